"""CPU oracle for the routed multi-tenant LoRA delta (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (``lora_delta_gb300``)
never touches it and shares no code with it; the two meet only through the
seeded inputs of ``lora_delta_gb300.inputs``.

The arithmetic lives in ``lora_oracle.c`` (plain loops, fp32 or fp64
accumulation, OpenMP over independent rows); this module only marshals numpy
arrays into it.  bf16 values are carried as ``uint16`` bit patterns.

Pages followed (cited per function in the C source):
  * "vllm/lora/punica_wrapper/punica_base.py": add_shrink / add_expand /
    add_lora_linear "Semantics", prefill_metadata.
  * "Module lora_delta" (metrale): LoraPair / LoraRoute layouts, the padded-rank
    invariant, apply_lora_bgmv, the scale rule.
  * "flashinfer.fused_moe.bgmv_moe_gemm1_lora_delta": the MoE FC1 formula,
    regular and shared-A / fused-B modes.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

import numpy as np

from .build_oracle import build as _build, library_path, override_path

_LIB = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_vpp = ctypes.c_void_p


def lib() -> ctypes.CDLL:
    """Load (building first if needed) the oracle shared library."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = override_path() or _build()  # _build is a no-op when up to date
    L = ctypes.CDLL(path)
    L.oracle_bf16_to_f32.restype = ctypes.c_float
    L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.oracle_f32_to_bf16.restype = ctypes.c_uint16
    L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    L.oracle_f64_to_bf16.restype = ctypes.c_uint16
    L.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
    L.oracle_lora_scale.restype = ctypes.c_float
    L.oracle_lora_scale.argtypes = [ctypes.c_float, ctypes.c_int, ctypes.c_int]
    L.oracle_pool_pack.restype = ctypes.c_int
    L.oracle_pool_pack.argtypes = [_vpp, _vpp, _vpp, _vpp] + [ctypes.c_int] * 4
    L.oracle_segments.restype = ctypes.c_int
    L.oracle_segments.argtypes = [_vpp, ctypes.c_int, ctypes.c_int, _vpp, _vpp, _u32p]
    L.oracle_shrink.restype = ctypes.c_int
    L.oracle_shrink.argtypes = [_vpp, _vpp, ctypes.c_int, ctypes.c_int, _vpp, _vpp, _vpp,
                                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _u32p]
    L.oracle_expand.restype = ctypes.c_int
    L.oracle_expand.argtypes = [_vpp, ctypes.c_int64, _vpp, _vpp, _vpp, _vpp, _vpp,
                                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                ctypes.c_int, ctypes.c_int, _u32p]
    L.oracle_delta.restype = ctypes.c_int
    L.oracle_delta.argtypes = [_vpp, ctypes.c_int64, _vpp, ctypes.c_int, ctypes.c_int, _vpp,
                               _vpp, _vpp, _vpp, _vpp, ctypes.c_int, ctypes.c_int,
                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _u32p]
    L.oracle_moe_fc1.restype = ctypes.c_int
    L.oracle_moe_fc1.argtypes = [_vpp, _vpp, _vpp, ctypes.c_int64, _vpp, ctypes.c_int64,
                                 ctypes.c_int, _vpp, _vpp] + [ctypes.c_int] * 7 + [
                                     ctypes.c_float, ctypes.c_int, _u32p]
    L.oracle_moe_w13.restype = ctypes.c_int
    L.oracle_moe_w13.argtypes = [_vpp, _vpp, _vpp, ctypes.c_int64, _vpp, ctypes.c_int64,
                                 ctypes.c_int, _vpp, _vpp, _vpp, ctypes.c_int, _vpp] + [
                                     ctypes.c_int] * 7 + [ctypes.c_float, ctypes.c_int,
                                                          ctypes.c_int, _u32p]
    L.oracle_moe_w2.restype = ctypes.c_int
    L.oracle_moe_w2.argtypes = [_vpp, _vpp, _vpp, ctypes.c_int64, _vpp, ctypes.c_int64,
                                _vpp, _vpp, _vpp, ctypes.c_int, _vpp, _vpp] + [
                                    ctypes.c_int] * 7 + [ctypes.c_float, ctypes.c_int,
                                                         ctypes.c_int, _u32p]
    L.oracle_gather_rank_blocks.restype = ctypes.c_int
    L.oracle_gather_rank_blocks.argtypes = [_vpp, _vpp] + [ctypes.c_int] * 4
    L.oracle_rank_sum.restype = ctypes.c_int
    L.oracle_rank_sum.argtypes = [_vpp, _vpp, ctypes.c_int, ctypes.c_int64]
    _LIB = L
    return L


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: bad argument (status {rc})")


# ---------------------------------------------------------------- bf16 ----

def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(a) -> np.ndarray:
    """Round-to-nearest-even float32 -> bf16 bits, element by element in C."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    f = lib().oracle_f32_to_bf16
    return np.array([f(float(v)) for v in a.ravel()], dtype=np.uint16).reshape(a.shape)


def f64_to_bf16(a) -> np.ndarray:
    """Round-to-nearest-even float64 -> bf16 bits (a single rounding)."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    f = lib().oracle_f64_to_bf16
    return np.array([f(float(v)) for v in a.ravel()], dtype=np.uint16).reshape(a.shape)


def lora_scale(alpha: float, r: int, use_rslora: bool = False) -> float:
    return float(lib().oracle_lora_scale(alpha, int(r), int(bool(use_rslora))))


# ---------------------------------------------------------------- pool ----

def pool_pack(a_r: np.ndarray, b_r: np.ndarray, R: int):
    """Pack one PEFT adapter (A_r [r,k_in], B_r [w,r]) into padded [R,k_in] / [w,R]."""
    a_r = np.ascontiguousarray(a_r, dtype=np.uint16)
    b_r = np.ascontiguousarray(b_r, dtype=np.uint16)
    r, k_in = a_r.shape
    w = b_r.shape[0]
    assert b_r.shape[1] == r
    a_slot = np.full((R, k_in), 0xFFFF, dtype=np.uint16)  # poison: pack must overwrite all
    b_slot = np.full((w, R), 0xFFFF, dtype=np.uint16)
    _check(lib().oracle_pool_pack(_p(a_slot), _p(b_slot), _p(a_r), _p(b_r), r, R, k_in, w),
           "pool_pack")
    return a_slot, b_slot


@dataclass
class OraclePool:
    """Host copy of one projection's adapter pool plus its routing tables.

    ``A[j]`` is ``[max_loras, R, k_in]`` and ``B[j]`` is ``[max_loras, w_j, R]``
    (bf16 bits); ``a_table``/``b_table`` are ``[S * max_loras]`` arrays of host
    addresses, 0 where a slot does not adapt slice j ("Module lora_delta",
    LoraRoute); ``scale_table`` is ``[max_loras]`` float32.
    """
    k_in: int
    widths: tuple
    max_loras: int
    R: int
    A: list = field(default_factory=list)
    B: list = field(default_factory=list)
    a_table: np.ndarray = None
    b_table: np.ndarray = None
    scale_table: np.ndarray = None

    @property
    def S(self):
        return len(self.widths)


def build_pool(case_adapters, k_in: int, widths, max_loras: int, R: int,
               use_rslora: bool = False) -> OraclePool:
    """Pack ``case_adapters`` (one entry per slot: None or an object with
    ``rank``, ``alpha``, ``A`` (per-slice [r,k_in]), ``B`` (per-slice [w_j,r]) and
    ``adapted`` (per-slice bool)) into an OraclePool using the oracle's packer."""
    S = len(widths)
    pool = OraclePool(k_in=k_in, widths=tuple(widths), max_loras=max_loras, R=R)
    pool.A = [np.zeros((max_loras, R, k_in), dtype=np.uint16) for _ in range(S)]
    pool.B = [np.zeros((max_loras, w, R), dtype=np.uint16) for w in widths]
    pool.a_table = np.zeros(S * max_loras, dtype=np.uint64)
    pool.b_table = np.zeros(S * max_loras, dtype=np.uint64)
    pool.scale_table = np.zeros(max_loras, dtype=np.float32)
    for s, ad in enumerate(case_adapters):
        if ad is None:
            continue
        pool.scale_table[s] = lora_scale(ad.alpha, ad.rank, use_rslora)
        for j in range(S):
            if not ad.adapted[j]:
                continue
            a_slot, b_slot = pool_pack(ad.A[j], ad.B[j], R)
            pool.A[j][s] = a_slot
            pool.B[j][s] = b_slot
            pool.a_table[j * max_loras + s] = pool.A[j][s].ctypes.data
            pool.b_table[j * max_loras + s] = pool.B[j][s].ctypes.data
    return pool


# ------------------------------------------------------------- routing ----

def segments(seq_slot: np.ndarray, max_loras: int):
    """Stable clustering of rows by slot: (perm, seg_start, err_word)."""
    seq_slot = np.ascontiguousarray(seq_slot, dtype=np.int32)
    n = seq_slot.shape[0]
    perm = np.full(max(n, 1), -1, dtype=np.int32)
    seg = np.zeros(max_loras + 1, dtype=np.int32)
    err = ctypes.c_uint32(0)
    _check(lib().oracle_segments(_p(seq_slot), n, max_loras, _p(perm), _p(seg),
                                 ctypes.byref(err)), "segments")
    return perm[: seg[-1]].copy(), seg, int(err.value)


# ----------------------------------------------------------- the delta ----

def shrink(x: np.ndarray, seq_slot: np.ndarray, pool: OraclePool, scale_table=None,
           h: np.ndarray | None = None, acc64: bool = False):
    """h[j, i, :] += scale_s * x[i] @ A_j,s^T; returns (h, err_word)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    seq_slot = np.ascontiguousarray(seq_slot, dtype=np.int32)
    n, k_in = x.shape
    if h is None:
        h = np.zeros((pool.S, n, pool.R), dtype=np.float32)
    st = None if scale_table is None else np.ascontiguousarray(scale_table, dtype=np.float32)
    err = ctypes.c_uint32(0)
    _check(lib().oracle_shrink(_p(h), _p(x), n, k_in, _p(seq_slot), _p(pool.a_table), _p(st),
                               pool.S, pool.R, pool.max_loras, int(acc64), ctypes.byref(err)),
           "shrink")
    return h, int(err.value)


def expand(out: np.ndarray, h: np.ndarray, seq_slot: np.ndarray, pool: OraclePool,
           scale_table=None, offset_start: int = 0, add_inputs: bool = True):
    """out[i, off_j + c] (+)= scale_s * h[j,i] . B_j,s[c]  (in place); returns err_word."""
    assert out.dtype == np.uint16 and out.flags["C_CONTIGUOUS"]
    h = np.ascontiguousarray(h, dtype=np.float32)
    seq_slot = np.ascontiguousarray(seq_slot, dtype=np.int32)
    n = seq_slot.shape[0]
    widths = np.ascontiguousarray(pool.widths, dtype=np.int32)
    st = None if scale_table is None else np.ascontiguousarray(scale_table, dtype=np.float32)
    err = ctypes.c_uint32(0)
    _check(lib().oracle_expand(_p(out), out.shape[1], _p(h), _p(seq_slot), _p(pool.b_table),
                               _p(st), _p(widths), pool.S, pool.R, n, pool.max_loras,
                               offset_start, int(add_inputs), ctypes.byref(err)), "expand")
    return int(err.value)


def delta(out: np.ndarray, x: np.ndarray, seq_slot: np.ndarray, pool: OraclePool,
          offset_start: int = 0, add_inputs: bool = True, acc64: bool = False,
          scale_table=None):
    """The routed delta, in place on ``out`` ([n, ld_out] bf16 bits); returns err_word."""
    assert out.dtype == np.uint16 and out.flags["C_CONTIGUOUS"]
    x = np.ascontiguousarray(x, dtype=np.uint16)
    seq_slot = np.ascontiguousarray(seq_slot, dtype=np.int32)
    n, k_in = x.shape
    widths = np.ascontiguousarray(pool.widths, dtype=np.int32)
    st = pool.scale_table if scale_table is None else np.ascontiguousarray(scale_table,
                                                                            dtype=np.float32)
    err = ctypes.c_uint32(0)
    _check(lib().oracle_delta(_p(out), out.shape[1], _p(x), n, k_in, _p(seq_slot),
                              _p(pool.a_table), _p(pool.b_table), _p(st), _p(widths), pool.S,
                              pool.R, pool.max_loras, offset_start, int(add_inputs), int(acc64),
                              ctypes.byref(err)), "delta")
    return int(err.value)


# ------------------------------------------------------------- MoE FC1 ----

def moe_fc1(x: np.ndarray, banks_a: list, banks_b: list, topk_ids: np.ndarray,
            lora_ids: np.ndarray, I: int, rank: int, scale: float, shared_a: bool,
            num_loras: int, acc64: bool = False):
    """MoE FC1 LoRA delta [T, top_k, 2I] (bf16 bits) and the error word.

    ``banks_a`` is ``[A_gate, A_up]`` (regular) or ``[A_shared]`` (shared mode),
    each ``[E, L, rank, H]``; ``banks_b`` is ``[B_gate, B_up]`` each ``[E, L, I, rank]``
    or ``[B_fused]`` ``[E, L, 2I, rank]``.  The pointer tables and element
    strides are derived from these arrays as the flashinfer page describes.
    """
    x = np.ascontiguousarray(x, dtype=np.uint16)
    T, H = x.shape
    topk_ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    lora_ids = np.ascontiguousarray(lora_ids, dtype=np.int32)
    top_k = topk_ids.shape[1]
    E = banks_a[0].shape[0]
    wa = np.array([bank[e].ctypes.data for bank in banks_a for e in range(E)], dtype=np.uint64)
    wb = np.array([bank[e].ctypes.data for bank in banks_b for e in range(E)], dtype=np.uint64)
    stride_a = int(np.prod(banks_a[0].shape[2:]))
    stride_b = int(np.prod(banks_b[0].shape[2:]))
    out = np.full((T, top_k, 2 * I), 0xFFFF, dtype=np.uint16)  # poison: every pair is written
    err = ctypes.c_uint32(0)
    _check(lib().oracle_moe_fc1(_p(out), _p(x), _p(wa), stride_a, _p(wb), stride_b,
                                int(bool(shared_a)), _p(topk_ids), _p(lora_ids), T, top_k, E, H,
                                I, rank, num_loras, float(scale), int(acc64), ctypes.byref(err)),
           "moe_fc1")
    return out, int(err.value)


# ------------------------------------------------- in-place MoE w13 / w2 ----

def _bank_tables(banks_a: list, banks_b: list):
    E = banks_a[0].shape[0]
    wa = np.array([bank[e].ctypes.data for bank in banks_a for e in range(E)], dtype=np.uint64)
    wb = np.array([bank[e].ctypes.data for bank in banks_b for e in range(E)], dtype=np.uint64)
    return E, wa, wb, int(np.prod(banks_a[0].shape[2:])), int(np.prod(banks_b[0].shape[2:]))


def _opt_i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def moe_w13(y: np.ndarray, x: np.ndarray, banks_a: list, banks_b: list, topk_ids: np.ndarray,
            lora_ids: np.ndarray, I: int, rank: int, scale: float, shared_a: bool,
            num_loras: int, expert_map=None, adapter_enabled=None, add_inputs: bool = True,
            acc64: bool = False):
    """add_lora_w13 on a copy of ``y`` [T, top_k, 2I] (bf16 bits); returns (y, err).

    Banks as for :func:`moe_fc1`, indexed by the local expert id.  ``expert_map``
    [n_global] int32 maps global expert ids to local ones (-1: not local);
    ``adapter_enabled`` [num_loras] int32 (0: the adapter adds nothing)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    T, H = x.shape
    topk_ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    lora_ids = np.ascontiguousarray(lora_ids, dtype=np.int32)
    top_k = topk_ids.shape[1]
    E, wa, wb, stride_a, stride_b = _bank_tables(banks_a, banks_b)
    emap, en = _opt_i32(expert_map), _opt_i32(adapter_enabled)
    out = np.array(y, dtype=np.uint16, copy=True, order="C")
    assert out.shape == (T, top_k, 2 * I)
    err = ctypes.c_uint32(0)
    _check(lib().oracle_moe_w13(_p(out), _p(x), _p(wa), stride_a, _p(wb), stride_b,
                                int(bool(shared_a)), _p(topk_ids), _p(lora_ids), _p(emap),
                                0 if emap is None else int(emap.size), _p(en), T, top_k, E, H,
                                I, rank, num_loras, float(scale), int(bool(add_inputs)),
                                int(acc64), ctypes.byref(err)), "moe_w13")
    return out, int(err.value)


def moe_w2(y: np.ndarray, x: np.ndarray, banks_a: list, banks_b: list, topk_ids: np.ndarray,
           lora_ids: np.ndarray, rank: int, scale: float, num_loras: int, expert_map=None,
           adapter_enabled=None, topk_weights=None, add_inputs: bool = True,
           acc64: bool = False):
    """add_lora_w2 on a copy of ``y`` [T, top_k, H] (bf16 bits); returns (y, err).

    ``x`` [T * top_k, I] holds one activation row per (token, slot);
    ``banks_a = [A_down]`` [E, L, rank, I], ``banks_b = [B_down]`` [E, L, H, rank];
    ``topk_weights`` [T, top_k] float32 or None."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    topk_ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    lora_ids = np.ascontiguousarray(lora_ids, dtype=np.int32)
    T, top_k = topk_ids.shape
    I = x.shape[1]
    assert x.shape[0] == T * top_k
    E, wa, wb, stride_a, stride_b = _bank_tables(banks_a, banks_b)
    H = banks_b[0].shape[2]
    emap, en = _opt_i32(expert_map), _opt_i32(adapter_enabled)
    wts = None if topk_weights is None else np.ascontiguousarray(topk_weights, dtype=np.float32)
    out = np.array(y, dtype=np.uint16, copy=True, order="C")
    assert out.shape == (T, top_k, H)
    err = ctypes.c_uint32(0)
    _check(lib().oracle_moe_w2(_p(out), _p(x), _p(wa), stride_a, _p(wb), stride_b,
                               _p(topk_ids), _p(lora_ids), _p(emap),
                               0 if emap is None else int(emap.size), _p(en), _p(wts), T, top_k,
                               E, H, I, rank, num_loras, float(scale), int(bool(add_inputs)),
                               int(acc64), ctypes.byref(err)), "moe_w2")
    return out, int(err.value)


# ------------------------------------------- tensor-parallel sharded forms ----
# "vllm.lora.fully_sharded_layers": the shrink and the expand run per rank on
# sharded adapters, with one collective on the fp32 h buffer in between.

def gather_rank_blocks(shards) -> np.ndarray:
    """Column parallel (_mcp_apply): the all-gather of the rank shards of h,
    ``shards`` [tp, S, n, Rs] -> h [S, n, tp * Rs] (rank p's block at p * Rs)."""
    sh = np.ascontiguousarray(shards, dtype=np.float32)
    tp, S, n, Rs = sh.shape
    h = np.empty((S, n, tp * Rs), dtype=np.float32)
    _check(lib().oracle_gather_rank_blocks(_p(h), _p(sh), tp, S, n, Rs), "gather_rank_blocks")
    return h


def rank_sum(parts) -> np.ndarray:
    """Row parallel (RowParallelLinearWithShardedLoRA apply): the all-reduce of
    the rank partials of h, ``parts`` [tp, ...] -> fp32 sum in rank order."""
    pa = np.ascontiguousarray(parts, dtype=np.float32)
    tp = pa.shape[0]
    h = np.empty(pa.shape[1:], dtype=np.float32)
    _check(lib().oracle_rank_sum(_p(h), _p(pa), tp, h.size), "rank_sum")
    return h


def shard_pool_a_rows(pool: OraclePool, tp: int, p: int) -> OraclePool:
    """Rank p's pool of the column-parallel form: rows p*R/tp .. (p+1)*R/tp - 1
    of every slot's padded A (the rank slice), B left whole (unused)."""
    Rs = pool.R // tp
    sp = OraclePool(k_in=pool.k_in, widths=pool.widths, max_loras=pool.max_loras, R=Rs)
    sp.A = [np.ascontiguousarray(a[:, p * Rs:(p + 1) * Rs, :]) for a in pool.A]
    sp.B = pool.B
    sp.scale_table = pool.scale_table
    sp.a_table = _table_like(pool.a_table, pool.A, sp.A)
    sp.b_table = pool.b_table
    return sp


def shard_pool_a_cols(pool: OraclePool, tp: int, p: int) -> OraclePool:
    """Rank p's pool of the row-parallel form: columns p*k_in/tp .. of every
    slot's A (the input slice, as x is sliced), B left whole (unused)."""
    ks = pool.k_in // tp
    sp = OraclePool(k_in=ks, widths=pool.widths, max_loras=pool.max_loras, R=pool.R)
    sp.A = [np.ascontiguousarray(a[:, :, p * ks:(p + 1) * ks]) for a in pool.A]
    sp.B = pool.B
    sp.scale_table = pool.scale_table
    sp.a_table = _table_like(pool.a_table, pool.A, sp.A)
    sp.b_table = pool.b_table
    return sp


def shard_pool_b_rows(pool: OraclePool, tp: int, p: int) -> OraclePool:
    """Rank p's pool for the expand of either form: output columns p*w_j/tp ..
    of every slice (rows of B), A left whole (unused)."""
    ws = tuple(w // tp for w in pool.widths)
    sp = OraclePool(k_in=pool.k_in, widths=ws, max_loras=pool.max_loras, R=pool.R)
    sp.A = pool.A
    sp.B = [np.ascontiguousarray(b[:, p * w:(p + 1) * w, :]) for b, w in zip(pool.B, ws)]
    sp.scale_table = pool.scale_table
    sp.a_table = pool.a_table
    sp.b_table = _table_like(pool.b_table, pool.B, sp.B)
    return sp


def _table_like(table, old, new):
    """Pointer table of ``new`` with the entries that are 0 in ``table`` kept 0."""
    S = len(old)
    L = old[0].shape[0]
    t = np.zeros_like(table)
    for j in range(S):
        for s in range(L):
            if table[j * L + s]:
                t[j * L + s] = new[j][s].ctypes.data
    return t
