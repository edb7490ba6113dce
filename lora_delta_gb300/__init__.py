"""GB300-native (sm_103a) routed multi-tenant LoRA delta.

Thin Python binding over the C ABI in ``include/lora_delta.h``: every function
here only marshals torch tensors into pointers and sizes, passes torch's
current CUDA stream, and turns a nonzero status into an exception.  All of the
arithmetic runs in the library's CUDA kernels; if the library is missing the
calls raise (there is no CPU or PyTorch fallback).

Pages the calls follow: "vllm/lora/punica_wrapper/punica_base.py" (add_shrink,
add_expand, add_lora_linear, prefill_metadata), "Module lora_delta" (LoraPair,
LoraRoute, apply_lora_bgmv, the scale rule) and
"flashinfer.fused_moe.bgmv_moe_gemm1_lora_delta".
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import LibraryMissing, lib, status_string

__all__ = [
    "LoraError", "LibraryMissing", "LoraPool", "lora_scale", "lora_pool_pack",
    "lora_workspace_size", "lora_workspace_min_size", "lora_route", "lora_route_scratch_size",
    "lora_route_with_scratch", "lora_shrink", "lora_expand", "lora_expand_gathered",
    "lora_delta_fused",
    "lora_delta_segmented", "lora_delta_fused_floor",
    "lora_moe_workspace_size", "lora_moe_fc1_delta", "lora_moe_w13_delta",
    "lora_moe_w2_delta", "lora_moe_w2_delta_routed", "lora_get_error", "new_error_word",
    "lora_delta_fused_noalloc", "lora_noalloc_scratch_bytes", "lora_set_wait_limit_ns",
    "WAIT_LIMIT_DEFAULT_NS",
]

# Default limit of the kernels' bounded waits (2 s of the GPU's global timer).
WAIT_LIMIT_DEFAULT_NS = 2_000_000_000


class LoraError(RuntimeError):
    def __init__(self, what: str, code: int):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


def _check(what: str, code: int):
    if code != 0:
        raise LoraError(what, code)


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def new_error_word(device=None) -> torch.Tensor:
    """A zeroed device error word (int32 view of the C uint32)."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def _widths_arg(widths):
    arr = (ctypes.c_int32 * len(widths))(*[int(w) for w in widths])
    return arr


# ---------------------------------------------------------------- scalars --

def lora_scale(alpha: float, r: int, use_rslora: bool = False) -> float:
    return float(lib().lora_scale(float(alpha), int(r), int(bool(use_rslora))))


def lora_set_wait_limit_ns(ns: int) -> int:
    """Set the limit of the kernels' bounded waits (ns of the GPU's global timer;
    0: give up at the first incomplete poll, for tests of the time-out path);
    returns the previous limit.  Process-wide, read by each launch."""
    return int(lib().lora_set_wait_limit_ns(int(ns)))


def lora_workspace_size(n: int, S: int, R: int, max_loras: int) -> int:
    return int(lib().lora_workspace_size(int(n), int(S), int(R), int(max_loras)))


def lora_workspace_min_size(n: int, S: int, R: int, max_loras: int) -> int:
    return int(lib().lora_workspace_min_size(int(n), int(S), int(R), int(max_loras)))


def lora_moe_workspace_size(T: int, top_k: int, E: int, num_loras: int, rank: int,
                            shared_a: bool) -> int:
    return int(lib().lora_moe_workspace_size(int(T), int(top_k), int(E), int(num_loras),
                                             int(rank), int(bool(shared_a))))


# Scratch workspaces the binding keeps for callers that pass none: one per
# (device, stream), grown when a call needs more and otherwise reused, so a
# steady stream of calls allocates nothing.  Calls on one stream run in
# order, so they may share one; calls on different streams get different ones.
_WS_CACHE: dict = {}


def _workspace(nbytes: int, workspace, device, stream=None):
    if workspace is not None:
        return workspace, workspace.numel() * workspace.element_size()
    if nbytes == 0:
        return None, 0
    device = torch.device(device)
    s = torch.cuda.current_stream(device) if stream is None else stream
    key = (device.index if device.index is not None else torch.cuda.current_device(),
           s.cuda_stream)
    ws = _WS_CACHE.get(key)
    if ws is None or ws.numel() < nbytes:
        _WS_CACHE.pop(key, None)
        with torch.cuda.stream(s):  # the allocator then reuses it on this stream only
            ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _WS_CACHE[key] = ws
    return ws, ws.numel()


# -------------------------------------------------------------------- pack --

def lora_pool_pack(a_slot: torch.Tensor, b_slot: torch.Tensor, a_r: torch.Tensor,
                   b_r: torch.Tensor, stream=None):
    """Pack PEFT ``a_r`` [r, k_in] / ``b_r`` [w, r] into padded ``a_slot`` [R, k_in] /
    ``b_slot`` [w, R] (all bf16 device tensors)."""
    for t, nm in ((a_slot, "a_slot"), (b_slot, "b_slot"), (a_r, "a_r"), (b_r, "b_r")):
        _dev(t, nm, torch.bfloat16)
    R, k_in = a_slot.shape
    r = a_r.shape[0]
    w = b_slot.shape[0]
    if a_r.shape[1] != k_in or b_r.shape != (w, r) or b_slot.shape[1] != R:
        raise ValueError("lora_pool_pack: inconsistent shapes")
    _check("lora_pool_pack", lib().lora_pool_pack(_ptr(a_slot), _ptr(b_slot), _ptr(a_r),
                                                  _ptr(b_r), r, R, k_in, w, _stream(stream)))


class LoraPool:
    """Device adapter pool of one projection plus its routing tables.

    Per slice j: ``A[j]`` [max_loras, R, k_in] and ``B[j]`` [max_loras, w_j, R] bf16,
    zeroed at creation ("Module lora_delta": the pool is zeroed before packing);
    ``a_table`` / ``b_table`` [S * max_loras] int64 device addresses (0 = slot does
    not adapt the slice); ``scale_table`` [max_loras] float32.
    """

    def __init__(self, k_in: int, widths, max_loras: int, R: int, device="cuda"):
        self.k_in, self.widths, self.max_loras, self.R = int(k_in), tuple(widths), max_loras, R
        self.device = torch.device(device)
        S = len(self.widths)
        self.A = [torch.zeros(max_loras, R, k_in, dtype=torch.bfloat16, device=device)
                  for _ in range(S)]
        self.B = [torch.zeros(max_loras, w, R, dtype=torch.bfloat16, device=device)
                  for w in self.widths]
        self._a_host = [0] * (S * max_loras)
        self._b_host = [0] * (S * max_loras)
        self.scale_table = torch.zeros(max_loras, dtype=torch.float32, device=device)
        self.a_table = torch.zeros(S * max_loras, dtype=torch.int64, device=device)
        self.b_table = torch.zeros(S * max_loras, dtype=torch.int64, device=device)

    @property
    def S(self):
        return len(self.widths)

    def pack(self, slot: int, a_r_list, b_r_list, alpha: float, rank: int,
             use_rslora: bool = False, adapted=None):
        """Pack one slot's PEFT tensors (device bf16: per slice [rank, k_in] / [w_j, rank])."""
        adapted = [True] * self.S if adapted is None else list(adapted)
        self.scale_table[slot] = lora_scale(alpha, rank, use_rslora)
        for j in range(self.S):
            if adapted[j]:
                lora_pool_pack(self.A[j][slot], self.B[j][slot], a_r_list[j], b_r_list[j])
                self._a_host[j * self.max_loras + slot] = self.A[j][slot].data_ptr()
                self._b_host[j * self.max_loras + slot] = self.B[j][slot].data_ptr()
            else:
                self._a_host[j * self.max_loras + slot] = 0
                self._b_host[j * self.max_loras + slot] = 0
        self.a_table.copy_(torch.tensor(self._a_host, dtype=torch.int64))
        self.b_table.copy_(torch.tensor(self._b_host, dtype=torch.int64))

    def nbytes(self) -> int:
        return sum(t.numel() * 2 for t in self.A + self.B)


# ----------------------------------------------------------------- routing --

def lora_route(seq_slot: torch.Tensor, max_loras: int, perm=None, seg_start=None, err=None,
               stream=None):
    """Stable clustering of rows by slot: returns (perm [n], seg_start [max_loras+2])."""
    _dev(seq_slot, "seq_slot", torch.int32)
    n = seq_slot.numel()
    dev = seq_slot.device
    perm = torch.empty(max(n, 1), dtype=torch.int32, device=dev) if perm is None else perm
    seg_start = (torch.empty(max_loras + 2, dtype=torch.int32, device=dev)
                 if seg_start is None else seg_start)
    _check("lora_route", lib().lora_route(_ptr(perm), _ptr(seg_start), _ptr(seq_slot), n,
                                          int(max_loras), _ptr(err), _stream(stream)))
    return perm, seg_start


def lora_route_scratch_size(n: int, max_loras: int) -> int:
    return int(lib().lora_route_scratch_size(int(n), int(max_loras)))


def lora_route_with_scratch(seq_slot: torch.Tensor, max_loras: int, scratch=None, perm=None,
                            seg_start=None, err=None, stream=None):
    """lora_route for large batches (many CTAs), with caller scratch; same result."""
    _dev(seq_slot, "seq_slot", torch.int32)
    n = seq_slot.numel()
    dev = seq_slot.device
    perm = torch.empty(max(n, 1), dtype=torch.int32, device=dev) if perm is None else perm
    seg_start = (torch.empty(max_loras + 2, dtype=torch.int32, device=dev)
                 if seg_start is None else seg_start)
    scratch, sbytes = _workspace(lora_route_scratch_size(n, max_loras), scratch, dev, stream)
    _check("lora_route_with_scratch",
           lib().lora_route_with_scratch(_ptr(perm), _ptr(seg_start), _ptr(seq_slot), n,
                                         int(max_loras), _ptr(scratch), sbytes, _ptr(err),
                                         _stream(stream)))
    return perm, seg_start


# --------------------------------------------------------------- the delta --

def lora_shrink(h, x, seq_slot, pool: LoraPool, scale_table=None, workspace=None, err=None,
                stream=None):
    """h[j, i, :] += scale_s * x[i] A_j,s^T (h [S, n, R] float32)."""
    _dev(h, "h", torch.float32)
    _dev(x, "x", torch.bfloat16)
    _dev(seq_slot, "seq_slot", torch.int32)
    n, k_in = x.shape
    ws, wsb = _workspace(lora_workspace_size(n, pool.S, pool.R, pool.max_loras) if n > 1024
                         else 0, workspace, x.device, stream)
    _check("lora_shrink", lib().lora_shrink(
        _ptr(h), _ptr(x), n, k_in, _ptr(seq_slot), _ptr(pool.a_table), _ptr(scale_table),
        pool.S, pool.R, pool.max_loras, _ptr(ws), wsb, _ptr(err), _stream(stream)))


def lora_expand(out, h, seq_slot, pool: LoraPool, scale_table=None, offset_start: int = 0,
                add_inputs: bool = True, workspace=None, err=None, stream=None):
    """out[i, off_j + c] (+)= scale_s * h[j, i] . B_j,s[c] (out [n, ld_out] bf16)."""
    _dev(out, "out", torch.bfloat16)
    _dev(h, "h", torch.float32)
    _dev(seq_slot, "seq_slot", torch.int32)
    n, ld_out = out.shape
    ws, wsb = _workspace(lora_workspace_size(n, pool.S, pool.R, pool.max_loras) if n > 1024
                         else 0, workspace, out.device, stream)
    w = _widths_arg(pool.widths)
    _check("lora_expand", lib().lora_expand(
        _ptr(out), ld_out, _ptr(h), _ptr(seq_slot), _ptr(pool.b_table), _ptr(scale_table), w,
        pool.S, pool.R, n, pool.max_loras, int(offset_start), int(bool(add_inputs)), _ptr(ws),
        wsb, _ptr(err), _stream(stream)))


def lora_expand_gathered(out, h_parts, seq_slot, pool: LoraPool, scale_table=None,
                         offset_start: int = 0, add_inputs: bool = True, workspace=None,
                         err=None, stream=None):
    """lora_expand on the all-gather of rank-sharded shrinks: ``h_parts``
    [parts, S, n, R / parts] float32 (rank-major), ``pool`` the pool of this rank's
    output columns with the whole rank R."""
    _dev(out, "out", torch.bfloat16)
    _dev(h_parts, "h_parts", torch.float32)
    _dev(seq_slot, "seq_slot", torch.int32)
    n, ld_out = out.shape
    parts = h_parts.shape[0]
    if h_parts.dim() != 4 or h_parts.shape[1:3] != (pool.S, n) or \
            h_parts.shape[3] * parts != pool.R:
        raise ValueError("h_parts must be [parts, S, n, R / parts]")
    ws, wsb = _workspace(lora_workspace_size(n, pool.S, pool.R, pool.max_loras) if n > 1024
                         else 0, workspace, out.device, stream)
    w = _widths_arg(pool.widths)
    _check("lora_expand_gathered", lib().lora_expand_gathered(
        _ptr(out), ld_out, _ptr(h_parts), parts, _ptr(seq_slot), _ptr(pool.b_table),
        _ptr(scale_table), w, pool.S, pool.R, n, pool.max_loras, int(offset_start),
        int(bool(add_inputs)), _ptr(ws), wsb, _ptr(err), _stream(stream)))


def lora_delta_fused(out, x, seq_slot, pool: LoraPool, offset_start: int = 0,
                     add_inputs: bool = True, scale_table=None, workspace=None, err=None,
                     stream=None):
    """out[i, slices] (+)= scale_s * (x[i] A_s^T) B_s^T over the pool's slices, in place."""
    _dev(out, "out", torch.bfloat16)
    _dev(x, "x", torch.bfloat16)
    _dev(seq_slot, "seq_slot", torch.int32)
    n, k_in = x.shape
    if out.shape[0] != n:
        raise ValueError("out and x must have the same number of rows")
    st = pool.scale_table if scale_table is None else scale_table
    # batches of >= 256 rows get a workspace: they are clustered by slot, and
    # slots with many rows take the tensor-core path
    ws, wsb = _workspace(lora_workspace_size(n, pool.S, pool.R, pool.max_loras) if n >= 256
                         else 0, workspace, x.device, stream)
    w = _widths_arg(pool.widths)
    _check("lora_delta_fused", lib().lora_delta_fused(
        _ptr(out), out.shape[1], _ptr(x), n, k_in, _ptr(seq_slot), _ptr(pool.a_table),
        _ptr(pool.b_table), _ptr(st), w, pool.S, pool.R, pool.max_loras, int(offset_start),
        int(bool(add_inputs)), _ptr(ws), wsb, _ptr(err), _stream(stream)))


def lora_delta_fused_floor(out, x, seq_slot, pool: LoraPool, offset_start: int = 0, stream=None):
    """Measurement aid: the bytes and launch plan of ``lora_delta_fused`` on a small
    batch with no arithmetic (``out`` is written back unchanged)."""
    _dev(out, "out", torch.bfloat16)
    _dev(x, "x", torch.bfloat16)
    _dev(seq_slot, "seq_slot", torch.int32)
    n, k_in = x.shape
    w = _widths_arg(pool.widths)
    _check("lora_delta_fused_floor", lib().lora_delta_fused_floor(
        _ptr(out), out.shape[1], _ptr(x), n, k_in, _ptr(seq_slot), _ptr(pool.a_table),
        _ptr(pool.b_table), w, pool.S, pool.R, pool.max_loras, int(offset_start),
        _stream(stream)))


def lora_delta_segmented(out, x, seg_start, pool: LoraPool, offset_start: int = 0,
                         add_inputs: bool = True, scale_table=None, workspace=None, err=None,
                         stream=None):
    """The delta on rows grouped by adapter: rows seg_start[s]..seg_start[s+1]
    take pool slot s (e.g. expert-sorted MoE rows, one adapter per expert)."""
    _dev(out, "out", torch.bfloat16)
    _dev(x, "x", torch.bfloat16)
    _dev(seg_start, "seg_start", torch.int32)
    n, k_in = x.shape
    if out.shape[0] != n:
        raise ValueError("out and x must have the same number of rows")
    n_segs = seg_start.numel() - 1
    if n_segs != pool.max_loras:
        raise ValueError("seg_start must have pool.max_loras + 1 entries")
    st = pool.scale_table if scale_table is None else scale_table
    ws, wsb = _workspace(lora_workspace_size(n, pool.S, pool.R, n_segs), workspace, x.device,
                         stream)
    w = _widths_arg(pool.widths)
    _check("lora_delta_segmented", lib().lora_delta_segmented(
        _ptr(out), out.shape[1], _ptr(x), n, k_in, _ptr(seg_start), n_segs, _ptr(pool.a_table),
        _ptr(pool.b_table), _ptr(st), w, pool.S, pool.R, int(offset_start),
        int(bool(add_inputs)), _ptr(ws), wsb, _ptr(err), _stream(stream)))


def lora_delta_fused_noalloc(out, x, seq_slot, pool: LoraPool, offset_start: int = 0,
                             add_inputs: bool = True, scale_table=None, err=None, stream=None):
    """``lora_delta_fused`` for callers that cannot allocate: the scratch is the
    library's own fixed buffer (``lora_noalloc_scratch_bytes()``), shared by all
    calls; calls that overlap on the GPU race, and a batch that needs more scratch
    raises LoraError(LORA_ERR_TOO_LARGE)."""
    _dev(out, "out", torch.bfloat16)
    _dev(x, "x", torch.bfloat16)
    _dev(seq_slot, "seq_slot", torch.int32)
    n, k_in = x.shape
    if out.shape[0] != n:
        raise ValueError("out and x must have the same number of rows")
    st = pool.scale_table if scale_table is None else scale_table
    w = _widths_arg(pool.widths)
    _check("lora_delta_fused_noalloc", lib().lora_delta_fused_noalloc(
        _ptr(out), out.shape[1], _ptr(x), n, k_in, _ptr(seq_slot), _ptr(pool.a_table),
        _ptr(pool.b_table), _ptr(st), w, pool.S, pool.R, pool.max_loras, int(offset_start),
        int(bool(add_inputs)), _ptr(err), _stream(stream)))


def lora_noalloc_scratch_bytes() -> int:
    return int(lib().lora_noalloc_scratch_bytes())


def lora_moe_fc1_delta(out, x, w_ptr_a, stride_a: int, w_ptr_b, stride_b: int, shared_a: bool,
                       topk_ids, lora_ids, E: int, I: int, rank: int, num_loras: int,
                       scale: float, workspace=None, err=None, stream=None):
    """MoE FC1 delta into ``out`` [T, top_k, 2I] bf16 (fully written)."""
    _dev(out, "out", torch.bfloat16)
    _dev(x, "x", torch.bfloat16)
    _dev(topk_ids, "topk_ids", torch.int32)
    _dev(lora_ids, "lora_ids", torch.int32)
    _dev(w_ptr_a, "w_ptr_a", torch.int64)
    _dev(w_ptr_b, "w_ptr_b", torch.int64)
    T, H = x.shape
    top_k = topk_ids.shape[1]
    ws, wsb = _workspace(lora_moe_workspace_size(T, top_k, E, num_loras, rank, shared_a),
                         workspace, x.device, stream)
    _check("lora_moe_fc1_delta", lib().lora_moe_fc1_delta(
        _ptr(out), _ptr(x), _ptr(w_ptr_a), int(stride_a), _ptr(w_ptr_b), int(stride_b),
        int(bool(shared_a)), _ptr(topk_ids), _ptr(lora_ids), T, top_k, int(E), H, int(I),
        int(rank), int(num_loras), float(scale), _ptr(ws), wsb, _ptr(err), _stream(stream)))


def _opt_dev(t, name, dtype):
    if t is None:
        return None
    _dev(t, name, dtype)
    return t


def lora_moe_w13_delta(y, x, w_ptr_a, stride_a: int, w_ptr_b, stride_b: int, shared_a: bool,
                       topk_ids, lora_ids, E: int, I: int, rank: int, num_loras: int,
                       scale: float, expert_map=None, adapter_enabled=None,
                       add_inputs: bool = True, workspace=None, err=None, stream=None):
    """add_lora_w13: the gate/up delta added in place to ``y`` [T, top_k, 2I] bf16."""
    _dev(y, "y", torch.bfloat16)
    _dev(x, "x", torch.bfloat16)
    _dev(topk_ids, "topk_ids", torch.int32)
    _dev(lora_ids, "lora_ids", torch.int32)
    _dev(w_ptr_a, "w_ptr_a", torch.int64)
    _dev(w_ptr_b, "w_ptr_b", torch.int64)
    _opt_dev(expert_map, "expert_map", torch.int32)
    _opt_dev(adapter_enabled, "adapter_enabled", torch.int32)
    T, H = x.shape
    top_k = topk_ids.shape[1]
    ws, wsb = _workspace(lora_moe_workspace_size(T, top_k, E, num_loras, rank, shared_a),
                         workspace, x.device, stream)
    _check("lora_moe_w13_delta", lib().lora_moe_w13_delta(
        _ptr(y), _ptr(x), _ptr(w_ptr_a), int(stride_a), _ptr(w_ptr_b), int(stride_b),
        int(bool(shared_a)), _ptr(topk_ids), _ptr(lora_ids), _ptr(expert_map),
        0 if expert_map is None else expert_map.numel(), _ptr(adapter_enabled), T, top_k,
        int(E), H, int(I), int(rank), int(num_loras), float(scale), int(bool(add_inputs)),
        _ptr(ws), wsb, _ptr(err), _stream(stream)))


def lora_moe_w2_delta(y, x, w_ptr_a, stride_a: int, w_ptr_b, stride_b: int, topk_ids,
                      lora_ids, E: int, H: int, rank: int, num_loras: int, scale: float,
                      expert_map=None, adapter_enabled=None, topk_weights=None,
                      add_inputs: bool = True, workspace=None, err=None, stream=None):
    """add_lora_w2: the down delta added in place to ``y`` [T, top_k, H] bf16 from the
    per-pair activations ``x`` [T * top_k, I]."""
    _dev(y, "y", torch.bfloat16)
    _dev(x, "x", torch.bfloat16)
    _dev(topk_ids, "topk_ids", torch.int32)
    _dev(lora_ids, "lora_ids", torch.int32)
    _dev(w_ptr_a, "w_ptr_a", torch.int64)
    _dev(w_ptr_b, "w_ptr_b", torch.int64)
    _opt_dev(expert_map, "expert_map", torch.int32)
    _opt_dev(adapter_enabled, "adapter_enabled", torch.int32)
    _opt_dev(topk_weights, "topk_weights", torch.float32)
    T, top_k = topk_ids.shape
    I = x.shape[1]
    if x.shape[0] != T * top_k:
        raise ValueError("x must hold one row per (token, slot) pair")
    ws, wsb = _workspace(lora_moe_workspace_size(T, top_k, E, num_loras, rank, True),
                         workspace, x.device, stream)
    _check("lora_moe_w2_delta", lib().lora_moe_w2_delta(
        _ptr(y), _ptr(x), _ptr(w_ptr_a), int(stride_a), _ptr(w_ptr_b), int(stride_b),
        _ptr(topk_ids), _ptr(lora_ids), _ptr(expert_map),
        0 if expert_map is None else expert_map.numel(), _ptr(adapter_enabled),
        _ptr(topk_weights), T, top_k, int(E), int(H), I, int(rank), int(num_loras),
        float(scale), int(bool(add_inputs)), _ptr(ws), wsb, _ptr(err), _stream(stream)))


def lora_moe_w2_delta_routed(y, x, w_ptr_a, stride_a: int, w_ptr_b, stride_b: int, T: int,
                             top_k: int, E: int, H: int, rank: int, num_loras: int,
                             scale: float, workspace, topk_weights=None, add_inputs: bool = True,
                             err=None, stream=None):
    """add_lora_w2 on the routing that the preceding ``lora_moe_w13_delta`` left in
    ``workspace`` (the same T, top_k, E, num_loras and routing arrays; the
    workspace untouched since): no second sort of the pairs."""
    _dev(y, "y", torch.bfloat16)
    _dev(x, "x", torch.bfloat16)
    _dev(w_ptr_a, "w_ptr_a", torch.int64)
    _dev(w_ptr_b, "w_ptr_b", torch.int64)
    _opt_dev(topk_weights, "topk_weights", torch.float32)
    if workspace is None:
        raise ValueError("lora_moe_w2_delta_routed needs the w13 call's workspace")
    I = x.shape[1]
    if x.shape[0] != T * top_k:
        raise ValueError("x must hold one row per (token, slot) pair")
    _check("lora_moe_w2_delta_routed", lib().lora_moe_w2_delta_routed(
        _ptr(y), _ptr(x), _ptr(w_ptr_a), int(stride_a), _ptr(w_ptr_b), int(stride_b),
        _ptr(topk_weights), int(T), int(top_k), int(E), int(H), I, int(rank), int(num_loras),
        float(scale), int(bool(add_inputs)), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(err), _stream(stream)))


def lora_get_error(err: torch.Tensor, clear: bool = True, stream=None) -> int:
    """Synchronize the stream and return the device error word (clearing it)."""
    host = ctypes.c_uint32(0)
    _check("lora_get_error", lib().lora_get_error(_ptr(err), ctypes.byref(host), int(clear),
                                                  _stream(stream)))
    return int(host.value)
