"""Seeded synthetic inputs for the routed LoRA delta and the MoE FC1 delta.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no packing, no scale rule, no contraction).  The GPU path
and the CPU oracle each consume its output on their own.

Distributions (the workloads' stated recipe; readings of what the recipe
leaves open are marked "reading"):
  * x ~ N(0, 1) (reading: an activation has no fan-in), or, with
    ``x_scaled=True``, N(0, 1) / sqrt(k_in) (the literal reading).
  * PEFT lora_A [r, k_in] ~ N(0, 1) / sqrt(k_in); lora_B [w, r] ~ N(0, 1) /
    sqrt(r) with r the adapter's true rank (reading: the pad columns are zero
    anyway).
  * the initial ``out`` ~ N(0, 1), or all zeros with ``out0="zero"``.
  * every value drawn in float32 and rounded to bf16 (round-to-nearest-even,
    done by torch's dtype conversion); bf16 travels as uint16 bit patterns.
Seeds: numpy ``default_rng(seed)``; the five standard workloads use seeds
1234 .. 1238 in the order tiny, decode qkv, prefill gate_up, skewed, MoE FC1.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 array -> bf16 bit patterns (uint16), round-to-nearest-even."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return to_bf16_bits(a)


@dataclass
class Adapter:
    """One slot's PEFT adapter: per slice A_r [rank, k_in] and B_r [w_j, rank]."""
    rank: int
    alpha: float
    A: list
    B: list
    adapted: list  # per slice: does this slot adapt the slice at all


@dataclass
class LinearCase:
    """A routed-delta workload: rows x, routing seq_slot, the slot adapters and
    the initial output (which the delta updates in place)."""
    name: str
    seed: int
    n: int
    k_in: int
    widths: tuple
    max_loras: int
    max_rank: int
    x: np.ndarray          # [n, k_in] bf16 bits
    out0: np.ndarray       # [n, ld_out] bf16 bits
    seq_slot: np.ndarray   # [n] int32
    adapters: list         # [max_loras] Adapter | None
    use_rslora: bool = False
    offset_start: int = 0

    @property
    def ld_out(self) -> int:
        return int(self.out0.shape[1])

    @property
    def S(self) -> int:
        return len(self.widths)


def make_adapters(rng, k_in: int, widths, ranks, alpha: float, adapted=None) -> list:
    """Adapters for slots with ``ranks[s] > 0`` (None where ranks[s] <= 0)."""
    out = []
    for s, r in enumerate(ranks):
        if r is None or r <= 0:
            out.append(None)
            continue
        A = [_normal_bf16(rng, (r, k_in), 1.0 / np.sqrt(k_in)) for _ in widths]
        B = [_normal_bf16(rng, (w, r), 1.0 / np.sqrt(r)) for w in widths]
        ad = [True] * len(widths) if adapted is None else list(adapted[s])
        out.append(Adapter(rank=int(r), alpha=float(alpha), A=A, B=B, adapted=ad))
    return out


def linear_case(seed: int, n: int, k_in: int, widths, max_loras: int, max_rank: int,
                ranks, alpha: float, seq_slot: np.ndarray | None = None,
                p_none: float = 0.0, x_scaled: bool = False, out0: str = "normal",
                ld_out: int | None = None, offset_start: int = 0, adapted=None,
                use_rslora: bool = False, name: str = "custom") -> LinearCase:
    """Generic routed-delta case.  Without ``seq_slot`` the slots are uniform over
    ``[0, max_loras)`` with probability ``p_none`` of -1 (no delta)."""
    rng = np.random.default_rng(seed)
    widths = tuple(int(w) for w in widths)
    if seq_slot is None:
        seq_slot = rng.integers(0, max_loras, size=n).astype(np.int32)
        if p_none > 0:
            seq_slot[rng.random(n) < p_none] = -1
    seq_slot = np.ascontiguousarray(seq_slot, dtype=np.int32)
    adapters = make_adapters(rng, k_in, widths, ranks, alpha, adapted)
    x = _normal_bf16(rng, (n, k_in), (1.0 / np.sqrt(k_in)) if x_scaled else 1.0)
    if ld_out is None:
        ld_out = offset_start + sum(widths)
    if out0 == "zero":
        o = np.zeros((n, ld_out), dtype=np.uint16)
    else:
        o = _normal_bf16(rng, (n, ld_out))
    return LinearCase(name=name, seed=seed, n=n, k_in=k_in, widths=widths,
                      max_loras=max_loras, max_rank=max_rank, x=x, out0=o,
                      seq_slot=seq_slot, adapters=adapters, use_rslora=use_rslora,
                      offset_start=offset_start)


# ----------------------------------------------------- standard workloads --

def tiny_case(seed: int = 1234, **kw) -> LinearCase:
    """n=8, k_in=256, one 256-wide slice, 4 slots of ranks 8,16,4,16 padded to 16,
    slots uniform in {-1,0,1,2,3}, alpha 16 (scale 16/r)."""
    rng = np.random.default_rng(seed + 10_000)
    seq = rng.integers(-1, 4, size=8).astype(np.int32)
    return linear_case(seed, 8, 256, (256,), 4, 16, [8, 16, 4, 16], 16.0, seq_slot=seq,
                       name="tiny routed delta n=8 k_in=256 n_out=256", **kw)


def decode_qkv_case(seed: int = 1235, **kw) -> LinearCase:
    """Decode BGMV qkv: n=64, k_in=4096, slices (4096,1024,1024), 16 slots all rank 16,
    slots uniform over 16 with 10% -1, alpha 32."""
    return linear_case(seed, 64, 4096, (4096, 1024, 1024), 16, 16, [16] * 16, 32.0,
                       p_none=0.10, name="decode BGMV qkv n=64 k_in=4096 slices 4096/1024/1024",
                       **kw)


def prefill_segments(rng: np.random.Generator, n_tokens: int, n_segments: int,
                     lo: int, hi: int) -> np.ndarray:
    """Segment lengths drawn uniform in [lo, hi], rescaled to sum to n_tokens
    (reading: floor, then the remainder to the largest fractional parts, min 1)."""
    raw = rng.integers(lo, hi + 1, size=n_segments).astype(np.float64)
    scaled = raw * (n_tokens / raw.sum())
    lens = np.floor(scaled).astype(np.int64)
    lens = np.maximum(lens, 1)
    rem = n_tokens - int(lens.sum())
    if rem > 0:
        order = np.argsort(-(scaled - np.floor(scaled)), kind="stable")
        for i in range(rem):
            lens[order[i % n_segments]] += 1
    while lens.sum() > n_tokens:  # only reachable when the min-1 rule bit
        lens[int(np.argmax(lens))] -= 1
    return lens


def prefill_gate_up_case(seed: int = 1236, n_tokens: int = 8192, n_segments: int = 32,
                         seg_lo: int = 16, seg_hi: int = 1024, k_in: int = 4096,
                         widths=(14336, 14336), **kw) -> LinearCase:
    """Prefill SGMV gate_up: 8192 tokens in 32 segments (lengths uniform 16..1024,
    rescaled to 8192), each segment on a slot uniform over 8, rows then randomly
    permuted (rows unsorted); k_in 4096, slices (14336, 14336), max_rank 32 (all
    ranks 32, reading), alpha 32 (reading: as the decode workload)."""
    rng = np.random.default_rng(seed + 10_000)
    lens = prefill_segments(rng, n_tokens, n_segments, seg_lo, seg_hi)
    seg_slot = rng.integers(0, 8, size=n_segments)
    seq = np.repeat(seg_slot, lens).astype(np.int32)
    seq = seq[rng.permutation(n_tokens)]
    return linear_case(seed, n_tokens, k_in, widths, 8, 32, [32] * 8, 32.0, seq_slot=seq,
                       name=f"prefill SGMV gate_up {n_tokens} tokens in {n_segments} segments",
                       **kw)


def zipf_slots(rng: np.random.Generator, n: int, n_slots: int, a: float,
               p_none: float) -> np.ndarray:
    """Slot k-1 with probability proportional to k^-a (k = 1..n_slots), -1 with p_none."""
    w = np.arange(1, n_slots + 1, dtype=np.float64) ** (-a)
    w /= w.sum()
    seq = rng.choice(n_slots, size=n, p=w).astype(np.int32)
    seq[rng.random(n) < p_none] = -1
    return seq


SKEWED_PROJECTIONS = ((5120, 5120), (13824, 5120))


def skewed_case(proj: int, seed: int = 1237, **kw) -> LinearCase:
    """Skewed many-adapter decode, projection ``proj`` (0: 5120->5120, 1: 13824->5120):
    n=1024, 128 slots, ranks uniform in {8,16,32,64} padded to 64, Zipf(1.1)
    popularity with 5% -1, alpha 32 (reading).  Both projections share the
    routing and the ranks; their weights differ."""
    rng = np.random.default_rng(seed + 10_000)
    seq = zipf_slots(rng, 1024, 128, 1.1, 0.05)
    ranks = rng.choice(np.array([8, 16, 32, 64]), size=128).tolist()
    k_in, n_out = SKEWED_PROJECTIONS[proj]
    return linear_case(seed + 100 * proj, 1024, k_in, (n_out,), 128, 64, ranks, 32.0,
                       seq_slot=seq, name=f"skewed decode proj{proj + 1} {k_in}->{n_out}", **kw)


# ---------------------------------------------------------------- MoE FC1 --

@dataclass
class MoeCase:
    """Routed-MoE FC1 workload.  Banks are per expert: ``A_banks`` is
    ``[A_gate, A_up]`` (regular) or ``[A_shared]``, each ``[E, L, rank, H]``;
    ``B_banks`` is ``[B_gate, B_up]`` each ``[E, L, I, rank]`` or ``[B_fused]``
    ``[E, L, 2I, rank]``.  Adapter l of expert e's bank starts l * stride
    elements after the bank base, stride = rank*H (A) or I*rank / 2I*rank (B)."""
    name: str
    seed: int
    T: int
    top_k: int
    E: int
    H: int
    I: int
    rank: int
    L: int
    scale: float
    shared_a: bool
    x: np.ndarray
    topk_ids: np.ndarray
    lora_ids: np.ndarray
    A_banks: list
    B_banks: list = field(default_factory=list)


def duplicate_experts(topk: np.ndarray, frac: float, seed: int) -> np.ndarray:
    """A copy of ``topk`` [T, top_k] in which a fraction ``frac`` of the tokens
    repeat experts: in each such token, between 1 and top_k - 1 of its slots
    (chosen at random) take the id of another slot of the same token, so that
    one token reaches one expert through two or more slots.  Nothing in the
    pages makes a token's experts distinct, so the path has to accept this.
    Drawn from its own generator: the default workloads do not change."""
    out = np.array(topk, dtype=np.int32, copy=True)
    T, k = out.shape
    if k < 2 or frac <= 0:
        return out
    rng = np.random.default_rng(seed + 50_000)
    for t in np.flatnonzero(rng.random(T) < frac):
        n_dup = int(rng.integers(1, k))
        slots = rng.permutation(k)
        src = slots[n_dup:]
        for j in slots[:n_dup]:
            out[t, j] = out[t, int(rng.choice(src))]
    return out


def moe_case(shared_a: bool = False, seed: int = 1238, T: int = 2048, top_k: int = 8,
             E: int = 64, H: int = 2048, I: int = 768, rank: int = 16, L: int = 8,
             scale: float = 2.0, p_none: float = 0.2, x_scaled: bool = False,
             dup_frac: float = 0.0) -> MoeCase:
    """MoE FC1 LoRA delta: T tokens, top_k distinct experts of E per token (uniform),
    lora_ids uniform over L with p_none of -1, A ~ N(0,1)/sqrt(H), B ~ N(0,1)/sqrt(rank).
    With ``dup_frac`` > 0, that fraction of the tokens repeat experts
    (``duplicate_experts``)."""
    rng = np.random.default_rng(seed + (1 if shared_a else 0) * 7)
    topk = np.stack([rng.permutation(E)[:top_k] for _ in range(T)]).astype(np.int32)
    lora = rng.integers(0, L, size=T).astype(np.int32)
    lora[rng.random(T) < p_none] = -1
    x = _normal_bf16(rng, (T, H), (1.0 / np.sqrt(H)) if x_scaled else 1.0)
    n_a = 1 if shared_a else 2
    A = [_normal_bf16(rng, (E, L, rank, H), 1.0 / np.sqrt(H)) for _ in range(n_a)]
    if shared_a:
        B = [_normal_bf16(rng, (E, L, 2 * I, rank), 1.0 / np.sqrt(rank))]
    else:
        B = [_normal_bf16(rng, (E, L, I, rank), 1.0 / np.sqrt(rank)) for _ in range(2)]
    if dup_frac > 0:
        topk = duplicate_experts(topk, dup_frac, seed)
    return MoeCase(name=("MoE FC1 shared-A/fused-B" if shared_a else "MoE FC1 regular")
                   + f" T={T} top_k={top_k} E={E} H={H} I={I} rank={rank}",
                   seed=seed, T=T, top_k=top_k, E=E, H=H, I=I, rank=rank, L=L, scale=scale,
                   shared_a=shared_a, x=x, topk_ids=topk, lora_ids=lora, A_banks=A, B_banks=B)


def expert_sorted_case(seed: int = 1239, T: int = 2048, top_k: int = 8, E: int = 64,
                       k_in: int = 2048, width: int = 1536, rank: int = 16,
                       p_unadapted: float = 0.1, alpha: float = 32.0, tail_rows: int = 0):
    """Expert-sorted rows of a grouped MoE GEMM ("expert_apply.rs",
    apply_expert_lora_sorted): T tokens each route to top_k distinct experts
    of E (uniform); the T * top_k (token, slot) rows are sorted by expert, so
    expert e owns rows offsets[e] .. offsets[e+1] - 1.  One adapter per expert
    (rank `rank`, padded to itself), a fraction p_unadapted of experts with
    none; x [rows, k_in] (the sorted grouped-GEMM input), out0 [rows, width]
    (its output, w13 = 2I by default).  `tail_rows` extra rows follow the last
    expert's block (no adapter).  Returns (LinearCase with seq_slot = the
    row's expert, or -1 for tail rows, offsets [E + 1] int32)."""
    rng = np.random.default_rng(seed + 20_000)
    topk = np.stack([rng.permutation(E)[:top_k] for _ in range(T)])
    counts = np.bincount(topk.ravel(), minlength=E)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    n = int(offsets[-1]) + tail_rows
    seq = np.full(n, -1, dtype=np.int32)
    seq[: offsets[-1]] = np.repeat(np.arange(E, dtype=np.int32), counts)
    adapted_expert = rng.random(E) >= p_unadapted
    ranks = [rank if adapted_expert[e] else 0 for e in range(E)]
    case = linear_case(seed, n, k_in, (width,), E, rank, ranks, alpha, seq_slot=seq,
                       name=f"expert-sorted fold {n} rows, {E} experts")
    return case, offsets


def moe_y0(seed: int, shape) -> np.ndarray:
    """The expert GEMM's output that an in-place MoE delta updates (w13:
    [T, top_k, 2I]; w2: [T, top_k, H]), N(0, 1) in bf16."""
    return _normal_bf16(np.random.default_rng(seed + 30_000), shape)


@dataclass
class MoeDownCase:
    """Routed-MoE down projection (w2): one activation row per (token, slot),
    x [T * top_k, I]; banks ``A_banks = [A_down]`` [E, L, rank, I] and
    ``B_banks = [B_down]`` [E, L, H, rank]; y0 [T, top_k, H] the down GEMM's
    output; topk_weights [T, top_k] float32 routing weights."""
    name: str
    seed: int
    T: int
    top_k: int
    E: int
    H: int
    I: int
    rank: int
    L: int
    scale: float
    x: np.ndarray
    y0: np.ndarray
    topk_ids: np.ndarray
    lora_ids: np.ndarray
    topk_weights: np.ndarray
    A_banks: list
    B_banks: list


def moe_w2_case(seed: int = 1240, T: int = 2048, top_k: int = 8, E: int = 64, H: int = 2048,
                I: int = 768, rank: int = 16, L: int = 8, scale: float = 2.0,
                p_none: float = 0.2, dup_frac: float = 0.0) -> MoeDownCase:
    """The FC1 workload's routing and shapes seen from the down projection:
    top_k distinct experts of E per token (uniform), lora_ids uniform over L
    with p_none of -1; x ~ N(0, 1) (reading: the activation has no fan-in),
    A ~ N(0,1)/sqrt(I), B ~ N(0,1)/sqrt(rank); routing weights a softmax of
    N(0, 1) logits over the token's top_k (reading: the pages fix no router).
    With ``dup_frac`` > 0, that fraction of the tokens repeat experts
    (``duplicate_experts``)."""
    rng = np.random.default_rng(seed + 40_000)
    topk = np.stack([rng.permutation(E)[:top_k] for _ in range(T)]).astype(np.int32)
    lora = rng.integers(0, L, size=T).astype(np.int32)
    lora[rng.random(T) < p_none] = -1
    logits = rng.standard_normal(size=(T, top_k))
    w = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    x = _normal_bf16(rng, (T * top_k, I))
    A = [_normal_bf16(rng, (E, L, rank, I), 1.0 / np.sqrt(I))]
    B = [_normal_bf16(rng, (E, L, H, rank), 1.0 / np.sqrt(rank))]
    y0 = _normal_bf16(rng, (T, top_k, H))
    if dup_frac > 0:
        topk = duplicate_experts(topk, dup_frac, seed)
    return MoeDownCase(name=f"MoE w2 T={T} top_k={top_k} E={E} H={H} I={I} rank={rank}",
                       seed=seed, T=T, top_k=top_k, E=E, H=H, I=I, rank=rank, L=L,
                       scale=scale, x=x, y0=y0, topk_ids=topk, lora_ids=lora, topk_weights=w,
                       A_banks=A, B_banks=B)
