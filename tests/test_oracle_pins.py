"""Pins of the CPU oracle to facts other than itself (CPU only).

Each test names the page passage or the mathematics that fixes the expected
value.  None of the expected values below comes from the GPU path, and none
comes from the oracle alone: they are library routines (torch dtype
conversion, numpy fp64 matmul), exact rational arithmetic, brute force, closed
forms, or invariants the pages state.
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

from lora_delta_gb300 import inputs
from tests.exact import bf16_ulp_distance, bf16_value, rne_bf16


def f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ bf16 --

def test_bf16_widening_matches_torch_for_every_pattern(oracle):
    """bf16 -> f32 is the exact upper-half embedding (torch's conversion)."""
    L = oracle.lib()
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = np.array([L.oracle_bf16_to_f32(int(p)) for p in pats], dtype=np.float32)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_f32_to_bf16_is_round_to_nearest_even_like_torch(oracle):
    """fp32 -> bf16 rounding agrees with torch's RNE conversion, ties included."""
    rng = np.random.default_rng(7)
    vals = [rng.standard_normal(20000).astype(np.float32),
            (rng.standard_normal(2000) * 1e30).astype(np.float32),
            (rng.standard_normal(2000) * 1e-39).astype(np.float32)]  # fp32 subnormals
    # exact ties: lower 16 bits == 0x8000, with even and odd upper halves
    ups = rng.integers(0, 0x7F7F, size=4000, dtype=np.uint32)
    vals.append(((ups << 16) | 0x8000).view(np.float32))
    vals.append(np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, 3.4028235e38, -3.4028235e38,
                          np.inf, -np.inf, 1.00390625, 1.01171875], dtype=np.float32))
    v = np.concatenate(vals)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f32_to_bf16(v)
    assert np.array_equal(got, ref)
    # textbook cases: 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even (1.0)
    assert int(oracle.f32_to_bf16(np.array([1.0 + 2.0 ** -8]))[0]) == 0x3F80
    # 1 + 3*2^-8 is a tie between 1+2^-7 (odd) and 1+2^-6 (even) -> 1+2^-6
    assert int(oracle.f32_to_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0]) == 0x3F82


def test_f64_to_bf16_single_rounding_matches_exact_rationals(oracle):
    """fp64 -> bf16 is one correctly rounded step (checked with exact Fractions)."""
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-40, 39, 3000),
                        # values a hair off bf16 ties: a single rounding differs from f64->f32->bf16
                        (1.0 + 2.0 ** -8 + 2.0 ** -30) * np.ones(1),
                        (1.0 + 2.0 ** -8 - 2.0 ** -40) * np.ones(1),
                        np.array([1e-45, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135, 3.4e38,
                                  3.3961e38, 0.0])])
    got = oracle.f64_to_bf16(v)
    want = np.array([rne_bf16(Fraction(float(x))) for x in v], dtype=np.uint16)
    assert np.array_equal(got, want)
    assert int(oracle.f64_to_bf16(np.array([1.0 + 2.0 ** -8 + 2.0 ** -30]))[0]) == 0x3F81


# ----------------------------------------------------------------- scale --

@pytest.mark.parametrize("alpha,r", [(16.0, 8), (16.0, 4), (32.0, 16), (32.0, 64), (8.0, 3)])
def test_scale_rule_closed_form(oracle, alpha, r):
    """'Module lora_delta', LoraPair: scale = alpha / r, or alpha / sqrt(r) with rsLoRA."""
    assert oracle.lora_scale(alpha, r, False) == np.float32(alpha / r)
    assert oracle.lora_scale(alpha, r, True) == np.float32(alpha / math.sqrt(r))


# ------------------------------------------------------------------ pack --

def test_pool_pack_layout(oracle):
    """'Module lora_delta', LoraPair: A_r fills the first r rows of [R, k_in], zero rows
    after; B_r fills the first r columns of each row of [w, R], zero columns after."""
    rng = np.random.default_rng(3)
    r, R, k_in, w = 5, 16, 40, 24
    a_r = rng.integers(1, 0x7F00, size=(r, k_in)).astype(np.uint16)
    b_r = rng.integers(1, 0x7F00, size=(w, r)).astype(np.uint16)
    a, b = oracle.pool_pack(a_r, b_r, R)
    assert np.array_equal(a[:r], a_r) and not a[r:].any()
    assert np.array_equal(b[:, :r], b_r) and not b[:, r:].any()


# --------------------------------------------------------------- routing --

def test_segments_brute_force(oracle):
    """'punica_base.py', prefill_metadata: rows clustered by identical lora index;
    -1 applies none.  Reading: a stable sort by slot (Python's sort is stable)."""
    rng = np.random.default_rng(5)
    for n, L in [(0, 3), (1, 1), (37, 4), (500, 16), (1000, 128)]:
        seq = rng.integers(-2, L + 2, size=n).astype(np.int32)
        perm, seg, err = oracle.segments(seq, L)
        keep = [i for i in range(n) if 0 <= seq[i] < L]
        want = sorted(keep, key=lambda i: seq[i])
        assert perm.tolist() == want
        counts = np.bincount(seq[(seq >= 0) & (seq < L)], minlength=L)
        assert seg.tolist() == [0] + np.cumsum(counts).tolist()
        assert err == (1 if (seq >= L).any() else 0)


# ---------------------------------------------------------------- shrink --

def test_shrink_matches_fp64_library_matmul(oracle):
    """'punica_base.py', add_shrink: y[i] += (x @ A_i) * scale, with A in the LoRA
    pair layout [R, k_in] (x @ A^T).  fp64 numpy matmul is the reference; the fp32
    oracle sits within the textbook summation bound gamma_k * sum|x*A|."""
    case = inputs.linear_case(21, n=24, k_in=192, widths=(32, 16), max_loras=3, max_rank=8,
                              ranks=[8, 5, 0], alpha=4.0, p_none=0.2)
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, 3, 8)
    h0 = np.full((2, case.n, 8), 0.25, dtype=np.float32)
    for acc64 in (False, True):
        h, err = oracle.shrink(case.x, case.seq_slot, pool, pool.scale_table, h=h0.copy(),
                               acc64=acc64)
        assert err == 0
        xf = f32(case.x).astype(np.float64)
        for i in range(case.n):
            s = case.seq_slot[i]
            for j in range(2):
                if s < 0 or case.adapters[s] is None:
                    assert np.array_equal(h[j, i], h0[j, i])
                    continue
                ad = case.adapters[s]
                Af = f32(ad.A[j]).astype(np.float64)              # unpadded [r, k_in]
                exact = xf[i] @ Af.T                                # [r]
                sc = float(pool.scale_table[s])
                ref = 0.25 + sc * np.concatenate([exact, np.zeros(8 - ad.rank)])
                bound = case.k_in * 2.0 ** -24 * sc * (np.abs(xf[i]) @ np.abs(Af.T))
                bound = np.concatenate([bound, np.zeros(8 - ad.rank)]) + 2e-7 * np.abs(ref)
                tol = 1e-12 * np.abs(ref) + 1e-7 if acc64 else bound + 1e-7
                assert np.all(np.abs(h[j, i] - ref) <= tol)


# ----------------------------------------------------------------- delta --

def _dense_ref_f64(case, pool_scale, rows=None):
    """out0 + scale_s * (x A_r^T) B_r^T per row and slice in fp64 numpy (unpadded ranks)."""
    ref = f32(case.out0).astype(np.float64).copy()
    xf = f32(case.x).astype(np.float64)
    rows = range(case.n) if rows is None else rows
    for i in rows:
        s = case.seq_slot[i]
        if s < 0 or s >= case.max_loras or case.adapters[s] is None:
            continue
        ad = case.adapters[s]
        off = case.offset_start
        for j, w in enumerate(case.widths):
            if ad.adapted[j]:
                hA = xf[i] @ f32(ad.A[j]).astype(np.float64).T
                d = hA @ f32(ad.B[j]).astype(np.float64).T
                ref[i, off:off + w] += float(pool_scale[s]) * d
            off += w
    return ref


def test_single_adapter_equals_dense_composition(oracle):
    """'Module lora_delta', apply_lora_delta: base_out += scale * (x @ a^T) @ b^T for
    one pair; every row routed to one slot reduces the routed delta to it.  The
    fp64 oracle is the correctly rounded bf16 of the fp64 library result; the fp32
    oracle is within one bf16 step of it."""
    seq = np.zeros(32, dtype=np.int32)
    case = inputs.linear_case(31, n=32, k_in=128, widths=(96,), max_loras=1, max_rank=16,
                              ranks=[11], alpha=16.0, seq_slot=seq)
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, 1, 16)
    ref = _dense_ref_f64(case, pool.scale_table)
    want = np.array([rne_bf16(Fraction(float(v))) for v in ref.ravel()],
                    dtype=np.uint16).reshape(ref.shape)
    o64 = case.out0.copy()
    assert oracle.delta(o64, case.x, case.seq_slot, pool, acc64=True) == 0
    assert np.array_equal(o64, want)
    o32 = case.out0.copy()
    oracle.delta(o32, case.x, case.seq_slot, pool)
    assert bf16_ulp_distance(o32, want).max() <= 1


def test_routed_delta_brute_force_exact_rationals(oracle):
    """'punica_base.py', add_lora_linear semantics / 'Module lora_delta',
    apply_lora_bgmv: per row, per slice, the exact rational
    out + scale_s * sum_r (sum_k x A[r,k]) B[c,r], rounded once to bf16, equals
    the fp64 oracle bit for bit; the fp32 oracle is within one bf16 step."""
    case = inputs.linear_case(41, n=6, k_in=12, widths=(8, 4), max_loras=3, max_rank=4,
                              ranks=[3, 4, 2], alpha=6.0, p_none=0.0, offset_start=8,
                              ld_out=24, seq_slot=np.array([2, 0, -1, 1, 2, 0], np.int32))
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, 3, 4)
    want = case.out0.copy()
    for i in range(case.n):
        s = int(case.seq_slot[i])
        if s < 0:
            continue
        ad = case.adapters[s]
        sc = Fraction(float(pool.scale_table[s]))
        off = case.offset_start
        for j, w in enumerate(case.widths):
            h = [sum(bf16_value(case.x[i, k]) * bf16_value(ad.A[j][q, k])
                     for k in range(case.k_in)) for q in range(ad.rank)]
            for c in range(w):
                d = sum(h[q] * bf16_value(ad.B[j][c, q]) for q in range(ad.rank))
                want[i, off + c] = rne_bf16(bf16_value(case.out0[i, off + c]) + sc * d)
            off += w
    o64 = case.out0.copy()
    oracle.delta(o64, case.x, case.seq_slot, pool, offset_start=case.offset_start, acc64=True)
    assert np.array_equal(o64, want)
    o32 = case.out0.copy()
    oracle.delta(o32, case.x, case.seq_slot, pool, offset_start=case.offset_start)
    assert bf16_ulp_distance(o32, want).max() <= 1
    assert np.array_equal(o32[:, :8], case.out0[:, :8])  # left of offset_start untouched


def test_padding_is_invisible(oracle):
    """'Module lora_delta', invariants: both stages contract at the padded max_rank;
    zero pad rows/columns give the same result as the unpadded adapter, bit for bit."""
    case = inputs.linear_case(51, n=40, k_in=256, widths=(64, 32), max_loras=4, max_rank=8,
                              ranks=[8, 8, 8, 8], alpha=16.0, p_none=0.1)
    padded = oracle.build_pool(case.adapters, case.k_in, case.widths, 4, 32)
    tight = oracle.build_pool(case.adapters, case.k_in, case.widths, 4, 8)
    a, b = case.out0.copy(), case.out0.copy()
    oracle.delta(a, case.x, case.seq_slot, padded)
    oracle.delta(b, case.x, case.seq_slot, tight)
    assert np.array_equal(a, b)


def test_skip_semantics(oracle):
    """'Module lora_delta', apply_lora_bgmv: a negative slot gets no delta;
    LoraRoute: a table entry of 0 means the slot does not adapt that module; a
    scale of 0 adds exact zeros (RN(out + 0) = out for nonzero out)."""
    adapted = [[True, True], [True, False], [False, False]]
    case = inputs.linear_case(61, n=64, k_in=64, widths=(32, 32), max_loras=3, max_rank=8,
                              ranks=[8, 4, 8], alpha=8.0, p_none=0.25, adapted=adapted)
    assert (case.out0 & 0x7FFF).all(), "precondition: no signed zeros in out0"
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, 3, 8)
    o = case.out0.copy()
    oracle.delta(o, case.x, case.seq_slot, pool)
    none = case.seq_slot < 0
    assert none.any() and np.array_equal(o[none], case.out0[none])
    s1 = case.seq_slot == 1
    assert np.array_equal(o[s1, 32:], case.out0[s1, 32:])         # slice 1 not adapted
    assert (o[s1, :32] != case.out0[s1, :32]).mean() > 0.9       # slice 0 adapted
    s2 = case.seq_slot == 2
    assert np.array_equal(o[s2], case.out0[s2])                   # nothing adapted
    zero = np.zeros(3, dtype=np.float32)
    oz = case.out0.copy()
    oracle.delta(oz, case.x, case.seq_slot, pool, scale_table=zero)
    assert np.array_equal(oz, case.out0)


def test_slices_equal_single_slice_calls(oracle):
    """'punica_base.py', add_expand: slice i lands at offset_start + sum of the earlier
    slice widths, so an S-slice call equals S one-slice calls at those offsets."""
    case = inputs.linear_case(71, n=50, k_in=96, widths=(40, 16, 24), max_loras=5,
                              max_rank=8, ranks=[8, 2, 0, 6, 8], alpha=8.0, p_none=0.1,
                              offset_start=8, ld_out=96)
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, 5, 8)
    o = case.out0.copy()
    oracle.delta(o, case.x, case.seq_slot, pool, offset_start=8)
    seq_o = case.out0.copy()
    off = 8
    for j, w in enumerate(case.widths):
        one = [None if ad is None else inputs.Adapter(ad.rank, ad.alpha, [ad.A[j]], [ad.B[j]],
                                                        [ad.adapted[j]])
               for ad in case.adapters]
        pj = oracle.build_pool(one, case.k_in, (w,), 5, 8)
        oracle.delta(seq_o, case.x, case.seq_slot, pj, offset_start=off)
        off += w
    assert np.array_equal(o, seq_o)
    assert np.array_equal(o[:, :8], case.out0[:, :8]) and np.array_equal(o[:, 88:],
                                                                         case.out0[:, 88:])


def test_row_permutation_equivariance(oracle):
    """Rows are independent: permuting (x, out, seq_slot) permutes the result."""
    case = inputs.linear_case(81, n=70, k_in=64, widths=(48,), max_loras=6, max_rank=16,
                              ranks=[16, 8, 4, 16, 2, 1], alpha=16.0, p_none=0.1)
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, 6, 16)
    o = case.out0.copy()
    oracle.delta(o, case.x, case.seq_slot, pool)
    p = np.random.default_rng(0).permutation(case.n)
    op = case.out0[p].copy()
    oracle.delta(op, case.x[p].copy(), case.seq_slot[p].copy(), pool)
    assert np.array_equal(op, o[p])


def test_shrink_then_expand_equals_fused(oracle):
    """'fully_sharded_layers' apply: shrink with scale 1.0 into an fp32 buffer, then
    expand; folding the scale in the expand reproduces the fused delta exactly.
    The 'punica_base.py' form (scale in the shrink) agrees within one bf16 step."""
    case = inputs.linear_case(91, n=33, k_in=160, widths=(64, 32), max_loras=4, max_rank=8,
                              ranks=[8, 4, 8, 3], alpha=8.0, p_none=0.15)
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, 4, 8)
    fused = case.out0.copy()
    oracle.delta(fused, case.x, case.seq_slot, pool)
    h, _ = oracle.shrink(case.x, case.seq_slot, pool, None)
    two = case.out0.copy()
    oracle.expand(two, h, case.seq_slot, pool, pool.scale_table)
    assert np.array_equal(two, fused)
    h2, _ = oracle.shrink(case.x, case.seq_slot, pool, pool.scale_table)
    p1 = case.out0.copy()
    oracle.expand(p1, h2, case.seq_slot, pool, None)
    assert bf16_ulp_distance(p1, fused).max() <= 1


def test_add_inputs_false_overwrites_routed_rows(oracle):
    """'punica_base.py', add_expand add_inputs flag: with add_inputs False the routed
    columns are set to the delta; starting from +0 with add_inputs True gives the
    same bits (RN(+0 + v) = RN(v))."""
    case = inputs.linear_case(101, n=30, k_in=64, widths=(32,), max_loras=2, max_rank=4,
                              ranks=[4, 4], alpha=4.0, p_none=0.3)
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, 2, 4)
    o = case.out0.copy()
    oracle.delta(o, case.x, case.seq_slot, pool, add_inputs=False)
    z = np.zeros_like(case.out0)
    oracle.delta(z, case.x, case.seq_slot, pool, add_inputs=True)
    routed = case.seq_slot >= 0
    assert np.array_equal(o[routed], z[routed])
    assert np.array_equal(o[~routed], case.out0[~routed])


def test_expand_overwrite_from_poisoned_out_equals_add_from_zero(oracle):
    """'punica_base.py', add_expand add_inputs flag, on the two-step form: with
    add_inputs False the expand sets the routed columns to RN(scale * h.B), so a
    poisoned starting out (huge values, infinities, NaN patterns) must give the
    bits that add_inputs True gives from +0 (RN(+0 + v) = RN(v)); rows without a
    slot keep their poison bit for bit, and columns outside the slices too."""
    case = inputs.linear_case(103, n=41, k_in=96, widths=(40, 24), max_loras=3, max_rank=8,
                              ranks=[8, 5, 8], alpha=8.0, p_none=0.25, offset_start=8,
                              ld_out=80)
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, 3, 8)
    h, _ = oracle.shrink(case.x, case.seq_slot, pool, None)
    rng = np.random.default_rng(5)
    poison = rng.choice(np.array([0x7F7F, 0xFF7F, 0x7F80, 0xFF80, 0x7FC0, 0x4480],
                                 dtype=np.uint16), size=case.out0.shape)
    o = poison.copy()
    oracle.expand(o, h, case.seq_slot, pool, pool.scale_table, offset_start=8,
                  add_inputs=False)
    z = np.zeros_like(poison)
    oracle.expand(z, h, case.seq_slot, pool, pool.scale_table, offset_start=8,
                  add_inputs=True)
    routed = case.seq_slot >= 0
    cols = slice(8, 8 + 64)
    assert np.array_equal(o[routed][:, cols], z[routed][:, cols])
    assert np.array_equal(o[~routed], poison[~routed])
    assert np.array_equal(o[:, :8], poison[:, :8]) and np.array_equal(o[:, 72:], poison[:, 72:])
    # and the overwritten values are the correctly rounded fp64 expand within one
    # bf16 step (fp32 accumulation of R = 8 terms)
    B = [f32(b).astype(np.float64) for b in pool.B]
    for i in np.flatnonzero(routed):
        s = case.seq_slot[i]
        ref = np.concatenate([float(pool.scale_table[s]) * (h[j, i].astype(np.float64) @ B[j][s].T)
                              for j in range(2)])
        assert bf16_ulp_distance(o[i, cols], oracle.f64_to_bf16(ref)).max() <= 1


def test_bad_slot_sets_error_and_skips_row(oracle):
    """Reading (no page fixes it): a slot >= max_loras applies no delta and sets
    error bit 1 instead of trapping."""
    seq = np.array([0, 5, -1, 1], dtype=np.int32)
    case = inputs.linear_case(111, n=4, k_in=32, widths=(16,), max_loras=2, max_rank=4,
                              ranks=[4, 4], alpha=4.0, seq_slot=seq)
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, 2, 4)
    o = case.out0.copy()
    assert oracle.delta(o, case.x, case.seq_slot, pool) == 1
    assert np.array_equal(o[1], case.out0[1])


def test_fp32_oracle_within_one_step_of_fp64_on_tiny_workload(oracle):
    case = inputs.tiny_case()
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, 4, 16)
    a, b = case.out0.copy(), case.out0.copy()
    oracle.delta(a, case.x, case.seq_slot, pool)
    oracle.delta(b, case.x, case.seq_slot, pool, acc64=True)
    assert bf16_ulp_distance(a, b).max() <= 1


# ------------------------------------------------------------------- MoE --

def _moe_small(shared, seed=5, **kw):
    args = dict(T=24, top_k=3, E=5, H=48, I=16, rank=4, L=3, scale=2.0, p_none=0.25)
    args.update(kw)
    return inputs.moe_case(shared_a=shared, seed=seed, **args)


def test_moe_matches_fp64_formula_per_pair(oracle):
    """'bgmv_moe_gemm1_lora_delta': delta[t, j] = scale * concat(B_gate[l,e] @ (A_gate[l,e]
    @ x[t]), B_up[l,e] @ (A_up[l,e] @ x[t])), unweighted, per (token, slot), l < 0 skipped
    (written as zeros).  fp64 oracle == correctly rounded fp64 numpy; fp32 within a step."""
    for shared in (False, True):
        c = _moe_small(shared)
        o64, err = oracle.moe_fc1(c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids, c.I,
                                  c.rank, c.scale, shared, c.L, acc64=True)
        assert err == 0
        xf = f32(c.x).astype(np.float64)
        want = np.zeros_like(o64)
        for t in range(c.T):
            l = int(c.lora_ids[t])
            for j in range(c.top_k):
                e = int(c.topk_ids[t, j])
                if l < 0:
                    continue
                if shared:
                    h = f32(c.A_banks[0][e, l]).astype(np.float64) @ xf[t]
                    d = c.scale * (f32(c.B_banks[0][e, l]).astype(np.float64) @ h)
                else:
                    hg = f32(c.A_banks[0][e, l]).astype(np.float64) @ xf[t]
                    hu = f32(c.A_banks[1][e, l]).astype(np.float64) @ xf[t]
                    d = c.scale * np.concatenate(
                        [f32(c.B_banks[0][e, l]).astype(np.float64) @ hg,
                         f32(c.B_banks[1][e, l]).astype(np.float64) @ hu])
                want[t, j] = [rne_bf16(Fraction(float(v))) for v in d]
        assert np.array_equal(o64, want)
        o32, _ = oracle.moe_fc1(c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids, c.I,
                                c.rank, c.scale, shared, c.L)
        assert bf16_ulp_distance(o32, want).max() <= 1


def test_moe_duplicate_experts_follow_the_formula_per_slot(oracle):
    """'bgmv_moe_gemm1_lora_delta', topk_ids: a token may name one expert in two
    or more slots.  Each slot is still its own (token, slot) row of the formula:
    the rows of the repeated expert are equal bit for bit, and each equals the
    correctly rounded fp64 formula (fp64 oracle) and a bf16 step of it (fp32)."""
    for shared in (False, True):
        c = _moe_small(shared, seed=23, dup_frac=0.6)
        dup_rows = [(t, j1, j2) for t in range(c.T) for j1 in range(c.top_k)
                    for j2 in range(j1 + 1, c.top_k)
                    if c.topk_ids[t, j1] == c.topk_ids[t, j2] and c.lora_ids[t] >= 0]
        assert dup_rows
        o64, err = oracle.moe_fc1(c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids, c.I,
                                  c.rank, c.scale, shared, c.L, acc64=True)
        o32, err32 = oracle.moe_fc1(c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids, c.I,
                                    c.rank, c.scale, shared, c.L)
        assert err == err32 == 0
        for t, j1, j2 in dup_rows:
            assert np.array_equal(o32[t, j1], o32[t, j2])
            assert np.array_equal(o64[t, j1], o64[t, j2])
        xf = f32(c.x).astype(np.float64)
        for t, j1, _ in dup_rows:
            e, l = int(c.topk_ids[t, j1]), int(c.lora_ids[t])
            hs = [f32(a[e, l]).astype(np.float64) @ xf[t] for a in c.A_banks]
            if shared:
                d = c.scale * (f32(c.B_banks[0][e, l]).astype(np.float64) @ hs[0])
            else:
                d = c.scale * np.concatenate([f32(c.B_banks[i][e, l]).astype(np.float64) @ hs[i]
                                              for i in range(2)])
            want = np.array([rne_bf16(Fraction(float(v))) for v in d], dtype=np.uint16)
            assert np.array_equal(o64[t, j1], want)
            assert bf16_ulp_distance(o32[t, j1], want).max() <= 1


def test_moe_shared_a_equals_regular_with_equal_a(oracle):
    """'bgmv_moe_gemm1_lora_delta', performant LoRA: one shared A and B fused as
    [2I, rank] (gate rows 0:I, up rows I:2I) is the two-slice form with
    A_gate = A_up; the two modes agree bit for bit."""
    c = _moe_small(False, seed=9)
    A = c.A_banks[0]
    reg, _ = oracle.moe_fc1(c.x, [A, A], c.B_banks, c.topk_ids, c.lora_ids, c.I, c.rank,
                            c.scale, False, c.L)
    fused = np.ascontiguousarray(np.concatenate(c.B_banks, axis=2))  # [E, L, 2I, rank]
    sh, _ = oracle.moe_fc1(c.x, [A], [fused], c.topk_ids, c.lora_ids, c.I, c.rank, c.scale,
                           True, c.L)
    assert np.array_equal(reg, sh)


def test_moe_pairs_are_independent_of_slot_order(oracle):
    """'bgmv_moe_gemm1_lora_delta': the delta is kept per (token, slot), unweighted and
    not summed over experts, so reordering a token's top_k permutes its rows."""
    c = _moe_small(False, seed=13)
    o, _ = oracle.moe_fc1(c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids, c.I, c.rank,
                          c.scale, False, c.L)
    p = np.array([2, 0, 1])
    op, _ = oracle.moe_fc1(c.x, c.A_banks, c.B_banks, c.topk_ids[:, p].copy(), c.lora_ids,
                           c.I, c.rank, c.scale, False, c.L)
    assert np.array_equal(op, o[:, p])


def test_moe_skipped_pairs_are_zero_and_flag_errors(oracle):
    """l < 0 is skipped (zeros, no error); l >= num_loras and e outside [0, E) are
    readings: zeros plus error bits 4 and 2."""
    c = _moe_small(False, seed=17, p_none=0.0)
    topk = c.topk_ids.copy()
    lora = c.lora_ids.copy()
    lora[0] = -1
    lora[1] = c.L            # out of range adapter
    topk[2, 1] = c.E         # out of range expert
    o, err = oracle.moe_fc1(c.x, c.A_banks, c.B_banks, topk, lora, c.I, c.rank, c.scale,
                            False, c.L)
    assert not o[0].any() and not o[1].any() and not o[2, 1].any()
    assert o[2, 0].any() and o[3].any()
    assert err == (4 | 2)


# ----------------------------------------------------- in-place MoE w13 / w2 --

def _pair_delta64(A, B, xrow, scale):
    """scale * B @ (A @ x) in fp64 numpy (A [rank, k], B [w, rank] bf16 bits)."""
    h = f32(A).astype(np.float64) @ f32(xrow).astype(np.float64)
    return scale * (f32(B).astype(np.float64) @ h)


def _rne_row(vals):
    return [rne_bf16(Fraction(float(v))) for v in vals]


def test_moe_w13_in_place_matches_fp64_formula(oracle):
    """'punica_base.py' add_lora_w13: the gate/up delta of 'bgmv_moe_gemm1_lora_delta'
    added to intermediate_cache1 in place, y = RN(y + delta); pairs with no adapter
    keep y bit for bit.  fp64 oracle == correctly rounded fp64 numpy."""
    for shared in (False, True):
        c = _moe_small(shared, seed=21)
        y0 = inputs.moe_y0(21, (c.T, c.top_k, 2 * c.I))
        y, err = oracle.moe_w13(y0, c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids, c.I,
                                c.rank, c.scale, shared, c.L, acc64=True)
        assert err == 0
        want = y0.copy()
        for t in range(c.T):
            l = int(c.lora_ids[t])
            if l < 0:
                continue
            for j in range(c.top_k):
                e = int(c.topk_ids[t, j])
                if shared:
                    d = _pair_delta64(c.A_banks[0][e, l], c.B_banks[0][e, l], c.x[t], c.scale)
                else:
                    d = np.concatenate([
                        _pair_delta64(c.A_banks[0][e, l], c.B_banks[0][e, l], c.x[t], c.scale),
                        _pair_delta64(c.A_banks[1][e, l], c.B_banks[1][e, l], c.x[t], c.scale)])
                want[t, j] = _rne_row(f32(y0[t, j]).astype(np.float64) + d)
        assert np.array_equal(y, want)
        assert np.array_equal(y[c.lora_ids < 0], y0[c.lora_ids < 0])
        y32, _ = oracle.moe_w13(y0, c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids, c.I,
                                c.rank, c.scale, shared, c.L)
        assert bf16_ulp_distance(y32, want).max() <= 1


def test_moe_w13_overwrite_writes_only_adapted_pairs(oracle):
    """add_inputs=False writes RN(delta) on the pairs that have an adapter (the FC1
    values of 'bgmv_moe_gemm1_lora_delta'); the other pairs keep the caller's y."""
    c = _moe_small(False, seed=23)
    poison = np.full((c.T, c.top_k, 2 * c.I), 0x7FC1, dtype=np.uint16)
    y, _ = oracle.moe_w13(poison, c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids, c.I,
                          c.rank, c.scale, False, c.L, add_inputs=False, acc64=True)
    fc1, _ = oracle.moe_fc1(c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids, c.I, c.rank,
                            c.scale, False, c.L, acc64=True)
    ad = c.lora_ids >= 0
    assert np.array_equal(y[ad], fc1[ad])
    assert (y[~ad] == 0x7FC1).all()


def test_moe_expert_map_selects_local_experts(oracle):
    """'punica_base.py' add_lora_w13 expert_map: global expert ids map to this rank's
    local ids, -1 = not local.  Eight global experts, four local (global 1, 3, 6, 7 in
    a shuffled local order): pairs on a local expert get that expert's adapter, the
    others keep y; an id past the map or a map entry >= E flags bit 2."""
    c = _moe_small(False, seed=25, E=8, p_none=0.0)
    local_of = {1: 2, 3: 0, 6: 3, 7: 1}
    emap = np.full(8, -1, dtype=np.int32)
    for g, loc in local_of.items():
        emap[g] = loc
    inv = {loc: g for g, loc in local_of.items()}
    banks_a = [np.ascontiguousarray(b[[inv[i] for i in range(4)]]) for b in c.A_banks]
    banks_b = [np.ascontiguousarray(b[[inv[i] for i in range(4)]]) for b in c.B_banks]
    y0 = inputs.moe_y0(25, (c.T, c.top_k, 2 * c.I))
    y, err = oracle.moe_w13(y0, c.x, banks_a, banks_b, c.topk_ids, c.lora_ids, c.I, c.rank,
                            c.scale, False, c.L, expert_map=emap, acc64=True)
    assert err == 0
    want = y0.copy()
    for t in range(c.T):
        l = int(c.lora_ids[t])
        for j in range(c.top_k):
            g = int(c.topk_ids[t, j])
            if g not in local_of:
                continue
            d = np.concatenate([
                _pair_delta64(c.A_banks[0][g, l], c.B_banks[0][g, l], c.x[t], c.scale),
                _pair_delta64(c.A_banks[1][g, l], c.B_banks[1][g, l], c.x[t], c.scale)])
            want[t, j] = _rne_row(f32(y0[t, j]).astype(np.float64) + d)
    assert np.array_equal(y, want)
    assert any(int(g) not in local_of for g in c.topk_ids.ravel())
    bad_map = emap.copy()
    bad_map[3] = 4  # local id past E
    topk = c.topk_ids.copy()
    topk[0, 0] = 8  # global id past the map
    yb, err = oracle.moe_w13(y0, c.x, banks_a, banks_b, topk, c.lora_ids, c.I, c.rank,
                             c.scale, False, c.L, expert_map=bad_map)
    assert err == 2
    assert np.array_equal(yb[0, 0], y0[0, 0])


def test_moe_adapter_enabled_switches_adapters_off(oracle):
    """adapter_enabled: an adapter marked 0 adds nothing (its pairs keep y bit for
    bit); all ones is the same as no table."""
    c = _moe_small(False, seed=27)
    y0 = inputs.moe_y0(27, (c.T, c.top_k, 2 * c.I))
    args = (c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids, c.I, c.rank, c.scale, False, c.L)
    base, _ = oracle.moe_w13(y0, *args)
    ones, _ = oracle.moe_w13(y0, *args, adapter_enabled=np.ones(c.L, np.int32))
    assert np.array_equal(base, ones)
    en = np.ones(c.L, np.int32)
    en[1] = 0
    part, _ = oracle.moe_w13(y0, *args, adapter_enabled=en)
    off = c.lora_ids == 1
    assert off.any()
    assert np.array_equal(part[off], y0[off])
    assert np.array_equal(part[~off], base[~off])


def _w2_small(seed=31, **kw):
    args = dict(T=20, top_k=3, E=5, H=40, I=24, rank=4, L=3, scale=2.0, p_none=0.25)
    args.update(kw)
    return inputs.moe_w2_case(seed=seed, **args)


def test_moe_w2_matches_fp64_formula_per_pair_row(oracle):
    """'punica_base.py' add_lora_w2: intermediate_cache3 [T, top_k, H] gets, in place,
    w[t, j] * scale * B_down[l,e] @ (A_down[l,e] @ x[t*top_k + j]), x being the
    activation row of that (token, slot); fp64 oracle == correctly rounded numpy,
    with and without routing weights."""
    c = _w2_small()
    for weights in (None, c.topk_weights):
        y, err = oracle.moe_w2(c.y0, c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids, c.rank,
                               c.scale, c.L, topk_weights=weights, acc64=True)
        assert err == 0
        want = c.y0.copy()
        for t in range(c.T):
            l = int(c.lora_ids[t])
            if l < 0:
                continue
            for j in range(c.top_k):
                e = int(c.topk_ids[t, j])
                d = _pair_delta64(c.A_banks[0][e, l], c.B_banks[0][e, l], c.x[t * c.top_k + j],
                                  c.scale)
                if weights is not None:
                    d = float(weights[t, j]) * d
                want[t, j] = _rne_row(f32(c.y0[t, j]).astype(np.float64) + d)
        assert np.array_equal(y, want)
        y32, _ = oracle.moe_w2(c.y0, c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids, c.rank,
                               c.scale, c.L, topk_weights=weights)
        assert bf16_ulp_distance(y32, want).max() <= 1


def test_moe_w2_weight_two_is_double_scale(oracle):
    """Multiplying by two is exact in binary floating point, so a routing weight of 2
    on every pair gives bit for bit the result of twice the scale and no weights."""
    c = _w2_small(seed=33)
    w2x = np.full((c.T, c.top_k), 2.0, np.float32)
    a, _ = oracle.moe_w2(c.y0, c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids, c.rank,
                         c.scale, c.L, topk_weights=w2x)
    b, _ = oracle.moe_w2(c.y0, c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids, c.rank,
                         2 * c.scale, c.L)
    assert np.array_equal(a, b)
    plain, _ = oracle.moe_w2(c.y0, c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids, c.rank,
                             c.scale, c.L)
    assert not np.array_equal(a, plain)


# ------------------------------------------- tensor-parallel sharded forms --

def test_gather_rank_blocks_is_numpy_concatenation_along_the_rank(oracle):
    """'vllm.lora.fully_sharded_layers', _mcp_apply: the all-gather of the h shards
    along the last dimension is numpy's concatenation of the rank blocks."""
    rng = np.random.default_rng(3)
    for tp, S, n, Rs in [(1, 2, 5, 8), (2, 3, 7, 8), (4, 1, 9, 4)]:
        shards = rng.standard_normal((tp, S, n, Rs)).astype(np.float32)
        want = np.concatenate(list(shards), axis=2)
        assert np.array_equal(oracle.gather_rank_blocks(shards), want)


def test_rank_sum_is_the_rank_order_fp32_sum(oracle):
    """RowParallelLinearWithShardedLoRA apply: the all-reduce of the h partials.
    Integer-valued partials sum exactly; random partials stay within tp - 1 fp32
    roundings of the exact sum; one rank is the identity."""
    rng = np.random.default_rng(4)
    ints = rng.integers(-1000, 1000, size=(4, 6, 5)).astype(np.float32)
    assert np.array_equal(oracle.rank_sum(ints), ints.astype(np.int64).sum(0).astype(np.float32))
    for tp in (2, 3, 4):
        parts = rng.standard_normal((tp, 3, 7, 16)).astype(np.float32)
        exact = parts.astype(np.float64).sum(0)
        bound = (tp - 1) * 2.0 ** -24 * np.abs(parts.astype(np.float64)).sum(0) + 1e-30
        assert np.all(np.abs(oracle.rank_sum(parts) - exact) <= bound)
    one = rng.standard_normal((1, 4, 4)).astype(np.float32)
    assert np.array_equal(oracle.rank_sum(one), one[0])


def _tp_case():
    return inputs.linear_case(131, n=37, k_in=96, widths=(64, 32), max_loras=3, max_rank=16,
                              ranks=[16, 8, 12], alpha=16.0, p_none=0.2)


def _rank_columns(case, tp, p, offset_start=0):
    """Columns of out that rank p's shard of the expand covers (per slice j:
    off_j + p * w_j / tp ...)."""
    cols, off = [], offset_start
    for w in case.widths:
        ws = w // tp
        cols.extend(range(off + p * ws, off + (p + 1) * ws))
        off += w
    return np.array(cols)


@pytest.mark.parametrize("tp", [2, 4])
def test_column_sharded_form_equals_the_unsharded_delta_bit_for_bit(oracle, tp):
    """'vllm.lora.fully_sharded_layers', _mcp_apply (ColumnParallelLinearWithShardedLoRA,
    MergedColumnParallelLinearWithShardedLoRA): A sliced along the rank, each rank's
    shrink (scale 1) into an fp32 buffer, all-gather, then each rank expands with the
    B rows of its output columns.  Every rank then holds the unsharded h exactly, so
    its output columns equal the unsharded delta's bit for bit (over two slices)."""
    case = _tp_case()
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, 3, 16)
    full = case.out0.copy()
    oracle.delta(full, case.x, case.seq_slot, pool)
    shards = np.stack([oracle.shrink(case.x, case.seq_slot,
                                     oracle.shard_pool_a_rows(pool, tp, p), None)[0]
                       for p in range(tp)])
    h = oracle.gather_rank_blocks(shards)
    for p in range(tp):
        cols = _rank_columns(case, tp, p)
        out_p = np.ascontiguousarray(case.out0[:, cols])
        oracle.expand(out_p, h, case.seq_slot, oracle.shard_pool_b_rows(pool, tp, p),
                      pool.scale_table)
        assert np.array_equal(out_p, full[:, cols])


@pytest.mark.parametrize("tp", [1, 2, 4])
def test_row_sharded_form_matches_the_dense_composition(oracle, tp):
    """RowParallelLinearWithShardedLoRA apply: x and A sliced along the input; each
    rank's shrink gives a partial h over its k columns; the all-reduce sums them;
    rank p expands with its B rows into its slice of the (partial-sum) output at
    offset_start = p * shard.  Within the slice the result is RN(out + scale * h.B)
    with h the reduced sum: within the parity tolerance of the fp64 dense
    composition (one rank: the unsharded delta bit for bit); outside the slice
    nothing changes; over all ranks every column gets its delta from one rank."""
    case = inputs.linear_case(133, n=29, k_in=128, widths=(64,), max_loras=3, max_rank=16,
                              ranks=[16, 4, 12], alpha=16.0, p_none=0.2)
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, 3, 16)
    ks = case.k_in // tp
    parts = np.stack([oracle.shrink(np.ascontiguousarray(case.x[:, p * ks:(p + 1) * ks]),
                                    case.seq_slot, oracle.shard_pool_a_cols(pool, tp, p),
                                    None)[0] for p in range(tp)])
    h = oracle.rank_sum(parts)
    xf = f32(case.x).astype(np.float64)
    A = f32(pool.A[0]).astype(np.float64)
    B = f32(pool.B[0]).astype(np.float64)
    full = case.out0.copy()
    oracle.delta(full, case.x, case.seq_slot, pool)
    ws = case.widths[0] // tp
    covered = np.zeros(case.out0.shape, dtype=bool)
    for p in range(tp):
        out_p = case.out0.copy()
        oracle.expand(out_p, h, case.seq_slot, oracle.shard_pool_b_rows(pool, tp, p),
                      pool.scale_table, offset_start=p * ws)
        inside = np.zeros(case.ld_out, dtype=bool)
        inside[p * ws:(p + 1) * ws] = True
        assert np.array_equal(out_p[:, ~inside], case.out0[:, ~inside])
        routed = case.seq_slot >= 0
        assert np.array_equal(out_p[~routed], case.out0[~routed])
        covered[:, inside] = True
        for i in np.flatnonzero(routed):
            s = case.seq_slot[i]
            ref = f32(case.out0[i, inside]).astype(np.float64) + float(pool.scale_table[s]) * (
                (A[s] @ xf[i]) @ B[s][p * ws:(p + 1) * ws].T)
            got = f32(out_p[i, inside]).astype(np.float64)
            assert np.all(np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref))
        if tp == 1:
            assert np.array_equal(out_p, full)
    assert covered.all()
