"""GPU parity: every entry point of the C ABI against the CPU oracle on the same
seeded inputs (marked gpu).

Bar: bf16 outputs within max|err| <= 1e-2 + 1e-2*|ref|; rows that get no delta,
routing (perm / segment starts) and packing bit-exact.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from lora_delta_gb300 import inputs
from tests.gpu_util import assert_close, oracle_delta

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ld():
    import __graft_entry__
    __graft_entry__.build()
    import lora_delta_gb300
    assert torch.cuda.is_available()
    return lora_delta_gb300


@pytest.fixture(scope="module")
def di(ld):
    from lora_delta_gb300 import device_inputs
    return device_inputs


def run_fused(ld, di, case, R=None, add_inputs=True, scale_table=None):
    d = di.linear_to_device(case, R=R)
    out = d.out0.clone()
    err = ld.new_error_word()
    ld.lora_delta_fused(out, d.x, d.seq_slot, d.pool, offset_start=case.offset_start,
                        add_inputs=add_inputs, scale_table=scale_table, err=err)
    e = ld.lora_get_error(err)
    return di.bits(out), e, d


def check_linear(oracle, case, got, err, rows=None, R=None, add_inputs=True):
    ref, ref_err = oracle_delta(oracle, case, rows=rows, R=R, add_inputs=add_inputs)
    sub = got if rows is None else got[np.asarray(rows)]
    out0 = case.out0 if rows is None else case.out0[np.asarray(rows)]
    seq = case.seq_slot if rows is None else case.seq_slot[np.asarray(rows)]
    assert_close(sub, ref, case.name)
    none = (seq < 0) | (seq >= case.max_loras)
    assert np.array_equal(sub[none], out0[none]), "rows without a delta must be untouched"
    assert err == ref_err


# ------------------------------------------------------------------ pack --

def test_pool_pack_bit_exact(ld, di, oracle):
    rng = np.random.default_rng(0)
    for r, R, k_in, w in [(5, 16, 40, 24), (16, 16, 256, 64), (1, 64, 8, 8), (0, 8, 16, 16)]:
        a_r = inputs.to_bf16_bits(rng.standard_normal((r, k_in), dtype=np.float32))
        b_r = inputs.to_bf16_bits(rng.standard_normal((w, r), dtype=np.float32))
        a_slot = torch.full((R, k_in), 7.0, dtype=torch.bfloat16, device="cuda")
        b_slot = torch.full((w, R), 7.0, dtype=torch.bfloat16, device="cuda")
        ld.lora_pool_pack(a_slot, b_slot, di.bf16(a_r.reshape(r, k_in)),
                          di.bf16(b_r.reshape(w, r)))
        a_ref, b_ref = oracle.pool_pack(a_r.reshape(r, k_in), b_r.reshape(w, r), R)
        assert np.array_equal(di.bits(a_slot), a_ref)
        assert np.array_equal(di.bits(b_slot), b_ref)


# --------------------------------------------------------------- routing --

@pytest.mark.parametrize("n,L", [(0, 3), (1, 1), (37, 4), (1000, 16), (8192, 8), (20000, 128),
                                 (5000, 3071)])
def test_route_bit_exact(ld, oracle, n, L):
    rng = np.random.default_rng(n + L)
    seq = rng.integers(-2, L + 2, size=n).astype(np.int32)
    err = ld.new_error_word()
    perm, seg = ld.lora_route(torch.from_numpy(seq).cuda(), L, err=err)
    e = ld.lora_get_error(err)
    ref_perm, ref_seg, ref_err = oracle.segments(seq, L)
    seg = seg.cpu().numpy()
    assert np.array_equal(seg[: L + 1], ref_seg)
    assert seg[L + 1] == n
    assert np.array_equal(perm.cpu().numpy()[: ref_seg[-1]], ref_perm)
    rest = np.sort(perm.cpu().numpy()[ref_seg[-1]:n])
    assert np.array_equal(rest, np.flatnonzero((seq < 0) | (seq >= L)))
    assert e == ref_err


@pytest.mark.parametrize("n,L", [(2048, 8), (5003, 8), (20000, 8), (16384, 512), (9000, 3071),
                                 (100, 8)])
def test_chunked_route_bit_exact(ld, oracle, n, L):
    """The many-CTA routing sort gives the one-CTA sort's output bit for bit
    (the same stable order) and the oracle's segments: the one-launch cluster
    sort (2 to 16 chunks of 1024 items, the last one ragged at 5003) and the
    two-kernel sort (20000 items: 20 chunks; 3072 keys: more than the cluster
    sort's shared memory holds)."""
    rng = np.random.default_rng(7 * n + L)
    seq = rng.integers(-2, L + 2, size=n).astype(np.int32)
    seq_d = torch.from_numpy(seq).cuda()
    err = ld.new_error_word()
    perm, seg = ld.lora_route_with_scratch(seq_d, L, err=err)
    e = ld.lora_get_error(err)
    perm1, seg1 = ld.lora_route(seq_d, L)
    ref_perm, ref_seg, ref_err = oracle.segments(seq, L)
    seg = seg.cpu().numpy()
    assert np.array_equal(seg, seg1.cpu().numpy())
    assert np.array_equal(seg[: L + 1], ref_seg)
    assert seg[L + 1] == n
    p = perm.cpu().numpy()
    assert np.array_equal(p[: ref_seg[-1]], ref_perm)
    assert np.array_equal(p[:n], perm1.cpu().numpy()[:n])
    assert e == ref_err


def test_chunked_route_rejects_missing_scratch(ld):
    seq = torch.zeros(5000, dtype=torch.int32, device="cuda")
    perm = torch.empty(5000, dtype=torch.int32, device="cuda")
    seg = torch.empty(10, dtype=torch.int32, device="cuda")
    rc = ld.lib().lora_route_with_scratch(perm.data_ptr(), seg.data_ptr(), seq.data_ptr(), 5000,
                                          8, None, 0, None, None)
    assert rc == 5  # LORA_ERR_WORKSPACE


# ------------------------------------------------------- the fused delta --

def test_tiny_workload(ld, di, oracle):
    case = inputs.tiny_case()
    got, err, _ = run_fused(ld, di, case)
    check_linear(oracle, case, got, err)


def test_decode_qkv_workload(ld, di, oracle):
    case = inputs.decode_qkv_case()
    got, err, _ = run_fused(ld, di, case)
    check_linear(oracle, case, got, err)


@pytest.mark.parametrize("proj", [0, 1])
def test_skewed_workload(ld, di, oracle, proj):
    case = inputs.skewed_case(proj)
    got, err, _ = run_fused(ld, di, case)
    check_linear(oracle, case, got, err)


def test_prefill_workload_all_rows(ld, di, oracle):
    """Full prefill gate_up size (8192 rows, 28672 columns), the launch the
    benchmark times, compared with the oracle on every row and column."""
    case = inputs.prefill_gate_up_case()
    got, err, _ = run_fused(ld, di, case)
    check_linear(oracle, case, got, err)


def test_prefill_shaped_small(ld, di, oracle):
    """Routed path (n > 1024) at a size the oracle finishes whole: ragged
    segments, several row passes per slot, unsorted rows."""
    case = inputs.prefill_gate_up_case(seed=77, n_tokens=3000, n_segments=12, seg_lo=16,
                                       seg_hi=700, k_in=512, widths=(1024, 776))
    got, err, _ = run_fused(ld, di, case)
    check_linear(oracle, case, got, err)


def test_x_scaled_reading(ld, di, oracle):
    case = inputs.decode_qkv_case(x_scaled=True)
    got, err, _ = run_fused(ld, di, case)
    check_linear(oracle, case, got, err)


def test_out_zero_start(ld, di, oracle):
    case = inputs.decode_qkv_case(out0="zero")
    got, err, _ = run_fused(ld, di, case)
    check_linear(oracle, case, got, err)


# ------------------------------------------------------------ edge cases --

def test_all_rows_unrouted_is_a_bitwise_no_op(ld, di, oracle):
    case = inputs.linear_case(5, n=50, k_in=64, widths=(32,), max_loras=3, max_rank=16,
                              ranks=[16, 8, 4], alpha=16.0,
                              seq_slot=np.full(50, -1, np.int32))
    got, err, _ = run_fused(ld, di, case)
    assert np.array_equal(got, case.out0) and err == 0


def test_single_slot_many_rows_and_rank8(ld, di, oracle):
    seq = np.zeros(900, dtype=np.int32)
    case = inputs.linear_case(6, n=900, k_in=256, widths=(128, 64), max_loras=1, max_rank=8,
                              ranks=[8], alpha=8.0, seq_slot=seq)
    got, err, _ = run_fused(ld, di, case)
    check_linear(oracle, case, got, err)


def test_single_row_and_true_rank_one(ld, di, oracle):
    """One row (on a rank-1 adapter padded to 16), and a batch over adapters of true
    ranks 1, 2, 5 and 16 with rsLoRA scales."""
    case = inputs.linear_case(7, n=1, k_in=264, widths=(136,), max_loras=2, max_rank=16,
                              ranks=[1, 16], alpha=4.0, seq_slot=np.array([0], np.int32))
    got, err, _ = run_fused(ld, di, case)
    check_linear(oracle, case, got, err)
    case = inputs.linear_case(8, n=37, k_in=264, widths=(136, 40), max_loras=4, max_rank=16,
                              ranks=[1, 2, 5, 16], alpha=4.0, p_none=0.1, use_rslora=True)
    got, err, _ = run_fused(ld, di, case)
    check_linear(oracle, case, got, err)


def test_table_zero_scale_zero_and_offsets(ld, di, oracle):
    adapted = [[True, False, True], [False, False, False], [True, True, True],
               [False, True, False]]
    case = inputs.linear_case(7, n=77, k_in=320, widths=(64, 40, 24), max_loras=4,
                              max_rank=16, ranks=[16, 8, 4, 12], alpha=16.0, p_none=0.2,
                              adapted=adapted, offset_start=16, ld_out=160)
    got, err, _ = run_fused(ld, di, case)
    check_linear(oracle, case, got, err)
    zero = torch.zeros(4, dtype=torch.float32, device="cuda")
    got0, _, _ = run_fused(ld, di, case, scale_table=zero)
    assert np.array_equal(got0, case.out0)


def test_add_inputs_false(ld, di, oracle):
    case = inputs.linear_case(8, n=40, k_in=128, widths=(48, 16), max_loras=3, max_rank=16,
                              ranks=[16, 16, 8], alpha=16.0, p_none=0.3)
    got, err, _ = run_fused(ld, di, case, add_inputs=False)
    check_linear(oracle, case, got, err, add_inputs=False)


def _stream_case(which):
    rng = np.random.default_rng(91 + which)
    if which == 0:  # two slices, one stage per CTA, keys of 1 to 40 rows
        seq = np.concatenate([np.zeros(40), np.ones(17), np.full(5, 2), [3], np.full(6, -1)])
        rng.shuffle(seq)
        return inputs.linear_case(91, n=len(seq), k_in=1024, widths=(6144, 2056), max_loras=4,
                                  max_rank=64, ranks=[64, 32, 48, 8], alpha=32.0,
                                  seq_slot=seq.astype(np.int32),
                                  adapted=[[True, True], [True, False], [False, True],
                                           [True, True]])
    # 56 keys (clusters of 8), so each CTA's k share takes two stages; one key of
    # 40 rows, the others 1 to 3
    seq = np.concatenate([np.zeros(40)] + [np.full(1 + s % 3, s) for s in range(1, 56)])
    rng.shuffle(seq)
    return inputs.linear_case(92, n=len(seq), k_in=3072, widths=(4096,), max_loras=56,
                              max_rank=64, ranks=rng.choice([8, 16, 32, 64], 56).tolist(),
                              alpha=32.0, seq_slot=seq.astype(np.int32))


@pytest.mark.parametrize("which", [0, 1])
@pytest.mark.parametrize("add_inputs", [True, False])
def test_rank_64_wide_outputs_stream_b_rows_in_chunks(ld, di, oracle, which, add_inputs):
    """Rank 64 where a CTA's B rows exceed the staged slab: the expand streams B rows
    and out segments in chunks through the shrink's stage buffers; keys span several
    16-row passes (the A rows are copied again each pass)."""
    case = _stream_case(which)
    got, err, _ = run_fused(ld, di, case, add_inputs=add_inputs)
    check_linear(oracle, case, got, err, add_inputs=add_inputs)


@pytest.mark.parametrize("R,add_inputs", [(32, True), (32, False), (16, True), (64, True)])
def test_small_slots_with_large_adapters(ld, di, oracle, R, add_inputs):
    """Adapters of at least 512 KiB (the tensor-core threshold drops to 16 rows):
    slots with 1 to 15 rows go to the small-segment kernel on the second stream,
    slots with 16 or more to the tensor-core path.  Two ragged slices, ranks
    under R, slots with an inactive slice, 40 slots."""
    rng = np.random.default_rng(101 + R)
    k_in = 524288 // (2 * 2 * R) + 8 * (R // 16)  # S * R * k_in * 2 just over 512 KiB
    counts = rng.choice([1, 2, 3, 5, 9, 15, 16, 23], size=40)
    seq = np.concatenate([np.full(c, s) for s, c in enumerate(counts)] + [np.full(7, -1)])
    rng.shuffle(seq)
    adapted = [[bool(rng.random() > 0.15), bool(rng.random() > 0.15)] for _ in range(40)]
    ranks = rng.choice([R // 2, R], size=40).tolist()
    case = inputs.linear_case(102 + R, n=len(seq), k_in=k_in, widths=(2048, 1032), max_loras=40,
                              max_rank=R, ranks=ranks, alpha=float(R), seq_slot=seq.astype(np.int32),
                              adapted=adapted)
    got, err, _ = run_fused(ld, di, case, add_inputs=add_inputs)
    check_linear(oracle, case, got, err, add_inputs=add_inputs)


def test_bad_slot_sets_error_and_skips(ld, di, oracle):
    seq = np.array([0, 9, -1, 1, 2, 7, 0, 1], dtype=np.int32)
    case = inputs.linear_case(9, n=8, k_in=64, widths=(32,), max_loras=3, max_rank=8,
                              ranks=[8, 8, 8], alpha=8.0, seq_slot=seq)
    got, err, _ = run_fused(ld, di, case)
    assert err & 1
    check_linear(oracle, case, got, err)


def test_bad_slot_is_flagged_when_slot_0_adapts_nothing(ld, di, oracle):
    """The out-of-range check does not depend on slot 0 having an adapter."""
    seq = np.array([1, 5, -1, 1, 2, 2, 1, 2], dtype=np.int32)
    case = inputs.linear_case(19, n=8, k_in=64, widths=(32,), max_loras=3, max_rank=8,
                              ranks=[8, 8, 8], alpha=8.0, seq_slot=seq,
                              adapted=[[False], [True], [True]])
    got, err, _ = run_fused(ld, di, case)
    assert err & 1
    check_linear(oracle, case, got, err)


def test_misaligned_table_entry_is_skipped_and_flagged(ld, di, oracle):
    case = inputs.linear_case(10, n=16, k_in=64, widths=(32,), max_loras=2, max_rank=8,
                              ranks=[8, 8], alpha=8.0, seq_slot=np.array([0, 1] * 8, np.int32))
    d = di.linear_to_device(case)
    d.pool.a_table[1] += 2  # slot 1: not 16-byte aligned
    out = d.out0.clone()
    err = ld.new_error_word()
    ld.lora_delta_fused(out, d.x, d.seq_slot, d.pool, err=err)
    assert ld.lora_get_error(err) & 16
    got = di.bits(out)
    assert np.array_equal(got[1::2], case.out0[1::2])
    ref, _ = oracle_delta(oracle, case)
    assert_close(got[0::2], ref[0::2], "slot 0 still applies")


def test_deterministic(ld, di):
    case = inputs.skewed_case(0)
    a, _, _ = run_fused(ld, di, case)
    b, _, _ = run_fused(ld, di, case)
    assert np.array_equal(a, b)


def test_empty_batch_is_a_no_op(ld, di):
    case = inputs.tiny_case()
    d = di.linear_to_device(case)
    out = d.out0[:0]
    ld.lora_delta_fused(out, d.x[:0], d.seq_slot[:0], d.pool)
    torch.cuda.synchronize()


# ------------------------------------------------- shrink / expand alone --

def test_shrink_matches_oracle(ld, di, oracle):
    case = inputs.linear_case(11, n=1500, k_in=1024, widths=(64, 32), max_loras=5,
                              max_rank=16, ranks=[16, 8, 0, 16, 4], alpha=16.0, p_none=0.1)
    d = di.linear_to_device(case)
    h = torch.full((2, case.n, 16), 0.5, dtype=torch.float32, device="cuda")
    err = ld.new_error_word()
    ld.lora_shrink(h, d.x, d.seq_slot, d.pool, scale_table=d.pool.scale_table, err=err)
    assert ld.lora_get_error(err) == 0
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, 5, 16)
    href, _ = oracle.shrink(case.x, case.seq_slot, pool, pool.scale_table,
                            h=np.full((2, case.n, 16), 0.5, np.float32), acc64=True)
    got = h.cpu().numpy()
    xf = (case.x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    # rigorous fp32 summation bound: k_in * 2^-24 * scale * sum |x||A| (+ the add)
    for j in range(2):
        Aabs = np.abs((pool.A[j].astype(np.uint32) << 16).view(np.float32).astype(np.float64))
        for i in range(case.n):
            s = case.seq_slot[i]
            if s < 0 or case.adapters[s] is None:
                assert np.array_equal(got[j, i], np.full(16, 0.5, np.float32))
                continue
            sc = float(pool.scale_table[s])
            bound = 2 * case.k_in * 2.0 ** -24 * sc * (np.abs(xf[i]) @ Aabs[s].T) + 1e-6
            assert np.all(np.abs(got[j, i] - href[j, i]) <= bound)


def test_expand_matches_oracle_and_composes(ld, di, oracle):
    case = inputs.linear_case(12, n=1300, k_in=256, widths=(96, 32), max_loras=4, max_rank=16,
                              ranks=[16, 8, 16, 4], alpha=16.0, p_none=0.15, offset_start=8,
                              ld_out=144)
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, 4, 16)
    h, _ = oracle.shrink(case.x, case.seq_slot, pool, None)
    ref = case.out0.copy()
    oracle.expand(ref, h, case.seq_slot, pool, pool.scale_table, offset_start=8)
    d = di.linear_to_device(case)
    out = d.out0.clone()
    ld.lora_expand(out, torch.from_numpy(h).cuda(), d.seq_slot, d.pool,
                   scale_table=d.pool.scale_table, offset_start=8)
    got = di.bits(out)
    assert_close(got, ref, "expand")
    # GPU shrink (scale 1) then GPU expand (scale folded) == the fused delta
    hg = torch.zeros(2, case.n, 16, dtype=torch.float32, device="cuda")
    ld.lora_shrink(hg, d.x, d.seq_slot, d.pool)
    two = d.out0.clone()
    ld.lora_expand(two, hg, d.seq_slot, d.pool, scale_table=d.pool.scale_table, offset_start=8)
    fused = d.out0.clone()
    ld.lora_delta_fused(fused, d.x, d.seq_slot, d.pool, offset_start=8)
    assert_close(di.bits(two), di.bits(fused), "shrink+expand vs fused")


# ------------------------------------------- logits and embedding variants --

@pytest.mark.parametrize("n", [48, 1500])
def test_logits_variant_at_vocabulary_width(ld, di, oracle, n):
    """"punica_base.py", add_lora_logits: buffer = (x A^T) * scale, y += buffer
    B^T, with the LM head's vocabulary-wide output as one slice of 32064
    columns (its last 128-column chunk is ragged: 64 columns).  48 rows stay
    on the small-segment path; 1500 rows over 5 slots (~270 each) take the
    tensor-core path.  The scale may sit in the shrink (the page's form) or
    in the fold: the two-step form with the scale in lora_shrink matches."""
    case = inputs.linear_case(31, n=n, k_in=1024, widths=(32064,), max_loras=5, max_rank=16,
                              ranks=[16, 8, 16, 16, 4], alpha=16.0, p_none=0.1, name="logits")
    got, err, d = run_fused(ld, di, case)
    rows = None if n < 100 else np.sort(np.random.default_rng(3).choice(n, 128, replace=False))
    check_linear(oracle, case, got, err, rows=rows)
    if n < 100:
        hg = torch.zeros(1, n, 16, dtype=torch.float32, device="cuda")
        ld.lora_shrink(hg, d.x, d.seq_slot, d.pool, scale_table=d.pool.scale_table)
        two = d.out0.clone()
        ld.lora_expand(two, hg, d.seq_slot, d.pool, scale_table=None)
        assert_close(di.bits(two), got, "logits, scale in the shrink")


def test_embedding_variant_expands_looked_up_rows(ld, di, oracle):
    """"punica_base.py", add_lora_embedding: y += x B^T, expand only, where x is
    the rank-space row an embedding lookup gives each token:
    x[i] = A_emb[slot_i][token_i] (taken here as an fp32 table)."""
    rng = np.random.default_rng(41)
    n, vocab, R, L, hidden = 700, 3000, 16, 4, 2048
    seq = rng.integers(-1, L, size=n).astype(np.int32)
    tokens = rng.integers(0, vocab, size=n)
    a_emb = (rng.standard_normal((L, vocab, R)) / 4).astype(np.float32)
    h = np.zeros((1, n, R), dtype=np.float32)
    ok = seq >= 0
    h[0, ok] = a_emb[seq[ok], tokens[ok]]
    case = inputs.linear_case(42, n=n, k_in=64, widths=(hidden,), max_loras=L, max_rank=R,
                              ranks=[16] * L, alpha=16.0, seq_slot=seq, name="embedding")
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, L, R)
    ref = case.out0.copy()
    oracle.expand(ref, h, seq, pool, None)  # no scale: y += x B^T
    d = di.linear_to_device(case)
    out = d.out0.clone()
    ld.lora_expand(out, torch.from_numpy(h).cuda(), d.seq_slot, d.pool, scale_table=None)
    got = di.bits(out)
    assert_close(got, ref, "embedding")
    assert np.array_equal(got[~ok], case.out0[~ok])


# ------------------------------------------------ expert-sorted fold --

def run_segmented(ld, di, case, offsets, add_inputs=True):
    d = di.linear_to_device(case)
    out = d.out0.clone()
    err = ld.new_error_word()
    ld.lora_delta_segmented(out, d.x, torch.from_numpy(offsets).cuda(), d.pool,
                            add_inputs=add_inputs, err=err)
    return di.bits(out), ld.lora_get_error(err)


@pytest.mark.parametrize("T,top_k,add", [(512, 8, True), (64, 2, False)])
def test_segmented_expert_fold(ld, di, oracle, T, top_k, add):
    """"expert_apply.rs", apply_expert_lora_sorted: each expert's block of
    sorted rows gets that expert's adapter, the blocks read from device
    offsets.  512 tokens x 8: ~64 rows per expert (both paths); 64 tokens x 2:
    many empty experts.  20% of experts unadapted; 37 rows past the last block."""
    case, offsets = inputs.expert_sorted_case(seed=17, T=T, top_k=top_k, E=64, k_in=1024,
                                              width=768, p_unadapted=0.2, tail_rows=37)
    got, err = run_segmented(ld, di, case, offsets, add_inputs=add)
    check_linear(oracle, case, got, err, add_inputs=add)


def test_segmented_expert_fold_full_size_sampled(ld, di, oracle):
    """2048 tokens x top-8 of 64 experts: 16,384 sorted rows, w13 width 1536."""
    case, offsets = inputs.expert_sorted_case()
    got, err = run_segmented(ld, di, case, offsets)
    rows = np.sort(np.random.default_rng(5).choice(case.n, 192, replace=False))
    check_linear(oracle, case, got, err, rows=rows)


def test_segmented_bad_offsets_are_clamped_and_flagged(ld, di):
    case, offsets = inputs.expert_sorted_case(seed=18, T=64, top_k=4, E=16, k_in=256, width=256)
    bad = offsets.copy()
    bad[5] = bad[7] + 50  # out of order
    bad[-1] = case.n + 1000  # past the batch
    _, err = run_segmented(ld, di, case, bad)
    assert err & 64  # LORA_DEV_ERR_SEGMENT


# ------------------------------------------------------------------- MoE --

def run_moe(ld, di, mc, topk=None, lora=None):
    dm = di.moe_to_device(mc)
    if topk is not None:
        dm.topk_ids = torch.from_numpy(topk).cuda()
    if lora is not None:
        dm.lora_ids = torch.from_numpy(lora).cuda()
    out = torch.full((mc.T, mc.top_k, 2 * mc.I), 3.0, dtype=torch.bfloat16, device="cuda")
    err = ld.new_error_word()
    ld.lora_moe_fc1_delta(out, dm.x, dm.w_ptr_a, dm.stride_a, dm.w_ptr_b, dm.stride_b,
                          mc.shared_a, dm.topk_ids, dm.lora_ids, mc.E, mc.I, mc.rank, mc.L,
                          mc.scale, err=err)
    return di.bits(out), ld.lora_get_error(err)


@pytest.mark.parametrize("shared", [False, True])
def test_moe_fc1_workload(ld, di, oracle, shared):
    mc = inputs.moe_case(shared_a=shared)
    got, err = run_moe(ld, di, mc)
    ref, ref_err = oracle.moe_fc1(mc.x, mc.A_banks, mc.B_banks, mc.topk_ids, mc.lora_ids, mc.I,
                                  mc.rank, mc.scale, shared, mc.L)
    assert err == ref_err == 0
    assert_close(got, ref, mc.name)
    skipped = mc.lora_ids < 0
    assert not got[skipped].any()


def test_moe_bad_ids(ld, di, oracle):
    mc = inputs.moe_case(T=40, top_k=3, E=6, H=64, I=24, rank=16, L=3, p_none=0.0)
    topk = mc.topk_ids.copy()
    lora = mc.lora_ids.copy()
    lora[0], lora[1] = -1, 3
    topk[2, 1], topk[3, 0] = 6, -5
    got, err = run_moe(ld, di, mc, topk, lora)
    ref, ref_err = oracle.moe_fc1(mc.x, mc.A_banks, mc.B_banks, topk, lora, mc.I, mc.rank,
                                  mc.scale, False, mc.L)
    assert err == ref_err == (2 | 4)
    assert_close(got, ref, "moe bad ids")
    assert not got[0].any() and not got[1].any() and not got[2, 1].any()


# ------------------------------------------- in-place MoE w13 / w2 deltas --

def _opt_cuda(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_w13(ld, di, mc, y0, expert_map=None, adapter_enabled=None, add_inputs=True, topk=None,
            lora=None):
    dm = di.moe_to_device(mc)
    if topk is not None:
        dm.topk_ids = torch.from_numpy(topk).cuda()
    if lora is not None:
        dm.lora_ids = torch.from_numpy(lora).cuda()
    y = di.bf16(y0, "cuda")
    err = ld.new_error_word()
    ld.lora_moe_w13_delta(y, dm.x, dm.w_ptr_a, dm.stride_a, dm.w_ptr_b, dm.stride_b,
                          mc.shared_a, dm.topk_ids, dm.lora_ids, dm.A_banks[0].shape[0], mc.I,
                          mc.rank, mc.L, mc.scale, expert_map=_opt_cuda(expert_map),
                          adapter_enabled=_opt_cuda(adapter_enabled), add_inputs=add_inputs,
                          err=err)
    return di.bits(y), ld.lora_get_error(err)


def run_w2(ld, di, c, expert_map=None, adapter_enabled=None, weights=None, add_inputs=True):
    dm = di.moe_to_device(c)
    y = di.bf16(c.y0, "cuda")
    err = ld.new_error_word()
    ld.lora_moe_w2_delta(y, dm.x, dm.w_ptr_a, dm.stride_a, dm.w_ptr_b, dm.stride_b,
                         dm.topk_ids, dm.lora_ids, dm.A_banks[0].shape[0], c.H, c.rank, c.L,
                         c.scale, expert_map=_opt_cuda(expert_map),
                         adapter_enabled=_opt_cuda(adapter_enabled),
                         topk_weights=_opt_cuda(weights), add_inputs=add_inputs, err=err)
    return di.bits(y), ld.lora_get_error(err)


@pytest.mark.parametrize("shared", [False, True])
def test_moe_w13_in_place_workload(ld, di, oracle, shared):
    """add_lora_w13 at the FC1 workload's size: 2048 tokens x top-8 of 64 experts."""
    mc = inputs.moe_case(shared_a=shared)
    y0 = inputs.moe_y0(mc.seed, (mc.T, mc.top_k, 2 * mc.I))
    got, err = run_w13(ld, di, mc, y0)
    ref, ref_err = oracle.moe_w13(y0, mc.x, mc.A_banks, mc.B_banks, mc.topk_ids, mc.lora_ids,
                                  mc.I, mc.rank, mc.scale, shared, mc.L)
    assert err == ref_err == 0
    assert_close(got, ref, "w13 " + mc.name)
    skipped = mc.lora_ids < 0
    assert np.array_equal(got[skipped], y0[skipped])


@pytest.mark.parametrize("add_inputs", [True, False])
def test_moe_w13_expert_map_switch_and_bad_ids(ld, di, oracle, add_inputs):
    """Expert parallel view: 12 global experts, 5 local (shuffled); adapter 1 switched
    off; an adapter id past the table, a global id past the map, a map entry past E."""
    mc = inputs.moe_case(seed=41, T=150, top_k=4, E=12, H=136, I=40, rank=8, L=3,
                         p_none=0.1)
    local = {2: 3, 5: 0, 7: 4, 8: 1, 11: 2}
    emap = np.full(12, -1, np.int32)
    for g, loc in local.items():
        emap[g] = loc
    emap[9] = 5  # past the 5 local experts
    inv = {loc: g for g, loc in local.items()}
    lc = inputs.MoeCase(**{**mc.__dict__, "E": 5,
                           "A_banks": [np.ascontiguousarray(b[[inv[i] for i in range(5)]])
                                       for b in mc.A_banks],
                           "B_banks": [np.ascontiguousarray(b[[inv[i] for i in range(5)]])
                                       for b in mc.B_banks]})
    en = np.array([1, 0, 1], np.int32)
    topk = mc.topk_ids.copy()
    lora = mc.lora_ids.copy()
    lora[3] = 3
    lora[4] = 0
    topk[4, 2] = 12
    y0 = inputs.moe_y0(41, (mc.T, mc.top_k, 2 * mc.I))
    got, err = run_w13(ld, di, lc, y0, expert_map=emap, adapter_enabled=en,
                       add_inputs=add_inputs, topk=topk, lora=lora)
    ref, ref_err = oracle.moe_w13(y0, lc.x, lc.A_banks, lc.B_banks, topk, lora, mc.I, mc.rank,
                                  mc.scale, False, mc.L, expert_map=emap, adapter_enabled=en,
                                  add_inputs=add_inputs)
    assert ref_err == (2 | 4)
    assert err == ref_err
    assert_close(got, ref, "w13 expert map")
    keep = np.all(ref == y0, axis=2)
    assert np.array_equal(got[keep], y0[keep])


@pytest.mark.parametrize("weighted", [False, True])
def test_moe_w2_in_place_workload(ld, di, oracle, weighted):
    """add_lora_w2 at the FC1 workload's routing: 2048 tokens x top-8 of 64 experts,
    per-pair activations [16384, 768] into intermediate_cache3 [2048, 8, 2048]."""
    c = inputs.moe_w2_case()
    w = c.topk_weights if weighted else None
    got, err = run_w2(ld, di, c, weights=w)
    ref, ref_err = oracle.moe_w2(c.y0, c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids,
                                 c.rank, c.scale, c.L, topk_weights=w)
    assert err == ref_err == 0
    assert_close(got, ref, c.name)
    skipped = c.lora_ids < 0
    assert np.array_equal(got[skipped], c.y0[skipped])


@pytest.mark.parametrize("add_inputs", [True, False])
def test_moe_w2_ragged_with_map_and_weights(ld, di, oracle, add_inputs):
    """Small ragged shapes: H 264 (a 64-column tail), I 40, rank 24 (a half MMA
    k-step), 7 global experts of which 4 local, routing weights, a switched-off adapter."""
    c = inputs.moe_w2_case(seed=43, T=70, top_k=3, E=7, H=264, I=40, rank=24, L=4, p_none=0.15)
    local = {0: 1, 3: 0, 4: 3, 6: 2}
    emap = np.full(7, -1, np.int32)
    for g, loc in local.items():
        emap[g] = loc
    inv = {loc: g for g, loc in local.items()}
    lc = inputs.MoeDownCase(**{**c.__dict__, "E": 4,
                               "A_banks": [np.ascontiguousarray(c.A_banks[0][[inv[i] for i in range(4)]])],
                               "B_banks": [np.ascontiguousarray(c.B_banks[0][[inv[i] for i in range(4)]])]})
    en = np.array([1, 1, 0, 1], np.int32)
    got, err = run_w2(ld, di, lc, expert_map=emap, adapter_enabled=en, weights=c.topk_weights,
                      add_inputs=add_inputs)
    ref, ref_err = oracle.moe_w2(c.y0, c.x, lc.A_banks, lc.B_banks, c.topk_ids, c.lora_ids,
                                 c.rank, c.scale, c.L, expert_map=emap, adapter_enabled=en,
                                 topk_weights=c.topk_weights, add_inputs=add_inputs)
    assert err == ref_err == 0
    assert_close(got, ref, "w2 ragged")
    keep = np.all(ref == c.y0, axis=2)
    assert keep.any() and np.array_equal(got[keep], c.y0[keep])


@pytest.mark.parametrize("shared", [False, True])
def test_moe_many_rows_per_key_rank_32(ld, di, oracle, shared):
    """Few keys with ~50 pairs each (two 32-row passes of the per-key kernel),
    rank 32 (two MMA k-steps), H 520 (a k tail of 8 after eight 64-column chunks)."""
    mc = inputs.moe_case(shared_a=shared, seed=47, T=150, top_k=2, E=3, H=520, I=48, rank=32,
                         L=2, p_none=0.05)
    got, err = run_moe(ld, di, mc)
    ref, ref_err = oracle.moe_fc1(mc.x, mc.A_banks, mc.B_banks, mc.topk_ids, mc.lora_ids, mc.I,
                                  mc.rank, mc.scale, shared, mc.L)
    assert err == ref_err == 0
    assert_close(got, ref, "moe many rows rank 32")
    y0 = inputs.moe_y0(47, (mc.T, mc.top_k, 2 * mc.I))
    got, err = run_w13(ld, di, mc, y0)
    ref, _ = oracle.moe_w13(y0, mc.x, mc.A_banks, mc.B_banks, mc.topk_ids, mc.lora_ids, mc.I,
                            mc.rank, mc.scale, shared, mc.L)
    assert err == 0
    assert_close(got, ref, "w13 many rows rank 32")


def test_moe_w2_contraction_longer_than_output(ld, di, oracle):
    """A down projection with I > H: per-pair input rows, routing weights, ~40 pairs per
    key, a k tail of 8."""
    c = inputs.moe_w2_case(seed=49, T=120, top_k=2, E=3, H=64, I=136, rank=16, L=2,
                           p_none=0.1)
    got, err = run_w2(ld, di, c, weights=c.topk_weights)
    ref, ref_err = oracle.moe_w2(c.y0, c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids,
                                 c.rank, c.scale, c.L, topk_weights=c.topk_weights)
    assert err == ref_err == 0
    assert_close(got, ref, "w2 I > H")
    keep = np.all(ref == c.y0, axis=2)
    assert np.array_equal(got[keep], c.y0[keep])


def test_moe_rank_64_takes_the_cluster_kernel(ld, di, oracle):
    """Rank 64 (S * R = 128 for the regular banks; rank above the per-key kernel's 32):
    FC1, w13 and w2 with routing weights on the cluster kernel."""
    mc = inputs.moe_case(seed=51, T=60, top_k=3, E=4, H=128, I=40, rank=64, L=2, p_none=0.1)
    got, err = run_moe(ld, di, mc)
    ref, ref_err = oracle.moe_fc1(mc.x, mc.A_banks, mc.B_banks, mc.topk_ids, mc.lora_ids, mc.I,
                                  mc.rank, mc.scale, False, mc.L)
    assert err == ref_err == 0
    assert_close(got, ref, "moe fc1 rank 64")
    y0 = inputs.moe_y0(51, (mc.T, mc.top_k, 2 * mc.I))
    got, err = run_w13(ld, di, mc, y0)
    ref, _ = oracle.moe_w13(y0, mc.x, mc.A_banks, mc.B_banks, mc.topk_ids, mc.lora_ids, mc.I,
                            mc.rank, mc.scale, False, mc.L)
    assert err == 0
    assert_close(got, ref, "w13 rank 64")
    c = inputs.moe_w2_case(seed=53, T=60, top_k=3, E=4, H=96, I=48, rank=64, L=2, p_none=0.1)
    got, err = run_w2(ld, di, c, weights=c.topk_weights)
    ref, ref_err = oracle.moe_w2(c.y0, c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids,
                                 c.rank, c.scale, c.L, topk_weights=c.topk_weights)
    assert err == ref_err == 0
    assert_close(got, ref, "w2 rank 64")


def test_moe_edge_cases_on_the_per_key_kernel(ld, di, oracle):
    """Pass boundaries (keys with exactly 32 and 33 pairs at top-1), no local expert at all
    (an expert map of -1: y untouched, no error), every adapter switched off (w2: y
    untouched), and an empty batch (T = 0: nothing launched, status OK)."""
    import torch
    # top-1, two experts, one adapter: expert 0 gets 32 tokens, expert 1 gets 33
    mc = inputs.moe_case(seed=55, T=65, top_k=1, E=2, H=64, I=16, rank=16, L=1, p_none=0.0)
    topk = np.array([[0]] * 32 + [[1]] * 33, dtype=np.int32)
    got, err = run_moe(ld, di, mc, topk=topk)
    ref, ref_err = oracle.moe_fc1(mc.x, mc.A_banks, mc.B_banks, topk, mc.lora_ids, mc.I,
                                  mc.rank, mc.scale, False, mc.L)
    assert err == ref_err == 0
    assert_close(got, ref, "moe 32 / 33 pairs per key")

    y0 = inputs.moe_y0(55, (mc.T, mc.top_k, 2 * mc.I))
    none_local = np.full(4, -1, np.int32)
    got, err = run_w13(ld, di, mc, y0, expert_map=none_local, topk=topk)
    assert err == 0 and np.array_equal(got, y0)

    c = inputs.moe_w2_case(seed=57, T=40, top_k=2, E=3, H=64, I=32, rank=16, L=2, p_none=0.0)
    got, err = run_w2(ld, di, c, adapter_enabled=np.zeros(2, np.int32), weights=c.topk_weights)
    assert err == 0 and np.array_equal(got, c.y0)

    dm = di.moe_to_device(mc)
    empty_x = torch.empty(0, mc.H, dtype=torch.bfloat16, device="cuda")
    empty_ids = torch.empty(0, 1, dtype=torch.int32, device="cuda")
    empty_l = torch.empty(0, dtype=torch.int32, device="cuda")
    out = torch.empty(0, 1, 2 * mc.I, dtype=torch.bfloat16, device="cuda")
    e = ld.new_error_word()
    ld.lora_moe_fc1_delta(out, empty_x, dm.w_ptr_a, dm.stride_a, dm.w_ptr_b, dm.stride_b, False,
                          empty_ids, empty_l, mc.E, mc.I, mc.rank, mc.L, mc.scale, err=e)
    assert ld.lora_get_error(e) == 0


# ------------------------------------------ duplicate experts in top-k --
# "bgmv_moe_gemm1_lora_delta", topk_ids: nothing makes a token's experts
# distinct.  A token that reaches one expert through two or more of its slots
# puts the same x row into one (adapter, expert) key more than once; every such
# pair is still its own output row.

@pytest.mark.parametrize("rank", [16, 64])
@pytest.mark.parametrize("shared", [False, True])
def test_moe_fc1_and_w13_with_duplicate_experts(ld, di, oracle, shared, rank):
    """30% of the tokens repeat experts.  Rank 16 at the FC1 workload's full size
    (2048 tokens x top-8 of 64: the per-key kernel); rank 64 on a smaller case
    (the cluster kernel)."""
    if rank == 16:
        mc = inputs.moe_case(shared_a=shared, dup_frac=0.3)
    else:
        mc = inputs.moe_case(shared_a=shared, seed=61, T=200, top_k=4, E=6, H=256, I=64,
                             rank=64, L=3, p_none=0.1, dup_frac=0.4)
    assert any(len(set(r)) < mc.top_k for r in mc.topk_ids.tolist())
    got, err = run_moe(ld, di, mc)
    ref, ref_err = oracle.moe_fc1(mc.x, mc.A_banks, mc.B_banks, mc.topk_ids, mc.lora_ids, mc.I,
                                  mc.rank, mc.scale, shared, mc.L)
    assert err == ref_err == 0
    assert_close(got, ref, "fc1 duplicates " + mc.name)
    assert not got[mc.lora_ids < 0].any()
    y0 = inputs.moe_y0(mc.seed + 1, (mc.T, mc.top_k, 2 * mc.I))
    got, err = run_w13(ld, di, mc, y0)
    ref, ref_err = oracle.moe_w13(y0, mc.x, mc.A_banks, mc.B_banks, mc.topk_ids, mc.lora_ids,
                                  mc.I, mc.rank, mc.scale, shared, mc.L)
    assert err == ref_err == 0
    assert_close(got, ref, "w13 duplicates " + mc.name)
    assert np.array_equal(got[mc.lora_ids < 0], y0[mc.lora_ids < 0])


@pytest.mark.parametrize("rank", [16, 64])
def test_moe_w2_weighted_with_duplicate_experts(ld, di, oracle, rank):
    """The down projection with routing weights when 30% of the tokens repeat
    experts: each duplicated pair folds its own activation row and weight."""
    if rank == 16:
        c = inputs.moe_w2_case(dup_frac=0.3)
    else:
        c = inputs.moe_w2_case(seed=63, T=150, top_k=4, E=5, H=192, I=96, rank=64, L=3,
                               p_none=0.1, dup_frac=0.4)
    assert any(len(set(r)) < c.top_k for r in c.topk_ids.tolist())
    got, err = run_w2(ld, di, c, weights=c.topk_weights)
    ref, ref_err = oracle.moe_w2(c.y0, c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids,
                                 c.rank, c.scale, c.L, topk_weights=c.topk_weights)
    assert err == ref_err == 0
    assert_close(got, ref, "w2 duplicates " + c.name)
    assert np.array_equal(got[c.lora_ids < 0], c.y0[c.lora_ids < 0])


def test_moe_duplicates_inside_a_key_that_spans_several_passes(ld, di, oracle):
    """Every token sends three of its four slots to expert 0 and one to expert 1,
    with one adapter: key (0, 0) holds 72 pairs (passes of 32, 32 and 8 rows of
    the per-key kernel) and the three copies of a token's row fall inside one
    pass or across a pass boundary.  FC1 regular, w13 and weighted w2."""
    mc = inputs.moe_case(seed=65, T=24, top_k=4, E=2, H=328, I=40, rank=16, L=1, p_none=0.0)
    topk = np.tile(np.array([0, 0, 1, 0], np.int32), (mc.T, 1))
    got, err = run_moe(ld, di, mc, topk=topk)
    ref, ref_err = oracle.moe_fc1(mc.x, mc.A_banks, mc.B_banks, topk, mc.lora_ids, mc.I,
                                  mc.rank, mc.scale, False, mc.L)
    assert err == ref_err == 0
    assert_close(got, ref, "fc1 72-pair key with duplicates")
    y0 = inputs.moe_y0(65, (mc.T, mc.top_k, 2 * mc.I))
    got, err = run_w13(ld, di, mc, y0, topk=topk)
    ref, _ = oracle.moe_w13(y0, mc.x, mc.A_banks, mc.B_banks, topk, mc.lora_ids, mc.I,
                            mc.rank, mc.scale, False, mc.L)
    assert err == 0
    assert_close(got, ref, "w13 72-pair key with duplicates")
    c = inputs.moe_w2_case(seed=67, T=24, top_k=4, E=2, H=136, I=72, rank=16, L=1, p_none=0.0)
    c.topk_ids = np.tile(np.array([1, 0, 0, 0], np.int32), (c.T, 1))
    got, err = run_w2(ld, di, c, weights=c.topk_weights)
    ref, ref_err = oracle.moe_w2(c.y0, c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids,
                                 c.rank, c.scale, c.L, topk_weights=c.topk_weights)
    assert err == ref_err == 0
    assert_close(got, ref, "w2 72-pair key with duplicates")


# ------------------------------------------------- tensor-core (SGMV) path --

def _hot_slots_case(seed, n, k_in, widths, R, ranks, hot=(0, 1), **kw):
    """Two hot slots (well over the tensor-core threshold, ragged 128-row tiles)
    and a sprinkle of rows on the other slots (small-segment kernel)."""
    rng = np.random.default_rng(seed + 500)
    L = len(ranks)
    seq = rng.integers(0, L, size=n).astype(np.int32)
    hot_mask = rng.random(n) < 0.8
    seq[hot_mask] = rng.choice(np.array(hot), size=int(hot_mask.sum()))
    seq[rng.random(n) < 0.05] = -1
    return inputs.linear_case(seed, n=n, k_in=k_in, widths=widths, max_loras=L, max_rank=R,
                              ranks=ranks, alpha=float(R), seq_slot=seq, **kw)


@pytest.mark.parametrize("k_in,widths,R,ranks", [
    (200, (136, 24), 8, [8, 4, 8, 2]),            # k tail of 8, half column tiles, R < 16
    (328, (64, 40, 24), 24, [24, 16, 24, 8]),     # R not a power of two, three slices
    (256, (96, 160), 128, [128, 64, 96, 128]),    # largest rank: two 64-wide k-blocks
])
def test_sgmv_edge_shapes(ld, di, oracle, k_in, widths, R, ranks):
    case = _hot_slots_case(3 + R, 1500, k_in, widths, R, ranks)
    got, err, _ = run_fused(ld, di, case)
    check_linear(oracle, case, got, err)


def test_sgmv_inactive_slice_offsets_and_no_add(ld, di, oracle):
    adapted = [[True, False], [True, True], [False, True], [True, True]]
    case = _hot_slots_case(21, 1300, 512, (128, 64), 16, [16, 16, 8, 16], hot=(0, 2),
                           adapted=adapted, offset_start=24, ld_out=240)
    got, err, _ = run_fused(ld, di, case)
    check_linear(oracle, case, got, err)
    got2, err2, _ = run_fused(ld, di, case, add_inputs=False)
    check_linear(oracle, case, got2, err2, add_inputs=False)


def test_sgmv_and_small_path_agree_on_a_hot_slot(ld, di, oracle):
    """The same batch through the tensor-core path (workspace given) and the
    small-segment kernel alone (no workspace, n <= 1024) agree within tolerance."""
    case = _hot_slots_case(33, 1000, 384, (256,), 32, [32, 16, 32], hot=(0,))
    d = di.linear_to_device(case)
    a = d.out0.clone()
    ws = torch.empty(ld.lora_workspace_size(case.n, 1, 32, 3), dtype=torch.uint8, device="cuda")
    ld.lora_delta_fused(a, d.x, d.seq_slot, d.pool, workspace=ws)
    b = d.out0.clone()
    L = ld.lib()
    import ctypes
    w = (ctypes.c_int32 * 1)(256)
    rc = L.lora_delta_fused(ctypes.c_void_p(b.data_ptr()), 256, ctypes.c_void_p(d.x.data_ptr()),
                            case.n, 384, ctypes.c_void_p(d.seq_slot.data_ptr()),
                            ctypes.c_void_p(d.pool.a_table.data_ptr()),
                            ctypes.c_void_p(d.pool.b_table.data_ptr()),
                            ctypes.c_void_p(d.pool.scale_table.data_ptr()), w, 1, 32, 3, 0, 1,
                            None, 0, None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert_close(di.bits(a), di.bits(b), "tensor-core vs small-segment path")
    ref, _ = oracle_delta(oracle, case)
    assert_close(di.bits(a), ref, "tensor-core path vs oracle")


@pytest.mark.parametrize("n", [1000, 1500])
def test_split_call_replays_from_a_cuda_graph(ld, di, oracle, n):
    """A call whose keys split between the tensor-core path and the small-segment
    kernel runs the latter on a second stream, forked and joined by events (at
    1000 rows before the routing sort, the kernel scanning its rows itself; at
    1500 after it).  Captured in a CUDA graph on a side stream and replayed, it
    gives the eager call's bits, and those match the oracle."""
    # two hot slots of 400-600 rows, ten others of 15-30 (below the threshold of 64)
    case = _hot_slots_case(41, n, 512, (384, 128), 16,
                           [16, 8, 16, 4, 16, 12, 16, 8, 2, 16, 1, 16], hot=(0, 3))
    counts = np.bincount(case.seq_slot[case.seq_slot >= 0], minlength=12)
    assert counts[[0, 3]].min() >= 64 and 0 < np.delete(counts, [0, 3]).max() < 64
    d = di.linear_to_device(case)
    ws = torch.empty(ld.lora_workspace_size(case.n, 2, 16, 12), dtype=torch.uint8, device="cuda")
    eager = d.out0.clone()
    ld.lora_delta_fused(eager, d.x, d.seq_slot, d.pool, workspace=ws)
    torch.cuda.synchronize()
    got = d.out0.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            ld.lora_delta_fused(got, d.x, d.seq_slot, d.pool, workspace=ws, stream=s)
    torch.cuda.synchronize()
    for _ in range(2):  # replays start from the same out
        got.copy_(d.out0)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(di.bits(got), di.bits(eager))
    ref, _ = oracle_delta(oracle, case)
    assert_close(di.bits(eager), ref, case.name)


def test_split_call_on_the_legacy_default_stream(ld, di, oracle):
    """The C ABI with stream NULL (the legacy default stream) on a call whose keys
    split between the two paths: the second stream is forked from and joined to
    it like any other; the result equals the same call on a created stream."""
    import ctypes
    case = _hot_slots_case(43, 1500, 512, (384, 128), 16,
                           [16, 8, 16, 4, 16, 12, 16, 8, 2, 16, 1, 16], hot=(0, 3))
    d = di.linear_to_device(case)
    ws = torch.empty(ld.lora_workspace_size(case.n, 2, 16, 12), dtype=torch.uint8, device="cuda")
    ref = d.out0.clone()
    ld.lora_delta_fused(ref, d.x, d.seq_slot, d.pool, workspace=ws)
    torch.cuda.synchronize()
    got = d.out0.clone()
    torch.cuda.synchronize()
    L = ld.lib()
    w = (ctypes.c_int32 * 2)(384, 128)
    rc = L.lora_delta_fused(ctypes.c_void_p(got.data_ptr()), 512, ctypes.c_void_p(d.x.data_ptr()),
                            case.n, 512, ctypes.c_void_p(d.seq_slot.data_ptr()),
                            ctypes.c_void_p(d.pool.a_table.data_ptr()),
                            ctypes.c_void_p(d.pool.b_table.data_ptr()),
                            ctypes.c_void_p(d.pool.scale_table.data_ptr()), w, 2, 16, 12, 0, 1,
                            ctypes.c_void_p(ws.data_ptr()), ws.numel(), None, None)
    assert rc == 0
    torch.cuda.synchronize()
    assert np.array_equal(di.bits(got), di.bits(ref))
    ref_o, _ = oracle_delta(oracle, case)
    assert_close(di.bits(got), ref_o, case.name)


def test_split_calls_from_two_host_threads(ld, di):
    """Two host threads making split calls on their own streams at once (the library
    call releases the interpreter lock): the forks and joins of the shared second
    stream are recorded under the library's lock, and every output equals the same
    call made alone."""
    import threading
    cases = [_hot_slots_case(44 + t, 1500, 512, (384, 128), 16,
                             [16, 8, 16, 4, 16, 12, 16, 8, 2, 16, 1, 16], hot=(0, 3))
             for t in range(2)]
    devs = [di.linear_to_device(c) for c in cases]
    wss = [torch.empty(ld.lora_workspace_size(c.n, 2, 16, 12), dtype=torch.uint8, device="cuda")
           for c in cases]
    refs = []
    for d, ws in zip(devs, wss):
        o = d.out0.clone()
        ld.lora_delta_fused(o, d.x, d.seq_slot, d.pool, workspace=ws)
        refs.append(di.bits(o))
    torch.cuda.synchronize()
    reps = 12
    outs = [[d.out0.clone() for _ in range(reps)] for d in devs]
    streams = [torch.cuda.Stream() for _ in devs]
    errors = []

    def worker(t):
        try:
            with torch.cuda.stream(streams[t]):
                for k in range(reps):
                    ld.lora_delta_fused(outs[t][k], devs[t].x, devs[t].seq_slot, devs[t].pool,
                                        workspace=wss[t], stream=streams[t])
        except Exception as e:  # (reported below)
            errors.append(e)

    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    threads = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for t in range(2):
        for k in range(reps):
            assert np.array_equal(di.bits(outs[t][k]), refs[t]), (t, k)


# ------------------------------------------------------ bounded waits --

def test_wait_time_out_sets_the_error_bit_and_the_next_call_is_correct(ld, di, oracle):
    """Every mbarrier wait of the tensor-core kernels is bounded.  With the limit
    at 0 (lora_set_wait_limit_ns) a wait that finds its phase incomplete gives up
    at once: its CTA records LORA_DEV_ERR_TIMEOUT (8), skips its stores, lets its
    issued MMAs finish, frees its tensor memory and returns.  A call on a hot slot
    (the tensor-core path) must report the bit and end; the next call, at the
    default limit, must be correct: the tensor memory was released and nothing
    hangs."""
    case = _hot_slots_case(71, 1200, 512, (256, 128), 16, [16, 16, 8, 16], hot=(0,))
    d = di.linear_to_device(case)
    ws = torch.empty(ld.lora_workspace_size(case.n, 2, 16, 4), dtype=torch.uint8,
                     device="cuda")
    out = d.out0.clone()
    err = ld.new_error_word()
    prev = ld.lora_set_wait_limit_ns(0)
    try:
        ld.lora_delta_fused(out, d.x, d.seq_slot, d.pool, workspace=ws, err=err)
        e = ld.lora_get_error(err)
    finally:
        assert ld.lora_set_wait_limit_ns(prev) == 0
    assert prev == ld.WAIT_LIMIT_DEFAULT_NS
    assert e & 8, f"no wait gave up (error word {e})"
    for _ in range(2):
        out2 = d.out0.clone()
        err2 = ld.new_error_word()
        ld.lora_delta_fused(out2, d.x, d.seq_slot, d.pool, workspace=ws, err=err2)
        e2 = ld.lora_get_error(err2)
        check_linear(oracle, case, di.bits(out2), e2)


# ------------------------------------------- w13 -> w2 routing hand-over --

@pytest.mark.parametrize("full", [True, False])
def test_moe_w2_on_the_routing_of_w13(ld, di, oracle, full):
    """"punica_base.py", add_lora_w2: "Reuses routing tensors returned by
    add_lora_w13".  lora_moe_w2_delta_routed reads the clustering that the
    preceding lora_moe_w13_delta left in its workspace.  Its result equals
    lora_moe_w2_delta's (which sorts again) bit for bit, and the oracle's within
    the tolerance; pairs with no delta keep y.  Full size: the FC1 workload's
    routing with routing weights.  Small: an expert map (5 of 12 experts local),
    a switched-off adapter and repeated experts."""
    if full:
        mc = inputs.moe_case(seed=1240)
        c = inputs.moe_w2_case()
        mc.topk_ids, mc.lora_ids = c.topk_ids, c.lora_ids
        emap = en = None
        E_loc = c.E
    else:
        mc = inputs.moe_case(seed=73, T=90, top_k=4, E=12, H=136, I=48, rank=16, L=3,
                             p_none=0.1, dup_frac=0.3)
        c = inputs.moe_w2_case(seed=75, T=90, top_k=4, E=12, H=136, I=48, rank=16, L=3)
        c.topk_ids, c.lora_ids = mc.topk_ids, mc.lora_ids
        local = {2: 3, 5: 0, 7: 4, 8: 1, 11: 2}
        emap = np.full(12, -1, np.int32)
        for g, loc in local.items():
            emap[g] = loc
        inv = {loc: g for g, loc in local.items()}
        pick = lambda b: np.ascontiguousarray(b[[inv[i] for i in range(5)]])
        mc = inputs.MoeCase(**{**mc.__dict__, "E": 5, "A_banks": [pick(b) for b in mc.A_banks],
                               "B_banks": [pick(b) for b in mc.B_banks]})
        c = inputs.MoeDownCase(**{**c.__dict__, "E": 5, "A_banks": [pick(c.A_banks[0])],
                                  "B_banks": [pick(c.B_banks[0])]})
        en = np.array([1, 0, 1], np.int32)
        E_loc = 5
    dm = di.moe_to_device(mc)
    d2 = di.moe_to_device(c)
    topk, lora = dm.topk_ids, dm.lora_ids
    y13 = di.bf16(inputs.moe_y0(mc.seed, (mc.T, mc.top_k, 2 * mc.I)), "cuda")
    ws = torch.empty(ld.lora_moe_workspace_size(mc.T, mc.top_k, E_loc, mc.L, mc.rank, False),
                     dtype=torch.uint8, device="cuda")
    wts = torch.from_numpy(c.topk_weights).cuda()
    err = ld.new_error_word()
    ld.lora_moe_w13_delta(y13, dm.x, dm.w_ptr_a, dm.stride_a, dm.w_ptr_b, dm.stride_b, False,
                          topk, lora, E_loc, mc.I, mc.rank, mc.L, mc.scale,
                          expert_map=_opt_cuda(emap), adapter_enabled=_opt_cuda(en),
                          workspace=ws, err=err)
    y_routed = di.bf16(c.y0, "cuda")
    ld.lora_moe_w2_delta_routed(y_routed, d2.x, d2.w_ptr_a, d2.stride_a, d2.w_ptr_b, d2.stride_b,
                                c.T, c.top_k, E_loc, c.H, c.rank, c.L, c.scale, ws,
                                topk_weights=wts, err=err)
    e = ld.lora_get_error(err)
    y_own = di.bf16(c.y0, "cuda")
    ld.lora_moe_w2_delta(y_own, d2.x, d2.w_ptr_a, d2.stride_a, d2.w_ptr_b, d2.stride_b, topk,
                         lora, E_loc, c.H, c.rank, c.L, c.scale, expert_map=_opt_cuda(emap),
                         adapter_enabled=_opt_cuda(en), topk_weights=wts)
    got = di.bits(y_routed)
    assert np.array_equal(got, di.bits(y_own))
    ref, ref_err = oracle.moe_w2(c.y0, c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids,
                                 c.rank, c.scale, c.L, expert_map=emap, adapter_enabled=en,
                                 topk_weights=c.topk_weights)
    assert e == ref_err
    assert_close(got, ref, "w2 on the routing of w13")
    keep = np.all(ref == c.y0, axis=2)
    assert keep.any() and np.array_equal(got[keep], c.y0[keep])


# ------------------------------------------- tensor-parallel sharded forms --

@pytest.mark.parametrize("tp_n", [2, 4])
def test_tensor_parallel_forms_with_the_ranks_in_turn_on_one_gpu(ld, di, oracle, tp_n):
    """"vllm.lora.fully_sharded_layers": the kernels of both sharded forms, each
    rank's step run in turn on this GPU, the collective between them done by a
    stack (the all-gather) or by adds in rank order (the all-reduce); no kernel
    waits on another rank.  Column parallel (_mcp_apply): every rank's output
    columns within the tolerance of the oracle's column form, which equals the
    unsharded delta bit for bit.  Row parallel (RowParallelLinearWithShardedLoRA
    apply): every rank's slice within the tolerance of the oracle's row form, the
    rest of its partial-sum output untouched."""
    from lora_delta_gb300 import tp
    case = inputs.linear_case(141, n=300, k_in=512, widths=(256, 128), max_loras=5,
                              max_rank=32, ranks=[32, 16, 8, 32, 24], alpha=32.0, p_none=0.1)
    d = di.linear_to_device(case)
    opool = oracle.build_pool(case.adapters, case.k_in, case.widths, 5, 32)
    want, _ = oracle_delta(oracle, case)
    shards = []
    for p in range(tp_n):
        h_p = torch.zeros(2, case.n, 32 // tp_n, dtype=torch.float32, device="cuda")
        ld.lora_shrink(h_p, d.x, d.seq_slot, tp.shard_pool_a_rows(d.pool, tp_n, p))
        shards.append(h_p)
    h_all = torch.stack(shards)
    routed = case.seq_slot >= 0
    for p in range(tp_n):
        cols = np.concatenate([np.arange(off + p * (w // tp_n), off + (p + 1) * (w // tp_n))
                               for off, w in ((0, 256), (256, 128))])
        out_p = d.out0[:, torch.from_numpy(cols).cuda()].contiguous()
        pb = tp.shard_pool_b_rows(d.pool, tp_n, p)
        ld.lora_expand_gathered(out_p, h_all, d.seq_slot, pb, scale_table=pb.scale_table)
        got = di.bits(out_p)
        assert_close(got, want[:, cols], f"column parallel rank {p}")
        assert np.array_equal(got[~routed], case.out0[~routed][:, cols])

    rc = inputs.linear_case(143, n=200, k_in=1024, widths=(512,), max_loras=4, max_rank=16,
                            ranks=[16, 8, 16, 4], alpha=32.0, p_none=0.1)
    rd = di.linear_to_device(rc)
    rpool = oracle.build_pool(rc.adapters, rc.k_in, rc.widths, 4, 16)
    ks, wsl = rc.k_in // tp_n, rc.widths[0] // tp_n
    parts, oparts = [], []
    for p in range(tp_n):
        h_p = torch.zeros(1, rc.n, 16, dtype=torch.float32, device="cuda")
        ld.lora_shrink(h_p, rd.x[:, p * ks:(p + 1) * ks].contiguous(), rd.seq_slot,
                       tp.shard_pool_a_cols(rd.pool, tp_n, p))
        parts.append(h_p)
        oparts.append(oracle.shrink(np.ascontiguousarray(rc.x[:, p * ks:(p + 1) * ks]),
                                    rc.seq_slot, oracle.shard_pool_a_cols(rpool, tp_n, p),
                                    None)[0])
    h = parts[0]
    for h_p in parts[1:]:
        h = h + h_p
    oh = oracle.rank_sum(np.stack(oparts))
    for p in range(tp_n):
        out_p = rd.out0.clone()
        pb = tp.shard_pool_b_rows(rd.pool, tp_n, p)
        ld.lora_expand(out_p, h, rd.seq_slot, pb, scale_table=pb.scale_table,
                       offset_start=p * wsl)
        ref = rc.out0.copy()
        oracle.expand(ref, oh, rc.seq_slot, oracle.shard_pool_b_rows(rpool, tp_n, p),
                      rpool.scale_table, offset_start=p * wsl)
        got = di.bits(out_p)
        assert_close(got, ref, f"row parallel rank {p}")
        inside = np.zeros(rc.ld_out, dtype=bool)
        inside[p * wsl:(p + 1) * wsl] = True
        assert np.array_equal(got[:, ~inside], rc.out0[:, ~inside])
