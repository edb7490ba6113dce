"""The data-parallel split, on two CPU processes over gloo.

Rows of the linear delta and tokens of the MoE deltas are independent
("Module lora_delta": one adapter per row through LoraRoute;
"bgmv_moe_gemm1_lora_delta": the delta stays per (token, slot); the in-place w2
delta of "punica_base.py" reads each pair's own activation row).  Ranks that
each apply the delta to their own contiguous shard, with the adapter pool
replicated, therefore reproduce the whole batch bit for bit, with no
collective on the data path.  The test also checks the host reductions the
benchmark's timing uses: barrier, max over ranks (the slowest rank's time) and
sum over ranks (the rows all ranks processed).

Each rank runs the oracle on its shard: what is tested here is the host-side
sharding logic, which is the same on a GPU machine.
"""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORLD = 2


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    try:
        import torch.distributed as dist

        import oracle
        from lora_delta_gb300 import dist as ldist
        from lora_delta_gb300 import inputs

        r, w = ldist.init("gloo")
        assert (r, w) == (rank, world)
        res = {}

        # linear delta: contiguous row shards of a decode-shaped batch (67 rows:
        # shards of 34 and 33; 3 slices, 6 slots of mixed rank, 10% unrouted)
        case = inputs.linear_case(4321, 67, 512, (256, 128, 128), 6, 16, [16, 8, 16, 4, 16, 8],
                                  32.0, p_none=0.1)
        pool = oracle.build_pool(case.adapters, case.k_in, case.widths, case.max_loras,
                                 case.max_rank)
        lo, hi = ldist.shard_rows(case.n, r, w)
        out = case.out0[lo:hi].copy()  # (a row slice can be a view of out0)
        err = oracle.delta(out, case.x[lo:hi], case.seq_slot[lo:hi], pool)
        shards = [None] * w
        dist.all_gather_object(shards, (lo, hi, out, err))

        # MoE FC1: token shards
        mc = inputs.moe_case(T=37, top_k=4, E=8, H=256, I=64, rank=16, L=4)
        tlo, thi = ldist.shard_rows(mc.T, r, w)
        mo, merr = oracle.moe_fc1(np.ascontiguousarray(mc.x[tlo:thi]), mc.A_banks, mc.B_banks,
                                  np.ascontiguousarray(mc.topk_ids[tlo:thi]),
                                  np.ascontiguousarray(mc.lora_ids[tlo:thi]), mc.I, mc.rank,
                                  mc.scale, mc.shared_a, mc.L)
        mshards = [None] * w
        dist.all_gather_object(mshards, (tlo, thi, mo, merr))

        # in-place w2 on token shards: the shard's pairs are rows tlo*top_k .. thi*top_k
        # of the activations, its y rows are tokens tlo .. thi
        dc = inputs.moe_w2_case(T=37, top_k=4, E=8, H=64, I=32, rank=16, L=4)
        dlo, dhi = ldist.shard_rows(dc.T, r, w)
        dy, derr = oracle.moe_w2(np.ascontiguousarray(dc.y0[dlo:dhi]),
                                 np.ascontiguousarray(dc.x[dlo * dc.top_k:dhi * dc.top_k]),
                                 dc.A_banks, dc.B_banks,
                                 np.ascontiguousarray(dc.topk_ids[dlo:dhi]),
                                 np.ascontiguousarray(dc.lora_ids[dlo:dhi]), dc.rank, dc.scale,
                                 dc.L, topk_weights=np.ascontiguousarray(dc.topk_weights[dlo:dhi]))
        dshards = [None] * w
        dist.all_gather_object(dshards, (dlo, dhi, dy, derr))

        ldist.barrier()
        res["max"] = ldist.max_over_ranks(1.5 + rank)
        res["sum"] = ldist.sum_over_ranks(10 * (rank + 1))
        if rank == 0:
            whole = case.out0.copy()
            werr = oracle.delta(whole, case.x, case.seq_slot, pool)
            got = np.concatenate([s[2] for s in sorted(shards, key=lambda s: s[0])])
            res["cover"] = sorted((s[0], s[1]) for s in shards)
            res["linear_equal"] = bool(np.array_equal(got, whole))
            res["linear_err"] = (werr, [s[3] for s in shards])
            mwhole, mwerr = oracle.moe_fc1(mc.x, mc.A_banks, mc.B_banks, mc.topk_ids,
                                           mc.lora_ids, mc.I, mc.rank, mc.scale, mc.shared_a,
                                           mc.L)
            mgot = np.concatenate([s[2] for s in sorted(mshards, key=lambda s: s[0])])
            res["moe_equal"] = bool(np.array_equal(mgot, mwhole))
            res["moe_cover"] = sorted((s[0], s[1]) for s in mshards)
            dwhole, _ = oracle.moe_w2(dc.y0, dc.x, dc.A_banks, dc.B_banks, dc.topk_ids,
                                      dc.lora_ids, dc.rank, dc.scale, dc.L,
                                      topk_weights=dc.topk_weights)
            dgot = np.concatenate([s[2] for s in sorted(dshards, key=lambda s: s[0])])
            res["w2_equal"] = bool(np.array_equal(dgot, dwhole))
        dist.destroy_process_group()
        q.put((rank, res, None))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, None, repr(e)))


def test_shard_rows_partitions_contiguously():
    from lora_delta_gb300.dist import shard_rows
    for n in (0, 1, 7, 64, 67, 8192):
        for w in (1, 2, 3, 8):
            parts = [shard_rows(n, r, w) for r in range(w)]
            assert parts[0][0] == 0 and parts[-1][1] == n
            assert all(parts[i][1] == parts[i + 1][0] for i in range(w - 1))
            sizes = [hi - lo for lo, hi in parts]
            assert max(sizes) - min(sizes) <= 1


def test_two_rank_shards_reproduce_the_whole_batch(oracle):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, WORLD, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    results = {}
    try:
        for _ in range(WORLD):
            rank, res, err = q.get(timeout=240)
            assert err is None, f"rank {rank}: {err}"
            results[rank] = res
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    for rank in range(WORLD):
        assert results[rank]["max"] == 1.5 + (WORLD - 1)
        assert results[rank]["sum"] == sum(10 * (r + 1) for r in range(WORLD))
    r0 = results[0]
    assert r0["cover"] == [(0, 34), (34, 67)]
    assert r0["linear_equal"]
    werr, shard_errs = r0["linear_err"]
    assert werr == (shard_errs[0] | shard_errs[1])
    assert r0["moe_cover"] == [(0, 19), (19, 37)]
    assert r0["moe_equal"]
    assert r0["w2_equal"]


# ------------------------------------------- tensor-parallel sharded forms --
# "vllm.lora.fully_sharded_layers": the collective steps of lora_delta_gb300.tp
# (the all-gather of the column-parallel h shards, the all-reduce of the
# row-parallel h partials) between per-rank oracle shrinks and expands.

def _tp_worker(rank: int, world: int, port: int, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    try:
        import torch
        import torch.distributed as dist

        import oracle
        from lora_delta_gb300 import dist as ldist
        from lora_delta_gb300 import inputs, tp

        r, w = ldist.init("gloo")
        res = {}
        # column parallel: two slices, ranks 16 split in two 8-row halves
        case = inputs.linear_case(4401, 45, 256, (128, 64), 5, 16, [16, 8, 16, 12, 16], 32.0,
                                  p_none=0.1)
        pool = oracle.build_pool(case.adapters, case.k_in, case.widths, 5, 16)
        h_shard, _ = oracle.shrink(case.x, case.seq_slot, oracle.shard_pool_a_rows(pool, w, r),
                                   None)
        h_all = tp.gather_rank_shards(torch.from_numpy(h_shard)).numpy()
        mine = [None] * w
        dist.all_gather_object(mine, h_shard)
        res["gather_rank_major"] = bool(np.array_equal(h_all, np.stack(mine)))
        h = oracle.gather_rank_blocks(h_all)
        cols, off = [], 0
        for wd in case.widths:
            cols.extend(range(off + r * (wd // w), off + (r + 1) * (wd // w)))
            off += wd
        cols = np.array(cols)
        out_c = np.ascontiguousarray(case.out0[:, cols])
        oracle.expand(out_c, h, case.seq_slot, oracle.shard_pool_b_rows(pool, w, r),
                      pool.scale_table)
        col_shards = [None] * w
        dist.all_gather_object(col_shards, (cols, out_c))

        # row parallel: one slice, k_in split in two
        rc = inputs.linear_case(4403, 39, 256, (96,), 4, 16, [16, 4, 16, 8], 32.0, p_none=0.1)
        rpool = oracle.build_pool(rc.adapters, rc.k_in, rc.widths, 4, 16)
        ks = rc.k_in // w
        part, _ = oracle.shrink(np.ascontiguousarray(rc.x[:, r * ks:(r + 1) * ks]), rc.seq_slot,
                                oracle.shard_pool_a_cols(rpool, w, r), None)
        parts = [None] * w
        dist.all_gather_object(parts, part)
        hr = tp.reduce_rank_partials(torch.from_numpy(part.copy())).numpy()
        res["reduce_is_rank_sum"] = bool(np.array_equal(hr, oracle.rank_sum(np.stack(parts))))
        wsl = rc.widths[0] // w
        out_r = rc.out0.copy()
        oracle.expand(out_r, hr, rc.seq_slot, oracle.shard_pool_b_rows(rpool, w, r),
                      rpool.scale_table, offset_start=r * wsl)
        row_shards = [None] * w
        dist.all_gather_object(row_shards, out_r)

        if rank == 0:
            whole = case.out0.copy()
            oracle.delta(whole, case.x, case.seq_slot, pool)
            res["column_equal"] = all(bool(np.array_equal(o, whole[:, c])) for c, o in col_shards)
            res["column_cover"] = sorted(np.concatenate([c for c, _ in col_shards]).tolist()) == \
                list(range(case.ld_out))
            rwhole = rc.out0.copy()
            oracle.delta(rwhole, rc.x, rc.seq_slot, rpool)
            ok_in, ok_out = True, True
            for p, o in enumerate(row_shards):
                inside = np.zeros(rc.ld_out, dtype=bool)
                inside[p * wsl:(p + 1) * wsl] = True
                ok_out &= bool(np.array_equal(o[:, ~inside], rc.out0[:, ~inside]))
                g = (o[:, inside].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
                f = (rwhole[:, inside].astype(np.uint32) << 16).view(np.float32).astype(
                    np.float64)
                ok_in &= bool(np.all(np.abs(g - f) <= 1e-2 + 1e-2 * np.abs(f)))
            res["row_slices_close"] = ok_in
            res["row_outside_untouched"] = ok_out
        dist.destroy_process_group()
        q.put((rank, res, None))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, None, repr(e)))


def test_two_rank_tensor_parallel_forms(oracle):
    """Column parallel: every rank's output columns equal the unsharded delta's bit
    for bit, the gather is rank-major, the columns cover the output once.  Row
    parallel: the all-reduce of the partials is their rank-order sum, each rank's
    slice is within the parity tolerance of the unsharded delta, and the rest of
    its partial-sum output is untouched."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_tp_worker, args=(r, WORLD, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    results = {}
    try:
        for _ in range(WORLD):
            rank, res, err = q.get(timeout=240)
            assert err is None, f"rank {rank}: {err}"
            results[rank] = res
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    for rank in range(WORLD):
        assert results[rank]["gather_rank_major"]
        assert results[rank]["reduce_is_rank_sum"]
    r0 = results[0]
    assert r0["column_equal"] and r0["column_cover"]
    assert r0["row_slices_close"] and r0["row_outside_untouched"]
