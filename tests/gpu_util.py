"""Helpers of the GPU parity tests: run a case through the C ABI and through the
oracle, and compare with the stated tolerance."""
from __future__ import annotations

import numpy as np

# Tolerance on bf16 outputs: max |err| <= ATOL + RTOL * |ref| (the stated bar).
ATOL = 1e-2
RTOL = 1e-2


def f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)


def assert_close(got_bits: np.ndarray, ref_bits: np.ndarray, what: str = ""):
    g, r = f64(got_bits), f64(ref_bits)
    assert g.shape == r.shape
    bad = ~(np.abs(g - r) <= ATOL + RTOL * np.abs(r))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first {idx.tolist()}: "
            f"got {g[bad][:5].tolist()} ref {r[bad][:5].tolist()}")


def oracle_delta(oracle, case, rows=None, R=None, add_inputs=True):
    """Oracle result of the routed delta on the case (optionally on a subset of rows;
    rows are independent, so a subset is computed on its own)."""
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, case.max_loras,
                             R or case.max_rank, case.use_rslora)
    if rows is None:
        out = case.out0.copy()
        err = oracle.delta(out, case.x, case.seq_slot, pool, offset_start=case.offset_start,
                           add_inputs=add_inputs)
        return out, err
    rows = np.asarray(rows)
    out = np.ascontiguousarray(case.out0[rows])
    err = oracle.delta(out, np.ascontiguousarray(case.x[rows]),
                       np.ascontiguousarray(case.seq_slot[rows]), pool,
                       offset_start=case.offset_start, add_inputs=add_inputs)
    return out, err
