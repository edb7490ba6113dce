"""Write the oracle's golden fixtures (calls only oracle/ and the seeded inputs).

The pages print no worked numeric example, so these fixtures are not page
values: they lock the oracle's output on the seeded tiny workloads, so that a
later change to the oracle's arithmetic shows up as a failing test and must be
justified by a passage of the pages.

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from lora_delta_gb300 import inputs  # noqa: E402


def tiny_delta():
    c = inputs.tiny_case()
    pool = oracle.build_pool(c.adapters, c.k_in, c.widths, c.max_loras, c.max_rank)
    out = c.out0.copy()
    err = oracle.delta(out, c.x, c.seq_slot, pool)
    return c, out, err


def tiny_moe(shared):
    c = inputs.moe_case(shared_a=shared, T=6, top_k=2, E=4, H=32, I=8, rank=4, L=2)
    out, err = oracle.moe_fc1(c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids, c.I, c.rank,
                              c.scale, shared, c.L)
    return c, out, err


def tiny_w13():
    c = inputs.moe_case(shared_a=False, T=6, top_k=2, E=4, H=32, I=8, rank=4, L=2)
    y0 = inputs.moe_y0(c.seed, (c.T, c.top_k, 2 * c.I))
    emap = np.array([1, -1, 0, 3, 2, -1], dtype=np.int32)  # 6 global experts, 4 local
    topk = np.minimum(c.topk_ids * 2, 5).astype(np.int32)  # global ids
    y, err = oracle.moe_w13(y0, c.x, c.A_banks, c.B_banks, topk, c.lora_ids, c.I, c.rank,
                            c.scale, False, c.L, expert_map=emap)
    return c, y, err


def tiny_w2():
    c = inputs.moe_w2_case(T=6, top_k=2, E=4, H=16, I=24, rank=8, L=2)
    y, err = oracle.moe_w2(c.y0, c.x, c.A_banks, c.B_banks, c.topk_ids, c.lora_ids, c.rank,
                           c.scale, c.L, topk_weights=c.topk_weights)
    return c, y, err


def write(path, header, arr):
    with open(path, "w") as f:
        for line in header:
            f.write(f"# {line}\n")
        f.write(f"# shape {' '.join(str(d) for d in arr.shape)}\n")
        flat = arr.reshape(arr.shape[0], -1)
        for row in flat:
            f.write(" ".join(f"{int(v):04x}" for v in row) + "\n")


def main():
    c, out, err = tiny_delta()
    write(os.path.join(HERE, "tiny_delta_oracle.txt"), [
        "oracle output (bf16 bits, hex) of the tiny routed delta: n=8, k_in=256, one",
        "256-wide slice, 4 slots (ranks 8,16,4,16 padded to 16), alpha 16, seed 1234.",
        "Semantics: 'Module lora_delta', apply_lora_bgmv; 'punica_base.py', add_lora_linear.",
        f"seq_slot {' '.join(str(int(s)) for s in c.seq_slot)}; error word {err}",
        "Written by tests/golden/make_golden.py (oracle only).",
    ], out)
    for shared in (False, True):
        c, out, err = tiny_moe(shared)
        mode = "shared" if shared else "regular"
        write(os.path.join(HERE, f"tiny_moe_{mode}_oracle.txt"), [
            f"oracle output (bf16 bits, hex) of a tiny MoE FC1 delta, {mode} mode:",
            "T=6, top_k=2, E=4, H=32, I=8, rank=4, L=2, scale 2, seed 1238.",
            "Semantics: 'flashinfer.fused_moe.bgmv_moe_gemm1_lora_delta'.",
            f"lora_ids {' '.join(str(int(v)) for v in c.lora_ids)}; error word {err}",
            "Written by tests/golden/make_golden.py (oracle only).",
        ], out)
    c, y, err = tiny_w13()
    write(os.path.join(HERE, "tiny_moe_w13_oracle.txt"), [
        "oracle output (bf16 bits, hex) of a tiny in-place w13 delta with an expert map",
        "(6 global experts, 4 local): T=6, top_k=2, H=32, I=8, rank=4, L=2, scale 2, seed 1238.",
        "Semantics: 'punica_base.py', add_lora_w13 (the delta of",
        "'flashinfer.fused_moe.bgmv_moe_gemm1_lora_delta', added in place).",
        f"error word {err}",
        "Written by tests/golden/make_golden.py (oracle only).",
    ], y)
    c, y, err = tiny_w2()
    write(os.path.join(HERE, "tiny_moe_w2_oracle.txt"), [
        "oracle output (bf16 bits, hex) of a tiny in-place w2 delta with routing weights:",
        "T=6, top_k=2, E=4, H=16, I=24, rank=8, L=2, scale 2, seed 1240.",
        "Semantics: 'punica_base.py', add_lora_w2.",
        f"error word {err}",
        "Written by tests/golden/make_golden.py (oracle only).",
    ], y)


if __name__ == "__main__":
    main()
