"""Move the seeded synthetic workloads of ``inputs`` onto the GPU.

Pure marshalling: bf16 bit patterns become torch.bfloat16 device tensors, the
PEFT adapters are packed by the library's own ``lora_pool_pack`` kernel into a
``LoraPool``, and the MoE banks get their int64 pointer tables.  No LoRA
arithmetic happens here.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import LoraPool
from .inputs import LinearCase, MoeCase


def bf16(a: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def pool_from_case(case: LinearCase, device="cuda", R: int | None = None) -> LoraPool:
    pool = LoraPool(case.k_in, case.widths, case.max_loras, R or case.max_rank, device=device)
    for s, ad in enumerate(case.adapters):
        if ad is None:
            continue
        a_r = [bf16(a, device) for a in ad.A]
        b_r = [bf16(b, device) for b in ad.B]
        pool.pack(s, a_r, b_r, ad.alpha, ad.rank, case.use_rslora, ad.adapted)
    torch.cuda.synchronize(device)
    return pool


@dataclass
class DeviceLinear:
    x: torch.Tensor
    out0: torch.Tensor
    seq_slot: torch.Tensor
    pool: LoraPool


def linear_to_device(case: LinearCase, device="cuda", R: int | None = None) -> DeviceLinear:
    return DeviceLinear(x=bf16(case.x, device), out0=bf16(case.out0, device),
                        seq_slot=torch.from_numpy(case.seq_slot).to(device),
                        pool=pool_from_case(case, device, R))


@dataclass
class DeviceMoe:
    x: torch.Tensor
    topk_ids: torch.Tensor
    lora_ids: torch.Tensor
    A_banks: list
    B_banks: list
    w_ptr_a: torch.Tensor
    w_ptr_b: torch.Tensor
    stride_a: int
    stride_b: int


def moe_to_device(case: MoeCase, device="cuda") -> DeviceMoe:
    A = [bf16(a, device) for a in case.A_banks]
    B = [bf16(b, device) for b in case.B_banks]
    E = case.E
    wa = torch.tensor([bank[e].data_ptr() for bank in A for e in range(E)], dtype=torch.int64,
                      device=device)
    wb = torch.tensor([bank[e].data_ptr() for bank in B for e in range(E)], dtype=torch.int64,
                      device=device)
    return DeviceMoe(x=bf16(case.x, device), topk_ids=torch.from_numpy(case.topk_ids).to(device),
                     lora_ids=torch.from_numpy(case.lora_ids).to(device), A_banks=A, B_banks=B,
                     w_ptr_a=wa, w_ptr_b=wb, stride_a=int(np.prod(case.A_banks[0].shape[2:])),
                     stride_b=int(np.prod(case.B_banks[0].shape[2:])))
