"""Tensor-parallel sharded LoRA ("vllm.lora.fully_sharded_layers", the S-LoRA
layers): one rank's step of the two sharded forms.

Both run the shrink and the expand on this library's kernels, with one
collective on the fp32 h buffer in between (torch.distributed: NCCL between
GPUs, gloo on the CPU):

* column parallel (``_mcp_apply``; ColumnParallelLinearWithShardedLoRA and
  MergedColumnParallelLinearWithShardedLoRA): x is whole on every rank; A is
  sliced along the rank (rank p holds rows p*R/tp .. of every adapter's A),
  B along the output (rank p holds the B rows of its output columns).  Each
  rank shrinks its R/tp rows (scale 1) into h [S, n, R/tp]; the buffers are
  all-gathered rank-major into [tp, S, n, R/tp]; each rank expands its output
  columns with the whole h.  Every rank ends with the unsharded h exactly, so
  its columns equal the unsharded delta's bit for bit.
* row parallel (RowParallelLinearWithShardedLoRA ``apply``): x and A are
  sliced along the input (rank p holds k columns p*k_in/tp ..); each rank's
  shrink gives a partial h [S, n, R] over its k columns; the partials are
  all-reduced (summed); rank p expands with the B rows of its slice of the
  output into that slice of its partial-sum output (offset_start = p * the
  slice width), which the caller's own all-reduce of the layer output then
  completes, as the page notes.

The collective step is the only exchange on the path; there is no
multicast.  Every call of this build has one GPU, so the NCCL form is
unmeasured on hardware: the GPU kernels of both forms are tested with the ranks
emulated on one GPU, and the collective steps on CPU ranks over gloo.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import LoraPool, lora_expand, lora_expand_gathered, lora_shrink


def _shard_pool(pool: LoraPool, A, B, R: int, k_in: int, widths) -> LoraPool:
    """A pool over the given (already sliced, contiguous) A / B tensors, with the
    table entries of ``pool`` that are 0 kept 0 and the others pointed at the
    slices; the scale table is shared."""
    sp = LoraPool.__new__(LoraPool)
    sp.k_in, sp.widths, sp.max_loras, sp.R = int(k_in), tuple(widths), pool.max_loras, int(R)
    sp.device = pool.device
    sp.A, sp.B = A, B
    L = pool.max_loras
    at, bt = pool.a_table.cpu().tolist(), pool.b_table.cpu().tolist()
    sp._a_host = [A[j][s].data_ptr() if at[j * L + s] else 0 for j in range(pool.S)
                  for s in range(L)]
    sp._b_host = [B[j][s].data_ptr() if bt[j * L + s] else 0 for j in range(pool.S)
                  for s in range(L)]
    sp.scale_table = pool.scale_table
    sp.a_table = torch.tensor(sp._a_host, dtype=torch.int64, device=pool.device)
    sp.b_table = torch.tensor(sp._b_host, dtype=torch.int64, device=pool.device)
    return sp


def shard_pool_a_rows(pool: LoraPool, tp: int, p: int) -> LoraPool:
    """Rank p's pool of the column-parallel shrink: rows p*R/tp .. (p+1)*R/tp - 1
    of every adapter's padded A (set-up; copies the slices)."""
    if pool.R % tp or (pool.R // tp) % 8:
        raise ValueError("R / tp must be a multiple of 8")
    Rs = pool.R // tp
    A = [a[:, p * Rs:(p + 1) * Rs, :].contiguous() for a in pool.A]
    return _shard_pool(pool, A, pool.B, Rs, pool.k_in, pool.widths)


def shard_pool_a_cols(pool: LoraPool, tp: int, p: int) -> LoraPool:
    """Rank p's pool of the row-parallel shrink: input columns p*k_in/tp .. of
    every adapter's A (set-up; copies the slices)."""
    if pool.k_in % tp or (pool.k_in // tp) % 8:
        raise ValueError("k_in / tp must be a multiple of 8")
    ks = pool.k_in // tp
    A = [a[:, :, p * ks:(p + 1) * ks].contiguous() for a in pool.A]
    return _shard_pool(pool, A, pool.B, pool.R, ks, pool.widths)


def shard_pool_b_rows(pool: LoraPool, tp: int, p: int) -> LoraPool:
    """Rank p's pool of the expand of either form: output columns p*w_j/tp .. of
    every slice (rows of B), the whole rank (set-up; copies the slices)."""
    if any(w % tp or (w // tp) % 8 for w in pool.widths):
        raise ValueError("every width / tp must be a multiple of 8")
    ws = [w // tp for w in pool.widths]
    B = [b[:, p * w:(p + 1) * w, :].contiguous() for b, w in zip(pool.B, ws)]
    return _shard_pool(pool, pool.A, B, pool.R, pool.k_in, ws)


def gather_rank_shards(h_shard: torch.Tensor, group=None) -> torch.Tensor:
    """The all-gather of the rank shards of h ([S, n, R/tp] each) into
    [tp, S, n, R/tp], rank-major (rank p's shard at index p)."""
    tp = dist.get_world_size(group)
    h_shard = h_shard.contiguous()
    S = h_shard.shape[0]
    # (the concatenation along dim 0, which every backend takes, is the
    # rank-major stack in memory)
    out = torch.empty((tp * S,) + tuple(h_shard.shape[1:]), dtype=h_shard.dtype,
                      device=h_shard.device)
    dist.all_gather_into_tensor(out, h_shard, group=group)
    return out.view((tp,) + tuple(h_shard.shape))


def reduce_rank_partials(h: torch.Tensor, group=None) -> torch.Tensor:
    """The all-reduce (sum) of the rank partials of h, in place."""
    dist.all_reduce(h, op=dist.ReduceOp.SUM, group=group)
    return h


def column_parallel_delta(out, x, seq_slot, pool_a: LoraPool, pool_b: LoraPool, group=None,
                          add_inputs: bool = True, workspace=None, err=None, stream=None):
    """This rank's step of the column-parallel form: ``out`` [n, ld_out] holds the
    rank's output columns (pool_b's widths, offset 0); ``pool_a`` the rank's rows of
    every A (R / tp of them), ``pool_b`` the B rows of the rank's columns with the
    whole rank R.  Returns the gathered h [tp, S, n, R / tp]."""
    n = x.shape[0]
    h_shard = torch.zeros(pool_a.S, n, pool_a.R, dtype=torch.float32, device=x.device)
    lora_shrink(h_shard, x, seq_slot, pool_a, scale_table=None, workspace=workspace, err=err,
                stream=stream)
    h_all = gather_rank_shards(h_shard, group)
    lora_expand_gathered(out, h_all, seq_slot, pool_b, scale_table=pool_b.scale_table,
                         add_inputs=add_inputs, workspace=workspace, err=err, stream=stream)
    return h_all


def row_parallel_delta(out, x_shard, seq_slot, pool_a: LoraPool, pool_b: LoraPool, group=None,
                       add_inputs: bool = True, workspace=None, err=None, stream=None):
    """This rank's step of the row-parallel form: ``x_shard`` [n, k_in / tp] the
    rank's input columns, ``pool_a`` A on the same columns (whole rank R),
    ``pool_b`` the B rows of the rank's slice of the output; ``out`` [n, ld_out]
    the rank's partial-sum output, updated in its slice only.  Returns the
    reduced h [S, n, R]."""
    if pool_b.S != 1:
        raise ValueError("the row-parallel form has one output slice")
    rank = dist.get_rank(group)
    n = x_shard.shape[0]
    h = torch.zeros(pool_a.S, n, pool_a.R, dtype=torch.float32, device=x_shard.device)
    lora_shrink(h, x_shard, seq_slot, pool_a, scale_table=None, workspace=workspace, err=err,
                stream=stream)
    reduce_rank_partials(h, group)
    lora_expand(out, h, seq_slot, pool_b, scale_table=pool_b.scale_table,
                offset_start=rank * pool_b.widths[0], add_inputs=add_inputs,
                workspace=workspace, err=err, stream=stream)
    return h
