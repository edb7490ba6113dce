// Data-movement floor of the fused small-segment kernel: the same grid,
// cluster size, shared-memory plan and programmatic dependent launch as
// bgmv_fused_kernel, the same bytes (each routed key's A share and B rows of
// every CTA, the key's x rows and out rows, out written back), and no
// arithmetic: the prologue streams the weights before the dependency wait,
// the key's rows are found, x and out rows are staged, the cluster meets once
// (the exchange's barrier) and the out rows go back unchanged.  Timing it
// next to lora_delta_fused says how much of a decode step is fixed cost of
// moving these bytes in this shape.  None of the pages has this kernel.
#pragma once

#include "bgmv_fused.cuh"

namespace lora {

__global__ void __launch_bounds__(kThreads, 3)
    bgmv_floor_kernel(const DeltaArgs a, const LinearTables tb) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ SlotView v;
  __shared__ int nrows_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int key = (int)cluster_index_x();
  const uint32_t crank = cluster_rank();
  const FusedPlan pl = fused_plan(a);
  int* prow = reinterpret_cast<int*>(smem + 64);
  int* rows_s = reinterpret_cast<int*>(smem + pl.rows_off);
  __nv_bfloat16* As = reinterpret_cast<__nv_bfloat16*>(smem + pl.As_off);
  __nv_bfloat16* Xs = reinterpret_cast<__nv_bfloat16*>(smem + pl.Xs_off);
  __nv_bfloat16* Bs = reinterpret_cast<__nv_bfloat16*>(smem + pl.Bs_off);
  __nv_bfloat16* Os = reinterpret_cast<__nv_bfloat16*>(smem + pl.Os_off);
  if (tid == 0) {
    uint32_t bad = 0;
    tb.resolve(key, a.sl.S, kModeFused, v, bad);
  }
  __syncthreads();
  const int SRa = v.nact * a.R;
  const int k_lo = min(a.k_in, (int)crank * a.kc);
  const int kw = min(a.k_in, k_lo + a.kc) - k_lo;
  const int cb = min(a.sl.n_cols, (int)crank * a.cpc);
  const int ce = min(a.sl.n_cols, cb + a.cpc);
  if (v.nact > 0) {
    if (kw > 0) copy_a_rows(a, v, SRa, k_lo, kw, As, pl.stride, tid);
    copy_b_rows(a, v, cb, ce, Bs, tid);
  }
  cp_async_commit();
  cudaTriggerProgrammaticLaunchCompletion();
  cudaGridDependencySynchronize();
  if (v.nact == 0) return;  // (uniform over the cluster)
  if (warp == 0) {
    int total = 0;
    for (int base = 0; base < a.n; base += 32 * 8) {
      int sl[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * 32 + lane;
        sl[u] = i < a.n ? a.seq_slot[i] : -1;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const bool hit = sl[u] == key;
        const unsigned m = __ballot_sync(0xffffffffu, hit);
        if (hit) rows_s[total + __popc(m & ((1u << lane) - 1u))] = base + u * 32 + lane;
        total += __popc(m);
      }
    }
    if (lane == 0) nrows_s = total;
  }
  __syncthreads();
  const int nrows = nrows_s;
  if (nrows == 0) {
    cp_async_wait<0>();
    return;
  }
  for (int p0 = 0; p0 < nrows; p0 += kFusedRows) {
    const int nr = min(kFusedRows, nrows - p0);
    if (p0 > 0) __syncthreads();
    if (tid < nr) prow[tid] = rows_s[p0 + tid];
    __syncthreads();
    if (kw > 0) copy_x_rows(a, tb, prow, nr, k_lo, kw, Xs, pl.stride, tid);
    copy_out_rows(a, tb, v, prow, nr, cb, ce, Os, pl.o_stride, tid);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    cluster_arrive_release_smem();  // the exchange's meeting point
    cluster_wait();
    for (int r = warp; r < nr; r += kWarps) {
      __nv_bfloat16* orow = a.out + (int64_t)prow[r] * a.ld_out;
      const __nv_bfloat16* srow = Os + (size_t)r * pl.o_stride - cb;
      for (int j = 0; j < a.sl.S; ++j) {
        const int c0 = max(cb, a.rel[j]), c1 = min(ce, a.rel[j + 1]);
        if (c1 <= c0 || v.ja[j] < 0) continue;
        __nv_bfloat16* dst = orow + a.sl.off[j] - a.rel[j];
        for (int c = c0 + lane * 8; c < c1; c += 256)
          *reinterpret_cast<uint4*>(dst + c) = *reinterpret_cast<const uint4*>(srow + c);
      }
    }
  }
}

}  // namespace lora
