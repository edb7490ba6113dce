// The routed delta for small row groups when a CTA's whole share of a key's A
// fits in shared memory at once (decode: "Module lora_delta", apply_lora_bgmv;
// "punica_base.py", add_lora_linear; the routed-MoE forms on their keys).
//
// One thread-block cluster of CS CTAs per key, as in the general cluster
// kernel, with the per-pass work cut to few dependent steps:
//   * prologue, before the grid dependency wait: the key's table entries; the
//     CTA's A share (its 1/CS of k_in, every active (slice, rank) row) and the
//     B rows of its 1/CS of the output columns start streaming into shared
//     memory (adapter weights are never written by the preceding kernel);
//   * the key's rows (own ballot scan, or the routing kernel's clusters), in
//     passes of 8: x rows of the CTA's k share and out segments of its columns
//     by cp.async, in separate groups, so the shrink waits for x only;
//   * shrink on mma.sync m16n8k16 (pairs x rows x k): warp w owns the 16-pair
//     tiles w and w + 8 over the CTA's whole k share, in two accumulator
//     chains on alternate k-steps, and writes its sums straight to the
//     buffer the cluster reads (nothing to combine inside the CTA);
//   * the CS partials meet through distributed shared memory: each CTA reads
//     the CS partials of every entry of the pass from its peers in one round
//     (all loads in flight together), sums them in a fixed order, and holds
//     the whole fp32 h;
//   * expand + fold on mma.sync with M = 16 output columns (B rows by
//     ldmatrix) and N = 8 rows (h as a bf16 (hi, lo) pair, so the rank
//     contraction keeps ~fp32 accuracy); each product is folded into the
//     staged out rows in shared memory, RN_bf16(out + scale * w * d), and the
//     rows go back to global memory as coalesced 16-byte stores.
#pragma once

#include "bgmv.cuh"
#include "common.cuh"

namespace lora {

constexpr int kFusedRows = 8;  // rows of one pass: one 8-row MMA tile

// Shared-memory plan (bytes) of bgmv_fused_kernel, identical on host and device.
struct FusedPlan {
  int rows_off, As_off, Xs_off, Bs_off, Os_off, Rx_off, H_off, total;
  int stride;    // elements per staged A / x row: the k share + 8 (ldmatrix conflict-free)
  int o_stride;  // elements per staged out row: the CTA's columns + 8
  int sr16;      // S * R rounded up to 16
};
__host__ __device__ inline FusedPlan fused_plan(const DeltaArgs& a) {
  FusedPlan p;
  p.sr16 = (a.sr_max + 15) / 16 * 16;
  p.stride = a.kc + 8;
  p.o_stride = a.cpc + 8;
  int o = 128;  // the pass's row ids (8 ints) at offset 64
  p.rows_off = o;
  o += ((a.row_cap * 4 + 127) / 128) * 128;
  p.As_off = o;
  o += p.sr16 * p.stride * 2;
  p.Xs_off = o;
  o += kFusedRows * p.stride * 2;
  o = (o + 127) / 128 * 128;
  p.Bs_off = o;  // the CTA's B rows [cpc][R], + 16 rows of slack (read by a half tile)
  o += (a.cpc + 16) * a.R * 2;
  o = (o + 127) / 128 * 128;
  p.Os_off = o;
  o += kFusedRows * p.o_stride * 2;
  o = (o + 127) / 128 * 128;
  p.Rx_off = o;  // this CTA's partial h, read by the cluster: [8 rows][sr16]
  o += kFusedRows * p.sr16 * 4;
  p.H_off = o;   // the pass's h [8 rows][sr16]
  o += kFusedRows * p.sr16 * 4;
  p.total = o;
  return p;
}

// Shapes the kernel takes: one k stage per CTA (kst == kc), R a multiple of
// 16 up to 64, S * R up to 256 (at most two 16-pair tiles per warp).
inline bool fused_kernel_fits(const DeltaArgs& a) {
  return a.nbuf == 1 && a.kst == a.kc && a.R % 16 == 0 && a.R <= 64 && a.sr_max <= 256;
}

template <int RMAX, class Tables>
__global__ void __launch_bounds__(kThreads, 3)
    bgmv_fused_kernel(const DeltaArgs a, const Tables tb) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ SlotView v;
  __shared__ int nrows_s, rows_base_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3;  // MMA fragment coordinates
  const int key = (int)cluster_index_x();
  const uint32_t crank = cluster_rank();
  const int ncta = a.cs;

  const FusedPlan pl = fused_plan(a);
  int* prow = reinterpret_cast<int*>(smem + 64);
  int* rows_s = reinterpret_cast<int*>(smem + pl.rows_off);
  __nv_bfloat16* As = reinterpret_cast<__nv_bfloat16*>(smem + pl.As_off);
  __nv_bfloat16* Xs = reinterpret_cast<__nv_bfloat16*>(smem + pl.Xs_off);
  __nv_bfloat16* Bs = reinterpret_cast<__nv_bfloat16*>(smem + pl.Bs_off);
  __nv_bfloat16* Os = reinterpret_cast<__nv_bfloat16*>(smem + pl.Os_off);
  float* Rx = reinterpret_cast<float*>(smem + pl.Rx_off);
  float* H = reinterpret_cast<float*>(smem + pl.H_off);
  const int stride = pl.stride, SR16 = pl.sr16;

  // ---- prologue: independent of the preceding kernel's outputs ----------
  if (tid == 0) {
    uint32_t bad = 0;
    tb.resolve(key, a.sl.S, kModeFused, v, bad);
    if (bad && crank == 0) set_error(a.err, bad);
  }
  __syncthreads();
  const int R = a.R;
  const int SRa = v.nact * R;
  const int k_lo = min(a.k_in, (int)crank * a.kc);
  const int kw = min(a.k_in, k_lo + a.kc) - k_lo;  // this CTA's k share (may be 0)
  const int cb = min(a.sl.n_cols, (int)crank * a.cpc);
  const int ce = min(a.sl.n_cols, cb + a.cpc);
  auto weight_copies = [&]() {
    if (kw > 0) copy_a_rows(a, v, SRa, k_lo, kw, As, stride, tid);
    copy_b_rows(a, v, cb, ce, Bs, tid);
  };
  const bool early = a.early && v.nact > 0;
  if (early) weight_copies();
  cp_async_commit();  // group 0: the weights (empty when not early)
  cudaTriggerProgrammaticLaunchCompletion();
  cudaGridDependencySynchronize();
  // Without a routing pass, CTA 0 of key 0 also checks every slot for
  // LORA_DEV_ERR_SLOT, so it scans even when key 0 adapts nothing.
  const bool slot_check = !a.perm && key == 0 && crank == 0;
  if (v.nact == 0 && !slot_check) return;  // the same in every CTA of the cluster

  // ---- the key's rows, in ascending row order (warp 0) -----------------
  if (warp == 0) {
    int total = 0, s0 = 0;
    if (a.perm) {
      s0 = a.seg_start[key];
      total = a.seg_start[key + 1] - s0;
    } else {
      bool bad_slot = false;
      for (int base = 0; base < a.n; base += 32 * 8) {
        int sl[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {  // independent loads, one round trip
          const int i = base + u * 32 + lane;
          sl[u] = i < a.n ? a.seq_slot[i] : -1;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const bool hit = sl[u] == key;
          bad_slot |= sl[u] >= a.n_keys;
          const unsigned m = __ballot_sync(0xffffffffu, hit);
          if (hit) rows_s[total + __popc(m & ((1u << lane) - 1u))] = base + u * 32 + lane;
          total += __popc(m);
        }
      }
      if (__any_sync(0xffffffffu, bad_slot) && key == 0 && crank == 0 && lane == 0)
        set_error(a.err, LORA_DEV_ERR_SLOT);
    }
    if (lane == 0) {
      nrows_s = total;
      rows_base_s = s0;
    }
  }
  __syncthreads();
  if (v.nact == 0) return;
  const int nrows = nrows_s;
  const int* rows = a.perm ? a.perm + rows_base_s : rows_s;
  if (nrows == 0 || nrows < a.min_rows || nrows >= a.max_rows) {  // uniform
    cp_async_wait<0>();  // no copy may land in a CTA that has exited
    return;
  }
  if (!early) weight_copies();
  cp_async_commit();  // group 1: the weights when not early (else empty)
  // the k tail: a half k-step reads 8 columns past kw, never copied: zeros
  if (kw & 15)
    for (int i = tid; i < SR16; i += kThreads)
      *reinterpret_cast<uint4*>(As + (size_t)i * stride + kw) = make_uint4(0, 0, 0, 0);

  const int mt = (SRa + 15) / 16;  // 16-pair tiles of the shrink (<= 16: two per warp)
  const int ksteps = (kw + 15) / 16;
  const int ng = (SRa >> 2);  // 4-pair groups per row (SRa is a multiple of 16)

  for (int p0 = 0; p0 < nrows; p0 += kFusedRows) {
    const int nr = min(kFusedRows, nrows - p0);
    if (p0 > 0) __syncthreads();  // the previous pass is done with prow, Xs and Os
    if (tid < nr) prow[tid] = rows[p0 + tid];
    __syncthreads();
    if (kw > 0) copy_x_rows(a, tb, prow, nr, k_lo, kw, Xs, stride, tid);
    cp_async_commit();  // group: x rows
    if (a.add_inputs) copy_out_rows(a, tb, v, prow, nr, cb, ce, Os, pl.o_stride, tid);
    cp_async_commit();  // group: out segments (waited for before the expand)
    if (kw & 15)
      for (int i = tid; i < kFusedRows; i += kThreads)
        *reinterpret_cast<uint4*>(Xs + (size_t)i * stride + kw) = make_uint4(0, 0, 0, 0);
    cp_async_wait<1>();  // weights and x rows landed (the out segments may still fly)
    __syncthreads();

    // ---- shrink: warp w owns pair tiles w and w + 8 over the whole k share,
    // each in two accumulator chains on alternate k-steps (no partials to
    // combine inside the CTA); the sums are this CTA's partial of h, written
    // straight to Rx[row][pair] for the cluster ------------------------------
    if (p0 > 0) cluster_wait();  // the previous pass's readers are done with Rx
    {
      // x fragments (rows 0..7 of the pass, k halves) by ldmatrix.x2 (lanes
      // 0-15); A fragments (16 pairs) by ldmatrix.x4
      const uint32_t xaddr = smem_addr(Xs + (size_t)(lane & 7) * stride + ((lane >> 3) & 1) * 8);
      const uint32_t arow = (uint32_t)((((lane >> 3) & 1) << 3) + (lane & 7));
      const uint32_t acol = (uint32_t)((lane >> 4) << 3);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int m = warp + i * kWarps;
        if (m >= mt) break;  // (uniform)
        const uint32_t aaddr = smem_addr(As + (size_t)(m * 16 + arow) * stride + acol);
        float acc[2][4];  // [chain][fragment]
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[c][e] = 0.0f;
        int ks = 0;
        for (; ks + 1 < ksteps; ks += 2) {
          uint32_t b0, b1, c0, c1, a0, a1, a2, a3, d0, d1, d2, d3;
          ldsm_x2(xaddr + ks * 32, b0, b1);
          ldsm_x4(aaddr + ks * 32, a0, a1, a2, a3);
          ldsm_x2(xaddr + (ks + 1) * 32, c0, c1);
          ldsm_x4(aaddr + (ks + 1) * 32, d0, d1, d2, d3);
          mma_16816(acc[0], a0, a1, a2, a3, b0, b1);
          mma_16816(acc[1], d0, d1, d2, d3, c0, c1);
        }
        if (ks < ksteps) {
          uint32_t b0, b1, a0, a1, a2, a3;
          ldsm_x2(xaddr + ks * 32, b0, b1);
          ldsm_x4(aaddr + ks * 32, a0, a1, a2, a3);
          mma_16816(acc[0], a0, a1, a2, a3, b0, b1);
        }
        // C[pair m*16 + gq (+8)][row 2tq (+1)] -> Rx[row][pair]
        float* rx = Rx + (2 * tq) * SR16 + m * 16 + gq;
        rx[0] = acc[0][0] + acc[1][0];
        rx[SR16] = acc[0][1] + acc[1][1];
        rx[8] = acc[0][2] + acc[1][2];
        rx[SR16 + 8] = acc[0][3] + acc[1][3];
      }
    }
    __syncthreads();  // (the whole CTA's partial is in Rx before the release)
    cluster_arrive_release_smem();  // partials in place
    cluster_wait();
    // ---- the cluster's partials: lg lanes per 4-entry group (4, or 2 when
    // the pass's groups would not fit one round of 4), lane qq reading peers
    // qq, qq + lg, ... (all in flight together), then xor-shuffles add the
    // lanes: the same summation order in every CTA ------------------------
    {
      const uint32_t rx_addr = smem_addr(Rx);
      const int ngrp = nr * ng;
      const int lg = ngrp * 4 <= kThreads ? 4 : 2;  // (uniform)
      const int gpr = kThreads / lg, qq = lane & (lg - 1);
      for (int gb0 = 0; gb0 < ngrp; gb0 += gpr) {  // (uniform rounds)
        const int gb = gb0 + tid / lg;
        const bool valid = gb < ngrp;  // (the warp's lanes stay together)
        const int e = valid ? gb : 0;
        const int r = e / ng, p = (e - r * ng) * 4;
        const uint32_t addr = rx_addr + 4u * (uint32_t)(r * SR16 + p);
        float4 part[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = qq + lg * u;
          part[u] = (valid && c < ncta) ? dsmem_ld_f32x4(dsmem_map(addr, (uint32_t)c))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float4 hv = part[0];
#pragma unroll
        for (int u = 1; u < 8; ++u) {
          hv.x += part[u].x;
          hv.y += part[u].y;
          hv.z += part[u].z;
          hv.w += part[u].w;
        }
        for (int off = 1; off < lg; off <<= 1) {
          hv.x += __shfl_xor_sync(0xffffffffu, hv.x, off);
          hv.y += __shfl_xor_sync(0xffffffffu, hv.y, off);
          hv.z += __shfl_xor_sync(0xffffffffu, hv.z, off);
          hv.w += __shfl_xor_sync(0xffffffffu, hv.w, off);
        }
        if (valid && qq == 0) *reinterpret_cast<float4*>(H + r * SR16 + p) = hv;
      }
    }
    cluster_arrive_relaxed();  // done reading the peers' Rx (waited on later)
    cp_async_wait<0>();        // the out segments landed
    __syncthreads();           // H complete, Os complete

    // ---- expand + fold: tiles of 16 columns x 8 rows ----------------------
    {
      constexpr int KS = RMAX / 16;
      const int ks_n = R / 16;
      // this thread's rows (2tq, 2tq + 1) and their scales
      float sc[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r = 2 * tq + e;
        sc[e] = r < nr ? v.scale * tb.row_weight(prow[r]) : 0.0f;
      }
      // tiles of every active slice's part of [cb, ce), 16 columns each (the
      // last of a slice may be 8 wide), dealt to the warps in turn
      int tile_base = 0;
      for (int j = 0; j < a.sl.S; ++j) {
        const int ja = v.ja[j];
        const int c0 = max(cb, a.rel[j]), c1 = min(ce, a.rel[j + 1]);
        if (ja < 0 || c1 <= c0) continue;
        const int ntl = (c1 - c0 + 15) / 16;
        const int t_first = ((warp - tile_base) % kWarps + kWarps) % kWarps;
        tile_base += ntl;
        if (t_first >= ntl) continue;
        // B operand: h of this slice, row gq of the pass, as bf16 (hi, lo)
        uint32_t bhi[KS][2], blo[KS][2];
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const bool ok = kk < ks_n && gq < nr;
          const float* hp = H + gq * SR16 + ja * R + kk * 16 + 2 * tq;
          split_bf16x2(ok ? hp[0] : 0.f, ok ? hp[1] : 0.f, bhi[kk][0], blo[kk][0]);
          split_bf16x2(ok ? hp[8] : 0.f, ok ? hp[9] : 0.f, bhi[kk][1], blo[kk][1]);
        }
        const uint32_t brow = (uint32_t)((((lane >> 3) & 1) << 3) + (lane & 7));
        const uint32_t bcol = (uint32_t)((lane >> 4) << 3);
#pragma unroll 4
        for (int t = t_first; t < ntl; t += kWarps) {
          const int col0 = c0 + t * 16;  // first column of the tile (CTA-relative: - cb)
          const uint32_t baddr = smem_addr(Bs + (size_t)(col0 - cb + brow) * R + bcol);
          float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            if (kk < ks_n) {
              uint32_t a0, a1, a2, a3;
              ldsm_x4(baddr + kk * 32, a0, a1, a2, a3);
              mma_16816(d, a0, a1, a2, a3, bhi[kk][0], bhi[kk][1]);
              mma_16816(d, a0, a1, a2, a3, blo[kk][0], blo[kk][1]);
            }
          }
          // fold: d = C[col gq / gq + 8][rows 2tq, 2tq + 1]; every staged value
          // is read before any is written (the accesses could alias as far as
          // the compiler knows, which would serialize each read behind the
          // previous write)
          const int wtile = min(16, c1 - col0);
          __nv_bfloat16* ob = Os + (col0 - cb + gq);
          float ov[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = 2 * tq + (e & 1), cc = (e >> 1) * 8;
            const bool ok = r < nr && gq + cc < wtile && a.add_inputs;
            ov[e] = ok ? __bfloat162float(ob[(size_t)r * pl.o_stride + cc]) : 0.0f;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = 2 * tq + (e & 1), cc = (e >> 1) * 8;
            if (r < nr && gq + cc < wtile)
              ob[(size_t)r * pl.o_stride + cc] = __float2bfloat16_rn(ov[e] + sc[e & 1] * d[e]);
          }
        }
      }
    }
    __syncthreads();
    // ---- the pass's out segments back to global memory: a warp per row,
    // 16-byte stores ------------------------------------------------------
    for (int r = warp; r < nr; r += kWarps) {
      __nv_bfloat16* orow = a.out + tb.out_row(prow[r]) * a.ld_out;
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
  // the last exchange's readers are done before this CTA's Rx goes away
  cluster_wait();
}

}  // namespace lora
