// The routed LoRA delta for small row groups, one thread-block cluster per
// adapter key ("Module lora_delta", apply_lora_bgmv; "punica_base.py",
// add_lora_linear / add_shrink / add_expand; the MoE FC1 variant of
// "flashinfer.fused_moe.bgmv_moe_gemm1_lora_delta").
//
// One cluster of CS CTAs per key (a slot, or an (adapter, expert) pair):
//   * prologue, before the grid dependency wait of programmatic dependent
//     launch: the key's table entries are resolved and, when nearly every key
//     has rows, the CTA's share of the A rows starts streaming into shared
//     memory and the B rows of its columns into L2 -- adapter weights are
//     never produced by the preceding kernel, so this overlaps its tail;
//   * the key's rows are found on the device (own ballot scan for small n,
//     else the routing kernel's stable clusters) and handled in passes of 16;
//     keys whose row count falls outside [min_rows, max_rows) are skipped;
//   * shrink: CTA c contracts its 1/CS share of k_in.  A rows and x rows are
//     staged in padded (ldmatrix-conflict-free) shared rows by 16-byte
//     cp.async copies from all threads, and the contraction runs as
//     mma.sync m16n8k16 tiles (16 (slice, rank) pairs x 8 rows, fp32
//     accumulate) split over the warps by k-group;
//   * the CS partial sums meet through distributed shared memory with two
//     rounds of remote stores and no remote loads: each CTA pushes its
//     partial of entry e to e's owner, each owner sums its entries over the
//     cluster in rank order and pushes the sum into every CTA's h, so all
//     CTAs hold the same fp32 h, which never goes to global memory;
//   * expand + fold: CTA c owns 1/CS of the concatenated output columns.  h
//     of the pass is split into a bf16 (hi, lo) pair -- the rank contraction
//     keeps ~fp32 accuracy -- and multiplied by 8-column tiles of B on the
//     tensor cores; every tile's B and out loads are issued before its MMAs,
//     and out is updated in place, RN_bf16(out + scale * d), one rounding.
// A key's A and B come from HBM once per call for the usual decode case of
// at most 16 rows per slot.
#pragma once

#include "common.cuh"

namespace lora {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxRowsPerPass = 16;

enum DeltaMode { kModeFused = 0, kModeShrink = 1, kModeExpand = 2 };

struct SlotView {
  const __nv_bfloat16* A[kMaxSlices];
  const __nv_bfloat16* B[kMaxSlices];
  int ja[kMaxSlices];  // ordinal among the active slices, -1 if inactive
  int act_slice[kMaxSlices];
  int nact;
  float scale;
};

// Linear delta: "Module lora_delta", LoraRoute tables.
struct LinearTables {
  const uint64_t* a_table;
  const uint64_t* b_table;
  const float* scale_table;
  int max_loras;
  __device__ void resolve(int key, int S, int mode, SlotView& v, uint32_t& bad) const {
    uint64_t av[kMaxSlices], bv[kMaxSlices];
#pragma unroll
    for (int j = 0; j < kMaxSlices; ++j) {  // independent loads, one round trip
      av[j] = (j < S && mode != kModeExpand) ? a_table[(size_t)j * max_loras + key] : 16u;
      bv[j] = (j < S && mode != kModeShrink) ? b_table[(size_t)j * max_loras + key] : 16u;
    }
    v.scale = scale_table ? scale_table[key] : 1.0f;
    v.nact = 0;
#pragma unroll
    for (int j = 0; j < kMaxSlices; ++j) {
      v.ja[j] = -1;
      if (j >= S) continue;
      const uint64_t a = av[j], b = bv[j];
      if ((a & 15u) || (b & 15u)) {
        bad |= LORA_DEV_ERR_ALIGN;
        continue;
      }
      if (a == 0 || b == 0) continue;
      v.A[j] = reinterpret_cast<const __nv_bfloat16*>(a);
      v.B[j] = reinterpret_cast<const __nv_bfloat16*>(b);
      v.act_slice[v.nact] = j;
      v.ja[j] = v.nact++;
    }
  }
  __device__ int64_t x_row(int item) const { return item; }
  __device__ int64_t out_row(int item) const { return item; }
  __device__ float row_weight(int) const { return 1.0f; }
};

// MoE: key = l * E + e (local expert e); slices = (gate, up) or one fused
// slice for FC1 / w13, one down slice for w2.  Items are (token, slot)
// pairs; the input row is the token's (x_div = top_k) or the pair's own
// (x_div = 1, the down projection).
struct MoeTables {
  const int64_t* w_ptr_a;
  const int64_t* w_ptr_b;
  int64_t stride_a, stride_b;
  int E, x_div, n_slices;
  float scale;
  const float* pair_weight;  // [T * top_k] routing weights folded with scale, or null
  __device__ void resolve(int key, int S, int mode, SlotView& v, uint32_t& bad) const {
    const int l = key / E, e = key - (key / E) * E;
    v.scale = scale;
    v.nact = 0;
    for (int j = 0; j < kMaxSlices; ++j) {
      v.ja[j] = -1;
      if (j >= n_slices) continue;
      const uint64_t a = (uint64_t)w_ptr_a[(size_t)j * E + e] + (uint64_t)l * stride_a * 2u;
      const uint64_t b = (uint64_t)w_ptr_b[(size_t)j * E + e] + (uint64_t)l * stride_b * 2u;
      if ((a & 15u) || (b & 15u)) {
        bad |= LORA_DEV_ERR_ALIGN;
        continue;
      }
      v.A[j] = reinterpret_cast<const __nv_bfloat16*>(a);
      v.B[j] = reinterpret_cast<const __nv_bfloat16*>(b);
      v.act_slice[v.nact] = j;
      v.ja[j] = v.nact++;
    }
  }
  __device__ int64_t x_row(int item) const { return item / x_div; }
  __device__ int64_t out_row(int item) const { return item; }
  __device__ float row_weight(int item) const { return pair_weight ? pair_weight[item] : 1.0f; }
};

struct DeltaArgs {
  __nv_bfloat16* out;
  int64_t ld_out;
  const __nv_bfloat16* x;
  int64_t ld_x;
  int k_in;
  float* h;  // [S, n, R] fp32 for the shrink / expand modes
  int h_parts;  // expand: h as [h_parts][S][n][R / h_parts] (0 or 1: [S, n, R])
  int n;     // rows (items)
  const int32_t* seq_slot;  // own clustering by scan when perm == nullptr
  const int32_t* perm;
  const int32_t* seg_start;
  int n_keys;
  int R;
  Slices sl;
  int rel[kMaxSlices + 1];  // slice starts relative to the first slice; rel[S..] = n_cols
  int add_inputs;
  int kc;     // k-range per CTA (multiple of 16)
  int kst;    // k per shared-memory stage (multiple of 16)
  int nbuf;   // stage buffers (1 or 2)
  int cpc;    // output columns per CTA (multiple of 8)
  int cs;     // CTAs per cluster
  int early;  // start the weight copies before the grid dependency wait
  int row_cap;
  int b_stage_max;         // largest B slab (bytes) staged in shared memory
  int sr_max;              // S * R: shared-memory sizing
  int min_rows, max_rows;  // keys with a row count outside [min, max) are skipped
  uint32_t* err;
};

constexpr int kRowsPerPass = 16;  // rows of one pass: two 8-wide MMA column tiles

// Shared-memory plan (bytes), identical on host and device.
struct SmemPlan {
  int rows_off, As_off, Xs_off, Pw_off, Rx_off, H_off, Bs_off, Os_off, total;
  int b_staged;   // the CTA's B rows fit in shared memory
  int o_stride;   // elements per staged out row (padded)
  int as_stride;  // elements per A / x row in shared memory (padded)
  int sr16;       // S * R rounded up to 16
};
__host__ __device__ inline SmemPlan smem_plan(const DeltaArgs& a, int mode) {
  SmemPlan p;
  p.sr16 = (a.sr_max + 15) / 16 * 16;
  p.as_stride = a.kst + 8;
  int o = 128;  // the pass's row ids (16 ints) at offset 64
  p.rows_off = o;
  o += ((a.row_cap * 4 + 127) / 128) * 128;
  p.As_off = o;
  if (mode != kModeExpand) o += a.nbuf * p.sr16 * p.as_stride * 2;
  p.Xs_off = o;
  if (mode != kModeExpand) o += a.nbuf * kRowsPerPass * p.as_stride * 2;
  o = (o + 127) / 128 * 128;
  p.Pw_off = o;
  if (mode != kModeExpand) o += (p.sr16 > 128 ? p.sr16 : 128) * kRowsPerPass * 4;
  p.Rx_off = o;  // this CTA's partial h, read by the cluster: [kRowsPerPass][sr16]
  if (mode != kModeExpand) o += kRowsPerPass * p.sr16 * 4;
  p.H_off = o;
  o += kRowsPerPass * p.sr16 * 4;
  // expand operands: the CTA's B rows and the pass's out segments
  p.b_staged = (mode != kModeShrink && a.cpc * a.R * 2 <= a.b_stage_max) ? 1 : 0;
  p.o_stride = a.cpc + 8;
  p.Bs_off = o;
  if (p.b_staged) o += a.cpc * a.R * 2;
  p.Os_off = o;
  if (p.b_staged && a.add_inputs) o += kRowsPerPass * p.o_stride * 2;
  p.total = o;
  return p;
}

// 16-byte cp.async copies of the A rows (columns [k0, k0 + kw) of the key's
// active (slice, rank) pairs) into As, by `nw` warps (`tid` counts from the
// first of them).  Warp w copies rows w, w + nw, ...; its lanes cover the
// row's 16-byte pieces.  Row t is pair (jj, q) = (t / R, t % R), tracked
// incrementally (R >= 8 >= nw, so q wraps at most once per step), so the
// loop carries no division and only one pointer reload per slice.
__device__ __forceinline__ void copy_a_rows(const DeltaArgs& a, const SlotView& v, int SRa,
                                            int k0, int kw, __nv_bfloat16* As, int stride,
                                            int tid, int nw = kWarps) {
  const int R = a.R, vpr = kw >> 3, warp = tid >> 5, lane = tid & 31;
  const size_t kin = (size_t)a.k_in;
  int jj = 0, q = warp;
  const __nv_bfloat16* base = v.A[v.act_slice[0]] + k0 + lane * 8;
  __nv_bfloat16* dst = As + (size_t)warp * stride + lane * 8;
#pragma unroll 2
  for (int t = warp; t < SRa; t += nw) {
    const __nv_bfloat16* src = base + (size_t)q * kin;
    for (int c = 0; c < vpr - lane; c += 32) cp_async16(dst + c * 8, src + c * 8);
    dst += (size_t)nw * stride;
    q += nw;
    if (q >= R) {
      q -= R;
      if (++jj < v.nact) base = v.A[v.act_slice[jj]] + k0 + lane * 8;
    }
  }
}

// ... and of the pass's x rows into Xs (warp per row, as above).
template <class Tables>
__device__ __forceinline__ void copy_x_rows(const DeltaArgs& a, const Tables& tb, const int* prow,
                                            int nr, int k0, int kw, __nv_bfloat16* Xs,
                                            int stride, int tid, int nw = kWarps) {
  const int vpr = kw >> 3, warp = tid >> 5, lane = tid & 31;
  for (int r = warp; r < nr; r += nw) {
    const __nv_bfloat16* src = a.x + tb.x_row(prow[r]) * a.ld_x + k0 + lane * 8;
    __nv_bfloat16* dst = Xs + (size_t)r * stride + lane * 8;
    for (int c = 0; c < vpr - lane; c += 32) cp_async16(dst + c * 8, src + c * 8);
  }
}

// cp.async copies of the B rows of this CTA's columns [cb, ce) into Bs
// (column c at Bs[(c - cb) * R]).  Each slice's part is one contiguous run.
__device__ __forceinline__ void copy_b_rows(const DeltaArgs& a, const SlotView& v, int cb, int ce,
                                            __nv_bfloat16* Bs, int tid, int nthr = kThreads) {
  for (int j = 0; j < a.sl.S; ++j) {
    const int c0 = max(cb, a.rel[j]), c1 = min(ce, a.rel[j + 1]);
    if (c1 <= c0 || v.ja[j] < 0) continue;
    const int nvec = (c1 - c0) * a.R / 8;
    const __nv_bfloat16* src = v.B[j] + (size_t)(c0 - a.rel[j]) * a.R + tid * 8;
    __nv_bfloat16* dst = Bs + (size_t)(c0 - cb) * a.R + tid * 8;
#pragma unroll 4
    for (int i = 0; i < nvec - tid; i += nthr) cp_async16(dst + i * 8, src + i * 8);
  }
}

// cp.async copies of the pass's out segments in this CTA's columns into Os
// (row r, column c at Os[r * o_stride + (c - cb)]); warp per row.
template <class Tables>
__device__ __forceinline__ void copy_out_rows(const DeltaArgs& a, const Tables& tb,
                                              const SlotView& v, const int* prow, int nr, int cb,
                                              int ce, __nv_bfloat16* Os, int o_stride, int tid,
                                              int nw = kWarps) {
  const int warp = tid >> 5, lane = tid & 31;
  for (int j = 0; j < a.sl.S; ++j) {
    const int c0 = max(cb, a.rel[j]), c1 = min(ce, a.rel[j + 1]);
    if (c1 <= c0 || v.ja[j] < 0) continue;
    const int vpr = (c1 - c0) >> 3;
    const int64_t col = a.sl.off[j] + (c0 - a.rel[j]) + lane * 8;
    for (int r = warp; r < nr; r += nw) {
      const __nv_bfloat16* src = a.out + tb.out_row(prow[r]) * a.ld_out + col;
      __nv_bfloat16* dst = Os + (size_t)r * o_stride + (c0 - cb) + lane * 8;
      for (int c = 0; c < vpr - lane; c += 32) cp_async16(dst + c * 8, src + c * 8);
    }
  }
}

// L2 prefetch (by the lanes of one warp) of the B rows of this CTA's columns.
__device__ __forceinline__ void prefetch_b(const DeltaArgs& a, const SlotView& v, int cb, int ce,
                                           int lane) {
  for (int j = lane; j < a.sl.S; j += 32) {
    if (v.ja[j] < 0) continue;
    const int c0 = max(cb, a.rel[j]), c1 = min(ce, a.rel[j + 1]);
    if (c1 > c0)
      bulk_prefetch_l2(v.B[j] + (size_t)(c0 - a.rel[j]) * a.R, (uint32_t)((c1 - c0) * a.R * 2));
  }
}

// L2 prefetch of the out segments of the pass's rows in this CTA's columns.
template <class Tables>
__device__ __forceinline__ void prefetch_out(const DeltaArgs& a, const Tables& tb,
                                             const SlotView& v, const int* prow, int nr, int cb,
                                             int ce, int lane) {
  for (int j = 0; j < a.sl.S; ++j) {
    if (v.ja[j] < 0) continue;
    const int c0 = max(cb, a.rel[j]), c1 = min(ce, a.rel[j + 1]);
    if (c1 <= c0) continue;
    for (int r = lane; r < nr; r += 32)
      bulk_prefetch_l2(a.out + tb.out_row(prow[r]) * a.ld_out + a.sl.off[j] + (c0 - a.rel[j]),
                       (uint32_t)((c1 - c0) * 2));
  }
}

template <int RMAX, int MODE, class Tables>
__global__ void __launch_bounds__(kThreads, (RMAX <= 32 ? 3 : 2))
    delta_cluster_kernel(const DeltaArgs a, const Tables tb) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ SlotView v;
  __shared__ int nrows_s, rows_base_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3;  // MMA fragment coordinates
  const int key = (int)cluster_index_x();
  const uint32_t crank = cluster_rank();
  const int ncta = a.cs;

  const SmemPlan plan = smem_plan(a, MODE);
  int* prow = reinterpret_cast<int*>(smem + 64);  // this pass's row ids
  int* rows_s = reinterpret_cast<int*>(smem + plan.rows_off);
  __nv_bfloat16* As = reinterpret_cast<__nv_bfloat16*>(smem + plan.As_off);
  __nv_bfloat16* Xs = reinterpret_cast<__nv_bfloat16*>(smem + plan.Xs_off);
  float* Pw = reinterpret_cast<float*>(smem + plan.Pw_off);
  float* Rx = reinterpret_cast<float*>(smem + plan.Rx_off);
  float* H = reinterpret_cast<float*>(smem + plan.H_off);
  __nv_bfloat16* Bs = reinterpret_cast<__nv_bfloat16*>(smem + plan.Bs_off);
  __nv_bfloat16* Os = reinterpret_cast<__nv_bfloat16*>(smem + plan.Os_off);
  const int stride = plan.as_stride, SR16 = plan.sr16;
  const bool b_staged = plan.b_staged != 0;
  const bool o_staged = b_staged && a.add_inputs;

  // ---- prologue: independent of the preceding kernel's outputs ----------
  if (tid == 0) {
    uint32_t bad = 0;
    tb.resolve(key, a.sl.S, MODE, v, bad);
    if (bad && crank == 0) set_error(a.err, bad);
  }
  __syncthreads();
  const int R = a.R;
  const int SRa = v.nact * R;
  const int k_lo = min(a.k_in, (int)crank * a.kc);
  const int k_hi = min(a.k_in, k_lo + a.kc);
  const int nst = (k_hi - k_lo + a.kst - 1) / a.kst;  // shrink stages of this CTA
  const int cb = min(a.sl.n_cols, (int)crank * a.cpc);
  const int ce = min(a.sl.n_cols, cb + a.cpc);
  // Adapter weights are never produced by the preceding kernel, so their
  // copies may start before the dependency wait and overlap its tail.  Warps
  // 1.. issue them while warp 0 waits for the dependency, finds the key's
  // rows and starts the first pass's x / out copies.
  const bool early = MODE != kModeExpand && a.early && v.nact > 0 && nst > 0;
  if (early && warp > 0) {
    copy_a_rows(a, v, SRa, k_lo, min(a.kst, k_hi - k_lo), As, stride, tid - 32, kWarps - 1);
    if (b_staged) copy_b_rows(a, v, cb, ce, Bs, tid - 32, kThreads - 32);
    cp_async_commit();
  }
  bool b_loaded = early && b_staged;
  if (v.nact > 0 && MODE != kModeShrink && !b_staged && warp == 1) prefetch_b(a, v, cb, ce, lane);
  cudaTriggerProgrammaticLaunchCompletion();
  cudaGridDependencySynchronize();
  // Without a routing pass, CTA 0 of key 0 also checks every slot for
  // LORA_DEV_ERR_SLOT, so it scans even when key 0 adapts nothing.
  const bool slot_check = !a.perm && key == 0 && crank == 0;
  if (v.nact == 0 && !slot_check) return;  // the same in every CTA of the cluster

  // ---- the key's rows, in ascending row order (warp 0) -----------------
  // Warp 0 also starts the first pass's x / out copies when they are few
  // (decode-sized: at most 16 per lane); larger ones are left to every warp.
  // The choice depends only on the key's row count, which warp 0 knows first
  // and every thread reads after the barrier below.
  const int w0_chunks = min(a.kst, k_hi - k_lo) / 8 + (o_staged ? a.cpc / 8 : 0);
  auto warp0_copies_for = [&](int total) {
    return early && min(kRowsPerPass, total) * w0_chunks <= 512;
  };
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
    __syncwarp();
    if (warp0_copies_for(total) && total > 0 && total >= a.min_rows && total < a.max_rows) {
      const int* rows0 = a.perm ? a.perm + s0 : rows_s;
      const int nr0 = min(kRowsPerPass, total);
      copy_x_rows(a, tb, rows0, nr0, k_lo, min(a.kst, k_hi - k_lo), Xs, stride, lane, 1);
      if (o_staged) copy_out_rows(a, tb, v, rows0, nr0, cb, ce, Os, plan.o_stride, lane, 1);
      cp_async_commit();
    }
  }
  __syncthreads();
  if (v.nact == 0) return;
  const int nrows = nrows_s;
  const bool warp0_copies = warp0_copies_for(nrows);
  const int* rows = a.perm ? a.perm + rows_base_s : rows_s;
  if (nrows == 0 || nrows < a.min_rows || nrows >= a.max_rows) {  // uniform
    if (early) cp_async_wait<0>();  // no copy may land in a CTA that has exited
    return;
  }

  const int mt = (SRa + 15) / 16;  // 16-pair tiles of the shrink
  const int SRk = mt * 16;         // this key's padded pair count (Pw row stride)
  // shrink work split: G k-groups x mt pair tiles over the 8 warps
  const int G = mt >= kWarps ? 1 : kWarps / mt;
  const int my_g = mt >= kWarps ? 0 : warp / mt;
  const int my_m0 = mt >= kWarps ? warp : warp % mt;
  const bool shrink_warp = mt >= kWarps || warp < G * mt;
  const bool timed_out = false;  // (no bounded waits in this kernel)
  bool skip_a0 = early;  // stage-0 A rows already in shared memory (early copy / resident)

  if (MODE != kModeExpand && SRa < SR16) {  // pad pair rows contract to zero
    const int per_buf = (SR16 - SRa) * stride / 8;
    for (int i = tid; i < a.nbuf * per_buf; i += kThreads) {
      const int b = i / per_buf, rem = i - b * per_buf;
      reinterpret_cast<uint4*>(As + (size_t)b * SR16 * stride + (size_t)SRa * stride)[rem] =
          make_uint4(0, 0, 0, 0);
    }
  }

  for (int p0 = 0; p0 < nrows; p0 += kRowsPerPass) {
    const int nr = min(kRowsPerPass, nrows - p0);
    __syncthreads();  // the previous pass is done with prow and the buffers
    if (tid < nr) prow[tid] = rows[p0 + tid];
    if (MODE != kModeExpand) {  // pad x rows of the pass contract to zero
      const int pad = (kRowsPerPass - nr) * stride / 8;  // 16-byte units
      for (int i = tid; i < a.nbuf * pad; i += kThreads) {
        const int b = i / pad, rem = i - b * pad;
        reinterpret_cast<uint4*>(Xs + (size_t)b * kRowsPerPass * stride + (size_t)nr * stride)[rem] =
            make_uint4(0, 0, 0, 0);
      }
    }
    __syncthreads();
    if (MODE != kModeShrink) {
      // expand operands of the pass: into shared memory when they fit, else L2
      if (b_staged && !b_loaded) copy_b_rows(a, v, cb, ce, Bs, tid);
      b_loaded = b_staged;
      if (o_staged) {
        if (!(warp0_copies && p0 == 0))  // (the first pass's were started by warp 0)
          copy_out_rows(a, tb, v, prow, nr, cb, ce, Os, plan.o_stride, tid);
      } else if (warp == 2)
        prefetch_out(a, tb, v, prow, nr, cb, ce, lane);
      cp_async_commit();  // (its own group, so the stage waits below stay in order)
    }

    if (MODE != kModeExpand) {
      // ---- copies of the first two stages ---------------------------------
      if (nst > 0) {
        if (!skip_a0) copy_a_rows(a, v, SRa, k_lo, min(a.kst, k_hi - k_lo), As, stride, tid);
        if (!(warp0_copies && p0 == 0))  // (the first pass's were started by warp 0)
          copy_x_rows(a, tb, prow, nr, k_lo, min(a.kst, k_hi - k_lo), Xs, stride, tid);
        cp_async_commit();
        if (nst > 1) {
          const int k1 = k_lo + a.kst;
          copy_a_rows(a, v, SRa, k1, min(a.kst, k_hi - k1), As + (size_t)SR16 * stride, stride,
                      tid);
          copy_x_rows(a, tb, prow, nr, k1, min(a.kst, k_hi - k1),
                      Xs + (size_t)kRowsPerPass * stride, stride, tid);
          cp_async_commit();
        }
      }
      skip_a0 = (nst == 1);  // a single stage keeps its A rows for the next passes

      // ---- shrink on the tensor cores: partial P[pair][row] over this CTA's k
      // pair tiles per warp: mt <= S * R / 16 <= 8 * RMAX / 16, so at most RMAX / 16
      constexpr int MI = RMAX / 16 < 4 ? RMAX / 16 : 4;
      float acc[MI][8];
#pragma unroll
      for (int i = 0; i < MI; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = 0.0f;
      for (int st = 0; st < nst; ++st) {
        const int buf = st & 1;
        const int k0 = k_lo + st * a.kst;
        const int kw = min(a.kst, k_hi - k0);
        if (st + 1 < nst)
          cp_async_wait<1>();  // this stage landed; the next may still be in flight
        else
          cp_async_wait<0>();
        __nv_bfloat16* Ab = As + (size_t)buf * SR16 * stride;
        __nv_bfloat16* Xb = Xs + (size_t)buf * kRowsPerPass * stride;
        if (kw & 15) {  // odd half k-step: zero the 8 columns after kw (never copied)
          for (int i = tid; i < SRa + nr; i += kThreads) {
            __nv_bfloat16* rowp = (i < SRa) ? Ab + (size_t)i * stride : Xb + (size_t)(i - SRa) * stride;
            *reinterpret_cast<uint4*>(rowp + kw) = make_uint4(0, 0, 0, 0);
          }
        }
        __syncthreads();
        if (shrink_warp) {
          const int ksteps = (kw + 15) / 16;
          const uint32_t xaddr = smem_addr(Xb + (size_t)(((lane >> 4) << 3) + (lane & 7)) * stride +
                                           ((lane >> 3) & 1) * 8);
          const uint32_t aaddr = smem_addr(Ab + (size_t)(my_m0 * 16 + (((lane >> 3) & 1) << 3) +
                                                         (lane & 7)) * stride + ((lane >> 4) << 3));
          const uint32_t mstep = 8u * 16u * (uint32_t)stride * 2u;  // 8 pair tiles, bytes
          if (mt >= kWarps) {  // up to 4 pair tiles per warp: 4 independent chains
            for (int ks = my_g; ks < ksteps; ks += G) {
              uint32_t b0, b1, b2, b3;
              ldsm_x4(xaddr + ks * 32, b0, b1, b2, b3);
#pragma unroll
              for (int i = 0; i < MI; ++i) {
                if (my_m0 + i * kWarps < mt) {
                  uint32_t a0, a1, a2, a3;
                  ldsm_x4(aaddr + i * mstep + ks * 32, a0, a1, a2, a3);
                  mma_16816(&acc[i][0], a0, a1, a2, a3, b0, b1);
                  mma_16816(&acc[i][4], a0, a1, a2, a3, b2, b3);
                }
              }
            }
          } else {  // one pair tile: two chains over alternate k-steps
            float acc2[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc2[e] = 0.0f;
            int ks = my_g;
            for (; ks + G < ksteps; ks += 2 * G) {
              uint32_t b0, b1, b2, b3, c0, c1, c2, c3, a0, a1, a2, a3, d0, d1, d2, d3;
              ldsm_x4(xaddr + ks * 32, b0, b1, b2, b3);
              ldsm_x4(aaddr + ks * 32, a0, a1, a2, a3);
              ldsm_x4(xaddr + (ks + G) * 32, c0, c1, c2, c3);
              ldsm_x4(aaddr + (ks + G) * 32, d0, d1, d2, d3);
              mma_16816(&acc[0][0], a0, a1, a2, a3, b0, b1);
              mma_16816(&acc[0][4], a0, a1, a2, a3, b2, b3);
              mma_16816(&acc2[0], d0, d1, d2, d3, c0, c1);
              mma_16816(&acc2[4], d0, d1, d2, d3, c2, c3);
            }
            if (ks < ksteps) {
              uint32_t b0, b1, b2, b3, a0, a1, a2, a3;
              ldsm_x4(xaddr + ks * 32, b0, b1, b2, b3);
              ldsm_x4(aaddr + ks * 32, a0, a1, a2, a3);
              mma_16816(&acc[0][0], a0, a1, a2, a3, b0, b1);
              mma_16816(&acc[0][4], a0, a1, a2, a3, b2, b3);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[0][e] += acc2[e];
          }
        }
        __syncthreads();  // buffer `buf` free
        if (st + 2 < nst) {
          const int k2 = k0 + 2 * a.kst;
          copy_a_rows(a, v, SRa, k2, min(a.kst, k_hi - k2), Ab, stride, tid);
          copy_x_rows(a, tb, prow, nr, k2, min(a.kst, k_hi - k2), Xb, stride, tid);
          cp_async_commit();
        }
      }
      // per-warp k-group partials -> Pw[g][pair][row]
      if (shrink_warp) {
#pragma unroll
        for (int i = 0; i < MI; ++i) {
          const int m = my_m0 + i * kWarps;
          if (m < mt && (i == 0 || mt >= kWarps)) {
            float* base = Pw + ((size_t)my_g * SRk + m * 16 + gq) * kRowsPerPass + 2 * tq;
            base[0] = acc[i][0];
            base[1] = acc[i][1];
            base[8 * kRowsPerPass] = acc[i][2];
            base[8 * kRowsPerPass + 1] = acc[i][3];
            base[8] = acc[i][4];
            base[9] = acc[i][5];
            base[8 * kRowsPerPass + 8] = acc[i][6];
            base[8 * kRowsPerPass + 9] = acc[i][7];
          }
        }
      }
      __syncthreads();
      // ---- the cluster's partials meet in one exchange: every CTA leaves its
      // partial (summed over its k-groups) in its own Rx; after one cluster
      // barrier each CTA reads the ncta partials of its entries from the
      // peers' shared memory, all loads in flight together, and sums them in
      // rank order into H.  A second barrier phase, arrived at right after the
      // reads and waited on only before Rx is rewritten (the next pass) or the
      // CTA exits, keeps every Rx alive while peers may still read it. ----
      const int nel = nr * SRa;
      if (p0 > 0) cluster_wait();  // the previous pass's readers are done with Rx
      // this thread's entries: groups of 4 consecutive pairs (SRa is a
      // multiple of 8), group g = tid + i * kThreads as (row r, pair p)
      const int gpr = SRa >> 2;  // groups per row
      const int dr = kThreads / gpr, dp = (kThreads - dr * gpr) * 4;
      const int r_first = tid / gpr, p_first = (tid - r_first * gpr) * 4;
      {
        int r = r_first, p = p_first;
        for (int e = tid * 4; e < nel; e += kThreads * 4) {
          float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int g = 0; g < G; ++g) {
            const float* src = Pw + ((size_t)g * SRk + p) * kRowsPerPass + r;
            s.x += src[0];
            s.y += src[kRowsPerPass];
            s.z += src[2 * kRowsPerPass];
            s.w += src[3 * kRowsPerPass];
          }
          *reinterpret_cast<float4*>(Rx + r * SR16 + p) = s;
          p += dp;
          r += dr;
          if (p >= SRa) {
            p -= SRa;
            ++r;
          }
        }
      }
      cluster_arrive_release_smem();  // partials in place
      cluster_wait();
      {
        // 4 lanes per 4-entry group; lane qq reads peers qq, qq + 4, qq + 8,
        // qq + 12 (all in flight together), then two xor-shuffles add the
        // lanes: one round trip, the same summation order in every CTA
        const uint32_t rx_addr = smem_addr(Rx);
        const int ngrp = nel >> 2, qq = lane & 3;
        for (int gb = (tid >> 2); gb - (lane >> 2) < ngrp; gb += kThreads / 4) {
          const bool valid = gb < ngrp;  // (the warp's lanes stay together)
          const int e = 4 * (valid ? gb : 0);
          const int r = e / SRa, p = e - r * SRa;
          const uint32_t addr = rx_addr + 4u * (uint32_t)(r * SR16 + p);
          float4 part[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c = qq + 4 * u;
            part[u] = (valid && c < ncta) ? dsmem_ld_f32x4(dsmem_map(addr, (uint32_t)c))
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
          }
          float4 v = part[0];
#pragma unroll
          for (int u = 1; u < 4; ++u) {
            v.x += part[u].x;
            v.y += part[u].y;
            v.z += part[u].z;
            v.w += part[u].w;
          }
#pragma unroll
          for (int off = 1; off < 4; off <<= 1) {
            v.x += __shfl_xor_sync(0xffffffffu, v.x, off);
            v.y += __shfl_xor_sync(0xffffffffu, v.y, off);
            v.z += __shfl_xor_sync(0xffffffffu, v.z, off);
            v.w += __shfl_xor_sync(0xffffffffu, v.w, off);
          }
          if (valid && qq == 0) *reinterpret_cast<float4*>(H + r * SR16 + p) = v;
        }
      }
      cluster_arrive_relaxed();  // done reading the peers' Rx (waited on later)
      __syncthreads();   // H complete
    } else {
      // (h in rank parts, as the all-gather of rank-sharded shrinks leaves it:
      // rank q of slice j, row i at [q / rp][j][i][q % rp])
      const int rp = a.h_parts > 1 ? R / a.h_parts : R;
      for (int i = tid; i < nr * SRa; i += kThreads) {
        const int r = i / SRa, t = i - r * SRa;
        const int jj = t / R, q = t - jj * R;
        const int part = q / rp, qq = q - part * rp;
        H[r * SR16 + t] =
            a.h[(((size_t)part * a.sl.S + v.act_slice[jj]) * a.n + prow[r]) * rp + qq];
      }
      __syncthreads();
    }

    if (MODE == kModeShrink) {
      // h[j, row, q] += scale * H, the cluster's CTAs splitting the entries.
      for (int i = (int)crank * kThreads + tid; i < nr * SRa; i += ncta * kThreads) {
        const int r = i / SRa, t = i - r * SRa, jj = t / R, q = t - jj * R;
        const int j = v.act_slice[jj];
        float* dst = a.h + ((size_t)j * a.n + prow[r]) * R + q;
        *dst = *dst + H[r * SR16 + t] * v.scale;
      }
    } else if (!timed_out) {
      // ---- expand + fold on the tensor cores, 8 columns per tile ----------
      // A operand: the pass's h rows of one slice as a bf16 (hi, lo) pair, so
      // the rank contraction keeps ~fp32 accuracy (rows >= nr only feed
      // discarded outputs); B operand: B rows from shared memory (or L2).
      if (b_staged) {
        cp_async_wait<0>();  // B rows and out segments landed
        __syncthreads();
      }
      constexpr int KS = RMAX / 16;
      constexpr int NB = KS == 4 ? 4 : (KS > 4 ? 1 : 4 / KS);  // column tiles per load batch
      const int row0 = gq, row1 = gq + 8;
      const bool ok0 = row0 < nr, ok1 = row1 < nr;
      const int64_t orow0 = ok0 ? tb.out_row(prow[row0]) : 0;
      const int64_t orow1 = ok1 ? tb.out_row(prow[row1]) : 0;
      const float sc0 = ok0 ? v.scale * tb.row_weight(prow[row0]) : 0.f;
      const float sc1 = ok1 ? v.scale * tb.row_weight(prow[row1]) : 0.f;
      for (int j = 0; j < a.sl.S; ++j) {
        const int ja = v.ja[j];
        if (ja < 0) continue;
        const int c0 = max(cb, a.rel[j]), c1 = min(ce, a.rel[j + 1]);
        if (c1 <= c0) continue;
        const int ntl = (c1 - c0) / 8;
        if (warp >= ntl) continue;
        uint32_t ahi[KS][4], alo[KS][4];
        {
          const float* hb = H + ja * R + 2 * tq;
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            const bool lo_ok = kk * 16 < R, hi_ok = kk * 16 + 8 < R;
            const float* h0 = hb + row0 * SR16 + kk * 16;
            const float* h1 = hb + row1 * SR16 + kk * 16;
            split_bf16x2(lo_ok ? h0[0] : 0.f, lo_ok ? h0[1] : 0.f, ahi[kk][0], alo[kk][0]);
            split_bf16x2(lo_ok ? h1[0] : 0.f, lo_ok ? h1[1] : 0.f, ahi[kk][1], alo[kk][1]);
            split_bf16x2(hi_ok ? h0[8] : 0.f, hi_ok ? h0[9] : 0.f, ahi[kk][2], alo[kk][2]);
            split_bf16x2(hi_ok ? h1[8] : 0.f, hi_ok ? h1[9] : 0.f, ahi[kk][3], alo[kk][3]);
          }
        }
        const int cl0 = c0 - a.rel[j];
        __nv_bfloat16* o0base = a.out + orow0 * a.ld_out + a.sl.off[j] + cl0 + 2 * tq;
        __nv_bfloat16* o1base = a.out + orow1 * a.ld_out + a.sl.off[j] + cl0 + 2 * tq;
        if (b_staged) {
          // operands in shared memory: one tile at a time
          const __nv_bfloat16* bsb = Bs + (size_t)(c0 - cb + gq) * R + 2 * tq;
          const __nv_bfloat16* os0 = Os + (size_t)row0 * plan.o_stride + (c0 - cb) + 2 * tq;
          const __nv_bfloat16* os1 = Os + (size_t)row1 * plan.o_stride + (c0 - cb) + 2 * tq;
          // batches of NS tiles: every shared-memory load first, then the
          // NS independent MMA chains, then the stores
          constexpr int NS = KS <= 2 ? 2 : 1;
          for (int t0 = warp; t0 < ntl; t0 += kWarps * NS) {
            uint32_t bf[NS][KS][2], ov[NS][2];
#pragma unroll
            for (int b = 0; b < NS; ++b) {
              const int t = t0 + b * kWarps;
              if (t < ntl) {
                const __nv_bfloat16* brow = bsb + (size_t)t * 8 * R;
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                  bf[b][kk][0] =
                      (kk * 16 < R) ? *reinterpret_cast<const uint32_t*>(brow + kk * 16) : 0u;
                  bf[b][kk][1] =
                      (kk * 16 + 8 < R) ? *reinterpret_cast<const uint32_t*>(brow + kk * 16 + 8) : 0u;
                }
                ov[b][0] = (a.add_inputs && ok0) ? *reinterpret_cast<const uint32_t*>(os0 + t * 8) : 0u;
                ov[b][1] = (a.add_inputs && ok1) ? *reinterpret_cast<const uint32_t*>(os1 + t * 8) : 0u;
              }
            }
#pragma unroll
            for (int b = 0; b < NS; ++b) {
              const int t = t0 + b * kWarps;
              if (t < ntl) {
                float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                  if (kk * 16 < R) {
                    mma_16816(d, ahi[kk][0], ahi[kk][1], ahi[kk][2], ahi[kk][3], bf[b][kk][0], bf[b][kk][1]);
                    mma_16816(d, alo[kk][0], alo[kk][1], alo[kk][2], alo[kk][3], bf[b][kk][0], bf[b][kk][1]);
                  }
                }
                if (ok0)
                  *reinterpret_cast<uint32_t*>(o0base + t * 8) =
                      pack_bf16x2(bf16lo(ov[b][0]) + sc0 * d[0], bf16hi(ov[b][0]) + sc0 * d[1]);
                if (ok1)
                  *reinterpret_cast<uint32_t*>(o1base + t * 8) =
                      pack_bf16x2(bf16lo(ov[b][1]) + sc1 * d[2], bf16hi(ov[b][1]) + sc1 * d[3]);
              }
            }
          }
          continue;
        }
        const __nv_bfloat16* bbase = v.B[j] + (size_t)(cl0 + gq) * R + 2 * tq;
        for (int t0 = warp; t0 < ntl; t0 += kWarps * NB) {
          uint32_t bf[NB][KS][2], ov[NB][2];
#pragma unroll
          for (int b = 0; b < NB; ++b) {  // every load of the batch first (L2 hits)
            const int t = t0 + b * kWarps;
            if (t < ntl) {
              const __nv_bfloat16* brow = bbase + (size_t)t * 8 * R;
#pragma unroll
              for (int kk = 0; kk < KS; ++kk) {
                bf[b][kk][0] = (kk * 16 < R) ? ldg_nc_u32(brow + kk * 16) : 0u;
                bf[b][kk][1] = (kk * 16 + 8 < R) ? ldg_nc_u32(brow + kk * 16 + 8) : 0u;
              }
              ov[b][0] = (a.add_inputs && ok0) ? *reinterpret_cast<const uint32_t*>(o0base + t * 8) : 0u;
              ov[b][1] = (a.add_inputs && ok1) ? *reinterpret_cast<const uint32_t*>(o1base + t * 8) : 0u;
            }
          }
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const int t = t0 + b * kWarps;
            if (t < ntl) {
              float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int kk = 0; kk < KS; ++kk) {
                if (kk * 16 < R) {
                  mma_16816(d, ahi[kk][0], ahi[kk][1], ahi[kk][2], ahi[kk][3], bf[b][kk][0], bf[b][kk][1]);
                  mma_16816(d, alo[kk][0], alo[kk][1], alo[kk][2], alo[kk][3], bf[b][kk][0], bf[b][kk][1]);
                }
              }
              if (ok0)
                *reinterpret_cast<uint32_t*>(o0base + t * 8) =
                    pack_bf16x2(bf16lo(ov[b][0]) + sc0 * d[0], bf16hi(ov[b][0]) + sc0 * d[1]);
              if (ok1)
                *reinterpret_cast<uint32_t*>(o1base + t * 8) =
                    pack_bf16x2(bf16lo(ov[b][1]) + sc1 * d[2], bf16hi(ov[b][1]) + sc1 * d[3]);
            }
          }
        }
      }
    }
  }
  if (timed_out && tid == 0) set_error(a.err, LORA_DEV_ERR_TIMEOUT);
  // the last exchange's readers are done before this CTA's Rx goes away
  if (MODE != kModeExpand) cluster_wait();
}

// Zeros for the MoE pairs that get no delta (the no-key bucket).
__global__ void zero_rows_kernel(__nv_bfloat16* out, int64_t ld_out, int width,
                                 const int32_t* perm, const int32_t* seg_start, int bucket) {
  cudaGridDependencySynchronize();
  const int s0 = seg_start[bucket], s1 = seg_start[bucket + 1];
  const int vec_per_row = width / 8;
  const int64_t total = (int64_t)(s1 - s0) * vec_per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / vec_per_row), v = (int)(i - (int64_t)r * vec_per_row);
    *reinterpret_cast<uint4*>(out + (int64_t)perm[s0 + r] * ld_out + v * 8) =
        make_uint4(0, 0, 0, 0);
  }
}

}  // namespace lora
