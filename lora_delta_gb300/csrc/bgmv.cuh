// The routed LoRA delta on CUDA cores, one thread-block cluster per adapter
// key ("Module lora_delta", apply_lora_bgmv; "punica_base.py",
// add_lora_linear / add_shrink / add_expand; the MoE FC1 variant of
// "flashinfer.fused_moe.bgmv_moe_gemm1_lora_delta").
//
// Work decomposition (one cluster of CS CTAs per key = slot, or (l, e) for MoE):
//   * the key's rows are found on the device (own scan for small n, else the
//     routing kernel's stable clusters) and handled in passes of kRowsPerPass;
//   * shrink: CTA c contracts its 1/CS share of k_in for every row of the pass
//     and every active (slice, rank) pair.  The A rows and x rows of that
//     k-range are pulled into shared memory by 1-D TMA bulk copies
//     (cp.async.bulk) completing on one mbarrier, so every byte a CTA needs is
//     in flight at once; lanes take 16-byte vectors along k and a warp-shuffle
//     tree reduces each dot product;
//   * the CS partial sums meet through distributed shared memory (DSMEM): after
//     a cluster barrier every CTA sums the CS partials in rank order, so all
//     CTAs hold the same fp32 h, which never leaves the chip;
//   * expand + fold: CTA c owns 1/CS of the concatenated output columns; a
//     thread takes two adjacent columns, keeps their B rows in registers and
//     updates out in place, RN_bf16(out + scale * (h . B)), one rounding.
// Each key's A and B are read from HBM once per pass (once in total for the
// usual decode case of <= kRowsPerPass rows per slot).
#pragma once

#include "common.cuh"

namespace lora {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerPass = 16;

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
    v.scale = scale_table ? scale_table[key] : 1.0f;
    v.nact = 0;
    for (int j = 0; j < kMaxSlices; ++j) {
      v.ja[j] = -1;
      if (j >= S) continue;
      uint64_t a = (mode != kModeExpand) ? a_table[(size_t)j * max_loras + key] : 16u;
      uint64_t b = (mode != kModeShrink) ? b_table[(size_t)j * max_loras + key] : 16u;
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
};

// MoE FC1: key = l * E + e; slices = (gate, up) or one fused slice.
struct MoeTables {
  const int64_t* w_ptr_a;
  const int64_t* w_ptr_b;
  int64_t stride_a, stride_b;
  int E, top_k, n_slices;
  float scale;
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
  __device__ int64_t x_row(int item) const { return item / top_k; }
  __device__ int64_t out_row(int item) const { return item; }
};

struct DeltaArgs {
  __nv_bfloat16* out;
  int64_t ld_out;
  const __nv_bfloat16* x;
  int64_t ld_x;
  int k_in;
  float* h;  // [S, n, R] fp32 for the shrink / expand modes
  int n;     // rows (items)
  const int32_t* seq_slot;  // own clustering by scan when perm == nullptr
  const int32_t* perm;
  const int32_t* seg_start;
  int n_keys;
  int R;
  Slices sl;
  int rel[kMaxSlices];  // slice starts relative to the first slice
  int add_inputs;
  int kc;   // k-range per CTA (multiple of 8)
  int ks;   // k per pipeline stage (multiple of 8)
  int cpc;  // output columns per CTA (multiple of 8)
  int row_cap;
  int sr_max;  // S * R: shared-memory sizing
  uint32_t* err;
};

// Shared-memory plan (bytes), identical on host and device.
struct SmemPlan {
  int rows_off, P_off, H_off, A_off, X_off, total;
};
__host__ __device__ inline SmemPlan smem_plan(int row_cap, int sr_max, int ks, int mode) {
  SmemPlan p;
  int o = 128;  // mbarrier + the pass's row ids
  p.rows_off = o;
  o += ((row_cap * 4 + 127) / 128) * 128;
  p.P_off = o;
  o += (mode == kModeExpand) ? 0 : kRowsPerPass * sr_max * 4;
  p.H_off = o;
  o += kRowsPerPass * sr_max * 4;
  p.A_off = o;
  o += (mode == kModeExpand) ? 0 : sr_max * ks * 2;
  p.X_off = o;
  o += (mode == kModeExpand) ? 0 : kRowsPerPass * ks * 2;
  p.total = o;
  return p;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

__device__ __forceinline__ float dot8(const uint4& a, const uint4& b) {
  float s = bf16lo(a.x) * bf16lo(b.x);
  s = fmaf(bf16hi(a.x), bf16hi(b.x), s);
  s = fmaf(bf16lo(a.y), bf16lo(b.y), s);
  s = fmaf(bf16hi(a.y), bf16hi(b.y), s);
  s = fmaf(bf16lo(a.z), bf16lo(b.z), s);
  s = fmaf(bf16hi(a.z), bf16hi(b.z), s);
  s = fmaf(bf16lo(a.w), bf16lo(b.w), s);
  s = fmaf(bf16hi(a.w), bf16hi(b.w), s);
  return s;
}

__device__ __forceinline__ float dot8h(const float* h, const uint4& b) {
  const float4 h0 = *reinterpret_cast<const float4*>(h);
  const float4 h1 = *reinterpret_cast<const float4*>(h + 4);
  float s = h0.x * bf16lo(b.x);
  s = fmaf(h0.y, bf16hi(b.x), s);
  s = fmaf(h0.z, bf16lo(b.y), s);
  s = fmaf(h0.w, bf16hi(b.y), s);
  s = fmaf(h1.x, bf16lo(b.z), s);
  s = fmaf(h1.y, bf16hi(b.z), s);
  s = fmaf(h1.z, bf16lo(b.w), s);
  s = fmaf(h1.w, bf16hi(b.w), s);
  return s;
}

template <int RMAX, int MODE, class Tables>
__global__ void __launch_bounds__(kThreads) delta_cluster_kernel(const DeltaArgs a, const Tables tb) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int key = (int)cluster_index_x();
  const uint32_t crank = cluster_rank();
  uint32_t ncta;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(ncta));

  __shared__ SlotView v;
  if (tid == 0) {
    uint32_t bad = 0;
    tb.resolve(key, a.sl.S, MODE, v, bad);
    if (bad && crank == 0) set_error(a.err, bad);
  }
  __syncthreads();
  if (v.nact == 0) return;  // the same decision in every CTA of the cluster

  const SmemPlan plan = smem_plan(a.row_cap, a.sr_max, a.ks, MODE);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  int* prow = reinterpret_cast<int*>(smem + 16);  // this pass's row ids
  int* rows_s = reinterpret_cast<int*>(smem + plan.rows_off);
  float* P = reinterpret_cast<float*>(smem + plan.P_off);
  float* H = reinterpret_cast<float*>(smem + plan.H_off);
  __nv_bfloat16* As = reinterpret_cast<__nv_bfloat16*>(smem + plan.A_off);
  __nv_bfloat16* Xs = reinterpret_cast<__nv_bfloat16*>(smem + plan.X_off);
  __shared__ int warp_cnt[kWarps];

  // ---- the key's rows, in ascending row order --------------------------
  int nrows;
  const int* rows;
  if (a.perm) {
    const int s0 = a.seg_start[key];
    nrows = a.seg_start[key + 1] - s0;
    rows = a.perm + s0;
  } else {
    int total = 0;
    bool bad_slot = false;
    for (int base = 0; base < a.n; base += kThreads) {
      const int i = base + tid;
      const int s = (i < a.n) ? a.seq_slot[i] : -1;
      const bool hit = (s == key);
      bad_slot |= (s >= a.n_keys);
      const unsigned m = __ballot_sync(0xffffffffu, hit);
      if (lane == 0) warp_cnt[warp] = __popc(m);
      __syncthreads();
      int before = total, sum = 0;
      for (int w = 0; w < kWarps; ++w) {
        before += (w < warp) ? warp_cnt[w] : 0;
        sum += warp_cnt[w];
      }
      if (hit) rows_s[before + __popc(m & ((1u << lane) - 1u))] = i;
      total += sum;
      __syncthreads();
    }
    if (key == 0 && crank == 0 && __syncthreads_or(bad_slot) && tid == 0)
      set_error(a.err, LORA_DEV_ERR_SLOT);
    nrows = total;
    rows = rows_s;
  }
  if (nrows == 0) return;  // uniform across the cluster

  const int R = a.R;
  const int SRa = v.nact * R;
  const int k_lo = (int)crank * a.kc;
  const int k_hi = min(a.k_in, k_lo + a.kc);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  uint32_t phase = 0;
  bool timed_out = false;

  for (int p0 = 0; p0 < nrows; p0 += kRowsPerPass) {
    const int nr = min(kRowsPerPass, nrows - p0);
    __syncthreads();  // the previous pass's readers of prow are done
    if (tid < nr) prow[tid] = rows[p0 + tid];
    if (MODE != kModeExpand)
      for (int i = tid; i < nr * SRa; i += kThreads) P[i] = 0.0f;

    if (MODE != kModeExpand) {
      // ---- shrink over this CTA's k-range ---------------------------------
      for (int k0 = k_lo; k0 < k_hi; k0 += a.ks) {
        const int kw = min(a.ks, k_hi - k0);
        __syncthreads();  // stage buffers free, prow / P visible
        if (warp == 0) {
          if (lane == 0) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar, (uint32_t)((SRa + nr) * kw * 2));
          }
          __syncwarp();
          for (int t = lane; t < SRa + nr; t += 32) {
            const __nv_bfloat16* src;
            __nv_bfloat16* dst;
            if (t < SRa) {
              const int jj = t / R, q = t - jj * R;
              src = v.A[v.act_slice[jj]] + (size_t)q * a.k_in + k0;
              dst = As + (size_t)t * a.ks;
            } else {
              const int r = t - SRa;
              src = a.x + tb.x_row(prow[r]) * a.ld_x + k0;
              dst = Xs + (size_t)r * a.ks;
            }
            bulk_g2s(dst, src, (uint32_t)kw * 2u, bar);
          }
        }
        if (!mbar_wait_bounded(bar, phase)) timed_out = true;
        phase ^= 1u;
        for (int pr = warp; pr < SRa; pr += kWarps) {
          float acc[kRowsPerPass];
#pragma unroll
          for (int r = 0; r < kRowsPerPass; ++r) acc[r] = 0.0f;
          for (int kv = lane * 8; kv < kw; kv += 256) {
            const uint4 av = *reinterpret_cast<const uint4*>(As + (size_t)pr * a.ks + kv);
#pragma unroll
            for (int r = 0; r < kRowsPerPass; ++r)
              if (r < nr)
                acc[r] += dot8(av, *reinterpret_cast<const uint4*>(Xs + (size_t)r * a.ks + kv));
          }
#pragma unroll
          for (int r = 0; r < kRowsPerPass; ++r) {
            if (r < nr) {
              const float s = warp_sum(acc[r]);
              if (lane == 0) P[r * SRa + pr] += s;
            }
          }
        }
      }
      __syncthreads();
      // ---- the CS partials meet in every CTA through DSMEM ----------------
      cluster_arrive();
      cluster_wait();
      const uint32_t P_addr = smem_addr(P);
      for (int i = tid; i < nr * SRa; i += kThreads) {
        float s = 0.0f;
        for (uint32_t c = 0; c < ncta; ++c) s += dsmem_ld_f32(dsmem_map(P_addr + 4u * i, c));
        H[i] = s;
      }
      __syncthreads();
      cluster_arrive();  // this CTA is done reading the others' partials
    } else {
      __syncthreads();
      for (int i = tid; i < nr * SRa; i += kThreads) {
        const int r = i / SRa, t = i - r * SRa, jj = t / R, q = t - jj * R;
        const int j = v.act_slice[jj];
        H[i] = a.h[((size_t)j * a.n + prow[r]) * R + q];
      }
      __syncthreads();
    }

    if (MODE == kModeShrink) {
      // h[j, row, q] += scale * H, the cluster's CTAs splitting the entries.
      for (int i = (int)crank * kThreads + tid; i < nr * SRa; i += (int)ncta * kThreads) {
        const int r = i / SRa, t = i - r * SRa, jj = t / R, q = t - jj * R;
        const int j = v.act_slice[jj];
        float* dst = a.h + ((size_t)j * a.n + prow[r]) * R + q;
        *dst = *dst + H[i] * v.scale;
      }
    } else if (!timed_out) {
      // ---- expand + fold over this CTA's columns --------------------------
      const int cb = (int)crank * a.cpc;
      const int ce = min(a.sl.n_cols, cb + a.cpc);
      for (int c2 = cb + 2 * tid; c2 < ce; c2 += 2 * kThreads) {
        int j = 0;
#pragma unroll
        for (int jj = 1; jj < kMaxSlices; ++jj)
          if (jj < a.sl.S && c2 >= a.rel[jj]) j = jj;
        const int ja = v.ja[j];
        if (ja < 0) continue;
        const int cl = c2 - a.rel[j];
        const __nv_bfloat16* b0 = v.B[j] + (size_t)cl * R;
        uint4 bq0[RMAX / 8], bq1[RMAX / 8];
#pragma unroll
        for (int u = 0; u < RMAX / 8; ++u) {
          if (u * 8 < R) {
            bq0[u] = ldg_nc_v4(b0 + u * 8);
            bq1[u] = ldg_nc_v4(b0 + R + u * 8);
          }
        }
        const float* Hj = H + ja * R;
        for (int r = 0; r < nr; ++r) {
          const float* hr = Hj + r * SRa;
          float d0 = 0.0f, d1 = 0.0f;
#pragma unroll
          for (int u = 0; u < RMAX / 8; ++u) {
            if (u * 8 < R) {
              d0 += dot8h(hr + u * 8, bq0[u]);
              d1 += dot8h(hr + u * 8, bq1[u]);
            }
          }
          const float v0 = v.scale * d0, v1 = v.scale * d1;
          uint32_t* o = reinterpret_cast<uint32_t*>(a.out + tb.out_row(prow[r]) * a.ld_out +
                                                    a.sl.off[j] + cl);
          if (a.add_inputs) {
            const uint32_t ov = *o;
            *o = pack_bf16x2(bf16lo(ov) + v0, bf16hi(ov) + v1);
          } else {
            *o = pack_bf16x2(v0, v1);
          }
        }
      }
    }
    if (MODE != kModeExpand) cluster_wait();  // peers done with this CTA's partials
  }
  if (timed_out && tid == 0) set_error(a.err, LORA_DEV_ERR_TIMEOUT);
}

// Zeros for the MoE pairs that get no delta (the no-key bucket).
__global__ void zero_rows_kernel(__nv_bfloat16* out, int64_t ld_out, int width,
                                 const int32_t* perm, const int32_t* seg_start, int bucket) {
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
