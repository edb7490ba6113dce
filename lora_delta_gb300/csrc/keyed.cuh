// The routed delta for many keys with a few dozen rows each (the routed-MoE
// deltas: "flashinfer.fused_moe.bgmv_moe_gemm1_lora_delta" and the in-place
// w13 / w2 deltas of "punica_base.py"): one CTA per key, which streams the
// key's whole A through a deep cp.async ring, then its B through the same
// ring for the expand.  There are hundreds of keys, so the grid fills the GPU without
// splitting a key over a cluster, and no partial sums cross CTAs.
//
// Per key (rows from the routing sort, in passes of 32):
//   * shrink: k_in in chunks of 64 columns; stage s of a kKeyStages ring holds
//     the chunk of the key's active (slice, rank) A rows and of the pass's x
//     rows.  Every thread copies one fixed 16-byte column of one A row and of
//     one x row per stage (its source pointers are set once per key), so the
//     copy issue costs a few instructions per stage, and kKeyStages - 1
//     stages stay in flight.  The A rows of the first stages are requested
//     before the grid dependency wait: adapter weights are never written by
//     the preceding kernel.  Warps own (16 pairs x 16 rows) tiles of the
//     product and split the k-steps of a chunk when there are fewer tiles
//     than warps; mma.sync m16n8k16, fp32 accumulate.
//   * the k-group partials meet in shared memory as the fp32 h [rows][pairs];
//   * expand + fold: the key's B rows (and, in place, the pass's out
//     segments) go through the idle ring in (slice, column chunk) items,
//     double-buffered in its two halves; every warp takes 8-column tiles of
//     the chunk, h as a bf16 (hi, lo) pair on the A side (rows), B fragments
//     by ldmatrix, then RN_bf16(out + scale * w_row * d) stored in place (or
//     RN_bf16(scale * w_row * d) without add_inputs).
#pragma once

#include "bgmv.cuh"
#include "common.cuh"

namespace lora {

constexpr int kKeyThreads = 256;
constexpr int kKeyWarps = kKeyThreads / 32;
constexpr int kKeyRows = 32;              // rows per pass
constexpr int kKeyKC = 64;                // k columns per stage
constexpr int kKeyStages = 5;             // ring depth
constexpr int kKeyStride = kKeyKC + 8;    // padded row (elements): ldmatrix conflict-free
constexpr int kKeyMaxSR = 64;             // largest S * R (rounded to 16) this kernel takes

// 16-byte asynchronous global -> shared copy to a shared-window address.
__device__ __forceinline__ void cp_async16_s(uint32_t saddr, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(gsrc) : "memory");
}

// Shared-memory plan (bytes), identical on host and device.
struct KeySmem {
  int stage_bytes, ring_off, ring_bytes, p_off, h_off, total;
};
__host__ __device__ inline KeySmem key_smem(int sr16) {
  KeySmem p;
  p.stage_bytes = (sr16 + kKeyRows) * kKeyStride * 2;
  p.ring_off = 0;
  // at least the ring of S * R = 32: the expand stages its B / out chunks in
  // the two halves of this region, and a small S * R has a long expand
  p.ring_bytes = kKeyStages * p.stage_bytes;
  const int min_ring = kKeyStages * (32 + kKeyRows) * kKeyStride * 2;
  if (p.ring_bytes < min_ring) p.ring_bytes = min_ring;
  int o = p.ring_bytes;
  o = (o + 127) / 128 * 128;
  p.p_off = o;  // k-group partials [G - 1][rows][sr16] (group 0 writes h directly)
  const int mt = sr16 / 16;
  const int units = mt * 2;
  const int G = units >= kKeyWarps ? 1 : kKeyWarps / units;
  o += (G - 1) * kKeyRows * sr16 * 4;
  p.h_off = o;
  o += kKeyRows * sr16 * 4 + 128;  // (+ slack: no guarded read of h can leave the plan)
  p.total = o;
  return p;
}

template <int RMAX, class Tables>
__global__ void __launch_bounds__(kKeyThreads, RMAX <= 16 ? 4 : 3)
    delta_key_kernel(const DeltaArgs a, const Tables tb, int zero_ctas, int halves) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ SlotView v;
  __shared__ int prow[kKeyRows];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3;
  // CTA (key, half): with halves == 2, CTAs n_keys .. 2 n_keys - 1 take the
  // odd passes of their key (keys of more than one pass share the work; for
  // the others the second CTA ends at once), the rest the even passes.
  const int nk_ctas = a.n_keys * halves;
  const int half = (int)blockIdx.x >= a.n_keys && (int)blockIdx.x < nk_ctas ? 1 : 0;
  const int key = (int)blockIdx.x < nk_ctas ? (int)blockIdx.x - half * a.n_keys
                                            : a.n_keys + ((int)blockIdx.x - nk_ctas);

  if (key >= a.n_keys) {
    // The last zero_ctas CTAs write zeros on the rows of the no-key bucket
    // (MoE pairs without an adapter, when the output is written fresh).
    cudaTriggerProgrammaticLaunchCompletion();
    cudaGridDependencySynchronize();
    const int z0 = a.seg_start[a.n_keys], z1 = a.seg_start[a.n_keys + 1];
    const int vpr = a.sl.n_cols / 8;
    const int64_t total = (int64_t)(z1 - z0) * vpr;
    for (int64_t i = (int64_t)(key - a.n_keys) * kKeyThreads + tid; i < total;
         i += (int64_t)zero_ctas * kKeyThreads) {
      const int r = (int)(i / vpr), c = (int)(i - (int64_t)r * vpr);
      *reinterpret_cast<uint4*>(a.out + tb.out_row(a.perm[z0 + r]) * a.ld_out + c * 8) =
          make_uint4(0, 0, 0, 0);
    }
    return;
  }

  if (tid == 0) {
    uint32_t bad = 0;
    tb.resolve(key, a.sl.S, kModeFused, v, bad);
    if (bad) set_error(a.err, bad);
  }
  __syncthreads();
  const int R = a.R;
  const int SRa = v.nact * R;
  const int SR16 = (a.sr_max + 15) / 16 * 16;
  const KeySmem plan = key_smem(SR16);
  uint8_t* ring = smem + plan.ring_off;
  float* P = reinterpret_cast<float*>(smem + plan.p_off);
  float* H = reinterpret_cast<float*>(smem + plan.h_off);
  const int nchunks = (a.k_in + kKeyKC - 1) / kKeyKC;

  // this thread's copy slots: 16-byte column `cq` of A rows ar0 (and ar0 + 32)
  // and of x row `ar0` of every stage
  const int cq = tid & 7, ar0 = tid >> 3;
  const __nv_bfloat16* asrc[2] = {nullptr, nullptr};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = ar0 + 32 * h;
    if (t < SRa) {
      const int jj = t / R, q = t - jj * R;
      asrc[h] = v.A[v.act_slice[jj]] + (size_t)q * a.k_in + cq * 8;
    }
  }
  // Stage layout: A rows [SR16][kKeyStride], then x rows [kKeyRows][kKeyStride].
  // Addresses are 32-bit shared-window offsets, advanced per stage without
  // divisions: the copy issue and the fragment loads cost a few integer
  // instructions per chunk.
  const uint32_t ring_s = smem_addr(ring);
  const uint32_t sbytes = (uint32_t)plan.stage_bytes;
  const uint32_t ring_end = ring_s + kKeyStages * sbytes;
  const uint32_t a_off = (uint32_t)(ar0 * kKeyStride + cq * 8) * 2u;
  const uint32_t a_off2 = a_off + 32u * kKeyStride * 2u;
  const uint32_t x_off = (uint32_t)((SR16 + ar0) * kKeyStride + cq * 8) * 2u;
  const int full = a.k_in / kKeyKC;  // chunks with all 64 columns
  const int tail_kw = a.k_in - full * kKeyKC;
  const bool tail_col = cq * 8 < tail_kw;  // this thread's column exists in the last chunk
  auto next_slot = [&](uint32_t sb) { sb += sbytes; return sb == ring_end ? ring_s : sb; };
  // copies of chunk c's A rows into the slot at sb (the x rows follow separately)
  auto copy_a = [&](int c, uint32_t sb) {
    if (c < full || tail_col) {
      const size_t k0 = (size_t)c * kKeyKC;
      if (asrc[0]) cp_async16_s(sb + a_off, asrc[0] + k0);
      if (asrc[1]) cp_async16_s(sb + a_off2, asrc[1] + k0);
    }
  };

  const bool early = a.early && v.nact > 0 && half == 0;
  if (early) {  // A rows of the first stages, before the dependency wait
    uint32_t sb = ring_s;
    for (int c = 0; c < kKeyStages - 1 && c < nchunks; ++c, sb += sbytes) copy_a(c, sb);
    cp_async_commit();
    // ... and the whole of the key's A and B on their way to L2: the routing
    // sort this launch waits for leaves DRAM nearly idle
    if (warp == kKeyWarps - 1 && lane < a.sl.S && v.ja[lane] >= 0) {
      bulk_prefetch_l2(v.A[lane], (uint32_t)(R * a.k_in * 2));
      bulk_prefetch_l2(v.B[lane], (uint32_t)(a.sl.width[lane] * R * 2));
    }
  }
  cudaTriggerProgrammaticLaunchCompletion();
  cudaGridDependencySynchronize();
  const int s0 = a.seg_start[key];
  const int nrows = v.nact > 0 ? a.seg_start[key + 1] - s0 : 0;
  if (nrows <= half * kKeyRows || nrows < a.min_rows || nrows >= a.max_rows) {
    if (early) cp_async_wait<0>();  // no copy may land in a CTA that has exited
    return;
  }
  const int* rows = a.perm + s0;

  // shrink work split: units of (16 pairs x 16 rows), k-groups over the warps
  const int mt = SR16 / 16, units = mt * 2;
  const int G = units >= kKeyWarps ? 1 : kKeyWarps / units;
  const int my_u = warp % units, my_g = warp / units;
  const bool mma_warp = warp < G * units;
  const int my_m = my_u >> 1, my_rg = my_u & 1;
  // ldmatrix row addresses of this lane inside a stage (bytes)
  const uint32_t a_frag =
      (uint32_t)((my_m * 16 + (((lane >> 3) & 1) << 3) + (lane & 7)) * kKeyStride +
                 ((lane >> 4) << 3)) * 2u;
  const uint32_t x_frag =
      (uint32_t)((SR16 + my_rg * 16 + ((lane >> 4) << 3) + (lane & 7)) * kKeyStride +
                 ((lane >> 3) & 1) * 8) * 2u;
  constexpr int KS = RMAX / 16;
  bool first_pass = true;

  for (int p0 = half * kKeyRows; p0 < nrows; p0 += halves * kKeyRows) {
    const int nr = min(kKeyRows, nrows - p0);
    if (!first_pass) __syncthreads();  // the previous pass is done with prow, H and the ring
    if (tid < nr) prow[tid] = rows[p0 + tid];
    __syncthreads();
    // L2 prefetch of the pass's expand operands (B of the key; out rows)
    if (warp == kKeyWarps - 1) {
      if (first_pass && !early)  // (prefetched before the dependency wait otherwise)
        for (int j = lane; j < a.sl.S; j += 32)
          if (v.ja[j] >= 0)
            bulk_prefetch_l2(v.B[j], (uint32_t)(a.sl.width[j] * R * 2));
      if (a.add_inputs)
        for (int r = lane; r < nr; r += 32)
          for (int j = 0; j < a.sl.S; ++j)
            if (v.ja[j] >= 0 && a.sl.width[j] > 0)
              bulk_prefetch_l2(a.out + tb.out_row(prow[r]) * a.ld_out + a.sl.off[j],
                               (uint32_t)(a.sl.width[j] * 2));
    }
    const __nv_bfloat16* xsrc =
        ar0 < nr ? a.x + tb.x_row(prow[ar0]) * a.ld_x + cq * 8 : nullptr;
    // chunk c's A (unless already requested) and x rows into the slot at sb;
    // the partial last chunk also zeroes its columns [kw, round16(kw))
    auto issue = [&](int c, uint32_t sb, bool with_a) {
      if (with_a) copy_a(c, sb);
      if (xsrc && (c < full || tail_col)) cp_async16_s(sb + x_off, xsrc + (size_t)c * kKeyKC);
      if (c == full && (tail_kw & 15)) {
        __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(ring + (sb - ring_s));
        for (int i = tid; i < SR16 + kKeyRows; i += kKeyThreads)
          *reinterpret_cast<uint4*>(st + (size_t)i * kKeyStride + tail_kw) = make_uint4(0, 0, 0, 0);
      }
    };

    // ---- ring prologue: chunks 0 .. kKeyStages - 2 ----------------------
    const bool a_done = early && first_pass;
    uint32_t sb_issue = ring_s;
    for (int c = 0; c < kKeyStages - 1; ++c) {
      if (c < nchunks) issue(c, sb_issue, !a_done);
      cp_async_commit();  // (empty groups keep the count uniform)
      sb_issue = next_slot(sb_issue);
    }
    first_pass = false;

    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    const bool rg_live = my_rg * 16 < nr;  // (warp-uniform)
    uint32_t sb = ring_s;
    for (int c = 0; c < nchunks; ++c) {
      cp_async_wait<kKeyStages - 2>();  // chunk c landed
      __syncthreads();                  // ... for every thread; the slot of c - 1 is free
      if (c + kKeyStages - 1 < nchunks) issue(c + kKeyStages - 1, sb_issue, true);
      cp_async_commit();
      sb_issue = next_slot(sb_issue);
      if (mma_warp && rg_live) {
        const uint32_t aaddr = sb + a_frag, xaddr = sb + x_frag;
        const int ksteps = c < full ? kKeyKC / 16 : (tail_kw + 15) / 16;
        for (int ks = my_g; ks < ksteps; ks += G) {
          uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
          ldsm_x4(aaddr + ks * 32, a0, a1, a2, a3);
          ldsm_x4(xaddr + ks * 32, b0, b1, b2, b3);
          mma_16816(&acc[0], a0, a1, a2, a3, b0, b1);
          mma_16816(&acc[4], a0, a1, a2, a3, b2, b3);
        }
      }
      sb = next_slot(sb);
    }
    cp_async_wait<0>();  // (only empty groups remain)

    // ---- k-group partials -> h [rows][pairs] -----------------------------
    if (mma_warp && rg_live) {
      float* dst = my_g == 0 ? H : P + (size_t)(my_g - 1) * kKeyRows * SR16;
      const int pr = my_m * 16 + gq;       // pair of acc[0], acc[1]
      const int xr = my_rg * 16 + 2 * tq;  // x row of acc[0]
      dst[(xr) * SR16 + pr] = acc[0];
      dst[(xr + 1) * SR16 + pr] = acc[1];
      dst[(xr) * SR16 + pr + 8] = acc[2];
      dst[(xr + 1) * SR16 + pr + 8] = acc[3];
      dst[(xr + 8) * SR16 + pr] = acc[4];
      dst[(xr + 9) * SR16 + pr] = acc[5];
      dst[(xr + 8) * SR16 + pr + 8] = acc[6];
      dst[(xr + 9) * SR16 + pr + 8] = acc[7];
    }
    __syncthreads();
    if (G > 1) {
      for (int i = tid; i < nr * SR16; i += kKeyThreads) {
        float s = H[i];
        for (int g = 1; g < G; ++g) s += P[(size_t)(g - 1) * kKeyRows * SR16 + i];
        H[i] = s;
      }
      __syncthreads();
    }

    // ---- expand + fold ------------------------------------------------------
    // The key's B goes through the idle ring in (slice, column chunk) items,
    // double-buffered in its two halves; fragments come from shared memory
    // by ldmatrix (B rows padded to R + 8 elements: conflict-free), so a
    // chunk costs one copy round trip instead of one per batch of tiles.
    const int nm = nr > 16 ? 2 : 1;  // 16-row m-tiles of the pass
    int orow[2][2];  // (row < n <= 2^30)
    float sc[2][2];
    bool ok[2][2];
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = mi * 16 + gq + 8 * h;
        ok[mi][h] = r < nr;
        orow[mi][h] = ok[mi][h] ? (int)tb.out_row(prow[r]) : 0;
        sc[mi][h] = ok[mi][h] ? v.scale * tb.row_weight(prow[r]) : 0.f;
      }
    // A half holds the chunk's B rows [cc][bstride] and, with add_inputs, its
    // out segments [kKeyRows][ostride] (a stride of 4 words mod 8: the
    // fragment reads are conflict-free); cc is chosen so that both fit.
    const int bstride = R + 8;
    const uint32_t half_bytes = ((uint32_t)plan.ring_bytes / 2u) & ~15u;
    const int per_col = bstride * 2 + (a.add_inputs ? kKeyRows * 2 : 0);
    const int cc = (int)((half_bytes - (a.add_inputs ? kKeyRows * 32u : 0u)) / (uint32_t)per_col) / 8 * 8;
    const int ostride = cc + (cc % 16 == 0 ? 8 : 16);  // elements, 8 mod 16: <= cc + 16
    const uint32_t o_off = (uint32_t)(cc * bstride * 2);
    const int vpc = R / 8;  // 16-byte pieces per B column
    // (a power of two for R = 8, 16, 32, 64: shifts instead of divisions)
    const int vpc_shift = (vpc & (vpc - 1)) == 0 ? __ffs(vpc) - 1 : -1;
    auto first_slice = [&](int j) {
      while (j < a.sl.S && v.ja[j] < 0) ++j;
      return j;
    };
    auto issue_b = [&](int j, int c0, uint32_t hb) {
      const int cw = min(cc, a.sl.width[j] - c0);
      const __nv_bfloat16* src = v.B[j] + (size_t)c0 * R;
      for (int i = tid; i < cw * vpc; i += kKeyThreads) {
        const int col = vpc_shift >= 0 ? i >> vpc_shift : i / vpc, part = i - col * vpc;
        cp_async16_s(hb + (uint32_t)(col * bstride + part * 8) * 2u, src + (size_t)col * R + part * 8);
      }
      if (a.add_inputs) {  // a warp per out row, its lanes over the row's pieces
        const int ppr = cw / 8;  // pieces per out row
        for (int r = warp; r < nr; r += kKeyWarps) {
          const __nv_bfloat16* orow = a.out + tb.out_row(prow[r]) * a.ld_out + a.sl.off[j] + c0;
          const uint32_t dst = hb + o_off + (uint32_t)(r * ostride) * 2u;
          for (int q = lane; q < ppr; q += 32) cp_async16_s(dst + (uint32_t)q * 16u, orow + q * 8);
        }
      }
    };
    // ldmatrix row address of this lane inside a chunk (matrix lane / 8 is k
    // block lane / 8 of the tile's 8 columns)
    const uint32_t b_frag = (uint32_t)((lane & 7) * bstride + ((lane >> 3) & (KS * 2 - 1)) * 8) * 2u;
    int j = first_slice(0), c0 = 0, hsel = 0;
    if (j < a.sl.S) issue_b(j, c0, ring_s);
    cp_async_commit();
    int ja_split = -1;  // slice whose h fragments are in registers
    uint32_t ahi[2][KS][4], alo[2][KS][4];
    while (j < a.sl.S) {
      // the next item into the other half
      int jn = j, cn = c0 + cc;
      if (cn >= a.sl.width[j]) {
        cn = 0;
        jn = first_slice(j + 1);
      }
      if (jn < a.sl.S) issue_b(jn, cn, ring_s + (hsel ^ 1) * half_bytes);
      cp_async_commit();
      cp_async_wait<1>();  // this item's chunk landed
      __syncthreads();
      const int ja = v.ja[j];
      if (ja != ja_split) {  // h of the slice as bf16 (hi, lo) A fragments
        ja_split = ja;
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
          const float* hb = H + ja * R + 2 * tq + (mi * 16 + gq) * SR16;
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            const bool lo_ok = mi < nm && kk * 16 < R, hi_ok = mi < nm && kk * 16 + 8 < R;
            const float* h0 = hb + kk * 16;
            const float* h1 = h0 + 8 * SR16;
            split_bf16x2(lo_ok ? h0[0] : 0.f, lo_ok ? h0[1] : 0.f, ahi[mi][kk][0], alo[mi][kk][0]);
            split_bf16x2(lo_ok ? h1[0] : 0.f, lo_ok ? h1[1] : 0.f, ahi[mi][kk][1], alo[mi][kk][1]);
            split_bf16x2(hi_ok ? h0[8] : 0.f, hi_ok ? h0[9] : 0.f, ahi[mi][kk][2], alo[mi][kk][2]);
            split_bf16x2(hi_ok ? h1[8] : 0.f, hi_ok ? h1[9] : 0.f, ahi[mi][kk][3], alo[mi][kk][3]);
          }
        }
      }
      const int cw = min(cc, a.sl.width[j] - c0);
      const uint32_t hbase = ring_s + hsel * half_bytes + b_frag;
      const int64_t cbase = a.sl.off[j] + c0 + 2 * tq;
      const __nv_bfloat16* os = reinterpret_cast<const __nv_bfloat16*>(
          ring + (size_t)hsel * half_bytes + o_off) + 2 * tq;
      // this lane's four output row pointers for the item, so that the tile
      // loop only adds the tile's column (rank <= 16: the larger instance
      // has no registers to spare for them)
      constexpr bool kHoist = RMAX <= 16;
      __nv_bfloat16* op[2][2];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          op[mi][h] = kHoist ? a.out + (int64_t)orow[mi][h] * a.ld_out + cbase : nullptr;
      for (int t = warp; t < cw / 8; t += kKeyWarps) {
        uint32_t bf[KS][2];
        const uint32_t ba = hbase + (uint32_t)(t * 8 * bstride) * 2u;
        if (KS == 1) {
          ldsm_x2(ba, bf[0][0], bf[0][1]);
        } else {
          ldsm_x4(ba, bf[0][0], bf[0][1], bf[KS - 1][0], bf[KS - 1][1]);
        }
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          if (kk * 16 + 8 >= R) bf[kk][1] = 0u;  // k past the rank: padding
        }
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
          if (mi >= nm) continue;
          float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            if (kk * 16 < R) {
              mma_16816(d, ahi[mi][kk][0], ahi[mi][kk][1], ahi[mi][kk][2], ahi[mi][kk][3],
                        bf[kk][0], bf[kk][1]);
              mma_16816(d, alo[mi][kk][0], alo[mi][kk][1], alo[mi][kk][2], alo[mi][kk][3],
                        bf[kk][0], bf[kk][1]);
            }
          }
#pragma unroll
          for (int h = 0; h < 2; ++h)
            if (ok[mi][h]) {
              const uint32_t o =
                  a.add_inputs ? *reinterpret_cast<const uint32_t*>(
                                     os + (mi * 16 + gq + 8 * h) * ostride + t * 8)
                               : 0u;
              *reinterpret_cast<uint32_t*>(
                  (kHoist ? op[mi][h] : a.out + (int64_t)orow[mi][h] * a.ld_out + cbase) + t * 8) =
                  pack_bf16x2(bf16lo(o) + sc[mi][h] * d[2 * h], bf16hi(o) + sc[mi][h] * d[2 * h + 1]);
            }
        }
      }
      __syncthreads();  // this half is free for the item after next
      j = jn;
      c0 = cn;
      hsel ^= 1;
    }
    cp_async_wait<0>();  // (an empty group)
  }
}

}  // namespace lora
