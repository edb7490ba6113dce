// Segmented (SGMV) path of the routed delta on the 5th-generation tensor cores
// (tcgen05 MMA, accumulators in tensor memory), for adapter keys with many
// rows ("punica_base.py", prefill_metadata / add_lora_linear; "Module
// lora_delta", lora_gemv_max_m: below a row threshold the GEMV-style path is
// cheaper, above it a real tensor-core GEMM is).
//
// The rows of a key are taken in the routing kernel's stable order and cut
// into tiles of 128 rows (the last one ragged).  Two kernels:
//   * shrink: one CTA per tile computes h[tile rows, active (slice, rank)
//     pairs] = x[rows] A^T over all of k_in: 64-wide k-blocks of the gathered
//     x rows and of the key's A rows are staged by cp.async into 128-byte
//     swizzled shared-memory tiles (4-stage ring), one thread issues the
//     M=128 MMAs, and h goes to the workspace in fp32;
//   * expand: one CTA per (tile, 128-column chunk of one slice) multiplies the
//     tile's h -- split into a bf16 (hi, lo) pair so the rank contraction keeps
//     ~fp32 accuracy -- by the chunk's B rows (both 128-byte swizzled tiles),
//     and folds scale * d into out in place, one rounding; the out segments
//     are staged in shared memory while the MMAs run.
// Every wait on an mbarrier is bounded; on a time-out the CTA records
// LORA_DEV_ERR_TIMEOUT, skips its writes and still releases its TMEM.
#pragma once

#include "bgmv.cuh"
#include "common.cuh"
#include "tc.cuh"

namespace lora {

constexpr int kTileRows = 128;      // MMA M
constexpr int kSgmvThreads = 128;   // 4 warps = the 4 TMEM lane quarters
constexpr int kShrinkStages = 4;
constexpr int kExpandCols = 128;    // output columns per expand CTA
constexpr int kSgmvMaxSR = 256;     // MMA N of the shrink

struct SgmvTile {
  int key, pos0, rows, pad;
};

// ---------------------------------------------------------------- tiles --
// Tile list from the routing kernel's cluster starts: keys with at least
// min_rows rows get ceil(rows / 128) tiles.  One CTA.
__global__ void __launch_bounds__(256)
    sgmv_tiles_kernel(const int32_t* __restrict__ seg_start, int n_keys, int min_rows,
                      SgmvTile* __restrict__ tiles, int* __restrict__ n_tiles, int max_tiles) {
  __shared__ int warp_sums[8];
  cudaGridDependencySynchronize();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kpt = (n_keys + 255) / 256;
  const int k0 = min(n_keys, tid * kpt), k1 = min(n_keys, k0 + kpt);
  int mine = 0;
  for (int k = k0; k < k1; ++k) {
    const int c = seg_start[k + 1] - seg_start[k];
    if (c >= min_rows && c > 0) mine += (c + kTileRows - 1) / kTileRows;
  }
  int incl = mine;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  int base = incl - mine;
  for (int w = 0; w < warp; ++w) base += warp_sums[w];
  for (int k = k0; k < k1; ++k) {
    const int s0 = seg_start[k], c = seg_start[k + 1] - s0;
    if (c < min_rows || c <= 0) continue;
    for (int r = 0; r < c; r += kTileRows) {
      if (base < max_tiles) tiles[base] = SgmvTile{k, s0 + r, min(kTileRows, c - r), 0};
      ++base;
    }
  }
  if (tid == 255) *n_tiles = min(base, max_tiles);
}

struct SgmvArgs {
  __nv_bfloat16* out;
  int64_t ld_out;
  const __nv_bfloat16* x;
  int64_t ld_x;
  int k_in;
  const int32_t* perm;
  const SgmvTile* tiles;
  const int* n_tiles;
  float* hbuf;  // [sorted rows, hs] fp32
  int hs;       // row stride of hbuf (S * R rounded up to 16)
  int R;
  Slices sl;
  int rel[kMaxSlices + 1];
  int chunk0[kMaxSlices + 1];  // first expand chunk of each slice; chunk0[S] = chunks total
  int add_inputs;
  uint32_t* err;
};

__device__ __forceinline__ void cp_async16_zfill(void* smem_dst, const void* gsrc, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(smem_dst)),
               "l"(gsrc), "r"(valid ? 16 : 0)
               : "memory");
}

// ---------------------------------------------------------------- shrink --
template <class Tables>
__global__ void __launch_bounds__(kSgmvThreads)
    sgmv_shrink_kernel(const SgmvArgs a, const Tables tb) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ SlotView v;
  __shared__ uint32_t taddr_s;
  __shared__ __align__(8) uint64_t mma_bar[kShrinkStages];
  __shared__ __align__(8) uint64_t done_bar;
  cudaGridDependencySynchronize();
  const int tile_id = blockIdx.x;
  if (tile_id >= *a.n_tiles) return;
  const SgmvTile tile = a.tiles[tile_id];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  if (tid == 0) {
    uint32_t bad = 0;
    tb.resolve(tile.key, a.sl.S, kModeFused, v, bad);
    for (int s = 0; s < kShrinkStages; ++s) mbar_init(&mma_bar[s], 1);
    mbar_init(&done_bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  const int R = a.R;
  const int SRa = v.nact * R;
  if (SRa == 0) return;
  const int N = (SRa + 15) / 16 * 16;
  uint32_t ncols = 32;
  while ((int)ncols < N) ncols <<= 1;
  if (warp == 0) tc::tmem_alloc(&taddr_s, ncols);

  const int xbytes = kTileRows * 128, abytes = N * 128;
  const int stage_bytes = xbytes + abytes;  // multiple of 1024
  const int nkb = (a.k_in + 63) / 64;

  // one 64-wide k-block of the gathered x rows and of the A rows, zero-filled
  // past the tile's rows, the key's pairs and k_in
  auto load_block = [&](int kb, int s) {
    uint8_t* xs = smem + (size_t)s * stage_bytes;
    uint8_t* as = xs + xbytes;
    const int kbase = kb * 64;
    for (int i = tid; i < (kTileRows + N) * 8; i += kSgmvThreads) {
      const int r = i >> 3, c = i & 7;
      const int k = kbase + c * 8;
      const bool kin = k < a.k_in;
      if (r < kTileRows) {
        const bool ok = kin && r < tile.rows;
        const __nv_bfloat16* src =
            ok ? a.x + tb.x_row(a.perm[tile.pos0 + r]) * a.ld_x + k : a.x;
        cp_async16_zfill(xs + tc::sw128_offset(r, c * 8), src, ok);
      } else {
        const int t = r - kTileRows;
        const bool ok = kin && t < SRa;
        const __nv_bfloat16* src = a.x;
        if (ok) {
          const int jj = t / R, q = t - jj * R;
          src = v.A[v.act_slice[jj]] + (size_t)q * a.k_in + k;
        }
        cp_async16_zfill(as + tc::sw128_offset(t, c * 8), src, ok);
      }
    }
  };

  for (int s = 0; s < kShrinkStages - 1; ++s) {
    if (s < nkb) load_block(s, s);
    cp_async_commit();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t taddr = taddr_s;
  const uint32_t idesc = tc::idesc_bf16_f32(kTileRows, N);
  bool ok = true;
  for (int kb = 0; kb < nkb; ++kb) {
    const int s = kb % kShrinkStages;
    cp_async_wait<kShrinkStages - 2>();  // block kb landed (this thread's copies)
    fence_proxy_async_smem();            // make them visible to the tensor core
    if (tid == 0 && kb >= 1) {           // the MMAs of block kb-1 released its stage
      const int sp = (kb - 1) % kShrinkStages;
      if (!mbar_wait_bounded(&mma_bar[sp], (uint32_t)(((kb - 1) / kShrinkStages) & 1))) ok = false;
    }
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
      const uint32_t xa = smem_addr(smem + (size_t)s * stage_bytes);
      const uint32_t aa = xa + xbytes;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        tc::mma_bf16(taddr, tc::sw128_desc(xa + ks * 32), tc::sw128_desc(aa + ks * 32), idesc,
                     (kb > 0 || ks > 0) ? 1u : 0u);
      tc::mma_commit(&mma_bar[s]);
    }
    const int nxt = kb + kShrinkStages - 1;  // refill the stage block kb-1 used
    if (nxt < nkb) load_block(nxt, nxt % kShrinkStages);
    cp_async_commit();
  }
  if (tid == 0) {
    tc::mma_commit(&done_bar);
    if (!mbar_wait_bounded(&done_bar, 0)) ok = false;
  }
  cp_async_wait<0>();
  __syncthreads();
  tc::fence_after_sync();
  const bool all_ok = __syncthreads_and(ok);
  if (!all_ok && tid == 0) set_error(a.err, LORA_DEV_ERR_TIMEOUT);
  // epilogue: TMEM row r -> hbuf[pos0 + r][0 .. SRa)
  if (all_ok) {
    const int r = warp * 32 + lane;
    float* dst = a.hbuf + (size_t)(tile.pos0 + r) * a.hs;
    for (int c = 0; c < N; c += 16) {
      float vals[16];
      tc::tmem_ld16(taddr + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, vals);
      if (r < tile.rows) {
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          if (c + i < SRa)
            *reinterpret_cast<float4*>(dst + c + i) =
                make_float4(vals[i], vals[i + 1], vals[i + 2], vals[i + 3]);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(taddr, ncols);
}

// ---------------------------------------------------------------- expand --
template <int RMAX, class Tables>
__global__ void __launch_bounds__(kSgmvThreads)
    sgmv_expand_kernel(const SgmvArgs a, const Tables tb, int n_chunks) {
  constexpr int KB = (RMAX + 63) / 64;  // 64-wide k-blocks of the rank
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ SlotView v;
  __shared__ uint32_t taddr_s;
  __shared__ __align__(8) uint64_t done_bar;
  __shared__ int orow_s[kTileRows];
  cudaGridDependencySynchronize();
  const int tile_id = blockIdx.x / n_chunks, chunk = blockIdx.x - tile_id * n_chunks;
  if (tile_id >= *a.n_tiles) return;
  const SgmvTile tile = a.tiles[tile_id];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int j = 0;
#pragma unroll
  for (int jj = 1; jj < kMaxSlices; ++jj)
    if (jj < a.sl.S && chunk >= a.chunk0[jj]) j = jj;
  const int c0 = (chunk - a.chunk0[j]) * kExpandCols;  // first column inside slice j
  const int nc = min(kExpandCols, a.sl.width[j] - c0);
  if (tid == 0) {
    uint32_t bad = 0;
    tb.resolve(tile.key, a.sl.S, kModeFused, v, bad);
    mbar_init(&done_bar, 1);
    fence_barrier_init();
  }
  for (int r = tid; r < kTileRows; r += kSgmvThreads)
    orow_s[r] = r < tile.rows ? (int)tb.out_row(a.perm[tile.pos0 + r]) : 0;
  __syncthreads();
  const int ja = v.ja[j];
  if (ja < 0 || nc <= 0) return;
  const int R = a.R;
  const int N = (nc + 15) / 16 * 16;
  uint8_t* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint8_t* hhi = smem;                                 // [KB][128 rows][128 B]
  uint8_t* hlo = hhi + KB * kTileRows * 128;
  uint8_t* bsm = hlo + KB * kTileRows * 128;           // [KB][kExpandCols rows][128 B]
  __nv_bfloat16* os = reinterpret_cast<__nv_bfloat16*>(bsm + KB * kExpandCols * 128);
  constexpr int kOStride = kExpandCols + 8;             // staged out row (elements)
  if (warp == 0) tc::tmem_alloc(&taddr_s, kExpandCols);

  // B rows of the chunk (zero past nc and past R inside the k-block)
  const __nv_bfloat16* bsrc = v.B[j] + (size_t)c0 * R;
  for (int i = tid; i < KB * kExpandCols * 8; i += kSgmvThreads) {
    const int kb = i / (kExpandCols * 8), rem = i - kb * kExpandCols * 8;
    const int c = rem >> 3, g = rem & 7, k = kb * 64 + g * 8;
    const bool ok = c < nc && k < R;
    cp_async16_zfill(bsm + (size_t)kb * kExpandCols * 128 + tc::sw128_offset(c, g * 8),
                     ok ? bsrc + (size_t)c * R + k : bsrc, ok);
  }
  cp_async_commit();
  // out segments of the tile's rows
  const int64_t ocol = a.sl.off[j] + c0;
  if (a.add_inputs) {
    for (int i = tid; i < tile.rows * (nc / 8); i += kSgmvThreads) {
      const int r = i / (nc / 8), g = i - r * (nc / 8);
      cp_async16(os + (size_t)r * kOStride + g * 8, a.out + (int64_t)orow_s[r] * a.ld_out + ocol + g * 8);
    }
  }
  cp_async_commit();
  // h of the tile's rows, slice ja, as a bf16 (hi, lo) pair
  for (int i = tid; i < KB * kTileRows * 8; i += kSgmvThreads) {
    const int kb = i / (kTileRows * 8), rem = i - kb * kTileRows * 8;
    const int r = rem >> 3, g = rem & 7, k = kb * 64 + g * 8;
    float hv[8];
    if (r < tile.rows && k < R) {
      const float* hp = a.hbuf + (size_t)(tile.pos0 + r) * a.hs + ja * R + k;
      const float4 h0 = *reinterpret_cast<const float4*>(hp);
      const float4 h1 = *reinterpret_cast<const float4*>(hp + 4);
      hv[0] = h0.x; hv[1] = h0.y; hv[2] = h0.z; hv[3] = h0.w;
      hv[4] = h1.x; hv[5] = h1.y; hv[6] = h1.z; hv[7] = h1.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) hv[e] = 0.0f;
    }
    uint4 hi, lo;
    split_bf16x2(hv[0], hv[1], hi.x, lo.x);
    split_bf16x2(hv[2], hv[3], hi.y, lo.y);
    split_bf16x2(hv[4], hv[5], hi.z, lo.z);
    split_bf16x2(hv[6], hv[7], hi.w, lo.w);
    const uint32_t off = (uint32_t)kb * kTileRows * 128 + tc::sw128_offset(r, g * 8);
    *reinterpret_cast<uint4*>(hhi + off) = hi;
    *reinterpret_cast<uint4*>(hlo + off) = lo;
  }
  cp_async_wait<1>();  // B rows landed (the out segments may still be in flight)
  fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t taddr = taddr_s;
  bool ok = true;
  if (tid == 0) {
    const uint32_t idesc = tc::idesc_bf16_f32(kTileRows, N);
    const int ksteps = (R + 15) / 16;
    for (int pass = 0; pass < 2; ++pass) {
      const uint8_t* hsrc = pass == 0 ? hhi : hlo;
      for (int s = 0; s < ksteps; ++s) {
        const int kb = s >> 2, ks = s & 3;
        const uint32_t ha = smem_addr(hsrc + (size_t)kb * kTileRows * 128) + ks * 32;
        const uint32_t ba = smem_addr(bsm + (size_t)kb * kExpandCols * 128) + ks * 32;
        tc::mma_bf16(taddr, tc::sw128_desc(ha), tc::sw128_desc(ba), idesc,
                     (pass > 0 || s > 0) ? 1u : 0u);
      }
    }
    tc::mma_commit(&done_bar);
    if (!mbar_wait_bounded(&done_bar, 0)) ok = false;
  }
  cp_async_wait<0>();  // out segments landed
  __syncthreads();
  tc::fence_after_sync();
  const bool all_ok = __syncthreads_and(ok);
  if (!all_ok && tid == 0) set_error(a.err, LORA_DEV_ERR_TIMEOUT);
  if (all_ok) {
    // epilogue: thread = tile row; RN_bf16(out + scale * d), 16 columns at a time
    const int r = warp * 32 + lane;
    const float sc = v.scale;
    __nv_bfloat16* orow = a.out + (int64_t)orow_s[r] * a.ld_out + ocol;
    const __nv_bfloat16* srow = os + (size_t)r * kOStride;
    for (int c = 0; c < N; c += 16) {
      float d[16];
      tc::tmem_ld16(taddr + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, d);
      if (r < tile.rows) {
#pragma unroll
        for (int h = 0; h < 16; h += 8) {
          if (c + h < nc) {
            uint4 o = make_uint4(0, 0, 0, 0);
            if (a.add_inputs) o = *reinterpret_cast<const uint4*>(srow + c + h);
            uint4 res;
            res.x = pack_bf16x2(bf16lo(o.x) + sc * d[h + 0], bf16hi(o.x) + sc * d[h + 1]);
            res.y = pack_bf16x2(bf16lo(o.y) + sc * d[h + 2], bf16hi(o.y) + sc * d[h + 3]);
            res.z = pack_bf16x2(bf16lo(o.z) + sc * d[h + 4], bf16hi(o.z) + sc * d[h + 5]);
            res.w = pack_bf16x2(bf16lo(o.w) + sc * d[h + 6], bf16hi(o.w) + sc * d[h + 7]);
            *reinterpret_cast<uint4*>(orow + c + h) = res;
          }
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(taddr, kExpandCols);
}

inline int sgmv_shrink_smem(int sr_max) {
  const int N = (sr_max + 15) / 16 * 16;
  return kShrinkStages * (kTileRows * 128 + N * 128) + 1024;
}
inline int sgmv_expand_smem(int R) {
  const int KB = (R + 63) / 64;
  return KB * (2 * kTileRows * 128 + kExpandCols * 128) + kTileRows * (kExpandCols + 8) * 2 + 1024;
}

}  // namespace lora
