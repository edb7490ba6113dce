// Segmented (SGMV) path of the routed delta on the 5th-generation tensor cores
// (tcgen05 MMA, accumulators in tensor memory), for adapter keys with many
// rows ("punica_base.py", prefill_metadata / add_lora_linear; "Module
// lora_delta", lora_gemv_max_m: below a row threshold the GEMV-style path is
// cheaper, above it a real tensor-core GEMM is).
//
// The rows of a key are taken in the routing kernel's stable order and cut
// into tiles of 128 rows (the last one ragged).  Two kernels:
//   * shrink: CTA (tile, k-split) computes the tile's partial h[rows, active
//     (slice, rank) pairs] = x[rows] A^T over its share of k_in: 64-wide
//     k-blocks of the gathered x rows and of the key's A rows are staged by
//     cp.async into 128-byte swizzled shared-memory tiles (4-stage ring), one
//     thread issues the M=128 MMAs, and the fp32 partial goes to the split's
//     own plane of the workspace (summed later in a fixed order: deterministic);
//   * expand: a persistent grid walks (tile, 128-column chunk of one slice)
//     items.  The tile's h -- the planes summed, then split into a bf16 (hi,
//     lo) pair so the rank contraction keeps ~fp32 accuracy -- is multiplied by
//     the chunk's B rows (both 128-byte swizzled tiles) and scale * d is folded
//     into out in place, one rounding; the next item's B chunk and out
//     segments stream into shared memory while the current one computes.
// Every wait on an mbarrier is bounded (the limit is a launch argument); on a
// time-out the CTA records LORA_DEV_ERR_TIMEOUT, skips its writes, lets its
// MMA thread's issued MMAs finish and still releases its TMEM.
#pragma once

#include <cuda.h>

#include "bgmv.cuh"
#include "common.cuh"
#include "tc.cuh"

namespace lora {

constexpr int kTileRows = 128;      // MMA M
constexpr int kShrinkStages = 4;
constexpr int kExpandCols = 128;    // output columns per expand CTA
constexpr int kSgmvMaxSR = 256;     // MMA N of the shrink

struct SgmvTile {
  int key, pos0, rows, pad;
};

// ---------------------------------------------------------------- tiles --
// Tile list from the routing kernel's cluster starts: keys with at least
// min_rows rows get ceil(rows / 128) tiles.  One CTA.
// n_tiles[0] = tiles, n_tiles[1] = k-splits of the shrink: enough (tile,
// split) items to fill the `slots` resident shrink CTAs, at most ks_max.
// (Measured on GB300 with the split capped at 1, 2, 3, 4 and 8: this rule is
// within 2% of the best cap on the prefill, skewed and expert-fold
// workloads; balancing the last wave more finely loses to the cost of the
// extra h planes.)
__global__ void __launch_bounds__(256)
    sgmv_tiles_kernel(const int32_t* __restrict__ seg_start, int n_keys, int min_rows,
                      SgmvTile* __restrict__ tiles, int* __restrict__ n_tiles, int max_tiles,
                      int slots, int ks_max) {
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
  if (tid == 255) {
    const int nt = min(base, max_tiles);
    n_tiles[0] = nt;
    n_tiles[1] = nt > 0 ? max(1, min(ks_max, slots / nt)) : 1;
  }
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
  float* hbuf;         // [ksplit planes][sorted rows, hs] fp32 partial sums of h
  int64_t plane;       // elements per plane
  const int* ksplit;   // k-splits of the shrink (planes to sum), set by the tile kernel
  int hs;         // row stride of hbuf (S * R rounded up to 16)
  int R;
  Slices sl;
  int rel[kMaxSlices + 1];
  int chunk0[kMaxSlices + 1];  // first expand chunk of each slice; chunk0[S] = chunks total
  int add_inputs;
  uint32_t* err;
  uint64_t wait_ns;  // limit of every bounded wait (kWaitLimitNs unless a test lowers it)
  // The rows of every tile are consecutive items that are also consecutive
  // rows of x and out (rows already grouped by adapter: perm is the
  // identity), and the kernels' tensor-map arguments describe x and out: the
  // tile's x k-blocks and out segments then arrive by 2-D TMA loads.
  int contig;
};

__device__ __forceinline__ void cp_async16_zfill(void* smem_dst, const void* gsrc, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(smem_dst)),
               "l"(gsrc), "r"(valid ? 16 : 0)
               : "memory");
}

// ---------------------------------------------------------------- shrink --
// CTA (tile, split): the tile's 128 rows against the key's A rows over the
// split's share of the 64-wide k-blocks; the fp32 partial goes to plane
// `split` of hbuf (the expand sums the planes in order, so the result does not
// depend on scheduling).  Producer warps stream each k-block of the gathered
// x rows and of the A rows by cp.async into a ring of swizzled stages and
// arrive on full[stage] as their copies land; one thread issues the MMAs of a
// block and commits them to empty[stage].  No CTA-wide barrier inside the
// loop.  Afterwards warps 0-3 (the TMEM lane quarters) write the accumulator.
constexpr int kShrinkProducers = 256;
constexpr int kShrinkMmaWarp = kShrinkProducers / 32;
constexpr int kShrinkThreads = kShrinkProducers + 32;

template <class Tables>
__global__ void __launch_bounds__(kShrinkThreads)
    sgmv_shrink_kernel(const SgmvArgs a, const Tables tb, const __grid_constant__ CUtensorMap tm_x) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ SlotView v;
  __shared__ uint32_t taddr_s;
  __shared__ __align__(8) uint64_t full_bar[kShrinkStages], empty_bar[kShrinkStages], done_bar,
      drain_bar;
  __shared__ const __nv_bfloat16* xrow_s[kTileRows];
  __shared__ const __nv_bfloat16* arow_s[kSgmvMaxSR];
  cudaGridDependencySynchronize();
  const int ks = *a.ksplit, n_items = *a.n_tiles * ks;
  if ((int)blockIdx.x >= n_items) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  if (tid == 0) {
    for (int s = 0; s < kShrinkStages; ++s) {
      mbar_init(&full_bar[s], kShrinkProducers);  // every producer thread's copies
      mbar_init(&empty_bar[s], 1);                // the MMA commit
    }
    mbar_init(&done_bar, 1);
    mbar_init(&drain_bar, 1);  // the MMA thread's last commit after a time-out
    fence_barrier_init();
  }
  if (warp == 0) tc::tmem_alloc(&taddr_s, kSgmvMaxSR);  // room for any N
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t taddr = taddr_s;
  const int R = a.R;
  const int nkb_all = (a.k_in + 63) / 64;
  int kbg = 0;  // k-blocks streamed through the stage ring so far
  int nd = 0;   // items committed to done_bar so far
  bool ok = true;
  bool issued = false;  // (MMA thread) some MMA was issued
  // persistent: items (tile, split), tile-major
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int tile_id = item / ks, split = item - tile_id * ks;
    const SgmvTile tile = a.tiles[tile_id];
    // the previous item is done (accumulator read, row tables no longer used);
    // after a timed-out wait anywhere in the CTA, all threads stop together
    if (!__syncthreads_and(ok)) break;
    if (tid == 0) {
      uint32_t bad = 0;
      tb.resolve(tile.key, a.sl.S, kModeFused, v, bad);
      if (bad) set_error(a.err, bad);
    }
    for (int r = tid; r < kTileRows; r += kShrinkThreads)
      xrow_s[r] = r < tile.rows ? a.x + tb.x_row(a.perm[tile.pos0 + r]) * a.ld_x : nullptr;
    __syncthreads();
    const int SRa = v.nact * R;
    if (SRa == 0) continue;  // (uniform) no active slice: no planes for this tile
    const int N = (SRa + 15) / 16 * 16;
    for (int t = tid; t < N; t += kShrinkThreads) {
      const __nv_bfloat16* p = nullptr;
      if (t < SRa) {
        const int jj = t / R, q = t - jj * R;
        p = v.A[v.act_slice[jj]] + (size_t)q * a.k_in;
      }
      arow_s[t] = p;
    }
    __syncthreads();
    const int xbytes = kTileRows * 128;
    const int stage_bytes = xbytes + N * 128;  // multiple of 1024
    const int kb_begin = (int)((int64_t)nkb_all * split / ks);
    const int nkb = (int)((int64_t)nkb_all * (split + 1) / ks) - kb_begin;
    if (warp < kShrinkMmaWarp) {
      // -------------------------------------------------------- producer --
      // piece (row, 16-byte chunk c) of a block: rows of x then of A,
      // zero-filled past the tile's rows, the key's pairs and k_in; with
      // contiguous tile rows the x block is one TMA load (rows past the
      // tile feed accumulator rows nobody writes; columns past k_in arrive
      // as zeros)
      // Rows past the tile's and pairs past the key's feed accumulator rows
      // and columns that nobody writes: they are not copied at all (a small
      // tile moves its own rows only); columns past k_in are zeros.
      const int c = tid & 7;
      const int x_rows = a.contig ? 0 : tile.rows;  // (contiguous rows: one TMA load)
      const int n_rows = x_rows + SRa;
      for (int kb = 0; kb < nkb; ++kb) {
        const int g = kbg + kb, s = g % kShrinkStages, k = g / kShrinkStages;
        if (k > 0 && !mbar_wait_bounded(&empty_bar[s], (k - 1) & 1, a.wait_ns)) {
          ok = false;
          break;
        }
        uint8_t* xs = smem + (size_t)s * stage_bytes;
        uint8_t* as = xs + xbytes;
        if (a.contig && tid == 0) {
          mbar_expect_tx(&full_bar[s], (uint32_t)xbytes);
          tma_load_2d(xs, &tm_x, (kb_begin + kb) * 64, tile.pos0, &full_bar[s]);
        }
        const int kk = (kb_begin + kb) * 64 + c * 8;
        const bool kin = kk < a.k_in;
        for (int i = tid >> 3; i < n_rows; i += kShrinkProducers / 8) {
          const bool is_x = i < x_rows;
          const __nv_bfloat16* row = is_x ? xrow_s[i] : arow_s[i - x_rows];
          uint8_t* dst = is_x ? xs + tc::sw128_offset(i, c * 8)
                              : as + tc::sw128_offset(i - x_rows, c * 8);
          cp_async16_zfill(dst, kin ? row + kk : a.x, kin);
        }
        cp_async_arrive(&full_bar[s]);
      }
    } else if (lane == 0) {
      // ------------------------------------------------------------- MMA --
      const uint32_t idesc = tc::idesc_bf16_f32(kTileRows, N);
      for (int kb = 0; kb < nkb; ++kb) {
        const int g = kbg + kb, s = g % kShrinkStages, k = g / kShrinkStages;
        if (!mbar_wait_bounded(&full_bar[s], k & 1, a.wait_ns)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        fence_proxy_async_smem();  // the block came through cp.async (generic proxy)
        const uint32_t xa = smem_addr(smem + (size_t)s * stage_bytes);
        const uint32_t aa = xa + xbytes;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          tc::mma_bf16(taddr, tc::sw128_desc(xa + q * 32), tc::sw128_desc(aa + q * 32), idesc,
                       (kb > 0 || q > 0) ? 1u : 0u);
        issued = true;
        tc::mma_commit(&empty_bar[s]);  // the stage is free once these MMAs are done
      }
      tc::mma_commit(&done_bar);
    }
    kbg += nkb;
    // -------------------------------------------------------------- epilogue
    // warps 0-3: TMEM lane quarter q = tile rows 32q.., columns [0, SRa) ->
    // plane `split` of hbuf, row pos0 + r
    if (warp < 4) {
      // (uniform over the warp before the warp-collective TMEM loads: a lane
      // may have given up in the producer loop, or see the phase later)
      const bool done = ok && mbar_wait_bounded(&done_bar, nd & 1, a.wait_ns);
      ok = __all_sync(0xffffffffu, done);
      tc::fence_after_sync();
      const int r = warp * 32 + lane;
      float* dst = a.hbuf + (size_t)split * a.plane + (size_t)(tile.pos0 + r) * a.hs;
      if (ok && warp * 32 < tile.rows)  // (a lane quarter past the tile's rows: nothing)
        for (int c0 = 0; c0 < N; c0 += 16) {
          float vals[16];
          tc::tmem_ld16(taddr + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, vals);
          if (r < tile.rows) {
#pragma unroll
            for (int i = 0; i < 16; i += 4)
              if (c0 + i < SRa)
                *reinterpret_cast<float4*>(dst + c0 + i) =
                    make_float4(vals[i], vals[i + 1], vals[i + 2], vals[i + 3]);
          }
        }
      tc::fence_before_sync();
    }
    ++nd;
  }
  if (warp < kShrinkMmaWarp) asm volatile("cp.async.wait_all;" ::: "memory");
  if (!ok) set_error(a.err, LORA_DEV_ERR_TIMEOUT);
  // After a time-out the MMAs issued last may still be running: one more
  // commit tracks every earlier MMA of the thread, and TMEM is freed only
  // after it has arrived.
  if (!__syncthreads_and(ok) && warp == kShrinkMmaWarp && lane == 0 && issued) {
    tc::mma_commit(&drain_bar);
    mbar_wait_bounded(&drain_bar, 0, kWaitLimitNs);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(taddr, kSgmvMaxSR);
}

// ---------------------------------------------------------------- expand --
// Persistent CTA over a contiguous range of (tile, 128-column chunk) items,
// one role per warp group:
//   producer warps: per item, the B chunk and the tile's out rows (16
//              lanes per 256-byte row) by cp.async into the 128-byte-swizzled
//              buffers of a ring of kStages stages; each thread's copies
//              arrive on full[stage] as they land;
//   MMA warp:  one thread issues the hi and lo MMAs of an item into one
//              of two TMEM accumulators and commits to acc_full[acc];
//   8 epilogue warps, one (TMEM lane quarter = 32 tile rows, 64-column
//              half) each: read the accumulator, fold scale * d into the
//              staged out rows in place, write them back (8 lanes per
//              128-byte row segment) and release the stage.  They also
//              rebuild h -- the shrink's
//              planes summed, split into bf16 (hi, lo) -- when an item starts
//              a new (tile, slice), after the last MMA that read the old h.
// Stage buffers, accumulators and h are handed over through mbarriers; every
// wait is bounded.
constexpr int kExpandProducers = 256;  // warps [0, kMmaWarp)
constexpr int kMmaWarp = kExpandProducers / 32;
constexpr int kExpandEpilogue = 256;   // warps (kMmaWarp, ...]
constexpr int kEpiWarp0 = kMmaWarp + 1;
constexpr int kExpandThreads = kExpandProducers + 32 + kExpandEpilogue;
constexpr int kExpandMaxTiles = 8;  // tiles one expand CTA may span (the grid ensures it)

template <int RMAX>
struct ExpandSmem {
  static constexpr int KB = (RMAX + 63) / 64;
  static constexpr int kStages = KB == 1 ? 3 : 2;
  static constexpr int kH = KB * kTileRows * 128;          // one of hi / lo
  static constexpr int kB = KB * kExpandCols * 128;        // one B chunk
  static constexpr int kHalf = kTileRows * 128;            // out rows, 64 columns
  static constexpr int kO = 2 * kHalf;                     // out rows, 128 columns
  static constexpr int kTotal = 2 * kH + kStages * (kB + kO) + 1024;
};

template <int RMAX, class Tables>
__global__ void __launch_bounds__(kExpandThreads, 1)
    sgmv_expand_kernel(const SgmvArgs a, const Tables tb, int n_chunks,
                       const __grid_constant__ CUtensorMap tm_out) {
  using SM = ExpandSmem<RMAX>;
  constexpr int KB = SM::KB, NS = SM::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ SlotView vt[kExpandMaxTiles];  // adapter tables of each tile's key
  __shared__ SgmvTile tiles_s[kExpandMaxTiles];
  __shared__ int orow_map[kExpandMaxTiles][kTileRows];  // out row of each tile row
  __shared__ uint32_t taddr_s;
  __shared__ __align__(8) uint64_t full_bar[NS], empty_bar[NS], accf_bar[2], acce_bar[2], h_bar,
      drain_bar;
  cudaGridDependencySynchronize();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int total = *a.n_tiles * n_chunks;
  const int ksplit = *a.ksplit;  // planes of h to sum
  const int w0 = (int)((int64_t)total * blockIdx.x / gridDim.x);
  const int w1 = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
  if (w0 >= w1) return;
  const int t_first = w0 / n_chunks;
  const int n_my_tiles = (w1 - 1) / n_chunks - t_first + 1;
  if (n_my_tiles > kExpandMaxTiles) {  // the launch sizes the grid so that this cannot be
    if (tid == 0) set_error(a.err, LORA_DEV_ERR_INTERNAL);
    return;
  }
  uint8_t* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint8_t* hhi = smem;
  uint8_t* hlo = hhi + SM::kH;
  uint8_t* stage0 = hlo + SM::kH;  // stage s: B chunk [KB][128][128 B], then out [2][128][128 B]
  auto stage_b = [&](int s) { return stage0 + (size_t)s * (SM::kB + SM::kO); };
  auto stage_o = [&](int s) { return stage0 + (size_t)s * (SM::kB + SM::kO) + SM::kB; };
  const int R = a.R;
  if (tid < n_my_tiles) {  // this CTA's tiles and their tables
    const SgmvTile t = a.tiles[t_first + tid];
    tiles_s[tid] = t;
    uint32_t bad = 0;
    tb.resolve(t.key, a.sl.S, kModeFused, vt[tid], bad);
    if (bad) set_error(a.err, bad);
  }
  for (int i = tid; i < n_my_tiles * kTileRows; i += kExpandThreads) {
    const int lt = i / kTileRows, r = i - lt * kTileRows;
    const SgmvTile t = a.tiles[t_first + lt];
    orow_map[lt][r] = r < t.rows ? (int)tb.out_row(a.perm[t.pos0 + r]) : 0;
  }
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full_bar[s], kExpandProducers);  // every producer thread's copies
      mbar_init(&empty_bar[s], kExpandEpilogue / 32);  // the epilogue warps
    }
    for (int c = 0; c < 2; ++c) {
      mbar_init(&accf_bar[c], 1);  // MMA commit
      mbar_init(&acce_bar[c], kExpandEpilogue / 32);  // the epilogue warps
    }
    mbar_init(&h_bar, kExpandEpilogue);  // every epilogue thread
    mbar_init(&drain_bar, 1);            // the MMA thread's last commit after a time-out
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tc::tmem_alloc(&taddr_s, 2 * kExpandCols);  // two accumulators
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t taddr = taddr_s;

  // Item w: (tile, slice j, first column c0, width nc) from arithmetic and the
  // preloaded tables; every role computes it itself.
  struct Item {
    int lt, j, ja, c0, nc;
  };
  auto item_of = [&](int w) {
    Item it;
    const int tile_id = w / n_chunks, chunk = w - tile_id * n_chunks;
    it.lt = tile_id - t_first;
    int j = 0;
#pragma unroll
    for (int jj = 1; jj < kMaxSlices; ++jj)
      if (jj < a.sl.S && chunk >= a.chunk0[jj]) j = jj;
    it.j = j;
    it.ja = vt[it.lt].ja[j];
    it.c0 = (chunk - a.chunk0[j]) * kExpandCols;
    it.nc = min(kExpandCols, a.sl.width[j] - it.c0);
    return it;
  };
  bool ok = true;
  int na_issued = 0;  // (MMA thread) items whose MMAs were issued

  if (warp < kMmaWarp) {
    // ---------------------------------------------------------- producer --
    const int cpr = (R + 15) >> 4 << 1;  // 16-byte pieces per B row that the K-steps read
    // (a power of two unless R is 48, 80, ...: a shift instead of a division)
    const int cpr_shift = (cpr & (cpr - 1)) == 0 ? __ffs(cpr) - 1 : -1;
    for (int w = w0; w < w1 && ok; ++w) {
      const int i = w - w0, s = i % NS, k = i / NS;
      const Item it = item_of(w);
      // the epilogue released this stage's previous use
      if (k > 0 && !mbar_wait_bounded(&empty_bar[s], (k - 1) & 1, a.wait_ns)) {
        ok = false;
        break;
      }
      if (it.ja >= 0 && it.nc > 0) {
        const __nv_bfloat16* bsrc = vt[it.lt].B[it.j] + (size_t)it.c0 * R;
        uint8_t* bb = stage_b(s);
        for (int idx = tid; idx < kExpandCols * cpr; idx += kExpandProducers) {
          const int c = cpr_shift >= 0 ? idx >> cpr_shift : idx / cpr, kk = (idx - c * cpr) * 8;
          const bool v = c < it.nc && kk < R;  // zeros past the slice's end and past R
          cp_async16_zfill(bb + (size_t)(kk >> 6) * kExpandCols * 128 + tc::sw128_offset(c, kk & 63),
                           v ? bsrc + (size_t)c * R + kk : bsrc, v);
        }
        if (a.add_inputs && a.contig) {
          // out rows: each 64-column half one TMA load of the tile's 128 rows
          // in the 128-byte swizzle (the epilogue's layout); rows past the
          // tile and columns past the slice are not written back
          if (tid == 0) {
            const SgmvTile& t = tiles_s[it.lt];
            const int halves = it.nc > 64 ? 2 : 1;
            fence_proxy_async_smem();  // the epilogue's writes to this stage come first
            mbar_expect_tx(&full_bar[s], (uint32_t)(halves * SM::kHalf));
            for (int h = 0; h < halves; ++h)
              tma_load_2d(stage_o(s) + h * SM::kHalf, &tm_out, a.sl.off[it.j] + it.c0 + 64 * h,
                          t.pos0, &full_bar[s]);
          }
        } else if (a.add_inputs) {
          // out rows: piece p (8 columns) of row r at half p / 8, chunk (p mod 8) ^ (r mod 8)
          const SgmvTile& t = tiles_s[it.lt];
          const int* om = orow_map[it.lt];
          const __nv_bfloat16* src = a.out + a.sl.off[it.j] + it.c0;
          uint8_t* ob = stage_o(s);
          const int p = tid & 15, np = it.nc >> 3;
          for (int r = tid >> 4; r < t.rows; r += kExpandProducers / 16)
            if (p < np)
              cp_async16(ob + (p >> 3) * SM::kHalf + r * 128 + (((p & 7) ^ (r & 7)) << 4),
                         src + (int64_t)om[r] * a.ld_out + p * 8);
        }
      }
      cp_async_arrive(&full_bar[s]);
    }
    // nothing may land in this CTA's shared memory after it exits
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------------- MMA --
    if (lane == 0) {
      const int ksteps = (R + 15) / 16;
      int na = 0, hv = -1, h_lt = -1, h_ja = -1;  // active items so far; h version
      for (int w = w0; w < w1; ++w) {
        const int i = w - w0, s = i % NS, k = i / NS;
        const Item it = item_of(w);
        if (it.ja < 0 || it.nc <= 0) continue;
        if (it.lt != h_lt || it.ja != h_ja) {  // the epilogue rebuilds h first
          ++hv;
          h_lt = it.lt;
          h_ja = it.ja;
          if (!mbar_wait_bounded(&h_bar, hv & 1, a.wait_ns)) {
            ok = false;
            break;
          }
        }
        const int acc = na & 1, u = na >> 1;
        if (!mbar_wait_bounded(&full_bar[s], k & 1, a.wait_ns) ||
            (u > 0 && !mbar_wait_bounded(&acce_bar[acc], (u - 1) & 1, a.wait_ns))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        fence_proxy_async_smem();  // the B chunk came through cp.async (generic proxy)
        const uint32_t idesc = tc::idesc_bf16_f32(kTileRows, (it.nc + 15) / 16 * 16);
        const uint8_t* bb = stage_b(s);
        const uint32_t dt = taddr + (uint32_t)(acc * kExpandCols);
        for (int pass = 0; pass < 2; ++pass) {
          const uint8_t* hsrc = pass == 0 ? hhi : hlo;
          for (int st = 0; st < ksteps; ++st) {
            const int kb = st >> 2, ks = st & 3;
            const uint32_t ha = smem_addr(hsrc + (size_t)kb * kTileRows * 128) + ks * 32;
            const uint32_t ba = smem_addr(bb + (size_t)kb * kExpandCols * 128) + ks * 32;
            tc::mma_bf16(dt, tc::sw128_desc(ha), tc::sw128_desc(ba), idesc,
                         (pass > 0 || st > 0) ? 1u : 0u);
          }
        }
        tc::mma_commit(&accf_bar[acc]);
        ++na;
        na_issued = na;
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue --
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int hf = (warp - kEpiWarp0) >> 2;  // 64-column half
    const int r = q * 32 + lane;             // this thread's tile row
    const int et = tid - kEpiWarp0 * 32;     // index among the epilogue threads
    int na = 0, h_lt = -1, h_ja = -1;
    for (int w = w0; w < w1 && ok; ++w) {
      const int i = w - w0, s = i % NS, k = i / NS;
      const Item it = item_of(w);
      if (it.ja < 0 || it.nc <= 0) {
        // nothing to compute: release the stage once its (empty) fill completed
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full_bar[s], k & 1, a.wait_ns))) {
          ok = false;
          break;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
        continue;
      }
      const SgmvTile& t = tiles_s[it.lt];
      if (it.lt != h_lt || it.ja != h_ja) {
        // every MMA that read the old h has completed (its accumulator was
        // waited for below), and the MMA thread waits for this arrival
        h_lt = it.lt;
        h_ja = it.ja;
        for (int e = et; e < KB * kTileRows * 8; e += kExpandEpilogue) {
          const int kb = e / (kTileRows * 8), rem = e - kb * kTileRows * 8;
          const int hr = rem >> 3, g = rem & 7, kk = kb * 64 + g * 8;
          float hv[8];
#pragma unroll
          for (int x = 0; x < 8; ++x) hv[x] = 0.0f;
          if (hr < t.rows && kk < R) {
            const float* hp = a.hbuf + (size_t)(t.pos0 + hr) * a.hs + it.ja * R + kk;
            for (int sp = 0; sp < ksplit; ++sp) {
              const float4 h0 = *reinterpret_cast<const float4*>(hp + sp * a.plane);
              const float4 h1 = *reinterpret_cast<const float4*>(hp + sp * a.plane + 4);
              hv[0] += h0.x; hv[1] += h0.y; hv[2] += h0.z; hv[3] += h0.w;
              hv[4] += h1.x; hv[5] += h1.y; hv[6] += h1.z; hv[7] += h1.w;
            }
          }
          uint4 hi, lo;
          split_bf16x2(hv[0], hv[1], hi.x, lo.x);
          split_bf16x2(hv[2], hv[3], hi.y, lo.y);
          split_bf16x2(hv[4], hv[5], hi.z, lo.z);
          split_bf16x2(hv[6], hv[7], hi.w, lo.w);
          const uint32_t off = (uint32_t)kb * kTileRows * 128 + tc::sw128_offset(hr, g * 8);
          *reinterpret_cast<uint4*>(hhi + off) = hi;
          *reinterpret_cast<uint4*>(hlo + off) = lo;
        }
        fence_proxy_async_smem();
        mbar_arrive(&h_bar);
      }
      const int acc = na & 1, u = na >> 1;
      // (every lane of the warp takes the same branch: the TMEM loads below
      // are warp-collective)
      const bool ready = mbar_wait_bounded(&accf_bar[acc], u & 1, a.wait_ns) &&
                         mbar_wait_bounded(&full_bar[s], k & 1, a.wait_ns);
      if (!__all_sync(0xffffffffu, ready)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      // fold scale * d into this warp's rows and half of the staged out tile
      // (in place; 16-byte chunk c of row r sits at chunk c ^ (r mod 8))
      const float sc = vt[it.lt].scale;
      uint8_t* hb = stage_o(s) + hf * SM::kHalf;
      // (uniform across the warp; a lane quarter past the tile's rows has
      // nothing to read or write back)
      const bool mine = hf * 64 < it.nc && q * 32 < t.rows;
      if (mine) {
        float d[64];
        tc::tmem_ld64(taddr + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kExpandCols + hf * 64),
                      d);
        uint8_t* rowp = hb + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4* p = reinterpret_cast<uint4*>(rowp + ((c ^ (r & 7)) << 4));
          const uint4 o = a.add_inputs ? *p : make_uint4(0, 0, 0, 0);
          uint4 res;
          res.x = pack_bf16x2(bf16lo(o.x) + sc * d[8 * c + 0], bf16hi(o.x) + sc * d[8 * c + 1]);
          res.y = pack_bf16x2(bf16lo(o.y) + sc * d[8 * c + 2], bf16hi(o.y) + sc * d[8 * c + 3]);
          res.z = pack_bf16x2(bf16lo(o.z) + sc * d[8 * c + 4], bf16hi(o.z) + sc * d[8 * c + 5]);
          res.w = pack_bf16x2(bf16lo(o.w) + sc * d[8 * c + 6], bf16hi(o.w) + sc * d[8 * c + 7]);
          *p = res;
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce_bar[acc]);  // accumulator free for the MMA thread
      if (mine) {
        // write back the warp's 32 row segments: 8 lanes per 128 bytes, 4 rows per step
        const int* om = orow_map[it.lt];
        __nv_bfloat16* dst0 = a.out + a.sl.off[it.j] + it.c0 + hf * 64;
        const int p = lane & 7, np = min(8, (it.nc - hf * 64) >> 3);
#pragma unroll 4
        for (int v = 0; v < 8; ++v) {  // (rows written by other lanes: the __syncwarp above)
          const int rr = q * 32 + v * 4 + (lane >> 3);
          if (rr < t.rows && p < np)
            *reinterpret_cast<uint4*>(dst0 + (int64_t)om[rr] * a.ld_out + p * 8) =
                *reinterpret_cast<const uint4*>(hb + rr * 128 + ((p ^ (rr & 7)) << 4));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);  // stage read: free for the producer
      ++na;
    }
    __syncwarp();
  }
  if (!ok) set_error(a.err, LORA_DEV_ERR_TIMEOUT);
  // After a time-out the MMAs issued last may still be running: one more
  // commit tracks every earlier MMA of the thread, and TMEM is freed only
  // after it has arrived.
  if (!__syncthreads_and(ok) && warp == kMmaWarp && lane == 0 && na_issued > 0) {
    tc::mma_commit(&drain_bar);
    mbar_wait_bounded(&drain_bar, 0, kWaitLimitNs);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) tc::tmem_dealloc(taddr, 2 * kExpandCols);
}
inline int sgmv_shrink_smem(int sr_max) {
  const int N = (sr_max + 15) / 16 * 16;
  return kShrinkStages * (kTileRows * 128 + N * 128) + 1024;
}
inline int sgmv_expand_smem(int R) {
  return R <= 64 ? ExpandSmem<64>::kTotal : ExpandSmem<128>::kTotal;
}

}  // namespace lora
