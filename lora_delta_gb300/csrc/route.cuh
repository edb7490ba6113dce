// Device-side routing: a stable counting sort of rows (or MoE (token, slot)
// pairs) by adapter key.  "vllm/lora/punica_wrapper/punica_base.py",
// prefill_metadata: the batch clustered by identical lora index, -1 applying
// none.  Our rows arrive unsorted, so the clusters are built here, on the
// device, with no host round trip.
//
// One CTA of kRouteThreads threads.  The items are cut into one contiguous
// block per warp, read kRouteBatch keys per lane at a time; pass 1 counts keys
// per (warp, key) with __match_any_sync,
// a block scan turns the counts into per-(warp, key) output positions, and
// pass 2 scatters every item to its position -- the rank inside a warp
// iteration comes from the match mask, so the order within a key is the
// original item order (stable).  Bucket n_keys collects the items with no
// valid key; seg_start[n_keys + 1] == n.
#pragma once

#include "common.cuh"

namespace lora {

constexpr int kRouteThreads = 512;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kRouteBatch = 16;  // keys per lane loaded together

// Key of a linear-delta row: its slot, or n_keys (no delta) for slot < 0 and
// for slot >= max_loras (which also sets LORA_DEV_ERR_SLOT).
struct SlotKey {
  const int32_t* seq_slot;
  int max_loras;
  __device__ int operator()(int i, uint32_t& err) const {
    const int s = seq_slot[i];
    if (s < 0) return max_loras;
    if (s >= max_loras) {
      err |= LORA_DEV_ERR_SLOT;
      return max_loras;
    }
    return s;
  }
};

// Key of an MoE (token, slot) pair p: l * E + e, or the no-key bucket.
struct MoeKey {
  const int32_t* topk_ids;
  const int32_t* lora_ids;
  const int32_t* expert_map;       // [n_global] global -> local expert id (-1: not local), or null
  const int32_t* adapter_enabled;  // [num_loras], 0: the adapter adds nothing; or null
  int top_k, E, num_loras, n_global;
  __device__ int operator()(int p, uint32_t& err) const {
    const int l = lora_ids[p / top_k];
    int e = topk_ids[p];
    const int none = num_loras * E;
    if (l < 0) return none;
    if (l >= num_loras) {
      err |= LORA_DEV_ERR_LORA;
      return none;
    }
    if (adapter_enabled && adapter_enabled[l] == 0) return none;
    if (expert_map) {
      if (e < 0 || e >= n_global) {
        err |= LORA_DEV_ERR_EXPERT;
        return none;
      }
      e = expert_map[e];
      if (e < 0) return none;  // the expert lives on another rank
    }
    if (e < 0 || e >= E) {
      err |= LORA_DEV_ERR_EXPERT;
      return none;
    }
    return l * E + e;
  }
};

inline size_t route_smem_bytes(int n_keys) {
  return sizeof(uint32_t) * (size_t)kRouteWarps * (size_t)(n_keys + 1);
}

// Per-warp pieces shared by the one-CTA sort and the chunked sort.  A warp
// owns the items [b0, b1) and reads BATCH keys per lane before using them
// (one memory round trip per 32 * BATCH items).  With at most 32
// key values, lane k counts key k from one ballot per key value; otherwise
// __match_any_sync groups the lanes by key.

// my[k] += number of items of key k in [b0, b1).
template <int BATCH, class KeyFn>
__device__ __forceinline__ void warp_count(const KeyFn& key_of, int b0, int b1, int nkb,
                                           uint32_t* my, uint32_t& errbits) {
  const int lane = threadIdx.x & 31;
  const bool few = nkb <= 32;
  uint32_t mine = 0;  // (few keys) this lane's count of key `lane`
  for (int base = b0; base < b1; base += 32 * BATCH) {
    int keys[BATCH];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int i = base + u * 32 + lane;
      keys[u] = (i < b1) ? key_of(i, errbits) : -1;
    }
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      if (few) {
        for (int kk = 0; kk < nkb; ++kk) {
          const unsigned m = __ballot_sync(0xffffffffu, keys[u] == kk);
          if (lane == kk) mine += __popc(m);
        }
      } else {
        const unsigned peers = __match_any_sync(0xffffffffu, keys[u]);
        if (keys[u] >= 0 && lane == __ffs(peers) - 1) my[keys[u]] += __popc(peers);
        __syncwarp();
      }
    }
  }
  if (few && lane < nkb) my[lane] += mine;
  __syncwarp();
}

// Scatter the items of [b0, b1) to perm; my[k] holds the next position of
// key k and is advanced.
template <int BATCH, class KeyFn>
__device__ __forceinline__ void warp_scatter(const KeyFn& key_of, int b0, int b1, int nkb,
                                             uint32_t* my, int32_t* __restrict__ perm) {
  const int lane = threadIdx.x & 31;
  const bool few = nkb <= 32;
  uint32_t next = (few && lane < nkb) ? my[lane] : 0u;  // (few keys) next position of key `lane`
  const unsigned lt = (1u << lane) - 1u;
  for (int base = b0; base < b1; base += 32 * BATCH) {
    int keys[BATCH];
    uint32_t dummy = 0;
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int i = base + u * 32 + lane;
      keys[u] = (i < b1) ? key_of(i, dummy) : -1;
    }
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int key = keys[u];
      if (few) {
        unsigned peers = 0, cnt = 0;
        for (int kk = 0; kk < nkb; ++kk) {
          const unsigned m = __ballot_sync(0xffffffffu, key == kk);
          if (key == kk) peers = m;
          if (lane == kk) cnt = __popc(m);
        }
        const uint32_t at = __shfl_sync(0xffffffffu, next, key < 0 ? 0 : key);
        if (key >= 0) perm[at + __popc(peers & lt)] = base + u * 32 + lane;
        next += cnt;
      } else {
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        if (key >= 0) perm[my[key] + __popc(peers & lt)] = base + u * 32 + lane;
        __syncwarp();
        if (key >= 0 && lane == __ffs(peers) - 1) my[key] += __popc(peers);
        __syncwarp();
      }
    }
  }
}

// Block-wide exclusive scan over keys [0, nkb) of total(k); each thread owns
// a contiguous run of keys; returns, in `first`, the scan value at this
// thread's first key (k0) and in k0 / k1 its run.
template <class TotalFn>
__device__ __forceinline__ uint32_t block_scan_keys(int nkb, const TotalFn& total, int& k0,
                                                    int& k1, uint32_t* warp_sums) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kpt = (nkb + kRouteThreads - 1) / kRouteThreads;
  k0 = min(nkb, tid * kpt);
  k1 = min(nkb, k0 + kpt);
  uint32_t tsum = 0;
  for (int k = k0; k < k1; ++k) tsum += total(k);
  uint32_t incl = tsum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  uint32_t run = incl - tsum;
  for (int w = 0; w < warp; ++w) run += warp_sums[w];
  return run;
}

// One CTA sorts all n items: one contiguous block per warp.
template <class KeyFn>
__global__ void __launch_bounds__(kRouteThreads)
    route_kernel(KeyFn key_of, int n, int n_keys, int32_t* __restrict__ perm,
                 int32_t* __restrict__ seg_start, uint32_t* err_word) {
  extern __shared__ uint32_t cnt[];  // [kRouteWarps][n_keys + 1]
  __shared__ uint32_t warp_sums[kRouteWarps];
  // The next launch may start its prologue (adapter weight copies) now: it
  // reads this sort's output only after its own dependency wait.
  cudaTriggerProgrammaticLaunchCompletion();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nkb = n_keys + 1;
  for (int i = tid; i < kRouteWarps * nkb; i += kRouteThreads) cnt[i] = 0;
  __syncthreads();
  const int per = (n + kRouteWarps - 1) / kRouteWarps;
  const int b0 = min(n, warp * per), b1 = min(n, b0 + per);
  uint32_t errbits = 0;
  uint32_t* my = cnt + warp * nkb;
  warp_count<kRouteBatch>(key_of, b0, b1, nkb, my, errbits);
  errbits = __reduce_or_sync(0xffffffffu, errbits);
  if (lane == 0 && errbits) set_error(err_word, errbits);
  __syncthreads();
  int k0, k1;
  uint32_t run = block_scan_keys(
      nkb,
      [&](int k) {
        uint32_t t = 0;
        for (int w = 0; w < kRouteWarps; ++w) t += cnt[w * nkb + k];
        return t;
      },
      k0, k1, warp_sums);
  for (int k = k0; k < k1; ++k) {
    seg_start[k] = (int32_t)run;
    for (int w = 0; w < kRouteWarps; ++w) {
      const uint32_t c = cnt[w * nkb + k];
      cnt[w * nkb + k] = run;
      run += c;
    }
  }
  if (tid == 0) seg_start[nkb] = n;
  __syncthreads();
  warp_scatter<kRouteBatch>(key_of, b0, b1, nkb, my, perm);
}

// ------------------------------------------------------- chunked sort ---
// For large batches: chunks of kRouteChunk items, one CTA each, in two
// kernels.  route_count_kernel writes chunk b's count of every key to
// counts[b][key]; route_scatter_kernel scans those counts (key-major, then
// chunk) into each chunk's starting position per key and scatters the chunk
// exactly as the one-CTA kernel does.  Chunk-major, then warp, then lane
// order: the same stable order.
constexpr int kRouteChunk = 1024;
constexpr int kRoutePerWarp = kRouteChunk / kRouteWarps;

inline size_t route_chunk_smem_bytes(int n_keys) {
  return sizeof(uint32_t) * ((size_t)kRouteWarps + 2) * (size_t)(n_keys + 1);
}

template <class KeyFn>
__global__ void __launch_bounds__(kRouteThreads)
    route_count_kernel(KeyFn key_of, int n, int n_keys, uint32_t* __restrict__ counts,
                       uint32_t* err_word) {
  extern __shared__ uint32_t cnt[];  // [kRouteWarps][n_keys + 1]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nkb = n_keys + 1;
  for (int i = tid; i < kRouteWarps * nkb; i += kRouteThreads) cnt[i] = 0;
  __syncthreads();
  const int b0 = min(n, (int)blockIdx.x * kRouteChunk + warp * kRoutePerWarp);
  const int b1 = min(n, b0 + kRoutePerWarp);
  uint32_t errbits = 0;
  warp_count<kRoutePerWarp / 32>(key_of, b0, b1, nkb, cnt + warp * nkb, errbits);
  errbits = __reduce_or_sync(0xffffffffu, errbits);
  if (lane == 0 && errbits) set_error(err_word, errbits);
  __syncthreads();
  for (int k = tid; k < nkb; k += kRouteThreads) {
    uint32_t t = 0;
    for (int w = 0; w < kRouteWarps; ++w) t += cnt[w * nkb + k];
    counts[(size_t)blockIdx.x * nkb + k] = t;
  }
}

template <class KeyFn>
__global__ void __launch_bounds__(kRouteThreads)
    route_scatter_kernel(KeyFn key_of, int n, int n_keys, const uint32_t* __restrict__ counts,
                         int32_t* __restrict__ perm, int32_t* __restrict__ seg_start) {
  // [kRouteWarps][n_keys + 1] per-warp counts, then before[n_keys + 1] (this
  // chunk's start within each key) and total[n_keys + 1]
  extern __shared__ uint32_t cnt[];
  __shared__ uint32_t warp_sums[kRouteWarps];
  cudaGridDependencySynchronize();
  cudaTriggerProgrammaticLaunchCompletion();  // (as in route_kernel)
  const int tid = threadIdx.x, warp = tid >> 5;
  const int nkb = n_keys + 1, nblk = (int)gridDim.x, blk = (int)blockIdx.x;
  uint32_t* before = cnt + kRouteWarps * nkb;
  uint32_t* total = before + nkb;
  for (int i = tid; i < kRouteWarps * nkb; i += kRouteThreads) cnt[i] = 0;
  for (int k = tid; k < nkb; k += kRouteThreads) {  // one pass, loads in flight together
    uint32_t b = 0, t = 0;
#pragma unroll 8
    for (int c = 0; c < nblk; ++c) {
      const uint32_t v = counts[(size_t)c * nkb + k];
      t += v;
      b += c < blk ? v : 0u;
    }
    before[k] = b;
    total[k] = t;
  }
  __syncthreads();
  const int b0 = min(n, blk * kRouteChunk + warp * kRoutePerWarp);
  const int b1 = min(n, b0 + kRoutePerWarp);
  uint32_t dummy = 0;
  uint32_t* my = cnt + warp * nkb;
  warp_count<kRoutePerWarp / 32>(key_of, b0, b1, nkb, my, dummy);
  __syncthreads();
  int k0, k1;
  uint32_t run = block_scan_keys(nkb, [&](int k) { return total[k]; }, k0, k1, warp_sums);
  for (int k = k0; k < k1; ++k) {
    if (blk == 0) seg_start[k] = (int32_t)run;
    uint32_t at = run + before[k];
    for (int w = 0; w < kRouteWarps; ++w) {
      const uint32_t c = cnt[w * nkb + k];
      cnt[w * nkb + k] = at;
      at += c;
    }
    run += total[k];
  }
  if (blk == 0 && tid == 0) seg_start[nkb] = n;
  __syncthreads();
  warp_scatter<kRoutePerWarp / 32>(key_of, b0, b1, nkb, my, perm);
}

// ------------------------------------------------------- cluster sort ---
// Up to kRouteClusterMax chunks in one launch: one CTA per chunk, all in one
// thread-block cluster.  Each CTA counts its chunk once (per warp, as above)
// and leaves the chunk's per-key totals in its shared memory; after one
// cluster barrier every CTA reads the totals of all chunks from its peers'
// shared memory (distributed shared memory) into its start within each key
// and the keys' totals, scans and scatters its chunk as route_scatter_kernel
// does -- the same positions, so the same stable order -- with no counts in
// global memory and one launch instead of two.
constexpr int kRouteClusterMax = 16;

inline size_t route_cluster_smem_bytes(int n_keys) {
  return sizeof(uint32_t) * ((size_t)kRouteWarps + 3) * (size_t)(n_keys + 1);
}

template <class KeyFn>
__global__ void __launch_bounds__(kRouteThreads)
    route_cluster_kernel(KeyFn key_of, int n, int n_keys, int32_t* __restrict__ perm,
                         int32_t* __restrict__ seg_start, uint32_t* err_word) {
  // [kRouteWarps][n_keys + 1] per-warp counts, then this chunk's totals
  // mine[n_keys + 1] (read by the peers), before[] and total[]
  extern __shared__ uint32_t cnt[];
  __shared__ uint32_t warp_sums[kRouteWarps];
  cudaGridDependencySynchronize();
  cudaTriggerProgrammaticLaunchCompletion();  // (as in route_kernel)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nkb = n_keys + 1, nblk = (int)gridDim.x, blk = (int)blockIdx.x;
  uint32_t* mine = cnt + kRouteWarps * nkb;
  uint32_t* before = mine + nkb;
  uint32_t* total = before + nkb;
  for (int i = tid; i < kRouteWarps * nkb; i += kRouteThreads) cnt[i] = 0;
  __syncthreads();
  const int b0 = min(n, blk * kRouteChunk + warp * kRoutePerWarp);
  const int b1 = min(n, b0 + kRoutePerWarp);
  uint32_t errbits = 0;
  uint32_t* my = cnt + warp * nkb;
  // A warp's items are one round of kRoutePerWarp / 32 keys per lane: they are
  // read once and kept in registers for both the count and the scatter.
  static_assert(kRoutePerWarp == 64, "two keys per lane");
  int kr[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int i = b0 + u * 32 + lane;
    kr[u] = i < b1 ? key_of(i, errbits) : -1;
  }
  // (item i of the warp's block is round (i - b0) / 32 of this lane)
  auto kept = [&](int i, uint32_t&) { return ((i - b0) >> 5) == 0 ? kr[0] : kr[1]; };
  warp_count<kRoutePerWarp / 32>(kept, b0, b1, nkb, my, errbits);
  errbits = __reduce_or_sync(0xffffffffu, errbits);
  if (lane == 0 && errbits) set_error(err_word, errbits);
  __syncthreads();
  for (int k = tid; k < nkb; k += kRouteThreads) {
    uint32_t t = 0;
    for (int w = 0; w < kRouteWarps; ++w) t += cnt[w * nkb + k];
    mine[k] = t;
  }
  cluster_arrive_release_smem();  // this chunk's totals in place
  cluster_wait();
  const uint32_t mine_addr = smem_addr(mine);
  for (int k = tid; k < nkb; k += kRouteThreads) {
    uint32_t b = 0, t = 0;
#pragma unroll 8
    for (int c = 0; c < nblk; ++c) {  // (loads in flight together)
      const uint32_t v = __float_as_uint(dsmem_ld_f32(dsmem_map(mine_addr + 4u * (uint32_t)k,
                                                                  (uint32_t)c)));
      t += v;
      b += c < blk ? v : 0u;
    }
    before[k] = b;
    total[k] = t;
  }
  cluster_arrive_relaxed();  // done reading the peers (waited on before exit)
  __syncthreads();
  int k0, k1;
  uint32_t run = block_scan_keys(nkb, [&](int k) { return total[k]; }, k0, k1, warp_sums);
  for (int k = k0; k < k1; ++k) {
    if (blk == 0) seg_start[k] = (int32_t)run;
    uint32_t at = run + before[k];
    for (int w = 0; w < kRouteWarps; ++w) {
      const uint32_t c = cnt[w * nkb + k];
      cnt[w * nkb + k] = at;
      at += c;
    }
    run += total[k];
  }
  if (blk == 0 && tid == 0) seg_start[nkb] = n;
  __syncthreads();
  warp_scatter<kRoutePerWarp / 32>(kept, b0, b1, nkb, my, perm);
  cluster_wait();  // the peers have read this CTA's totals
}

}  // namespace lora
