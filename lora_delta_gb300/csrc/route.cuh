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
  int top_k, E, num_loras;
  __device__ int operator()(int p, uint32_t& err) const {
    const int l = lora_ids[p / top_k];
    const int e = topk_ids[p];
    const int none = num_loras * E;
    if (l < 0) return none;
    if (l >= num_loras) {
      err |= LORA_DEV_ERR_LORA;
      return none;
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

template <class KeyFn>
__global__ void __launch_bounds__(kRouteThreads)
    route_kernel(KeyFn key_of, int n, int n_keys, int32_t* __restrict__ perm,
                 int32_t* __restrict__ seg_start, uint32_t* err_word) {
  extern __shared__ uint32_t cnt[];  // [kRouteWarps][n_keys + 1]
  __shared__ uint32_t warp_sums[kRouteWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nkb = n_keys + 1;
  for (int i = tid; i < kRouteWarps * nkb; i += kRouteThreads) cnt[i] = 0;
  __syncthreads();

  const int per = (n + kRouteWarps - 1) / kRouteWarps;
  const int b0 = min(n, warp * per), b1 = min(n, b0 + per);
  uint32_t errbits = 0;
  uint32_t* my = cnt + warp * nkb;
  // kRouteBatch keys per lane are loaded before any is used, so a warp's
  // block costs one memory round trip per 32 * kRouteBatch items
  // With at most 32 key values, lane k counts key k from one ballot per key
  // value; otherwise __match_any_sync groups the lanes by key.
  const bool few = nkb <= 32;
  uint32_t mine = 0;  // (few keys) this lane's count of key `lane`
  for (int base = b0; base < b1; base += 32 * kRouteBatch) {
    int keys[kRouteBatch];
#pragma unroll
    for (int u = 0; u < kRouteBatch; ++u) {
      const int i = base + u * 32 + lane;
      keys[u] = (i < b1) ? key_of(i, errbits) : -1;
    }
#pragma unroll
    for (int u = 0; u < kRouteBatch; ++u) {
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
  if (few && lane < nkb) my[lane] = mine;
  errbits = __reduce_or_sync(0xffffffffu, errbits);
  if (lane == 0 && errbits) set_error(err_word, errbits);
  __syncthreads();

  // Block-wide exclusive scan over keys of the per-key totals; each thread
  // owns a contiguous run of keys.
  const int kpt = (nkb + kRouteThreads - 1) / kRouteThreads;
  const int k0 = min(nkb, tid * kpt), k1 = min(nkb, k0 + kpt);
  uint32_t tsum = 0;
  for (int k = k0; k < k1; ++k)
    for (int w = 0; w < kRouteWarps; ++w) tsum += cnt[w * nkb + k];
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

  uint32_t next = (few && lane < nkb) ? my[lane] : 0u;  // (few keys) next position of key `lane`
  const unsigned lt = (1u << lane) - 1u;
  for (int base = b0; base < b1; base += 32 * kRouteBatch) {
    int keys[kRouteBatch];
    uint32_t dummy = 0;
#pragma unroll
    for (int u = 0; u < kRouteBatch; ++u) {
      const int i = base + u * 32 + lane;
      keys[u] = (i < b1) ? key_of(i, dummy) : -1;
    }
#pragma unroll
    for (int u = 0; u < kRouteBatch; ++u) {
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

}  // namespace lora
