// C ABI of the routed LoRA delta: host-side validation, launch planning and
// dispatch onto the caller's stream.  Nothing here allocates or synchronizes
// (lora_get_error excepted); every failure is a status code.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>
#include <unordered_map>

#include "bgmv.cuh"
#include "bgmv_fused.cuh"
#include "floor.cuh"
#include "common.cuh"
#include "keyed.cuh"
#include "lora_delta.h"
#include "route.cuh"
#include "sgmv.cuh"

using namespace lora;

namespace {

constexpr int kAbiVersion = 2;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

int env_int(const char* name, int dflt) {
  const char* v = getenv(name);
  if (!v || !*v) return dflt;
  char* end = nullptr;
  long x = strtol(v, &end, 10);
  return (end && *end == 0) ? (int)x : dflt;
}

// Cluster size of the small-segment kernel: 16 CTAs per key when there are few
// keys (decode: spread each adapter's bytes over many SMs), fewer when there
// are many keys (MoE); LORA_CLUSTER_SIZE (1..16) overrides, read once.
int cluster_size_for(int n_keys) {
  static const int forced = [] {
    const int v = env_int("LORA_CLUSTER_SIZE", 0);
    return (v >= 1 && v <= 16) ? v : 0;
  }();
  if (forced) return forced;
  // measured on GB300 (152 SMs): 16 slots run best at 12 CTAs per cluster
  // (192 CTAs: 9.8 us per decode step against 10.8 us at 16, and 17 us at 14
  // or 15, where the clusters no longer fit in one wave); 128 slots at 8 and
  // 512 MoE keys at 4
  if (n_keys <= 8) return 16;
  if (n_keys <= 16) return 12;
  if (n_keys <= 48) return 16;
  if (n_keys <= 192) return 8;
  return 4;
}
// Shared memory for the A rows of the cluster kernel's shrink stages (both
// buffers); LORA_STAGE_KB overrides (16..192), read once.
int stage_bytes() {
  static const int v = [] {
    const int kb = env_int("LORA_STAGE_KB", 64);
    return (kb >= 16 && kb <= 192 ? kb : 64) * 1024;
  }();
  return v;
}
// Largest B slab the cluster kernel stages in shared memory; LORA_BSTAGE_KB
// overrides (8..96), read once.
int b_stage_bytes() {
  static const int v = [] {
    const int kb = env_int("LORA_BSTAGE_KB", 32);
    return (kb >= 8 && kb <= 96 ? kb : 32) * 1024;
  }();
  return v;
}
bool use_pdl() {
  static const bool on = env_int("LORA_PDL", 1) != 0;
  return on;
}
// Limit of the kernels' bounded waits, read at each launch
// (lora_set_wait_limit_ns).
std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};

// Per-(kernel, device) function attributes, set once: the dynamic shared
// memory opt-in (to the largest size requested so far) and the non-portable
// cluster size.
struct KernelAttrCache {
  std::mutex mu;
  std::unordered_map<uint64_t, int> smem;  // (kernel, device) -> bytes granted
  std::unordered_map<uint64_t, bool> cluster;
  std::unordered_map<uint64_t, int> occupancy;  // (kernel, device, smem) -> CTAs per SM
};
KernelAttrCache& attr_cache() {
  static KernelAttrCache c;
  return c;
}

// Resident CTAs per SM of `kernel` with `threads` threads and `smem_bytes` of
// dynamic shared memory, ignoring tensor memory; at least 1.
template <class K>
int ctas_per_sm(K kernel, int threads, int smem_bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  const uint64_t id = (reinterpret_cast<uint64_t>(reinterpret_cast<const void*>(kernel)) << 6) ^
                      ((uint64_t)dev << 40) ^ (uint64_t)smem_bytes;
  KernelAttrCache& c = attr_cache();
  std::lock_guard<std::mutex> lock(c.mu);
  auto it = c.occupancy.find(id);
  if (it != c.occupancy.end()) return it->second;
  // From the SM's shared memory, registers and threads (the runtime's
  // occupancy query answers 1 for any kernel that allocates tensor memory,
  // although CTAs whose columns fit share an SM).
  int n = 1;
  cudaFuncAttributes fa;
  int smem_sm = 0, resv = 0, regs_sm = 0, thr_sm = 0;
  if (cudaFuncGetAttributes(&fa, kernel) == cudaSuccess &&
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) ==
          cudaSuccess &&
      cudaDeviceGetAttribute(&resv, cudaDevAttrReservedSharedMemoryPerBlock, dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) ==
          cudaSuccess &&
      cudaDeviceGetAttribute(&thr_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) == cudaSuccess) {
    const long per_cta = (long)smem_bytes + (long)fa.sharedSizeBytes + resv;
    const int warps = (threads + 31) / 32;
    const int regs = ((fa.numRegs * 32 + 255) / 256) * 256 * warps;  // 256-register granules
    n = (int)(smem_sm / per_cta);
    if (regs > 0 && regs_sm / regs < n) n = regs_sm / regs;
    if (thr_sm / (warps * 32) < n) n = thr_sm / (warps * 32);
    if (n < 1) n = 1;
  }
  c.occupancy[id] = n;
  return n;
}

template <class K>
cudaError_t prepare_kernel(K kernel, int smem_bytes, bool big_cluster) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t id = (reinterpret_cast<uint64_t>(reinterpret_cast<const void*>(kernel)) << 6) ^
                      (uint64_t)dev;
  KernelAttrCache& c = attr_cache();
  std::lock_guard<std::mutex> lock(c.mu);
  if (smem_bytes > 48 * 1024) {
    auto it = c.smem.find(id);
    if (it == c.smem.end() || it->second < smem_bytes) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
      if (e != cudaSuccess) return e;
      // all of the unified L1 as shared memory, so that several such CTAs fit
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
      c.smem[id] = smem_bytes;
    }
  }
  if (big_cluster && !c.cluster[id]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    c.cluster[id] = true;
  }
  return cudaSuccess;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? LORA_OK : LORA_ERR_CUDA; }

int make_slices(const int32_t* widths, int S, int offset_start, Slices& sl, int* rel) {
  if (!widths || S < 1 || S > kMaxSlices) return S > kMaxSlices ? LORA_ERR_UNSUPPORTED : LORA_ERR_ARG;
  if (offset_start < 0) return LORA_ERR_ARG;
  if (offset_start % 8) return LORA_ERR_ALIGN;
  sl.S = S;
  int o = 0;
  for (int j = 0; j < kMaxSlices; ++j) {
    sl.width[j] = 0;
    sl.off[j] = 0;
  }
  for (int j = 0; j < S; ++j) {
    if (widths[j] < 0) return LORA_ERR_ARG;
    if (widths[j] % 8) return LORA_ERR_ALIGN;
    sl.width[j] = widths[j];
    sl.off[j] = offset_start + o;
    rel[j] = o;
    o += widths[j];
  }
  for (int j = S; j <= kMaxSlices; ++j) rel[j] = o;
  sl.n_cols = o;
  return LORA_OK;
}

int check_rank(int S, int R) {
  if (R < 1) return LORA_ERR_ARG;
  if (R % 8) return LORA_ERR_ALIGN;
  if (R > kMaxRank || S * R > kMaxSR) return LORA_ERR_UNSUPPORTED;
  return LORA_OK;
}

// Per-CTA k-range and shrink stage width (multiples of 16: whole MMA k-steps,
// except at the end of k_in) and columns per CTA (multiple of 8: whole MMA
// column tiles).
void plan_tiles(DeltaArgs& a, int k_in, int n_cols, int sr_max, int mode) {
  const int cs = cluster_size_for(a.n_keys);
  a.cs = cs;
  const int sr16 = (sr_max + 15) / 16 * 16;
  a.kc = ((k_in + cs - 1) / cs + 15) / 16 * 16;
  if (a.kc < 16) a.kc = 16;
  if (mode == kModeExpand) {
    a.kst = 16;
    a.nbuf = 1;
  } else if (sr16 * (a.kc + 8) * 2 <= stage_bytes()) {
    a.kst = a.kc;  // one stage: A stays resident across row passes
    a.nbuf = 1;
  } else {
    int ks = stage_bytes() / 2 / (sr16 * 2) - 8;
    ks = ks >= 64 ? ks / 64 * 64 : ks / 16 * 16;
    a.kst = ks < 16 ? 16 : ks;
    a.nbuf = 2;
  }
  a.b_stage_max = b_stage_bytes();
  a.cpc = ((n_cols + cs - 1) / cs + 7) / 8 * 8;
  if (a.cpc < 8) a.cpc = 8;
  a.min_rows = 0;
  a.max_rows = 0x7fffffff;
  // start the weight copies before the dependency wait when nearly every key
  // has rows (an empty key's early copies are wasted traffic)
  a.early = (mode != kModeExpand && a.n >= 2 * a.n_keys) ? 1 : 0;
}

template <int RMAX, int MODE, class Tables>
int launch_delta_r(const DeltaArgs& a, const Tables& tb, int n_keys, int smem,
                   cudaStream_t stream) {
  auto kernel = delta_cluster_kernel<RMAX, MODE, Tables>;
  const int cs = a.cs;
  cudaError_t e = prepare_kernel(kernel, smem, cs > 8);
  if (e != cudaSuccess) return LORA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(n_keys * cs), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = use_pdl() ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, kernel, a, tb);
  return cuda_status(e);
}

// The fused small-segment kernel for one k stage per CTA (bgmv_fused_kernel);
// LORA_FUSED_KERNEL=0 keeps every fused call on the general cluster kernel.
bool fused_kernel_on() {
  static const bool on = env_int("LORA_FUSED_KERNEL", 1) != 0;
  return on;
}

template <int RMAX, class Tables>
int launch_fused_r(const DeltaArgs& a, const Tables& tb, int n_keys, int smem,
                   cudaStream_t stream) {
  auto kernel = bgmv_fused_kernel<RMAX, Tables>;
  const int cs = a.cs;
  if (prepare_kernel(kernel, smem, cs > 8) != cudaSuccess) return LORA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(n_keys * cs), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = use_pdl() ? 2 : 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, kernel, a, tb));
}

template <int MODE, class Tables>
int launch_delta(const DeltaArgs& a, const Tables& tb, int n_keys, cudaStream_t s) {
  if (MODE == kModeFused && fused_kernel_on() && fused_kernel_fits(a)) {
    const int smem = fused_plan(a).total;
    if (smem <= 226 * 1024) {
      if (a.R <= 16) return launch_fused_r<16>(a, tb, n_keys, smem, s);
      if (a.R <= 32) return launch_fused_r<32>(a, tb, n_keys, smem, s);
      return launch_fused_r<64>(a, tb, n_keys, smem, s);
    }
  }
  const int smem = smem_plan(a, MODE).total;
  if (smem > 226 * 1024) return LORA_ERR_UNSUPPORTED;  // leaves room for static smem
  if (a.R <= 16) return launch_delta_r<16, MODE>(a, tb, n_keys, smem, s);
  if (a.R <= 32) return launch_delta_r<32, MODE>(a, tb, n_keys, smem, s);
  if (a.R <= 64) return launch_delta_r<64, MODE>(a, tb, n_keys, smem, s);
  return launch_delta_r<128, MODE>(a, tb, n_keys, smem, s);
}

// One CTA per key (the routed-MoE deltas): S * R up to kKeyMaxSR, R <= 32.
// zero_ctas extra CTAs write zeros on the no-key bucket's rows.
template <class Tables>
int launch_key(const DeltaArgs& a, const Tables& tb, int n_keys, int zero_ctas,
               cudaStream_t stream) {
  const int sr16 = (a.sr_max + 15) / 16 * 16;
  if (sr16 > kKeyMaxSR || a.R > 32) return LORA_ERR_UNSUPPORTED;
  const int smem = key_smem(sr16).total;
  auto kernel = a.R <= 16 ? delta_key_kernel<16, Tables> : delta_key_kernel<32, Tables>;
  if (prepare_kernel(kernel, smem, false) != cudaSuccess) return LORA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  // two CTAs per key (the second takes the odd 32-row passes): keys with more
  // than one pass no longer set the length of the launch; LORA_MOE_HALVES=1
  // keeps one CTA per key
  static const int halves = env_int("LORA_MOE_HALVES", 2) == 1 ? 1 : 2;
  cfg.gridDim = dim3((unsigned)(n_keys * halves + zero_ctas), 1, 1);
  cfg.blockDim = dim3(kKeyThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = use_pdl() ? 1 : 0;
  return cuda_status(cudaLaunchKernelEx(&cfg, kernel, a, tb, zero_ctas, halves));
}

// The one-CTA-per-key kernel for the routed-MoE deltas (LORA_MOE_KEYED=0
// falls back to the cluster kernel).
bool moe_keyed() {
  static const bool on = env_int("LORA_MOE_KEYED", 1) != 0;
  return on;
}

template <class KeyFn>
int launch_route(const KeyFn& kf, int n, int n_keys, int32_t* perm, int32_t* seg_start,
                 uint32_t* err, cudaStream_t stream) {
  const int smem = (int)route_smem_bytes(n_keys);
  auto kernel = route_kernel<KeyFn>;
  cudaError_t e = prepare_kernel(kernel, smem, false);
  if (e != cudaSuccess) return LORA_ERR_CUDA;
  kernel<<<1, kRouteThreads, smem, stream>>>(kf, n, n_keys, perm, seg_start, err);
  return cuda_status(cudaGetLastError());
}

// Scratch of the chunked sort: one count per (chunk, key).
constexpr int kRouteChunkedMinItems = 2 * kRouteChunk;  // below this one CTA sorts
size_t route_counts_bytes(int n, int n_keys) {
  const int nb = (n + kRouteChunk - 1) / kRouteChunk;
  return (size_t)(nb > 0 ? nb : 1) * (size_t)(n_keys + 1) * 4;
}

// The routing sort with scratch `counts` (route_counts_bytes): chunked over
// many CTAs for large batches, one CTA otherwise.
template <class KeyFn>
int launch_route_scratch(const KeyFn& kf, int n, int n_keys, int32_t* perm, int32_t* seg_start,
                         uint32_t* counts, uint32_t* err, cudaStream_t stream) {
  if (n < kRouteChunkedMinItems) return launch_route(kf, n, n_keys, perm, seg_start, err, stream);
  const int nb = (n + kRouteChunk - 1) / kRouteChunk;
  // up to kRouteClusterMax chunks: the one-launch cluster sort
  // (LORA_ROUTE_CLUSTER=0 keeps the two kernels)
  static const bool cluster_on = env_int("LORA_ROUTE_CLUSTER", 1) != 0;
  const size_t smem_cl = route_cluster_smem_bytes(n_keys);
  if (cluster_on && nb <= kRouteClusterMax && smem_cl <= 200 * 1024) {
    auto kcl = route_cluster_kernel<KeyFn>;
    if (prepare_kernel(kcl, (int)smem_cl, nb > 8) == cudaSuccess) {
      cudaLaunchAttribute attr[2];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)nb;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[1].val.programmaticStreamSerializationAllowed = 1;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)nb);
      cfg.blockDim = dim3(kRouteThreads);
      cfg.dynamicSmemBytes = smem_cl;
      cfg.stream = stream;
      cfg.attrs = attr;
      cfg.numAttrs = use_pdl() ? 2 : 1;
      if (cudaLaunchKernelEx(&cfg, kcl, kf, n, n_keys, perm, seg_start, err) == cudaSuccess)
        return LORA_OK;
    }
    cudaGetLastError();  // (not launched: the two kernels below)
  }
  const int smem_c = (int)route_smem_bytes(n_keys), smem_s = (int)route_chunk_smem_bytes(n_keys);
  auto kc = route_count_kernel<KeyFn>;
  auto ks = route_scatter_kernel<KeyFn>;
  if (prepare_kernel(kc, smem_c, false) != cudaSuccess ||
      prepare_kernel(ks, smem_s, false) != cudaSuccess)
    return LORA_ERR_CUDA;
  kc<<<nb, kRouteThreads, smem_c, stream>>>(kf, n, n_keys, counts, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return LORA_ERR_CUDA;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nb);
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = (size_t)smem_s;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = use_pdl() ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, ks, kf, n, n_keys, (const uint32_t*)counts, perm, seg_start);
  return e == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

// Workspace layout: perm [n] int32 | seg_start [n_keys + 2] int32 |
// SGMV tiles [max_tiles] + their count | routing-sort counts [chunks, n_keys + 1] |
// h planes of the tensor-core path [planes][n, hs] fp32.
int max_sgmv_tiles(int n, int n_keys) { return n / kTileRows + (n_keys < n ? n_keys : n) + 1; }

struct Workspace {
  int32_t* perm;
  int32_t* seg;
  SgmvTile* tiles;
  int* n_tiles;
  uint32_t* rcounts;
  float* hbuf;
  size_t bytes;  // size of the whole buffer
};

constexpr int kMaxKSplit = 8;  // planes of the SGMV shrink's partial h

// Bytes before the h planes, and bytes of one plane.
size_t ws_head_bytes(int n, int n_keys) {
  const int nn = n > 0 ? n : 1;
  return align256((size_t)nn * 4) + align256((size_t)(n_keys + 2) * 4) +
         align256((size_t)max_sgmv_tiles(nn, n_keys) * sizeof(SgmvTile) + 16) +
         align256(route_counts_bytes(nn, n_keys));
}
size_t ws_plane_bytes(int n, int hs) { return align256((size_t)(n > 0 ? n : 1) * hs * 4); }

// Minimum workspace: one plane; the size query asks for kMaxKSplit planes so
// the tensor-core shrink can split k across more CTAs.
size_t ws_bytes_for(int n, int n_keys, int hs, int planes = 1) {
  return ws_head_bytes(n, n_keys) + (size_t)planes * ws_plane_bytes(n, hs);
}

int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cache[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = v > 0 ? v : 148;
  }
  return cache[dev];
}

Workspace carve(void* ws, int n, int n_keys) {
  const int nn = n > 0 ? n : 1;
  char* p = reinterpret_cast<char*>(ws);
  Workspace w;
  w.perm = reinterpret_cast<int32_t*>(p);
  p += align256((size_t)nn * 4);
  w.seg = reinterpret_cast<int32_t*>(p);
  p += align256((size_t)(n_keys + 2) * 4);
  w.n_tiles = reinterpret_cast<int*>(p);
  w.tiles = reinterpret_cast<SgmvTile*>(p + 16);
  p += align256((size_t)max_sgmv_tiles(nn, n_keys) * sizeof(SgmvTile) + 16);
  w.rcounts = reinterpret_cast<uint32_t*>(p);
  p += align256(route_counts_bytes(nn, n_keys));
  w.hbuf = reinterpret_cast<float*>(p);
  w.bytes = 0;
  return w;
}

// Rows per key from which the tensor-core (SGMV) path takes a key over from
// the small-segment kernel, by the size of a slot's weights;
// LORA_SGMV_MIN_ROWS overrides, read once.
int sgmv_min_rows(int S, int R, int k_in) {
  static const int forced = env_int("LORA_SGMV_MIN_ROWS", 0);
  if (forced >= 1) return forced;
  // Measured on GB300: a slot whose weights are large (the skewed workload,
  // R 64 over k_in 5120 / 13824: 0.64 / 1.7 MiB) streams them faster on the
  // tensor-core path from 16 rows on (0.288 against 0.331 ms at 64); a small
  // one (the expert fold, 64 KiB) keeps the cluster kernel below 64 rows.
  const int64_t slot_bytes = (int64_t)S * R * k_in * 2;
  return slot_bytes >= (512 << 10) ? 16 : 64;
}

// Batches of at least this many rows are clustered by the routing kernel when
// a workspace is given (and always above kInlineRowsMax).
constexpr int kRouteMinRows = 256;

// Common front half of the linear calls: row clustering (own scan or routing
// kernel into the workspace).  Sets *routed when the routing kernel ran.
int prepare_rows(DeltaArgs& a, const int32_t* seq_slot, int n, int max_loras, int hs,
                 void* workspace, size_t ws_bytes, uint32_t* err, cudaStream_t stream,
                 Workspace* wout) {
  a.seq_slot = seq_slot;
  a.n = n;
  a.n_keys = max_loras;
  a.err = err;
  const bool want_route = n > kInlineRowsMax || (workspace != nullptr && n >= kRouteMinRows);
  if (!want_route) {
    a.perm = nullptr;
    a.seg_start = nullptr;
    a.row_cap = n;
    return LORA_OK;
  }
  if (!workspace || ws_bytes < ws_bytes_for(n, max_loras, hs)) return LORA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LORA_ERR_ALIGN;
  const Workspace w = carve(workspace, n, max_loras);
  const int rc = launch_route_scratch(SlotKey{seq_slot, max_loras}, n, max_loras, w.perm, w.seg,
                                      w.rcounts, err, stream);
  if (rc) return rc;
  a.perm = w.perm;
  a.seg_start = w.seg;
  a.row_cap = 0;
  if (wout) {
    *wout = w;
    wout->bytes = ws_bytes;
  }
  return LORA_OK;
}

// 2-D tensor maps for TMA loads of row blocks (128 rows x 64 columns, bf16,
// 128-byte swizzle) of a row-major [rows, cols] matrix with leading dimension
// ld; the encoder comes from the driver through the runtime, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      p = nullptr;
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}
bool encode_row_blocks(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc || rows < 1 || cols < 1) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kTileRows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// TMA loads of the activation tiles on the tensor-core path when the rows of
// each key are already contiguous; LORA_SGMV_TMA=0 keeps the cp.async copies.
bool sgmv_tma_on() {
  static const bool on = env_int("LORA_SGMV_TMA", 1) != 0;
  return on;
}

// Launch of the tensor-core path for the keys with >= min_rows rows.  With
// tmx and tmo (tensor maps of x and out), the tiles' rows are contiguous.
template <class Tables>
int launch_sgmv(const DeltaArgs& d, const Tables& tb, const Workspace& w, int n_keys,
                int min_rows, cudaStream_t stream, const CUtensorMap* tmx = nullptr,
                const CUtensorMap* tmo = nullptr) {
  static const CUtensorMap no_map = {};
  SgmvArgs s = {};
  s.out = d.out;
  s.ld_out = d.ld_out;
  s.x = d.x;
  s.ld_x = d.ld_x;
  s.k_in = d.k_in;
  s.perm = w.perm;
  s.tiles = w.tiles;
  s.n_tiles = w.n_tiles;
  s.hbuf = w.hbuf;
  s.hs = (d.sr_max + 15) / 16 * 16;
  const int max_tiles = max_sgmv_tiles(d.n, n_keys);
  // the shrink runs persistent: `slots` resident CTAs walk (tile, split)
  // items; the tile kernel picks the split from the true tile count, within
  // the planes the workspace holds
  const int shrink_smem = sgmv_shrink_smem(d.sr_max);
  if (prepare_kernel(sgmv_shrink_kernel<Tables>, shrink_smem, false) != cudaSuccess)
    return LORA_ERR_CUDA;
  // (each shrink CTA holds kSgmvMaxSR of the SM's 512 TMEM columns)
  int per_sm = ctas_per_sm(sgmv_shrink_kernel<Tables>, kShrinkThreads, shrink_smem);
  if (per_sm > 512 / kSgmvMaxSR) per_sm = 512 / kSgmvMaxSR;
  const int slots = per_sm * sm_count();
  static const int ks_cap = [] {
    const int v = env_int("LORA_SHRINK_KS_MAX", kMaxKSplit);
    return v >= 1 && v <= kMaxKSplit ? v : kMaxKSplit;
  }();
  int ks_max = ks_cap;
  {
    const int nkb = (d.k_in + 63) / 64;
    if (ks_max > nkb) ks_max = nkb;
    const size_t head = ws_head_bytes(d.n, n_keys), plane = ws_plane_bytes(d.n, s.hs);
    const int fit = w.bytes > head ? (int)((w.bytes - head) / plane) : 0;
    if (ks_max > fit) ks_max = fit;
    if (ks_max < 1) ks_max = 1;
    s.ksplit = w.n_tiles + 1;
    s.plane = (int64_t)(plane / 4);
  }
  s.R = d.R;
  s.sl = d.sl;
  for (int j = 0; j <= kMaxSlices; ++j) s.rel[j] = d.rel[j];
  int nch = 0;
  for (int j = 0; j < kMaxSlices; ++j) {
    s.chunk0[j] = nch;
    if (j < d.sl.S) nch += (d.sl.width[j] + kExpandCols - 1) / kExpandCols;
  }
  s.chunk0[kMaxSlices] = nch;
  s.add_inputs = d.add_inputs;
  s.err = d.err;
  s.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  s.contig = (tmx && tmo) ? 1 : 0;
  const CUtensorMap& map_x = s.contig ? *tmx : no_map;
  const CUtensorMap& map_out = s.contig ? *tmo : no_map;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = use_pdl() ? 1 : 0;
  // tile list
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, sgmv_tiles_kernel, (const int32_t*)d.seg_start, n_keys,
                                     min_rows, w.tiles, w.n_tiles, max_tiles, slots, ks_max);
  if (e != cudaSuccess) return LORA_ERR_CUDA;
  // shrink
  {
    auto kernel = sgmv_shrink_kernel<Tables>;
    const int64_t most = (int64_t)max_tiles * ks_max;  // items at most
    cfg.gridDim = dim3((unsigned)(most < slots ? most : slots));
    cfg.blockDim = dim3(kShrinkThreads);
    cfg.dynamicSmemBytes = (size_t)shrink_smem;
    if ((e = cudaLaunchKernelEx(&cfg, kernel, s, tb, map_x)) != cudaSuccess) return LORA_ERR_CUDA;
  }
  // expand: persistent, one CTA per SM
  {
    const int smem = sgmv_expand_smem(d.R);
    // one CTA per SM, more if needed so that no CTA spans more than
    // kExpandMaxTiles tiles (<= kExpandMaxTiles - 2 tiles' worth of items each)
    const int64_t items = (int64_t)max_tiles * nch;
    int64_t grid = sm_count();
    const int64_t need = (max_tiles + (kExpandMaxTiles - 2) - 1) / (kExpandMaxTiles - 2);
    if (grid < need) grid = need;
    if (grid > items) grid = items;
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kExpandThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    if (d.R <= 64) {
      auto kernel = sgmv_expand_kernel<64, Tables>;
      if ((e = prepare_kernel(kernel, smem, false)) != cudaSuccess) return LORA_ERR_CUDA;
      e = cudaLaunchKernelEx(&cfg, kernel, s, tb, nch, map_out);
    } else {
      auto kernel = sgmv_expand_kernel<128, Tables>;
      if ((e = prepare_kernel(kernel, smem, false)) != cudaSuccess) return LORA_ERR_CUDA;
      e = cudaLaunchKernelEx(&cfg, kernel, s, tb, nch, map_out);
    }
    if (e != cudaSuccess) return LORA_ERR_CUDA;
  }
  return LORA_OK;
}

int check_max_loras(int max_loras) {
  if (max_loras < 1) return LORA_ERR_ARG;
  if (max_loras > kMaxKeys) return LORA_ERR_UNSUPPORTED;
  return LORA_OK;
}

// A call whose keys split between the small-segment kernel and the
// tensor-core path runs the two on disjoint rows and separate weights, so the
// small-segment launch goes to a second stream of the device (forked from the
// caller's stream by an event and joined back by another) and the two share
// the GPU: each leaves DRAM idle in phases the other fills (the skewed decode
// workload: 0.284 -> 0.245 ms).  One side stream and event pair per device,
// created outside stream capture on first use; a call made while the caller's
// stream is being captured before that runs both parts on the caller's stream.
// Fork and join are recorded under a lock, so calls from several host threads
// keep their pairs apart (their small-segment launches then queue on the one
// side stream).  LORA_FORK=0 keeps everything on the caller's stream.
struct ForkStreams {
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxDevices = 64;
std::mutex g_fork_mu;
ForkStreams g_fork[kMaxDevices];

bool fork_on() {
  static const bool on = env_int("LORA_FORK", 1) != 0;
  return on;
}

// The device's side stream and events, or nullptr (fork off, not creatable
// now, or an unknown device); called with g_fork_mu held.
ForkStreams* fork_streams(cudaStream_t caller) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  ForkStreams& f = g_fork[dev];
  if (f.side) return &f;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(caller, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return nullptr;
  }
  ForkStreams g;
  if (cudaStreamCreateWithFlags(&g.side, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&g.fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&g.join, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    if (g.join) cudaEventDestroy(g.join);
    if (g.fork) cudaEventDestroy(g.fork);
    if (g.side) cudaStreamDestroy(g.side);
    return nullptr;
  }
  f = g;
  return &f;
}

// launch_delta<kModeFused> for the small keys and launch_sgmv for the others,
// forked as above when possible.
template <class Tables>
int launch_split(const DeltaArgs& a, const Tables& tb, const Workspace& w, int n_keys, int thr,
                 cudaStream_t s, const CUtensorMap* tmx = nullptr,
                 const CUtensorMap* tmo = nullptr) {
  if (fork_on()) {
    std::lock_guard<std::mutex> lock(g_fork_mu);
    ForkStreams* f = fork_streams(s);
    if (f) {
      if (cudaEventRecord(f->fork, s) != cudaSuccess ||
          cudaStreamWaitEvent(f->side, f->fork, 0) != cudaSuccess)
        return LORA_ERR_CUDA;
      const int rc1 = launch_delta<kModeFused>(a, tb, n_keys, f->side);
      const int rc2 = launch_sgmv(a, tb, w, n_keys, thr, s, tmx, tmo);
      // joined whatever the launches returned (a capture must not be left forked)
      const bool joined = cudaEventRecord(f->join, f->side) == cudaSuccess &&
                          cudaStreamWaitEvent(s, f->join, 0) == cudaSuccess;
      if (rc1) return rc1;
      if (rc2) return rc2;
      return joined ? LORA_OK : LORA_ERR_CUDA;
    }
  }
  const int rc = launch_delta<kModeFused>(a, tb, n_keys, s);
  return rc ? rc : launch_sgmv(a, tb, w, n_keys, thr, s, tmx, tmo);
}

// A batch small enough for the kernels' own row scan that still goes through
// the routing sort for the tensor-core path: forked before the sort, the
// small-segment kernel finds its keys' rows by that scan on the side stream
// (skipping keys with thr rows or more), so it does not wait for the sort.
// Returns kNoFork, having launched nothing, when there is no side stream.
constexpr int kNoFork = -1;
int launch_split_scan(DeltaArgs& a, const LinearTables& tb, const int32_t* seq_slot, int n,
                      int n_keys, int hs, int thr, void* workspace, size_t ws_bytes,
                      uint32_t* err, cudaStream_t s) {
  if (!fork_on()) return kNoFork;
  // (the checks of the routing pass, before anything is launched)
  if (ws_bytes < ws_bytes_for(n, n_keys, hs)) return LORA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LORA_ERR_ALIGN;
  DeltaArgs c = a;
  prepare_rows(c, seq_slot, n, n_keys, hs, nullptr, 0, err, s, nullptr);  // (own scan)
  plan_tiles(c, a.k_in, a.sl.n_cols, a.sr_max, kModeFused);
  c.max_rows = thr;
  if (n >= (int64_t)thr * n_keys) c.early = 0;
  std::lock_guard<std::mutex> lock(g_fork_mu);
  ForkStreams* f = fork_streams(s);
  if (!f) return kNoFork;
  if (cudaEventRecord(f->fork, s) != cudaSuccess ||
      cudaStreamWaitEvent(f->side, f->fork, 0) != cudaSuccess)
    return LORA_ERR_CUDA;
  const int rc1 = launch_delta<kModeFused>(c, tb, n_keys, f->side);
  Workspace w = {};
  int rc2 = prepare_rows(a, seq_slot, n, n_keys, hs, workspace, ws_bytes, err, s, &w);
  if (!rc2) {
    plan_tiles(a, a.k_in, a.sl.n_cols, a.sr_max, kModeFused);
    rc2 = launch_sgmv(a, tb, w, n_keys, thr, s);
  }
  const bool joined = cudaEventRecord(f->join, f->side) == cudaSuccess &&
                      cudaStreamWaitEvent(s, f->join, 0) == cudaSuccess;
  if (rc1) return rc1;
  if (rc2) return rc2;
  return joined ? LORA_OK : LORA_ERR_CUDA;
}

}  // namespace

// ------------------------------------------------------------------ pack --
__global__ void pool_pack_kernel(__nv_bfloat16* __restrict__ a_slot,
                                 __nv_bfloat16* __restrict__ b_slot,
                                 const __nv_bfloat16* __restrict__ a_r,
                                 const __nv_bfloat16* __restrict__ b_r, int r, int R, int k_in,
                                 int w) {
  const int64_t na = (int64_t)R * k_in, nb = (int64_t)w * R;
  const __nv_bfloat16 zero = __float2bfloat16_rn(0.0f);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < na + nb;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < na) {
      const int q = (int)(i / k_in);
      a_slot[i] = (q < r) ? a_r[i] : zero;  // row q < r of a_r sits at the same offset
    } else {
      const int64_t t = i - na;
      const int c = (int)(t / R), q = (int)(t - (int64_t)c * R);
      b_slot[t] = (q < r) ? b_r[(int64_t)c * r + q] : zero;
    }
  }
}

__global__ void clear_word_kernel(uint32_t* w) { *w = 0u; }

// Plan of a call on rows already grouped by adapter ("expert_apply.rs",
// expert_delta_workitems, done on the device from the device offsets): the
// identity row permutation, and the segment starts made nondecreasing within
// [0, n] (a start out of order or past n is clamped, nothing is read outside
// the batch, and LORA_DEV_ERR_SEGMENT is set); rows past the last segment
// form the no-adapter bucket.
__global__ void segment_plan_kernel(const int32_t* __restrict__ offsets, int n_segs, int n,
                                    int32_t* __restrict__ perm, int32_t* __restrict__ seg,
                                    uint32_t* err) {
  __shared__ int off_s[kMaxKeys + 1];
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) perm[i] = i;
  if (blockIdx.x != 0) return;
  for (int s = threadIdx.x; s <= n_segs; s += blockDim.x) off_s[s] = offsets[s];  // one round trip
  __syncthreads();
  if (threadIdx.x == 0) {
    int prev = 0;
    bool bad = false;
    for (int s = 0; s <= n_segs; ++s) {
      int v = off_s[s];
      if (s == 0 && v != 0) bad = true;  // segment 0 starts at row 0
      if (v < prev || v > n) {
        bad = true;
        v = v < prev ? prev : n;
      }
      if (s == 0) v = 0;
      seg[s] = v;
      prev = v;
    }
    seg[n_segs + 1] = n;
    if (bad) set_error(err, LORA_DEV_ERR_SEGMENT);
  }
}

namespace {

// lora_expand and lora_expand_gathered: h as [parts][S][n][R / parts].
int expand_parts(void* out, int64_t ld_out, const float* h, int parts, const int32_t* seq_slot,
                 const uint64_t* b_table, const float* scale_table, const int32_t* widths, int S,
                 int R, int n, int max_loras, int offset_start, int add_inputs, void* workspace,
                 size_t ws_bytes, uint32_t* err_word, lora_stream_t stream) {
  if (n < 0) return LORA_ERR_ARG;
  if (n == 0) return LORA_OK;
  if (!out || !h || !seq_slot || !b_table) return LORA_ERR_ARG;
  int rc = check_max_loras(max_loras);
  if (rc) return rc;
  DeltaArgs a = {};
  if ((rc = make_slices(widths, S, offset_start, a.sl, a.rel))) return rc;
  if ((rc = check_rank(S, R))) return rc;
  if (ld_out < (int64_t)offset_start + a.sl.n_cols) return LORA_ERR_SHAPE;
  if (ld_out % 8 || !aligned16(out) || !aligned16(h)) return LORA_ERR_ALIGN;
  if (a.sl.n_cols == 0) return LORA_OK;
  a.out = (__nv_bfloat16*)out;
  a.ld_out = ld_out;
  a.h = (float*)h;
  a.R = R;
  a.add_inputs = add_inputs ? 1 : 0;
  a.sr_max = S * R;
  rc = prepare_rows(a, seq_slot, n, max_loras, (S * R + 15) / 16 * 16, workspace, ws_bytes,
                    err_word, (cudaStream_t)stream, nullptr);
  if (rc) return rc;
  a.h_parts = parts;
  plan_tiles(a, 8, a.sl.n_cols, a.sr_max, kModeExpand);
  LinearTables tb{nullptr, b_table, scale_table, max_loras};
  return launch_delta<kModeExpand>(a, tb, max_loras, (cudaStream_t)stream);
}

}  // namespace

extern "C" {

const char* lora_status_string(int status) {
  switch (status) {
    case LORA_OK: return "LORA_OK";
    case LORA_ERR_ARG: return "LORA_ERR_ARG";
    case LORA_ERR_SHAPE: return "LORA_ERR_SHAPE";
    case LORA_ERR_ALIGN: return "LORA_ERR_ALIGN";
    case LORA_ERR_CUDA: return "LORA_ERR_CUDA";
    case LORA_ERR_WORKSPACE: return "LORA_ERR_WORKSPACE";
    case LORA_ERR_UNSUPPORTED: return "LORA_ERR_UNSUPPORTED";
    case LORA_ERR_TOO_LARGE: return "LORA_ERR_TOO_LARGE";
    default: return "LORA_ERR_UNKNOWN";
  }
}

int lora_abi_version(void) { return kAbiVersion; }

uint64_t lora_set_wait_limit_ns(uint64_t ns) {
  return g_wait_limit_ns.exchange(ns, std::memory_order_relaxed);
}

float lora_scale(float alpha, int r, int use_rslora) {
  if (r <= 0) return 0.0f;
  return use_rslora ? (float)((double)alpha / sqrt((double)r)) : (float)((double)alpha / r);
}

int lora_pool_pack(void* a_slot, void* b_slot, const void* a_r, const void* b_r, int r, int R,
                   int k_in, int w, lora_stream_t stream) {
  if (!a_slot || !b_slot || r < 0 || r > R || k_in < 0 || w < 0) return LORA_ERR_ARG;
  if (r > 0 && (!a_r || !b_r)) return LORA_ERR_ARG;
  const int64_t total = (int64_t)R * k_in + (int64_t)w * R;
  if (total == 0) return LORA_OK;
  const int blocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
  pool_pack_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(
      (__nv_bfloat16*)a_slot, (__nv_bfloat16*)b_slot, (const __nv_bfloat16*)a_r,
      (const __nv_bfloat16*)b_r, r, R, k_in, w);
  return cuda_status(cudaGetLastError());
}

size_t lora_workspace_size(int n, int S, int R, int max_loras) {
  if (n < 0 || max_loras < 1 || S < 1 || R < 1) return 0;
  return ws_bytes_for(n, max_loras, (S * R + 15) / 16 * 16, kMaxKSplit);
}

size_t lora_workspace_min_size(int n, int S, int R, int max_loras) {
  if (n < 0 || max_loras < 1 || S < 1 || R < 1) return 0;
  return ws_bytes_for(n, max_loras, (S * R + 15) / 16 * 16, 1);
}

size_t lora_route_scratch_size(int n, int max_loras) {
  if (n < 0 || max_loras < 1) return 0;
  return route_counts_bytes(n, max_loras);
}

int lora_route_with_scratch(int32_t* perm, int32_t* seg_start, const int32_t* seq_slot, int n,
                            int max_loras, void* scratch, size_t scratch_bytes,
                            uint32_t* err_word, lora_stream_t stream) {
  if (n < 0 || !seg_start || (n > 0 && (!perm || !seq_slot))) return LORA_ERR_ARG;
  int rc = check_max_loras(max_loras);
  if (rc) return rc;
  if (!scratch || scratch_bytes < route_counts_bytes(n, max_loras)) return LORA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(scratch) & 15u) != 0) return LORA_ERR_ALIGN;
  return launch_route_scratch(SlotKey{seq_slot, max_loras}, n, max_loras, perm, seg_start,
                              reinterpret_cast<uint32_t*>(scratch), err_word,
                              (cudaStream_t)stream);
}

int lora_route(int32_t* perm, int32_t* seg_start, const int32_t* seq_slot, int n, int max_loras,
               uint32_t* err_word, lora_stream_t stream) {
  if (n < 0 || !seg_start || (n > 0 && (!perm || !seq_slot))) return LORA_ERR_ARG;
  int rc = check_max_loras(max_loras);
  if (rc) return rc;
  return launch_route(SlotKey{seq_slot, max_loras}, n, max_loras, perm, seg_start, err_word,
                      (cudaStream_t)stream);
}

int lora_shrink(float* h, const void* x, int n, int k_in, const int32_t* seq_slot,
                const uint64_t* a_table, const float* scale_table, int S, int R, int max_loras,
                void* workspace, size_t ws_bytes, uint32_t* err_word, lora_stream_t stream) {
  if (n < 0 || k_in < 0) return LORA_ERR_ARG;
  if (n == 0) return LORA_OK;
  if (!h || !x || !seq_slot || !a_table) return LORA_ERR_ARG;
  int rc = check_max_loras(max_loras);
  if (rc) return rc;
  if (S < 1 || S > kMaxSlices) return S > kMaxSlices ? LORA_ERR_UNSUPPORTED : LORA_ERR_ARG;
  if ((rc = check_rank(S, R))) return rc;
  if (k_in % 8 || !aligned16(x) || !aligned16(h)) return LORA_ERR_ALIGN;
  if (k_in == 0) return LORA_OK;
  DeltaArgs a = {};
  a.x = (const __nv_bfloat16*)x;
  a.ld_x = k_in;
  a.k_in = k_in;
  a.h = h;
  a.R = R;
  a.sl.S = S;
  a.sr_max = S * R;
  rc = prepare_rows(a, seq_slot, n, max_loras, (S * R + 15) / 16 * 16, workspace, ws_bytes,
                    err_word, (cudaStream_t)stream, nullptr);
  if (rc) return rc;
  plan_tiles(a, k_in, 8, a.sr_max, kModeShrink);
  LinearTables tb{a_table, nullptr, scale_table, max_loras};
  return launch_delta<kModeShrink>(a, tb, max_loras, (cudaStream_t)stream);
}

int lora_expand(void* out, int64_t ld_out, const float* h, const int32_t* seq_slot,
                const uint64_t* b_table, const float* scale_table, const int32_t* widths, int S,
                int R, int n, int max_loras, int offset_start, int add_inputs, void* workspace,
                size_t ws_bytes, uint32_t* err_word, lora_stream_t stream) {
  return expand_parts(out, ld_out, h, 1, seq_slot, b_table, scale_table, widths, S, R, n,
                      max_loras, offset_start, add_inputs, workspace, ws_bytes, err_word, stream);
}

int lora_expand_gathered(void* out, int64_t ld_out, const float* h, int parts,
                         const int32_t* seq_slot, const uint64_t* b_table,
                         const float* scale_table, const int32_t* widths, int S, int R, int n,
                         int max_loras, int offset_start, int add_inputs, void* workspace,
                         size_t ws_bytes, uint32_t* err_word, lora_stream_t stream) {
  if (parts < 1 || R < 1 || R % parts) return LORA_ERR_ARG;
  return expand_parts(out, ld_out, h, parts, seq_slot, b_table, scale_table, widths, S, R, n,
                      max_loras, offset_start, add_inputs, workspace, ws_bytes, err_word, stream);
}


int lora_delta_segmented(void* out, int64_t ld_out, const void* x, int n, int k_in,
                         const int32_t* seg_start, int n_segs, const uint64_t* a_table,
                         const uint64_t* b_table, const float* scale_table, const int32_t* widths,
                         int S, int R, int offset_start, int add_inputs, void* workspace,
                         size_t ws_bytes, uint32_t* err_word, lora_stream_t stream) {
  if (n < 0 || k_in < 0) return LORA_ERR_ARG;
  if (n == 0) return LORA_OK;
  if (!out || !x || !seg_start || !a_table || !b_table) return LORA_ERR_ARG;
  int rc = check_max_loras(n_segs);
  if (rc) return rc;
  DeltaArgs a = {};
  if ((rc = make_slices(widths, S, offset_start, a.sl, a.rel))) return rc;
  if ((rc = check_rank(S, R))) return rc;
  if (ld_out < (int64_t)offset_start + a.sl.n_cols) return LORA_ERR_SHAPE;
  if (k_in % 8 || ld_out % 8 || !aligned16(out) || !aligned16(x)) return LORA_ERR_ALIGN;
  if (a.sl.n_cols == 0) return LORA_OK;
  const int hs = (S * R + 15) / 16 * 16;
  if (!workspace || ws_bytes < ws_bytes_for(n, n_segs, hs)) return LORA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LORA_ERR_ALIGN;
  cudaStream_t st = (cudaStream_t)stream;
  Workspace w = carve(workspace, n, n_segs);
  w.bytes = ws_bytes;
  segment_plan_kernel<<<(n + 1023) / 1024, 1024, 0, st>>>(seg_start, n_segs, n, w.perm, w.seg,
                                                         err_word);
  if (cudaGetLastError() != cudaSuccess) return LORA_ERR_CUDA;
  a.out = (__nv_bfloat16*)out;
  a.ld_out = ld_out;
  a.x = (const __nv_bfloat16*)x;
  a.ld_x = k_in;
  a.k_in = k_in;
  a.R = R;
  a.add_inputs = add_inputs ? 1 : 0;
  a.sr_max = S * R;
  a.seq_slot = nullptr;
  a.n = n;
  a.n_keys = n_segs;
  a.err = err_word;
  a.perm = w.perm;
  a.seg_start = w.seg;
  a.row_cap = 0;
  plan_tiles(a, k_in, a.sl.n_cols, a.sr_max, kModeFused);
  LinearTables tb{a_table, b_table, scale_table, n_segs};
  const bool sgmv = a.sr_max <= kSgmvMaxSR;
  const int thr = sgmv_min_rows(S, R, k_in);
  if (sgmv) a.max_rows = thr;
  if (!sgmv) return launch_delta<kModeFused>(a, tb, n_segs, st);
  // the rows of a segment are consecutive rows of x and out: the tensor-core
  // tiles take them by TMA
  CUtensorMap tmx, tmo;
  const bool tma = sgmv_tma_on() && encode_row_blocks(&tmx, x, n, k_in, k_in) &&
                   encode_row_blocks(&tmo, out, n, ld_out, ld_out);
  return tma ? launch_split(a, tb, w, n_segs, thr, st, &tmx, &tmo)
             : launch_split(a, tb, w, n_segs, thr, st);
}

int lora_delta_fused(void* out, int64_t ld_out, const void* x, int n, int k_in,
                     const int32_t* seq_slot, const uint64_t* a_table, const uint64_t* b_table,
                     const float* scale_table, const int32_t* widths, int S, int R,
                     int max_loras, int offset_start, int add_inputs, void* workspace,
                     size_t ws_bytes, uint32_t* err_word, lora_stream_t stream) {
  if (n < 0 || k_in < 0) return LORA_ERR_ARG;
  if (n == 0) return LORA_OK;
  if (!out || !x || !seq_slot || !a_table || !b_table) return LORA_ERR_ARG;
  int rc = check_max_loras(max_loras);
  if (rc) return rc;
  DeltaArgs a = {};
  if ((rc = make_slices(widths, S, offset_start, a.sl, a.rel))) return rc;
  if ((rc = check_rank(S, R))) return rc;
  if (ld_out < (int64_t)offset_start + a.sl.n_cols) return LORA_ERR_SHAPE;
  if (k_in % 8 || ld_out % 8 || !aligned16(out) || !aligned16(x)) return LORA_ERR_ALIGN;
  if (a.sl.n_cols == 0) return LORA_OK;
  a.out = (__nv_bfloat16*)out;
  a.ld_out = ld_out;
  a.x = (const __nv_bfloat16*)x;
  a.ld_x = k_in;
  a.k_in = k_in;
  a.R = R;
  a.add_inputs = add_inputs ? 1 : 0;
  a.sr_max = S * R;
  const int hs = (S * R + 15) / 16 * 16;
  const int thr = sgmv_min_rows(S, R, k_in);
  LinearTables tb{a_table, b_table, scale_table, max_loras};
  if (n <= kInlineRowsMax && workspace && n >= kRouteMinRows && a.sr_max <= kSgmvMaxSR) {
    rc = launch_split_scan(a, tb, seq_slot, n, max_loras, hs, thr, workspace, ws_bytes, err_word,
                           (cudaStream_t)stream);
    if (rc != kNoFork) return rc;
  }
  Workspace w = {};
  rc = prepare_rows(a, seq_slot, n, max_loras, hs, workspace, ws_bytes, err_word,
                    (cudaStream_t)stream, &w);
  if (rc) return rc;
  plan_tiles(a, k_in, a.sl.n_cols, a.sr_max, kModeFused);
  // keys with many rows go to the tensor-core path, the others stay here
  const bool sgmv = a.perm != nullptr && a.sr_max <= kSgmvMaxSR;
  if (sgmv) a.max_rows = thr;
  // when the average slot has enough rows for the tensor-core path, most
  // slots will leave the cluster kernel at once: no early weight copies
  if (sgmv && n >= (int64_t)thr * max_loras) a.early = 0;
  if (!sgmv) return launch_delta<kModeFused>(a, tb, max_loras, (cudaStream_t)stream);
  return launch_split(a, tb, w, max_loras, thr, (cudaStream_t)stream);
}

int lora_delta_fused_floor(void* out, int64_t ld_out, const void* x, int n, int k_in,
                           const int32_t* seq_slot, const uint64_t* a_table,
                           const uint64_t* b_table, const int32_t* widths, int S, int R,
                           int max_loras, int offset_start, lora_stream_t stream) {
  if (n < 0 || k_in < 0) return LORA_ERR_ARG;
  if (n == 0) return LORA_OK;
  if (!out || !x || !seq_slot || !a_table || !b_table) return LORA_ERR_ARG;
  int rc = check_max_loras(max_loras);
  if (rc) return rc;
  DeltaArgs a = {};
  if ((rc = make_slices(widths, S, offset_start, a.sl, a.rel))) return rc;
  if ((rc = check_rank(S, R))) return rc;
  if (ld_out < (int64_t)offset_start + a.sl.n_cols) return LORA_ERR_SHAPE;
  if (k_in % 8 || ld_out % 8 || !aligned16(out) || !aligned16(x)) return LORA_ERR_ALIGN;
  if (a.sl.n_cols == 0) return LORA_OK;
  if (n > kInlineRowsMax) return LORA_ERR_UNSUPPORTED;  // (rows found by the kernel's own scan)
  a.out = (__nv_bfloat16*)out;
  a.ld_out = ld_out;
  a.x = (const __nv_bfloat16*)x;
  a.ld_x = k_in;
  a.k_in = k_in;
  a.R = R;
  a.add_inputs = 1;
  a.sr_max = S * R;
  rc = prepare_rows(a, seq_slot, n, max_loras, (S * R + 15) / 16 * 16, nullptr, 0, nullptr,
                    (cudaStream_t)stream, nullptr);
  if (rc) return rc;
  plan_tiles(a, k_in, a.sl.n_cols, a.sr_max, kModeFused);
  if (!fused_kernel_fits(a)) return LORA_ERR_UNSUPPORTED;
  const int smem = fused_plan(a).total;
  if (smem > 226 * 1024) return LORA_ERR_UNSUPPORTED;
  LinearTables tb{a_table, b_table, nullptr, max_loras};
  auto kernel = bgmv_floor_kernel;
  if (prepare_kernel(kernel, smem, a.cs > 8) != cudaSuccess) return LORA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(max_loras * a.cs), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = use_pdl() ? 2 : 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, kernel, a, tb));
}

size_t lora_moe_workspace_size(int T, int top_k, int E, int num_loras, int rank, int shared_a) {
  if (T < 0 || top_k < 0 || E < 1 || num_loras < 1 || rank < 1) return 0;
  const int hs = ((shared_a ? 1 : 2) * rank + 15) / 16 * 16;
  return ws_bytes_for(T * top_k, E * num_loras, hs, kMaxKSplit);
}

}  // extern "C"

namespace {

// One routed-MoE delta over the T * top_k (token, slot) pairs, keyed by
// (adapter, local expert): FC1 (fresh output), w13 and w2 (in place).
struct MoeCall {
  void* out;
  int64_t ld_out;
  const void* x;
  int64_t ld_x;
  int k_in, x_div, n_slices;
  int32_t widths[2];
  const int64_t *w_ptr_a, *w_ptr_b;
  int64_t stride_a, stride_b;
  const int32_t *topk_ids, *lora_ids, *expert_map, *adapter_enabled;
  const float* pair_weight;
  int n_global, T, top_k, E, H, I, rank, num_loras;
  float scale;
  int add_inputs;
  int zero_skipped;  // write zeros on the pairs with no delta (fresh output)
  int routed;        // the workspace already holds this call's routing (w2 after w13)
};

int moe_delta(const MoeCall& c, void* workspace, size_t ws_bytes, uint32_t* err_word,
              cudaStream_t s) {
  const int64_t n64 = (int64_t)c.T * c.top_k;
  const int n_cols = c.widths[0] + (c.n_slices > 1 ? c.widths[1] : 0);
  if (n64 == 0 || n_cols == 0) return LORA_OK;
  if (n64 > (1 << 30)) return LORA_ERR_UNSUPPORTED;
  if (!c.out || !c.x || !c.w_ptr_a || !c.w_ptr_b || (!c.routed && (!c.topk_ids || !c.lora_ids)))
    return LORA_ERR_ARG;
  if (c.expert_map && c.n_global < 1) return LORA_ERR_ARG;
  if ((int64_t)c.E * c.num_loras > kMaxKeys) return LORA_ERR_UNSUPPORTED;
  int rc = check_rank(c.n_slices, c.rank);
  if (rc) return rc;
  if (c.H % 8 || c.I % 8 || c.k_in % 8 || n_cols % 8 || c.ld_x % 8 || c.ld_out % 8 || c.stride_a % 8 ||
      c.stride_b % 8 || !aligned16(c.out) || !aligned16(c.x))
    return LORA_ERR_ALIGN;
  const int n = (int)n64, n_keys = c.E * c.num_loras;
  const int hs = (c.n_slices * c.rank + 15) / 16 * 16;
  if (!workspace || ws_bytes < ws_bytes_for(n, n_keys, hs)) return LORA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LORA_ERR_ALIGN;
  const Workspace w = carve(workspace, n, n_keys);
  int32_t* perm = w.perm;
  int32_t* seg = w.seg;
  if (!c.routed) {
    rc = launch_route_scratch(MoeKey{c.topk_ids, c.lora_ids, c.expert_map, c.adapter_enabled,
                                     c.top_k, c.E, c.num_loras, c.n_global},
                              n, n_keys, perm, seg, w.rcounts, err_word, s);
    if (rc) return rc;
  }

  DeltaArgs a = {};
  if ((rc = make_slices(c.widths, c.n_slices, 0, a.sl, a.rel))) return rc;
  a.out = (__nv_bfloat16*)c.out;
  a.ld_out = c.ld_out;
  a.x = (const __nv_bfloat16*)c.x;
  a.ld_x = c.ld_x;
  a.k_in = c.k_in;
  a.R = c.rank;
  a.add_inputs = c.add_inputs;
  a.sr_max = c.n_slices * c.rank;
  a.n = n;
  a.n_keys = n_keys;
  a.perm = perm;
  a.seg_start = seg;
  a.row_cap = 0;
  a.err = err_word;
  plan_tiles(a, c.k_in, a.sl.n_cols, a.sr_max, kModeFused);
  MoeTables tb{c.w_ptr_a, c.w_ptr_b, c.stride_a, c.stride_b, c.E, c.x_div, c.n_slices,
               c.scale, c.pair_weight};
  // With LORA_MOE_SGMV_MIN_ROWS set, keys with at least that many pairs go to
  // the tensor-core path.  Off by default: at the ~26 pairs per key of a
  // top-8-of-64 routing the cluster kernel is faster (0.139 against 0.187 ms
  // on GB300), and the tensor-core kernels cost ~10 us of launches per call
  // even when no key qualifies.  Its epilogue folds one scale per key, so
  // calls with routing weights stay on the cluster kernel.
  static const int moe_thr = env_int("LORA_MOE_SGMV_MIN_ROWS", 0);
  const bool sgmv = moe_thr >= 1 && a.sr_max <= kSgmvMaxSR && !c.pair_weight;
  if (sgmv) a.max_rows = moe_thr;
  // One CTA per key (S * R <= 64, rank <= 32): FC1 regular 0.107 against
  // 0.135 ms on the cluster kernel (GB300), w13 0.126 against 0.154, w2
  // 0.115 against 0.117.
  const bool keyed = moe_keyed() && (a.sr_max + 15) / 16 * 16 <= kKeyMaxSR && c.rank <= 32;
  // the per-key kernel also zeroes the pairs without an adapter (fresh output)
  const int zero_ctas = keyed && c.zero_skipped && !sgmv ? 64 : 0;
  rc = keyed ? launch_key(a, tb, n_keys, zero_ctas, s)
             : launch_delta<kModeFused>(a, tb, n_keys, s);
  if (rc) return rc;
  if (sgmv) {
    Workspace wb = w;
    wb.bytes = ws_bytes;
    if ((rc = launch_sgmv(a, tb, wb, n_keys, moe_thr, s))) return rc;
  }
  if (!c.zero_skipped || zero_ctas) return LORA_OK;
  // the pairs with no adapter (the no-key bucket) are written as zeros
  zero_rows_kernel<<<1024, 256, 0, s>>>(a.out, a.ld_out, n_cols, perm, seg, n_keys);
  return cuda_status(cudaGetLastError());
}

}  // namespace

extern "C" {

int lora_moe_fc1_delta(void* out, const void* x, const int64_t* w_ptr_a, int64_t stride_a,
                       const int64_t* w_ptr_b, int64_t stride_b, int shared_a,
                       const int32_t* topk_ids, const int32_t* lora_ids, int T, int top_k, int E,
                       int H, int I, int rank, int num_loras, float scale, void* workspace,
                       size_t ws_bytes, uint32_t* err_word, lora_stream_t stream) {
  if (T < 0 || top_k < 0 || E < 1 || H < 0 || I < 0 || num_loras < 1 || stride_a < 0 ||
      stride_b < 0)
    return LORA_ERR_ARG;
  MoeCall c = {};
  c.out = out;
  c.ld_out = 2 * (int64_t)I;
  c.x = x;
  c.ld_x = H;
  c.k_in = H;
  c.x_div = top_k > 0 ? top_k : 1;
  c.n_slices = shared_a ? 1 : 2;
  c.widths[0] = shared_a ? 2 * I : I;
  c.widths[1] = I;
  c.w_ptr_a = w_ptr_a;
  c.w_ptr_b = w_ptr_b;
  c.stride_a = stride_a;
  c.stride_b = stride_b;
  c.topk_ids = topk_ids;
  c.lora_ids = lora_ids;
  c.T = T;
  c.top_k = top_k;
  c.E = E;
  c.H = H;
  c.I = I;
  c.rank = rank;
  c.num_loras = num_loras;
  c.scale = scale;
  c.zero_skipped = 1;
  return moe_delta(c, workspace, ws_bytes, err_word, (cudaStream_t)stream);
}

int lora_moe_w13_delta(void* y, const void* x, const int64_t* w_ptr_a, int64_t stride_a,
                       const int64_t* w_ptr_b, int64_t stride_b, int shared_a,
                       const int32_t* topk_ids, const int32_t* lora_ids,
                       const int32_t* expert_map, int n_global_experts,
                       const int32_t* adapter_enabled, int T, int top_k, int E, int H, int I,
                       int rank, int num_loras, float scale, int add_inputs, void* workspace,
                       size_t ws_bytes, uint32_t* err_word, lora_stream_t stream) {
  if (T < 0 || top_k < 0 || E < 1 || H < 0 || I < 0 || num_loras < 1 || stride_a < 0 ||
      stride_b < 0)
    return LORA_ERR_ARG;
  MoeCall c = {};
  c.out = y;
  c.ld_out = 2 * (int64_t)I;
  c.x = x;
  c.ld_x = H;
  c.k_in = H;
  c.x_div = top_k > 0 ? top_k : 1;
  c.n_slices = shared_a ? 1 : 2;
  c.widths[0] = shared_a ? 2 * I : I;
  c.widths[1] = I;
  c.w_ptr_a = w_ptr_a;
  c.w_ptr_b = w_ptr_b;
  c.stride_a = stride_a;
  c.stride_b = stride_b;
  c.topk_ids = topk_ids;
  c.lora_ids = lora_ids;
  c.expert_map = expert_map;
  c.n_global = n_global_experts;
  c.adapter_enabled = adapter_enabled;
  c.T = T;
  c.top_k = top_k;
  c.E = E;
  c.H = H;
  c.I = I;
  c.rank = rank;
  c.num_loras = num_loras;
  c.scale = scale;
  c.add_inputs = add_inputs ? 1 : 0;
  return moe_delta(c, workspace, ws_bytes, err_word, (cudaStream_t)stream);
}

int lora_moe_w2_delta(void* y, const void* x, const int64_t* w_ptr_a, int64_t stride_a,
                      const int64_t* w_ptr_b, int64_t stride_b, const int32_t* topk_ids,
                      const int32_t* lora_ids, const int32_t* expert_map, int n_global_experts,
                      const int32_t* adapter_enabled, const float* topk_weights, int T,
                      int top_k, int E, int H, int I, int rank, int num_loras, float scale,
                      int add_inputs, void* workspace, size_t ws_bytes, uint32_t* err_word,
                      lora_stream_t stream) {
  if (T < 0 || top_k < 0 || E < 1 || H < 0 || I < 0 || num_loras < 1 || stride_a < 0 ||
      stride_b < 0)
    return LORA_ERR_ARG;
  MoeCall c = {};
  c.out = y;
  c.ld_out = H;
  c.x = x;
  c.ld_x = I;
  c.k_in = I;
  c.x_div = 1;
  c.n_slices = 1;
  c.widths[0] = H;
  c.w_ptr_a = w_ptr_a;
  c.w_ptr_b = w_ptr_b;
  c.stride_a = stride_a;
  c.stride_b = stride_b;
  c.topk_ids = topk_ids;
  c.lora_ids = lora_ids;
  c.expert_map = expert_map;
  c.n_global = n_global_experts;
  c.adapter_enabled = adapter_enabled;
  c.pair_weight = topk_weights;
  c.T = T;
  c.top_k = top_k;
  c.E = E;
  c.H = H;
  c.I = I;
  c.rank = rank;
  c.num_loras = num_loras;
  c.scale = scale;
  c.add_inputs = add_inputs ? 1 : 0;
  return moe_delta(c, workspace, ws_bytes, err_word, (cudaStream_t)stream);
}

int lora_moe_w2_delta_routed(void* y, const void* x, const int64_t* w_ptr_a, int64_t stride_a,
                             const int64_t* w_ptr_b, int64_t stride_b, const float* topk_weights,
                             int T, int top_k, int E, int H, int I, int rank, int num_loras,
                             float scale, int add_inputs, void* workspace, size_t ws_bytes,
                             uint32_t* err_word, lora_stream_t stream) {
  if (T < 0 || top_k < 0 || E < 1 || H < 0 || I < 0 || num_loras < 1 || stride_a < 0 ||
      stride_b < 0)
    return LORA_ERR_ARG;
  MoeCall c = {};
  c.out = y;
  c.ld_out = H;
  c.x = x;
  c.ld_x = I;
  c.k_in = I;
  c.x_div = 1;
  c.n_slices = 1;
  c.widths[0] = H;
  c.w_ptr_a = w_ptr_a;
  c.w_ptr_b = w_ptr_b;
  c.stride_a = stride_a;
  c.stride_b = stride_b;
  c.pair_weight = topk_weights;
  c.T = T;
  c.top_k = top_k;
  c.E = E;
  c.H = H;
  c.I = I;
  c.rank = rank;
  c.num_loras = num_loras;
  c.scale = scale;
  c.add_inputs = add_inputs ? 1 : 0;
  c.routed = 1;
  return moe_delta(c, workspace, ws_bytes, err_word, (cudaStream_t)stream);
}

int lora_get_error(uint32_t* err_word, uint32_t* host_out, int clear, lora_stream_t stream) {
  if (!err_word || !host_out) return LORA_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(host_out, err_word, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear) {
    clear_word_kernel<<<1, 1, 0, s>>>(err_word);
    e = cudaGetLastError();
  }
  return cuda_status(e);
}

}  // extern "C"
