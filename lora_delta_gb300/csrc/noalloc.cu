// lora_delta_fused_noalloc: the routed delta for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) on the path
// that applies the delta: code that runs inside a memory budget fixed at start
// up, custom allocators that forbid allocations after warm-up, or runtimes that
// hand this library only the tensors they already own.  lora_delta_fused needs
// a scratch workspace for large batches (the row clustering by slot), which
// such a caller cannot provide.  This entry point takes that scratch from a
// fixed array that lives in the library itself.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes bytes.
// This file is its own CUDA module, and the runtime loads modules lazily by
// default (CUDA_MODULE_LOADING=LAZY): the driver reserves the array on a
// device when the first call on that device looks its address up with
// cudaGetSymbolAddress (with that device current), not when the library is
// loaded.  From then on the device holds it until the process exits.  So a
// caller makes one warm-up call on every device it uses before its memory
// budget is fixed and before any stream capture; after that no call reserves
// anything.  The address is cached per device; it is stale after a
// cudaDeviceReset of that device.  Every call shares the one array,
// so calls that overlap on the GPU (for example on two streams) race on it;
// serialize them.  The array keeps whatever the last call left in it; the
// kernels that use it overwrite every entry they read (the clustering writes
// the whole row permutation and every cluster start), so nothing in it has to
// start at zero.
#include <mutex>

#include "lora_delta.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return LORA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      // (e.g. out of memory while the module loads): clear the runtime's last
      // error, so that a later, unrelated launch check does not report it
      cudaGetLastError();
      return LORA_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return LORA_OK;
}

}  // namespace

extern "C" {

size_t lora_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int lora_delta_fused_noalloc(void* out, int64_t ld_out, const void* x, int n, int k_in,
                             const int32_t* seq_slot, const uint64_t* a_table,
                             const uint64_t* b_table, const float* scale_table,
                             const int32_t* widths, int S, int R, int max_loras,
                             int offset_start, int add_inputs, uint32_t* err_word,
                             lora_stream_t stream) {
  if (n < 0 || max_loras < 1 || S < 1 || R < 1) return LORA_ERR_ARG;
  const size_t need = lora_workspace_min_size(n, S, R, max_loras);
  if (need > kNoAllocScratchBytes) return LORA_ERR_TOO_LARGE;
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != LORA_OK) return rc;
  return lora_delta_fused(out, ld_out, x, n, k_in, seq_slot, a_table, b_table, scale_table,
                          widths, S, R, max_loras, offset_start, add_inputs, scratch,
                          kNoAllocScratchBytes, err_word, stream);
}

}  // extern "C"
