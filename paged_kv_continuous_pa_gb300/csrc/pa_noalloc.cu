// pa_noalloc.cu -- pa_attention_noalloc: paged attention for callers that
// cannot allocate device memory.
//
// Some callers only ever receive input and output buffers: a plugin invoked
// by a host inference runtime that owns and budgets all device memory, or a
// serving loop that forbids cudaMalloc after start-up because an allocation
// on the hot path can synchronise the device or fail under memory pressure in
// the middle of a request.  Such callers cannot provide pa_attention's split-KV
// workspace.  This entry point uses a fixed scratch array that lives in this
// library's device image instead: every GPU that loads the library holds
// kNoallocScratchBytes of it until the process exits.
//
// The array is shared by every call on a device and keeps the last call's
// contents; each call clears the split counters of its plan on its stream
// before the attention launch (every partial is written before it is read).
// Calls that overlap on the GPU (different streams, no ordering between them)
// race on it.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/pa.h"
#include "pa_kernels.h"

namespace {

constexpr size_t kNoallocScratchBytes = 32u << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

// Split-KV partials and counters for pa_attention_noalloc.  In host code this
// name is only a stand-in for the symbol; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// The address found for a device, and the context it was found in: a device
// reset (or a primary context released and created again) gives the device a
// new context, where the array has a new address, so the lookup is repeated.
struct CachedAddress {
  CUcontext ctx;
  void* ptr;
};

std::mutex g_mu;
CachedAddress g_scratch_dev[kMaxDevices] = {};

// cuCtxGetCurrent from the driver, looked up once through the runtime.
PFN_cuCtxGetCurrent_v4000 ctx_getter() {
  static std::once_flag once;
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
  });
  return fn;
}

// Device address of the scratch array on the current device, looked up with
// that device current the first time a call needs it there (and again after
// the device's context changed).  Returns nullptr (and sets the last-error
// text) on failure.
void* scratch_on_current_device() {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    pa::set_last_error("pa_attention_noalloc: no current CUDA device (%s)", cudaGetErrorString(e));
    return nullptr;
  }
  PFN_cuCtxGetCurrent_v4000 get = ctx_getter();
  if (get == nullptr) {
    pa::set_last_error("pa_attention_noalloc: cuCtxGetCurrent is not available from the driver");
    return nullptr;
  }
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  CachedAddress& c = g_scratch_dev[dev];
  if (ctx == nullptr || c.ptr == nullptr || c.ctx != ctx) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);  // makes the device's context current if none was
    if (e != cudaSuccess || ptr == nullptr) {
      pa::set_last_error("pa_attention_noalloc: cudaGetSymbolAddress failed on device %d (%s)", dev,
                         cudaGetErrorString(e));
      return nullptr;
    }
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
      pa::set_last_error("pa_attention_noalloc: cannot read the current CUDA context on device %d", dev);
      return nullptr;
    }
    c.ctx = ctx;
    c.ptr = ptr;
  }
  return c.ptr;
}

}  // namespace

extern "C" pa_status pa_attention_noalloc(const pa_pool* pool, int32_t n_rows, const void* q, pa_dtype q_dtype,
                                          int32_t num_q_heads, const int32_t* seq_ids, const int32_t* positions,
                                          const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                                          const pa_chunk* chunks, int32_t n_chunks, float softmax_scale, void* out,
                                          int32_t* status_dev, void* stream) {
  const pa::FixedScratch scratch{kNoallocScratchBytes, &scratch_on_current_device};
  return pa::attention_fixed_scratch(pool, n_rows, q, q_dtype, num_q_heads, seq_ids, positions, block_tables,
                                     num_seqs, max_blocks_per_seq, chunks, n_chunks, softmax_scale, out, status_dev,
                                     stream, scratch);
}
