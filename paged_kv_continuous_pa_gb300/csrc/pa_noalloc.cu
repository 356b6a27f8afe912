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
// contents; each call clears the part it uses on its stream before the
// attention launch.  Calls that overlap on the GPU (different streams, no
// ordering between them) race on it.
#include <cuda_runtime.h>

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

std::mutex g_mu;
void* g_scratch_dev[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (the first call on a device does it, with that device current).
// Returns nullptr (and sets the last-error text) on failure.
void* scratch_on_current_device() {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    pa::set_last_error("pa_attention_noalloc: no current CUDA device (%s)", cudaGetErrorString(e));
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_dev[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      pa::set_last_error("pa_attention_noalloc: cudaGetSymbolAddress failed on device %d (%s)", dev,
                         cudaGetErrorString(e));
      return nullptr;
    }
    g_scratch_dev[dev] = ptr;
  }
  return g_scratch_dev[dev];
}

}  // namespace

extern "C" pa_status pa_attention_noalloc(const pa_pool* pool, int32_t n_rows, const void* q, pa_dtype q_dtype,
                                          int32_t num_q_heads, const int32_t* seq_ids, const int32_t* positions,
                                          const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                                          const pa_chunk* chunks, int32_t n_chunks, float softmax_scale, void* out,
                                          int32_t* status_dev, void* stream) {
  const size_t need = pa_attention_workspace_bytes(pool, n_rows, num_q_heads, max_blocks_per_seq, chunks, n_chunks);
  if (need > kNoallocScratchBytes) {
    pa::set_last_error(
        "pa_attention_noalloc: this call needs %zu bytes of split-KV scratch but the static scratch holds %zu; "
        "use pa_attention with a caller workspace, fewer rows or a shorter block table",
        need, kNoallocScratchBytes);
    return PA_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  if (need > 0) {
    scratch = scratch_on_current_device();
    if (scratch == nullptr) return PA_ERR_CUDA;
    cudaError_t e = cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
      pa::set_last_error("pa_attention_noalloc: clearing the scratch failed (%s)", cudaGetErrorString(e));
      return PA_ERR_CUDA;
    }
  }
  return pa_attention(pool, n_rows, q, q_dtype, num_q_heads, seq_ids, positions, block_tables, num_seqs,
                      max_blocks_per_seq, chunks, n_chunks, softmax_scale, out, scratch, need, status_dev, stream);
}
