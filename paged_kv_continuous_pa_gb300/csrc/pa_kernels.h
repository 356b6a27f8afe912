// pa_kernels.h -- launch parameters shared by the host API (pa_api.cu) and the
// kernels.  Internal: not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/pa.h"

namespace pa {

constexpr int kMaxChunks = 16;          // prefill chunks per pa_attention call
constexpr int kDefaultSplitTokens = 4096;
constexpr uint32_t kDefaultWaitLimit = 1000000;  // microseconds one bounded wait may take (one second)
constexpr uint32_t kDrainWaitLimit = 1000000;    // microseconds spent draining copies on an error path
#ifndef PA_WAIT_HINT_NS
#define PA_WAIT_HINT_NS 10000
#endif
constexpr uint32_t kWaitHintNs = PA_WAIT_HINT_NS;  // longest sleep inside one mbarrier poll (0: poll without a hint)
constexpr int kMaxStages = 16;          // decode pipeline depth upper bound
constexpr int kDecodeWarps = 4;         // warps of a decode CTA
constexpr int kStageTokens = 32;        // tokens per decode pipeline stage
constexpr int kMaxUnitPages = 256;      // page ids a decode unit caches (split_tokens <= 256 * 16)
constexpr int kMaxSplitTokens = 4096;
constexpr float kRescaleSlack = 8.0f;   // log2-domain headroom before the running max is moved

// Decode occupancy target and the stage-ring budget that goes with it: the
// ring is sized so that kDecodeMinCtas CTAs fit in an SM's shared memory, and
// registers are capped so that they fit in its register file.
#ifndef PA_DECODE_MIN_CTAS
#define PA_DECODE_MIN_CTAS 4
#endif
#ifndef PA_DECODE_RING_KB
#define PA_DECODE_RING_KB 48
#endif
constexpr int kDecodeMinCtas = PA_DECODE_MIN_CTAS;
constexpr int kDecodeRingBytes = PA_DECODE_RING_KB * 1024;   // at four CTAs per SM
constexpr int kDecodeRingBytes3 = 64 * 1024;                 // at three CTAs per SM

enum KvType { KV_F32 = 0, KV_BF16 = 1, KV_E4M3 = 2 };

// Device status codes (same values as pa_status in include/pa.h).
enum { ST_OK = 0, ST_OUT_OF_RANGE = 3, ST_TIMEOUT = 4, ST_LAUNCH = 5 };  // ST_LAUNCH: a kernel found its launch inconsistent

constexpr int kMaxHeadScales = 64;  // kv heads a pool with per-head fp8 scales may have

// The scale entry of kv head h: per head, or the per-tensor entry 0.
#define PA_HEAD(p, h) ((p).head_scales ? (h) : 0)

// The launch order of a call's decode rows (pa_set_unit_order): a single
// CTA writes the row indices longest first into `order`, either as a launch of
// its own or as one more CTA of the append launch that precedes the attention.
struct OrderParams {
  const int32_t* seq_ids;
  const int32_t* positions;
  int32_t n_rows, num_seqs;
  int32_t max_pos;        // max_blocks * P: positions at or past it are out of range
  int32_t split_tokens;   // a unit holds at most this many keys
  int32_t n_skip;         // rows of tile-path chunks: no decode units, listed last
  int32_t skip_begin[kMaxChunks];
  int32_t skip_end[kMaxChunks];
  int32_t* order;         // out: [n_rows] row indices
};

struct AppendParams {
  void* k_pool;
  void* v_pool;
  const void* k_new;
  const void* v_new;
  const int32_t* seq_ids;
  const int32_t* positions;
  const int32_t* block_tables;
  int32_t n_rows, num_seqs, max_blocks, num_pages;
  int32_t P, Hkv, D;
  int32_t in_dtype;  // KV_F32 or KV_BF16
  int32_t kv_dtype;  // KvType
  int32_t head_scales;  // 1: k_scale_h / v_scale_h hold one scale per kv head; 0: entry 0 holds the per-tensor scale
  float k_scale_h[kMaxHeadScales], v_scale_h[kMaxHeadScales];
  int32_t* status;
  // 0: rows 0 .. n_rows-1.  Otherwise only the rows of these ranges (the
  // chunks of a pa_step whose other rows append inside the attention units):
  // range k is rows range_begin[k] .. + range_rows[k] - 1, and range_first[k]
  // is the number of rows in the ranges before it.
  int32_t n_ranges;
  int32_t range_begin[kMaxChunks];
  int32_t range_first[kMaxChunks + 1];
  // 1: one more CTA, after the rows' CTAs, writes `order` (the attention that
  // follows as a programmatic dependent reads it)
  int32_t with_order;
  OrderParams order;
};

struct AttnParams {
  const void* k_pool;
  const void* v_pool;
  const void* q;
  void* out;
  const int32_t* seq_ids;
  const int32_t* positions;
  const int32_t* block_tables;
  int32_t n_rows, num_seqs, max_blocks, num_pages;
  int32_t P, Hq, Hkv, D;
  int32_t q_is_bf16;
  int32_t split_tokens;  // split-KV chunk length (multiple of P)
  int32_t max_splits;    // ceil(max_blocks * P / split_tokens)
  int32_t head_scales;   // 1: the two arrays below hold one entry per kv head; 0: entry 0 for every head
  float qk_scale_log2_h[kMaxHeadScales];  // softmax scale * log2(e) * k scale (scores live in the log2 domain)
  float v_scale_h[kMaxHeadScales];        // fp8 value scale, 1 otherwise
  float* ws_o;           // [n_rows][Hq][max_splits][D] partial accumulators (split rows only)
  float* ws_ml;          // [n_rows][Hq][max_splits][2] partial (max, sum)
  int32_t* ws_count;     // [n_rows][Hkv] finished-split counters, zero between calls
  int32_t* status;
  uint32_t wait_limit;   // microseconds
  int32_t debug_stall;   // 1: every CTA also waits on a barrier nothing completes (failure-path test)
  int32_t n_stages;      // decode pipeline depth (set per instantiation at launch)
  int32_t n_prefill_ctas;  // CTAs [0, n_prefill_ctas) run prefill tiles, the rest decode units
  int32_t n_chunks;                       // chunks on the tensor-core tile path
  int32_t chunk_begin[kMaxChunks];        // their rows [chunk_begin, chunk_end)
  int32_t chunk_end[kMaxChunks];
  int32_t chunk_cta_begin[kMaxChunks + 1];  // prefix sums of tile CTAs per chunk
  int32_t chunk_row_begin[kMaxChunks];    // prefix sums of chunk rows (tile partial slots)
  int32_t chunk_tile_begin[kMaxChunks];   // prefix sums of tiles (tile counters)
  int32_t tile_rows;                      // positions per 128-row tile: 128 / G
  int32_t tile_splits;                    // key-range splits per tile (CTAs per tile)
  float* ws_tile_o;                       // [chunk rows][Hq][tile_splits][D] partial accumulators
  float* ws_tile_ml;                      // [chunk rows][Hq][tile_splits][2] partial (max, sum)
  int32_t* ws_tile_count;                 // [tiles] finished-split counters, zero between calls
  float sm_scale_log2;                    // softmax scale * log2(e) for the tile path
  int32_t dependent;                      // host: launch as a programmatic dependent of the append
  int32_t row_group;                      // e4m3 tensor-core decode: rows per CTA (1, 2, 4 or 8)
  // Decode units in launch order: unit slot i runs row row_order[i], written
  // by the launch this one depends on (read after griddep_wait); null: row i
  const int32_t* row_order;
  // rows that get decode units: n_rows, or with a launch order the rows it
  // lists (every row but those of tile-path chunks)
  int32_t n_unit_rows;
  // pa_step: every row outside the caller's chunks appends its own new K/V
  // row inside the attention launch (the unit of its last split, per kv
  // head), with the encoder of the append kernel; chunk rows were appended
  // by the launch this one depends on.
  int32_t fuse_append;
  int32_t in_dtype;                       // KV_F32 or KV_BF16: dtype of k_new / v_new
  const void* k_new;                      // [n_rows][Hkv][D]
  const void* v_new;
  float k_enc_scale_h[kMaxHeadScales];    // fp8 key scale (stored code = e4m3(x / scale)), 1 otherwise
  int32_t n_all_chunks;                   // every chunk the caller listed (tile path or not)
  int32_t all_chunk_begin[kMaxChunks];
  int32_t all_chunk_end[kMaxChunks];
  CUtensorMap kmap;                       // bf16 K pool as [num_pages * Hkv * P][D], box 64 x P, 128B swizzle;
                                          // e4m3 pool (D = 128): bytes [num_pages * Hkv * P][128], box 128 x min(P, 32)
  CUtensorMap vmap;                       // V pool, same geometry
  CUtensorMap kmap_dec;                   // D = 128 pools for the tensor-core decode units: bf16 boxes of
  CUtensorMap vmap_dec;                   //   64 x min(P, 32), e4m3 boxes of 128 bytes x min(P, 32); 128B swizzle
};

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);

// One CTA that writes o.order (the rows longest first); the attention launched
// after it as a programmatic dependent may start its setup at once.
cudaError_t launch_order_rows(const OrderParams& o, cudaStream_t stream);

// Let `kernel` use `bytes` of dynamic shared memory on the current device.
// The attribute is per device, so it is set once for each device this process
// launches on (`done`: one bit per device, kept by the caller per kernel).
// Every thread sets the same value, so concurrent first calls are harmless.
template <typename Kernel>
cudaError_t allow_dynamic_smem(Kernel kernel, std::atomic<unsigned long long>& done, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// CTAs of `kernel` (`threads` threads, `bytes` of dynamic shared memory)
// resident on the current device at once, computed once per device (`cache`:
// value + 1 per device, 0 until known).  0 if it cannot be queried.
template <typename Kernel>
long long resident_ctas(Kernel kernel, std::atomic<long long> (&cache)[64], std::atomic<unsigned long long>& smem_done,
                        int threads, size_t bytes) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64) {
    const long long c = cache[dev].load(std::memory_order_acquire);
    if (c > 0) return c - 1;
  }
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      allow_dynamic_smem(kernel, smem_done, bytes) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, bytes) != cudaSuccess)
    return 0;
  const long long cap = static_cast<long long>(sms) * per_sm;
  if (dev < 64) cache[dev].store(cap + 1, std::memory_order_release);
  return cap;
}


// Launch `kernel` normally, or (dependent) as a programmatic dependent of the
// previous kernel in the stream: it may start while that kernel runs and must
// call griddep_wait() before reading anything that kernel writes.
template <typename Kernel, typename... Args>
inline cudaError_t launch_kernel(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool dependent,
                                 Args... args) {
  if (!dependent) {
    kernel<<<grid, block, smem, stream>>>(args...);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Process-wide count of kernel launches made by the library (pa_kernel_launches).
void count_launch();

// A scratch array of `bytes` bytes that the library owns (pa_attention_noalloc):
// address() returns its device address on the current device, or nullptr
// after setting the last-error text.
struct FixedScratch {
  size_t bytes;
  void* (*address)();
};

// pa_attention with `scratch` as its workspace: the arguments are checked as
// pa_attention checks them, the plan is made once (one read of the split
// length), a plan larger than the scratch is refused with PA_ERR_UNSUPPORTED,
// and the plan's split counters are cleared on `stream` before the launch.
pa_status attention_fixed_scratch(const pa_pool* pool, int32_t n_rows, const void* q, pa_dtype q_dtype,
                                  int32_t num_q_heads, const int32_t* seq_ids, const int32_t* positions,
                                  const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                                  const pa_chunk* chunks, int32_t n_chunks, float softmax_scale, void* out,
                                  int32_t* status_dev, void* stream, const FixedScratch& scratch);

// Set the calling thread's pa_last_error() text.
void set_last_error(const char* fmt, ...);

// Decode-unit kernels, one translation unit per K/V dtype.  Return
// cudaErrorNotSupported for a (G, D) pair without an instantiation.
cudaError_t launch_decode_f32(const AttnParams& p, cudaStream_t stream);
cudaError_t launch_decode_bf16(const AttnParams& p, cudaStream_t stream);
cudaError_t launch_decode_e4m3(const AttnParams& p, cudaStream_t stream);

// Tensor-core decode units for e4m3 pools, head_dim 128, bf16 queries,
// 1..8 query heads per kv head; p.kmap / p.vmap must be the pools' byte views
// [num_pages * Hkv * P][128], box 128 x min(P, 32), 128-byte swizzle.
bool decode_e4m3_mma_eligible(int D, int G, bool q_bf16);
cudaError_t launch_decode_e4m3_mma(const AttnParams& p, cudaStream_t stream);

// Tensor-core decode units for bf16 pools, head_dim 128, bf16 queries, 3..8
// query heads per kv head (p.kmap_dec / p.vmap_dec: bf16 boxes of 64 x
// min(P, 32) rows).  The mixed launch runs the same units for its decode rows.
bool decode_bf16_mma_eligible(int D, int G, bool q_bf16);
cudaError_t launch_decode_bf16_mma(const AttnParams& p, cudaStream_t stream);

// One launch whose first p.n_prefill_ctas CTAs run tensor-core prefill tiles
// (bf16 q and K/V) and whose remaining CTAs run decode units.
cudaError_t launch_mixed_bf16(const AttnParams& p, cudaStream_t stream);

// A launch of tensor-core prefill tiles only (every row of the call is in a
// chunk on the tile path): p.n_prefill_ctas warp-specialised tile CTAs with
// the same per-row arithmetic as the tiles of launch_mixed_bf16.
cudaError_t launch_prefill_bf16(const AttnParams& p, cudaStream_t stream);

constexpr int kMinTileRows = 16;     // shorter chunks run on the decode path
constexpr int kTileRowsTotal = 128;  // (position, head) rows of one tensor-core tile
#ifndef PA_TILE_SPLIT_KEYS
#define PA_TILE_SPLIT_KEYS 4096
#endif
constexpr int kTileSplitKeys = PA_TILE_SPLIT_KEYS;  // keys per CTA of a tile (a multiple of 64); longer tiles split


}  // namespace pa
