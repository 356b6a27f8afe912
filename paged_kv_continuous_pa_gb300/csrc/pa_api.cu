// pa_api.cu -- the C ABI declared in include/pa.h: argument validation, launch
// geometry and dispatch.  No allocation, no device synchronisation.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>

#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/pa.h"
#include "pa_kernels.h"

struct pa_pool {
  pa_pool_desc desc;
  bool head_scales;  // fp8 scales per kv head (pa_pool_set_head_scales)
  float k_scale_h[pa::kMaxHeadScales], v_scale_h[pa::kMaxHeadScales];
  void* k;
  void* v;
  bool tile_maps_ready;  // kmap / vmap encoded (on first use by the prefill tile path)
  bool dec_maps_ready;   // kmap_dec / vmap_dec encoded (on first use by tensor-core decode units)
  CUtensorMap kmap;      // 2-D views of the pools for tensor-map copies
  CUtensorMap vmap;
  CUtensorMap kmap_dec;
  CUtensorMap vmap_dec;
};

namespace {
std::atomic<unsigned long long> g_launches{0};
}  // namespace

void pa::count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {

thread_local char g_last_error[512] = "";
// process-wide settings; any thread may change them, and a call reads each once
std::atomic<int32_t> g_split_tokens{pa::kDefaultSplitTokens};
std::atomic<int32_t> g_row_groups{1};
std::atomic<int32_t> g_unit_order{PA_ORDER_AUTO};
std::atomic<uint32_t> g_wait_limit{pa::kDefaultWaitLimit};
std::atomic<int32_t> g_debug_stall{0};

pa_status fail(pa_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

pa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t elt_bytes(pa_dtype t) { return t == PA_F32 ? 4 : t == PA_BF16 ? 2 : 1; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int max_splits_for(const pa_pool_desc& d, int32_t max_blocks, int32_t split_tokens) {
  const long long cap = static_cast<long long>(max_blocks) * d.page_size;
  return static_cast<int>((cap + split_tokens - 1) / split_tokens);
}

// How one pa_attention call is laid out: which chunks take the tensor-core
// tile path, how many CTAs that takes, and where the split-KV partials live in
// the caller's workspace.  Decided from host-known sizes only.
struct Plan {
  int G = 1, R = 0;
  int max_splits = 1;     // decode splits per row
  int tile_splits = 0;    // key-range splits per tile (0: no tile path)
  int n_tile = 0;         // chunks on the tile path
  int src[pa::kMaxChunks];
  int cta_begin[pa::kMaxChunks + 1];
  int row_begin[pa::kMaxChunks];
  int tile_begin[pa::kMaxChunks];
  int total_tiles = 0, total_rows = 0;
  bool order_rows = false;  // decode units launch longest row first (the order goes to the workspace)
  // workspace byte offsets
  size_t d_count = 0, d_ml = 0, d_o = 0, t_count = 0, t_ml = 0, t_o = 0, order = 0, total = 0;
};

// Whether a call's decode rows launch longest first (pa_set_unit_order).
// Automatic: when the rows are many and a unit may be long (at least 1024
// keys), so that a long unit started late could outlast the rest of the
// launch by more than the order costs (one small launch, or one more CTA of
// the step's append launch); a call of short rows keeps its order.
bool want_order(int32_t mode, const pa_pool_desc& d, int32_t n_decode_rows, int32_t max_blocks, int32_t split_tokens) {
  if (mode == PA_ORDER_CALL || n_decode_rows < 2) return false;
  if (mode == PA_ORDER_LONGEST_FIRST) return true;
  const long long longest_unit = std::min<long long>(static_cast<long long>(max_blocks) * d.page_size, split_tokens);
  return n_decode_rows >= 128 && longest_unit >= 1024;
}

Plan make_plan(const pa_pool_desc& d, int32_t n_rows, int32_t hq, int32_t max_blocks, const pa_chunk* chunks,
               int32_t n_chunks, bool tile_dtypes, int32_t split_tokens, int32_t order_mode) {
  Plan pl;
  pl.G = hq / d.num_kv_heads;
  pl.max_splits = max_splits_for(d, max_blocks, split_tokens);
  pl.R = pa::kTileRowsTotal / pl.G;
  if (tile_dtypes && chunks != nullptr) {
    const long long keys = static_cast<long long>(max_blocks) * d.page_size;
    pl.tile_splits = static_cast<int>((keys + pa::kTileSplitKeys - 1) / pa::kTileSplitKeys);
    int ctas = 0;
    for (int c = 0; c < n_chunks && c < pa::kMaxChunks; ++c) {
      if (chunks[c].n_rows < pa::kMinTileRows) continue;
      const int k = pl.n_tile++;
      const int n_mt = (chunks[c].n_rows + pl.R - 1) / pl.R;
      pl.src[k] = c;
      pl.cta_begin[k] = ctas;
      pl.row_begin[k] = pl.total_rows;
      pl.tile_begin[k] = pl.total_tiles;
      ctas += d.num_kv_heads * n_mt * pl.tile_splits;
      pl.total_rows += chunks[c].n_rows;
      pl.total_tiles += d.num_kv_heads * n_mt;
    }
    pl.cta_begin[pl.n_tile] = ctas;
    if (pl.n_tile == 0) pl.tile_splits = 0;
  }
  auto pad = [](size_t x) { return (x + 255) / 256 * 256; };
  size_t off = 0;
  if (pl.max_splits > 1 && n_rows > 0) {
    const size_t slots = static_cast<size_t>(n_rows) * hq * pl.max_splits;
    pl.d_count = off;
    off += pad(static_cast<size_t>(n_rows) * d.num_kv_heads * sizeof(int32_t));
    pl.d_ml = off;
    off += pad(slots * 2 * sizeof(float));
    pl.d_o = off;
    off += pad(slots * d.head_dim * sizeof(float));
  }
  if (pl.tile_splits > 1) {
    // tile-major partials: per (tile, key range) all 128 tile rows
    const size_t slots = static_cast<size_t>(pl.total_tiles) * pl.tile_splits * pa::kTileRowsTotal;
    pl.t_count = off;
    off += pad(static_cast<size_t>(pl.total_tiles) * sizeof(int32_t));
    pl.t_ml = off;
    off += pad(slots * 2 * sizeof(float));
    pl.t_o = off;
    off += pad(slots * d.head_dim * sizeof(float));
  }
  // the order's room is kept whenever the rows could want it (chunk rows that
  // end up on the decode path count as decode rows), so that the workspace
  // size for a bf16 pool covers either query dtype
  if (want_order(order_mode, d, n_rows, max_blocks, split_tokens)) {
    pl.order_rows = want_order(order_mode, d, n_rows - pl.total_rows, max_blocks, split_tokens);
    pl.order = off;
    off += pad(static_cast<size_t>(n_rows) * sizeof(int32_t));
  }
  pl.total = off;
  return pl;
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// The pool as a 2-D tensor [num_pages * Hkv * P rows][D] with 128-byte
// swizzle, the layout the tensor-core paths read, boxes of `cols` elements x
// `rows` rows (one page of one kv head, or a part of it).
pa_status encode_map_pair(pa_pool* pool, CUtensorMap* km, CUtensorMap* vm, uint32_t cols, uint32_t rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const pa_pool_desc& d = pool->desc;
  const bool fp8 = d.kv_dtype == PA_FP8_E4M3;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d.head_dim),
                        static_cast<cuuint64_t>(d.num_pages) * d.num_kv_heads * d.page_size};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(d.head_dim) * elt_bytes(d.kv_dtype)};
  cuuint32_t box[2] = {cols, rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType ty = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  for (int i = 0; i < 2; ++i) {
    CUresult r = enc(i == 0 ? km : vm, ty, 2, i == 0 ? pool->k : pool->v, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  }
  return PA_OK;
}

// bf16 pools, prefill tiles: 64 elements x min(P, 64) rows (half or all of the head dim).
pa_status encode_tile_maps(pa_pool* pool) {
  if (pool->tile_maps_ready) return PA_OK;
  if (pool->desc.kv_dtype != PA_BF16) return fail(PA_ERR_UNSUPPORTED, "the tile path reads bf16 pools");
  const int P = pool->desc.page_size;
  const pa_status st = encode_map_pair(pool, &pool->kmap, &pool->vmap, 64u, static_cast<uint32_t>(P > 64 ? 64 : P));
  if (st == PA_OK) pool->tile_maps_ready = true;
  return st;
}

// D = 128 pools, tensor-core decode units: bf16 boxes of 64 elements x min(P, 32)
// rows (one head-dim half), e4m3 boxes of 128 bytes x min(P, 32) rows.
pa_status encode_decode_maps(pa_pool* pool) {
  if (pool->dec_maps_ready) return PA_OK;
  const pa_pool_desc& d = pool->desc;
  if (d.head_dim != 128 || (d.kv_dtype != PA_BF16 && d.kv_dtype != PA_FP8_E4M3))
    return fail(PA_ERR_UNSUPPORTED, "no tensor-core decode view for this pool's dtype / head_dim");
  const int P = d.page_size;
  const pa_status st = encode_map_pair(pool, &pool->kmap_dec, &pool->vmap_dec, d.kv_dtype == PA_BF16 ? 64u : 128u,
                                       static_cast<uint32_t>(P > 32 ? 32 : P));
  if (st == PA_OK) pool->dec_maps_ready = true;
  return st;
}

pa_status check_desc(const pa_pool_desc* d) {
  if (d == nullptr) return fail(PA_ERR_INVALID_ARG, "pool descriptor is NULL");
  if (d->num_pages <= 0 || d->num_kv_heads <= 0 || d->page_size <= 0 || d->head_dim <= 0)
    return fail(PA_ERR_INVALID_ARG, "pool sizes must be positive (pages %d, kv heads %d, page %d, head_dim %d)",
                d->num_pages, d->num_kv_heads, d->page_size, d->head_dim);
  if (d->kv_dtype != PA_F32 && d->kv_dtype != PA_BF16 && d->kv_dtype != PA_FP8_E4M3)
    return fail(PA_ERR_INVALID_ARG, "unknown kv dtype %d", static_cast<int>(d->kv_dtype));
  if (d->page_size < 16 || d->page_size > 256 || (d->page_size & (d->page_size - 1)) != 0)
    return fail(PA_ERR_UNSUPPORTED, "page_size %d not in {16, 32, 64, 128, 256}", d->page_size);
  if (d->head_dim != 64 && d->head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "head_dim %d not in {64, 128}", d->head_dim);
  if (d->kv_dtype == PA_FP8_E4M3 &&
      !(std::isfinite(d->k_scale) && d->k_scale > 0.f && std::isfinite(d->v_scale) && d->v_scale > 0.f))
    return fail(PA_ERR_INVALID_ARG, "fp8 scales must be finite and positive (k %g, v %g)", d->k_scale, d->v_scale);
  return PA_OK;
}

}  // namespace

void pa::set_last_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
}

namespace {

// pa_append_kv's argument checks and launch parameters; *empty when there is nothing to do.
pa_status build_append(const pa_pool* pool, int32_t n_rows, const void* k_new, const void* v_new, pa_dtype in_dtype,
                       const int32_t* seq_ids, const int32_t* positions, const int32_t* block_tables,
                       int32_t num_seqs, int32_t max_blocks_per_seq, int32_t* status_dev, pa::AppendParams* out,
                       bool* empty) {
  *empty = true;
  if (pool == nullptr) return fail(PA_ERR_INVALID_ARG, "pool is NULL");
  if (n_rows < 0) return fail(PA_ERR_INVALID_ARG, "n_rows %d < 0", n_rows);
  if (n_rows == 0) return PA_OK;
  *empty = false;
  if (in_dtype != PA_F32 && in_dtype != PA_BF16)
    return fail(PA_ERR_INVALID_ARG, "append input dtype must be f32 or bf16");
  if (!k_new || !v_new || !seq_ids || !positions || !block_tables)
    return fail(PA_ERR_INVALID_ARG, "append: a device pointer is NULL");
  if (!aligned(k_new, 16) || !aligned(v_new, 16)) return fail(PA_ERR_INVALID_ARG, "k_new / v_new must be 16-byte aligned");
  if (num_seqs <= 0 || max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG, "num_seqs and max_blocks_per_seq must be positive");
  pa::AppendParams p{};
  p.k_pool = pool->k;
  p.v_pool = pool->v;
  p.k_new = k_new;
  p.v_new = v_new;
  p.seq_ids = seq_ids;
  p.positions = positions;
  p.block_tables = block_tables;
  p.n_rows = n_rows;
  p.num_seqs = num_seqs;
  p.max_blocks = max_blocks_per_seq;
  p.num_pages = pool->desc.num_pages;
  p.P = pool->desc.page_size;
  p.Hkv = pool->desc.num_kv_heads;
  p.D = pool->desc.head_dim;
  p.in_dtype = in_dtype == PA_F32 ? pa::KV_F32 : pa::KV_BF16;
  p.kv_dtype = static_cast<int32_t>(pool->desc.kv_dtype);
  p.head_scales = pool->head_scales ? 1 : 0;
  for (int h = 0; h < (pool->head_scales ? pool->desc.num_kv_heads : 1); ++h) {
    p.k_scale_h[h] = pool->head_scales ? pool->k_scale_h[h] : pool->desc.k_scale;
    p.v_scale_h[h] = pool->head_scales ? pool->v_scale_h[h] : pool->desc.v_scale;
  }
  p.status = status_dev;
  *out = p;
  return PA_OK;
}

// pa_attention; with `pre` (pa_step), the append `pre` describes is launched
// once every attention argument has passed its checks, and the attention
// kernel follows it as a programmatic dependent: its CTAs start their
// query, sequence and page-id lookups while the append runs, and wait for it
// before the first pool read.  With `scratch` (pa_attention_noalloc) the
// workspace is the library's fixed scratch array instead of the caller's:
// the plan must fit in it, and the call clears the plan's split counters on
// the stream before its launch.
pa_status attention_impl(const pa_pool* pool, int32_t n_rows, const void* q, pa_dtype q_dtype, int32_t num_q_heads,
                         const int32_t* seq_ids, const int32_t* positions, const int32_t* block_tables,
                         int32_t num_seqs, int32_t max_blocks_per_seq, const pa_chunk* chunks, int32_t n_chunks,
                         float softmax_scale, void* out, void* workspace, size_t workspace_bytes,
                         int32_t* status_dev, void* stream, const pa::AppendParams* pre,
                         const pa::FixedScratch* scratch = nullptr) {
  if (pool == nullptr) return fail(PA_ERR_INVALID_ARG, "pool is NULL");
  const pa_pool_desc& d = pool->desc;
  if (n_rows < 0) return fail(PA_ERR_INVALID_ARG, "n_rows %d < 0", n_rows);
  if (q_dtype != PA_F32 && q_dtype != PA_BF16) return fail(PA_ERR_INVALID_ARG, "q dtype must be f32 or bf16");
  if (num_q_heads <= 0 || num_q_heads % d.num_kv_heads != 0)
    return fail(PA_ERR_INVALID_ARG, "num_q_heads %d is not a positive multiple of num_kv_heads %d", num_q_heads,
                d.num_kv_heads);
  const int G = num_q_heads / d.num_kv_heads;
  if (G > 8) return fail(PA_ERR_UNSUPPORTED, "query heads per kv head %d > 8", G);
  if (num_seqs <= 0 || max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG, "num_seqs and max_blocks_per_seq must be positive");
  if (n_chunks < 0 || n_chunks > pa::kMaxChunks)
    return fail(PA_ERR_INVALID_ARG, "n_chunks %d outside [0, %d]", n_chunks, pa::kMaxChunks);
  if (n_chunks > 0 && chunks == nullptr) return fail(PA_ERR_INVALID_ARG, "chunks is NULL");
  for (int c = 0; c < n_chunks; ++c) {
    if (chunks[c].n_rows <= 0 || chunks[c].row_begin < 0 ||
        static_cast<long long>(chunks[c].row_begin) + chunks[c].n_rows > n_rows)
      return fail(PA_ERR_INVALID_ARG, "chunk %d rows [%d, +%d) outside [0, %d)", c, chunks[c].row_begin,
                  chunks[c].n_rows, n_rows);
    for (int c2 = 0; c2 < c; ++c2)
      if (chunks[c].row_begin < chunks[c2].row_begin + chunks[c2].n_rows &&
          chunks[c2].row_begin < chunks[c].row_begin + chunks[c].n_rows)
        return fail(PA_ERR_INVALID_ARG, "chunks %d and %d overlap", c2, c);
  }
  if (n_rows == 0) {
    if (pre == nullptr) return PA_OK;
    const cudaError_t e = pa::launch_append(*pre, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "append launch");
  }
  if (!q || !seq_ids || !positions || !block_tables || !out)
    return fail(PA_ERR_INVALID_ARG, "attention: a device pointer is NULL");
  if (!aligned(q, 16) || !aligned(out, 16)) return fail(PA_ERR_INVALID_ARG, "q / out must be 16-byte aligned");
  const int32_t split_tokens = g_split_tokens.load(std::memory_order_relaxed);  // one value for the plan and the kernels
  const Plan pl = make_plan(d, n_rows, num_q_heads, max_blocks_per_seq, chunks, n_chunks,
                            q_dtype == PA_BF16 && d.kv_dtype == PA_BF16, split_tokens,
                            g_unit_order.load(std::memory_order_relaxed));
  if (scratch != nullptr && pl.total > 0) {
    if (pl.total > scratch->bytes)
      return fail(PA_ERR_UNSUPPORTED,
                  "pa_attention_noalloc: this call needs %zu bytes of split-KV scratch but the static scratch holds "
                  "%zu; use pa_attention with a caller workspace, fewer rows or a shorter block table",
                  pl.total, scratch->bytes);
    workspace = scratch->address();
    if (workspace == nullptr) return PA_ERR_CUDA;  // the lookup set the message
    workspace_bytes = scratch->bytes;
  }
  if (pl.total > 0) {
    if (workspace == nullptr || workspace_bytes < pl.total)
      return fail(PA_ERR_INVALID_ARG, "workspace of %zu bytes needed, %zu given", pl.total,
                  workspace == nullptr ? static_cast<size_t>(0) : workspace_bytes);
    if (!aligned(workspace, 256)) return fail(PA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  }
  const double sm = softmax_scale > 0.f ? static_cast<double>(softmax_scale) : 1.0 / std::sqrt(static_cast<double>(d.head_dim));

  pa::AttnParams p{};
  p.k_pool = pool->k;
  p.v_pool = pool->v;
  p.q = q;
  p.out = out;
  p.seq_ids = seq_ids;
  p.positions = positions;
  p.block_tables = block_tables;
  p.n_rows = n_rows;
  p.num_seqs = num_seqs;
  p.max_blocks = max_blocks_per_seq;
  p.num_pages = d.num_pages;
  p.P = d.page_size;
  p.Hq = num_q_heads;
  p.Hkv = d.num_kv_heads;
  p.D = d.head_dim;
  p.q_is_bf16 = q_dtype == PA_BF16;
  p.split_tokens = split_tokens;
  p.max_splits = pl.max_splits;
  p.n_unit_rows = n_rows;
  p.row_group = g_row_groups.load(std::memory_order_relaxed);
  // per kv head (or entry 0 for all): softmax scale * k scale * log2(e), and the v scale
  p.head_scales = pool->head_scales ? 1 : 0;
  for (int h = 0; h < (pool->head_scales ? d.num_kv_heads : 1); ++h) {
    const bool fp8 = d.kv_dtype == PA_FP8_E4M3;
    const double ks = fp8 ? static_cast<double>(pool->head_scales ? pool->k_scale_h[h] : d.k_scale) : 1.0;
    p.qk_scale_log2_h[h] = static_cast<float>(sm * ks * 1.4426950408889634073599246810018921);  // log2(e)
    p.v_scale_h[h] = fp8 ? (pool->head_scales ? pool->v_scale_h[h] : d.v_scale) : 1.0f;
  }
  if (pl.total > 0) {
    unsigned char* base = static_cast<unsigned char*>(workspace);
    if (pl.max_splits > 1) {
      p.ws_count = reinterpret_cast<int32_t*>(base + pl.d_count);
      p.ws_ml = reinterpret_cast<float*>(base + pl.d_ml);
      p.ws_o = reinterpret_cast<float*>(base + pl.d_o);
    }
    if (pl.tile_splits > 1) {
      p.ws_tile_count = reinterpret_cast<int32_t*>(base + pl.t_count);
      p.ws_tile_ml = reinterpret_cast<float*>(base + pl.t_ml);
      p.ws_tile_o = reinterpret_cast<float*>(base + pl.t_o);
    }
  }
  p.status = status_dev;
  p.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  p.debug_stall = g_debug_stall.load(std::memory_order_relaxed);
  p.n_prefill_ctas = 0;
  p.n_chunks = 0;
  p.sm_scale_log2 = static_cast<float>(sm * 1.4426950408889634073599246810018921);

  // Chunks long enough for the tensor-core tile path (bf16 q and K/V): their
  // rows run there; rows of other chunks run as decode rows.
  if (pl.n_tile > 0) {
    pa_status st = encode_tile_maps(const_cast<pa_pool*>(pool));
    if (st != PA_OK) return st;
    p.kmap = pool->kmap;
    p.vmap = pool->vmap;
    p.tile_rows = pl.R;
    p.tile_splits = pl.tile_splits;
    p.n_chunks = pl.n_tile;
    for (int k = 0; k < pl.n_tile; ++k) {
      p.chunk_begin[k] = chunks[pl.src[k]].row_begin;
      p.chunk_end[k] = chunks[pl.src[k]].row_begin + chunks[pl.src[k]].n_rows;
      p.chunk_cta_begin[k] = pl.cta_begin[k];
      p.chunk_row_begin[k] = pl.row_begin[k];
      p.chunk_tile_begin[k] = pl.tile_begin[k];
    }
    p.chunk_cta_begin[pl.n_tile] = pl.cta_begin[pl.n_tile];
    p.n_prefill_ctas = pl.cta_begin[pl.n_tile];
  }

  // Tensor-core decode units (chosen by pool dtype, head_dim, G and the query
  // dtype alone, so a row's bits never depend on the rest of the batch): e4m3
  // pools with D = 128, bf16 pools with D = 128 and G >= 3 (also inside the
  // mixed launch).  They read stages through the pool's decode tensor maps.
  const bool q16 = q_dtype == PA_BF16;
  const bool mma_e4m3 = d.kv_dtype == PA_FP8_E4M3 && pa::decode_e4m3_mma_eligible(d.head_dim, G, q16);
  const bool mma_bf16 = d.kv_dtype == PA_BF16 && pa::decode_bf16_mma_eligible(d.head_dim, G, q16);
  if (mma_e4m3 || mma_bf16) {
    pa_status st = encode_decode_maps(const_cast<pa_pool*>(pool));
    if (st != PA_OK) return st;
    p.kmap_dec = pool->kmap_dec;
    p.vmap_dec = pool->vmap_dec;
  }

  // Decode rows longest first: the order goes to the workspace, written by one
  // CTA of its own launch, or of the step's append launch when there is one;
  // the attention follows as its programmatic dependent.  Row groups keep the
  // caller's order (a group is consecutive rows of the call).
  const bool use_order = pl.order_rows && !(mma_e4m3 && p.row_group > 1);
  pa::OrderParams ord{};
  if (use_order) {
    ord.seq_ids = seq_ids;
    ord.positions = positions;
    ord.n_rows = n_rows;
    ord.num_seqs = num_seqs;
    ord.max_pos = static_cast<int32_t>(std::min<long long>(static_cast<long long>(max_blocks_per_seq) * d.page_size,
                                                           0x7fffffffLL));
    ord.split_tokens = split_tokens;
    ord.n_skip = p.n_chunks;
    for (int c = 0; c < p.n_chunks; ++c) {
      ord.skip_begin[c] = p.chunk_begin[c];
      ord.skip_end[c] = p.chunk_end[c];
    }
    ord.order = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(workspace) + pl.order);
    p.row_order = ord.order;
    p.n_unit_rows = n_rows - pl.total_rows;  // the order lists every row but the tile-path chunks'
  }
  bool order_in_append = false;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (scratch != nullptr && pl.total > 0) {
    // the counters of the finished splits must start at zero; every partial
    // is written before it is read, so nothing else needs clearing
    unsigned char* base = static_cast<unsigned char*>(workspace);
    if (pl.max_splits > 1) {
      const cudaError_t e = cudaMemsetAsync(base + pl.d_count, 0, static_cast<size_t>(n_rows) * d.num_kv_heads * 4, s);
      if (e != cudaSuccess) return cuda_fail(e, "pa_attention_noalloc: clearing the split counters");
    }
    if (pl.tile_splits > 1) {
      const cudaError_t e = cudaMemsetAsync(base + pl.t_count, 0, static_cast<size_t>(pl.total_tiles) * 4, s);
      if (e != cudaSuccess) return cuda_fail(e, "pa_attention_noalloc: clearing the tile counters");
    }
  }
  if (pre != nullptr) {
    // pa_step: rows outside the chunks append their own K/V inside the
    // attention launch (each is its sequence's only row in the step); the
    // chunks' rows, which read one another's keys, are appended first by a
    // launch the attention depends on.  No chunks: one launch.
    p.fuse_append = 1;
    p.in_dtype = pre->in_dtype;
    p.k_new = pre->k_new;
    p.v_new = pre->v_new;
    for (int h = 0; h < pa::kMaxHeadScales; ++h) p.k_enc_scale_h[h] = pre->k_scale_h[h];
    p.n_all_chunks = n_chunks;
    for (int c = 0; c < n_chunks; ++c) {
      p.all_chunk_begin[c] = chunks[c].row_begin;
      p.all_chunk_end[c] = chunks[c].row_begin + chunks[c].n_rows;
    }
    if (n_chunks > 0) {
      pa::AppendParams ap = *pre;
      ap.n_ranges = n_chunks;
      ap.range_first[0] = 0;
      for (int c = 0; c < n_chunks; ++c) {
        ap.range_begin[c] = chunks[c].row_begin;
        ap.range_first[c + 1] = ap.range_first[c] + chunks[c].n_rows;
      }
      if (use_order) {
        ap.with_order = 1;
        ap.order = ord;
        order_in_append = true;
      }
      const cudaError_t ea = pa::launch_append(ap, s);
      if (ea != cudaSuccess) return cuda_fail(ea, "append launch");
      p.dependent = 1;
    }
  }
  if (use_order && !order_in_append) {
    const cudaError_t eo = pa::launch_order_rows(ord, s);
    if (eo != cudaSuccess) return cuda_fail(eo, "order launch");
    p.dependent = 1;
  }
  cudaError_t e = cudaErrorNotSupported;
  if (p.n_prefill_ctas > 0) {
    // every row on the tile path: a launch of tile CTAs of their own shape;
    // else tiles and decode units share one launch (the tiles' bits are the
    // same either way)
    e = pl.total_rows == n_rows ? pa::launch_prefill_bf16(p, s) : pa::launch_mixed_bf16(p, s);
  } else if (mma_e4m3) {
    e = pa::launch_decode_e4m3_mma(p, s);
  } else if (mma_bf16) {
    e = pa::launch_decode_bf16_mma(p, s);
  } else {
    switch (d.kv_dtype) {
      case PA_F32: e = pa::launch_decode_f32(p, s); break;
      case PA_BF16: e = pa::launch_decode_bf16(p, s); break;
      default: e = pa::launch_decode_e4m3(p, s); break;
    }
  }
  if (e == cudaErrorNotSupported) return fail(PA_ERR_UNSUPPORTED, "no decode kernel for head_dim %d, group %d", d.head_dim, G);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return PA_OK;
}

}  // namespace

pa_status pa::attention_fixed_scratch(const pa_pool* pool, int32_t n_rows, const void* q, pa_dtype q_dtype,
                                      int32_t num_q_heads, const int32_t* seq_ids, const int32_t* positions,
                                      const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                                      const pa_chunk* chunks, int32_t n_chunks, float softmax_scale, void* out,
                                      int32_t* status_dev, void* stream, const FixedScratch& scratch) {
  return attention_impl(pool, n_rows, q, q_dtype, num_q_heads, seq_ids, positions, block_tables, num_seqs,
                        max_blocks_per_seq, chunks, n_chunks, softmax_scale, out, nullptr, 0, status_dev, stream,
                        nullptr, &scratch);
}

extern "C" {

size_t pa_pool_bytes(const pa_pool_desc* desc) {
  if (check_desc(desc) != PA_OK) return 0;
  return static_cast<size_t>(desc->num_pages) * desc->num_kv_heads * desc->page_size * desc->head_dim *
         elt_bytes(desc->kv_dtype);
}

pa_status pa_pool_create(const pa_pool_desc* desc, void* k_pool, void* v_pool, pa_pool** out) {
  if (out == nullptr) return fail(PA_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (k_pool == nullptr || v_pool == nullptr) return fail(PA_ERR_INVALID_ARG, "pool buffers must not be NULL");
  if (!aligned(k_pool, 16) || !aligned(v_pool, 16)) return fail(PA_ERR_INVALID_ARG, "pool buffers must be 16-byte aligned");
  pa_pool* p = new (std::nothrow) pa_pool;
  if (p == nullptr) return fail(PA_ERR_INVALID_ARG, "out of host memory");
  p->desc = *desc;
  if (p->desc.kv_dtype != PA_FP8_E4M3) p->desc.k_scale = p->desc.v_scale = 1.0f;
  p->head_scales = false;
  p->k = k_pool;
  p->v = v_pool;
  p->tile_maps_ready = false;
  p->dec_maps_ready = false;
  *out = p;
  return PA_OK;
}

void pa_pool_destroy(pa_pool* pool) { delete pool; }

pa_status pa_pool_set_head_scales(pa_pool* pool, const float* k_scales, const float* v_scales) {
  if (pool == nullptr) return fail(PA_ERR_INVALID_ARG, "pool is NULL");
  if (k_scales == nullptr && v_scales == nullptr) {
    pool->head_scales = false;  // back to the per-tensor scales of the pool descriptor
    return PA_OK;
  }
  if (k_scales == nullptr || v_scales == nullptr)
    return fail(PA_ERR_INVALID_ARG, "give both scale arrays (or neither)");
  if (pool->desc.kv_dtype != PA_FP8_E4M3) return fail(PA_ERR_INVALID_ARG, "per-head scales apply to fp8 pools only");
  const int H = pool->desc.num_kv_heads;
  if (H > pa::kMaxHeadScales)
    return fail(PA_ERR_UNSUPPORTED, "per-head scales for %d kv heads (at most %d)", H, pa::kMaxHeadScales);
  for (int h = 0; h < H; ++h)
    if (!(std::isfinite(k_scales[h]) && k_scales[h] > 0.f && std::isfinite(v_scales[h]) && v_scales[h] > 0.f))
      return fail(PA_ERR_INVALID_ARG, "scales of kv head %d must be finite and positive (k %g, v %g)", h, k_scales[h],
                  v_scales[h]);
  for (int h = 0; h < H; ++h) {
    pool->k_scale_h[h] = k_scales[h];
    pool->v_scale_h[h] = v_scales[h];
  }
  pool->head_scales = true;
  return PA_OK;
}

pa_status pa_append_kv(const pa_pool* pool, int32_t n_rows, const void* k_new, const void* v_new, pa_dtype in_dtype,
                       const int32_t* seq_ids, const int32_t* positions, const int32_t* block_tables,
                       int32_t num_seqs, int32_t max_blocks_per_seq, int32_t* status_dev, void* stream) {
  pa::AppendParams p{};
  bool empty = true;
  const pa_status st = build_append(pool, n_rows, k_new, v_new, in_dtype, seq_ids, positions, block_tables, num_seqs,
                                    max_blocks_per_seq, status_dev, &p, &empty);
  if (st != PA_OK || empty) return st;
  cudaError_t e = pa::launch_append(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  return PA_OK;
}

size_t pa_attention_workspace_bytes(const pa_pool* pool, int32_t n_rows, int32_t num_q_heads,
                                    int32_t max_blocks_per_seq, const pa_chunk* chunks, int32_t n_chunks) {
  if (pool == nullptr || n_rows <= 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 ||
      num_q_heads % pool->desc.num_kv_heads != 0 || n_chunks < 0)
    return 0;
  // chunks of a bf16 pool may take the tile path (with bf16 queries): size for it
  return make_plan(pool->desc, n_rows, num_q_heads, max_blocks_per_seq, chunks, n_chunks,
                   pool->desc.kv_dtype == PA_BF16, g_split_tokens.load(std::memory_order_relaxed),
                   g_unit_order.load(std::memory_order_relaxed))
      .total;
}

pa_status pa_attention(const pa_pool* pool, int32_t n_rows, const void* q, pa_dtype q_dtype, int32_t num_q_heads,
                       const int32_t* seq_ids, const int32_t* positions, const int32_t* block_tables,
                       int32_t num_seqs, int32_t max_blocks_per_seq, const pa_chunk* chunks, int32_t n_chunks,
                       float softmax_scale, void* out, void* workspace, size_t workspace_bytes,
                       int32_t* status_dev, void* stream) {
  return attention_impl(pool, n_rows, q, q_dtype, num_q_heads, seq_ids, positions, block_tables, num_seqs,
                        max_blocks_per_seq, chunks, n_chunks, softmax_scale, out, workspace, workspace_bytes, status_dev,
                        stream, nullptr);
}

pa_status pa_step(const pa_pool* pool, int32_t n_rows, const void* q, pa_dtype q_dtype, int32_t num_q_heads,
                  const void* k_new, const void* v_new, pa_dtype kv_in_dtype, const int32_t* seq_ids,
                  const int32_t* positions, const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                  const pa_chunk* chunks, int32_t n_chunks, float softmax_scale, void* out, void* workspace,
                  size_t workspace_bytes, int32_t* status_dev, void* stream) {
  pa::AppendParams ap{};
  bool empty = true;
  const pa_status st = build_append(pool, n_rows, k_new, v_new, kv_in_dtype, seq_ids, positions, block_tables,
                                    num_seqs, max_blocks_per_seq, status_dev, &ap, &empty);
  if (st != PA_OK) return st;
  return attention_impl(pool, n_rows, q, q_dtype, num_q_heads, seq_ids, positions, block_tables, num_seqs,
                        max_blocks_per_seq, chunks, n_chunks, softmax_scale, out, workspace, workspace_bytes, status_dev,
                        stream, empty ? nullptr : &ap);
}

pa_status pa_set_split_tokens(int32_t tokens) {
  if (tokens <= 0 || tokens % 64 != 0 || tokens > pa::kMaxSplitTokens)
    return fail(PA_ERR_INVALID_ARG, "split tokens %d is not a multiple of 64 in [64, %d]", tokens, pa::kMaxSplitTokens);
  g_split_tokens.store(tokens, std::memory_order_relaxed);
  return PA_OK;
}

int32_t pa_get_split_tokens(void) { return g_split_tokens.load(std::memory_order_relaxed); }

pa_status pa_set_row_groups(int32_t rows) {
  if (rows != 1 && rows != 2 && rows != 4 && rows != 8)
    return fail(PA_ERR_INVALID_ARG, "row groups %d is not 1, 2, 4 or 8", rows);
  g_row_groups.store(rows, std::memory_order_relaxed);
  return PA_OK;
}

int32_t pa_get_row_groups(void) { return g_row_groups.load(std::memory_order_relaxed); }

pa_status pa_set_unit_order(int32_t mode) {
  if (mode != PA_ORDER_AUTO && mode != PA_ORDER_CALL && mode != PA_ORDER_LONGEST_FIRST)
    return fail(PA_ERR_INVALID_ARG, "unit order %d is not PA_ORDER_AUTO, PA_ORDER_CALL or PA_ORDER_LONGEST_FIRST", mode);
  g_unit_order.store(mode, std::memory_order_relaxed);
  return PA_OK;
}

int32_t pa_get_unit_order(void) { return g_unit_order.load(std::memory_order_relaxed); }

void pa_set_wait_limit(uint32_t microseconds) {
  g_wait_limit.store(microseconds == 0 ? pa::kDefaultWaitLimit : microseconds, std::memory_order_relaxed);
}

void pa_debug_stall_waits(int32_t enable) { g_debug_stall.store(enable != 0, std::memory_order_relaxed); }

const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_OUT_OF_RANGE: return "PA_ERR_OUT_OF_RANGE";
    case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_NO_PAGES: return "PA_ERR_NO_PAGES";
  }
  return "PA_ERR_UNKNOWN";
}

const char* pa_last_error(void) { return g_last_error; }

uint64_t pa_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

const char* pa_version(void) { return "paged_kv_continuous_pa_gb300 0.1 (sm_103a)"; }

}  // extern "C"
