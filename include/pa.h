/*
 * pa.h -- C ABI of libpa_gb300: batched attention over a paged key/value pool
 * for a continuous-batching engine, on one NVIDIA GB300 (sm_103a).
 *
 * What it computes ("GPU inference engine engineering", section "Batching
 * without running out of cache"; "Building an LLM runtime from scratch on
 * NVIDIA H100", section "Bug #1"; "llm-rs: LLM Inference in Rust ...",
 * section "4. Going down a level: SIMT kernels"):
 *   - K/V live in a pool of fixed-size pages; each sequence owns a block table
 *     mapping its logical page j (tokens j*P .. j*P+P-1) to a physical page.
 *   - A step is a set of rows; each row carries its own query, sequence id and
 *     position.  pa_append_kv scatters the rows' new keys and values into their
 *     page slots; pa_attention then computes, for every row r and query head g,
 *         out[r][g] = softmax_t( scale * q[r][g] . K_s[t] ) . V_s[t],  t = 0..position
 *     over the row's own sequence s, with kv head g / (Hq / Hkv) (grouped-query
 *     heads), an FP32 online softmax, and a split-KV path for long contexts whose
 *     partial (max, sum, acc) triples are merged in a fixed order.
 *   - Rows listed in a prefill chunk (consecutive rows of one sequence at
 *     consecutive positions) run on a tensor-core tile path in the same launch.
 *
 * Conventions for every entry point:
 *   - All device memory (pools, q, k/v, out, tables, workspace, status) is
 *     allocated and owned by the caller.  The library owns only the small host
 *     pa_pool object.  No call allocates device memory or synchronises.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default).
 *   - Host-side argument errors return a status at once, launch nothing, and
 *     set a thread-local message readable with pa_last_error().  No C++
 *     exception crosses the ABI.
 *   - Device-side errors (a sequence id, position or page id out of range, a
 *     bounded wait that ran out) are recorded in *status_dev (int32 in device
 *     memory, may be NULL): the first error code wins (compare-and-swap from
 *     PA_OK).  The caller zeroes it and reads it back when it wants to know.
 *     Rows hit by such an error get unspecified output (zeros for rows whose
 *     sequence id or position is invalid); the kernels never trap.
 *
 * Layouts (row-major, innermost last):
 *   k_pool, v_pool   [num_pages][Hkv][P][D]     kv_dtype, 16-byte aligned
 *   q, out           [n_rows][Hq][D]            q_dtype (out has q's dtype), 16-byte aligned
 *   k_new, v_new     [n_rows][Hkv][D]           in_dtype
 *   seq_ids, positions [n_rows]                 int32
 *   block_tables     [num_seqs][max_blocks_per_seq] int32, unused entries -1
 */
#ifndef PA_GB300_H
#define PA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1, /* host-side: a bad pointer, size, dtype or alignment */
    PA_ERR_UNSUPPORTED = 2, /* host-side: a valid but unimplemented shape (e.g. head_dim 96) */
    PA_ERR_OUT_OF_RANGE = 3, /* device-side: sequence id, position or page id out of range */
    PA_ERR_TIMEOUT = 4,     /* device-side: a bounded wait on a copy gave up */
    PA_ERR_CUDA = 5,        /* a CUDA runtime call failed (launch, attribute, driver entry point), or a kernel found its launch configuration inconsistent */
    PA_ERR_NO_PAGES = 6     /* host-side: an admission needs more free pages than the pool has */
} pa_status;

typedef enum { PA_F32 = 0, PA_BF16 = 1, PA_FP8_E4M3 = 2 } pa_dtype;

/* Pool geometry.  page_size in {16, 32, 64, 128, 256}; head_dim in {64, 128};
 * kv_dtype PA_F32, PA_BF16 or PA_FP8_E4M3.  k_scale / v_scale are the fp8
 * per-tensor scales ("Engines for the card you have", section "One checkpoint,
 * many engines": an FP8 key/value cache, calibrated): a stored code c means
 * value(c) * scale, and appending x stores e4m3_satfinite_rne(x / scale).
 * They are ignored (taken as 1) for f32 and bf16 pools. */
typedef struct {
    int32_t num_pages;
    int32_t page_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    pa_dtype kv_dtype;
    float k_scale;
    float v_scale;
} pa_pool_desc;

typedef struct pa_pool pa_pool; /* opaque host object */

/* Rows row_begin .. row_begin + n_rows - 1 of a step form one causal prefill
 * chunk: they must share one sequence id and have consecutive increasing
 * positions.  Host memory. */
typedef struct {
    int32_t row_begin;
    int32_t n_rows;
} pa_chunk;

/* Bytes of ONE of the two pool buffers (K or V) for this geometry: the memory
 * need, computed without allocating ("GPU inference engine engineering",
 * "Batching without running out of cache": the engine computes its memory need
 * without allocating).  Returns 0 for an invalid descriptor. */
size_t pa_pool_bytes(const pa_pool_desc *desc);

/* Wrap caller-owned device buffers k_pool and v_pool (each pa_pool_bytes(desc)
 * bytes, 16-byte aligned) in a host object.  Contents are not touched.
 * Errors: PA_ERR_INVALID_ARG (NULL pointer, misaligned buffer, non-positive
 * sizes, fp8 scale not finite and > 0), PA_ERR_UNSUPPORTED (page_size or
 * head_dim outside the supported sets). */
pa_status pa_pool_create(const pa_pool_desc *desc, void *k_pool, void *v_pool, pa_pool **out);

/* Free the host object (not the device buffers).  NULL is allowed. */
void pa_pool_destroy(pa_pool *pool);

/* One fp8 scale per kv head instead of the descriptor's per-tensor scales
 * ("Engines for the card you have", section "One checkpoint, many engines":
 * a calibrated FP8 key/value cache; the calibration's granularity is the
 * caller's).  k_scales, v_scales: HOST arrays of num_kv_heads floats, copied;
 * kv head h stores e4m3_satfinite_rne(x / k_scales[h]) and decodes
 * value(c) * k_scales[h] (likewise V).  Both NULL: back to the per-tensor
 * scales.  Errors: PA_ERR_INVALID_ARG (one array NULL, a pool that is not
 * fp8, a scale not finite and positive), PA_ERR_UNSUPPORTED (more than 64 kv
 * heads).  Takes effect for calls made after it. */
pa_status pa_pool_set_head_scales(pa_pool *pool, const float *k_scales, const float *v_scales);

/* K/V append ("GPU inference engine engineering", "Batching without running
 * out of cache"): for each row r, kv head h and element d,
 *     pool[block_tables[s][p / P]][h][p % P][d] = enc(new[r][h][d]),  s = seq_ids[r], p = positions[r]
 * for K and V.  enc is a copy (f32->f32, bf16->bf16, bf16->f32 widening),
 * fp32->bf16 round-to-nearest-even, or for fp8 pools e4m3 satfinite
 * round-to-nearest-even of (x / scale) with one IEEE binary32 division.
 * in_dtype is PA_F32 or PA_BF16.  One launch on `stream`.
 * Precondition: no two rows of one call write the same (page, slot); shared
 * prefix pages are never append targets.  n_rows == 0 is a no-op.
 * Device-side: a row with s outside [0, num_seqs), p outside
 * [0, max_blocks_per_seq * P) or a page id outside [0, num_pages) is skipped
 * and records PA_ERR_OUT_OF_RANGE. */
pa_status pa_append_kv(const pa_pool *pool, int32_t n_rows, const void *k_new, const void *v_new,
                       pa_dtype in_dtype, const int32_t *seq_ids, const int32_t *positions,
                       const int32_t *block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                       int32_t *status_dev, void *stream);

/* Workspace bytes pa_attention needs for these rows, this block-table width
 * and these prefill chunks (the split-KV partial triples of decode rows and of
 * chunk tiles, their counters, and the decode rows' launch order when
 * pa_set_unit_order asks for one).  0 when nothing can be split or ordered.
 * Computed on the host from sizes only; for a bf16 pool it assumes the chunks
 * take the tensor-core tile path (bf16 queries), which never needs less. */
size_t pa_attention_workspace_bytes(const pa_pool *pool, int32_t n_rows, int32_t num_q_heads,
                                    int32_t max_blocks_per_seq, const pa_chunk *chunks, int32_t n_chunks);

/* Paged attention over a step's rows (see the top of this file).
 *   q_dtype      PA_F32 or PA_BF16; out has the same dtype, rounded to nearest even
 *   num_q_heads  a multiple of the pool's num_kv_heads, with Hq / Hkv in 1..8
 *   chunks       host array of n_chunks prefill chunks (may be NULL when n_chunks == 0);
 *                at most 16 chunks.  Rows not in a chunk are decode rows.
 *   softmax_scale <= 0 selects 1 / sqrt(head_dim)
 *   workspace    device memory of at least pa_attention_workspace_bytes(...), 256-byte
 *                aligned, ZERO-FILLED BEFORE ITS FIRST USE; every call leaves the split
 *                counters in it at zero again, so it is reused without clearing (except
 *                after a call that reported PA_ERR_TIMEOUT: clear it again); the other
 *                bytes are scratch that each call writes before it reads them.  Calls that
 *                share a workspace must not overlap on the GPU.  May be NULL when 0 bytes
 *                are needed.
 * Each row attends keys 0..positions[r] of its own sequence (its own token
 * included, so append the step's rows first).  A row's output bits depend only
 * on that row's inputs and on the rows of its own chunk, never on the other
 * rows of the call or the physical placement of its pages.
 * One launch on `stream` (split partials are merged inside it), preceded by
 * the one-CTA launch that orders the decode rows when pa_set_unit_order says
 * so; no allocation; graph-capturable.  Errors: PA_ERR_INVALID_ARG (NULL or misaligned pointer,
 * bad sizes, overlapping chunks, workspace too small), PA_ERR_UNSUPPORTED (a
 * group size or head_dim without a kernel), PA_ERR_CUDA (a failed launch). */
pa_status pa_attention(const pa_pool *pool, int32_t n_rows, const void *q, pa_dtype q_dtype,
                       int32_t num_q_heads, const int32_t *seq_ids, const int32_t *positions,
                       const int32_t *block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                       const pa_chunk *chunks, int32_t n_chunks, float softmax_scale, void *out,
                       void *workspace, size_t workspace_bytes, int32_t *status_dev, void *stream);

/* One decode/prefill step: pa_append_kv of the step's rows, then pa_attention
 * over the same rows ("GPU inference engine engineering", section "Speed that
 * counts end to end": fewer launches per step; "Building an LLM runtime from
 * scratch on NVIDIA H100", section "Bug #2: Eager Decode and the CUDA Graph
 * Necessity": the launch gaps of eager decoding).
 *   - Rows outside every chunk (decode rows) append their own new K/V inside
 *     the attention launch: for each kv head, the attention unit that holds
 *     the row's position stores the row's converted key and value in the pool
 *     before it copies that page, so a step without chunks is ONE attention
 *     launch (behind the one-CTA order launch when pa_set_unit_order orders
 *     its rows; a step with chunks has its append launch write the order).
 *   - Chunk rows read one another's keys, so they are appended first by an
 *     append launch over the chunks' rows only; the attention kernel is its
 *     programmatic dependent (its CTAs start their lookups while the append
 *     runs; chunk tiles and chunk rows wait for it before reading the pools,
 *     decode rows do not wait).
 * Precondition (beyond those of pa_append_kv and pa_attention): a row outside
 * every chunk is the only row of its sequence in the step; a sequence that
 * contributes several rows to one step lists them as a chunk.
 *   k_new, v_new, kv_in_dtype: as pa_append_kv's k_new, v_new, in_dtype
 *   the other arguments: as pa_attention
 * Results (pool bytes and outputs) are bit-identical to pa_append_kv followed
 * by pa_attention on the same stream.  Every argument of both is checked
 * before anything is launched; errors as for those two calls.  Capturable in
 * a CUDA graph. */
pa_status pa_step(const pa_pool *pool, int32_t n_rows, const void *q, pa_dtype q_dtype, int32_t num_q_heads,
                  const void *k_new, const void *v_new, pa_dtype kv_in_dtype, const int32_t *seq_ids,
                  const int32_t *positions, const int32_t *block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                  const pa_chunk *chunks, int32_t n_chunks, float softmax_scale, void *out, void *workspace,
                  size_t workspace_bytes, int32_t *status_dev, void *stream);

/* pa_attention without a workspace argument, for callers that cannot allocate
 * device memory: code handed only its input and output buffers by a host
 * runtime that owns and budgets all device memory (a plugin interface), or a
 * serving loop that forbids cudaMalloc after start-up because an allocation on
 * the hot path can synchronise the device or fail under memory pressure.  The
 * pages have no counterpart to this entry point; it exists for such callers.
 * The split-KV partials go to a scratch array of 32 MiB compiled into the
 * library's device image: every GPU that loads the library holds it until the
 * process exits, and this call allocates nothing (no cudaMalloc, no cudaFree,
 * no allocating library routine).  Arguments and results are those of
 * pa_attention, checked the same way first.  A call whose split-KV plan (the
 * bytes pa_attention would need for these rows, chunks, dtypes and split
 * length) exceeds 32 MiB is rejected with PA_ERR_UNSUPPORTED and a message in
 * pa_last_error(); the split length is read once per call.
 * The first call on a device that needs the array looks up its device
 * address (with that device current), and looks it up again when the
 * device's CUDA context has changed since (after cudaDeviceReset, for
 * instance); make that first call before any stream capture.  Every call
 * shares the one array and finds the previous call's contents in it; each
 * call clears its plan's split counters on `stream` first (every other byte
 * it reads, it has written).  Calls that can run at the same time on the GPU
 * (unordered streams) race on the array. */
pa_status pa_attention_noalloc(const pa_pool *pool, int32_t n_rows, const void *q, pa_dtype q_dtype,
                               int32_t num_q_heads, const int32_t *seq_ids, const int32_t *positions,
                               const int32_t *block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                               const pa_chunk *chunks, int32_t n_chunks, float softmax_scale, void *out,
                               int32_t *status_dev, void *stream);

/* Split-KV chunk length in tokens: a row at position p is cut into
 * ceil((p + 1) / split) pieces merged in ascending order.  A process-wide
 * constant (default 4096), a multiple of 64 up to 4096, never derived from the batch.
 * These settings (split length, row groups, wait limit, injected stall) may be changed from
 * any thread; a call reads each of them once, when it starts, so one call never
 * mixes two values.  A workspace sized by pa_attention_workspace_bytes before a
 * change may be too small after it: the call then returns PA_ERR_INVALID_ARG.
 * Changing it changes output bits (within tolerance) for rows longer than it.
 * Returns PA_ERR_INVALID_ARG for a value that is not a positive multiple of 64. */
pa_status pa_set_split_tokens(int32_t tokens);
int32_t pa_get_split_tokens(void);

/* Row groups for the FP8 (E4M3) tensor-core decode units (head_dim 128, bf16
 * queries): with rows = 2, 4 or 8, one CTA takes that many consecutive decode
 * rows of the call for one kv head and split, and the leading pages that all
 * of its rows share (the same physical page ids, full 32-token stages, none a
 * row's last) are copied into shared memory once and read by every row
 * ("GPU inference engine engineering", section "The same bits in any batch":
 * a shared prompt prefix staged once for eight rows).  Rows share pages only
 * when the caller lists the rows of one prefix next to one another (a
 * scheduler that groups its batches by prefix, section "Caching measured on
 * the real prompt structure").  1 (the default) runs one row per CTA.  Output
 * bits never depend on it: each row's arithmetic is the same in both forms.
 * Other pools and query dtypes ignore it.  A process-wide setting, read once
 * per call like the split length.  Returns PA_ERR_INVALID_ARG for a value
 * other than 1, 2, 4 or 8. */
pa_status pa_set_row_groups(int32_t rows);
int32_t pa_get_row_groups(void);

/* Launch order of the decode rows.  A decode launch runs one CTA per (row,
 * split, kv head) and the GPU starts CTAs roughly in index order, so a long
 * row listed late starts in the last wave and runs on after the rest of the
 * launch has finished, reading HBM at a fraction of its rate (the pages
 * measure a kernel by its fraction of the bandwidth ceiling: "llm-rs ...",
 * section "2. Why decode is a memory problem"; they describe no launch
 * order).  PA_ORDER_LONGEST_FIRST runs the units of the rows with the most
 * keys per unit first: one CTA, of a launch of its own or of pa_step's append
 * launch, sorts the rows by the key
 * count of their longest unit into the workspace, and the attention launch
 * reads the order (its programmatic dependent).  PA_ORDER_CALL keeps the
 * call's order, one launch fewer.  PA_ORDER_AUTO (the default) orders a call
 * of at least 128 decode rows whose units can hold 1024 keys or more
 * (max_blocks_per_seq * page_size and the split length both at least 1024),
 * and keeps the order of other calls.  Output bits never depend on it: a
 * row's arithmetic is the same wherever it runs.  Row groups (rows > 1 above)
 * keep the call's order.  A process-wide setting, read once per call like the
 * split length; the workspace size depends on it.  Returns PA_ERR_INVALID_ARG
 * for another value. */
enum { PA_ORDER_AUTO = 0, PA_ORDER_CALL = 1, PA_ORDER_LONGEST_FIRST = 2 };
pa_status pa_set_unit_order(int32_t mode);
int32_t pa_get_unit_order(void);

/* Longest time, in microseconds, one device-side wait (for a copy or an MMA
 * to complete) may take before it gives up with PA_ERR_TIMEOUT; 0 restores
 * the default of one second.  A debugging knob for failure-path tests. */
void pa_set_wait_limit(uint32_t microseconds);

/* Failure-path testing without a GPU fault: with enable != 0, every attention
 * CTA additionally waits on a barrier that nothing ever completes, so that
 * wait runs out after the current wait limit; the call then reports
 * PA_ERR_TIMEOUT in *status_dev, its outputs are unspecified, and the kernel
 * still returns normally.  Set a small wait limit first (e.g. 1000 us).
 * Off by default; affects calls made while it is on. */
void pa_debug_stall_waits(int32_t enable);

const char *pa_status_string(pa_status status);

/* Detail text of the last host-side error on this thread ("" if none). */
const char *pa_last_error(void);

/* Number of CUDA kernels this library has launched in this process (all
 * entry points, all devices): lets a caller count the launches of a region. */
uint64_t pa_kernel_launches(void);

/* Library version string. */
const char *pa_version(void);

/* ---- Page allocator with admission (host side) ----------------------------
 * "GPU inference engine engineering", section "Batching without running out of
 * cache": a request is admitted only if the pages for its whole prompt AND its
 * whole answer can be reserved up front; a refusal gives a typed reason and
 * the numbers; the need is computable without allocating; a refused admission
 * takes nothing.  The allocator owns page ids of one pool (0 .. num_pages-1)
 * and the block-table rows of num_seqs sequence slots; it fills rows of a
 * caller-owned HOST array int32 [num_seqs][max_blocks_per_seq] (unused
 * entries -1), which the caller copies to the device for pa_append_kv /
 * pa_attention.  Prefix sharing: a sequence may share the whole pages of an
 * admitted parent's prompt prefix (reference counted; the page holding the
 * prefix's last partial tokens is the sequence's own).  Page ids are handed
 * out in a deterministic order (lowest first from a fresh allocator; a
 * release followed by the same admission returns the same pages).  Not
 * thread-safe: one scheduler thread owns an allocator. */
typedef struct pa_pages pa_pages; /* opaque host object */

typedef enum {
    PA_ADMIT_OK = 0,
    PA_ADMIT_NO_PAGES = 1,   /* fewer free pages than the admission needs (status PA_ERR_NO_PAGES) */
    PA_ADMIT_TOO_LONG = 2,   /* prompt + answer exceed max_blocks_per_seq * page_size tokens */
    PA_ADMIT_SEQ_IN_USE = 3, /* the sequence slot already holds pages */
    PA_ADMIT_BAD_ARG = 4     /* slot out of range, negative counts, prefix parent not admitted */
} pa_admit_reason;

typedef struct {
    pa_admit_reason reason;
    int32_t pages_needed;  /* new pages the admission takes (shared prefix pages excluded) */
    int32_t pages_free;    /* free pages when the admission was asked */
    int32_t pages_shared;  /* whole prefix pages shared with the parent */
    int32_t tokens;        /* prompt + answer tokens asked for */
    int32_t max_tokens;    /* tokens one block-table row can hold */
} pa_admit_info;

/* Pages a sequence of prompt_tokens + max_new_tokens tokens needs:
 * ceil((prompt + answer) / page_size).  No state; -1 on bad arguments.
 * Times pa_pool_bytes(desc) / desc.num_pages it is the device memory. */
int32_t pa_pages_needed(int32_t page_size, int32_t prompt_tokens, int32_t max_new_tokens);

/* An allocator over num_pages pages of page_size tokens for num_seqs sequence
 * slots of max_blocks_per_seq pages.  Errors: PA_ERR_INVALID_ARG. */
pa_status pa_pages_create(int32_t num_pages, int32_t page_size, int32_t num_seqs, int32_t max_blocks_per_seq,
                          pa_pages **out);
void pa_pages_destroy(pa_pages *pages);

/* Admit sequence slot seq for prompt_tokens + max_new_tokens tokens: reserve
 * every page up front and write the slot's row of block_tables (host, may be
 * NULL).  prefix_parent >= 0 shares the parent's first prefix_tokens / page_size
 * pages (prefix_tokens <= prompt_tokens); -1 for none.  *info (may be NULL)
 * receives the reason and the numbers.  Returns PA_OK; PA_ERR_NO_PAGES when
 * too few pages are free; PA_ERR_INVALID_ARG for the other reasons.  A refused
 * admission changes nothing. */
pa_status pa_pages_admit(pa_pages *pages, int32_t seq, int32_t prompt_tokens, int32_t max_new_tokens,
                         int32_t prefix_parent, int32_t prefix_tokens, int32_t *block_tables, pa_admit_info *info);

/* Release slot seq: drop its hold on each page (a page returns to the free
 * list when no sequence holds it) and reset its block_tables row to -1
 * (block_tables may be NULL).  PA_ERR_INVALID_ARG if the slot holds nothing. */
pa_status pa_pages_release(pa_pages *pages, int32_t seq, int32_t *block_tables);

int32_t pa_pages_free_count(const pa_pages *pages);            /* -1 if pages is NULL */
int32_t pa_pages_refcount(const pa_pages *pages, int32_t page); /* sequences holding page; -1 if out of range */

#ifdef __cplusplus
}
#endif

#endif /* PA_GB300_H */
