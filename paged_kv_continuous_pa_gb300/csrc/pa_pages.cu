// pa_pages.cu -- the host-side page allocator with admission (pa_pages_* in
// include/pa.h).  Host code only: no kernel, no device memory.
//
// "GPU inference engine engineering", section "Batching without running out
// of cache": a request is admitted only if pages for its whole prompt and its
// whole answer can be reserved up front, a refusal says why and with which
// numbers, the need can be computed without allocating, and a failed
// admission leaves nothing allocated.  Prefix pages shared between sequences
// are reference counted; only whole pages of the prefix are shared (the page
// holding the prefix's last partial tokens belongs to each sequence).
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <new>
#include <vector>

#include "../../include/pa.h"
#include "pa_kernels.h"

struct pa_pages {
  int32_t num_pages, page_size, num_seqs, max_blocks;
  std::vector<int32_t> free_stack;             // free page ids; the next one handed out is at the back
  std::vector<int32_t> refs;                   // per page: sequences holding it
  std::vector<std::vector<int32_t>> seq_pages;  // per sequence slot: its pages in logical order
  std::vector<char> in_use;                    // per sequence slot: admitted and not yet released
};

namespace {

pa_status refuse(pa_admit_info* info, pa_admit_reason reason, pa_status st, const char* fmt, ...) {
  if (info != nullptr) info->reason = reason;
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  pa::set_last_error("%s", buf);
  return st;
}

int32_t ceil_div(int64_t a, int64_t b) { return static_cast<int32_t>((a + b - 1) / b); }

}  // namespace

extern "C" {

int32_t pa_pages_needed(int32_t page_size, int32_t prompt_tokens, int32_t max_new_tokens) {
  if (page_size <= 0 || prompt_tokens < 0 || max_new_tokens < 0) return -1;
  const int64_t tokens = static_cast<int64_t>(prompt_tokens) + max_new_tokens;
  const int64_t pages = (tokens + page_size - 1) / page_size;
  return pages > 0x7fffffff ? -1 : static_cast<int32_t>(pages);
}

pa_status pa_pages_create(int32_t num_pages, int32_t page_size, int32_t num_seqs, int32_t max_blocks_per_seq,
                          pa_pages** out) {
  if (out == nullptr) {
    pa::set_last_error("pa_pages_create: out is NULL");
    return PA_ERR_INVALID_ARG;
  }
  *out = nullptr;
  if (num_pages <= 0 || page_size <= 0 || num_seqs <= 0 || max_blocks_per_seq <= 0) {
    pa::set_last_error("pa_pages_create: sizes must be positive (pages %d, page size %d, sequences %d, blocks %d)",
                       num_pages, page_size, num_seqs, max_blocks_per_seq);
    return PA_ERR_INVALID_ARG;
  }
  pa_pages* a = new (std::nothrow) pa_pages;
  if (a == nullptr) {
    pa::set_last_error("pa_pages_create: out of host memory");
    return PA_ERR_INVALID_ARG;
  }
  try {
    a->num_pages = num_pages;
    a->page_size = page_size;
    a->num_seqs = num_seqs;
    a->max_blocks = max_blocks_per_seq;
    a->free_stack.resize(num_pages);
    for (int32_t i = 0; i < num_pages; ++i) a->free_stack[i] = num_pages - 1 - i;  // hands out 0, 1, 2, ...
    a->refs.assign(num_pages, 0);
    a->seq_pages.assign(num_seqs, std::vector<int32_t>());
    a->in_use.assign(num_seqs, 0);
  } catch (...) {
    delete a;
    pa::set_last_error("pa_pages_create: out of host memory");
    return PA_ERR_INVALID_ARG;
  }
  *out = a;
  return PA_OK;
}

void pa_pages_destroy(pa_pages* a) { delete a; }

int32_t pa_pages_free_count(const pa_pages* a) { return a == nullptr ? -1 : static_cast<int32_t>(a->free_stack.size()); }

int32_t pa_pages_refcount(const pa_pages* a, int32_t page) {
  if (a == nullptr || page < 0 || page >= a->num_pages) return -1;
  return a->refs[page];
}

pa_status pa_pages_admit(pa_pages* a, int32_t seq, int32_t prompt_tokens, int32_t max_new_tokens,
                         int32_t prefix_parent, int32_t prefix_tokens, int32_t* block_tables, pa_admit_info* info) {
  if (info != nullptr) *info = pa_admit_info{PA_ADMIT_OK, 0, 0, 0, 0, 0};
  if (a == nullptr) return refuse(info, PA_ADMIT_BAD_ARG, PA_ERR_INVALID_ARG, "pa_pages_admit: allocator is NULL");
  const int32_t max_tokens = a->max_blocks * a->page_size;
  if (info != nullptr) {
    info->pages_free = static_cast<int32_t>(a->free_stack.size());
    info->max_tokens = max_tokens;
  }
  if (seq < 0 || seq >= a->num_seqs)
    return refuse(info, PA_ADMIT_BAD_ARG, PA_ERR_INVALID_ARG, "pa_pages_admit: sequence %d outside [0, %d)", seq,
                  a->num_seqs);
  if (prompt_tokens < 0 || max_new_tokens < 0)
    return refuse(info, PA_ADMIT_BAD_ARG, PA_ERR_INVALID_ARG, "pa_pages_admit: negative token counts (%d, %d)",
                  prompt_tokens, max_new_tokens);
  if (a->in_use[seq])
    return refuse(info, PA_ADMIT_SEQ_IN_USE, PA_ERR_INVALID_ARG, "pa_pages_admit: sequence %d already holds %zu pages",
                  seq, a->seq_pages[seq].size());
  const int64_t tokens = static_cast<int64_t>(prompt_tokens) + max_new_tokens;
  if (info != nullptr) info->tokens = tokens > 0x7fffffff ? 0x7fffffff : static_cast<int32_t>(tokens);
  if (tokens > max_tokens)
    return refuse(info, PA_ADMIT_TOO_LONG, PA_ERR_INVALID_ARG,
                  "pa_pages_admit: %lld tokens (prompt %d + answer %d) exceed the %d a block-table row holds",
                  static_cast<long long>(tokens), prompt_tokens, max_new_tokens, max_tokens);
  const int32_t total = ceil_div(tokens, a->page_size);
  int32_t shared = 0;
  if (prefix_parent >= 0) {
    if (prefix_parent >= a->num_seqs || prefix_parent == seq || !a->in_use[prefix_parent])
      return refuse(info, PA_ADMIT_BAD_ARG, PA_ERR_INVALID_ARG,
                    "pa_pages_admit: prefix parent %d is not an admitted sequence", prefix_parent);
    if (prefix_tokens < 0 || prefix_tokens > prompt_tokens)
      return refuse(info, PA_ADMIT_BAD_ARG, PA_ERR_INVALID_ARG,
                    "pa_pages_admit: prefix of %d tokens outside the %d-token prompt", prefix_tokens, prompt_tokens);
    shared = std::min(prefix_tokens / a->page_size, static_cast<int32_t>(a->seq_pages[prefix_parent].size()));
  }
  const int32_t fresh = total - shared;
  if (info != nullptr) {
    info->pages_needed = fresh;
    info->pages_shared = shared;
  }
  if (fresh > static_cast<int32_t>(a->free_stack.size()))
    return refuse(info, PA_ADMIT_NO_PAGES, PA_ERR_NO_PAGES,
                  "pa_pages_admit: sequence %d needs %d new pages (%lld tokens, %d shared prefix pages) and %zu are free",
                  seq, fresh, static_cast<long long>(tokens), shared, a->free_stack.size());
  // every check passed: take the pages (nothing above has changed any state)
  std::vector<int32_t>& mine = a->seq_pages[seq];
  mine.clear();
  mine.reserve(total);
  for (int32_t i = 0; i < shared; ++i) {
    const int32_t pg = a->seq_pages[prefix_parent][i];
    ++a->refs[pg];
    mine.push_back(pg);
  }
  for (int32_t i = 0; i < fresh; ++i) {
    const int32_t pg = a->free_stack.back();
    a->free_stack.pop_back();
    a->refs[pg] = 1;
    mine.push_back(pg);
  }
  a->in_use[seq] = 1;
  if (block_tables != nullptr) {
    int32_t* row = block_tables + static_cast<size_t>(seq) * a->max_blocks;
    for (int32_t j = 0; j < a->max_blocks; ++j) row[j] = j < total ? mine[j] : -1;
  }
  return PA_OK;
}

pa_status pa_pages_release(pa_pages* a, int32_t seq, int32_t* block_tables) {
  if (a == nullptr) {
    pa::set_last_error("pa_pages_release: allocator is NULL");
    return PA_ERR_INVALID_ARG;
  }
  if (seq < 0 || seq >= a->num_seqs || !a->in_use[seq]) {
    pa::set_last_error("pa_pages_release: sequence %d holds no pages", seq);
    return PA_ERR_INVALID_ARG;
  }
  std::vector<int32_t>& mine = a->seq_pages[seq];
  // last page first, so that a release followed by the same admission gets the same pages back
  for (auto it = mine.rbegin(); it != mine.rend(); ++it)
    if (--a->refs[*it] == 0) a->free_stack.push_back(*it);
  mine.clear();
  a->in_use[seq] = 0;
  if (block_tables != nullptr) {
    int32_t* row = block_tables + static_cast<size_t>(seq) * a->max_blocks;
    for (int32_t j = 0; j < a->max_blocks; ++j) row[j] = -1;
  }
  return PA_OK;
}

}  // extern "C"
