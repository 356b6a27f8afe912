// pa_order.cuh -- the launch order of a call's decode rows: longest first.
//
// A decode launch runs one CTA per (row, split, kv head), and the GPU starts
// CTAs roughly in index order.  With the rows in the caller's order, a long
// row whose units start in the last wave runs on after everything else has
// finished, close to alone on the GPU, and the launch's end reads HBM at a
// fraction of its rate; listing the rows by decreasing work starts the long
// units in the first waves and lets the short ones fill the end.  (The
// yardstick is the fraction of the bandwidth ceiling a launch reaches,
// "llm-rs ...", section "2. Why decode is a memory problem"; the pages
// describe no launch order, this one is the library's own.)  The order only
// decides where a row's units run, never what they compute: a row's
// arithmetic and its output bits are the same at any place in the order.
//
// One CTA sorts the rows by counting: the key of a row is the number of
// 32-token stages of its longest unit, min(position + 1, split length) / 32
// rounded up; rows whose sequence or position is out of range take key 0 and
// go last (their units write zeros and report the error), and rows of
// tile-path chunks are left out (the launch has no decode units for them).  Rows with
// equal keys keep no particular order.  Counting and placing go through
// shared-memory atomics aggregated per warp over lanes of equal key, so a
// batch of equal keys costs one atomic per warp.
#pragma once

#include "pa_device.cuh"

namespace pa {

constexpr int kOrderBins = kMaxSplitTokens / kStageTokens + 1;  // keys 0 .. split / 32

__device__ __forceinline__ int order_key(const OrderParams& o, int r) {
  for (int c = 0; c < o.n_skip; ++c)
    if (r >= o.skip_begin[c] && r < o.skip_end[c]) return -1;  // left out: no decode units
  const int seq = __ldg(o.seq_ids + r), pos = __ldg(o.positions + r);
  if (seq < 0 || seq >= o.num_seqs || pos < 0 || pos >= o.max_pos) return 0;
  const int keys = min(pos + 1, o.split_tokens);
  return (keys + kStageTokens - 1) / kStageTokens;
}

// The whole CTA (any multiple of 32 threads) writes o.order.
__device__ __forceinline__ void order_rows_block(const OrderParams& o) {
  __shared__ int start[kOrderBins];
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31;
  const unsigned below = (1u << lane) - 1u;
  for (int b = tid; b < kOrderBins; b += nt) start[b] = 0;
  __syncthreads();
  // rows per key
  for (int base = 0; base < o.n_rows; base += nt) {  // uniform trip count: every lane takes part in the match
    const int r = base + tid;
    const int k = r < o.n_rows ? order_key(o, r) : -1;
    const unsigned same = __match_any_sync(0xffffffffu, k);
    if (k >= 0 && (same & below) == 0) atomicAdd(&start[k], __popc(same));
  }
  __syncthreads();
  if (tid < 32) {
    // start[k] = rows with a larger key: an exclusive scan from the top key
    // down, PER keys a lane, then across the lanes
    constexpr int PER = (kOrderBins + 31) / 32;
    int c[PER], sum = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int b = kOrderBins - 1 - (lane * PER + i);
      c[i] = b >= 0 ? start[b] : 0;
      sum += c[i];
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int acc = incl - sum;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int b = kOrderBins - 1 - (lane * PER + i);
      if (b >= 0) start[b] = acc;
      acc += c[i];
    }
  }
  __syncthreads();
  // each row into its key's range
  for (int base = 0; base < o.n_rows; base += nt) {
    const int r = base + tid;
    const int k = r < o.n_rows ? order_key(o, r) : -1;
    const unsigned same = __match_any_sync(0xffffffffu, k);
    const int leader = __ffs(same) - 1;
    int first = 0;
    if (k >= 0 && lane == leader) first = atomicAdd(&start[k], __popc(same));
    first = __shfl_sync(0xffffffffu, first, leader);
    if (k >= 0) o.order[first + __popc(same & below)] = r;
  }
}

}  // namespace pa
