// pa_prefill.cuh -- causal prefill-chunk tiles on the 5th-generation tensor
// cores (tcgen05), reading K/V straight from the paged pool.
//
// What it computes ("llm-rs ...", section "Prefill: tensor cores, written by
// hand": flash-style prefill attention over the paged cache, K/V tiles shared
// across query rows, tensor cores): for one kv head h and one tile of a chunk,
// the 128 rows (position, query head) = R = 128 / G consecutive chunk
// positions times the G query heads of h, attend causally to keys
// 0..position of the chunk's sequence:
//     S = Q K^T          tcgen05.mma, Q from tensor memory, K from shared memory,
//                        BF16 x BF16 -> FP32 in tensor memory
//     online softmax     FP32, one thread per row, masked by key <= position
//     O += P V           tcgen05.mma, P from tensor memory as a (hi, lo) BF16
//                        pair, V from shared memory, FP32 accumulator in TMEM
// over key tiles of 64 keys, then O / l rounded to BF16.
//
// The CTA has the decode unit's shape (4 warps, about 50 KB of shared memory,
// at most 128 registers a thread) so that tiles and decode units share one
// launch without lowering the decode occupancy.  Shared memory holds one K
// tile and two V tiles (128-byte swizzled, loaded by 2-D tensor-map copies of
// one page x 64 head elements each; the block table gives the row
// coordinate; no multicast).  Tensor memory (256 columns) holds S, then P in
// place, Q, and O.  Thread m owns TMEM lane m = tile row m.  Every wait is
// made by all 128 threads on an mbarrier (copies landed: bulk bytes; MMAs
// done: tcgen05.commit); thread 0 alone issues copies and MMAs between them.
//
// Precision: the scores and the softmax are FP32.  Each weight p enters the
// P.V product as hi = bf16(p) and lo = bf16(p - hi), so the product sees p to
// about 16 significant bits; the tensor core accumulates in FP32 and l sums
// the FP32 weights.
#pragma once

#include "pa_device.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

constexpr int kTileM = 128;  // rows per tile (TMEM lanes)
constexpr int kTileN = 64;   // keys per key tile

template <int D>
struct PrefillSmem {  // byte offsets from a 1024-byte aligned base
  static constexpr int NH = D / 64;        // 64-element halves of the head dim
  static constexpr int KH = kTileN * 128;  // one half of a K or V tile: 8 KiB
  static constexpr int TILE = NH * KH;     // one K or V tile
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + TILE;  // two value tiles
  static constexpr int BAR_OFF = V_OFF + 2 * TILE;
  static constexpr int TOTAL = BAR_OFF + 128;
  static constexpr int BYTES = TOTAL + 1024;  // slack for aligning the base
};

enum { BAR_K = 0, BAR_V0 = 1, BAR_V1 = 2, BAR_S = 3, BAR_O = 4, BAR_STALL = 5, BAR_COUNT = 6 };

// TMEM columns: [0, 64) S of one key tile, then P (hi in [0, 32), lo in [32, 64));
// [64, 64 + D/2) Q; [128, 128 + D) O.
constexpr uint32_t kColSP = 0, kColQ = 64, kColO = 128, kTmemCols = 256;

// Thread 0's record of the copies and MMAs it issued on each barrier; a barrier
// never has more than one phase outstanding, so after a failure each pending
// operation is drained by waiting for the parity of its own phase.
struct PrefillIssueLog {
  int issued[BAR_COUNT];
  int observed[BAR_COUNT];
  __device__ void issue(int b) { ++issued[b]; }
  __device__ void seen(int b) { observed[b] = issued[b]; }
  __device__ void drain(uint64_t* bar) {
    for (int b = 0; b < BAR_COUNT; ++b)
      if (issued[b] > observed[b]) mbar_wait(&bar[b], (issued[b] - 1) & 1, kDrainWaitLimit);
  }
};

template <int D>
__device__ __forceinline__ void prefill_load_kv(const AttnParams& p, const CUtensorMap* map, unsigned char* dst,
                                                uint64_t* bar, const int32_t* bt, int j, int h, int fallback_pid) {
  constexpr int NH = D / 64;
  const int P = p.P;
  const int BR = P < kTileN ? P : kTileN;  // rows of one box: a page, or a 64-key part of a larger page
  mbar_arrive_expect_tx(bar, static_cast<uint32_t>(kTileN * D * 2));
  for (int k = 0; k < kTileN / BR; ++k) {
    const int t = j * kTileN + k * BR;  // first key of the box
    const int jp = t / P;               // logical page
    int pid = jp < p.max_blocks ? __ldg(bt + jp) : -1;
    if (pid < 0 || pid >= p.num_pages) pid = fallback_pid;  // keys past the sequence: masked / zeroed later
    const int y = (pid * p.Hkv + h) * P + t % P;
#pragma unroll
    for (int half = 0; half < NH; ++half)
      tc::tma_load_2d(dst + half * PrefillSmem<D>::KH + k * BR * 128, map, half * 64, y, bar);
  }
}

template <int D, int G>
__device__ __forceinline__ void prefill_tile(const AttnParams& p, int cta, unsigned char* smem_raw) {
  using S = PrefillSmem<D>;
  constexpr int NH = S::NH;
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* Ks = sm + S::K_OFF;
  unsigned char* Vs = sm + S::V_OFF;  // buffer b at Vs + b * TILE
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + S::BAR_OFF);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + S::BAR_OFF + 64);
  int32_t* flag = reinterpret_cast<int32_t*>(sm + S::BAR_OFF + 72);
  int32_t* last_flag = reinterpret_cast<int32_t*>(sm + S::BAR_OFF + 76);

  int c = 0;
  while (c + 1 < p.n_chunks && cta >= p.chunk_cta_begin[c + 1]) ++c;
  const int local = cta - p.chunk_cta_begin[c];
  const int h = local % p.Hkv;
  const int split = (local / p.Hkv) % p.tile_splits;  // which 256-key range of the tile
  const int R = p.tile_rows;
  const int rb = p.chunk_begin[c];
  const int C = p.chunk_end[c] - rb;
  const int n_mt = (C + R - 1) / R;
  const int mt = n_mt - 1 - local / (p.Hkv * p.tile_splits);  // the tiles with the most keys start first
  const int t0 = mt * R;
  const int rows_here = min(R, C - t0);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int seq = __ldg(p.seq_ids + rb);
  const int p0 = __ldg(p.positions + rb);
  const int p_last = p0 + C - 1;
  const int p_max = p0 + t0 + rows_here - 1;
  const bool geom_ok = seq >= 0 && seq < p.num_seqs && p0 >= 0 && p_last < p.max_blocks * p.P;
  const int32_t* bt = p.block_tables + static_cast<size_t>(geom_ok ? seq : 0) * p.max_blocks;
  // key tiles of this CTA: [j_begin, j_end) of the tile's 0 .. p_max / kTileN
  constexpr int kTilesPerSplit = kTileSplitKeys / kTileN;
  const int nk_all = p_max / kTileN + 1;
  const int nsplit = (nk_all + kTilesPerSplit - 1) / kTilesPerSplit;
  if ((geom_ok && split >= nsplit) || (!geom_ok && split > 0)) {
    // the tile needs fewer splits than the launch has (or a bad chunk is
    // reported once per tile): nothing to do, and no tensor memory to take
    if (warp == 0) tc::tmem_relinquish();
    return;
  }
  const int j_begin = split * kTilesPerSplit;

  // allocate tensor memory first: until it has, this CTA keeps others off the SM
  if (warp == 0) tc::tmem_alloc(tslot, kTmemCols);
  if (tid == 0) {
    for (int i = 0; i < BAR_COUNT; ++i) mbar_init(&bar[i], 1);  // nothing ever arrives on BAR_STALL
    *flag = geom_ok ? 0 : 1;
    fence_barrier_init();
  }
  __syncthreads();
  // the tile's rows must be consecutive positions of one sequence; the pages its
  // keys need must be in range
  bool bad = !geom_ok;
  if (geom_ok) {
    for (int r = tid; r < rows_here; r += kTileM)
      bad |= __ldg(p.seq_ids + rb + t0 + r) != seq || __ldg(p.positions + rb + t0 + r) != p0 + t0 + r;
    for (int jp = tid; jp <= p_max / p.P; jp += kTileM) {
      const int pid = __ldg(bt + jp);
      bad |= pid < 0 || pid >= p.num_pages;
    }
  }
  if (bad) *flag = 1;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = *tslot;
  const bool run = *flag == 0;
  if (!run && tid == 0) record_error(p.status, ST_OUT_OF_RANGE);
  const int nk = run ? min(nk_all - j_begin, kTilesPerSplit) : 0;  // key tiles of this CTA
  const int fallback_pid = run ? __ldg(bt) : 0;

  // row m of the tile: chunk position t0 + m / G, query head h * G + m % G
  const int m = tid;
  const int r_local = m / G, g = m % G;
  const bool row_valid = m < R * G && r_local < rows_here;
  const int my_pos = p0 + t0 + min(r_local, rows_here - 1);
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const size_t row_off = (static_cast<size_t>(rb + t0 + min(r_local, rows_here - 1)) * p.Hq + h * G + g) * D;

  // Q row -> TMEM columns [kColQ, kColQ + D/2), two bf16 per column; all loads first
  {
    uint32_t w[D / 2];
    if (run && row_valid) {
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.q) + row_off);
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        const uint4 v = __ldg(src + i);
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < D / 2; ++i) w[i] = 0u;
    }
#pragma unroll
    for (int c16 = 0; c16 < D / 32; ++c16) tc::tmem_st16(tb + lane_base + kColQ + c16 * 16, *reinterpret_cast<uint32_t(*)[16]>(&w[16 * c16]));
  }
  tc::tmem_wait_st();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  constexpr uint32_t id_qk = tc::idesc_bf16_f32(kTileM, kTileN, false);
  constexpr uint32_t id_pv = tc::idesc_bf16_f32(kTileM, D, true);
  PrefillIssueLog log = {};
  griddep_wait();  // the chunk's own rows, appended by a preceding dependent-launch append, are visible from here
  if (tid == 0 && nk > 0) {
    prefill_load_kv<D>(p, &p.kmap, Ks, &bar[BAR_K], bt, j_begin, h, fallback_pid);
    log.issue(BAR_K);
    prefill_load_kv<D>(p, &p.vmap, Vs, &bar[BAR_V0], bt, j_begin, h, fallback_pid);
    log.issue(BAR_V0);
    if (nk > 1) {
      prefill_load_kv<D>(p, &p.vmap, Vs + S::TILE, &bar[BAR_V1], bt, j_begin + 1, h, fallback_pid);
      log.issue(BAR_V1);
    }
  }
  float m_ref = -INFINITY, l_run = 0.0f;
  bool ok = !(p.debug_stall && nk > 0) || mbar_wait(&bar[BAR_STALL], 0, p.wait_limit);  // the stall runs out
  ok = __syncthreads_and(ok);
  for (int j = 0; j < nk && ok; ++j) {
    const int vb = j & 1;  // value buffer of this tile
    if (j > 0) {
      // P.V of the previous tile is done: P's columns, O and its value buffer are free
      if (!(ok = __syncthreads_and(mbar_wait(&bar[BAR_O], (j - 1) & 1, p.wait_limit)))) break;
      tc::fence_after_sync();
      if (tid == 0) {
        log.seen(BAR_O);
        if (j + 1 < nk) {
          const int nb = (j + 1) & 1;
          prefill_load_kv<D>(p, &p.vmap, Vs + nb * S::TILE, &bar[BAR_V0 + nb], bt, j_begin + j + 1, h, fallback_pid);
          log.issue(BAR_V0 + nb);
        }
      }
    }
    // ---- S = Q K^T
    if (!(ok = __syncthreads_and(mbar_wait(&bar[BAR_K], j & 1, p.wait_limit)))) break;
    if (tid == 0) {
      log.seen(BAR_K);
      tc::fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const unsigned char* b = Ks + (kk / 4) * S::KH + (kk % 4) * 32;
        tc::mma_bf16_ts(tb + kColSP, tb + kColQ + kk * 8, tc::smem_desc(b, 16, 1024), id_qk, kk > 0);
      }
      tc::mma_commit(&bar[BAR_S]);
      log.issue(BAR_S);
    }
    if (!(ok = __syncthreads_and(mbar_wait(&bar[BAR_S], j & 1, p.wait_limit)))) break;
    tc::fence_after_sync();
    if (tid == 0) {
      log.seen(BAR_S);
      if (j + 1 < nk) {  // the K tile is free once S is done
        prefill_load_kv<D>(p, &p.kmap, Ks, &bar[BAR_K], bt, j_begin + j + 1, h, fallback_pid);
        log.issue(BAR_K);
      }
    }
    // ---- online softmax of this row's 64 scores (log2 domain)
    float s[kTileN];
    tc::tmem_ld32(tb + lane_base + kColSP, *reinterpret_cast<float(*)[32]>(&s[0]));
    tc::tmem_ld32(tb + lane_base + kColSP + 32, *reinterpret_cast<float(*)[32]>(&s[32]));
    const int key0 = (j_begin + j) * kTileN;
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kTileN; ++i) {
      s[i] = (key0 + i <= my_pos) ? __fmul_rn(s[i], p.sm_scale_log2) : -INFINITY;
      mx = fmaxf(mx, s[i]);
    }
    float alpha = 1.0f;
    if (mx > __fadd_rn(m_ref, kRescaleSlack)) {
      alpha = ex2(__fsub_rn(m_ref, mx));
      m_ref = mx;
      l_run = __fmul_rn(l_run, alpha);
    }
    // weights -> (hi, lo) bf16 pairs in place of S: hi in [0, 32), lo in [32, 64)
    float lsum = 0.0f;
#pragma unroll
    for (int q16 = 0; q16 < kTileN / 16; ++q16) {
      uint32_t hw[8], lw[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float a = s[16 * q16 + 2 * i] == -INFINITY ? 0.0f : ex2(__fsub_rn(s[16 * q16 + 2 * i], m_ref));
        const float b = s[16 * q16 + 2 * i + 1] == -INFINITY ? 0.0f : ex2(__fsub_rn(s[16 * q16 + 2 * i + 1], m_ref));
        lsum = __fadd_rn(__fadd_rn(lsum, a), b);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(a, b);
        const __nv_bfloat162 lo = __floats2bfloat162_rn(__fsub_rn(a, __low2float(hi)), __fsub_rn(b, __high2float(hi)));
        hw[i] = *reinterpret_cast<const uint32_t*>(&hi);
        lw[i] = *reinterpret_cast<const uint32_t*>(&lo);
      }
      tc::tmem_st8(tb + lane_base + kColSP + q16 * 8, hw);
      tc::tmem_st8(tb + lane_base + kColSP + 32 + q16 * 8, lw);
    }
    l_run = __fadd_rn(l_run, lsum);
    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {  // the reference max moved: rescale O
#pragma unroll 1
      for (int c4 = 0; c4 < D / 32; ++c4) {
        float o[32];
        tc::tmem_ld32(tb + lane_base + kColO + c4 * 32, o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __fmul_rn(o[i], alpha);
        tc::tmem_st32(tb + lane_base + kColO + c4 * 32, o);
      }
    }
    tc::tmem_wait_st();
    // ---- value tile: keys past the chunk's last position may hold stale or
    // poisoned values; zero those rows so that 0-weights never meet a NaN
    if (!(ok = __syncthreads_and(mbar_wait(&bar[BAR_V0 + vb], (j >> 1) & 1, p.wait_limit)))) break;
    if (key0 + kTileN - 1 > p_last) {
      unsigned char* V = Vs + vb * S::TILE;
      const int first = max(0, p_last + 1 - key0);
      const int n16 = (kTileN - first) * NH * 8;  // 16-byte pieces to clear
      for (int i = tid; i < n16; i += kTileM) {
        const int row = first + i / (NH * 8), piece = i % (NH * 8);
        *reinterpret_cast<uint4*>(V + (piece / 8) * S::KH + row * 128 + (piece % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      tc::fence_proxy_async_smem();
    }
    tc::fence_before_sync();
    __syncthreads();
    // ---- O += P V
    if (tid == 0) {
      log.seen(BAR_V0 + vb);
      tc::fence_after_sync();
      const unsigned char* V = Vs + vb * S::TILE;
#pragma unroll
      for (int kk = 0; kk < kTileN / 16; ++kk) {
        const uint64_t b = tc::smem_desc(V + kk * 2048, S::KH, 1024);  // 16 keys of the MN-major value tile
        tc::mma_bf16_ts(tb + kColO, tb + kColSP + kk * 8, b, id_pv, j > 0 || kk > 0);
        tc::mma_bf16_ts(tb + kColO, tb + kColSP + 32 + kk * 8, b, id_pv, true);
      }
      tc::mma_commit(&bar[BAR_O]);
      log.issue(BAR_O);
    }
  }
  if (ok && nk > 0) ok = __syncthreads_and(mbar_wait(&bar[BAR_O], (nk - 1) & 1, p.wait_limit));
  if (!ok && tid == 0) {
    record_error(p.status, ST_TIMEOUT);
    log.drain(bar);  // every copy and MMA in flight finishes before TMEM or shared memory is reused
  }
  __syncthreads();
  if (nk > 0) {
    tc::fence_after_sync();
    if (nsplit == 1) {
      if (ok) {
        const float inv = __fdiv_rn(1.0f, l_run);
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + row_off;
#pragma unroll 1
        for (int c4 = 0; c4 < D / 32; ++c4) {
          float o[32];
          tc::tmem_ld32(tb + lane_base + kColO + c4 * 32, o);
          if (row_valid) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t w[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const __nv_bfloat162 pr =
                    __floats2bfloat162_rn(__fmul_rn(o[8 * i + 2 * k], inv), __fmul_rn(o[8 * i + 2 * k + 1], inv));
                w[k] = *reinterpret_cast<const uint32_t*>(&pr);
              }
              *reinterpret_cast<uint4*>(orow + c4 * 32 + 8 * i) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
    } else {
      // publish this key range's partial (max, sum, unnormalised O) -- an empty
      // one after a failure, so that the counters still return to zero -- and
      // let the last of the tile's CTAs merge the ranges in ascending order
      const size_t slot0 = (static_cast<size_t>(p.chunk_row_begin[c] + t0 + min(r_local, rows_here - 1)) * p.Hq +
                            h * G + g) * p.tile_splits;
      const size_t slot = slot0 + split;
#pragma unroll 1
      for (int c4 = 0; c4 < D / 32; ++c4) {
        float o[32];
        if (ok) {
          tc::tmem_ld32(tb + lane_base + kColO + c4 * 32, o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0.0f;
        }
        if (row_valid) {
          float4* dst = reinterpret_cast<float4*>(p.ws_tile_o + slot * D + c4 * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        }
      }
      if (row_valid) {
        p.ws_tile_ml[slot * 2] = ok ? m_ref : -INFINITY;
        p.ws_tile_ml[slot * 2 + 1] = ok ? l_run : 0.0f;
      }
      __threadfence();
      __syncthreads();
      int32_t* counter = p.ws_tile_count + p.chunk_tile_begin[c] + mt * p.Hkv + h;
      if (tid == 0) *last_flag = atomicAdd(counter, 1) == nsplit - 1;
      __syncthreads();
      if (*last_flag) {
        __threadfence();
        // Merge in ascending key-range order.  Each row's weights f[row][sp] and
        // 1 / sum go to shared memory (the K/V buffers are free now); then all
        // threads sweep the rows together, one head element each, so the loads
        // of the partial accumulators are coalesced and independent.
        float* ftab = reinterpret_cast<float*>(sm);  // [kTileM][nsplit], then [kTileM] inverse sums
        const bool fits = (kTileM * (nsplit + 1)) * 4 <= S::BAR_OFF;
        if (fits) {
          float M = -INFINITY;
          for (int sp = 0; sp < nsplit; ++sp) {
            const float mv = row_valid ? __ldcg(p.ws_tile_ml + (slot0 + sp) * 2) : 0.0f;
            ftab[m * nsplit + sp] = mv;
            M = fmaxf(M, mv);
          }
          float lsum = 0.0f;
          for (int sp = 0; sp < nsplit; ++sp) {
            const float f = ex2(__fsub_rn(ftab[m * nsplit + sp], M));
            ftab[m * nsplit + sp] = f;
            lsum = fmaf(f, row_valid ? __ldcg(p.ws_tile_ml + (slot0 + sp) * 2 + 1) : 1.0f, lsum);
          }
          ftab[kTileM * nsplit + m] = __fdiv_rn(1.0f, lsum);
          __syncthreads();
          // thread t: head element t % D of rows t / D, t / D + 4 * (128 / D) ...: four rows
          // and four key ranges of loads in flight at a time
          constexpr int RPI = kTileM / D;  // rows per sweep step (1 for D = 128, 2 for D = 64)
          const int d = tid % D;
#pragma unroll 1
          for (int r0 = tid / D; r0 < kTileM; r0 += 4 * RPI) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            const float* o[4];
            bool use[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int rr = r0 + u * RPI;
              const int rl = rr / G, gg = rr % G;
              use[u] = rr < kTileM && rr < R * G && rl < rows_here;
              const size_t s0 = (static_cast<size_t>(p.chunk_row_begin[c] + t0 + (use[u] ? rl : 0)) * p.Hq + h * G + gg) *
                                p.tile_splits;
              o[u] = p.ws_tile_o + s0 * D + d;
            }
#pragma unroll 2
            for (int sp = 0; sp < nsplit; ++sp)
#pragma unroll
              for (int u = 0; u < 4; ++u)
                if (use[u]) acc[u] = fmaf(ftab[(r0 + u * RPI) * nsplit + sp], __ldcg(o[u] + static_cast<size_t>(sp) * D), acc[u]);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (!use[u]) continue;
              const int rr = r0 + u * RPI, rl = rr / G, gg = rr % G;
              reinterpret_cast<__nv_bfloat16*>(p.out)[(static_cast<size_t>(rb + t0 + rl) * p.Hq + h * G + gg) * D + d] =
                  __float2bfloat16_rn(__fmul_rn(acc[u], ftab[kTileM * nsplit + rr]));
            }
          }
        } else if (row_valid) {
          float M = -INFINITY;
          for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, __ldcg(p.ws_tile_ml + (slot0 + sp) * 2));
          float lsum = 0.0f;
          for (int sp = 0; sp < nsplit; ++sp)
            lsum = fmaf(ex2(__fsub_rn(__ldcg(p.ws_tile_ml + (slot0 + sp) * 2), M)),
                        __ldcg(p.ws_tile_ml + (slot0 + sp) * 2 + 1), lsum);
          const float inv = __fdiv_rn(1.0f, lsum);
          __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + row_off;
          for (int d = 0; d < D; ++d) {
            float acc = 0.0f;
            for (int sp = 0; sp < nsplit; ++sp)
              acc = fmaf(ex2(__fsub_rn(__ldcg(p.ws_tile_ml + (slot0 + sp) * 2), M)),
                         __ldcg(p.ws_tile_o + (slot0 + sp) * D + d), acc);
            orow[d] = __float2bfloat16_rn(__fmul_rn(acc, inv));
          }
        }
        if (tid == 0) *counter = 0;  // leave the workspace zero-filled for the next call
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tb, kTmemCols);
  }
}

}  // namespace pa
