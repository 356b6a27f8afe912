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
// launch without lowering the decode occupancy.  Shared memory holds two key
// tiles and one value tile (128-byte swizzled, loaded by 2-D tensor-map copies
// of one page x 64 head elements each; no multicast) and the page ids of the
// CTA's key range, read from the block table once.  Tensor memory (256
// columns, so that two tile CTAs share an SM and one's softmax overlaps the
// other's MMAs) holds S of the current key tile, then P of it in place, Q and
// O.  Thread m owns TMEM lane m = tile row m; thread 0 alone issues copies and
// MMAs.  Schedule of key tile j: P.V(j-1) done -> V(j) into the value buffer,
// S(j) issued (K(j) landed a key tile earlier) -> S(j) done: its key buffer
// takes K(j+2) -> softmax, one read of the 64 scores from tensor memory ->
// P.V(j).  A tile's key range is split across CTAs in fixed pieces of
// kTileSplitKeys keys, merged in ascending order.  Every barrier has at most
// one phase outstanding; every wait is bounded.
//
// Precision: the scores and the softmax are FP32.  Each weight p enters the
// P.V product as hi = bf16(p) and lo = bf16(p - hi), so the product sees p to
// about 16 significant bits; the tensor core accumulates in FP32 and l sums
// the FP32 weights (a fixed tree of eight partial sums per key tile).
#pragma once

#include "pa_device.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

constexpr int kTileM = 128;  // rows per tile (TMEM lanes)
constexpr int kTileN = 64;   // keys per key tile

constexpr int kTilePids = kTileSplitKeys / 16 + 1;  // page ids of one CTA's key range (pages >= 16 tokens)

template <int D>
struct PrefillSmem {  // byte offsets from a 1024-byte aligned base
  static constexpr int NH = D / 64;        // 64-element halves of the head dim
  static constexpr int KH = kTileN * 128;  // one half of a K or V tile: 8 KiB
  static constexpr int TILE = NH * KH;     // one K or V tile
  static constexpr int K_OFF = 0;          // two key tiles
  static constexpr int V_OFF = K_OFF + 2 * TILE;
  static constexpr int BAR_OFF = V_OFF + TILE;
  static constexpr int PID_OFF = BAR_OFF + 128;
  static constexpr int TOTAL = PID_OFF + ((kTilePids * 4 + 15) / 16) * 16;
  static constexpr int BYTES = TOTAL + 1024;  // slack for aligning the base
};

enum {
  BAR_K0 = 0,   // key buffer 0 / 1 landed
  BAR_K1 = 1,
  BAR_V = 2,    // value tile landed
  BAR_S = 3,    // S of the current key tile done
  BAR_O = 4,    // P.V of a key tile done
  BAR_STALL = 5,
  BAR_COUNT = 6
};

// TMEM columns: S of the current key tile in [0, 64), then P of it in place
// (keys 32h .. 32h+31: hi in columns 32h .. 32h+15, lo in the 16 after them);
// Q in [64, 64 + D/2); O in [128, 128 + D).  256 columns: two tile CTAs fit on
// an SM, so that one's softmax runs while the other's MMAs do.
template <int D>
struct PrefillTmem {
  static constexpr uint32_t S = 0;
  static constexpr uint32_t Q = 64;
  static constexpr uint32_t O = 128;
  static constexpr uint32_t COLS = 256;  // a power of two
  static_assert(O >= Q + D / 2 && O + D <= COLS, "tensor memory columns overlap");
};

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

// Key tile j (keys 64j .. 64j+63) of kv head h into a tile buffer: one box of
// min(P, 64) keys x 64 head elements per page piece and head-dim half.  Page
// ids come from the CTA's table in shared memory (pids[jp - jp0]); keys past
// the sequence read a valid page instead (masked or zeroed later).
template <int D>
__device__ __forceinline__ void prefill_load_kv(const AttnParams& p, const CUtensorMap* map, unsigned char* dst,
                                                uint64_t* bar, const int32_t* pids, int jp0, int j, int h,
                                                int fallback_pid) {
  constexpr int NH = D / 64;
  const int P = p.P;
  const int BR = P < kTileN ? P : kTileN;  // rows of one box: a page, or a 64-key part of a larger page
  mbar_arrive_expect_tx(bar, static_cast<uint32_t>(kTileN * D * 2));
  for (int k = 0; k < kTileN / BR; ++k) {
    const int t = j * kTileN + k * BR;  // first key of the box
    int pid = pids[t / P - jp0];
    if (pid < 0 || pid >= p.num_pages) pid = fallback_pid;
    const int y = (pid * p.Hkv + h) * P + t % P;
#pragma unroll
    for (int half = 0; half < NH; ++half)
      tc::tma_load_2d(dst + half * PrefillSmem<D>::KH + k * BR * 128, map, half * 64, y, bar);
  }
}

template <int D, int G>
__device__ __forceinline__ void prefill_tile(const AttnParams& p, int cta, unsigned char* smem_raw) {
  using S = PrefillSmem<D>;
  using T = PrefillTmem<D>;
  constexpr int NH = S::NH;
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* Ks = sm + S::K_OFF;  // key buffer b at Ks + b * TILE
  unsigned char* Vs = sm + S::V_OFF;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + S::BAR_OFF);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + S::BAR_OFF + 64);
  int32_t* last_flag = reinterpret_cast<int32_t*>(sm + S::BAR_OFF + 72);
  int32_t* pids = reinterpret_cast<int32_t*>(sm + S::PID_OFF);

  int c = 0;
  while (c + 1 < p.n_chunks && cta >= p.chunk_cta_begin[c + 1]) ++c;
  const int local = cta - p.chunk_cta_begin[c];
  const int h = local % p.Hkv;
  const int split = (local / p.Hkv) % p.tile_splits;  // which key range of the tile
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
  // key tiles of this CTA: [j_begin, j_begin + nk) of the tile's 0 .. p_max / kTileN
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
  const int nk_cta = min(nk_all - j_begin, kTilesPerSplit);
  const int jp0 = j_begin * kTileN / p.P;                       // first page of the CTA's keys
  const int jp_last = ((j_begin + nk_cta) * kTileN - 1) / p.P;  // last page its key tiles touch

  // row m of the tile: chunk position t0 + m / G, query head h * G + m % G
  const int m = tid;
  const int r_local = m / G, g = m % G;
  const bool row_valid = m < R * G && r_local < rows_here;
  const int my_pos = p0 + t0 + min(r_local, rows_here - 1);
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const size_t row_off = (static_cast<size_t>(rb + t0 + min(r_local, rows_here - 1)) * p.Hq + h * G + g) * D;

  // allocate tensor memory first: until it has, this CTA keeps others off the SM
  if (warp == 0) tc::tmem_alloc(tslot, T::COLS);
  if (tid == 0) {
    for (int i = 0; i < BAR_COUNT; ++i) mbar_init(&bar[i], 1);  // nothing ever arrives on BAR_STALL
    fence_barrier_init();
  }
  // the Q row (the query is the caller's input: no dependence on a preceding
  // append), then the checks: the tile's rows must be consecutive positions of
  // one sequence, the pages its keys need in range; the CTA's page ids go to
  // shared memory
  uint32_t w[D / 2];
  if (row_valid) {
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
  bool bad = !geom_ok;
  if (geom_ok) {
    for (int r = tid; r < rows_here; r += kTileM)
      bad |= __ldg(p.seq_ids + rb + t0 + r) != seq || __ldg(p.positions + rb + t0 + r) != p0 + t0 + r;
    const int jp_check = p_max / p.P;
    for (int jp = tid; jp <= max(jp_check, jp_last); jp += kTileM) {
      const int pid = jp < p.max_blocks ? __ldg(bt + jp) : -1;
      if (jp <= jp_check) bad |= pid < 0 || pid >= p.num_pages;
      if (jp >= jp0 && jp <= jp_last) pids[jp - jp0] = pid;
    }
  }
  tc::fence_before_sync();
  bad = __syncthreads_or(bad);
  tc::fence_after_sync();
  const uint32_t tb = *tslot;
  const bool run = !bad;
  if (!run && tid == 0) record_error(p.status, ST_OUT_OF_RANGE);
  const int nk = run ? nk_cta : 0;  // key tiles of this CTA
  const int fallback_pid = run ? pids[0] : 0;

  PrefillIssueLog log = {};
  griddep_wait();  // the chunk's own rows, appended by a preceding dependent-launch append, are visible from here
  if (tid == 0 && nk > 0) {
    prefill_load_kv<D>(p, &p.kmap, Ks, &bar[BAR_K0], pids, jp0, j_begin, h, fallback_pid);
    log.issue(BAR_K0);
    prefill_load_kv<D>(p, &p.vmap, Vs, &bar[BAR_V], pids, jp0, j_begin, h, fallback_pid);
    log.issue(BAR_V);
    if (nk > 1) {
      prefill_load_kv<D>(p, &p.kmap, Ks + S::TILE, &bar[BAR_K1], pids, jp0, j_begin + 1, h, fallback_pid);
      log.issue(BAR_K1);
    }
  }
  // Q row -> TMEM columns [T::Q, T::Q + D/2), two bf16 per column
#pragma unroll
  for (int c16 = 0; c16 < D / 32; ++c16) tc::tmem_st16(tb + lane_base + T::Q + c16 * 16, *reinterpret_cast<uint32_t(*)[16]>(&w[16 * c16]));
  tc::tmem_wait_st();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  constexpr uint32_t id_qk = tc::idesc_bf16_f32(kTileM, kTileN, false);
  constexpr uint32_t id_pv = tc::idesc_bf16_f32(kTileM, D, true);
  // S(j) = Q K(j)^T into the S columns from key buffer j % 2 (thread 0; K(j) has landed)
  auto issue_qk = [&](int j) {
    const unsigned char* K = Ks + (j & 1) * S::TILE;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const unsigned char* kb = K + (kk / 4) * S::KH + (kk % 4) * 32;
      tc::mma_bf16_ts(tb + T::S, tb + T::Q + kk * 8, tc::smem_desc(kb, 16, 1024), id_qk, kk > 0);
    }
    tc::mma_commit(&bar[BAR_S]);
  };
  // O += P(j) V(j), P as (hi, lo) from the S columns
  auto issue_pv = [&](int j) {
#pragma unroll
    for (int kk = 0; kk < kTileN / 16; ++kk) {
      const uint64_t vb = tc::smem_desc(Vs + kk * 2048, S::KH, 1024);  // 16 keys of the MN-major value tile
      const uint32_t ph = tb + T::S + (kk / 2) * 32 + (kk % 2) * 8;   // hi of keys 16kk .. 16kk+15; lo 16 columns on
      tc::mma_bf16_ts(tb + T::O, ph, vb, id_pv, j > 0 || kk > 0);
      tc::mma_bf16_ts(tb + T::O, ph + 16, vb, id_pv, true);
    }
    tc::mma_commit(&bar[BAR_O]);
  };

  // Key tile j: P.V(j-1) done (it has left the S columns and the value buffer)
  // -> V(j) into the value buffer, S(j) -> softmax -> P.V(j).  Every barrier has
  // at most one phase outstanding; every wait is bounded.
  float m_ref = -INFINITY, l_run = 0.0f;
  bool ok = !(p.debug_stall && nk > 0) || mbar_wait(&bar[BAR_STALL], 0, p.wait_limit);  // the stall runs out
  // thread 0's own waits; a failure there reaches the others through the next
  // collective wait (theirs then runs out too: bounded)
  bool issuer_ok = true;
  const uint32_t col_s = tb + lane_base + T::S;
  for (int j = 0; j < nk && ok; ++j) {
    if (tid == 0 && issuer_ok) {
      if (j > 0) {
        issuer_ok = mbar_wait(&bar[BAR_O], (j - 1) & 1, p.wait_limit);
        if (issuer_ok) {
          log.seen(BAR_O);
          prefill_load_kv<D>(p, &p.vmap, Vs, &bar[BAR_V], pids, jp0, j_begin + j, h, fallback_pid);
          log.issue(BAR_V);
        }
      }
      if (issuer_ok) issuer_ok = mbar_wait(&bar[BAR_K0 + (j & 1)], (j >> 1) & 1, p.wait_limit);
      if (issuer_ok) {
        log.seen(BAR_K0 + (j & 1));
        tc::fence_after_sync();
        issue_qk(j);
        log.issue(BAR_S);
      }
    }
    // ---- S(j) done
    if (!(ok = __syncthreads_and(issuer_ok && mbar_wait(&bar[BAR_S], j & 1, p.wait_limit)))) break;
    tc::fence_after_sync();
    if (tid == 0) {
      log.seen(BAR_S);
      if (j + 2 < nk) {  // S(j) has read key buffer j % 2: refill it
        prefill_load_kv<D>(p, &p.kmap, Ks + (j & 1) * S::TILE, &bar[BAR_K0 + (j & 1)], pids, jp0, j_begin + j + 2, h,
                           fallback_pid);
        log.issue(BAR_K0 + (j & 1));
      }
    }
    // ---- online softmax of this row's 64 scores (log2 domain), in two halves of
    // 32 read from tensor memory twice (for the maximum, then for the weights),
    // so that no more than 32 scores are live in registers
    const int key0 = (j_begin + j) * kTileN;
    const bool edge = key0 + kTileN - 1 > my_pos;  // the row's causal edge (or keys past the chunk) is in this tile
    float mx = -INFINITY;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      float sc[32];
      tc::tmem_ld32(col_s + 32 * half, sc);
      if (edge) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (key0 + 32 * half + i > my_pos) sc[i] = -INFINITY;
      }
      float mx4[4] = {sc[0], sc[1], sc[2], sc[3]};
#pragma unroll
      for (int i = 4; i < 32; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], sc[i]);
      mx = fmaxf(mx, fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])));
    }
    mx = __fmul_rn(mx, p.sm_scale_log2);  // the scale is positive: the largest scaled score is the scaled largest one
    float alpha = 1.0f;
    if (mx > __fadd_rn(m_ref, kRescaleSlack)) {
      alpha = ex2(__fsub_rn(m_ref, mx));
      m_ref = mx;
      l_run = __fmul_rn(l_run, alpha);
    }
    // every score so far masked: the weights are ex2(-inf) = 0 against any finite reference
    const float neg_ref = m_ref == -INFINITY ? 0.0f : -m_ref;
    // weights -> (hi, lo) bf16 pairs in place of S: keys 32h .. 32h+31 as hi
    // in columns 32h .. 32h+15 and lo in the 16 after them
    float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      float sc[32];
      tc::tmem_ld32(col_s + 32 * half, sc);
      if (edge) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (key0 + 32 * half + i > my_pos) sc[i] = -INFINITY;
      }
#pragma unroll
      for (int q8 = 0; q8 < 2; ++q8) {
        uint32_t hw[8], lw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float a = ex2(fmaf(sc[16 * q8 + 2 * i], p.sm_scale_log2, neg_ref));
          const float c = ex2(fmaf(sc[16 * q8 + 2 * i + 1], p.sm_scale_log2, neg_ref));
          ls[i] = __fadd_rn(ls[i], __fadd_rn(a, c));
          const __nv_bfloat162 hi = __floats2bfloat162_rn(a, c);
          const __nv_bfloat162 lo = __floats2bfloat162_rn(__fsub_rn(a, __low2float(hi)), __fsub_rn(c, __high2float(hi)));
          hw[i] = *reinterpret_cast<const uint32_t*>(&hi);
          lw[i] = *reinterpret_cast<const uint32_t*>(&lo);
        }
        tc::tmem_st8(col_s + 32 * half + q8 * 8, hw);
        tc::tmem_st8(col_s + 32 * half + 16 + q8 * 8, lw);
      }
    }
    const float lsum = __fadd_rn(__fadd_rn(__fadd_rn(ls[0], ls[1]), __fadd_rn(ls[2], ls[3])),
                                 __fadd_rn(__fadd_rn(ls[4], ls[5]), __fadd_rn(ls[6], ls[7])));
    l_run = __fadd_rn(l_run, lsum);
    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
      // the reference max moved: rescale O (P.V(j-1), its last writer, is done:
      // thread 0 saw it before issuing S(j); the others see it here)
      if (mbar_wait(&bar[BAR_O], (j - 1) & 1, p.wait_limit)) {
        tc::fence_after_sync();
#pragma unroll 1
        for (int c4 = 0; c4 < D / 32; ++c4) {
          float o[32];
          tc::tmem_ld32(tb + lane_base + T::O + c4 * 32, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __fmul_rn(o[i], alpha);
          tc::tmem_st32(tb + lane_base + T::O + c4 * 32, o);
        }
      } else {
        ok = false;
      }
    }
    tc::tmem_wait_st();
    // ---- value tile: keys past the chunk's last position may hold stale or
    // poisoned values; zero those rows so that 0-weights never meet a NaN
    if (!(ok = __syncthreads_and(ok && issuer_ok && mbar_wait(&bar[BAR_V], j & 1, p.wait_limit)))) break;
    if (key0 + kTileN - 1 > p_last) {
      const int first = max(0, p_last + 1 - key0);
      const int n16 = (kTileN - first) * NH * 8;  // 16-byte pieces to clear
      for (int i = tid; i < n16; i += kTileM) {
        const int row = first + i / (NH * 8), piece = i % (NH * 8);
        *reinterpret_cast<uint4*>(Vs + (piece / 8) * S::KH + row * 128 + (piece % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      tc::fence_proxy_async_smem();
    }
    tc::fence_before_sync();
    __syncthreads();
    // ---- O += P V
    if (tid == 0) {
      log.seen(BAR_V);
      tc::fence_after_sync();
      issue_pv(j);
      log.issue(BAR_O);
    }
  }
  if (ok && nk > 0) {
    // the last commit arrives when every MMA before it has completed too
    ok = __syncthreads_and(mbar_wait(&bar[BAR_O], (nk - 1) & 1, p.wait_limit));
    if (ok && tid == 0) log.seen(BAR_O);
  }
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
          tc::tmem_ld32(tb + lane_base + T::O + c4 * 32, o);
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
          tc::tmem_ld32(tb + lane_base + T::O + c4 * 32, o);
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
        // threads sweep the tile in 16-byte pieces (thread t: pieces t, t + 128,
        // ...; a row's pieces are consecutive), eight loads in flight a thread
        // (four pieces, two key ranges): the merge is bound by the loads one SM
        // keeps in flight.
        float* ftab = reinterpret_cast<float*>(sm);  // [kTileM][nsplit], then [kTileM] inverse sums
        const bool fits = (kTileM * (nsplit + 1)) * 4 <= S::BAR_OFF;
        if (fits) {
          float M = -INFINITY;
#pragma unroll 4
          for (int sp = 0; sp < nsplit; ++sp) {  // independent loads, several in flight
            const float mv = row_valid ? __ldcg(p.ws_tile_ml + (slot0 + sp) * 2) : 0.0f;
            ftab[m * nsplit + sp] = mv;
            M = fmaxf(M, mv);
          }
          float lsum = 0.0f;
#pragma unroll 4
          for (int sp = 0; sp < nsplit; ++sp) {
            const float f = ex2(__fsub_rn(ftab[m * nsplit + sp], M));
            ftab[m * nsplit + sp] = f;
            lsum = fmaf(f, row_valid ? __ldcg(p.ws_tile_ml + (slot0 + sp) * 2 + 1) : 1.0f, lsum);
          }
          ftab[kTileM * nsplit + m] = __fdiv_rn(1.0f, lsum);
          __syncthreads();
          constexpr int PPR = D / 4;  // 16-byte pieces per row
          constexpr int U = 4;        // pieces per thread per sweep step
#pragma unroll 1
          for (int q0 = tid; q0 < kTileM * PPR; q0 += kTileM * U) {
            float4 acc[U];
            const float4* src[U];
            int rr[U];
            bool use[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const int q = q0 + u * kTileM;
              rr[u] = q / PPR;
              const int rl = rr[u] / G, gg = rr[u] % G;
              use[u] = q < kTileM * PPR && rr[u] < R * G && rl < rows_here;
              const size_t s0 = (static_cast<size_t>(p.chunk_row_begin[c] + t0 + (use[u] ? rl : 0)) * p.Hq + h * G + gg) *
                                p.tile_splits;
              src[u] = reinterpret_cast<const float4*>(p.ws_tile_o + s0 * D) + q % PPR;
              acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll 2
            for (int sp = 0; sp < nsplit; ++sp) {
#pragma unroll
              for (int u = 0; u < U; ++u) {
                if (!use[u]) continue;
                const float f = ftab[rr[u] * nsplit + sp];
                const float4 v = __ldcg(src[u] + static_cast<size_t>(sp) * PPR);
                acc[u].x = fmaf(f, v.x, acc[u].x);
                acc[u].y = fmaf(f, v.y, acc[u].y);
                acc[u].z = fmaf(f, v.z, acc[u].z);
                acc[u].w = fmaf(f, v.w, acc[u].w);
              }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
              if (!use[u]) continue;
              const int q = q0 + u * kTileM, rl = rr[u] / G, gg = rr[u] % G;
              const float inv = ftab[kTileM * nsplit + rr[u]];
              const __nv_bfloat162 lo = __floats2bfloat162_rn(__fmul_rn(acc[u].x, inv), __fmul_rn(acc[u].y, inv));
              const __nv_bfloat162 hi = __floats2bfloat162_rn(__fmul_rn(acc[u].z, inv), __fmul_rn(acc[u].w, inv));
              __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + (static_cast<size_t>(rb + t0 + rl) * p.Hq + h * G + gg) * D;
              *reinterpret_cast<uint2*>(orow + (q % PPR) * 4) =
                  make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
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
    tc::tmem_dealloc(tb, T::COLS);
  }
}

}  // namespace pa
