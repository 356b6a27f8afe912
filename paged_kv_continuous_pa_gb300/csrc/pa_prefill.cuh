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
// Two CTA shapes run the same per-row arithmetic, so a chunk row's bits do
// not depend on which one ran it:
//   * in a launch that also runs decode units, the tile CTA has the decode
//     unit's shape (4 warps, about 51 KB of shared memory, at most 128
//     registers a thread) so that mixing lowers no decode occupancy.  Three
//     tile buffers form one ring that takes key and value tiles in the order
//     the MMAs read them; two S buffers let S(j+1) run while the threads turn
//     S(j) into P(j); four threads in four warps issue the copies and MMAs
//     (an MMA of these shapes holds its issuing thread ~100 cycles); the block
//     meets once per key tile, before P.V(j);
//   * in a launch of chunk tiles only, the CTA is warp-specialised: four
//     softmax warps and two issuing warps (key copies + S MMAs, value copies +
//     P.V MMAs), three S buffers and three key and three value buffers, and
//     the roles synchronise through mbarriers only.
// Tiles are 2-D tensor-map copies of one page x 64 head elements (128-byte
// swizzle, no multicast), the tensor-map row of each page of the CTA's key
// range computed once from the block table.  TMEM (512 columns) holds the S
// buffers (P in place), Q and O; thread m owns TMEM lane m = tile row m.  A
// tile's key range is split across CTAs in fixed pieces of kTileSplitKeys
// keys, merged in ascending order by the last CTA of the tile.  Every barrier
// has at most one phase outstanding; every wait is bounded.
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

template <int D, int SLOTS_>
struct PrefillSmem {  // byte offsets from a 1024-byte aligned base
  static constexpr int NH = D / 64;        // 64-element halves of the head dim
  static constexpr int KH = kTileN * 128;  // one half of a K or V tile: 8 KiB
  static constexpr int TILE = NH * KH;     // one K or V tile
  static constexpr int SLOTS = SLOTS_;     // key / value tile buffers, from offset 0
  static constexpr int BAR_OFF = SLOTS * TILE;  // barriers and small state (256 bytes), then the page rows
  static constexpr int TSLOT_OFF = BAR_OFF + 248;  // the TMEM base address
  static constexpr int LAST_OFF = BAR_OFF + 252;   // this CTA merges the tile's key ranges
  static constexpr int PID_OFF = BAR_OFF + 256;
  static constexpr int TOTAL = PID_OFF + ((kTilePids * 4 + 15) / 16) * 16;
  static constexpr int BYTES = TOTAL + 1024;  // slack for aligning the base
};

// The shared-memory layout of each tile CTA shape (its launcher sizes the
// dynamic shared memory from the same definition)
template <int D, bool WS>
using PrefillLayout = PrefillSmem<D, WS ? 6 : 3>;

// Barriers of the tile CTA that shares the decode CTA's shape (mixed launch)
enum {
  BAR_R0 = 0,     // ring slot 0 / 1 / 2 landed (a key or a value tile)
  BAR_S0 = 3,     // S of S buffer 0 / 1 done
  BAR_O = 5,      // P.V of a key tile done
  BAR_STALL = 6,
  BAR_COUNT = 7,
  BAR_M0 = 7,     // split merge: partial block landed in tile buffer 0 / 1 / 2
  BAR_ALL = 10    // barriers initialised (the merge's are not in the issue log)
};
// ... and of the warp-specialised tile CTA (a launch of chunk tiles only)
enum {
  WS_KF0 = 0,     // key buffer 0 / 1 / 2 landed
  WS_VF0 = 3,     // value buffer 0 / 1 / 2 landed
  WS_SD0 = 6,     // S of S buffer 0 / 1 / 2 done
  WS_PR0 = 9,     // P of S buffer 0 / 1 / 2 written (one arrival per row)
  WS_OD0 = 12,    // P.V of key tile j done, j % 3 = 0 / 1 / 2
  WS_STALL = 15,
  WS_COUNT = 16,
  WS_M0 = 16,     // split merge, as above
  WS_ALL = 19
};
constexpr int kMergeSlots = 3;

// TMEM columns: SB S buffers, S(j) in buffer j % SB = [64 b, 64 b + 64), then
// P(j) in place (keys 32h .. 32h+31: hi in columns 32h .. 32h+15, lo in the 16
// after them); Q in [64 SB, 64 SB + D/2); O in [256, 256 + D).  With two S
// buffers (the decode-shaped CTA) S(j+1) runs on the tensor cores while the
// threads turn S(j) into P(j); the warp-specialised CTA keeps three, so that
// S(j+1) waits only for P.V(j-2).
template <int D, int SB>
struct PrefillTmem {
  static constexpr uint32_t S = 0;  // S buffer b at S + 64 b
  static constexpr uint32_t Q = SB * kTileN;
  static constexpr uint32_t O = 256;
  static constexpr uint32_t COLS = 512;  // a power of two
  static_assert(O >= Q + D / 2 && O + D <= COLS, "tensor memory columns overlap");
};

// A role thread's record of the copies and MMAs it issued on each barrier, in
// two bit masks (registers, not local memory): a phase outstanding, and the
// parity of the last phase issued.  A barrier never has more than one phase
// outstanding, so after a failure each pending operation is drained by
// waiting for the parity of its own phase.
struct PrefillIssueLog {
  uint32_t pending = 0u, parity = 0u;
  __device__ void issue(int b) {
    parity ^= 1u << b;
    pending |= 1u << b;
  }
  __device__ void seen(int b) { pending &= ~(1u << b); }
  __device__ void drain(uint64_t* bar, int count) {
    for (int b = 0; b < count; ++b)
      if ((pending >> b) & 1u) mbar_wait(&bar[b], ((parity >> b) & 1u) ^ 1u, kDrainWaitLimit);
  }
};

// Key tile j (keys 64j .. 64j+63) into a tile buffer: one box of min(P, 64)
// keys x 64 head elements per page piece and head-dim half.  ybase[jp - jp0]
// is the tensor-map row of page jp's first slot for this kv head (built once
// from the block table; a page past the sequence has a valid page's row:
// masked or zeroed later).  P = 2^lg_p.  Called by all lanes of one warp:
// lane 0 posts the byte count, then lane l issues box l (2 to 8 boxes), so a
// tile's copies cost the warp about one copy's issue time.
template <int D>
__device__ __forceinline__ void prefill_load_kv(const CUtensorMap* map, unsigned char* dst, uint64_t* bar,
                                                const int32_t* ybase, int jp0, int j, int lg_p, int lane) {
  constexpr int NH = D / 64;
  const int lg_br = lg_p < 6 ? lg_p : 6;  // rows of one box: a page, or a 64-key part of a larger page
  if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(kTileN * D * 2));
  __syncwarp();
  if (lane < (kTileN >> lg_br) * NH) {
    const int k = lane / NH, half = lane % NH;
    const int t = j * kTileN + (k << lg_br);  // first key of the box
    const int y = ybase[(t >> lg_p) - jp0] + (t & ((1 << lg_p) - 1));
    tc::tma_load_2d(dst + half * (kTileN * 128) + (k << lg_br) * 128, map, half * 64, y, bar);
  }
}

// One tile CTA.  WS = false: the decode CTA's shape (4 warps, 3 tile buffers),
// in the launch that also runs decode units; WS = true: a launch of chunk
// tiles only, 6 warps (4 softmax warps, one issuing the S MMAs and key-tile
// copies, one the P.V MMAs and value-tile copies) and 6 tile buffers.  The
// per-row arithmetic and its order are the same in both, so a chunk row's
// output bits do not depend on which launch ran it.
template <int D, int G, bool WS>
__device__ __forceinline__ void prefill_tile(const AttnParams& p, int cta, unsigned char* smem_raw) {
  using S = PrefillLayout<D, WS>;
  constexpr int NT = WS ? 192 : kTileM;  // threads of the CTA
  constexpr int kBarAll = WS ? WS_ALL : BAR_ALL;
  constexpr int kStall = WS ? WS_STALL : BAR_STALL;
  constexpr int kM0 = WS ? WS_M0 : BAR_M0;
  using T = PrefillTmem<D, WS ? 3 : 2>;
  constexpr int NH = S::NH;
  {
    // a launch that gave less shared memory than this layout needs touches none of it
    uint32_t dyn;
    asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    if (dyn < static_cast<uint32_t>(S::BYTES)) {
      if (threadIdx.x == 0) record_error(p.status, ST_LAUNCH);
      if (threadIdx.x < 32) tc::tmem_relinquish();
      return;
    }
  }
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // ring slot r at sm + r * TILE
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + S::BAR_OFF);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + S::TSLOT_OFF);
  int32_t* last_flag = reinterpret_cast<int32_t*>(sm + S::LAST_OFF);
  int32_t* last_item = reinterpret_cast<int32_t*>(sm + S::BAR_OFF + kBarAll * 8);  // per ring slot: last item issued
  static_assert(kBarAll * 8 + S::SLOTS * 4 <= 248, "barriers overlap the TMEM slot");
  int32_t* pids = reinterpret_cast<int32_t*>(sm + S::PID_OFF);  // page ids, then tensor-map rows

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
    for (int i = 0; i < kBarAll; ++i)  // nothing ever arrives on the stall barrier
      mbar_init(&bar[i], (WS && i >= WS_PR0 && i < WS_PR0 + 3) ? kTileM : 1);
    for (int i = 0; i < S::SLOTS; ++i) last_item[i] = -1;
    fence_barrier_init();
    tc::prefetch_tensormap(&p.kmap);  // the copy issuer's descriptors, fetched while the setup runs
    tc::prefetch_tensormap(&p.vmap);
  }
  const int lg_p = 31 - __clz(p.P);
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
    for (int r = tid; r < rows_here; r += NT)
      bad |= __ldg(p.seq_ids + rb + t0 + r) != seq || __ldg(p.positions + rb + t0 + r) != p0 + t0 + r;
    const int jp_check = p_max / p.P;
    for (int jp = tid; jp <= max(jp_check, jp_last); jp += NT) {
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
  // page ids -> tensor-map rows (pages past the sequence take the first page's)
  if (run) {
    const int fallback_pid = __ldg(bt + jp0);  // = pids[0], read where no thread overwrites it
    for (int jp = jp0 + tid; jp <= jp_last; jp += NT) {
      int pid = pids[jp - jp0];
      if (pid < 0 || pid >= p.num_pages) pid = fallback_pid;
      pids[jp - jp0] = (pid * p.Hkv + h) << lg_p;
    }
  }
  __syncthreads();

  PrefillIssueLog log;
  const int lane = tid & 31;
  constexpr uint32_t id_qk = tc::idesc_bf16_f32(kTileM, kTileN, false);
  constexpr uint32_t id_pv = tc::idesc_bf16_f32(kTileM, D, true);
  // S(jj) = Q K(jj)^T into S buffer sb from the key tile at K (one thread;
  // K(jj) has landed); completion arrives on bar[cb]
  auto issue_qk = [&](const unsigned char* K, int cb, int sb) {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const unsigned char* kb = K + (kk / 4) * S::KH + (kk % 4) * 32;
      tc::mma_bf16_ts(tb + T::S + sb * kTileN, tb + T::Q + kk * 8, tc::smem_desc(kb, 16, 1024), id_qk, kk > 0);
    }
    tc::mma_commit(&bar[cb]);
    log.issue(cb);
  };
  // O += P(jj) V(jj), P as (hi, lo) from S buffer sb, V the tile at Vt
  auto issue_pv = [&](int jj, const unsigned char* Vt, int cb, int sb) {
#pragma unroll
    for (int kk = 0; kk < kTileN / 16; ++kk) {
      const uint64_t vb = tc::smem_desc(Vt + kk * 2048, S::KH, 1024);  // 16 keys of the MN-major value tile
      const uint32_t ph = tb + T::S + sb * kTileN + (kk / 2) * 32 + (kk % 2) * 8;  // hi of keys 16kk .. +15; lo 16 columns on
      tc::mma_bf16_ts(tb + T::O, ph, vb, id_pv, jj > 0 || kk > 0);
      tc::mma_bf16_ts(tb + T::O, ph + 16, vb, id_pv, true);
    }
    tc::mma_commit(&bar[cb]);
    log.issue(cb);
  };
  // Values past the chunk's last position may be stale or poisoned: zero
  // those rows of a value tile so that 0-weights never meet a NaN (threads
  // `first_thread` .. of a group of `nthreads`)
  auto zero_tail = [&](unsigned char* Vt, int key0, int first_thread, int nthreads) {
    const int first = max(0, p_last + 1 - key0);
    const int n16 = (kTileN - first) * NH * 8;  // 16-byte pieces to clear
    for (int i = first_thread; i < n16; i += nthreads) {
      const int row = first + i / (NH * 8), piece = i % (NH * 8);
      *reinterpret_cast<uint4*>(Vt + (piece / 8) * S::KH + row * 128 + (piece % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    tc::fence_proxy_async_smem();
  };

  // ---- the online softmax of this row's 64 scores of one key tile (log2
  // domain), in two halves of 32 read from tensor memory twice (for the
  // maximum, then for the weights), so that no more than 32 scores are live
  // in registers.  The same code runs in both CTA shapes.
  float m_ref = -INFINITY, l_run = 0.0f;
  auto softmax_max = [&](uint32_t col_s, int key0, bool edge) -> float {  // returns the rescale factor
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
    return alpha;
  };
  auto softmax_weights = [&](uint32_t col_s, int key0, bool edge) {
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
  };
  // O *= alpha (the reference max moved; P.V(j-1), O's last writer, is done)
  auto rescale_o = [&](float alpha) {
#pragma unroll 1
    for (int c4 = 0; c4 < D / 32; ++c4) {
      float o[32];
      tc::tmem_ld32(tb + lane_base + T::O + c4 * 32, o);
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = __fmul_rn(o[i], alpha);
      tc::tmem_st32(tb + lane_base + T::O + c4 * 32, o);
    }
  };
  // Q row -> TMEM columns [T::Q, T::Q + D/2), two bf16 per column (the
  // softmax warps), then the block meets before the first MMA
  auto q_to_tmem = [&]() {
    if (warp < 4) {
#pragma unroll
      for (int c16 = 0; c16 < D / 32; ++c16)
        tc::tmem_st16(tb + lane_base + T::Q + c16 * 16, *reinterpret_cast<uint32_t(*)[16]>(&w[16 * c16]));
      tc::tmem_wait_st();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
  };

  bool ok = !(p.debug_stall && nk > 0) || mbar_wait(&bar[kStall], 0, p.wait_limit);  // the stall runs out
  if constexpr (!WS) {
    // ---- the ring: the three tile buffers take key and value tiles in the
    // order the tensor pipe reads them, K(0), K(1), V(0), K(2), V(1), K(3), ...
    // (item i in slot i % 3); a slot takes item i + 3 once the MMA that read
    // item i is done, so a value tile is copied a key tile ahead of its P.V and
    // a key tile about one ahead of its S.
    auto item_tile = [](int i) { return i == 0 ? 0 : ((i & 1) ? (i + 1) / 2 : (i - 2) / 2); };
    auto k_item = [](int jj) { return jj == 0 ? 0 : 2 * jj - 1; };
    auto v_item = [](int jj) { return 2 * jj + 2; };
    auto issue_item = [&](int i) {  // all lanes of a loader warp; nothing past the CTA's key tiles
      const int jj = item_tile(i);
      if (jj >= nk) return;
      const bool is_k = i == 0 || (i & 1);
      prefill_load_kv<D>(is_k ? &p.kmap : &p.vmap, sm + (i % S::SLOTS) * S::TILE, &bar[BAR_R0 + i % S::SLOTS], pids,
                         jp0, j_begin + jj, lg_p, lane);
      if (lane == 0) last_item[i % S::SLOTS] = i;
    };
    auto wait_item = [&](int i) { return mbar_wait(&bar[BAR_R0 + i % S::SLOTS], (i / S::SLOTS) & 1, p.wait_limit); };
    griddep_wait();  // the chunk's own rows, appended by a preceding dependent-launch append, are visible from here
    if (warp == 0)
      for (int i = 0; i < S::SLOTS; ++i) issue_item(i);
    q_to_tmem();

    // Key tile j: S(j) done -> softmax(j) -> P.V(j).  Three threads issue the
    // asynchronous work, each also a softmax row: warps 0 and 3 the copies,
    // thread 32 S(j+1) during softmax(j) (once P.V(j-1) has left the other S
    // buffer and K(j+1) has landed), thread 64 P.V(j).  A tensor-core MMA of
    // these shapes keeps its issuing thread about 100 cycles, so spreading the
    // MMAs over two warps keeps either from holding back the block by a whole
    // key tile.  The threads meet once per key tile, before P.V(j).  Every
    // barrier has at most one phase outstanding; every wait is bounded.
    constexpr int kLoader = 0, kSIssuer = 32, kPvIssuer = 64;  // threads
    constexpr int kKWarp = 0, kVWarp = 3;                       // warps that issue key / value tile copies
    // a role thread's own waits; a failure there reaches the others at the next
    // block-wide meeting (their waits on its work run out too: bounded)
    bool role_ok = true;
    if (tid == kSIssuer && nk > 0 && ok) {
      role_ok = wait_item(k_item(0));
      if (role_ok) {
        tc::fence_after_sync();
        issue_qk(sm + (k_item(0) % S::SLOTS) * S::TILE, BAR_S0, 0);
      }
    }
    bool next_k_slot_refilled = false;  // warp 3: S(j)'s key slot already took its next item
    for (int j = 0; j < nk && ok; ++j) {
      // ---- S(j) done (each warp waits for itself)
      bool good = __all_sync(0xffffffffu, mbar_wait(&bar[BAR_S0 + (j & 1)], (j >> 1) & 1, p.wait_limit));
      tc::fence_after_sync();
      // S(j) has read K(j): its slot takes the item three on, K(2) after S(0)
      // (warp 0 issues key tiles), V(j) after S(j > 0) (warp 3 value tiles)
      if (good && warp == (j == 0 ? kKWarp : kVWarp)) {
        if (!next_k_slot_refilled) issue_item(k_item(j) + S::SLOTS);
        next_k_slot_refilled = false;
      }
      if (good && tid == kSIssuer) log.seen(BAR_S0 + (j & 1));
      const uint32_t col_s = tb + lane_base + T::S + (j & 1) * kTileN;
      const int key0 = (j_begin + j) * kTileN;
      const bool edge = key0 + kTileN - 1 > my_pos;  // the row's causal edge (or keys past the chunk) is in this tile
      float alpha = 1.0f;
      if (good) alpha = softmax_max(col_s, key0, edge);
      // ---- P.V(j-1) done: warp 0 refills its value slot (with K(j+2)); thread
      // 32 then issues S(j+1) into the other S buffer once K(j+1) has landed
      if (good && role_ok && j > 0 && (warp == kKWarp || tid == kSIssuer)) {
        role_ok = mbar_wait(&bar[BAR_O], (j - 1) & 1, p.wait_limit);
        if (warp == kKWarp) {
          role_ok = __all_sync(0xffffffffu, role_ok);
          if (role_ok) issue_item(v_item(j - 1) + S::SLOTS);
        }
      }
      if (good && role_ok && tid == kSIssuer && j + 1 < nk) {
        role_ok = wait_item(k_item(j + 1));
        if (role_ok) {
          tc::fence_after_sync();
          issue_qk(sm + (k_item(j + 1) % S::SLOTS) * S::TILE, BAR_S0 + ((j + 1) & 1), (j + 1) & 1);
        }
      }
      if (good) {
        softmax_weights(col_s, key0, edge);
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
          // threads 0 and 32 saw P.V(j-1) done before S(j+1); the others see it here
          if (__all_sync(0xffffffffu, mbar_wait(&bar[BAR_O], (j - 1) & 1, p.wait_limit))) {
            tc::fence_after_sync();
            rescale_o(alpha);
          } else {
            good = false;
          }
        }
      }
      tc::tmem_wait_st();
      const int vi = v_item(j);
      tc::fence_before_sync();
      if (!(ok = __syncthreads_and(good && role_ok && wait_item(vi)))) break;
      if (key0 + kTileN - 1 > p_last) {
        zero_tail(sm + (vi % S::SLOTS) * S::TILE, key0, tid, kTileM);
        __syncthreads();
      }
      // ---- O += P V
      if (tid == kPvIssuer) {
        tc::fence_after_sync();
        issue_pv(j, sm + (vi % S::SLOTS) * S::TILE, BAR_O, j & 1);
      }
      if (warp == kVWarp && j + 1 < nk) {
        // S(j+1) has usually finished by now: its key slot takes its next item
        // (V(j+1)) a little earlier
        if (__shfl_sync(0xffffffffu, mbar_test(&bar[BAR_S0 + ((j + 1) & 1)], ((j + 1) >> 1) & 1) ? 1 : 0, 0)) {
          issue_item(k_item(j + 1) + S::SLOTS);
          next_k_slot_refilled = true;
        }
      }
    }
    if (ok && nk > 0) {
      // the last commit arrives when every MMA before it has completed too
      ok = __syncthreads_and(mbar_wait(&bar[BAR_O], (nk - 1) & 1, p.wait_limit));
      if (ok && tid == kPvIssuer) log.seen(BAR_O);
    }
    if (!ok) {
      // every copy and MMA in flight finishes before TMEM or shared memory is
      // reused: each MMA issuer drains its barriers; thread 0 the ring slots,
      // whose loads two warps issue (each slot's last one, at most one in flight)
      __syncthreads();
      if (tid == kSIssuer || tid == kPvIssuer) log.drain(bar, BAR_COUNT);
      if (tid == kLoader) {
        record_error(p.status, ST_TIMEOUT);
        for (int r = 0; r < S::SLOTS; ++r)
          if (last_item[r] >= 0) mbar_wait(&bar[BAR_R0 + r], (last_item[r] / S::SLOTS) & 1, kDrainWaitLimit);
      }
    }
  } else {
    // ---- warp-specialised: warps 0-3 are the softmax rows; warp 4 issues the
    // key-tile copies (its lanes) and the S MMAs (lane 0), warp 5 the value-tile
    // copies and the P.V MMAs.  Key tile j uses key and value buffer j % 3 and
    // S buffer j % 3.  The warps never meet inside the loop; they wait on:
    //   K(j) / V(j) landed
    //   S(j) done        -> softmax(j) may read S; key buffer j % 3 is free
    //   P(j) written     -> P.V(j) may run (one arrival per row)
    //   P.V(j) done      -> S buffer j % 3 (P(j)) and value buffer j % 3 are
    //                       free; O may be rescaled for key tile j + 1
    // Every kind of barrier comes three to a kind, one per buffer, and key tile
    // j + 3 can only reuse one after every waiter of key tile j has passed it:
    // no waiter can mistake a later phase for its own.  A key or value tile is
    // copied two key tiles ahead of its MMA.
    constexpr int kSWarp = 4, kPvWarp = 5;
    auto kbuf = [&](int jj) { return sm + (jj % 3) * S::TILE; };
    auto vbuf = [&](int jj) { return sm + (3 + jj % 3) * S::TILE; };
    auto par3 = [](int jj) { return static_cast<uint32_t>((jj / 3) & 1); };  // phase parity of key tile jj's barrier
    griddep_wait();  // the chunk's own rows, appended by a preceding dependent-launch append, are visible from here
    if (warp == kSWarp) {
      for (int jj = 0; jj < 3 && jj < nk; ++jj) {
        prefill_load_kv<D>(&p.kmap, kbuf(jj), &bar[WS_KF0 + jj], pids, jp0, j_begin + jj, lg_p, lane);
        if (lane == 0) log.issue(WS_KF0 + jj);
      }
    } else if (warp == kPvWarp) {
      for (int jj = 0; jj < 3 && jj < nk; ++jj) {
        prefill_load_kv<D>(&p.vmap, vbuf(jj), &bar[WS_VF0 + jj], pids, jp0, j_begin + jj, lg_p, lane);
        if (lane == 0) log.issue(WS_VF0 + jj);
      }
    }
    q_to_tmem();
    bool wok = ok;  // this warp's waits (warp-uniform)
    if (warp == kSWarp) {
      for (int j = 0; j < nk && wok; ++j) {
        // S buffer j % 3 held P(j-3): P.V(j-3) must be done; K(j) landed
        if (j >= 3) wok = __all_sync(0xffffffffu, mbar_wait(&bar[WS_OD0 + j % 3], par3(j - 3), p.wait_limit));
        wok = wok && __all_sync(0xffffffffu, mbar_wait(&bar[WS_KF0 + j % 3], par3(j), p.wait_limit));
        if (!wok) break;
        if (lane == 0) {
          log.seen(WS_KF0 + j % 3);
          tc::fence_after_sync();
          issue_qk(kbuf(j), WS_SD0 + j % 3, j % 3);
        }
        __syncwarp();
        if (j + 2 < nk && j >= 1) {
          // S(j-1) has read key buffer (j-1) % 3: it takes K(j+2)
          wok = __all_sync(0xffffffffu, mbar_wait(&bar[WS_SD0 + (j - 1) % 3], par3(j - 1), p.wait_limit));
          if (!wok) break;
          if (lane == 0) log.seen(WS_SD0 + (j - 1) % 3);
          prefill_load_kv<D>(&p.kmap, kbuf(j + 2), &bar[WS_KF0 + (j + 2) % 3], pids, jp0, j_begin + j + 2, lg_p, lane);
          if (lane == 0) log.issue(WS_KF0 + (j + 2) % 3);
        }
      }
    } else if (warp == kPvWarp) {
      for (int j = 0; j < nk && wok; ++j) {
        wok = __all_sync(0xffffffffu, mbar_wait(&bar[WS_PR0 + j % 3], par3(j), p.wait_limit) &&
                                           mbar_wait(&bar[WS_VF0 + j % 3], par3(j), p.wait_limit));
        if (!wok) break;
        if (lane == 0) log.seen(WS_VF0 + j % 3);
        const int key0 = (j_begin + j) * kTileN;
        if (key0 + kTileN - 1 > p_last) {
          zero_tail(vbuf(j), key0, lane, 32);
          __syncwarp();
        }
        if (lane == 0) {
          tc::fence_after_sync();
          issue_pv(j, vbuf(j), WS_OD0 + j % 3, j % 3);
        }
        __syncwarp();
        if (j + 2 < nk && j >= 1) {
          // P.V(j-1) has read value buffer (j-1) % 3: it takes V(j+2)
          wok = __all_sync(0xffffffffu, mbar_wait(&bar[WS_OD0 + (j - 1) % 3], par3(j - 1), p.wait_limit));
          if (!wok) break;
          if (lane == 0) log.seen(WS_OD0 + (j - 1) % 3);
          prefill_load_kv<D>(&p.vmap, vbuf(j + 2), &bar[WS_VF0 + (j + 2) % 3], pids, jp0, j_begin + j + 2, lg_p, lane);
          if (lane == 0) log.issue(WS_VF0 + (j + 2) % 3);
        }
      }
    } else {
      for (int j = 0; j < nk && wok; ++j) {
        wok = __all_sync(0xffffffffu, mbar_wait(&bar[WS_SD0 + j % 3], par3(j), p.wait_limit));
        if (!wok) break;
        tc::fence_after_sync();
        const uint32_t col_s = tb + lane_base + T::S + (j % 3) * kTileN;
        const int key0 = (j_begin + j) * kTileN;
        const bool edge = key0 + kTileN - 1 > my_pos;  // the row's causal edge (or keys past the chunk) is in this tile
        const float alpha = softmax_max(col_s, key0, edge);
        softmax_weights(col_s, key0, edge);
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
          wok = __all_sync(0xffffffffu, mbar_wait(&bar[WS_OD0 + (j - 1) % 3], par3(j - 1), p.wait_limit));
          if (!wok) break;
          tc::fence_after_sync();
          rescale_o(alpha);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        mbar_arrive(&bar[WS_PR0 + j % 3]);
      }
      // the last P.V (its commit arrives when every MMA before it is done too)
      if (wok && nk > 0)
        wok = __all_sync(0xffffffffu, mbar_wait(&bar[WS_OD0 + (nk - 1) % 3], par3(nk - 1), p.wait_limit));
    }
    ok = __syncthreads_and(wok);
    if (!ok) {
      // every copy and MMA in flight finishes before TMEM or shared memory is
      // reused: lane 0 of each issuing warp drains what it issued
      if (lane == 0 && (warp == kSWarp || warp == kPvWarp)) log.drain(bar, WS_COUNT);
      if (tid == 0) record_error(p.status, ST_TIMEOUT);
    }
  }
  __syncthreads();
  const bool row_thread = warp < 4;  // the threads that own a TMEM lane (every thread of the decode-shaped CTA)
  if (nk > 0) {
    tc::fence_after_sync();
    if (nsplit == 1) {
      if (ok && row_thread) {
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
      // let the last of the tile's CTAs merge the ranges in ascending order.
      // A tile's partials are tile-major: per key range, D / CB blocks of CB
      // columns, each [CB / 4][128 rows][4] floats (one key or value buffer's
      // size), so that a warp's 16-byte stores and the merge's bulk copies
      // are contiguous; the (max, sum) pairs are [key range][128 rows].
      constexpr int CB = S::TILE / (kTileM * 4);  // columns per block
      constexpr int NBS = D / CB;                 // blocks per key range
      const int ti = p.chunk_tile_begin[c] + mt * p.Hkv + h;  // the tile (its counter)
      const size_t blk0 = static_cast<size_t>(ti) * p.tile_splits;
      float* po = p.ws_tile_o + (blk0 + split) * (kTileM * D);
      if (row_thread) {
#pragma unroll 1
        for (int c4 = 0; c4 < D / 32; ++c4) {
          float o[32];
          if (ok) {
            tc::tmem_ld32(tb + lane_base + T::O + c4 * 32, o);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0.0f;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int col = c4 * 32 + 4 * i;
            float4* dst = reinterpret_cast<float4*>(po + (col / CB) * (kTileM * CB)) + ((col % CB) / 4) * kTileM + m;
            *dst = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
          }
        }
        reinterpret_cast<float2*>(p.ws_tile_ml)[(blk0 + split) * kTileM + m] =
            make_float2(ok ? m_ref : -INFINITY, ok ? l_run : 0.0f);
      }
      __threadfence();
      __syncthreads();
      int32_t* counter = p.ws_tile_count + ti;
      if (tid == 0) *last_flag = atomicAdd(counter, 1) == nsplit - 1;
      __syncthreads();
      if (*last_flag) {
        __threadfence();
        // Merge in ascending key-range order.  Row m's max and 1 / sum first;
        // then the partial blocks stream through the three key and value
        // buffers (free now) by bulk copies, several in flight, in the order
        // (column block, key range); each thread accumulates its row's CB
        // columns of a block.
        const float2* mlt = reinterpret_cast<const float2*>(p.ws_tile_ml) + blk0 * kTileM;
        const float* pbase = p.ws_tile_o + blk0 * (kTileM * D);
        const int nb = NBS * nsplit;
        auto issue_block = [&](int b) {  // block b: column block b / nsplit of key range b % nsplit
          uint64_t* mb = &bar[kM0 + b % kMergeSlots];
          mbar_arrive_expect_tx(mb, static_cast<uint32_t>(S::TILE));
          bulk_g2s(sm + (b % kMergeSlots) * S::TILE,
                   pbase + static_cast<size_t>(b % nsplit) * (kTileM * D) + (b / nsplit) * (kTileM * CB),
                   static_cast<uint32_t>(S::TILE), mb, l2_policy_evict_first());
        };
        int issued = 0;
        if (tid == 0) {
          fence_proxy_async_global();  // the other CTAs' partials, seen through the counter, before the bulk reads
          for (; issued < min(kMergeSlots, nb); ++issued) issue_block(issued);
        }
        const int mr = row_thread ? m : 0;  // the issuing warps of the wider CTA own no row: they read row 0
        float M = -INFINITY;
#pragma unroll 4
        for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, __ldcg(mlt + sp * kTileM + mr).x);
        float lsum = 0.0f;
#pragma unroll 4
        for (int sp = 0; sp < nsplit; ++sp) {
          const float2 v = __ldcg(mlt + sp * kTileM + mr);
          lsum = fmaf(ex2(__fsub_rn(v.x, M)), v.y, lsum);
        }
        const float inv = __fdiv_rn(1.0f, lsum);
        bool mok = true;
#pragma unroll 1
        for (int cb = 0; cb < NBS && mok; ++cb) {
          float acc[CB];
#pragma unroll
          for (int i = 0; i < CB; ++i) acc[i] = 0.0f;
#pragma unroll 1
          for (int sp = 0; sp < nsplit; ++sp) {
            const int b = cb * nsplit + sp;
            const float mv = __ldcg(mlt + sp * kTileM + mr).x;
            const bool got = mbar_wait(&bar[kM0 + b % kMergeSlots], (b / kMergeSlots) & 1, p.wait_limit);
            if (got) {
              const float f = ex2(__fsub_rn(mv, M));
              const float4* src = reinterpret_cast<const float4*>(sm + (b % kMergeSlots) * S::TILE) + mr;
#pragma unroll
              for (int i = 0; i < CB / 4; ++i) {
                const float4 v = src[i * kTileM];
                acc[4 * i] = fmaf(f, v.x, acc[4 * i]);
                acc[4 * i + 1] = fmaf(f, v.y, acc[4 * i + 1]);
                acc[4 * i + 2] = fmaf(f, v.z, acc[4 * i + 2]);
                acc[4 * i + 3] = fmaf(f, v.w, acc[4 * i + 3]);
              }
            }
            if (!(mok = __syncthreads_and(got))) break;  // every thread is done with the slot
            if (tid == 0 && issued < nb) {
              tc::fence_proxy_async_smem();
              issue_block(issued++);
            }
          }
          if (mok && row_valid) {
            __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + row_off + cb * CB;
#pragma unroll
            for (int i = 0; i < CB / 8; ++i) {
              uint32_t w[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const __nv_bfloat162 pr = __floats2bfloat162_rn(__fmul_rn(acc[8 * i + 2 * k], inv),
                                                                __fmul_rn(acc[8 * i + 2 * k + 1], inv));
                w[k] = *reinterpret_cast<const uint32_t*>(&pr);
              }
              *reinterpret_cast<uint4*>(orow + 8 * i) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
        if (!mok && tid == 0) {
          record_error(p.status, ST_TIMEOUT);
          for (int b = max(0, issued - kMergeSlots); b < issued; ++b)  // copies in flight land before the CTA leaves
            mbar_wait(&bar[kM0 + b % kMergeSlots], (b / kMergeSlots) & 1, kDrainWaitLimit);
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
