// pa_decode_mma_bf16.cuh -- decode units for bf16 K/V pools with head_dim 128
// and 3..8 query heads per kv head on warp-level tensor-core MMAs
// (mma.sync m16n8k16, bf16 inputs, FP32 accumulation).
//
// With G query heads per kv head each K/V byte feeds G/2 FP32 FMAs in the SIMT
// units ("llm-rs ...", section "2. Why decode is a memory problem": decode is
// bound by memory only while the arithmetic per byte stays small); from G = 3
// on, the tensor cores take the arithmetic instead.  Same contract, unit
// decomposition (one warp, one CTA per (row, kv head, split)) and split merge
// as the e4m3 tensor-core units, with these differences:
//   * A 32-token stage holds K and V as two 128-byte-swizzled half tiles each
//     (head elements 0..63 and 64..127: boxes of 64 bf16 x min(P, 32) rows).
//   * S^T = K . Q^T: A = K fragments straight from ldmatrix (no conversion),
//     B = the bf16 query, exact.
//   * O^T += V^T . P^T: A = V^T fragments straight from ldmatrix.trans; B =
//     the softmax weights as bf16 hi = bf16(w) and lo = bf16(w - hi), two MMAs,
//     so the product sees w to about 2^-16 (the prefill tiles do the same).
//   * The accumulator rows are head elements 16 i + (lane / 4) and + 8: the
//     state goes through shared memory to the shared split-merge epilogue,
//     which writes coalesced rows.
#pragma once

#include "pa_decode_mma.cuh"

namespace pa {

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void* smem_row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(smem_row)));
}

// One 32-token stage: K half 0, K half 1, V half 0, V half 1 (32 rows x 128 B each).
constexpr int kBfHalfBytes = kStageTokens * 128;
constexpr int kBfStageBytes = 4 * kBfHalfBytes;

template <int G, int NST>
struct MmaBfGeom {
  static constexpr int THREADS = 32;
  static constexpr size_t SMEM = 1024 + mma_header_bytes() + static_cast<size_t>(NST) * kBfStageBytes;
  static_assert(NST >= 2 && NST <= kMaxStages, "ring depth");
  static_assert(G >= 1 && G <= 8, "query heads per kv head");
  static_assert(static_cast<size_t>(G) * (128 + 2) * 4 <= static_cast<size_t>(NST) * kBfStageBytes, "ring");
};

// Copy the token slots of stage n into ring slot s: boxes of BR = min(P, 32)
// rows, two head-dim halves each, for K and for V.
__device__ __forceinline__ void mma_bf_issue_stage(const AttnParams& p, MmaSmemHeader* hdr, unsigned char* ring, int n,
                                                   int s, int t_begin, int t_end, int j0, int h, int lg_p) {
  const int a = t_begin + n * kStageTokens;
  const int b = min(t_end, a + kStageTokens);
  const int P = 1 << lg_p;
  const int BR = P < kStageTokens ? P : kStageTokens;
  unsigned char* st = ring + static_cast<size_t>(s) * kBfStageBytes;
  const int nbox = (b - a + BR - 1) / BR;
  mbar_arrive_expect_tx(&hdr->full[s], static_cast<uint32_t>(4 * nbox * BR * 128));
  for (int k = 0; k < nbox; ++k) {
    const int t = a + k * BR;
    const int page = hdr->pid[(t >> lg_p) - j0];
    const int y = (page * p.Hkv + h) * P + (t & (P - 1));
    const int off = k * BR * 128;
    tc::tma_load_2d(st + off, &p.kmap_dec, 0, y, &hdr->full[s]);
    tc::tma_load_2d(st + kBfHalfBytes + off, &p.kmap_dec, 64, y, &hdr->full[s]);
    tc::tma_load_2d(st + 2 * kBfHalfBytes + off, &p.vmap_dec, 0, y, &hdr->full[s]);
    tc::tma_load_2d(st + 3 * kBfHalfBytes + off, &p.vmap_dec, 64, y, &hdr->full[s]);
  }
}

// One unit (row, kv head h, split) on one warp (lanes 0..31 of the CTA).
template <int G, int NST>
__device__ __forceinline__ void decode_unit_mma_bf16(const AttnParams& p, int unit, unsigned char* smem_raw) {
  constexpr int D = 128, ST = kStageTokens;

  const int h = unit % p.Hkv;
  const int rest = unit / p.Hkv;
  const int split = rest % p.max_splits;
  const int row = unit_row(p, rest / p.max_splits);
  if (row >= p.n_rows) return;
  if (p.n_chunks > 0 && row_in_chunk(p, row)) return;

  const int lane = threadIdx.x & 31;
  const int g4 = lane >> 2;  // fragment group: key row (QK), head element (PV), query head (B operand)
  const int t4 = lane & 3;   // thread in group
  const size_t out_row = static_cast<size_t>(row) * p.Hq + static_cast<size_t>(h) * G;
  // Query fragments (B of Q.K), loaded first so that their latency overlaps
  // the sequence and page-id lookups: head g4 of the group (zero if >= G),
  // elements 16kb + 2t4 .. +1 (b0) and 16kb + 8 + 2t4 .. +1 (b1).
  uint32_t qf[8][2];
  {
    const uint32_t* qs = reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint16_t*>(p.q) +
                                                           (out_row + (g4 < G ? g4 : 0)) * D);
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
      qf[kb][0] = g4 < G ? __ldg(qs + 8 * kb + t4) : 0u;
      qf[kb][1] = g4 < G ? __ldg(qs + 8 * kb + 4 + t4) : 0u;
    }
  }
  // a row that appends itself (pa_step): lane l loads elements 4l .. 4l+3 of
  // its new K and V before anything else, so that they have landed by the
  // time the page ids have
  const bool own_row = row_appends_itself(p, row);
  uint32_t kw[4], vw[4];
  if (own_row) {
    load_new_raw<4>(p, row, h, 4 * lane, false, kw);
    load_new_raw<4>(p, row, h, 4 * lane, true, vw);
  }
  const int seq = __ldg(p.seq_ids + row);
  const int pos = __ldg(p.positions + row);
  const int P = p.P;

  if (seq < 0 || seq >= p.num_seqs || pos < 0 || pos >= p.max_blocks * P) {
    if (split == 0) {
      for (int i = lane; i < G * D; i += 32) store_out(p.out, true, out_row * D + i, 0.0f);
      if (lane == 0) record_error(p.status, ST_OUT_OF_RANGE);
    }
    return;
  }
  const int L = pos + 1;
  const int nsplit = (L + p.split_tokens - 1) / p.split_tokens;
  if (split >= nsplit) return;
  const int t_begin = split * p.split_tokens;
  const int t_end = min(L, t_begin + p.split_tokens);
  const int j0 = t_begin / P;
  const int npg = (t_end + P - 1) / P - j0;
  const int nstage = (t_end - t_begin + ST - 1) / ST;
  const int lg_p = 31 - __clz(P);
  const bool append_here = own_row && split == nsplit - 1;

  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  MmaSmemHeader* hdr = reinterpret_cast<MmaSmemHeader*>(smem);
  unsigned char* ring = smem + mma_header_bytes();
  if (lane == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(&hdr->full[s], 1);
    mbar_init(&hdr->stall, 1);
    hdr->bad = 0;
    hdr->last = 0;
    fence_barrier_init();
  }
  bool unit_bad;
  {
    // the unit's page ids, range-checked before any copy
    const int32_t* bt = p.block_tables + static_cast<size_t>(seq) * p.max_blocks + j0;
    bool bad = false;
    for (int i = lane; i < npg && i < kMaxUnitPages; i += 32) {
      const int pid = __ldg(bt + i);
      bad |= pid < 0 || pid >= p.num_pages;
      hdr->pid[i] = pid;
    }
    unit_bad = __any_sync(0xffffffffu, bad);
    __syncwarp();  // page ids and barrier init visible to lane 0
    if (unit_bad && lane == 0) {
      hdr->bad = 1;
      record_error(p.status, ST_OUT_OF_RANGE);
    }
  }
  // the pool rows appended by a preceding dependent-launch append are visible
  // from here (a row that appends itself reads nothing that launch writes)
  if (!own_row) griddep_wait();
  if (lane == 0 && !unit_bad) {
    const int first = min(NST, nstage);
    for (int n = 0; n < first; ++n) mma_bf_issue_stage(p, hdr, ring, n, n, t_begin, t_end, j0, h, lg_p);
  }
  if (append_here) {  // the row's own K/V, converted, to the pool (and below to the stage)
    uint32_t raw[4] = {kw[0], kw[1], kw[2], kw[3]};
    convert_new<KV_BF16, 4>(p, h, false, raw, kw);
    raw[0] = vw[0]; raw[1] = vw[1]; raw[2] = vw[2]; raw[3] = vw[3];
    convert_new<KV_BF16, 4>(p, h, true, raw, vw);
    const int pid = hdr->pid[(pos >> lg_p) - j0];
    if (pid >= 0 && pid < p.num_pages) {
      store_piece<8>(pool_elem(p.k_pool, p, pid, h, pos & (P - 1), 4 * lane, 2), kw);
      store_piece<8>(pool_elem(p.v_pool, p, pid, h, pos & (P - 1), 4 * lane, 2), vw);
    }
  }
  const float score_scale = p.qk_scale_log2_h[PA_HEAD(p, h)];

  // per-lane ldmatrix row offsets (row r: chunk c at c ^ (r % 8)):
  //   Q.K, m-tile mi, head block kb: key row 16 mi + (lane & 7) + 8 ((lane >> 3) & 1), chunk 2 (kb % 4) + (lane >> 4)
  //   P.V, k-step ks, m-tile i:      key row 16 ks + (lane & 7) + 8 ((lane >> 4) & 1), chunk 2 (i % 4) + ((lane >> 3) & 1)
  const int kr_row = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int vr_row = (lane & 7) + ((lane >> 4) & 1) * 8;
  uint32_t k_off[4], v_off[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    k_off[c] = sw128(kr_row, 2 * c + (lane >> 4));
    v_off[c] = sw128(vr_row, 2 * c + ((lane >> 3) & 1));
  }

  // ---- softmax state: heads 2 t4 and 2 t4 + 1; O^T rows d = 16 i + g4 and
  // 16 i + 8 + g4 for m-tile i.  The weight sums come from MMAs with an
  // all-ones A over the same (hi, lo) weights that meet V.
  float m_ref[2] = {-INFINITY, -INFINITY};
  float o[8][4], lsum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  const uint32_t ones[4] = {0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u};  // bf16x2 (1, 1)

  int drain_n = -1;  // the stage a wait gave up on
  int s = 0;         // ring slot of stage n
  uint32_t ph = 0;   // its phase parity
  for (int n = 0; n < nstage && !unit_bad; ++n) {
    bool got = mbar_wait(&hdr->full[s], ph, p.wait_limit);
    if (p.debug_stall) got = got && mbar_wait(&hdr->stall, 0, p.wait_limit);  // runs out by construction
    if (!__all_sync(0xffffffffu, got)) {
      if (lane == 0) {
        record_error(p.status, ST_TIMEOUT);
        hdr->bad = 1;
      }
      drain_n = n;
      break;
    }
    unsigned char* st = ring + static_cast<size_t>(s) * kBfStageBytes;
    unsigned char* vs = st + 2 * kBfHalfBytes;
    if (append_here && n == nstage - 1) {  // the row's own slot, as appended: lane l's 8 bytes
      const int r = pos - (t_begin + n * ST);  // sit in half l / 16, 16-byte chunk (l % 16) / 2
      const uint32_t off = (lane >> 4) * kBfHalfBytes + sw128(r, (lane & 15) >> 1) + 8 * (lane & 1);
      store_piece<8>(st + off, kw);
      store_piece<8>(vs + off, vw);
      __syncwarp();
    }
    const int n_valid = min(ST, t_end - (t_begin + n * ST));  // 1..32
    const bool full = n_valid == ST;
    // ---- S^T = K . Q^T, even and odd head blocks in separate accumulators
    float sc[2][4];
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
      float sa[4] = {0.0f, 0.0f, 0.0f, 0.0f}, sb[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) {
        uint32_t a[4];
        ldmatrix_x4(a, st + (kb / 4) * kBfHalfBytes + mi * 2048 + k_off[kb % 4]);
        if (kb & 1)
          mma_bf16_16816(sb, a, qf[kb][0], qf[kb][1]);
        else
          mma_bf16_16816(sa, a, qf[kb][0], qf[kb][1]);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int key = 16 * mi + g4 + (c >> 1) * 8;
        sc[mi][c] = (full || key < n_valid) ? __fadd_rn(sa[c], sb[c]) : -INFINITY;
      }
    }
    // ---- online softmax (log2 domain), as in the e4m3 units
    float t[2][4];
    float tmax = -INFINITY;
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        t[mi][c] = (full || sc[mi][c] != -INFINITY) ? fmaf(sc[mi][c], score_scale, -m_ref[c & 1]) : -INFINITY;
        tmax = fmaxf(tmax, t[mi][c]);
      }
    if (__any_sync(0xffffffffu, tmax > kRescaleSlack)) {
      float alpha[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float mx = fmaxf(fmaxf(__fmul_rn(sc[0][hh], score_scale), __fmul_rn(sc[0][2 + hh], score_scale)),
                         fmaxf(__fmul_rn(sc[1][hh], score_scale), __fmul_rn(sc[1][2 + hh], score_scale)));
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        alpha[hh] = 1.0f;
        if (mx > __fadd_rn(m_ref[hh], kRescaleSlack)) {
          alpha[hh] = ex2(__fsub_rn(m_ref[hh], mx));
          m_ref[hh] = mx;
        }
      }
      if (n > 0) {  // the first stage sets the first reference: nothing accumulated yet
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          o[i][0] = __fmul_rn(o[i][0], alpha[0]);
          o[i][1] = __fmul_rn(o[i][1], alpha[1]);
          o[i][2] = __fmul_rn(o[i][2], alpha[0]);
          o[i][3] = __fmul_rn(o[i][3], alpha[1]);
        }
        lsum[0] = __fmul_rn(lsum[0], alpha[0]);
        lsum[1] = __fmul_rn(lsum[1], alpha[1]);
        lsum[2] = __fmul_rn(lsum[2], alpha[0]);
        lsum[3] = __fmul_rn(lsum[3], alpha[1]);
      }
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int c = 0; c < 4; ++c)
          t[mi][c] = (full || sc[mi][c] != -INFINITY) ? fmaf(sc[mi][c], score_scale, -m_ref[c & 1]) : -INFINITY;
    }
    // weights w = 2^t as hi = bf16(w), lo = bf16(w - hi), into B-fragment order:
    // C layout (key g4 / g4+8, heads 2t4, 2t4+1) -> B layout (head g4, keys 2t4, 2t4+1)
    uint32_t phi[2][2], plo[2][2];  // [k-step][keys 0..7 / 8..15 of it]
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float w0 = ex2(t[mi][2 * half]), w1 = ex2(t[mi][2 * half + 1]);
        const __nv_bfloat16 h0 = __float2bfloat16_rn(w0), h1 = __float2bfloat16_rn(w1);
        const float r0 = __fsub_rn(w0, __bfloat162float(h0)), r1 = __fsub_rn(w1, __bfloat162float(h1));
        phi[mi][half] = movmatrix_trans(static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
                                        (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16));
        plo[mi][half] = movmatrix_trans(pack_bf16x2(r0, r1));
      }
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
      mma_bf16_16816(lsum, ones, phi[mi][0], phi[mi][1]);
      mma_bf16_16816(lsum, ones, plo[mi][0], plo[mi][1]);
    }
    // ---- value rows past the row's position: zero them (both halves) before
    // they meet weight 0 (stale or NaN bytes times 0 would poison the sums)
    if (!full) {
      for (int i = lane; i < (ST - n_valid) * 16; i += 32) {
        const int r = n_valid + (i >> 4), c = i & 15;
        *reinterpret_cast<uint4*>(vs + (c >> 3) * kBfHalfBytes + r * 128 + (c & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }
    // ---- O^T += V^T . P^T: m-tile i = head elements 16 i .. 16 i + 15 (half i / 4),
    // k-step ks = keys 16 ks .. 16 ks + 15
#pragma unroll
    for (int ks = 0; ks < 2; ++ks)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t a[4];
        ldmatrix_x4_trans(a, vs + (i / 4) * kBfHalfBytes + ks * 2048 + v_off[i % 4]);
        mma_bf16_16816(o[i], a, phi[ks][0], phi[ks][1]);
        mma_bf16_16816(o[i], a, plo[ks][0], plo[ks][1]);
      }
    // ---- release the slot and refill it
    __syncwarp();
    if (lane == 0 && n + NST < nstage) {
      fence_proxy_async();
      mma_bf_issue_stage(p, hdr, ring, n + NST, s, t_begin, t_end, j0, h, lg_p);
    }
    if (++s == NST) {
      s = 0;
      ph ^= 1u;
    }
  }
  // After a wait gave up on stage m, stages m .. m + NST - 1 may still be in
  // flight: let them land before the ring is reused.
  if (drain_n >= 0 && lane == 0) {
    for (int m = drain_n; m < min(drain_n + NST, nstage); ++m)
      mbar_wait(&hdr->full[m % NST], (m / NST) & 1, kDrainWaitLimit);
  }
  __syncwarp();

  // ---- the state to shared memory in the SIMT unit's layout (one warp), then
  // the shared epilogue and split merge (coalesced output rows)
  float* red_acc = reinterpret_cast<float*>(ring);  // [G][D]
  float* red_ml = red_acc + G * D;                  // [G][2]
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int head = 2 * t4 + hh;
    if (head < G) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        red_acc[head * D + 16 * i + g4] = o[i][hh];
        red_acc[head * D + 16 * i + 8 + g4] = o[i][2 + hh];
      }
      if (g4 == 0) {
        red_ml[head * 2] = m_ref[hh];
        red_ml[head * 2 + 1] = lsum[hh];
      }
    }
  }
  __syncwarp();
  decode_finish<D, G, KV_BF16, 1, 32>(p, hdr->bad != 0, &hdr->last, red_acc, red_ml, out_row, row, h, split, nsplit,
                                      true, NST * kBfStageBytes);
}

template <int G, int NST>
__global__ void __launch_bounds__(32, 8) decode_mma_bf16_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(128) unsigned char smem[];  // aligned to 1024 by hand in the unit
  decode_unit_mma_bf16<G, NST>(p, static_cast<int>(blockIdx.x), smem);
}

// Devices on which decode_mma_bf16_kernel<G, NST> may use its dynamic shared memory.
template <int G, int NST>
std::atomic<unsigned long long>& mma_bf16_smem_done() {
  static std::atomic<unsigned long long> done{0};
  return done;
}

template <int G, int NST>
cudaError_t launch_decode_mma_bf16_nst(const AttnParams& p, cudaStream_t stream, unsigned units) {
  using Geo = MmaBfGeom<G, NST>;
  const cudaError_t ea = allow_dynamic_smem(decode_mma_bf16_kernel<G, NST>, mma_bf16_smem_done<G, NST>(), Geo::SMEM);
  if (ea != cudaSuccess) return ea;
  const cudaError_t e = launch_kernel(decode_mma_bf16_kernel<G, NST>, dim3(units), dim3(Geo::THREADS), Geo::SMEM,
                                      stream, p.dependent != 0, p);
  count_launch();
  return e;
}

template <int G, int NST>
long long mma_bf16_resident_units() {
  static std::atomic<long long> cache[64];  // per device: resident CTAs + 1, 0 until known
  return resident_ctas(decode_mma_bf16_kernel<G, NST>, cache, mma_bf16_smem_done<G, NST>(), 32,
                       MmaBfGeom<G, NST>::SMEM);
}

#ifndef PA_MMA_BF16_NST
#define PA_MMA_BF16_NST 0  // 0: ring depth by the number of units; 2, 4 or 6: that depth always
#endif

// Ring depth by the number of units, as for the e4m3 units (no effect on the bits).
template <int G>
cudaError_t launch_decode_mma_bf16_inst(const AttnParams& p, cudaStream_t stream) {
  const long long units = static_cast<long long>(p.n_unit_rows) * p.max_splits * p.Hkv;
  if (units <= 0) return cudaSuccess;
  if (units > 0x7fffffffLL) return cudaErrorNotSupported;
  const unsigned u = static_cast<unsigned>(units);
  if (PA_MMA_BF16_NST == 2) return launch_decode_mma_bf16_nst<G, 2>(p, stream, u);
  if (PA_MMA_BF16_NST == 4) return launch_decode_mma_bf16_nst<G, 4>(p, stream, u);
  if (PA_MMA_BF16_NST == 6) return launch_decode_mma_bf16_nst<G, 6>(p, stream, u);
  if (units <= mma_bf16_resident_units<G, 6>()) return launch_decode_mma_bf16_nst<G, 6>(p, stream, u);
  if (units <= mma_bf16_resident_units<G, 4>()) return launch_decode_mma_bf16_nst<G, 4>(p, stream, u);
  return launch_decode_mma_bf16_nst<G, 2>(p, stream, u);
}

}  // namespace pa
