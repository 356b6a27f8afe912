// pa_decode_mma.cuh -- decode units for FP8 (E4M3) K/V pools with head_dim 128,
// where the query-head group makes Q.K and P.V a small dense contraction
// (G query heads x 32 keys x 128 per stage): warp-level tensor-core MMAs
// (mma.sync m16n8k16, f16 inputs, FP32 accumulation) instead of FP32 FMAs.
//
// Why: with G = 7 query heads per KV head ("Engines for the card you have":
// a 7B model with an FP8 key/value cache), each K/V byte feeds 7 FMAs; at HBM
// rate that is more than the FP32 pipes deliver, so the SIMT decode path is
// compute-bound here.  The tensor cores make the arithmetic cheap; what is
// left per byte is one conversion (e4m3x2 -> f16x2, exact).
//
// Same contract as the SIMT decode unit (one CTA per (row, kv head, split),
// the same split merge and epilogue), with these differences:
//   * A CTA is ONE warp.  A unit's work is a short chain (a few stages at the
//     context lengths of a 7B-class decode batch), so many small CTAs per SM
//     keep more units' copies in flight than a few wide ones, and no
//     cross-warp merge is needed.  (Opt-in row groups put 2, 4 or 8 such
//     units in one CTA to share the copies of a common prefix: see
//     decode_mma_group_kernel below.)  The warp waits on, consumes and refills
//     its ring of NST slots in stage order; NST (2, 4 or 8) follows the
//     number of units in the launch.
//   * Stages of 32 tokens arrive by 2-D tensor-map copies (box: 128 bytes x
//     min(P, 32) rows of one page of one kv head) into 128-byte swizzled
//     shared-memory tiles, so that ldmatrix and 16-byte row loads are free of
//     bank conflicts.
//   * S^T = K . Q^T: A = K (16 keys x 16 head elements) from ldmatrix on the fp8
//     bytes; each 32-bit fragment word holds 4 consecutive fp8 elements, so the
//     two f16x2 conversions of a word feed two MMAs whose k order is permuted;
//     the query fragments (B, constant per unit) are laid out with the same
//     permutation.  Query heads are the MMA's n (8; heads >= G are zero).
//   * O^T += V^T . P^T: A = V^T (16 head elements x 16 keys) built from 16-byte
//     row loads with byte permutes and e4m3x2 -> f16x2 conversions; thread t
//     owns head elements 16 (t/4) .. 16 (t/4) + 15, so the MMA's m rows are a
//     fixed permutation of the head dim, undone when the accumulators are
//     written out.  B = P^T: each softmax weight w (<= 2^8 by the lazy
//     reference max) as two f16 parts, hi = f16(w) and lo = f16(w - hi), moved
//     into fragment order with movmatrix.trans; two MMAs per k-step, so the
//     product sees w to about 2^-22 relative (f16 alone would leave 2^-11,
//     an error that grows with the values' magnitude).  With G <= 4 the hi
//     and lo parts share one MMA: columns 4..7 repeat query heads 0..3, so
//     their scores, references and weights are the same, and they carry the
//     lo parts into accumulator columns of their own, added to the hi
//     columns once at the end of the unit.
//   * The query enters as f16, scaled by a power of two chosen per (row, kv
//     head) so that its largest element is below 2^15; the power is folded
//     back into the score scale.  bf16 values in the f16 normal range are exact.
//   * Value rows of keys past the row's position in the last stage are zeroed in
//     shared memory before P.V (zero weights must never meet stale or NaN bytes).
#pragma once

#include "pa_decode.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

// ------------------------------------------------------- warp-level MMA --

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* smem_row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(smem_row)));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// Two e4m3 codes in the low (lo = true) or high half of w -> f16x2, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w, bool lo) {
  uint32_t d;
  if (lo)
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t}" : "=r"(d) : "r"(w));
  else
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h;\n\t}" : "=r"(d) : "r"(w));
  return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Byte i of the 16-byte swizzled row r of a 128-byte-per-row tile: chunk c sits
// at chunk position c ^ (r % 8).
__device__ __forceinline__ uint32_t sw128(int r, int chunk) { return r * 128 + ((chunk ^ (r & 7)) << 4); }

constexpr int kMmaStageBytes = 2 * kStageTokens * 128;  // K and V rows of one stage

struct MmaSmemHeader {
  uint64_t full[kMaxStages];   // stage landed (tensor-map copy bytes)
  uint64_t stall;              // never completed: the injected-stall test waits here
  int32_t bad;                 // a page id was out of range or a wait gave up
  int32_t last;                // this CTA merges the splits of its (row, kv head)
  int32_t pid[kMaxUnitPages];  // the unit's physical page ids
};

__host__ __device__ constexpr size_t mma_header_bytes() { return (sizeof(MmaSmemHeader) + 1023) / 1024 * 1024; }

// One warp per CTA, one CTA per unit; NST ring slots of one stage each.
template <int G, int NST>
struct MmaGeom {
  static constexpr int D = 128;
  static constexpr int THREADS = 32;
  static constexpr int STAGES = NST;
  static constexpr size_t SMEM = 1024 + mma_header_bytes() + static_cast<size_t>(NST) * kMmaStageBytes;
  static_assert(NST >= 2 && NST <= kMaxStages, "ring depth");
  static_assert(G >= 1 && G <= 8, "query heads per kv head");
  // the epilogue's [G][D] accumulator and [G][2] (max, sum) sit in the ring
  static_assert(static_cast<size_t>(G) * (D + 2) * 4 <= static_cast<size_t>(NST) * kMmaStageBytes, "ring");
};

// Copy the token slots of stage n (32 tokens from t_begin + 32 n) into ring
// slot s by tensor-map boxes of BR = min(P, 32) rows; every box is whole, so
// the last stage may carry slots past the unit's end (masked / zeroed later).
__device__ __forceinline__ void mma_issue_stage(const AttnParams& p, MmaSmemHeader* hdr, unsigned char* ring, int n,
                                                int s, int t_begin, int t_end, int j0, int h, int lg_p) {
  const int a = t_begin + n * kStageTokens;
  const int b = min(t_end, a + kStageTokens);
  const int P = 1 << lg_p;
  const int BR = P < kStageTokens ? P : kStageTokens;
  unsigned char* ks = ring + static_cast<size_t>(s) * kMmaStageBytes;
  unsigned char* vs = ks + kStageTokens * 128;
  const int nbox = (b - a + BR - 1) / BR;
  mbar_arrive_expect_tx(&hdr->full[s], static_cast<uint32_t>(2 * nbox * BR * 128));
  for (int k = 0; k < nbox; ++k) {
    const int t = a + k * BR;
    const int page = hdr->pid[(t >> lg_p) - j0];
    const int y = (page * p.Hkv + h) * P + (t & (P - 1));
    tc::tma_load_2d(ks + k * BR * 128, &p.kmap_dec, 0, y, &hdr->full[s]);
    tc::tma_load_2d(vs + k * BR * 128, &p.vmap_dec, 0, y, &hdr->full[s]);
  }
}

// The running state of one unit (one warp): query fragments and the online
// softmax (heads 2 t4 and 2 t4 + 1 of each lane; O^T rows d(i, g4) = 16 g4 + i
// and d(i, g4 + 8) = 16 g4 + 8 + i for m-tile i).  The sums of the weights come
// from MMAs with an all-ones A: lsum[0] / lsum[1] hold heads 2 t4 / 2 t4 + 1
// (lsum[2..3] repeat them), summed from the same (hi, lo) f16 parts of the
// weights that meet V.
template <int G>
struct MmaState {
  uint32_t qf[4][4];  // [kb][mma0 b0, mma0 b1, mma1 b0, mma1 b1]
  float score_scale;
  float m_ref[2];
  float o[8][4];
  float lsum[4];
};

// Query fragments (B of Q.K), f16, in the permuted k order of the K fragments:
// for head block kb (32 elements) the first MMA reads elements 32kb + 4 t4 +
// {0,1} and 32kb + 16 + 4 t4 + {0,1}, the second + 2; the lane's query head
// qhead (-1: a zero column).  Also clears the softmax state.
template <int G>
__device__ __forceinline__ void mma_prep(const AttnParams& p, int h, int qhead, const uint2 (&qraw)[4][2],
                                         MmaState<G>& st) {
  {
    float qv[4][8];
    float amax = 0.0f;
    const bool head_ok = qhead >= 0;
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
      const uint2 w0 = qraw[kb][0], w1 = qraw[kb][1];
      const float f[8] = {bf16lo(w0.x), bf16hi(w0.x), bf16lo(w0.y), bf16hi(w0.y),
                          bf16lo(w1.x), bf16hi(w1.x), bf16lo(w1.y), bf16hi(w1.y)};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        qv[kb][i] = head_ok ? f[i] : 0.0f;
        amax = fmaxf(amax, fabsf(qv[kb][i]));
      }
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    // Scale by 2^-shift so that the largest element lands in [2^14, 2^15):
    // amax = 1.f * 2^(E - 127) for biased exponent E; subnormal or zero
    // queries take the clamp.
    const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 126;
    const int shift = min(100, max(-100, e - 15));
    const float down = __uint_as_float(static_cast<uint32_t>(127 - shift) << 23);
    st.score_scale = __fmul_rn(p.qk_scale_log2_h[PA_HEAD(p, h)], __uint_as_float(static_cast<uint32_t>(127 + shift) << 23));
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
      st.qf[kb][0] = pack_f16x2(qv[kb][0] * down, qv[kb][1] * down);  // mma0: elements 4t4 + {0,1}
      st.qf[kb][1] = pack_f16x2(qv[kb][4] * down, qv[kb][5] * down);  //       16 + 4t4 + {0,1}
      st.qf[kb][2] = pack_f16x2(qv[kb][2] * down, qv[kb][3] * down);  // mma1: 4t4 + {2,3}
      st.qf[kb][3] = pack_f16x2(qv[kb][6] * down, qv[kb][7] * down);  //       16 + 4t4 + {2,3}
    }
  }
  st.m_ref[0] = st.m_ref[1] = -INFINITY;
#pragma unroll
  for (int i = 0; i < 4; ++i) st.lsum[i] = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) st.o[i][0] = st.o[i][1] = st.o[i][2] = st.o[i][3] = 0.0f;
}

// One 32-token stage of one unit: K rows at ks, V rows at vs (128-byte
// swizzled; n_valid of the 32 are the unit's keys).  Q.K, the online softmax
// and P.V into st.  Value rows past n_valid are zeroed first.
template <int G>
__device__ __forceinline__ void mma_stage(MmaState<G>& st, unsigned char* ks, unsigned char* vs, int n_valid,
                                          int lane) {
  constexpr int ST = kStageTokens;
  constexpr bool PACK = G <= 4;
  const int g4 = lane >> 2, t4 = lane & 3;
  const uint32_t ones[4] = {0x3c003c00u, 0x3c003c00u, 0x3c003c00u, 0x3c003c00u};  // f16x2 (1, 1)
  auto& qf = st.qf;
  auto& m_ref = st.m_ref;
  auto& o = st.o;
  auto& lsum = st.lsum;
  const float score_scale = st.score_scale;
  const bool full = n_valid == ST;
  // ---- S^T = K . Q^T for the stage's two 16-key m-tiles; the two k halves
  // of each head block accumulate separately (shorter dependency chains)
  // and are added at the end
  float sc[2][4];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi) {
    float sa[4] = {0.0f, 0.0f, 0.0f, 0.0f}, sb[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const int r = 16 * mi + (lane & 7) + ((lane >> 3) & 1) * 8;  // row this lane addresses for ldmatrix
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
      uint32_t kr[4];
      ldmatrix_x4(kr, ks + sw128(r, 2 * kb + (lane >> 4)));
      const uint32_t a0[4] = {e4m3x2_to_f16x2(kr[0], true), e4m3x2_to_f16x2(kr[1], true),
                              e4m3x2_to_f16x2(kr[2], true), e4m3x2_to_f16x2(kr[3], true)};
      const uint32_t a1[4] = {e4m3x2_to_f16x2(kr[0], false), e4m3x2_to_f16x2(kr[1], false),
                              e4m3x2_to_f16x2(kr[2], false), e4m3x2_to_f16x2(kr[3], false)};
      mma_f16_16816(sa, a0, qf[kb][0], qf[kb][1]);
      mma_f16_16816(sb, a1, qf[kb][2], qf[kb][3]);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int key = 16 * mi + g4 + (c >> 1) * 8;
      sc[mi][c] = (full || key < n_valid) ? __fadd_rn(sa[c], sb[c]) : -INFINITY;
    }
  }
  // ---- online softmax (log2 domain): this lane holds keys 16 mi + g4 (+8)
  // for heads 2 t4 (+1).  t = score * scale - reference; the reference of a
  // head moves only when some weight would exceed 2^kRescaleSlack, which a
  // single vote detects, so the common stage needs no max reduction.
  float t[2][4];
  float tmax = -INFINITY;
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      t[mi][c] = fmaf(sc[mi][c], score_scale, -m_ref[c & 1]);
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
        alpha[hh] = ex2(__fsub_rn(m_ref[hh], mx));  // 0 on the first stage
        m_ref[hh] = mx;
      }
    }
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
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int c = 0; c < 4; ++c) t[mi][c] = fmaf(sc[mi][c], score_scale, -m_ref[c & 1]);
  }
  // weights w = 2^t (masked keys: 2^-inf = 0) as hi = f16(w), lo = f16(w - hi),
  // into B-fragment order:
  // C layout (key g4 / g4+8, heads 2t4, 2t4+1) -> B layout (head g4, keys 2t4, 2t4+1)
  uint32_t phi[2][2], plo[2][2];  // P^T fragments: [k-step][keys 0..7 / 8..15 of it]
#pragma unroll
  for (int mi = 0; mi < 2; ++mi) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const float w0 = ex2(t[mi][2 * half]), w1 = ex2(t[mi][2 * half + 1]);
      const __half2 hi = __floats2half2_rn(w0, w1);
      const float2 hf = __half22float2(hi);
      const uint32_t hi_w = *reinterpret_cast<const uint32_t*>(&hi);
      const uint32_t lo_w = pack_f16x2(__fsub_rn(w0, hf.x), __fsub_rn(w1, hf.y));
      if constexpr (PACK) {
        phi[mi][half] = movmatrix_trans(t4 < 2 ? hi_w : lo_w);  // columns 0..3 hi, 4..7 lo
      } else {
        phi[mi][half] = movmatrix_trans(hi_w);
        plo[mi][half] = movmatrix_trans(lo_w);
      }
    }
    mma_f16_16816(lsum, ones, phi[mi][0], phi[mi][1]);
    if constexpr (!PACK) mma_f16_16816(lsum, ones, plo[mi][0], plo[mi][1]);
  }
  // ---- value rows past the row's position: zero them before they meet weight 0
  if (!full) {
    for (int i = lane; i < (ST - n_valid) * 8; i += 32)
      *reinterpret_cast<uint4*>(vs + (n_valid + i / 8) * 128 + (i % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
  }
  // ---- O^T += V^T . P^T, two 16-key k-steps
#pragma unroll
  for (int mi = 0; mi < 2; ++mi) {
    const int ta = 16 * mi + 2 * t4;  // keys ta, ta+1 (k slots 2t4, 2t4+1) and ta+8, ta+9
    const uint4 va = *reinterpret_cast<const uint4*>(vs + sw128(ta, g4));
    const uint4 vb = *reinterpret_cast<const uint4*>(vs + sw128(ta + 1, g4));
    const uint4 vc = *reinterpret_cast<const uint4*>(vs + sw128(ta + 8, g4));
    const uint4 vd = *reinterpret_cast<const uint4*>(vs + sw128(ta + 9, g4));
    const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
    const uint32_t wc[4] = {vc.x, vc.y, vc.z, vc.w}, wd[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll
    for (int w = 0; w < 2; ++w) {  // head elements 4w .. 4w+3 (rows g4) and 8 + 4w .. (rows g4 + 8)
      // byte pairs (key ta, key ta+1) and (ta+8, ta+9) for element e: low byte from the first key
      const uint32_t ab_lo = __byte_perm(wa[w], wb[w], 0x5140), ab_hi = __byte_perm(wa[w], wb[w], 0x7362);
      const uint32_t ab8_lo = __byte_perm(wa[w + 2], wb[w + 2], 0x5140), ab8_hi = __byte_perm(wa[w + 2], wb[w + 2], 0x7362);
      const uint32_t cd_lo = __byte_perm(wc[w], wd[w], 0x5140), cd_hi = __byte_perm(wc[w], wd[w], 0x7362);
      const uint32_t cd8_lo = __byte_perm(wc[w + 2], wd[w + 2], 0x5140), cd8_hi = __byte_perm(wc[w + 2], wd[w + 2], 0x7362);
      // element 4w + j of the thread's 16: m-tile i = 4w + j
      const uint32_t a_j0[4] = {e4m3x2_to_f16x2(ab_lo, true), e4m3x2_to_f16x2(ab8_lo, true),
                                e4m3x2_to_f16x2(cd_lo, true), e4m3x2_to_f16x2(cd8_lo, true)};
      const uint32_t a_j1[4] = {e4m3x2_to_f16x2(ab_lo, false), e4m3x2_to_f16x2(ab8_lo, false),
                                e4m3x2_to_f16x2(cd_lo, false), e4m3x2_to_f16x2(cd8_lo, false)};
      const uint32_t a_j2[4] = {e4m3x2_to_f16x2(ab_hi, true), e4m3x2_to_f16x2(ab8_hi, true),
                                e4m3x2_to_f16x2(cd_hi, true), e4m3x2_to_f16x2(cd8_hi, true)};
      const uint32_t a_j3[4] = {e4m3x2_to_f16x2(ab_hi, false), e4m3x2_to_f16x2(ab8_hi, false),
                                e4m3x2_to_f16x2(cd_hi, false), e4m3x2_to_f16x2(cd8_hi, false)};
      mma_f16_16816(o[4 * w + 0], a_j0, phi[mi][0], phi[mi][1]);
      mma_f16_16816(o[4 * w + 1], a_j1, phi[mi][0], phi[mi][1]);
      mma_f16_16816(o[4 * w + 2], a_j2, phi[mi][0], phi[mi][1]);
      mma_f16_16816(o[4 * w + 3], a_j3, phi[mi][0], phi[mi][1]);
      if constexpr (!PACK) {
        mma_f16_16816(o[4 * w + 0], a_j0, plo[mi][0], plo[mi][1]);
        mma_f16_16816(o[4 * w + 1], a_j1, plo[mi][0], plo[mi][1]);
        mma_f16_16816(o[4 * w + 2], a_j2, plo[mi][0], plo[mi][1]);
        mma_f16_16816(o[4 * w + 3], a_j3, plo[mi][0], plo[mi][1]);
      }
    }
  }
}


// The end of one unit: the G <= 4 lo columns added to their hi columns, then
// the output straight from the fragments (one split) or the state through
// shared memory (ring) into the split merge.
template <int G, int NST>
__device__ __forceinline__ void mma_finish(const AttnParams& p, MmaState<G>& st, bool bad, MmaSmemHeader* hdr,
                                           unsigned char* ring, size_t out_row, int row, int h, int split, int nsplit,
                                           int lane) {
  constexpr int D = 128;
  constexpr bool PACK = G <= 4;
  const int g4 = lane >> 2, t4 = lane & 3;
  const bool q_bf16 = p.q_is_bf16 != 0;  // always true here: the tensor-core units take bf16 queries
  auto& m_ref = st.m_ref;
  auto& o = st.o;
  auto& lsum = st.lsum;
  if constexpr (PACK) {
    // add each head's lo columns (lane ^ 2) to its hi columns; their
    // references are the same (equal scores), so the factor is 1 -- it is
    // applied anyway so that the sum never mixes two references
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const float m_lo = __shfl_xor_sync(0xffffffffu, m_ref[hh], 2);
      const float f = m_lo == m_ref[hh] ? 1.0f : ex2(__fsub_rn(m_lo, m_ref[hh]));
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        o[i][hh] = fmaf(__shfl_xor_sync(0xffffffffu, o[i][hh], 2), f, o[i][hh]);
        o[i][2 + hh] = fmaf(__shfl_xor_sync(0xffffffffu, o[i][2 + hh], 2), f, o[i][2 + hh]);
      }
      lsum[hh] = fmaf(__shfl_xor_sync(0xffffffffu, lsum[hh], 2), f, lsum[hh]);
    }
  }

  if (nsplit == 1) {
    // ---- straight from the fragments: out = o * (v_scale / l), 16 bytes a store
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int head = 2 * t4 + hh;
      if (head < G) {
        const float r = __fdiv_rn(p.v_scale_h[PA_HEAD(p, h)], lsum[hh]);
        uint32_t w0[4], w1[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // a unit that hit an error writes zeros
          w0[i] = bad ? 0u : pack_bf16x2(__fmul_rn(o[2 * i][hh], r), __fmul_rn(o[2 * i + 1][hh], r));
          w1[i] = bad ? 0u : pack_bf16x2(__fmul_rn(o[2 * i][2 + hh], r), __fmul_rn(o[2 * i + 1][2 + hh], r));
        }
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + (out_row + head) * D + 16 * g4);
        dst[0] = make_uint4(w0[0], w0[1], w0[2], w0[3]);
        dst[1] = make_uint4(w1[0], w1[1], w1[2], w1[3]);
      }
    }
    return;
  }

  // ---- split row: the state to shared memory in the SIMT unit's layout (one
  // warp), then the same partial publication and split merge
  float* red_acc = reinterpret_cast<float*>(ring);  // [G][D]
  float* red_ml = red_acc + G * D;                  // [G][2]
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int head = 2 * t4 + hh;
    if (head < G) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        red_acc[head * D + 16 * g4 + i] = o[i][hh];
        red_acc[head * D + 16 * g4 + 8 + i] = o[i][2 + hh];
      }
      if (g4 == 0) {
        red_ml[head * 2] = m_ref[hh];
        red_ml[head * 2 + 1] = lsum[hh];
      }
    }
  }
  __syncwarp();
  decode_finish<D, G, KV_E4M3, 1, 32>(p, bad, &hdr->last, red_acc, red_ml, out_row, row, h, split, nsplit, q_bf16,
                                      NST * kMmaStageBytes);
}

template <int G, int NST>
__device__ __forceinline__ void decode_unit_mma(const AttnParams& p, int unit, unsigned char* smem_raw) {
  constexpr int D = 128, ST = kStageTokens;

  const int h = unit % p.Hkv;
  const int rest = unit / p.Hkv;
  const int split = rest % p.max_splits;
  const int row = unit_row(p, rest / p.max_splits);
  if (row >= p.n_rows) return;
  if (p.n_chunks > 0 && row_in_chunk(p, row)) return;

  const int lane = threadIdx.x;
  const int g4 = lane >> 2;  // fragment group: key row (QK), head element block (PV), query head (B operand)
  const int t4 = lane & 3;   // thread in group
  const size_t out_row = static_cast<size_t>(row) * p.Hq + static_cast<size_t>(h) * G;
  // G <= 4: MMA column n >= 4 repeats query head n - 4 and carries the lo
  // parts of its weights (the hi and lo products in one MMA)
  constexpr bool PACK = G <= 4;
  const int qhead = g4 < G ? g4 : ((PACK && g4 >= 4 && g4 - 4 < G) ? g4 - 4 : -1);  // -1: a zero column
  // The query words this lane needs (bf16), loaded first so that their latency
  // overlaps the sequence and page-id lookups: head g4 of the group (head 0
  // stands in for heads >= G), elements 32kb + 4 t4 .. +3 and 32kb + 16 + 4 t4 .. +3.
  uint2 qraw[4][2];
  {
    const uint2* qs = reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(p.q) +
                                                     (out_row + (qhead >= 0 ? qhead : 0)) * D);
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
      qraw[kb][0] = __ldg(qs + 8 * kb + t4);
      qraw[kb][1] = __ldg(qs + 8 * kb + 4 + t4);
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
  const bool q_bf16 = p.q_is_bf16 != 0;  // always true here: the tensor-core units take bf16 queries
  const int P = p.P;

  if (seq < 0 || seq >= p.num_seqs || pos < 0 || pos >= p.max_blocks * P) {
    if (split == 0) {
      for (int i = lane; i < G * D; i += 32) store_out(p.out, q_bf16, out_row * D + i, 0.0f);
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
    for (int n = 0; n < first; ++n) mma_issue_stage(p, hdr, ring, n, n, t_begin, t_end, j0, h, lg_p);
  }
  if (append_here) {  // the row's own K/V, converted, to the pool (and below to the stage)
    uint32_t raw[4] = {kw[0], kw[1], kw[2], kw[3]};
    convert_new<KV_E4M3, 4>(p, h, false, raw, kw);
    raw[0] = vw[0]; raw[1] = vw[1]; raw[2] = vw[2]; raw[3] = vw[3];
    convert_new<KV_E4M3, 4>(p, h, true, raw, vw);
    const int pid = hdr->pid[(pos >> lg_p) - j0];
    if (pid >= 0 && pid < p.num_pages) {
      store_piece<4>(pool_elem(p.k_pool, p, pid, h, pos & (P - 1), 4 * lane, 1), kw);
      store_piece<4>(pool_elem(p.v_pool, p, pid, h, pos & (P - 1), 4 * lane, 1), vw);
    }
  }

  MmaState<G> st;
  mma_prep<G>(p, h, qhead, qraw, st);

  int drain_n = -1;  // the stage a wait gave up on
  for (int n = 0; n < nstage && !unit_bad; ++n) {
    const int s = n % NST;
    bool got = mbar_wait(&hdr->full[s], (n / NST) & 1, p.wait_limit);
    if (p.debug_stall) got = got && mbar_wait(&hdr->stall, 0, p.wait_limit);  // runs out by construction
    if (!__all_sync(0xffffffffu, got)) {
      if (lane == 0) {
        record_error(p.status, ST_TIMEOUT);
        hdr->bad = 1;
      }
      drain_n = n;
      break;
    }
    unsigned char* ks = ring + static_cast<size_t>(s) * kMmaStageBytes;
    unsigned char* vs = ks + ST * 128;
    if (append_here && n == nstage - 1) {  // the row's own slot, as appended: lane l's 4 bytes
      const int r = pos - (t_begin + n * ST);  // sit in 16-byte chunk l / 4 of the swizzled row
      store_piece<4>(ks + sw128(r, lane >> 2) + 4 * (lane & 3), kw);
      store_piece<4>(vs + sw128(r, lane >> 2) + 4 * (lane & 3), vw);
      __syncwarp();
    }
    mma_stage<G>(st, ks, vs, min(ST, t_end - (t_begin + n * ST)), lane);
    // ---- release the slot and refill it
    __syncwarp();
    if (lane == 0 && n + NST < nstage) {
      fence_proxy_async();
      mma_issue_stage(p, hdr, ring, n + NST, s, t_begin, t_end, j0, h, lg_p);
    }
  }
  // After a wait gave up on stage n, stages n .. n + NST - 1 may still be in
  // flight: let them land before the ring is reused.
  if (drain_n >= 0 && lane == 0) {
    for (int m = drain_n; m < min(drain_n + NST, nstage); ++m)
      mbar_wait(&hdr->full[m % NST], (m / NST) & 1, kDrainWaitLimit);
  }
  __syncwarp();
  const bool bad = hdr->bad != 0;
  mma_finish<G, NST>(p, st, bad, hdr, ring, out_row, row, h, split, nsplit, lane);
}

template <int G, int NST>
__global__ void __launch_bounds__(32, 8) decode_mma_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(128) unsigned char smem[];  // aligned to 1024 by hand in the unit
  decode_unit_mma<G, NST>(p, static_cast<int>(blockIdx.x), smem);
}

// ------------------------------------------------------------ row groups --
//
// Row-tiled staging of shared prefix pages ("GPU inference engine
// engineering", section "The same bits in any batch": a shared prompt prefix
// staged once for eight rows).  A CTA of RG warps takes RG consecutive rows of
// the call for one kv head and split; warp w runs row RG b + w with the
// one-warp unit's arithmetic (mma_prep, mma_stage, mma_finish on the same
// bytes), so every output bit is the one-warp unit's.  What changes is where
// a stage's bytes come from:
//   * The group's shared stages are its leading stages whose page ids are the
//     same for every active row of the group, none of them a row's last stage
//     (which may be partial, or hold the row's own appended key).  They are
//     copied once, into the ring of the first active warp (the leader), and
//     every active warp reads them there; the last of the NP readers of a slot
//     refills it with the leader's next stage.
//   * Each row's other stages arrive in its own ring (the leader's in its own
//     ring after the shared ones); every warp issues its first copies at the
//     start, so they overlap the shared stages.
// Rows share pages only when the caller places rows of one prefix next to
// one another (a scheduler that groups its batches by prefix); a group whose
// rows share nothing runs as RG one-warp units side by side.  Every wait is
// bounded; a warp that gives up records PA_ERR_TIMEOUT, and the copies still
// in flight in any ring are drained before the CTA's shared memory is left.
struct MmaGroupHeader {
  int32_t done[kMaxStages];  // reads of each shared slot, a running count (every NP-th frees it)
  int32_t issued[8];         // stages issued into each warp's ring
  int32_t nst[8];            // stages each warp runs (0: none)
  int32_t t_end[8];          // end of each warp's key range
  int32_t waits[8];          // 1: the warp's row reads rows a preceding append launch writes
  int32_t S, leader, np, lwait, timeout;
};

template <int G, int NST, int RG>
struct MmaGroupGeom {
  static constexpr int THREADS = 32 * RG;
  static constexpr size_t SLICE = mma_header_bytes() + static_cast<size_t>(NST) * kMmaStageBytes;  // per warp
  static constexpr size_t SMEM = 1024 + 1024 + RG * SLICE;
  // CTAs an SM's 228 KB of shared memory holds (1 KB reserved per CTA): the
  // register budget the compiler is held to
  static constexpr int MIN_CTAS = static_cast<int>((228 * 1024) / (SMEM + 1024)) > 0
                                      ? static_cast<int>((228 * 1024) / (SMEM + 1024)) : 1;
  static_assert(RG == 2 || RG == 4 || RG == 8, "rows per group");
  static_assert(sizeof(MmaGroupHeader) <= 1024, "group header");
};

template <int G, int NST, int RG>
__global__ void __launch_bounds__(32 * RG, MmaGroupGeom<G, NST, RG>::MIN_CTAS) decode_mma_group_kernel(const __grid_constant__ AttnParams p) {
  constexpr int D = 128, ST = kStageTokens;
  using Geo = MmaGroupGeom<G, NST, RG>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  MmaGroupHeader* grp = reinterpret_cast<MmaGroupHeader*>(smem);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto slice_hdr = [&](int i) { return reinterpret_cast<MmaSmemHeader*>(smem + 1024 + i * Geo::SLICE); };
  auto slice_ring = [&](int i) { return smem + 1024 + i * Geo::SLICE + mma_header_bytes(); };
  MmaSmemHeader* hdr = slice_hdr(w);
  unsigned char* ring = slice_ring(w);

  const int h = static_cast<int>(blockIdx.x) % p.Hkv;
  const int rest = static_cast<int>(blockIdx.x) / p.Hkv;
  const int split = rest % p.max_splits;
  const int row = (rest / p.max_splits) * RG + w;
  const bool real = row < p.n_rows && !(p.n_chunks > 0 && row_in_chunk(p, row));

  const int g4 = lane >> 2, t4 = lane & 3;
  const size_t out_row = static_cast<size_t>(row) * p.Hq + static_cast<size_t>(h) * G;
  constexpr bool PACK = G <= 4;
  const int qhead = g4 < G ? g4 : ((PACK && g4 >= 4 && g4 - 4 < G) ? g4 - 4 : -1);
  uint2 qraw[4][2];
  bool own_row = false;
  uint32_t kw[4] = {0u, 0u, 0u, 0u}, vw[4] = {0u, 0u, 0u, 0u};
  int seq = -1, pos = -1;
  if (real) {
    const uint2* qs = reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(p.q) +
                                                     (out_row + (qhead >= 0 ? qhead : 0)) * D);
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
      qraw[kb][0] = __ldg(qs + 8 * kb + t4);
      qraw[kb][1] = __ldg(qs + 8 * kb + 4 + t4);
    }
    own_row = row_appends_itself(p, row);
    if (own_row) {
      load_new_raw<4>(p, row, h, 4 * lane, false, kw);
      load_new_raw<4>(p, row, h, 4 * lane, true, vw);
    }
    seq = __ldg(p.seq_ids + row);
    pos = __ldg(p.positions + row);
  } else {
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) qraw[kb][0] = qraw[kb][1] = make_uint2(0u, 0u);
  }
  const bool q_bf16 = p.q_is_bf16 != 0;  // always true here: the tensor-core units take bf16 queries
  const int P = p.P;
  const int lg_p = 31 - __clz(P);

  // this warp's unit: nstage = 0 when it has none (past the rows, a tile
  // chunk row, out of range, or no keys in this split)
  int nstage = 0, nsplit = 1, t_begin = split * p.split_tokens, t_end = 0;
  if (real) {
    if (seq < 0 || seq >= p.num_seqs || pos < 0 || pos >= p.max_blocks * P) {
      if (split == 0) {
        for (int i = lane; i < G * D; i += 32) store_out(p.out, q_bf16, out_row * D + i, 0.0f);
        if (lane == 0) record_error(p.status, ST_OUT_OF_RANGE);
      }
    } else {
      const int L = pos + 1;
      nsplit = (L + p.split_tokens - 1) / p.split_tokens;
      if (split < nsplit) {
        t_end = min(L, t_begin + p.split_tokens);
        nstage = (t_end - t_begin + ST - 1) / ST;
      }
    }
  }
  const int j0 = t_begin / P;
  const bool append_here = own_row && nstage > 0 && split == nsplit - 1;

  if (lane == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(&hdr->full[s], 1);
    mbar_init(&hdr->stall, 1);
    hdr->bad = 0;
    hdr->last = 0;
    if (w == 0) {
      for (int s = 0; s < NST; ++s) grp->done[s] = 0;
      grp->timeout = 0;
    }
    grp->issued[w] = 0;
    fence_barrier_init();
  }
  bool unit_bad = false;
  if (nstage > 0) {
    const int npg = (t_end + P - 1) / P - j0;
    const int32_t* bt = p.block_tables + static_cast<size_t>(seq) * p.max_blocks + j0;
    bool bad = false;
    for (int i = lane; i < npg && i < kMaxUnitPages; i += 32) {
      const int pid = __ldg(bt + i);
      bad |= pid < 0 || pid >= p.num_pages;
      hdr->pid[i] = pid;
    }
    unit_bad = __any_sync(0xffffffffu, bad);
    __syncwarp();
    if (unit_bad && lane == 0) {
      hdr->bad = 1;
      record_error(p.status, ST_OUT_OF_RANGE);
    }
  }
  const bool active = nstage > 0 && !unit_bad;  // runs the stage loop
  if (lane == 0) {
    grp->nst[w] = active ? nstage : 0;
    grp->t_end[w] = t_end;
    grp->waits[w] = own_row ? 0 : 1;
  }
  __syncthreads();  // page ids, barriers and the group's table visible to every warp

  // ---- the shared stages: warp 0 compares the page ids of stage n of every
  // active row with the leader's, 32 stages at a time
  if (w == 0) {
    int lead = -1, np = 0, lw = 0, mn = 0x7fffffff;
    for (int i = 0; i < RG; ++i) {
      const int ni = grp->nst[i];
      if (ni > 0) {
        if (lead < 0) lead = i;
        ++np;
        lw |= grp->waits[i];
        mn = min(mn, ni - 1);  // never a row's last stage
      }
    }
    int S = 0;
    if (np >= 2) {
      S = mn;
      const MmaSmemHeader* hl = slice_hdr(lead);
      for (int base = 0; base < mn; base += 32) {
        const int n = base + lane;
        bool same = true;
        if (n < mn) {
          const int a = t_begin + n * ST;
          const int ja = (a >> lg_p) - j0, jb = ((a + ST - 1) >> lg_p) - j0;
          for (int i = 0; i < RG; ++i) {
            if (i == lead || grp->nst[i] == 0) continue;
            const MmaSmemHeader* hi = slice_hdr(i);
            for (int j = ja; j <= jb; ++j) same &= hi->pid[j] == hl->pid[j];
          }
        }
        const unsigned diff = __ballot_sync(0xffffffffu, !same);
        if (diff != 0u) {
          S = base + __ffs(diff) - 1;
          break;
        }
      }
    }
    if (lane == 0) {
      grp->S = S;
      grp->leader = lead;
      grp->np = np;
      grp->lwait = lw;
    }
  }
  __syncthreads();
  const int S = grp->S, lead = grp->leader, NP = grp->np;
  const bool is_lead = w == lead;
  MmaSmemHeader* hl = slice_hdr(lead < 0 ? 0 : lead);
  unsigned char* rl = slice_ring(lead < 0 ? 0 : lead);

  // the pool rows appended by a preceding dependent-launch append are visible
  // from here; the leader also waits when any row of the group does, since it
  // copies the shared stages for all of them
  if (active && (!own_row || (is_lead && S > 0 && grp->lwait != 0))) griddep_wait();
  if (lane == 0 && active) {
    if (is_lead) {
      const int first = min(NST, nstage);
      for (int n = 0; n < first; ++n) mma_issue_stage(p, hdr, ring, n, n, t_begin, t_end, j0, h, lg_p);
      atomicMax(&grp->issued[w], first);
    } else {
      const int first = min(NST, nstage - S);
      for (int k = 0; k < first; ++k) mma_issue_stage(p, hdr, ring, S + k, k, t_begin, t_end, j0, h, lg_p);
      atomicMax(&grp->issued[w], first);
    }
  }
  if (append_here) {  // the row's own K/V, converted, to the pool (and below to its last stage)
    uint32_t raw[4] = {kw[0], kw[1], kw[2], kw[3]};
    convert_new<KV_E4M3, 4>(p, h, false, raw, kw);
    raw[0] = vw[0]; raw[1] = vw[1]; raw[2] = vw[2]; raw[3] = vw[3];
    convert_new<KV_E4M3, 4>(p, h, true, raw, vw);
    const int pid = hdr->pid[(pos >> lg_p) - j0];
    if (pid >= 0 && pid < p.num_pages) {
      store_piece<4>(pool_elem(p.k_pool, p, pid, h, pos & (P - 1), 4 * lane, 1), kw);
      store_piece<4>(pool_elem(p.v_pool, p, pid, h, pos & (P - 1), 4 * lane, 1), vw);
    }
  }

  MmaState<G> st;
  mma_prep<G>(p, h, qhead, qraw, st);

  if (active) {
    const int t_end_lead = grp->t_end[lead], nst_lead = grp->nst[lead];
    for (int n = 0; n < nstage; ++n) {
      const bool in_lead = n < S || is_lead;  // the stage sits in the leader's ring
      MmaSmemHeader* H = in_lead ? hl : hdr;
      unsigned char* R = in_lead ? rl : ring;
      const int k = in_lead ? n : n - S;  // stage index within that ring
      const int s = k % NST;
      bool got = mbar_wait(&H->full[s], (k / NST) & 1, p.wait_limit);
      if (p.debug_stall) got = got && mbar_wait(&hdr->stall, 0, p.wait_limit);  // runs out by construction
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) {
          record_error(p.status, ST_TIMEOUT);
          hdr->bad = 1;
          grp->timeout = 1;
        }
        break;
      }
      unsigned char* ks = R + static_cast<size_t>(s) * kMmaStageBytes;
      unsigned char* vs = ks + ST * 128;
      if (append_here && n == nstage - 1) {  // the row's own slot (never a shared stage)
        const int r = pos - (t_begin + n * ST);
        store_piece<4>(ks + sw128(r, lane >> 2) + 4 * (lane & 3), kw);
        store_piece<4>(vs + sw128(r, lane >> 2) + 4 * (lane & 3), vw);
        __syncwarp();
      }
      mma_stage<G>(st, ks, vs, min(ST, t_end - (t_begin + n * ST)), lane);
      // ---- release the slot; a shared slot is refilled by its last reader
      __syncwarp();
      if (lane == 0) {
        if (n < S) {
          __threadfence_block();
          if ((atomicAdd(&grp->done[s], 1) + 1) % NP == 0 && n + NST < nst_lead) {
            fence_proxy_async();
            mma_issue_stage(p, hl, rl, n + NST, s, t_begin, t_end_lead, j0, h, lg_p);
            atomicMax(&grp->issued[lead], n + NST + 1);
          }
        } else if (n + NST < nstage) {
          fence_proxy_async();
          mma_issue_stage(p, hdr, ring, n + NST, s, t_begin, t_end, j0, h, lg_p);
          atomicMax(&grp->issued[w], k + NST + 1);
        }
      }
    }
  }
  // Every warp is out of its loop: the leader's ring is no longer read.  After
  // a wait gave up, the last NST stages issued into each ring may still be in
  // flight: let them land before the ring is reused or left.
  __syncthreads();
  if (grp->timeout != 0 && lane == 0) {
    const int iss = grp->issued[w];
    for (int m = max(0, iss - NST); m < iss; ++m) mbar_wait(&hdr->full[m % NST], (m / NST) & 1, kDrainWaitLimit);
  }
  __syncwarp();
  if (nstage > 0) mma_finish<G, NST>(p, st, hdr->bad != 0, hdr, ring, out_row, row, h, split, nsplit, lane);
}

// Devices on which decode_mma_kernel<G, NST> may use its dynamic shared memory.
template <int G, int NST>
std::atomic<unsigned long long>& mma_smem_done() {
  static std::atomic<unsigned long long> done{0};
  return done;
}

template <int G, int NST>
cudaError_t launch_decode_mma_nst(const AttnParams& p, cudaStream_t stream, unsigned units) {
  using Geo = MmaGeom<G, NST>;
  const cudaError_t ea = allow_dynamic_smem(decode_mma_kernel<G, NST>, mma_smem_done<G, NST>(), Geo::SMEM);
  if (ea != cudaSuccess) return ea;
  const cudaError_t e = launch_kernel(decode_mma_kernel<G, NST>, dim3(units), dim3(Geo::THREADS), Geo::SMEM, stream,
                                      p.dependent != 0, p);
  count_launch();
  return e;
}

// Row groups (opt-in): ceil(n_rows / RG) groups per (split, kv head), two
// ring slots per warp.
template <int G, int NST, int RG>
std::atomic<unsigned long long>& mma_group_smem_done() {
  static std::atomic<unsigned long long> done{0};
  return done;
}

template <int G, int RG>
cudaError_t launch_decode_mma_group(const AttnParams& p, cudaStream_t stream) {
  constexpr int NST = 2;
  using Geo = MmaGroupGeom<G, NST, RG>;
  const long long groups = (static_cast<long long>(p.n_rows) + RG - 1) / RG * p.max_splits * p.Hkv;
  if (groups <= 0) return cudaSuccess;
  if (groups > 0x7fffffffLL) return cudaErrorNotSupported;
  const cudaError_t ea =
      allow_dynamic_smem(decode_mma_group_kernel<G, NST, RG>, mma_group_smem_done<G, NST, RG>(), Geo::SMEM);
  if (ea != cudaSuccess) return ea;
  const cudaError_t e = launch_kernel(decode_mma_group_kernel<G, NST, RG>, dim3(static_cast<unsigned>(groups)),
                                      dim3(Geo::THREADS), Geo::SMEM, stream, p.dependent != 0, p);
  count_launch();
  return e;
}

// Units resident on the GPU at once with an NST-slot ring (from the shared
// memory each one-warp CTA takes), queried once.
template <int G, int NST>
long long mma_resident_units() {
  static std::atomic<long long> cache[64];  // per device: resident CTAs + 1, 0 until known
  return resident_ctas(decode_mma_kernel<G, NST>, cache, mma_smem_done<G, NST>(), 32, MmaGeom<G, NST>::SMEM);
}

// The ring depth follows the number of units: many short units want many
// resident CTAs (two slots each); few long ones want each CTA to keep more
// copies in flight.  Take the deepest ring whose CTAs all fit on the GPU at
// once, else two slots.  The depth changes no arithmetic: a row's output bits
// do not depend on it.
template <int G>
cudaError_t launch_decode_mma_inst(const AttnParams& p, cudaStream_t stream) {
  if (p.row_group == 2) return launch_decode_mma_group<G, 2>(p, stream);
  if (p.row_group == 4) return launch_decode_mma_group<G, 4>(p, stream);
  if (p.row_group == 8) return launch_decode_mma_group<G, 8>(p, stream);
  const long long units = static_cast<long long>(p.n_unit_rows) * p.max_splits * p.Hkv;
  if (units <= 0) return cudaSuccess;
  if (units > 0x7fffffffLL) return cudaErrorNotSupported;
  const unsigned u = static_cast<unsigned>(units);
  if (units <= mma_resident_units<G, 8>()) return launch_decode_mma_nst<G, 8>(p, stream, u);
  if (units <= mma_resident_units<G, 4>()) return launch_decode_mma_nst<G, 4>(p, stream, u);
  return launch_decode_mma_nst<G, 2>(p, stream, u);
}

}  // namespace pa
