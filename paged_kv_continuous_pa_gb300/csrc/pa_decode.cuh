// pa_decode.cuh -- the decode-unit kernel: one CTA per (row, kv head, split).
//
// What it computes: for the G query heads of one row that share kv head h,
// the FP32 online softmax over the keys of one split of the row's context,
// reading K/V pages through the row's block table ("Building an LLM runtime
// from scratch on NVIDIA H100", section "Bug #1": pages of K and V are brought
// into shared memory by the bulk-copy engine, the softmax runs in FP32
// registers; "llm-rs ...", section "4. Going down a level: SIMT kernels":
// decode attention split into chunks of positions, each with its own online
// softmax, followed by a cheap merge).
//
// CTA layout: 4 warps, all of them consumers.  The unit's keys are cut into
// 32-token stages; a stage holds those tokens' K and V rows (for one kv head a
// page is contiguous, so a stage is one or two 1-D bulk copies per operand:
// half a 64-token page, a 32-token page, or two 16-token pages), and only the
// valid slots of the last page are copied.  Stages live in a ring of
// shared-memory slots whose `full` mbarrier counts the copied bytes.  Thread 0
// fills the ring at the start; afterwards the LAST warp to finish with a slot
// (a shared-memory counter) issues the copies of the stage that goes there
// next, so no warp ever waits for a slot to drain and no producer warp takes
// registers.  Page ids are read once per unit and range-checked before any
// copy.  No CTA-wide barrier sits inside a warp-dependent branch (the bug the
// H100 page describes cannot occur).
// Work split inside a stage: warp w owns tokens 8w .. 8w+7.  For Q.K, LPT
// lanes share one token and each dots its D / LPT elements with the matching
// slice of the G query vectors held in registers (packed two-wide FMAs, even
// and odd elements summed at the end); a fixed xor-butterfly over the LPT
// lanes completes the dot product.  One online-softmax update covers
// the warp's 8 tokens.  For P.V, PLT lanes share one token and each owns PE
// consecutive output elements.
//
// Determinism: every sum runs in an order fixed by (position, head, element)
// alone -- FMA chains in a fixed order, fixed shuffle trees, a fixed warp order
// when the 4 warps' partial states are merged, and ascending split order in
// the split merge.  The split count is ceil(L / split_tokens), a function of
// the row alone.  So a row's bits do not depend on which other rows share the
// launch, on the grid size, or on where its pages sit in the pool.
#pragma once

#include "pa_device.cuh"

namespace pa {

template <int KVT>
struct KvElt;
template <>
struct KvElt<KV_F32> {
  static constexpr int bytes = 4;
};
template <>
struct KvElt<KV_BF16> {
  static constexpr int bytes = 2;
};
template <>
struct KvElt<KV_E4M3> {
  static constexpr int bytes = 1;
};

// ------------------------------------------------ a row's own K/V append --
//
// In a pa_step, a row outside every chunk the caller listed is the only row
// of its sequence in the step, so no other row reads the slot its append
// writes.  Its attention units therefore append it themselves: the unit of
// its last split (per kv head) loads the row's new key and value when it
// starts, converts them exactly as the append kernel would, stores them in
// the pool, and writes the same bytes over that slot in its own shared-memory
// stage once the stage has landed (the copy may have read the slot before the
// store).  Nothing waits for the append, and such rows wait for no preceding
// launch.

__device__ __forceinline__ bool row_appends_itself(const AttnParams& p, int row) {
  if (!p.fuse_append) return false;
  for (int c = 0; c < p.n_all_chunks; ++c)
    if (row >= p.all_chunk_begin[c] && row < p.all_chunk_end[c]) return false;
  return true;
}

// Elements d0 .. d0 + E - 1 of row `row`, kv head h of the step's new K
// (is_v false) or V, as loaded: E f32 words, or E / 2 words of bf16 pairs.
template <int E>
__device__ __forceinline__ void load_new_raw(const AttnParams& p, int row, int h, int d0, bool is_v,
                                             uint32_t (&raw)[4]) {
  static_assert(E == 2 || E == 4, "elements per lane");
  const size_t i = (static_cast<size_t>(row) * p.Hkv + h) * p.D + d0;
  const void* src = is_v ? p.v_new : p.k_new;
  raw[0] = raw[1] = raw[2] = raw[3] = 0u;
  if (p.in_dtype == KV_F32) {
    const float* f = static_cast<const float*>(src) + i;
    if constexpr (E == 4) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(f));
      raw[0] = a.x; raw[1] = a.y; raw[2] = a.z; raw[3] = a.w;
    } else {
      const uint2 a = __ldg(reinterpret_cast<const uint2*>(f));
      raw[0] = a.x; raw[1] = a.y;
    }
  } else {
    const uint16_t* b = static_cast<const uint16_t*>(src) + i;
    if constexpr (E == 4) {
      const uint2 a = __ldg(reinterpret_cast<const uint2*>(b));
      raw[0] = a.x; raw[1] = a.y;
    } else {
      raw[0] = __ldg(reinterpret_cast<const uint32_t*>(b));
    }
  }
}

// Those elements in the pool's storage format: the input bits when the
// dtypes match, else the append kernel's conversion.  Packed little-endian
// into w (E * element bytes: 2 .. 16).
template <int KVT, int E>
__device__ __forceinline__ void convert_new(const AttnParams& p, int h, bool is_v, const uint32_t (&raw)[4],
                                            uint32_t (&w)[4]) {
  w[0] = w[1] = w[2] = w[3] = 0u;
  const bool in_f32 = p.in_dtype == KV_F32;
  if constexpr (KVT == KV_F32) {
    if (in_f32) {
#pragma unroll
      for (int e = 0; e < E; ++e) w[e] = raw[e];
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) w[e] = __float_as_uint((e & 1) ? bf16hi(raw[e / 2]) : bf16lo(raw[e / 2]));
    }
  } else if constexpr (KVT == KV_BF16) {
    if (in_f32) {
#pragma unroll
      for (int e = 0; e < E; e += 2)
        w[e / 2] = encode_bf16(__uint_as_float(raw[e])) | (encode_bf16(__uint_as_float(raw[e + 1])) << 16);
    } else {
#pragma unroll
      for (int e = 0; e < E / 2; ++e) w[e] = raw[e];
    }
  } else {
    const float scale = is_v ? p.v_scale_h[PA_HEAD(p, h)] : p.k_enc_scale_h[PA_HEAD(p, h)];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float x = in_f32 ? __uint_as_float(raw[e]) : ((e & 1) ? bf16hi(raw[e / 2]) : bf16lo(raw[e / 2]));
      w[0] |= encode_e4m3(x, scale) << (8 * e);
    }
  }
}

// Store BYTES (2 .. 16) bytes of w at dst (aligned to BYTES).
template <int BYTES>
__device__ __forceinline__ void store_piece(void* dst, const uint32_t (&w)[4]) {
  if constexpr (BYTES == 16)
    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  else if constexpr (BYTES == 8)
    *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
  else if constexpr (BYTES == 4)
    *reinterpret_cast<uint32_t*>(dst) = w[0];
  else
    *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(w[0]);
}

// Byte address, in a pool, of element d of slot `slot` of page `page`, kv head h.
__device__ __forceinline__ unsigned char* pool_elem(const void* pool, const AttnParams& p, int page, int h, int slot,
                                                    int d, int elt) {
  const size_t e = ((static_cast<size_t>(page) * p.Hkv + h) * p.P + slot) * p.D + d;
  return const_cast<unsigned char*>(static_cast<const unsigned char*>(pool)) + e * elt;
}

// Compile-time geometry of one decode instantiation.
//   QK layout: LPT lanes share one token; each holds D / LPT elements of the G
//   query vectors in registers.  A warp scores TPS tokens per sub-step and U
//   sub-steps cover its 8 tokens of a 32-token stage.
//   PV layout: PLT lanes share one token; each owns PE consecutive output
//   elements, so one 4..16-byte shared-memory load feeds G * PE FMAs.
template <int D, int G, int KVT>
struct DecodeGeom {
  static constexpr int ELT = KvElt<KVT>::bytes;
  static constexpr int RB = D * ELT;                     // bytes of one K or V row
  static constexpr int NW = kDecodeWarps;
  static constexpr int THREADS = NW * 32;
  static constexpr int ST = kStageTokens;                // tokens per stage
  static constexpr int WT = ST / NW;                     // tokens per warp per stage
  static constexpr int LPT_MIN = (G * D + 63) / 64;      // keep the query slice at <= 64 registers
  static constexpr int LPT = LPT_MIN <= 4 ? 4 : (LPT_MIN <= 8 ? 8 : 16);
  static constexpr int TPS = 32 / LPT;
  static constexpr int U = WT / TPS;
  static constexpr int EPL = D / LPT;                    // QK elements per lane
  static constexpr int LB = EPL * ELT;
  static constexpr int VEC = LB < 16 ? LB : 16;          // one shared-memory load
  static constexpr int NV = LB / VEC;                    // loads per lane per token
  static constexpr int EPV = VEC / ELT;
  static constexpr int PE_CAP = (32 / G) >= 16 ? 16 : (32 / G) >= 8 ? 8 : (32 / G) >= 4 ? 4 : 2;
  static constexpr int PE_WANT = (D / 32) > PE_CAP ? (D / 32) : PE_CAP;
  static constexpr int PE = (16 / ELT) < PE_WANT ? (16 / ELT) : PE_WANT;  // P.V elements per lane
  static constexpr int PLT = D / PE;                     // P.V lanes per token
  static constexpr int TPV = 32 / PLT;                   // P.V tokens per iteration
  static constexpr int NPV = WT / TPV;                   // P.V iterations per stage
  static constexpr int VB = PE * ELT;                    // P.V bytes per lane
  // Occupancy: four CTAs per SM (128 registers a thread) unless the register
  // estimate says that would spill, then three (168 registers).  The stage ring
  // takes what is left of the SM's shared memory at that occupancy.
  static constexpr int REG_EST = G * EPL + G * PE + U * G + 40;
  static constexpr int MIN_CTAS = REG_EST > 128 ? 3 : kDecodeMinCtas;
  static constexpr int RING_BYTES = MIN_CTAS >= 4 ? kDecodeRingBytes : kDecodeRingBytes3;
  static constexpr int STAGE_BYTES = 2 * kStageTokens * RB;
  static constexpr int STAGES_RAW = RING_BYTES / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW < 2 ? 2 : (STAGES_RAW > kMaxStages ? kMaxStages : STAGES_RAW);
  static_assert(WT % TPS == 0 && WT % TPV == 0 && PLT <= 32, "decode geometry");
  static_assert(D % LPT == 0 && LB % VEC == 0, "head_dim");
};

// Shared-memory header in front of the stage ring (the ring starts 128-byte aligned).
struct DecodeSmemHeader {
  uint64_t full[kMaxStages];   // stage landed (bulk-copy bytes)
  uint64_t stall;              // never completed: the injected-stall test waits here
  int32_t done[kMaxStages];    // warps finished with the stage; the last one refills it
  int32_t bad;                 // a page id was out of range or a wait gave up
  int32_t last;                // this CTA merges the splits of its (row, kv head)
  int32_t issued;              // stages issued so far
  int32_t pid[kMaxUnitPages];  // the unit's physical page ids
  alignas(16) float p[kDecodeWarps][kStageTokens / kDecodeWarps][8];  // softmax weights: [warp][token][head]
  alignas(16) uint32_t own[2][128];  // the row's own new K and V row in pool format (a row that appends itself)
};

__host__ __device__ constexpr size_t decode_header_bytes() { return (sizeof(DecodeSmemHeader) + 127) / 128 * 128; }

// --------------------------------------------------------- vector loads --

template <int BYTES>
struct VecT;
template <>
struct VecT<16> {
  using T = uint4;
};
template <>
struct VecT<8> {
  using T = uint2;
};
template <>
struct VecT<4> {
  using T = uint32_t;
};
template <>
struct VecT<2> {
  using T = uint16_t;
};

// Load BYTES bytes of K/V elements from shared memory and widen them to floats.
template <int KVT, int BYTES>
__device__ __forceinline__ void load_widen(const unsigned char* src, float* f) {
  using T = typename VecT<BYTES>::T;
  T raw = *reinterpret_cast<const T*>(src);
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&raw);
  if constexpr (KVT == KV_F32) {
#pragma unroll
    for (int i = 0; i < BYTES / 4; ++i) f[i] = __uint_as_float(w[i]);
  } else if constexpr (KVT == KV_BF16) {
    if constexpr (BYTES >= 4) {
#pragma unroll
      for (int i = 0; i < BYTES / 4; ++i) {
        f[2 * i] = bf16lo(w[i]);
        f[2 * i + 1] = bf16hi(w[i]);
      }
    } else {
      f[0] = __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&raw)) << 16);
    }
  } else {
    if constexpr (BYTES >= 4) {
#pragma unroll
      for (int i = 0; i < BYTES / 4; ++i) {
        float2 a = e4m3x2_to_float2(w[i] & 0xffffu);
        float2 b = e4m3x2_to_float2(w[i] >> 16);
        f[4 * i] = a.x;
        f[4 * i + 1] = a.y;
        f[4 * i + 2] = b.x;
        f[4 * i + 3] = b.y;
      }
    } else {
      float2 a = e4m3x2_to_float2(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&raw)));
      f[0] = a.x;
      f[1] = a.y;
    }
  }
}

// The G softmax weights of one token from the warp's exchange buffer (a broadcast read).
template <int G>
__device__ __forceinline__ void load_p(const float* src, float (&pv)[G]) {
  if constexpr (G == 1) {
    pv[0] = src[0];
  } else if constexpr (G == 2) {
    const float2 a = *reinterpret_cast<const float2*>(src);
    pv[0] = a.x;
    pv[1] = a.y;
  } else {
#pragma unroll
    for (int i = 0; i < (G + 3) / 4; ++i) {
      const float4 a = *reinterpret_cast<const float4*>(src + 4 * i);
      if (4 * i < G) pv[4 * i] = a.x;
      if (4 * i + 1 < G) pv[4 * i + 1] = a.y;
      if (4 * i + 2 < G) pv[4 * i + 2] = a.z;
      if (4 * i + 3 < G) pv[4 * i + 3] = a.w;
    }
  }
}

// N consecutive query elements starting at element i (i a multiple of N; q
// 16-byte aligned), widened to float, with 4..16-byte loads.
template <int N>
__device__ __forceinline__ void load_q_vec(const void* q, bool bf16, size_t i, float* f) {
  if (bf16) {
    const uint16_t* src = reinterpret_cast<const uint16_t*>(q) + i;
    if constexpr (N % 8 == 0) {
#pragma unroll
      for (int k = 0; k < N / 8; ++k) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(src) + k);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          f[8 * k + 2 * j] = bf16lo(ws[j]);
          f[8 * k + 2 * j + 1] = bf16hi(ws[j]);
        }
      }
    } else {
#pragma unroll
      for (int k = 0; k < N / 2; ++k) {
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(src) + k);
        f[2 * k] = bf16lo(w);
        f[2 * k + 1] = bf16hi(w);
      }
    }
  } else {
    const float* src = reinterpret_cast<const float*>(q) + i;
    if constexpr (N % 4 == 0) {
#pragma unroll
      for (int k = 0; k < N / 4; ++k) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(src) + k);
        f[4 * k] = v.x;
        f[4 * k + 1] = v.y;
        f[4 * k + 2] = v.z;
        f[4 * k + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int k = 0; k < N; ++k) f[k] = __ldg(src + k);
    }
  }
}

__device__ __forceinline__ float load_q(const void* q, bool bf16, size_t i) {
  if (bf16) return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(q)[i]) << 16);
  return reinterpret_cast<const float*>(q)[i];
}

__device__ __forceinline__ void store_out(void* out, bool bf16, size_t i, float v) {
  if (bf16)
    reinterpret_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float*>(out)[i] = v;
}

__device__ __forceinline__ bool row_in_chunk(const AttnParams& p, int row) {
  for (int c = 0; c < p.n_chunks; ++c)
    if (row >= p.chunk_begin[c] && row < p.chunk_end[c]) return true;
  return false;
}

// The row of decode-unit slot `slot`: the slot itself, or its entry in the
// launch order that the preceding launch wrote (this launch depends on it)
__device__ __forceinline__ int unit_row(const AttnParams& p, int slot) {
  if (p.row_order == nullptr) return slot;
  if (slot >= p.n_unit_rows) return p.n_rows;  // no such unit: it exits
  griddep_wait();
  return __ldcg(p.row_order + slot);
}

// Copy the valid token slots of stage n (tokens t_begin + 32n .. +32, clipped
// to t_end) into ring slot s: one bulk copy of K and one of V per page piece.
// P is a power of two (lg_p = log2 P).
template <int RB>
__device__ __forceinline__ void issue_stage(const AttnParams& p, DecodeSmemHeader* hdr, unsigned char* ring, int n,
                                            int s, int t_begin, int t_end, int j0, int h, int lg_p, uint64_t policy) {
  const int a = t_begin + n * kStageTokens;
  const int b = min(t_end, a + kStageTokens);
  unsigned char* ks = ring + static_cast<size_t>(s) * 2 * kStageTokens * RB;
  unsigned char* vs = ks + kStageTokens * RB;
  const size_t head_bytes = static_cast<size_t>(RB) << lg_p;
  const size_t page_bytes = head_bytes * p.Hkv;
  const unsigned char* kb = reinterpret_cast<const unsigned char*>(p.k_pool) + h * head_bytes;
  const unsigned char* vb = reinterpret_cast<const unsigned char*>(p.v_pool) + h * head_bytes;
  mbar_arrive_expect_tx(&hdr->full[s], static_cast<uint32_t>(2 * (b - a) * RB));
  for (int t = a; t < b;) {
    const int page = hdr->pid[(t >> lg_p) - j0];
    const int slot = t & ((1 << lg_p) - 1);
    const int cnt = min((1 << lg_p) - slot, b - t);
    const size_t src = static_cast<size_t>(page) * page_bytes + static_cast<size_t>(slot) * RB;
    const size_t dst = static_cast<size_t>(t - a) * RB;
    bulk_g2s(ks + dst, kb + src, static_cast<uint32_t>(cnt * RB), &hdr->full[s], policy);
    bulk_g2s(vs + dst, vb + src, static_cast<uint32_t>(cnt * RB), &hdr->full[s], policy);
    t += cnt;
  }
}

// A warp's running softmax state and its query slice (all in registers).
template <int G, int NV, int EPV, int PE>
struct DecodeState {
  float qr[G][NV][EPV];  // query slice, pre-scaled into the log2 domain
  float m_ref[G];        // reference maximum (log2 domain)
  float l_run[G];        // this lane's share of the sum of weights
  float acc[G][PE];      // this lane's share of sum(weight * V)
};

// One warp's work on one 32-token stage: scores of its WT tokens, one
// online-softmax update, weights to the warp's exchange buffer, P.V.  FULL:
// every token of the warp is valid (all stages but the last), no masking.
template <int D, int G, int KVT, bool FULL>
__device__ __forceinline__ void decode_stage(DecodeState<G, DecodeGeom<D, G, KVT>::NV, DecodeGeom<D, G, KVT>::EPV,
                                                         DecodeGeom<D, G, KVT>::PE>& st,
                                             const unsigned char* krows, const unsigned char* vrows, float* pbuf,
                                             int n_valid, int tok, int part, int pv_tok, int pv_off) {
  using Geo = DecodeGeom<D, G, KVT>;
  constexpr int LPT = Geo::LPT, TPS = Geo::TPS, U = Geo::U, NV = Geo::NV, EPV = Geo::EPV;
  constexpr int PE = Geo::PE, PLT = Geo::PLT, TPV = Geo::TPV, NPV = Geo::NPV, RB = Geo::RB;
  (void)PLT;
  // ---- scores of the warp's tokens (log2 domain), U sub-steps of TPS tokens
  float sc[U][G];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const unsigned char* krow = krows + static_cast<size_t>(u * TPS + tok) * RB;
    float partial[G][NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int vidx = part + LPT * ((i + tok) % NV);
      float kf[EPV];
      load_widen<KVT, Geo::VEC>(krow + vidx * Geo::VEC, kf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        // even and odd elements in the two halves of a packed FMA, then added
        float2 a = __fmul2_rn(make_float2(st.qr[g][i][0], st.qr[g][i][1]), make_float2(kf[0], kf[1]));
#pragma unroll
        for (int e = 2; e < EPV; e += 2)
          a = __ffma2_rn(make_float2(st.qr[g][i][e], st.qr[g][i][e + 1]), make_float2(kf[e], kf[e + 1]), a);
        partial[g][i] = __fadd_rn(a.x, a.y);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float a = partial[g][0];
#pragma unroll
      for (int i = 1; i < NV; ++i) a = __fadd_rn(a, partial[g][i]);
#pragma unroll
      for (int off = 1; off < LPT; off <<= 1) a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, off));
      sc[u][g] = (FULL || u * TPS + tok < n_valid) ? a : -INFINITY;
    }
  }
  // ---- online softmax: one reference-max update per stage.  The reference
  // only moves when the new maximum exceeds it by more than kRescaleSlack
  // (log2 units), so weights stay <= 2^kRescaleSlack and rescaling is rare.
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float mx = sc[0][g];
#pragma unroll
    for (int u = 1; u < U; ++u) mx = fmaxf(mx, sc[u][g]);
#pragma unroll
    for (int off = LPT; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (mx > __fadd_rn(st.m_ref[g], kRescaleSlack)) {
      const float alpha = ex2(__fsub_rn(st.m_ref[g], mx));
      st.m_ref[g] = mx;
      st.l_run[g] = __fmul_rn(st.l_run[g], alpha);
#pragma unroll
      for (int e = 0; e < PE; e += 2) {
        const float2 a = __fmul2_rn(make_float2(st.acc[g][e], st.acc[g][e + 1]), make_float2(alpha, alpha));
        st.acc[g][e] = a.x;
        st.acc[g][e + 1] = a.y;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {  // scores become weights in place
      sc[u][g] = (FULL || u * TPS + tok < n_valid) ? ex2(__fsub_rn(sc[u][g], st.m_ref[g])) : 0.0f;
      st.l_run[g] = __fadd_rn(st.l_run[g], sc[u][g]);
    }
  }
  __syncwarp();
  if (part == 0) {
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int g = 0; g < G; ++g) pbuf[(u * TPS + tok) * 8 + g] = sc[u][g];
  }
  __syncwarp();
  // ---- acc += p . V over the warp's valid tokens, TPV tokens per iteration
#pragma unroll
  for (int it = 0; it < NPV; ++it) {
    const int t = it * TPV + pv_tok;
    if (FULL || t < n_valid) {
      float vf[PE];
      load_widen<KVT, Geo::VB>(vrows + static_cast<size_t>(t) * RB + pv_off, vf);
      float pv[G];
      load_p<G>(pbuf + t * 8, pv);
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < PE; e += 2) {
          const float2 a = __ffma2_rn(make_float2(pv[g], pv[g]), make_float2(vf[e], vf[e + 1]),
                                      make_float2(st.acc[g][e], st.acc[g][e + 1]));
          st.acc[g][e] = a.x;
          st.acc[g][e + 1] = a.y;
        }
    }
  }
}

// The end of a decode unit, shared by the SIMT and tensor-core units: the NW
// warps' (max, sum, accumulator) states sit in shared memory as red_ml
// [NW][G][2] and red_acc [NW][G][D]; they are merged in warp order.  A row
// with one split writes its output; otherwise each split publishes its
// partial triple to the workspace and the last split to finish merges all of
// them in ascending split order (the counter is left at zero for the next
// call).  ring_bytes: shared memory from red_acc on, for the merge weights.
template <int D, int G, int KVT, int NW, int THREADS>
__device__ __forceinline__ void decode_finish(const AttnParams& p, bool bad, int32_t* last_flag, float* red_acc,
                                              const float* red_ml, size_t out_row, int row, int h, int split,
                                              int nsplit, bool q_bf16, int ring_bytes) {
  const int tid = static_cast<int>(threadIdx.x) % THREADS;  // a warp of a wider CTA runs it as its own
  if (nsplit == 1) {
    for (int i = tid; i < G * D; i += THREADS) {
      const int g = i / D, d = i % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, red_ml[(w * G + g) * 2]);
      float lsum = 0.0f, osum = 0.0f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = ex2(__fsub_rn(red_ml[(w * G + g) * 2], M));
        lsum = fmaf(f, red_ml[(w * G + g) * 2 + 1], lsum);
        osum = fmaf(f, red_acc[(w * G + g) * D + d], osum);
      }
      float o = __fdiv_rn(osum, lsum);
      if (KVT == KV_E4M3) o = __fmul_rn(o, p.v_scale_h[PA_HEAD(p, h)]);
      store_out(p.out, q_bf16, out_row * D + i, bad ? 0.0f : o);
    }
    return;
  }

  // ---- split row: publish this split's partial triple, the last split merges
  for (int i = tid; i < G * D; i += THREADS) {
    const int g = i / D, d = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, red_ml[(w * G + g) * 2]);
    float lsum = 0.0f, osum = 0.0f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float f = ex2(__fsub_rn(red_ml[(w * G + g) * 2], M));
      lsum = fmaf(f, red_ml[(w * G + g) * 2 + 1], lsum);
      osum = fmaf(f, red_acc[(w * G + g) * D + d], osum);
    }
    const size_t slot = (out_row + g) * p.max_splits + split;
    if (bad) {
      M = -INFINITY;
      lsum = 0.0f;
      osum = 0.0f;
    }
    p.ws_o[slot * D + d] = osum;
    if (d == 0) {
      p.ws_ml[slot * 2] = M;
      p.ws_ml[slot * 2 + 1] = lsum;
    }
  }
  __threadfence();
  sync_threads_n<THREADS>();
  int32_t* counter = p.ws_count + static_cast<size_t>(row) * p.Hkv + h;
  if (tid == 0) *last_flag = (atomicAdd(counter, 1) == nsplit - 1) ? 1 : 0;
  sync_threads_n<THREADS>();
  if (!*last_flag) return;
  __threadfence();
  // Merge the splits in ascending order.  The (max, sum) pairs go through
  // shared memory first, so the value loads below are independent and coalesced.
  const size_t slot_base = out_row * p.max_splits;  // slot of (head 0 of the group, split 0)
  float* fbuf = red_acc + NW * G * D + NW * G * 2;   // [G][nsplit] weights, then [G] sums
  const int ring_floats = ring_bytes / 4 - (NW * G * D + NW * G * 2);
  if (G * (nsplit + 1) <= ring_floats) {
    for (int i = tid; i < G * nsplit; i += THREADS) {
      const int g = i / nsplit, sp = i % nsplit;
      fbuf[i] = __ldcg(p.ws_ml + (slot_base + static_cast<size_t>(g) * p.max_splits + sp) * 2);
    }
    sync_threads_n<THREADS>();
    if (tid < G) {
      const int g = tid;
      float M = -INFINITY;
      for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, fbuf[g * nsplit + sp]);
      float lsum = 0.0f;
      for (int sp = 0; sp < nsplit; ++sp) {
        const float f = ex2(__fsub_rn(fbuf[g * nsplit + sp], M));
        fbuf[g * nsplit + sp] = f;
        lsum = fmaf(f, __ldcg(p.ws_ml + (slot_base + static_cast<size_t>(g) * p.max_splits + sp) * 2 + 1), lsum);
      }
      fbuf[G * nsplit + g] = lsum;
    }
    sync_threads_n<THREADS>();
    for (int i = tid; i < G * D; i += THREADS) {
      const int g = i / D, d = i % D;
      const float* o = p.ws_o + (slot_base + static_cast<size_t>(g) * p.max_splits) * D + d;
      float osum = 0.0f;
#pragma unroll 4
      for (int sp = 0; sp < nsplit; ++sp) osum = fmaf(fbuf[g * nsplit + sp], __ldcg(o + static_cast<size_t>(sp) * D), osum);
      float out = __fdiv_rn(osum, fbuf[G * nsplit + g]);
      if (KVT == KV_E4M3) out = __fmul_rn(out, p.v_scale_h[PA_HEAD(p, h)]);
      store_out(p.out, q_bf16, out_row * D + i, out);
    }
  } else {
    for (int i = tid; i < G * D; i += THREADS) {
      const int g = i / D, d = i % D;
      const size_t slot0 = (out_row + g) * p.max_splits;
      float M = -INFINITY;
      for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, __ldcg(p.ws_ml + (slot0 + sp) * 2));
      float lsum = 0.0f, osum = 0.0f;
      for (int sp = 0; sp < nsplit; ++sp) {
        const float f = ex2(__fsub_rn(__ldcg(p.ws_ml + (slot0 + sp) * 2), M));
        lsum = fmaf(f, __ldcg(p.ws_ml + (slot0 + sp) * 2 + 1), lsum);
        osum = fmaf(f, __ldcg(p.ws_o + (slot0 + sp) * D + d), osum);
      }
      float out = __fdiv_rn(osum, lsum);
      if (KVT == KV_E4M3) out = __fmul_rn(out, p.v_scale_h[PA_HEAD(p, h)]);
      store_out(p.out, q_bf16, out_row * D + i, out);
    }
  }
  if (tid == 0) *counter = 0;  // leave the workspace zero-filled for the next call
}

// ------------------------------------------------------------ the unit --

template <int D, int G, int KVT>
__device__ __forceinline__ void decode_unit(const AttnParams& p, int unit, unsigned char* smem) {
  using Geo = DecodeGeom<D, G, KVT>;
  constexpr int NW = Geo::NW, LPT = Geo::LPT, NV = Geo::NV, EPV = Geo::EPV;
  constexpr int PE = Geo::PE, PLT = Geo::PLT, RB = Geo::RB, WT = Geo::WT;
  constexpr int ST = kStageTokens;

  const int h = unit % p.Hkv;
  const int rest = unit / p.Hkv;
  const int split = rest % p.max_splits;
  const int row = unit_row(p, rest / p.max_splits);
  if (row >= p.n_rows) return;
  if (p.n_chunks > 0 && row_in_chunk(p, row)) return;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool own_row = row_appends_itself(p, row);
  const int seq = __ldg(p.seq_ids + row);
  const int pos = __ldg(p.positions + row);
  const bool q_bf16 = p.q_is_bf16 != 0;
  const int P = p.P;

  // A row whose sequence or position is out of range: zeros, error recorded once.
  if (seq < 0 || seq >= p.num_seqs || pos < 0 || pos >= p.max_blocks * P) {
    if (split == 0) {
      for (int i = tid; i < G * D; i += Geo::THREADS)
        store_out(p.out, q_bf16, (static_cast<size_t>(row) * p.Hq + h * G) * D + i, 0.0f);
      if (tid == 0) record_error(p.status, ST_OUT_OF_RANGE);
    }
    return;
  }
  const int L = pos + 1;  // keys 0..pos, own token included
  const int nsplit = (L + p.split_tokens - 1) / p.split_tokens;
  if (split >= nsplit) return;

  const int t_begin = split * p.split_tokens;
  const int t_end = min(L, t_begin + p.split_tokens);
  const int j0 = t_begin / P;
  const int npg = (t_end + P - 1) / P - j0;
  const int nstage = (t_end - t_begin + ST - 1) / ST;
  constexpr int NST = Geo::STAGES;
  const int lg_p = 31 - __clz(P);

  // this row's own K/V append (pa_step): in the unit of the last split, the
  // warp that owns the row's slot in the last stage loads the row's new K and V
  // (E elements a lane), converts them, stores them in the pool, and copies
  // them into that stage once it has landed
  constexpr int E = D / 32;
  constexpr int PB = E * Geo::ELT;  // bytes of a lane's piece
  const bool appends = own_row && split == nsplit - 1;
  // the stage in which this warp writes the row's slot: the last, for the warp
  // that owns the slot there (-1: none)
  const int patch_n = (appends && warp == (pos - (t_begin + (nstage - 1) * ST)) / WT) ? nstage - 1 : -1;
  uint32_t kraw[4], vraw[4];  // that warp's lanes: E elements each of the row's new K and V, loaded now
  if (patch_n >= 0) {
    load_new_raw<E>(p, row, h, E * lane, false, kraw);
    load_new_raw<E>(p, row, h, E * lane, true, vraw);
  }

  DecodeSmemHeader* hdr = reinterpret_cast<DecodeSmemHeader*>(smem);
  unsigned char* ring = smem + decode_header_bytes();
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&hdr->full[s], 1);
      hdr->done[s] = 0;
    }
    mbar_init(&hdr->stall, 1);
    hdr->bad = 0;
    hdr->last = 0;
    hdr->issued = 0;
    fence_barrier_init();
  }
  {
    // the unit's page ids, range-checked before any copy
    const int32_t* bt = p.block_tables + static_cast<size_t>(seq) * p.max_blocks + j0;
    bool bad = false;
    for (int i = tid; i < npg && i < kMaxUnitPages; i += Geo::THREADS) {
      const int pid = __ldg(bt + i);
      bad |= pid < 0 || pid >= p.num_pages;
      hdr->pid[i] = pid;
    }
    sync_threads_n<Geo::THREADS>();  // barrier init and zeroed flags visible before the error flag is raised
    if (bad) {
      hdr->bad = 1;
      record_error(p.status, ST_OUT_OF_RANGE);
    }
  }
  sync_threads_n<Geo::THREADS>();
  const bool unit_bad = hdr->bad != 0;
  const uint64_t policy = l2_policy_evict_first();
  // the pool rows appended by a preceding dependent-launch append are visible
  // from here (a row that appends itself reads nothing that launch writes)
  if (!own_row) griddep_wait();
  if (tid == 0 && !unit_bad) {
    const int first = min(NST, nstage);
    for (int n = 0; n < first; ++n) issue_stage<RB>(p, hdr, ring, n, n, t_begin, t_end, j0, h, lg_p, policy);
    hdr->issued = first;
  }
  if (patch_n >= 0) {
    // the row's own K/V, converted, to the pool, and to the header for this
    // warp's copy into the stage once it has landed
    uint32_t kw[4], vw[4];
    convert_new<KVT, E>(p, h, false, kraw, kw);
    convert_new<KVT, E>(p, h, true, vraw, vw);
    const int pid = hdr->pid[(pos >> lg_p) - j0];
    if (pid >= 0 && pid < p.num_pages) {
      store_piece<PB>(pool_elem(p.k_pool, p, pid, h, pos & (P - 1), E * lane, Geo::ELT), kw);
      store_piece<PB>(pool_elem(p.v_pool, p, pid, h, pos & (P - 1), E * lane, Geo::ELT), vw);
    }
    store_piece<PB>(reinterpret_cast<unsigned char*>(hdr->own[0]) + PB * lane, kw);
    store_piece<PB>(reinterpret_cast<unsigned char*>(hdr->own[1]) + PB * lane, vw);
    __syncwarp();
  }

  // ---- per-warp state
  DecodeState<G, NV, EPV, PE> st;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    st.m_ref[g] = -INFINITY;
    st.l_run[g] = 0.0f;
#pragma unroll
    for (int e = 0; e < PE; ++e) st.acc[g][e] = 0.0f;
  }
  const int tok = lane / LPT;   // QK: token of this lane within a sub-step
  const int part = lane % LPT;  // QK: which slice of the row
  // Query slice in registers, pre-scaled into the log2 domain.  Load i of a
  // lane reads vector part + LPT * ((i + tok) % NV) of the row: rotating by
  // the token spreads one sub-step's tokens over all shared-memory banks.
  {
    const size_t qrow = (static_cast<size_t>(row) * p.Hq + static_cast<size_t>(h) * G) * D;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int vidx = part + LPT * ((i + tok) % NV);
        load_q_vec<EPV>(p.q, q_bf16, qrow + static_cast<size_t>(g) * D + vidx * EPV, st.qr[g][i]);
#pragma unroll
        for (int e = 0; e < EPV; ++e) st.qr[g][i][e] = __fmul_rn(st.qr[g][i][e], p.qk_scale_log2_h[PA_HEAD(p, h)]);
      }
  }
  float* pbuf = &hdr->p[warp][0][0];
  const int pv_tok = lane / PLT;              // P.V: token of this lane within an iteration
  const int pv_off = (lane % PLT) * Geo::VB;  // P.V: byte offset of this lane's elements
  const int wtok0 = warp * WT;                // this warp's first token in a stage

  int s = 0;         // ring slot of stage n
  uint32_t ph = 0;   // phase parity of that slot's current use
  for (int n = 0; n < nstage && !unit_bad; ++n) {
    bool got = mbar_wait(&hdr->full[s], ph, p.wait_limit);
    if (p.debug_stall) got = got && mbar_wait(&hdr->stall, 0, p.wait_limit);  // runs out by construction
    if (!__all_sync(0xffffffffu, got)) {
      if (lane == 0) {
        record_error(p.status, ST_TIMEOUT);
        hdr->bad = 1;
      }
      break;
    }
    const unsigned char* ks = ring + static_cast<size_t>(s) * 2 * ST * RB + static_cast<size_t>(wtok0) * RB;
    const unsigned char* vs = ks + ST * RB;
    if (n == patch_n) {  // the row's own slot, as appended (this warp alone reads it)
      const size_t off = static_cast<size_t>(pos - (t_begin + n * ST) - wtok0) * RB + PB * lane;
      uint32_t w[4] = {0u, 0u, 0u, 0u};
      for (int i = 0; i < PB / 4; ++i) w[i] = hdr->own[0][(PB / 4) * lane + i];
      if constexpr (PB < 4) w[0] = reinterpret_cast<const uint16_t*>(hdr->own[0])[lane];
      store_piece<PB>(const_cast<unsigned char*>(ks) + off, w);
      for (int i = 0; i < PB / 4; ++i) w[i] = hdr->own[1][(PB / 4) * lane + i];
      if constexpr (PB < 4) w[0] = reinterpret_cast<const uint16_t*>(hdr->own[1])[lane];
      store_piece<PB>(const_cast<unsigned char*>(vs) + off, w);
      __syncwarp();
    }
    const int n_valid = min(WT, t_end - (t_begin + n * ST + wtok0));
    if (n_valid == WT)
      decode_stage<D, G, KVT, true>(st, ks, vs, pbuf, WT, tok, part, pv_tok, pv_off);
    else if (n_valid > 0)
      decode_stage<D, G, KVT, false>(st, ks, vs, pbuf, n_valid, tok, part, pv_tok, pv_off);
    // ---- release the slot; the last warp to finish refills it
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&hdr->done[s], 1) == NW - 1) {
        hdr->done[s] = 0;
        const int nn = n + NST;
        if (nn < nstage) {
          fence_proxy_async();
          issue_stage<RB>(p, hdr, ring, nn, s, t_begin, t_end, j0, h, lg_p, policy);
          atomicMax(&hdr->issued, nn + 1);
        }
      }
    }
    if (++s == NST) {
      s = 0;
      ph ^= 1u;
    }
  }
  // each lane summed only its own tokens: complete l over the token lanes and
  // acc over the P.V token groups (fixed xor trees)
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int off = LPT; off < 32; off <<= 1)
      st.l_run[g] = __fadd_rn(st.l_run[g], __shfl_xor_sync(0xffffffffu, st.l_run[g], off));
#pragma unroll
    for (int e = 0; e < PE; ++e)
#pragma unroll
      for (int off = PLT; off < 32; off <<= 1)
        st.acc[g][e] = __fadd_rn(st.acc[g][e], __shfl_xor_sync(0xffffffffu, st.acc[g][e], off));
  }

  sync_threads_n<Geo::THREADS>();
  if (tid == 0) {
    // every issued copy must land before the ring is reused (only matters after a timeout)
    const int issued = hdr->issued;
    for (int n = max(0, issued - NST); n < issued; ++n) mbar_wait(&hdr->full[n % NST], (n / NST) & 1, kDrainWaitLimit);
  }
  sync_threads_n<Geo::THREADS>();

  // ---- merge the 4 warps' states, warp 0 first
  float* red_acc = reinterpret_cast<float*>(ring);  // [NW][G][D]
  float* red_ml = red_acc + NW * G * D;             // [NW][G][2]
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane < PLT) {
#pragma unroll
      for (int e = 0; e < PE; ++e) red_acc[(warp * G + g) * D + lane * PE + e] = st.acc[g][e];
    }
    if (lane == 0) {
      red_ml[(warp * G + g) * 2] = st.m_ref[g];
      red_ml[(warp * G + g) * 2 + 1] = st.l_run[g];
    }
  }
  sync_threads_n<Geo::THREADS>();
  decode_finish<D, G, KVT, NW, Geo::THREADS>(p, hdr->bad != 0, &hdr->last, red_acc, red_ml,
                                             static_cast<size_t>(row) * p.Hq + static_cast<size_t>(h) * G, row, h,
                                             split, nsplit, q_bf16, NST * Geo::STAGE_BYTES);
}

template <int D, int G, int KVT>
__global__ void __launch_bounds__(DecodeGeom<D, G, KVT>::THREADS, DecodeGeom<D, G, KVT>::MIN_CTAS) decode_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  decode_unit<D, G, KVT>(p, static_cast<int>(blockIdx.x) - p.n_prefill_ctas, smem);
}

template <int D, int G, int KVT>
__host__ __device__ constexpr size_t decode_smem_for(int P, int n_stages) {
  using Geo = DecodeGeom<D, G, KVT>;
  (void)P;
  const size_t ring = static_cast<size_t>(n_stages) * 2 * kStageTokens * Geo::RB;
  const size_t merge = static_cast<size_t>(Geo::NW) * G * (D + 2) * sizeof(float);
  return decode_header_bytes() + (ring > merge ? ring : merge);
}

template <int D, int G, int KVT>
cudaError_t launch_decode_inst(const AttnParams& p0, cudaStream_t stream) {
  using Geo = DecodeGeom<D, G, KVT>;
  AttnParams p = p0;
  p.n_stages = Geo::STAGES;
  const size_t smem = decode_smem_for<D, G, KVT>(p.P, p.n_stages);
  static std::atomic<unsigned long long> smem_done{0};  // devices on which the size is allowed
  const cudaError_t ea = allow_dynamic_smem(decode_kernel<D, G, KVT>, smem_done, smem);
  if (ea != cudaSuccess) return ea;
  const long long units = static_cast<long long>(p.n_unit_rows) * p.max_splits * p.Hkv;
  if (units <= 0) return cudaSuccess;
  const cudaError_t e = launch_kernel(decode_kernel<D, G, KVT>, dim3(static_cast<unsigned>(units)), dim3(Geo::THREADS),
                                      smem, stream, p.dependent != 0, p);
  count_launch();
  return e;
}

template <int KVT>
cudaError_t launch_decode_dispatch(const AttnParams& p, cudaStream_t stream) {
  const int G = p.Hq / p.Hkv;
#define PA_DECODE_CASE(DD, GG) \
  if (p.D == DD && G == GG) return launch_decode_inst<DD, GG, KVT>(p, stream);
  PA_DECODE_CASE(128, 1)
  PA_DECODE_CASE(128, 2)
  PA_DECODE_CASE(128, 3)
  PA_DECODE_CASE(128, 4)
  PA_DECODE_CASE(128, 5)
  PA_DECODE_CASE(128, 6)
  PA_DECODE_CASE(128, 7)
  PA_DECODE_CASE(128, 8)
  PA_DECODE_CASE(64, 1)
  PA_DECODE_CASE(64, 2)
  PA_DECODE_CASE(64, 3)
  PA_DECODE_CASE(64, 4)
  PA_DECODE_CASE(64, 5)
  PA_DECODE_CASE(64, 6)
  PA_DECODE_CASE(64, 7)
  PA_DECODE_CASE(64, 8)
#undef PA_DECODE_CASE
  return cudaErrorNotSupported;
}

}  // namespace pa
