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
// CTA layout: warps 0..3 consume, warp 4 produces.
//   producer  one lane issues one 1-D bulk copy per page for K and one for V
//             (a page of one kv head is contiguous: P*D*elt bytes) into a ring
//             of shared-memory stages; completion is counted in bytes on the
//             stage's `full` mbarrier.  The last page of the row copies only its
//             valid slots.  Page ids are read 32 at a time, one per lane, and
//             range-checked before any copy is issued.
//   consumers wait on `full`, compute, then arrive on `empty` (one arrival per
//             warp).  There is no CTA-wide barrier inside the role branches; the
//             only __syncthreads are outside them (the bug the H100 page
//             describes cannot occur).
// Work split inside a page: the page's tokens are cut into steps of TPS
// tokens; step k of the unit's page n goes to warp (n * steps_per_page + k) % 4.
// Within a step, LPT lanes share one token: each lane dots its D / LPT
// elements of K with the matching slice of the G query vectors held in
// registers, and a fixed xor-butterfly over the LPT lanes completes the dot
// product.  For P.V each lane owns D / 32 consecutive output elements.
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

// Compile-time geometry of one decode instantiation.
template <int D, int G, int KVT>
struct DecodeGeom {
  static constexpr int ELT = KvElt<KVT>::bytes;
  static constexpr int RB = D * ELT;                     // bytes of one K or V row
  static constexpr int LPT_MIN = (G * D + 63) / 64;      // keep the query slice at <= 64 registers
  static constexpr int LPT = LPT_MIN <= 4 ? 4 : (LPT_MIN <= 8 ? 8 : 16);  // lanes per token
  static constexpr int TPS = 32 / LPT;                   // tokens per warp step
  static constexpr int EPL = D / LPT;                    // QK elements per lane
  static constexpr int LB = EPL * ELT;                   // QK bytes per lane
  static constexpr int VEC = LB < 16 ? LB : 16;          // one shared-memory load
  static constexpr int NV = LB / VEC;                    // loads per lane per token
  static constexpr int EPV = VEC / ELT;                  // elements per load
  static constexpr int DPL = D / 32;                     // P.V output elements per lane
  static constexpr int VB = DPL * ELT;                   // P.V bytes per lane
  static constexpr int NW = kDecodeWarps;
  static constexpr int THREADS = (NW + 1) * 32;
  static_assert(D % LPT == 0 && D % 32 == 0, "head_dim");
  static_assert(LB % VEC == 0, "vector split");
};

// Shared-memory header in front of the stage ring (stage ring starts at 128-byte alignment).
struct DecodeSmemHeader {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  int32_t bad;    // set when a page id was out of range or a wait gave up
  int32_t last;   // set in the CTA that merges the splits of its (row, kv head)
  float p[kDecodeWarps][8][8];  // softmax weights of one step: [warp][token][head]
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

// ------------------------------------------------------------ the unit --

template <int D, int G, int KVT>
__device__ __forceinline__ void decode_unit(const AttnParams& p, int unit, unsigned char* smem) {
  using Geo = DecodeGeom<D, G, KVT>;
  constexpr int NW = Geo::NW, LPT = Geo::LPT, TPS = Geo::TPS, NV = Geo::NV, EPV = Geo::EPV;
  constexpr int DPL = Geo::DPL, RB = Geo::RB;

  const int h = unit % p.Hkv;
  const int rest = unit / p.Hkv;
  const int split = rest % p.max_splits;
  const int row = rest / p.max_splits;
  if (row >= p.n_rows) return;
  if (p.n_chunks > 0 && row_in_chunk(p, row)) return;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seq = __ldg(p.seq_ids + row);
  const int pos = __ldg(p.positions + row);
  const bool q_bf16 = p.q_is_bf16 != 0;
  const int P = p.P;

  // A row whose sequence or position is out of range: zeros, error recorded once.
  if (seq < 0 || seq >= p.num_seqs || pos < 0 || pos >= p.max_blocks * P) {
    if (split == 0) {
      for (int i = tid; i < G * D; i += blockDim.x)
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
  const int npages = (t_end + P - 1) / P - j0;
  const int nst = p.n_stages;
  const uint32_t page_bytes = static_cast<uint32_t>(P) * RB;

  DecodeSmemHeader* hdr = reinterpret_cast<DecodeSmemHeader*>(smem);
  unsigned char* stages = smem + decode_header_bytes();
  if (tid == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&hdr->full[s], 1);
      mbar_init(&hdr->empty[s], NW);
    }
    hdr->bad = 0;
    hdr->last = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const size_t head_stride = static_cast<size_t>(P) * RB;  // bytes of one (page, kv head)
  const unsigned char* kbase = reinterpret_cast<const unsigned char*>(p.k_pool) + static_cast<size_t>(h) * head_stride;
  const unsigned char* vbase = reinterpret_cast<const unsigned char*>(p.v_pool) + static_cast<size_t>(h) * head_stride;
  const size_t page_stride = head_stride * p.Hkv;

  float m_run[G], l_run[G], acc[G][DPL];

  if (warp == NW) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = l2_policy_evict_first();
    const int32_t* bt = p.block_tables + static_cast<size_t>(seq) * p.max_blocks;
    int issued = 0;
    bool ok = true;
    for (int nb = 0; nb < npages && ok; nb += 32) {
      const int n_mine = nb + lane;
      int pid = 0;
      bool bad = false;
      if (n_mine < npages) {
        pid = __ldg(bt + j0 + n_mine);
        bad = pid < 0 || pid >= p.num_pages;
      }
      const unsigned bad_mask = __ballot_sync(0xffffffffu, bad);
      const int cnt = min(32, npages - nb);
      for (int k = 0; k < cnt; ++k) {
        const int page = __shfl_sync(0xffffffffu, pid, k);
        const int n = nb + k;
        const int s = n % nst, r = n / nst;
        if (lane == 0) {
          if (r > 0 && !mbar_wait(&hdr->empty[s], (r - 1) & 1, p.wait_limit)) {
            record_error(p.status, ST_TIMEOUT);
            hdr->bad = 1;
            ok = false;
          } else if ((bad_mask >> k) & 1u) {
            record_error(p.status, ST_OUT_OF_RANGE);
            hdr->bad = 1;
            mbar_arrive(&hdr->full[s]);  // completes the phase with no data
          } else {
            const int first_tok = (j0 + n) * P;
            const int valid = min(P, t_end - first_tok);
            const uint32_t bytes = static_cast<uint32_t>(valid) * RB;
            unsigned char* ks = stages + static_cast<size_t>(s) * 2 * page_bytes;
            mbar_arrive_expect_tx(&hdr->full[s], 2 * bytes);
            bulk_g2s(ks, kbase + static_cast<size_t>(page) * page_stride, bytes, &hdr->full[s], policy);
            bulk_g2s(ks + page_bytes, vbase + static_cast<size_t>(page) * page_stride, bytes, &hdr->full[s], policy);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        issued = n + 1;
      }
    }
    // Every issued copy must land before this CTA's shared memory is reused.
    if (lane == 0)
      for (int n = max(0, issued - nst); n < issued; ++n) mbar_wait(&hdr->full[n % nst], (n / nst) & 1, kDrainWaitLimit);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers
    const int tok = lane / LPT;   // token of this lane within a step
    const int part = lane % LPT;  // which slice of the row
    // Query slice in registers, pre-scaled into the log2 domain.  Load i of
    // token tok reads vector part + LPT * ((i + tok) % NV) of the row: the
    // rotation by tok spreads one step's tokens over all shared-memory banks.
    float qr[G][NV][EPV];
    {
      const size_t qrow = (static_cast<size_t>(row) * p.Hq + static_cast<size_t>(h) * G) * D;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          const int vidx = part + LPT * ((i + tok) % NV);
#pragma unroll
          for (int e = 0; e < EPV; ++e)
            qr[g][i][e] = __fmul_rn(load_q(p.q, q_bf16, qrow + static_cast<size_t>(g) * D + vidx * EPV + e), p.qk_scale_log2);
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m_run[g] = -INFINITY;
      l_run[g] = 0.0f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[g][e] = 0.0f;
    }
    const int steps_per_page = P / TPS;
    float* pbuf = &hdr->p[warp][0][0];

    for (int n = 0; n < npages; ++n) {
      const int s = n % nst, r = n / nst;
      const bool landed = __all_sync(0xffffffffu, mbar_wait(&hdr->full[s], r & 1, p.wait_limit));
      if (!landed) {
        if (lane == 0) {
          record_error(p.status, ST_TIMEOUT);
          hdr->bad = 1;
        }
        break;
      }
      const unsigned char* ks = stages + static_cast<size_t>(s) * 2 * page_bytes;
      const unsigned char* vs = ks + page_bytes;
      const int page_tok0 = (j0 + n) * P;
      for (int k = 0; k < steps_per_page; ++k) {
        if ((n * steps_per_page + k) % NW != warp) continue;
        const int t0 = page_tok0 + k * TPS;
        const int n_valid = min(TPS, t_end - t0);
        if (n_valid <= 0) break;
        // ---- scores of this step's tokens (log2 domain)
        float sc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) sc[g] = 0.0f;
        const unsigned char* krow = ks + static_cast<size_t>(k * TPS + tok) * RB;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          const int vidx = part + LPT * ((i + tok) % NV);
          float kf[EPV];
          load_widen<KVT, Geo::VEC>(krow + vidx * Geo::VEC, kf);
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < EPV; ++e) sc[g] = fmaf(qr[g][i][e], kf[e], sc[g]);
        }
#pragma unroll
        for (int off = 1; off < LPT; off <<= 1)
#pragma unroll
          for (int g = 0; g < G; ++g) sc[g] = __fadd_rn(sc[g], __shfl_xor_sync(0xffffffffu, sc[g], off));
        const bool valid = tok < n_valid;
        // ---- online softmax update (m is the same in every lane of the warp)
        float pw[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          if (!valid) sc[g] = -INFINITY;
          float mx = sc[g];
#pragma unroll
          for (int off = LPT; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
          if (mx > m_run[g]) {
            const float alpha = exp2f(__fsub_rn(m_run[g], mx));
            m_run[g] = mx;
            l_run[g] = __fmul_rn(l_run[g], alpha);
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[g][e] = __fmul_rn(acc[g][e], alpha);
          }
          pw[g] = valid ? exp2f(__fsub_rn(sc[g], m_run[g])) : 0.0f;
          l_run[g] = __fadd_rn(l_run[g], pw[g]);
        }
        __syncwarp();
        if (part == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g) pbuf[tok * 8 + g] = pw[g];
        }
        __syncwarp();
        // ---- acc += p . V over the step's valid tokens, in token order
        const unsigned char* vrow = vs + static_cast<size_t>(k * TPS) * RB + lane * Geo::VB;
        for (int tt = 0; tt < n_valid; ++tt) {
          float vf[DPL];
          load_widen<KVT, Geo::VB>(vrow + static_cast<size_t>(tt) * RB, vf);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float pv = pbuf[tt * 8 + g];
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[g][e] = fmaf(pv, vf[e], acc[g][e]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&hdr->empty[s]);
    }
    // each lane summed only its own token's weights: add over the token lanes
#pragma unroll
    for (int off = LPT; off < 32; off <<= 1)
#pragma unroll
      for (int g = 0; g < G; ++g) l_run[g] = __fadd_rn(l_run[g], __shfl_xor_sync(0xffffffffu, l_run[g], off));
  }

  __syncthreads();  // all copies landed and consumed: the stage ring is free

  // ---- merge the 4 consumer warps' states, warp 0 first
  float* red_acc = reinterpret_cast<float*>(stages);      // [NW][G][D]
  float* red_ml = red_acc + NW * G * D;                   // [NW][G][2]
  if (warp < NW) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int e = 0; e < DPL; ++e) red_acc[(warp * G + g) * D + lane * DPL + e] = acc[g][e];
      if (lane == 0) {
        red_ml[(warp * G + g) * 2] = m_run[g];
        red_ml[(warp * G + g) * 2 + 1] = l_run[g];
      }
    }
  }
  __syncthreads();
  const bool bad = hdr->bad != 0;
  const size_t out_row = static_cast<size_t>(row) * p.Hq + static_cast<size_t>(h) * G;

  if (nsplit == 1) {
    for (int i = tid; i < G * D; i += blockDim.x) {
      const int g = i / D, d = i % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, red_ml[(w * G + g) * 2]);
      float lsum = 0.0f, osum = 0.0f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = exp2f(__fsub_rn(red_ml[(w * G + g) * 2], M));
        lsum = fmaf(f, red_ml[(w * G + g) * 2 + 1], lsum);
        osum = fmaf(f, red_acc[(w * G + g) * D + d], osum);
      }
      float o = __fdiv_rn(osum, lsum);
      if (KVT == KV_E4M3) o = __fmul_rn(o, p.v_scale);
      store_out(p.out, q_bf16, out_row * D + i, bad ? 0.0f : o);
    }
    return;
  }

  // ---- split row: publish this split's partial triple, the last split merges
  for (int i = tid; i < G * D; i += blockDim.x) {
    const int g = i / D, d = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, red_ml[(w * G + g) * 2]);
    float lsum = 0.0f, osum = 0.0f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float f = exp2f(__fsub_rn(red_ml[(w * G + g) * 2], M));
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
  __syncthreads();
  int32_t* counter = p.ws_count + static_cast<size_t>(row) * p.Hkv + h;
  if (tid == 0) hdr->last = (atomicAdd(counter, 1) == nsplit - 1) ? 1 : 0;
  __syncthreads();
  if (!hdr->last) return;
  __threadfence();
  for (int i = tid; i < G * D; i += blockDim.x) {
    const int g = i / D, d = i % D;
    const size_t slot0 = (out_row + g) * p.max_splits;
    float M = -INFINITY;
    for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, __ldcg(p.ws_ml + (slot0 + sp) * 2));
    float lsum = 0.0f, osum = 0.0f;
    for (int sp = 0; sp < nsplit; ++sp) {
      const float f = exp2f(__fsub_rn(__ldcg(p.ws_ml + (slot0 + sp) * 2), M));
      lsum = fmaf(f, __ldcg(p.ws_ml + (slot0 + sp) * 2 + 1), lsum);
      osum = fmaf(f, __ldcg(p.ws_o + (slot0 + sp) * D + d), osum);
    }
    float o = __fdiv_rn(osum, lsum);
    if (KVT == KV_E4M3) o = __fmul_rn(o, p.v_scale);
    store_out(p.out, q_bf16, out_row * D + i, o);
  }
  if (tid == 0) *counter = 0;  // leave the workspace zero-filled for the next call
}

template <int D, int G, int KVT>
__global__ void __launch_bounds__(DecodeGeom<D, G, KVT>::THREADS, 3) decode_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  decode_unit<D, G, KVT>(p, static_cast<int>(blockIdx.x) - p.n_prefill_ctas, smem);
}

template <int D, int G, int KVT>
size_t decode_smem_for(int P, int n_stages) {
  using Geo = DecodeGeom<D, G, KVT>;
  const size_t ring = static_cast<size_t>(n_stages) * 2 * P * Geo::RB;
  const size_t merge = static_cast<size_t>(Geo::NW) * G * (D + 2) * sizeof(float);
  return decode_header_bytes() + (ring > merge ? ring : merge);
}

template <int D, int G, int KVT>
cudaError_t launch_decode_inst(const AttnParams& p, cudaStream_t stream) {
  const size_t smem = decode_smem_for<D, G, KVT>(p.P, p.n_stages);
  static int attr_bytes = 0;  // largest dynamic shared memory size already allowed
  if (static_cast<int>(smem) > attr_bytes) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, G, KVT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_bytes = static_cast<int>(smem);
  }
  const long long units = static_cast<long long>(p.n_rows) * p.max_splits * p.Hkv;
  if (units <= 0) return cudaSuccess;
  decode_kernel<D, G, KVT><<<static_cast<unsigned>(units), DecodeGeom<D, G, KVT>::THREADS, smem, stream>>>(p);
  count_launch();
  return cudaGetLastError();
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

template <int KVT>
size_t decode_smem_dispatch(int P, int D, int G, int n_stages) {
#define PA_SMEM_CASE(DD, GG) \
  if (D == DD && G == GG) return decode_smem_for<DD, GG, KVT>(P, n_stages);
  PA_SMEM_CASE(128, 1)
  PA_SMEM_CASE(128, 2)
  PA_SMEM_CASE(128, 3)
  PA_SMEM_CASE(128, 4)
  PA_SMEM_CASE(128, 5)
  PA_SMEM_CASE(128, 6)
  PA_SMEM_CASE(128, 7)
  PA_SMEM_CASE(128, 8)
  PA_SMEM_CASE(64, 1)
  PA_SMEM_CASE(64, 2)
  PA_SMEM_CASE(64, 3)
  PA_SMEM_CASE(64, 4)
  PA_SMEM_CASE(64, 5)
  PA_SMEM_CASE(64, 6)
  PA_SMEM_CASE(64, 7)
  PA_SMEM_CASE(64, 8)
#undef PA_SMEM_CASE
  return 0;
}

}  // namespace pa
