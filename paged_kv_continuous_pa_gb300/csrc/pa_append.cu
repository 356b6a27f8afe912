// pa_append.cu -- K/V append: scatter each row's new key and value into slot
// p % P of page block_tables[s][p / P] ("GPU inference engine engineering",
// section "Batching without running out of cache": a paged pool with a block
// table per sequence; rows carry their own sequence and position).
//
// One thread converts and stores 8 consecutive elements of one (row, K|V, kv
// head): a 16- or 32-byte load and a 32-, 16- or 8-byte store, so a warp moves
// whole contiguous rows.  Conversions:
//   f32 -> f32, bf16 -> bf16   copy
//   bf16 -> f32                exact widening
//   f32 -> bf16                round to nearest even (cvt.rn.bf16.f32)
//   f32|bf16 -> fp8 e4m3       IEEE binary32 division by the scale, then
//                              satfinite round-to-nearest-even (cvt.rn.satfinite)
#include "pa_order.cuh"

namespace pa {

__global__ void __launch_bounds__(256) append_kernel(const __grid_constant__ AppendParams p) {
  griddep_launch_dependents();  // an attention launched as a dependent may start its lookups now
  if (p.with_order && blockIdx.x == gridDim.x - 1) {  // the extra CTA: the decode rows' launch order
    order_rows_block(p.order);
    return;
  }
  const long long oct_per_row = static_cast<long long>(p.Hkv) * p.D / 8;  // octets of one K (or V) row
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long rows = p.n_ranges > 0 ? p.range_first[p.n_ranges] : p.n_rows;
  const long long total = rows * 2 * oct_per_row;
  if (idx >= total) return;
  long long row = idx / (2 * oct_per_row);
  if (p.n_ranges > 0) {  // the i-th row of the ranges
    int k = 0;
    while (k + 1 < p.n_ranges && row >= p.range_first[k + 1]) ++k;
    row = p.range_begin[k] + (row - p.range_first[k]);
  }
  const long long rem = idx % (2 * oct_per_row);
  const bool is_v = rem >= oct_per_row;
  const long long oct = is_v ? rem - oct_per_row : rem;  // octet within [Hkv][D]
  const int h = static_cast<int>(oct * 8 / p.D);
  const int d0 = static_cast<int>(oct * 8 % p.D);

  const int seq = __ldg(p.seq_ids + row);
  const int pos = __ldg(p.positions + row);
  if (seq < 0 || seq >= p.num_seqs || pos < 0 || pos >= p.max_blocks * p.P) {
    if (oct == 0 && !is_v) record_error(p.status, ST_OUT_OF_RANGE);
    return;
  }
  const int page = __ldg(p.block_tables + static_cast<long long>(seq) * p.max_blocks + pos / p.P);
  if (page < 0 || page >= p.num_pages) {
    if (oct == 0 && !is_v) record_error(p.status, ST_OUT_OF_RANGE);
    return;
  }
  const int slot = pos % p.P;
  const long long src = (row * p.Hkv + h) * p.D + d0;
  const long long dst = ((static_cast<long long>(page) * p.Hkv + h) * p.P + slot) * p.D + d0;
  const void* in = is_v ? p.v_new : p.k_new;
  void* pool = is_v ? p.v_pool : p.k_pool;

  float x[8];
  if (p.in_dtype == KV_F32) {
    const float4* s4 = reinterpret_cast<const float4*>(static_cast<const float*>(in) + src);
    const float4 a = __ldg(s4), b = __ldg(s4 + 1);
    if (p.kv_dtype == KV_F32) {
      float4* d4 = reinterpret_cast<float4*>(static_cast<float*>(pool) + dst);
      d4[0] = a;
      d4[1] = b;
      return;
    }
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(in) + src));
    if (p.kv_dtype == KV_BF16) {
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(pool) + dst) = w;
      return;
    }
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = bf16lo(ws[i]);
      x[2 * i + 1] = bf16hi(ws[i]);
    }
  }
  if (p.kv_dtype == KV_F32) {
    float4* d4 = reinterpret_cast<float4*>(static_cast<float*>(pool) + dst);
    d4[0] = make_float4(x[0], x[1], x[2], x[3]);
    d4[1] = make_float4(x[4], x[5], x[6], x[7]);
  } else if (p.kv_dtype == KV_BF16) {
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = encode_bf16(x[2 * i]) | (encode_bf16(x[2 * i + 1]) << 16);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(pool) + dst) = make_uint4(o[0], o[1], o[2], o[3]);
  } else {
    const float scale = is_v ? p.v_scale_h[PA_HEAD(p, h)] : p.k_scale_h[PA_HEAD(p, h)];
    uint32_t o[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i / 4] |= encode_e4m3(x[i], scale) << (8 * (i % 4));
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(pool) + dst) = make_uint2(o[0], o[1]);
  }
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  const long long rows = p.n_ranges > 0 ? p.range_first[p.n_ranges] : p.n_rows;
  const long long total = rows * 2 * p.Hkv * p.D / 8;
  if (total <= 0 && !p.with_order) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads + (p.with_order ? 1 : 0);
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  append_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(p);
  count_launch();
  return cudaGetLastError();
}

}  // namespace pa
