// One launch for a step that mixes decode rows and prefill chunks (bf16 q and
// K/V): CTAs [0, n_prefill_ctas) run tensor-core chunk tiles, the others run
// decode units ("GPU inference engine engineering", section "Batching without
// running out of cache": decode rows of many sequences and a slice of a long
// prompt share one launch).  A tile CTA has the decode CTA's shape (4 warps,
// the same shared memory and register budget), so mixing costs the decode
// units no occupancy.  The decode rows run the same units as in a decode-only
// launch, so their bits do not depend on a chunk being present: the SIMT units
// for G <= 2 or D = 64, the tensor-core units (on the CTA's first warp; the
// others leave at once) for D = 128 and G >= 3.  A call whose rows are all
// chunk tiles takes the warp-specialised tile launch instead
// (pa_prefill_bf16.cu), with the same per-row arithmetic.
#include "pa_decode.cuh"
#include "pa_decode_mma_bf16.cuh"
#include "pa_prefill.cuh"

namespace pa {

template <int D, int G>
__global__ void __launch_bounds__(DecodeGeom<D, G, KV_BF16>::THREADS, DecodeGeom<D, G, KV_BF16>::MIN_CTAS)
    mixed_kernel(const __grid_constant__ AttnParams p) {
  static_assert(DecodeGeom<D, G, KV_BF16>::THREADS == kTileM, "a tile CTA has one thread per tile row");
  extern __shared__ __align__(128) unsigned char smem[];  // the tile and tensor-core units align to 1024 by hand
  if (static_cast<int>(blockIdx.x) < p.n_prefill_ctas) {
    prefill_tile<D, G, false>(p, static_cast<int>(blockIdx.x), smem);
  } else {
    // a decode unit never allocates tensor memory: say so at once, or this CTA
    // would keep the SM's other CTA slots empty
    if (threadIdx.x < 32) tc::tmem_relinquish();
    if constexpr (D == 128 && G >= 3) {
      if (threadIdx.x < 32) decode_unit_mma_bf16<G, 2>(p, static_cast<int>(blockIdx.x) - p.n_prefill_ctas, smem);
    } else {
      decode_unit<D, G, KV_BF16>(p, static_cast<int>(blockIdx.x) - p.n_prefill_ctas, smem);
    }
  }
}

template <int D, int G>
cudaError_t launch_mixed_inst(const AttnParams& p0, cudaStream_t stream) {
  using Geo = DecodeGeom<D, G, KV_BF16>;
  AttnParams p = p0;
  p.n_stages = Geo::STAGES;
  const size_t tile_smem = PrefillLayout<D, false>::BYTES;
  const size_t dec_smem = (D == 128 && G >= 3) ? MmaBfGeom<G, 2>::SMEM
                                               : decode_smem_for<D, G, KV_BF16>(p.P, Geo::STAGES);
  const size_t smem = tile_smem > dec_smem ? tile_smem : dec_smem;
  static std::atomic<unsigned long long> smem_done{0};  // devices on which the size is allowed
  const cudaError_t ea = allow_dynamic_smem(mixed_kernel<D, G>, smem_done, smem);
  if (ea != cudaSuccess) return ea;
  const long long ctas = static_cast<long long>(p.n_prefill_ctas) + static_cast<long long>(p.n_unit_rows) * p.max_splits * p.Hkv;
  if (ctas <= 0) return cudaSuccess;
  const cudaError_t e = launch_kernel(mixed_kernel<D, G>, dim3(static_cast<unsigned>(ctas)), dim3(Geo::THREADS), smem,
                                      stream, p.dependent != 0, p);
  count_launch();
  return e;
}

cudaError_t launch_mixed_bf16(const AttnParams& p, cudaStream_t stream) {
  const int G = p.Hq / p.Hkv;
#define PA_MIXED_CASE(DD, GG) \
  if (p.D == DD && G == GG) return launch_mixed_inst<DD, GG>(p, stream);
  PA_MIXED_CASE(128, 1)
  PA_MIXED_CASE(128, 2)
  PA_MIXED_CASE(128, 3)
  PA_MIXED_CASE(128, 4)
  PA_MIXED_CASE(128, 5)
  PA_MIXED_CASE(128, 6)
  PA_MIXED_CASE(128, 7)
  PA_MIXED_CASE(128, 8)
  PA_MIXED_CASE(64, 1)
  PA_MIXED_CASE(64, 2)
  PA_MIXED_CASE(64, 3)
  PA_MIXED_CASE(64, 4)
  PA_MIXED_CASE(64, 5)
  PA_MIXED_CASE(64, 6)
  PA_MIXED_CASE(64, 7)
  PA_MIXED_CASE(64, 8)
#undef PA_MIXED_CASE
  return cudaErrorNotSupported;
}

}  // namespace pa
