// A launch of causal prefill-chunk tiles only (bf16 q and K/V): every row of
// the call is in a chunk on the tensor-core tile path, so the tile CTAs need
// not share the decode units' shape.  Each CTA has six warps: four own the
// tile's 128 rows (softmax), one issues the key-tile copies and the S MMAs,
// one the value-tile copies and the P.V MMAs, so that no softmax warp waits
// while an MMA is issued ("llm-rs ...", section "Prefill: tensor cores,
// written by hand": prefill is limited by compute).  The per-row arithmetic
// is the mixed launch's (pa_prefill.cuh), so a chunk row's output bits do not
// depend on whether decode rows share its call.
#include "pa_prefill.cuh"

namespace pa {

template <int D, int G>
__global__ void __launch_bounds__(192, 1) prefill_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(128) unsigned char smem[];  // aligned to 1024 by hand in the tile
  prefill_tile<D, G, true>(p, static_cast<int>(blockIdx.x), smem);
}

template <int D, int G>
cudaError_t launch_prefill_inst(const AttnParams& p, cudaStream_t stream) {
  const size_t smem = PrefillLayout<D, true>::BYTES;
  static std::atomic<unsigned long long> smem_done{0};  // devices on which the size is allowed
  const cudaError_t ea = allow_dynamic_smem(prefill_kernel<D, G>, smem_done, smem);
  if (ea != cudaSuccess) return ea;
  if (p.n_prefill_ctas <= 0) return cudaSuccess;
  const cudaError_t e = launch_kernel(prefill_kernel<D, G>, dim3(static_cast<unsigned>(p.n_prefill_ctas)), dim3(192),
                                      smem, stream, p.dependent != 0, p);
  count_launch();
  return e;
}

cudaError_t launch_prefill_bf16(const AttnParams& p, cudaStream_t stream) {
  const int G = p.Hq / p.Hkv;
#define PA_PREFILL_CASE(DD, GG) \
  if (p.D == DD && G == GG) return launch_prefill_inst<DD, GG>(p, stream);
  PA_PREFILL_CASE(128, 1)
  PA_PREFILL_CASE(128, 2)
  PA_PREFILL_CASE(128, 3)
  PA_PREFILL_CASE(128, 4)
  PA_PREFILL_CASE(128, 5)
  PA_PREFILL_CASE(128, 6)
  PA_PREFILL_CASE(128, 7)
  PA_PREFILL_CASE(128, 8)
  PA_PREFILL_CASE(64, 1)
  PA_PREFILL_CASE(64, 2)
  PA_PREFILL_CASE(64, 3)
  PA_PREFILL_CASE(64, 4)
  PA_PREFILL_CASE(64, 5)
  PA_PREFILL_CASE(64, 6)
  PA_PREFILL_CASE(64, 7)
  PA_PREFILL_CASE(64, 8)
#undef PA_PREFILL_CASE
  return cudaErrorNotSupported;
}

}  // namespace pa
