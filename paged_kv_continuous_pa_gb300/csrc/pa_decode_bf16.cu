// Decode-unit kernel instantiations for bf16 K/V pools (one translation unit
// per K/V dtype so the instantiations compile in parallel).
#include "pa_decode.cuh"

namespace pa {

cudaError_t launch_decode_bf16(const AttnParams& p, cudaStream_t stream) {
  return launch_decode_dispatch<KV_BF16>(p, stream);
}


}  // namespace pa
