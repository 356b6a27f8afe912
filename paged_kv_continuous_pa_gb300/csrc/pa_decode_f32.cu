// Decode-unit kernel instantiations for f32 K/V pools (one translation unit
// per K/V dtype so the instantiations compile in parallel).
#include "pa_decode.cuh"

namespace pa {

cudaError_t launch_decode_f32(const AttnParams& p, cudaStream_t stream) {
  return launch_decode_dispatch<KV_F32>(p, stream);
}


}  // namespace pa
