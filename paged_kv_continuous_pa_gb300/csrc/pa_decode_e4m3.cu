// Decode-unit kernel instantiations for e4m3 K/V pools (one translation unit
// per K/V dtype so the instantiations compile in parallel).
#include "pa_decode.cuh"

namespace pa {

cudaError_t launch_decode_e4m3(const AttnParams& p, cudaStream_t stream) {
  return launch_decode_dispatch<KV_E4M3>(p, stream);
}


}  // namespace pa
