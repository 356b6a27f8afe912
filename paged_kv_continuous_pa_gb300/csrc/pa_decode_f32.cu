// Decode-unit kernel instantiations for f32 K/V pools (one translation unit
// per K/V dtype so the instantiations compile in parallel).
#include "pa_decode.cuh"

namespace pa {

cudaError_t launch_decode_f32(const AttnParams& p, cudaStream_t stream) {
  return launch_decode_dispatch<KV_F32>(p, stream);
}

size_t decode_smem_bytes_f32(int P, int D, int G, int n_stages) {
  return decode_smem_dispatch<KV_F32>(P, D, G, n_stages);
}

}  // namespace pa
