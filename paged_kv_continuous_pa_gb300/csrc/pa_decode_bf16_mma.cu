// Tensor-core (mma.sync) decode-unit kernels for bf16 K/V pools with head_dim
// 128 and bf16 queries, G = 3..8 query heads per kv head.
#include "pa_decode_mma_bf16.cuh"

namespace pa {

bool decode_bf16_mma_eligible(int D, int G, bool q_bf16) { return D == 128 && G >= 3 && G <= 8 && q_bf16; }

cudaError_t launch_decode_bf16_mma(const AttnParams& p, cudaStream_t stream) {
  if (p.D != 128) return cudaErrorNotSupported;
  switch (p.Hq / p.Hkv) {
    case 3: return launch_decode_mma_bf16_inst<3>(p, stream);
    case 4: return launch_decode_mma_bf16_inst<4>(p, stream);
    case 5: return launch_decode_mma_bf16_inst<5>(p, stream);
    case 6: return launch_decode_mma_bf16_inst<6>(p, stream);
    case 7: return launch_decode_mma_bf16_inst<7>(p, stream);
    case 8: return launch_decode_mma_bf16_inst<8>(p, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace pa
