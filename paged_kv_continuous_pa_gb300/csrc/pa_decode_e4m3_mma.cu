// Tensor-core (mma.sync) decode-unit kernels for e4m3 K/V pools with head_dim
// 128 and bf16 queries, G = 1..8 query heads per kv head.  The e4m3 -> f16
// conversions, not the MMAs, set the cost per byte, so the unused query-head
// columns of the MMA at small G cost little.
#include "pa_decode_mma.cuh"

namespace pa {

bool decode_e4m3_mma_eligible(int D, int G, bool q_bf16) { return D == 128 && G >= 1 && G <= 8 && q_bf16; }

cudaError_t launch_decode_e4m3_mma(const AttnParams& p, cudaStream_t stream) {
  if (p.D != 128) return cudaErrorNotSupported;
  switch (p.Hq / p.Hkv) {
    case 1: return launch_decode_mma_inst<1>(p, stream);
    case 2: return launch_decode_mma_inst<2>(p, stream);
    case 3: return launch_decode_mma_inst<3>(p, stream);
    case 4: return launch_decode_mma_inst<4>(p, stream);
    case 5: return launch_decode_mma_inst<5>(p, stream);
    case 6: return launch_decode_mma_inst<6>(p, stream);
    case 7: return launch_decode_mma_inst<7>(p, stream);
    case 8: return launch_decode_mma_inst<8>(p, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace pa
