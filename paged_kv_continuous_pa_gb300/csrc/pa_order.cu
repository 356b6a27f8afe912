// pa_order.cu -- the order of a call's decode rows as a launch of its own
// (calls without an append launch to carry it; see pa_order.cuh).
#include "pa_order.cuh"

namespace pa {

__global__ void __launch_bounds__(1024) order_rows_kernel(const __grid_constant__ OrderParams o) {
  griddep_launch_dependents();  // the attention that reads the order may start its setup now
  order_rows_block(o);
}

cudaError_t launch_order_rows(const OrderParams& o, cudaStream_t stream) {
  if (o.n_rows <= 0) return cudaSuccess;
  const int threads = o.n_rows >= 1024 ? 1024 : (o.n_rows + 31) / 32 * 32;
  order_rows_kernel<<<1, threads, 0, stream>>>(o);
  count_launch();
  return cudaGetLastError();
}

}  // namespace pa
