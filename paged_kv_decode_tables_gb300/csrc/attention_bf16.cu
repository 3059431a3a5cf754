// Paged decode attention instances for element type __nv_bfloat16.
#include "attention_launch.cuh"

namespace pkv {

pkv_status_t launch_attention_bf16(const AttnParams &p, int D, int BS, int W, dim3 g,
                                  cudaStream_t s) {
  switch (D) {
    case 64: return detail::launch_d<__nv_bfloat16, 64>(p, BS, W, g, s);
    case 128: return detail::launch_d<__nv_bfloat16, 128>(p, BS, W, g, s);
    case 256: return detail::launch_d<__nv_bfloat16, 256>(p, BS, W, g, s);
    default: return PKV_ERR_UNSUPPORTED;
  }
}

size_t smem_attention_bf16(int D, int BS, int W) {
  switch (D) {
    case 64: return detail::smem_d<__nv_bfloat16, 64>(BS, W);
    case 128: return detail::smem_d<__nv_bfloat16, 128>(BS, W);
    case 256: return detail::smem_d<__nv_bfloat16, 256>(BS, W);
    default: return 0;
  }
}

}  // namespace pkv
