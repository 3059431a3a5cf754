// Host side of the tensor-memory decode kernel over fp8 caches: eligibility,
// instance selection and launch.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/paged_kv.h"
#include "attention_fp8_tc.cuh"
#include "attention_launch.cuh"
#include "pkv_launch.cuh"

namespace pkv {

namespace {

template <typename T, typename KV, int GP>
pkv_status_t launch_tc_instance(const AttnParams &p, dim3 grid, cudaStream_t stream) {
  using Cfg = TcCfg<T, GP>;
  static std::atomic<unsigned long long> done{0};
  auto kernel = paged_attention_fp8_tc_kernel<T, KV, GP>;
  if (!detail::ensure_smem_attr(kernel, Cfg::kSmemBytes, done)) return PKV_ERR_CUDA;
  return launch_programmatic(kernel, grid, dim3(kTcThreads), Cfg::kSmemBytes, stream, p) ==
                 cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

template <typename T, typename KV>
pkv_status_t launch_tc_t(const AttnParams &p, int gp, dim3 grid, cudaStream_t stream) {
  return gp == 4 ? launch_tc_instance<T, KV, 4>(p, grid, stream)
                 : launch_tc_instance<T, KV, 8>(p, grid, stream);
}

}  // namespace

bool fp8_tc_eligible(const pkv_decode_args_t *a) {
  if (a->kv_cache_dtype != PKV_KV_FP8_E4M3 && a->kv_cache_dtype != PKV_KV_FP8_E5M2) return false;
  if (a->dtype != PKV_F16 && a->dtype != PKV_BF16) return false;
  return a->head_size == kTcD && a->block_size == kTcBS;
}

pkv_status_t launch_attention_fp8_tc(const pkv_decode_args_t *a, const AttnParams &p, dim3 grid,
                                     cudaStream_t stream) {
  // Query heads per CTA: up to 4, or 5..8 (a kv head's group is served 8 at a time).
  const int gp = p.group <= 4 ? 4 : 8;
  const bool e5 = a->kv_cache_dtype == PKV_KV_FP8_E5M2;
  if (a->dtype == PKV_BF16)
    return e5 ? launch_tc_t<__nv_bfloat16, fp8_e5m2_t>(p, gp, grid, stream)
              : launch_tc_t<__nv_bfloat16, fp8_e4m3_t>(p, gp, grid, stream);
  return e5 ? launch_tc_t<__half, fp8_e5m2_t>(p, gp, grid, stream)
            : launch_tc_t<__half, fp8_e4m3_t>(p, gp, grid, stream);
}

}  // namespace pkv
