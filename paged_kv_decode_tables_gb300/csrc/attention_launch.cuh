// Host-side launcher of the paged decode attention kernel instances.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <type_traits>

#include "../../include/paged_kv.h"
#include "attention_kernel.cuh"
#include "pkv_launch.cuh"

namespace pkv {

// Launch one instance on `grid` = (partitions, num_kv_heads * sub-groups,
// num_seqs); `kv` selects the cache element format.
pkv_status_t launch_attention(pkv_dtype_t dtype, pkv_kv_cache_dtype_t kv, const AttnParams &p,
                              int head_size, int block_size, int warps, dim3 grid,
                              cudaStream_t stream);

// fp8 caches with head size 128 and block size 16 and f16/bf16 queries run on
// the tensor-memory kernel (attention_fp8_tc.cuh): fp8_tc_eligible tells,
// launch_attention_fp8_tc launches it.
bool fp8_tc_eligible(const pkv_decode_args_t *args);
pkv_status_t launch_attention_fp8_tc(const pkv_decode_args_t *args, const AttnParams &p, dim3 grid,
                                     cudaStream_t stream);

// The host-side argument checks of paged_attention_v2_partition (everything
// but its three scratch pointers), shared with the entry points built on it.
pkv_status_t check_partition_args(const pkv_decode_args_t *args, int32_t max_num_partitions,
                                  int32_t partition_size, const int32_t *num_kv_splits);

namespace detail {

// Opt every launched instance into its dynamic shared memory size, once per
// device (the attribute is per device).
template <typename Kernel>
bool ensure_smem_attr(Kernel kernel, int bytes, std::atomic<unsigned long long> &done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const unsigned long long bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return false;
  done.fetch_or(bit, std::memory_order_acq_rel);
  return true;
}

template <typename T, typename KV, int D, int BS, int W, bool PAIR>
pkv_status_t launch_kernel(const AttnParams &p, dim3 grid, cudaStream_t stream) {
  using Cfg = AttnCfg<KV, D, BS, W>;
  static std::atomic<unsigned long long> done{0};
  auto kernel = paged_attention_kernel<T, KV, D, BS, W, PAIR>;
  if (!ensure_smem_attr(kernel, Cfg::kSmemBytes, done)) return PKV_ERR_CUDA;
  return launch_programmatic(kernel, grid, dim3(Cfg::kThreads), Cfg::kSmemBytes, stream, p) ==
                 cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

// Every body has a column-pair form for groups of at most 4 query heads
// (every CTA then serves the whole group), compiled as its own kernel: one
// kernel holding both forms ran the other form 4 % slower.
template <typename T, typename KV, int D, int BS, int W>
pkv_status_t launch_instance(const AttnParams &p, dim3 grid, cudaStream_t stream) {
  if (p.group <= 4) return launch_kernel<T, KV, D, BS, W, true>(p, grid, stream);
  return launch_kernel<T, KV, D, BS, W, false>(p, grid, stream);
}

// Instances are built for WARPS in {1, 2, 4}; a 4-warp instance only when its
// shared memory stays within the per-CTA limit.
template <typename KV, int D, int BS, int W>
constexpr bool instance_fits() {
  return AttnCfg<KV, D, BS, W>::kSmemBytes <= 200 * 1024;
}

template <typename T, typename KV, int D, int BS>
pkv_status_t launch_bs(const AttnParams &p, int warps, dim3 grid, cudaStream_t stream) {
  if (warps == 1) return launch_instance<T, KV, D, BS, 1>(p, grid, stream);
  if constexpr (instance_fits<KV, D, BS, 2>()) {
    if (warps == 2) return launch_instance<T, KV, D, BS, 2>(p, grid, stream);
  }
  if constexpr (instance_fits<KV, D, BS, 4>()) {
    if (warps == 4) return launch_instance<T, KV, D, BS, 4>(p, grid, stream);
  }
  return PKV_ERR_UNSUPPORTED;
}

template <typename KV, int D, int BS>
size_t smem_bs(int warps) {
  if (warps == 1) return AttnCfg<KV, D, BS, 1>::kSmemBytes;
  if constexpr (instance_fits<KV, D, BS, 2>()) {
    if (warps == 2) return AttnCfg<KV, D, BS, 2>::kSmemBytes;
  }
  if constexpr (instance_fits<KV, D, BS, 4>()) {
    if (warps == 4) return AttnCfg<KV, D, BS, 4>::kSmemBytes;
  }
  return 0;
}

template <typename T, typename KV, int D>
pkv_status_t launch_d(const AttnParams &p, int BS, int W, dim3 g, cudaStream_t s) {
  switch (BS) {
    case 8: return launch_bs<T, KV, D, 8>(p, W, g, s);
    case 16: return launch_bs<T, KV, D, 16>(p, W, g, s);
    case 32: return launch_bs<T, KV, D, 32>(p, W, g, s);
    default: return PKV_ERR_UNSUPPORTED;
  }
}

template <typename KV, int D>
size_t smem_d(int BS, int W) {
  switch (BS) {
    case 8: return smem_bs<KV, D, 8>(W);
    case 16: return smem_bs<KV, D, 16>(W);
    case 32: return smem_bs<KV, D, 32>(W);
    default: return 0;
  }
}

// Head sizes built per element type: 64, 128, 256 (fp32: 64, 128).
template <typename T>
constexpr bool has_d256() {
  return !std::is_same<T, float>::value;
}

template <typename T, typename KV>
pkv_status_t launch_by_d(const AttnParams &p, int D, int BS, int W, dim3 g, cudaStream_t s) {
  switch (D) {
    case 64: return launch_d<T, KV, 64>(p, BS, W, g, s);
    case 128: return launch_d<T, KV, 128>(p, BS, W, g, s);
    case 256:
      if constexpr (has_d256<T>()) return launch_d<T, KV, 256>(p, BS, W, g, s);
      return PKV_ERR_UNSUPPORTED;
    default: return PKV_ERR_UNSUPPORTED;
  }
}

template <typename T, typename KV>
size_t smem_by_d(int D, int BS, int W) {
  switch (D) {
    case 64: return smem_d<KV, 64>(BS, W);
    case 128: return smem_d<KV, 128>(BS, W);
    case 256:
      if constexpr (has_d256<T>()) return smem_d<KV, 256>(BS, W);
      return 0;
    default: return 0;
  }
}

}  // namespace detail

// Per (query dtype, cache format) dispatch, one translation unit each.
#define PKV_DECLARE_ATTENTION(name)                                                      \
  pkv_status_t launch_attention_##name(const AttnParams &p, int D, int BS, int W, dim3 g, \
                                       cudaStream_t s);                                  \
  size_t smem_attention_##name(int D, int BS, int W);
PKV_DECLARE_ATTENTION(f32)
PKV_DECLARE_ATTENTION(f16)
PKV_DECLARE_ATTENTION(bf16)
PKV_DECLARE_ATTENTION(f16_e4m3)
PKV_DECLARE_ATTENTION(f16_e5m2)
PKV_DECLARE_ATTENTION(bf16_e4m3)
PKV_DECLARE_ATTENTION(bf16_e5m2)
#undef PKV_DECLARE_ATTENTION

#define PKV_DEFINE_ATTENTION(name, T, KV)                                                \
  pkv_status_t launch_attention_##name(const AttnParams &p, int D, int BS, int W, dim3 g, \
                                       cudaStream_t s) {                                 \
    return detail::launch_by_d<T, KV>(p, D, BS, W, g, s);                                \
  }                                                                                      \
  size_t smem_attention_##name(int D, int BS, int W) {                                   \
    return detail::smem_by_d<T, KV>(D, BS, W);                                           \
  }

}  // namespace pkv
