// Host-side launcher of the paged decode attention kernel instances.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "../../include/paged_kv.h"
#include "attention_kernel.cuh"
#include "pkv_launch.cuh"

namespace pkv {

// Shared memory a (dtype, head_size, block_size, warps) instance needs, or 0
// when that instance is not built.
size_t attention_smem_bytes(pkv_dtype_t dtype, int head_size, int block_size, int warps);

// Launch one instance on `grid` = (partitions, num_kv_heads, num_seqs).
pkv_status_t launch_attention(pkv_dtype_t dtype, const AttnParams &p, int head_size,
                              int block_size, int warps, dim3 grid, cudaStream_t stream);

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

template <typename T, int D, int BS, int W>
pkv_status_t launch_instance(const AttnParams &p, dim3 grid, cudaStream_t stream) {
  using Cfg = AttnCfg<T, D, BS, W>;
  static std::atomic<unsigned long long> done{0};
  auto kernel = paged_attention_kernel<T, D, BS, W>;
  if (!ensure_smem_attr(kernel, Cfg::kSmemBytes, done)) return PKV_ERR_CUDA;
  return launch_programmatic(kernel, grid, dim3(Cfg::kThreads), Cfg::kSmemBytes, stream, p) ==
                 cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

// Instances are built for WARPS in {1, 2, 4}; a 4-warp instance only when its
// shared memory stays within the per-CTA limit.
template <typename T, int D, int BS, int W>
constexpr bool instance_fits() {
  return AttnCfg<T, D, BS, W>::kSmemBytes <= 200 * 1024;
}

template <typename T, int D, int BS>
pkv_status_t launch_bs(const AttnParams &p, int warps, dim3 grid, cudaStream_t stream) {
  if (warps == 1) return launch_instance<T, D, BS, 1>(p, grid, stream);
  if constexpr (instance_fits<T, D, BS, 2>()) {
    if (warps == 2) return launch_instance<T, D, BS, 2>(p, grid, stream);
  }
  if constexpr (instance_fits<T, D, BS, 4>()) {
    if (warps == 4) return launch_instance<T, D, BS, 4>(p, grid, stream);
  }
  return PKV_ERR_UNSUPPORTED;
}

template <typename T, int D, int BS>
size_t smem_bs(int warps) {
  if (warps == 1) return AttnCfg<T, D, BS, 1>::kSmemBytes;
  if constexpr (instance_fits<T, D, BS, 2>()) {
    if (warps == 2) return AttnCfg<T, D, BS, 2>::kSmemBytes;
  }
  if constexpr (instance_fits<T, D, BS, 4>()) {
    if (warps == 4) return AttnCfg<T, D, BS, 4>::kSmemBytes;
  }
  return 0;
}

template <typename T, int D>
pkv_status_t launch_d(const AttnParams &p, int BS, int W, dim3 g, cudaStream_t s) {
  switch (BS) {
    case 8: return launch_bs<T, D, 8>(p, W, g, s);
    case 16: return launch_bs<T, D, 16>(p, W, g, s);
    case 32: return launch_bs<T, D, 32>(p, W, g, s);
    default: return PKV_ERR_UNSUPPORTED;
  }
}

template <typename T, int D>
size_t smem_d(int BS, int W) {
  switch (BS) {
    case 8: return smem_bs<T, D, 8>(W);
    case 16: return smem_bs<T, D, 16>(W);
    case 32: return smem_bs<T, D, 32>(W);
    default: return 0;
  }
}

}  // namespace detail

// Per-dtype dispatch (one translation unit each).
pkv_status_t launch_attention_f32(const AttnParams &p, int D, int BS, int W, dim3 g, cudaStream_t s);
pkv_status_t launch_attention_f16(const AttnParams &p, int D, int BS, int W, dim3 g, cudaStream_t s);
pkv_status_t launch_attention_bf16(const AttnParams &p, int D, int BS, int W, dim3 g, cudaStream_t s);
size_t smem_attention_f32(int D, int BS, int W);
size_t smem_attention_f16(int D, int BS, int W);
size_t smem_attention_bf16(int D, int BS, int W);

}  // namespace pkv
