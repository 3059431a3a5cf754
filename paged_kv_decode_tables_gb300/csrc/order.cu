// Launch order of single-pass decode units, longest sequence first.
//
// A single pass launches one CTA per (sequence, kv head group) in sequence
// order, so the batch's last CTAs to start decide when the grid ends.  Taking
// the longest sequences first shortens that tail (longest processing time
// first).  One CTA computes the order with a counting sort over 256 length
// buckets: bucket = (max_len - len) * 256 / (max_len + 1), so bucket 0 holds the
// longest sequences; within a bucket the order is unspecified.  No host sync.
#include <cuda_runtime.h>

#include "../../include/paged_kv.h"
#include "pkv_launch.cuh"
#include "pkv_ptx.cuh"

namespace pkv {

namespace {

constexpr int kOrderThreads = 1024;
constexpr int kBuckets = 256;

__device__ __forceinline__ int bucket_of(int len, int max_len) {
  const int l = len < 0 ? 0 : (len > max_len ? max_len : len);
  return int((int64_t(max_len - l) * kBuckets) / (int64_t(max_len) + 1));
}

__global__ void __launch_bounds__(kOrderThreads)
    order_by_length_kernel(int32_t *order, const int32_t *seq_lens, int n) {
  grid_dependency_wait();
  allow_dependent_launch();
  __shared__ int max_len;
  __shared__ unsigned count[kBuckets];
  const int tid = threadIdx.x;
  if (tid == 0) max_len = 0;
  for (int b = tid; b < kBuckets; b += kOrderThreads) count[b] = 0u;
  __syncthreads();
  int m = 0;
  for (int i = tid; i < n; i += kOrderThreads) m = max(m, seq_lens[i]);
  atomicMax(&max_len, m);
  __syncthreads();
  const int ml = max_len;
  for (int i = tid; i < n; i += kOrderThreads) atomicAdd(&count[bucket_of(seq_lens[i], ml)], 1u);
  __syncthreads();
  // Exclusive prefix sum of the bucket counts: one bucket per thread of the
  // first kBuckets threads, an inclusive scan within each warp by shuffles,
  // then the warps' totals added in.
  __shared__ unsigned warp_total[kBuckets / 32];
  const int lane = tid & 31, w = tid >> 5;
  unsigned c = 0, incl = 0;
  if (tid < kBuckets) {
    c = count[tid];
    incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_total[w] = incl;
  }
  __syncthreads();
  if (tid < kBuckets) {
    unsigned base = 0;
    for (int k = 0; k < w; ++k) base += warp_total[k];
    count[tid] = base + incl - c;  // first position of bucket tid
  }
  __syncthreads();
  for (int i = tid; i < n; i += kOrderThreads) {
    const unsigned pos = atomicAdd(&count[bucket_of(seq_lens[i], ml)], 1u);
    order[pos] = i;
  }
}

}  // namespace

}  // namespace pkv

extern "C" pkv_status_t pkv_order_by_length(int32_t *order, const int32_t *seq_lens,
                                            int32_t num_seqs, pkv_stream_t stream) {
  if (num_seqs < 0) return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (order == nullptr || seq_lens == nullptr) return PKV_ERR_INVALID_ARG;
  const cudaError_t e = pkv::launch_programmatic(
      pkv::order_by_length_kernel, dim3(1), dim3(pkv::kOrderThreads), 0,
      reinterpret_cast<cudaStream_t>(stream), order, seq_lens, int(num_seqs));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
