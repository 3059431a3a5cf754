// Host-side interface of the split-KV reduce kernel.
#pragma once

#include <cuda_runtime.h>

#include "../../include/paged_kv.h"
#include "pkv_ptx.cuh"

namespace pkv {

struct ReduceParams {
  void *out;
  int64_t o_s0, o_s1, o_s2;
  const float *tmp, *es, *ml;
  const int32_t *seq_lens;
  const int32_t *splits;  // may be null: fixed partition_size
  int32_t *err;
  int32_t num_seqs, num_heads, head_size, block_size, max_parts, partition_size;
};

pkv_status_t launch_reduce(const ReduceParams &p, pkv_dtype_t out_dtype, cudaStream_t stream);

}  // namespace pkv
