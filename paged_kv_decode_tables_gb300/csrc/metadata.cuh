// Host-side interface of the metadata kernels.
#pragma once

#include <cuda_runtime.h>

#include "../../include/paged_kv.h"
#include "pkv_ptx.cuh"

namespace pkv {

pkv_status_t launch_copy_page_indices(int32_t *page_indices, int64_t capacity,
                                      const int32_t *block_table, int32_t num_cols, int64_t s0,
                                      int64_t s1, const int32_t *cu, int32_t num_reqs,
                                      int32_t *err, cudaStream_t stream);

pkv_status_t launch_num_kv_splits(int32_t *out, const int32_t *seq_lens, int32_t num_seq,
                                  int32_t num_group, int32_t num_head, int32_t num_kv_head,
                                  int32_t max_kv_splits, int32_t core_count, cudaStream_t stream);

pkv_status_t launch_decode_metadata(int32_t *page_indices, int64_t capacity,
                                    const int32_t *block_table, int32_t num_cols, int64_t s0,
                                    int64_t s1, const int32_t *cu, int32_t num_reqs,
                                    int32_t *splits, const int32_t *seq_lens, int32_t num_group,
                                    int32_t num_head, int32_t num_kv_head, int32_t max_kv_splits,
                                    int32_t core_count, int32_t *err, cudaStream_t stream);

}  // namespace pkv
