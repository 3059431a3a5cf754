// Sliding-window page table for speculative decoding (sglang
// python/sglang/kernels/ops/attention/metadata.py:
// prepare_swa_spec_page_table_triton / _prepare_swa_spec_page_table_kernel).
//
// Output row m (one per draft token, bs * R rows) is request row m / R of
// table A cut to seq_len_a[m / R], followed by row m of table B cut to
// seq_len_b[m]; columns past a table's width read as 0 and columns at or past
// min(la + lb, LEN_A + LEN_B) are left untouched.  One CTA per (row, chunk of
// 1024 columns), four columns per thread.
#include <cuda_runtime.h>

#include "../../include/paged_kv.h"
#include "pkv_launch.cuh"
#include "pkv_ptx.cuh"

namespace pkv {

namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 4;
constexpr int kChunk = kThreads * kPerThread;

__global__ void __launch_bounds__(kThreads) swa_spec_kernel(const pkv_swa_spec_args_t a) {
  grid_dependency_wait();
  allow_dependent_launch();
  const int m = blockIdx.x;
  const int r = m / a.num_draft_tokens;
  int la = a.seq_len_a[int64_t(r) * a.seq_len_a_stride];
  int lb = a.seq_len_b[int64_t(m) * a.seq_len_b_stride];
  if (la < 0 || lb < 0) {
    if (threadIdx.x == 0) flag_error(a.err_flag, 2u);
    la = max(la, 0);
    lb = max(lb, 0);
  }
  const int64_t len_out = int64_t(a.len_a) + a.len_b;
  const int64_t limit = min(int64_t(la) + lb, len_out);
  const int32_t *row_a = a.page_table_a + int64_t(r) * a.a_stride[0];
  const int32_t *row_b = a.page_table_b + int64_t(m) * a.b_stride[0];
  int32_t *dst = a.dst + int64_t(m) * a.dst_stride[0];
  const int64_t base = int64_t(blockIdx.y) * kChunk + threadIdx.x;
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    const int64_t n = base + int64_t(k) * kThreads;
    if (n >= limit) continue;
    int32_t v = 0;
    if (n < la) {
      if (n < a.len_a) v = row_a[n * a.a_stride[1]];
    } else {
      const int64_t j = n - la;
      if (j < a.len_b) v = row_b[j * a.b_stride[1]];
    }
    dst[n * a.dst_stride[1]] = v;
  }
}

}  // namespace

}  // namespace pkv

extern "C" pkv_status_t prepare_swa_spec_page_table(const pkv_swa_spec_args_t *a,
                                                    pkv_stream_t stream) {
  if (a == nullptr) return PKV_ERR_INVALID_ARG;
  if (a->bs < 0 || a->num_draft_tokens < 1 || a->len_a < 0 || a->len_b < 0)
    return PKV_ERR_INVALID_ARG;
  const int64_t rows = int64_t(a->bs) * a->num_draft_tokens;
  const int64_t len_out = int64_t(a->len_a) + a->len_b;
  if (rows == 0 || len_out == 0) return PKV_OK;
  if (!a->dst || !a->seq_len_a || !a->seq_len_b) return PKV_ERR_INVALID_ARG;
  if ((a->len_a > 0 && !a->page_table_a) || (a->len_b > 0 && !a->page_table_b))
    return PKV_ERR_INVALID_ARG;
  const int64_t chunks = (len_out + pkv::kChunk - 1) / pkv::kChunk;
  if (rows > 0x7fffffff || chunks > 65535) return PKV_ERR_UNSUPPORTED;
  return pkv::launch_programmatic(pkv::swa_spec_kernel, dim3(unsigned(rows), unsigned(chunks)),
                                  dim3(pkv::kThreads), 0, reinterpret_cast<cudaStream_t>(stream),
                                  *a) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

extern "C" size_t pkv_swa_spec_args_size(void) { return sizeof(pkv_swa_spec_args_t); }
