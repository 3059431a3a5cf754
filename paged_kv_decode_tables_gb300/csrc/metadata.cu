// Sync-free decode metadata kernels.
//
// copy_page_indices: vLLM PR 35765 ("AITER MLA backend: Avoid CPU sync in
//   _build_decode"), _copy_page_indices_kernel with the review's stride_1
//   change.  One CTA per request row; the row's columns are copied with a
//   block-stride loop (coalesced stores, strided loads).
// compute_num_kv_splits: sglang metadata.py, get_num_kv_splits_triton.  One
//   CTA: block-wide max/min of the lengths, the split formula evaluated once,
//   then every thread writes its sequences' counts.
// prepare_decode_metadata: both of the above in one launch (a warp per
//   256-column segment of a table row, plus one CTA for the split counts).
#include "metadata.cuh"
#include "pkv_launch.cuh"

namespace pkv {

namespace {

constexpr int kCopyThreads = 128;
constexpr int kSplitThreads = 1024;
constexpr int kFusedThreads = 256;  // fused launch: a warp per row segment, one CTA for the splits
constexpr int kSegCols = 256;       // columns of a row segment: eight per lane

__device__ __forceinline__ int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Row i of the page-index copy, its columns shared by `nthreads` threads
// starting at `tid`.
__device__ __forceinline__ void copy_row(int32_t *__restrict__ out, int64_t capacity,
                                         const int32_t *__restrict__ bt, int32_t num_cols,
                                         int64_t s0, int64_t s1, const int32_t *__restrict__ cu,
                                         int32_t *err, int i, int tid, int nthreads) {
  const int64_t start = cu[i];
  int64_t n = int64_t(cu[i + 1]) - start;
  if (start < 0 || n < 0 || n > num_cols) {
    if (tid == 0) flag_error(err, 8u);
    if (start < 0) return;
    n = n < 0 ? 0 : num_cols;
  }
  if (start + n > capacity) {
    if (tid == 0) flag_error(err, 8u);
    n = capacity > start ? capacity - start : 0;
  }
  const int32_t *row = bt + int64_t(i) * s0;
  int32_t *dst = out + start;
  for (int64_t j = tid; j < n; j += nthreads) dst[j] = __ldg(row + j * s1);
}

// Columns [seg * kSegCols, (seg + 1) * kSegCols) of row i of the page-index
// copy, one warp, the lane's eight loads issued before its stores (the same
// checks as copy_row; a bad indptr row is flagged by its segment 0).
__device__ __forceinline__ void copy_row_segment(int32_t *__restrict__ out, int64_t capacity,
                                                 const int32_t *__restrict__ bt, int32_t num_cols,
                                                 int64_t s0, int64_t s1,
                                                 const int32_t *__restrict__ cu, int32_t *err,
                                                 int i, int seg, int lane) {
  const int64_t start = cu[i];
  int64_t n = int64_t(cu[i + 1]) - start;
  const bool report = seg == 0 && lane == 0;
  if (start < 0 || n < 0 || n > num_cols) {
    if (report) flag_error(err, 8u);
    if (start < 0) return;
    n = n < 0 ? 0 : num_cols;
  }
  if (start + n > capacity) {
    if (report) flag_error(err, 8u);
    n = capacity > start ? capacity - start : 0;
  }
  const int64_t j0 = int64_t(seg) * kSegCols;
  if (j0 >= n) return;
  const int32_t *row = bt + int64_t(i) * s0;
  int32_t v[kSegCols / 32];
#pragma unroll
  for (int k = 0; k < kSegCols / 32; ++k) {
    const int64_t j = j0 + lane + 32 * k;
    v[k] = j < n ? __ldg(row + j * s1) : 0;
  }
  int32_t *dst = out + start;
#pragma unroll
  for (int k = 0; k < kSegCols / 32; ++k) {
    const int64_t j = j0 + lane + 32 * k;
    if (j < n) dst[j] = v[k];
  }
}

// log2(x) correctly rounded to float32 through the float64 log2; not
// inlined, so that it runs only when called (the compiler would otherwise be
// free to evaluate it ahead of the branch that needs it).
__device__ __noinline__ float log2_rounded_f32(float x) {
  return __double2float_rn(log2(double(x)));
}

// trunc(core_count * max(r, 1)) in float32, where r is log2(ext_len)
// correctly rounded to float32.  Only that integer matters, so the float64
// log2 (float64 runs at a small fraction of the float32 rate on GB300) is
// needed only near a truncation boundary:
// log2f is within 1 ulp of log2 (its documented bound), so r is one of
// log2f(ext_len) and its two float neighbours; when all three give the same
// integer, that integer is the answer; otherwise r is computed from the
// float64 log2 rounded once.
__device__ __forceinline__ int64_t ext_core_count(float ext_len, float cores) {
  auto ext_of = [cores](float r) -> int64_t {
    return __float2int_rz(__fmul_rn(cores, fmaxf(r, 1.0f)));
  };
  const float y = log2f(ext_len);
  const int64_t e = ext_of(y);
  if (ext_of(nextafterf(y, -INFINITY)) == e && ext_of(nextafterf(y, INFINITY)) == e) return e;
  return ext_of(log2_rounded_f32(ext_len));
}

// The split-count heuristic on one CTA of THREADS threads.
template <int THREADS>
__device__ __forceinline__ void split_counts(int32_t *__restrict__ out,
                                             const int32_t *__restrict__ seq_lens, int32_t num_seq,
                                             int32_t num_group, int32_t num_head,
                                             int32_t num_kv_head, int32_t max_kv_splits,
                                             int32_t core_count) {
  __shared__ int red_max[THREADS / 32], red_min[THREADS / 32];
  __shared__ int64_t chunk[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int mx = 1, mn = 0x7fffffff;
  for (int s = tid; s < num_seq; s += THREADS) {
    const int L = max(seq_lens[s], 1);
    mx = max(mx, L);
    mn = min(mn, L);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  if (lane == 0) {
    red_max[warp] = mx;
    red_min[warp] = mn;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < THREADS / 32; ++w) {
      mx = max(mx, red_max[w]);
      mn = min(mn, red_min[w]);
    }
    int64_t mx64 = mx, mn64 = mn;
    if (mx64 * 8 < mn64 * 10) mn64 = mx64;
    const int64_t s1 = min(cdiv64(mx64, mn64), int64_t(max_kv_splits));
    const int64_t c1 = cdiv64(mx64, s1);
    // The one float32 step: log2(max_len / 64) rounded to float32, times the
    // core count in float32, truncated toward zero.
    const float ext_len = __fdiv_rn(__int2float_rn(mx), 64.0f);
    const int64_t ext = ext_core_count(ext_len, __int2float_rn(core_count));
    const int kv_group = num_head / num_kv_head;
    int64_t token_grid;
    if (kv_group == 1) {
      token_grid = int64_t(num_seq) * num_group * num_head;
    } else {
      const int block_h = min(16, kv_group);
      token_grid = int64_t(num_seq) * num_group * cdiv64(num_head, block_h);
    }
    const int64_t s2 = min(cdiv64(ext, token_grid), int64_t(max_kv_splits));
    const int64_t c2 = cdiv64(mx64, s2);
    chunk[0] = c1;
    chunk[1] = c2;
  }
  __syncthreads();
  const int64_t c1 = chunk[0], c2 = chunk[1];
  for (int s = tid; s < num_seq; s += THREADS) {
    const int64_t L = max(seq_lens[s], 0);
    const int v = int(max(cdiv64(L, c1), cdiv64(L, c2)));
    for (int i = 0; i < num_group; ++i) out[int64_t(s) * num_group + i] = v;
  }
}

__global__ void __launch_bounds__(kCopyThreads)
    copy_page_indices_kernel(int32_t *__restrict__ out, int64_t capacity,
                             const int32_t *__restrict__ bt, int32_t num_cols, int64_t s0,
                             int64_t s1, const int32_t *__restrict__ cu, int32_t *err) {
  grid_dependency_wait();
  allow_dependent_launch();
  copy_row(out, capacity, bt, num_cols, s0, s1, cu, err, blockIdx.x, threadIdx.x, kCopyThreads);
}

__global__ void __launch_bounds__(kSplitThreads)
    num_kv_splits_kernel(int32_t *__restrict__ out, const int32_t *__restrict__ seq_lens,
                         int32_t num_seq, int32_t num_group, int32_t num_head,
                         int32_t num_kv_head, int32_t max_kv_splits, int32_t core_count) {
  grid_dependency_wait();
  allow_dependent_launch();
  split_counts<kSplitThreads>(out, seq_lens, num_seq, num_group, num_head, num_kv_head,
                              max_kv_splits, core_count);
}

// Both metadata steps in one grid: blocks [0, copy_blocks) copy table rows (a
// warp per 256-column segment, so long rows do not set the grid's length),
// the last block computes the split counts.
__global__ void __launch_bounds__(kFusedThreads)
    decode_metadata_kernel(int32_t *__restrict__ page_indices, int64_t capacity,
                           const int32_t *__restrict__ bt, int32_t num_cols, int64_t s0,
                           int64_t s1, const int32_t *__restrict__ cu, int32_t num_reqs,
                           int32_t *__restrict__ splits, const int32_t *__restrict__ seq_lens,
                           int32_t num_group, int32_t num_head, int32_t num_kv_head,
                           int32_t max_kv_splits, int32_t core_count, int32_t *err,
                           int32_t segs) {
  grid_dependency_wait();
  allow_dependent_launch();
  if (blockIdx.x == gridDim.x - 1) {
    split_counts<kFusedThreads>(splits, seq_lens, num_reqs, num_group, num_head, num_kv_head,
                                max_kv_splits, core_count);
    return;
  }
  const int64_t w = int64_t(blockIdx.x) * (kFusedThreads / 32) + (threadIdx.x >> 5);
  const int64_t row = w / segs;
  if (row < num_reqs)
    copy_row_segment(page_indices, capacity, bt, num_cols, s0, s1, cu, err, int(row),
                     int(w - row * segs), threadIdx.x & 31);
}

}  // namespace

pkv_status_t launch_copy_page_indices(int32_t *page_indices, int64_t capacity,
                                      const int32_t *block_table, int32_t num_cols, int64_t s0,
                                      int64_t s1, const int32_t *cu, int32_t num_reqs,
                                      int32_t *err, cudaStream_t stream) {
  if (num_reqs == 0) return PKV_OK;
  return launch_programmatic(copy_page_indices_kernel, dim3(num_reqs), dim3(kCopyThreads), 0,
                             stream, page_indices, capacity, block_table, num_cols, s0, s1, cu,
                             err) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

pkv_status_t launch_num_kv_splits(int32_t *out, const int32_t *seq_lens, int32_t num_seq,
                                  int32_t num_group, int32_t num_head, int32_t num_kv_head,
                                  int32_t max_kv_splits, int32_t core_count,
                                  cudaStream_t stream) {
  return launch_programmatic(num_kv_splits_kernel, dim3(1), dim3(kSplitThreads), 0, stream, out,
                             seq_lens, num_seq, num_group, num_head, num_kv_head, max_kv_splits,
                             core_count) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

pkv_status_t launch_decode_metadata(int32_t *page_indices, int64_t capacity,
                                    const int32_t *block_table, int32_t num_cols, int64_t s0,
                                    int64_t s1, const int32_t *cu, int32_t num_reqs,
                                    int32_t *splits, const int32_t *seq_lens, int32_t num_group,
                                    int32_t num_head, int32_t num_kv_head, int32_t max_kv_splits,
                                    int32_t core_count, int32_t *err, cudaStream_t stream) {
  const int warps_per_block = kFusedThreads / 32;
  const int32_t segs = num_cols > 0 ? (num_cols + kSegCols - 1) / kSegCols : 1;
  const int64_t copy_blocks = (int64_t(num_reqs) * segs + warps_per_block - 1) / warps_per_block;
  if (copy_blocks + 1 > 0x7fffffff) return PKV_ERR_UNSUPPORTED;
  return launch_programmatic(decode_metadata_kernel, dim3(unsigned(copy_blocks + 1)),
                             dim3(kFusedThreads), 0, stream, page_indices, capacity, block_table,
                             num_cols, s0, s1, cu, num_reqs, splits, seq_lens, num_group,
                             num_head, num_kv_head, max_kv_splits, core_count, err,
                             segs) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

}  // namespace pkv
