// Fused decode metadata (sglang python/sglang/kernels/ops/attention/metadata.py:
// normal_decode_set_metadata with _fused_metadata_kernel_general and
// _fused_metadata_kernel_ps1_no_swa), one launch, no host sync:
//
//   cache_seqlens[i] = int32(seq_lens[i] + seq_len_delta)
//   cu_seqlens_k     = running int32 sum of cache_seqlens (cu[0] = 0, cu[B] = total)
//   page_index       = req_to_token[req_pool_indices[i], c << SHIFT],  c < max_seq_pages
//   page_table[i, c] = page_index >> SHIFT                     (SHIFT = log2(page_size))
//   swa_page_table[i, c] = full_to_swa_mapping[page_index] >> SHIFT   (optional)
//
// Blocks [0, B * chunks) gather one chunk of one request row each (the last
// block computes the lengths and the scan with warp shuffles, 256 at a time).
// General form: 2048-column chunks, eight columns per thread, their loads
// issued together.  Page size 1 without the sliding-window table over
// unit-stride, 16-byte aligned rows is a plain row copy: 4096-column chunks,
// sixteen columns per thread moved as four 16-byte loads and stores.  Row and
// column indices into the token pool and the mapping are bounds-checked: an
// out-of-range index writes 0 and sets PKV_ERRF_INDPTR.
#include <cuda_runtime.h>

#include "../../include/paged_kv.h"
#include "pkv_launch.cuh"
#include "pkv_ptx.cuh"

namespace pkv {

namespace {

constexpr int kCols = 256;                           // threads per block
constexpr int kPerThread = 8;                        // columns per thread
constexpr int kChunkCols = kCols * kPerThread;       // columns per block
constexpr int kVecPerThread = 4;                     // row copy: int4 per thread
constexpr int kVecChunkCols = kCols * kVecPerThread * 4;

// Page size 1, no sliding-window table: page_table row i = the first
// max_seq_pages entries of token-pool row req_pool_indices[i], 16 bytes at a
// time (columns past the pool's width or a bad row write 0 and flag).
__device__ __forceinline__ void copy_row_vec(const pkv_decode_metadata_args_t &a, int i, int chunk,
                                             int tid) {
  const int64_t row = a.req_pool_indices[int64_t(i) * a.req_pool_indices_stride];
  const bool row_ok = row >= 0 && row < a.req_to_token_rows;
  const int32_t *src = a.req_to_token + (row_ok ? row : 0) * a.req_to_token_stride[0];
  int32_t *dst = a.page_table + int64_t(i) * a.page_table_stride[0];
  const int cbase = chunk * kVecChunkCols + 4 * tid;
  int4 v[kVecPerThread];
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const int c = cbase + k * (4 * kCols);
    v[k] = make_int4(0, 0, 0, 0);
    if (c + 3 < a.max_seq_pages && row_ok && int64_t(c) + 3 < a.req_to_token_cols) {
      v[k] = __ldcs(reinterpret_cast<const int4 *>(src + c));
    } else {
      int e[4] = {0, 0, 0, 0};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (c + j < a.max_seq_pages) {
          if (row_ok && int64_t(c) + j < a.req_to_token_cols)
            e[j] = src[c + j];
          else
            flag_error(a.err_flag, 8u);
        }
      }
      v[k] = make_int4(e[0], e[1], e[2], e[3]);
    }
  }
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const int c = cbase + k * (4 * kCols);
    if (c + 3 < a.max_seq_pages) {
      __stcs(reinterpret_cast<int4 *>(dst + c), v[k]);
    } else {
      const int e[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (c + j < a.max_seq_pages) dst[c + j] = e[j];
    }
  }
}

template <bool kRowCopy>
__global__ void __launch_bounds__(kCols) decode_metadata_kernel(const pkv_decode_metadata_args_t a,
                                                                int shift, int chunks) {
  grid_dependency_wait();
  allow_dependent_launch();
  const int tid = threadIdx.x;
  const int64_t gather_blocks = int64_t(a.batch_size) * chunks;
  if (int64_t(blockIdx.x) == gather_blocks) {
    // lengths and their exclusive scan (int32 arithmetic, wrapping like a cast)
    // With cu_num_pages, the page counts ceil(len / page_size) (0 for a
    // length <= 0) are scanned alongside, in the same int32 arithmetic.
    __shared__ unsigned warp_sum[2][kCols / 32];
    const int lane = tid & 31, warp = tid >> 5;
    const bool pages_out = a.cu_num_pages != nullptr;
    unsigned carry = 0, carry_p = 0;
    for (int base = 0; base < a.batch_size; base += kCols) {
      const int i = base + tid;
      unsigned v = 0, np = 0;
      if (i < a.batch_size) {
        v = unsigned(a.seq_lens[int64_t(i) * a.seq_lens_stride] + a.seq_len_delta);
        a.cache_seqlens[int64_t(i) * a.cache_seqlens_stride] = int32_t(v);
        np = int32_t(v) > 0 ? ((v - 1u) >> shift) + 1u : 0u;
      }
      unsigned incl = v, incl_p = np;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_up_sync(0xffffffffu, incl, o);
        const unsigned tp = __shfl_up_sync(0xffffffffu, incl_p, o);
        if (lane >= o) {
          incl += t;
          incl_p += tp;
        }
      }
      if (lane == 31) {
        warp_sum[0][warp] = incl;
        warp_sum[1][warp] = incl_p;
      }
      __syncthreads();
      unsigned before = 0, total = 0, before_p = 0, total_p = 0;
#pragma unroll
      for (int w = 0; w < kCols / 32; ++w) {
        const unsigned ws = warp_sum[0][w], wp = warp_sum[1][w];
        if (w < warp) {
          before += ws;
          before_p += wp;
        }
        total += ws;
        total_p += wp;
      }
      if (i < a.batch_size) {
        a.cu_seqlens_k[int64_t(i) * a.cu_seqlens_k_stride] = int32_t(carry + before + incl - v);
        if (pages_out)
          a.cu_num_pages[int64_t(i) * a.cu_num_pages_stride] =
              int32_t(carry_p + before_p + incl_p - np);
      }
      carry += total;
      carry_p += total_p;
      __syncthreads();
    }
    if (tid == 0) {
      a.cu_seqlens_k[int64_t(a.batch_size) * a.cu_seqlens_k_stride] = int32_t(carry);
      if (pages_out)
        a.cu_num_pages[int64_t(a.batch_size) * a.cu_num_pages_stride] = int32_t(carry_p);
    }
    return;
  }
  const int i = int(blockIdx.x / unsigned(chunks));
  if constexpr (kRowCopy) {
    copy_row_vec(a, i, int(blockIdx.x % unsigned(chunks)), tid);
    return;
  }
  const int c0 = int(blockIdx.x % unsigned(chunks)) * kChunkCols + tid;
  const int64_t row = a.req_pool_indices[int64_t(i) * a.req_pool_indices_stride];
  const bool row_ok = row >= 0 && row < a.req_to_token_rows;
  const int32_t *src = a.req_to_token + (row_ok ? row : 0) * a.req_to_token_stride[0];
  // Column c = c0 + k * kCols: each warp touches 32 consecutive columns per k,
  // and the kPerThread loads of a thread are issued before any is used.
  int32_t page_index[kPerThread];
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    const int c = c0 + k * kCols;
    const int64_t col = int64_t(c) << shift;
    page_index[k] = 0;
    if (c < a.max_seq_pages) {
      if (row_ok && col < a.req_to_token_cols)
        page_index[k] = __ldcs(src + col * a.req_to_token_stride[1]);
      else
        flag_error(a.err_flag, 8u);
    }
  }
  int64_t slot[kPerThread];
  if (a.swa_page_table != nullptr) {
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
      slot[k] = 0;
      if (c0 + k * kCols < a.max_seq_pages) {
        if (page_index[k] >= 0 && page_index[k] < a.full_to_swa_len)
          slot[k] = a.full_to_swa_mapping[int64_t(page_index[k]) * a.full_to_swa_stride];
        else
          flag_error(a.err_flag, 8u);
      }
    }
  }
  int32_t *pt = a.page_table + int64_t(i) * a.page_table_stride[0];
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    const int c = c0 + k * kCols;
    if (c < a.max_seq_pages) __stcs(pt + int64_t(c) * a.page_table_stride[1], page_index[k] >> shift);
  }
  if (a.swa_page_table != nullptr) {
    int32_t *sp = a.swa_page_table + int64_t(i) * a.swa_page_table_stride[0];
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
      const int c = c0 + k * kCols;
      if (c < a.max_seq_pages)
        __stcs(sp + int64_t(c) * a.swa_page_table_stride[1], int32_t(slot[k] >> shift));
    }
  }
}

}  // namespace

}  // namespace pkv

extern "C" size_t pkv_decode_metadata_args_size(void) {
  return sizeof(pkv_decode_metadata_args_t);
}

extern "C" pkv_status_t normal_decode_set_metadata(const pkv_decode_metadata_args_t *a,
                                                   pkv_stream_t stream) {
  if (a == nullptr) return PKV_ERR_INVALID_ARG;
  if (a->batch_size < 1 || a->max_seq_pages < 0) return PKV_ERR_INVALID_ARG;
  if (a->page_size < 1 || (a->page_size & (a->page_size - 1)) != 0) return PKV_ERR_INVALID_ARG;
  if (!a->seq_lens || !a->cache_seqlens || !a->cu_seqlens_k) return PKV_ERR_INVALID_ARG;
  if (a->max_seq_pages > 0 && (!a->req_to_token || !a->req_pool_indices || !a->page_table))
    return PKV_ERR_INVALID_ARG;
  if (a->req_to_token_rows < 0 || a->req_to_token_cols < 0) return PKV_ERR_INVALID_ARG;
  if (a->swa_page_table != nullptr && (a->full_to_swa_mapping == nullptr || a->full_to_swa_len < 0))
    return PKV_ERR_INVALID_ARG;
  int shift = 0;
  while ((1 << shift) < a->page_size) ++shift;
  auto aligned16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const bool row_copy = shift == 0 && a->swa_page_table == nullptr && a->max_seq_pages > 0 &&
                        a->req_to_token_stride[1] == 1 && a->page_table_stride[1] == 1 &&
                        a->req_to_token_stride[0] % 4 == 0 && a->page_table_stride[0] % 4 == 0 &&
                        aligned16(a->req_to_token) && aligned16(a->page_table);
  const int chunk_cols = row_copy ? pkv::kVecChunkCols : pkv::kChunkCols;
  const int chunks = (a->max_seq_pages + chunk_cols - 1) / chunk_cols;
  const int64_t blocks = int64_t(a->batch_size) * chunks + 1;
  if (blocks > 0x7fffffff) return PKV_ERR_UNSUPPORTED;
  const cudaError_t e =
      row_copy ? pkv::launch_programmatic(pkv::decode_metadata_kernel<true>, dim3(unsigned(blocks)),
                                          dim3(pkv::kCols), 0,
                                          reinterpret_cast<cudaStream_t>(stream), *a, shift, chunks)
               : pkv::launch_programmatic(pkv::decode_metadata_kernel<false>,
                                          dim3(unsigned(blocks)), dim3(pkv::kCols), 0,
                                          reinterpret_cast<cudaStream_t>(stream), *a, shift, chunks);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
