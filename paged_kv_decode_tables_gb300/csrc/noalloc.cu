// Split-KV decode for callers that cannot allocate device memory.
//
// Some callers can't call cudaMalloc: an engine that reserves all device
// memory up front and forbids allocation while serving, a plugin running
// inside a host application that owns the CUDA allocator, or a latency path
// where cudaMalloc/cudaFree would add an implicit synchronisation.  For them
// this file keeps the split-KV scratch (per-partition outputs, exp sums and
// max logits) in one statically sized device array that every GPU loading the
// library holds until the process exits.  The caller passes only inputs and
// the output; nothing here allocates.
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>

#include "../../include/paged_kv.h"
#include "attention_launch.cuh"

static constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB per GPU

// The scratch itself: one file-scope array per GPU that loads the library.
static __device__ __align__(256) unsigned char g_split_scratch[kScratchBytes];

namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_addr[kMaxDevices];

size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Device address of the array on the current device.  Host code only sees a
// host-side stand-in under the array's name, so the address is looked up once
// per device (with that device current) and cached for the life of the
// process: a cudaDeviceReset reloads the module and leaves the cached address
// stale, so the entry point is not for processes that reset a device.
void *scratch_address(int dev) {
  void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p != nullptr) return p;
  void *q = nullptr;
  if (cudaGetSymbolAddress(&q, g_split_scratch) != cudaSuccess || q == nullptr) return nullptr;
  g_scratch_addr[dev].store(q, std::memory_order_release);
  return q;
}

// Bytes of the three scratch regions (tmp_out, exp_sums, max_logits, each
// rounded up to kAlign) for `rows` = num_seqs * num_heads * max_num_partitions
// rows of head_size floats; false when they exceed the array.  Every product
// is bounded by a division first, so no size computation can wrap whatever
// the (already validated, positive) factors are.
bool scratch_layout(int64_t num_seqs, int64_t num_heads, int64_t max_parts, int64_t head_size,
                    size_t *tmp_bytes, size_t *stat_bytes) {
  const uint64_t row_bytes = (uint64_t(head_size) + 2u) * sizeof(float);
  const uint64_t max_rows = kScratchBytes / row_bytes;
  uint64_t rows = uint64_t(num_seqs);
  if (rows > max_rows) return false;
  if (uint64_t(num_heads) > max_rows / rows) return false;
  rows *= uint64_t(num_heads);
  if (uint64_t(max_parts) > max_rows / rows) return false;
  rows *= uint64_t(max_parts);
  // rows * row_bytes <= kScratchBytes here, so nothing below wraps.
  *tmp_bytes = round_up(size_t(rows) * size_t(head_size) * sizeof(float));
  *stat_bytes = round_up(size_t(rows) * sizeof(float));
  return *tmp_bytes + 2 * *stat_bytes <= kScratchBytes;
}

}  // namespace

extern "C" size_t pkv_noalloc_scratch_bytes(void) { return kScratchBytes; }

extern "C" pkv_status_t paged_attention_v2_noalloc(void *out, const int64_t out_stride[3],
                                                   int32_t max_num_partitions,
                                                   int32_t partition_size,
                                                   const int32_t *num_kv_splits,
                                                   const pkv_decode_args_t *args,
                                                   pkv_stream_t stream) {
  // The partition pass's own checks come first, so a malformed call gets the
  // status that names its fault rather than a scratch-size refusal.
  pkv_status_t st =
      pkv::check_partition_args(args, max_num_partitions, partition_size, num_kv_splits);
  if (st != PKV_OK) return st;
  if (out == nullptr || out_stride == nullptr) return PKV_ERR_INVALID_ARG;
  if (args->num_seqs == 0) return PKV_OK;
  size_t tmp_bytes = 0, stat_bytes = 0;
  if (!scratch_layout(args->num_seqs, args->num_heads, max_num_partitions, args->head_size,
                      &tmp_bytes, &stat_bytes))
    return PKV_ERR_SCRATCH_TOO_SMALL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
  unsigned char *base = static_cast<unsigned char *>(scratch_address(dev));
  if (base == nullptr) return PKV_ERR_CUDA;
  float *tmp = reinterpret_cast<float *>(base);
  float *exp_sums = reinterpret_cast<float *>(base + tmp_bytes);
  float *max_logits = reinterpret_cast<float *>(base + tmp_bytes + stat_bytes);
  // Every entry the reduce reads is written by the partition pass first, so
  // nothing left from an earlier call needs clearing.
  st = paged_attention_v2_partition(tmp, exp_sums, max_logits, max_num_partitions,
                                    partition_size, num_kv_splits, args, stream);
  if (st != PKV_OK) return st;
  return paged_attention_v2_reduce(out, out_stride, tmp, exp_sums, max_logits, args->seq_lens,
                                   num_kv_splits, args->num_seqs, args->num_heads,
                                   args->head_size, args->block_size, max_num_partitions,
                                   partition_size, args->dtype, args->err_flag, stream);
}
