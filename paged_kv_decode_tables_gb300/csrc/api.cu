// C ABI of the paged-KV decode library: argument checks on the host, instance
// selection, launch on the caller's stream.  No allocation, no host sync.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "../../include/paged_kv.h"
#include "attention_launch.cuh"
#include "metadata.cuh"
#include "reduce.cuh"

namespace {

using pkv::AttnParams;

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_smem_per_sm[kMaxDevices];
std::atomic<int> g_forced_warps{0};
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};
std::atomic<unsigned> g_extra_expect_tx{0};
std::atomic<int> g_fp8_kernel{0};
std::atomic<int> g_split_fold{1};

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  int v = g_sm_count[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
    v = 148;
  g_sm_count[dev].store(v, std::memory_order_relaxed);
  return v;
}

// Shared memory of one SM in bytes (228 KiB on GB300 when the query fails).
int smem_per_sm() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 233472;
  int v = g_smem_per_sm[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
      v <= 0)
    v = 233472;
  g_smem_per_sm[dev].store(v, std::memory_order_relaxed);
  return v;
}

int elem_size(pkv_dtype_t t) {
  switch (t) {
    case PKV_F32: return 4;
    case PKV_F16: return 2;
    case PKV_BF16: return 2;
    default: return 0;
  }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool stride_bytes16(int64_t stride, int elem) {
  const int64_t b = stride * elem;
  return (b % 16) == 0;
}

bool is_fp8_cache(int32_t kv) { return kv == PKV_KV_FP8_E4M3 || kv == PKV_KV_FP8_E5M2; }

// Bytes of one cache element.
int cache_elem_size(const pkv_decode_args_t *a) {
  return is_fp8_cache(a->kv_cache_dtype) ? 1 : elem_size(a->dtype);
}

size_t smem_for(pkv_dtype_t t, int32_t kv, int D, int BS, int W) {
  if (kv == PKV_KV_AUTO) {
    switch (t) {
      case PKV_F32: return pkv::smem_attention_f32(D, BS, W);
      case PKV_F16: return pkv::smem_attention_f16(D, BS, W);
      case PKV_BF16: return pkv::smem_attention_bf16(D, BS, W);
      default: return 0;
    }
  }
  const bool e4m3 = kv == PKV_KV_FP8_E4M3;
  switch (t) {
    case PKV_F16:
      return e4m3 ? pkv::smem_attention_f16_e4m3(D, BS, W) : pkv::smem_attention_f16_e5m2(D, BS, W);
    case PKV_BF16:
      return e4m3 ? pkv::smem_attention_bf16_e4m3(D, BS, W)
                  : pkv::smem_attention_bf16_e5m2(D, BS, W);
    default: return 0;
  }
}

// Checks shared by decode and the v2 partition pass.
pkv_status_t check_decode_args(const pkv_decode_args_t *a) {
  if (a == nullptr) return PKV_ERR_INVALID_ARG;
  if (elem_size(a->dtype) == 0) return PKV_ERR_INVALID_ARG;
  if (a->kv_cache_dtype != PKV_KV_AUTO && !is_fp8_cache(a->kv_cache_dtype))
    return PKV_ERR_INVALID_ARG;
  if (is_fp8_cache(a->kv_cache_dtype)) {
    if (!std::isfinite(a->k_scale) || !std::isfinite(a->v_scale)) return PKV_ERR_INVALID_ARG;
    if (a->dtype == PKV_F32) return PKV_ERR_UNSUPPORTED;
  }
  if ((reinterpret_cast<uintptr_t>(a->alibi_slopes) & 3u) != 0) return PKV_ERR_INVALID_ARG;
  const int es = cache_elem_size(a);
  if (a->num_seqs < 0 || a->num_heads < 1 || a->num_kv_heads < 1) return PKV_ERR_INVALID_ARG;
  if (a->num_heads % a->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (a->x * es != 16) return PKV_ERR_INVALID_ARG;
  if (a->head_size < 1 || a->head_size % a->x != 0) return PKV_ERR_INVALID_ARG;
  if (a->block_size < 1 || a->max_blocks_per_seq < 0 || a->num_blocks < 1)
    return PKV_ERR_INVALID_ARG;
  if (!std::isfinite(a->scale)) return PKV_ERR_INVALID_ARG;
  const int64_t head_groups =
      (a->num_heads / a->num_kv_heads + pkv::kMaxGroup - 1) / pkv::kMaxGroup;
  if (a->num_seqs > 65535 || int64_t(a->num_kv_heads) * head_groups > 65535)
    return PKV_ERR_UNSUPPORTED;
  if (smem_for(a->dtype, a->kv_cache_dtype, a->head_size, a->block_size, 1) == 0)
    return PKV_ERR_UNSUPPORTED;
  if (a->num_seqs == 0) return PKV_OK;
  if (!a->query || !a->key_cache || !a->value_cache || !a->block_tables || !a->seq_lens)
    return PKV_ERR_INVALID_ARG;
  // Each (block, kv_head) page must be one contiguous run.
  const int64_t *ks = a->k_stride, *vs = a->v_stride;
  if (ks[4] != 1 || ks[3] != a->x || ks[2] != int64_t(a->block_size) * a->x)
    return PKV_ERR_UNSUPPORTED;
  if (vs[3] != 1 || vs[2] != a->block_size) return PKV_ERR_UNSUPPORTED;
  if (!aligned16(a->key_cache) || !aligned16(a->value_cache)) return PKV_ERR_INVALID_ARG;
  if (!stride_bytes16(ks[0], es) || !stride_bytes16(ks[1], es) || !stride_bytes16(vs[0], es) ||
      !stride_bytes16(vs[1], es))
    return PKV_ERR_INVALID_ARG;
  return PKV_OK;
}

AttnParams make_params(const pkv_decode_args_t *a) {
  AttnParams p{};
  p.q = a->query;
  p.q_s0 = a->q_stride[0];
  p.q_s1 = a->q_stride[1];
  p.q_s2 = a->q_stride[2];
  p.k = a->key_cache;
  p.k_s0 = a->k_stride[0];
  p.k_s1 = a->k_stride[1];
  p.v = a->value_cache;
  p.v_s0 = a->v_stride[0];
  p.v_s1 = a->v_stride[1];
  p.bt = a->block_tables;
  p.bt_s0 = a->bt_stride[0];
  p.bt_s1 = a->bt_stride[1];
  p.indptr = a->kv_indptr;
  p.seq_lens = a->seq_lens;
  p.err = a->err_flag;
  p.num_heads = a->num_heads;
  p.num_kv_heads = a->num_kv_heads;
  p.group = a->num_heads / a->num_kv_heads;
  p.head_groups = (p.group + pkv::kMaxGroup - 1) / pkv::kMaxGroup;
  p.num_blocks = a->num_blocks;
  p.max_blocks_per_seq = a->max_blocks_per_seq;
  const bool fp8 = is_fp8_cache(a->kv_cache_dtype);
  p.scale_log2 = (fp8 ? a->scale * a->k_scale : a->scale) * 1.44269504088896340736f;
  p.out_scale = fp8 ? a->v_scale : 1.0f;
  p.alibi = a->alibi_slopes;
  p.order = nullptr;  // set by paged_attention_decode only
  p.fold = 0;
  p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  // The test hook is one-shot: the launch that reads it clears it, so a hook
  // left set can delay at most one launch, never every later one.
  p.extra_expect_tx = g_extra_expect_tx.exchange(0u, std::memory_order_relaxed);
  return p;
}

// Warps per CTA, from measurements on GB300 (the instance must exist):
// - single pass: 4 (a unit is a whole sequence; more warps per CTA shorten
//   the tail of long sequences, at any batch size measured);
// - split-KV with enough units to fill every SM many times over: 1 for fixed
//   partitions of at most 512 tokens (short, even units), 2 for split counts
//   or longer partitions (units can be long and uneven), but 1 with pages of
//   32 tokens or more (a chunk is then a whole page: ragged batch at block
//   size 32, bf16 1.01 vs 0.95 of the copy bandwidth, fp8 0.93 vs 0.90);
// - split-KV with few units: 4;
// - fp32 caches: at most 2 (a warp's two 16-token stages take 32 KiB at head
//   size 128, so 4-warp CTAs leave one CTA and 4 warps per SM: the fp32 GQA
//   single pass ran 0.60 of the copy bandwidth on 4 warps, 0.90 on 2);
// - 2 instead of 4 whenever fewer than three 4-warp CTAs fit in an SM's shared
//   memory (16-bit caches at head size 256: the GQA single pass ran 0.91 of
//   the copy bandwidth on 4 warps, 0.975 on 2).
enum class Pass { kSingle, kFixed, kSplits };

int pick_warps(const pkv_decode_args_t *a, int64_t units, Pass pass, int partition_size) {
  const int forced = g_forced_warps.load(std::memory_order_relaxed);
  auto have = [&](int w) {
    return smem_for(a->dtype, a->kv_cache_dtype, a->head_size, a->block_size, w) != 0;
  };
  if ((forced == 1 || forced == 2 || forced == 4) && have(forced)) return forced;
  int want;
  if (pass == Pass::kSingle || units < int64_t(sm_count()) * 16)
    want = 4;
  else if (pass == Pass::kFixed && partition_size <= 512)
    want = 1;
  else
    want = a->block_size >= 32 ? 1 : 2;
  if (a->dtype == PKV_F32 && want > 2) want = 2;
  if (want == 4) {
    // 1 KiB per CTA is reserved by the system.
    const size_t s4 = smem_for(a->dtype, a->kv_cache_dtype, a->head_size, a->block_size, 4);
    if (s4 != 0 && (s4 + 1024) * 3 > size_t(smem_per_sm())) want = 2;
  }
  while (want > 1 && !have(want)) want /= 2;
  return want;
}

// fp8 caches of head size 128 / block size 16 run on the tensor-memory kernel
// when it is selected (pkv_set_fp8_kernel(1)) and no warp count is forced (a
// forced count names instances of the mma.sync kernel).
bool use_tensor_memory_kernel(const pkv_decode_args_t *a) {
  return g_fp8_kernel.load(std::memory_order_relaxed) == 1 &&
         g_forced_warps.load(std::memory_order_relaxed) == 0 && pkv::fp8_tc_eligible(a);
}

}  // namespace

extern "C" {

const char *pkv_version(void) { return "paged_kv 0.2.0 sm_103a"; }

const char *pkv_status_string(pkv_status_t s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape, dtype or layout";
    case PKV_ERR_CUDA: return "CUDA launch error";
    case PKV_ERR_SCRATCH_TOO_SMALL: return "request exceeds the fixed scratch of the no-allocation entry point";
    default: return "unknown status";
  }
}

size_t pkv_decode_args_size(void) { return sizeof(pkv_decode_args_t); }

pkv_status_t pkv_set_attention_warps(int32_t warps) {
  if (warps != 0 && warps != 1 && warps != 2 && warps != 4) return PKV_ERR_INVALID_ARG;
  g_forced_warps.store(warps, std::memory_order_relaxed);
  return PKV_OK;
}

pkv_status_t pkv_set_split_fold(int32_t mode) {
  if (mode < 0 || mode > 2) return PKV_ERR_INVALID_ARG;
  g_split_fold.store(mode, std::memory_order_relaxed);
  return PKV_OK;
}

pkv_status_t pkv_set_fp8_kernel(int32_t which) {
  if (which != 0 && which != 1) return PKV_ERR_INVALID_ARG;
  g_fp8_kernel.store(which, std::memory_order_relaxed);
  return PKV_OK;
}

pkv_status_t pkv_set_wait_limit_ns(uint64_t ns) {
  if (ns == 0) ns = 2000000000ull;
  if (ns > 60000000000ull) return PKV_ERR_INVALID_ARG;
  g_wait_limit_ns.store(ns, std::memory_order_relaxed);
  return PKV_OK;
}

pkv_status_t pkv_test_set_unarrived_bytes(uint32_t bytes) {
  if (bytes % 16 != 0 || bytes > 65536) return PKV_ERR_INVALID_ARG;
  g_extra_expect_tx.store(bytes, std::memory_order_relaxed);
  return PKV_OK;
}

pkv_status_t paged_attention_decode(void *out, const int64_t out_stride[3],
                                    const pkv_decode_args_t *args, pkv_stream_t stream) {
  pkv_status_t st = check_decode_args(args);
  if (st != PKV_OK) return st;
  if (!out || !out_stride) return PKV_ERR_INVALID_ARG;
  if (args->num_seqs == 0) return PKV_OK;
  AttnParams p = make_params(args);
  p.mode = pkv::kModeV1;
  p.out = out;
  p.o_s0 = out_stride[0];
  p.o_s1 = out_stride[1];
  p.o_s2 = out_stride[2];
  p.max_parts = 1;
  p.order = args->seq_order;
  dim3 grid(1, args->num_kv_heads * p.head_groups, args->num_seqs);
  if (use_tensor_memory_kernel(args))
    return pkv::launch_attention_fp8_tc(args, p, grid, reinterpret_cast<cudaStream_t>(stream));
  const int w = pick_warps(args, int64_t(grid.y) * args->num_seqs, Pass::kSingle, 0);
  return pkv::launch_attention(args->dtype, pkv_kv_cache_dtype_t(args->kv_cache_dtype), p,
                               args->head_size, args->block_size, w, grid,
                               reinterpret_cast<cudaStream_t>(stream));
}

pkv_status_t paged_attention_v2_partition(float *tmp_out, float *exp_sums, float *max_logits,
                                          int32_t max_num_partitions, int32_t partition_size,
                                          const int32_t *num_kv_splits,
                                          const pkv_decode_args_t *args, pkv_stream_t stream) {
  pkv_status_t st = pkv::check_partition_args(args, max_num_partitions, partition_size,
                                              num_kv_splits);
  if (st != PKV_OK) return st;
  if (!tmp_out || !exp_sums || !max_logits) return PKV_ERR_INVALID_ARG;
  if (args->num_seqs == 0) return PKV_OK;
  AttnParams p = make_params(args);
  p.mode = num_kv_splits ? pkv::kModeSplits : pkv::kModeFixed;
  p.tmp = tmp_out;
  p.es = exp_sums;
  p.ml = max_logits;
  p.max_parts = max_num_partitions;
  p.partition_size = num_kv_splits ? 0 : partition_size;
  p.splits = num_kv_splits;
  dim3 grid(max_num_partitions, args->num_kv_heads * p.head_groups, args->num_seqs);
  if (use_tensor_memory_kernel(args))
    return pkv::launch_attention_fp8_tc(args, p, grid, reinterpret_cast<cudaStream_t>(stream));
  const int64_t units = int64_t(max_num_partitions) * grid.y * args->num_seqs;
  const int w = pick_warps(args, units, num_kv_splits ? Pass::kSplits : Pass::kFixed,
                           partition_size);
  // Split-KV over an fp8 cache on two warps per CTA: a sequence fills
  // num_kv_splits[seq] of the max_num_partitions slots, and an empty slot's
  // CTA costs the latency-bound fp8 kernel about 0.6 ns of launch time.  Half
  // the slots, each CTA taking partitions x and x + slots of its sequence,
  // leave fewer empty CTAs (the instance runs its second partition without a
  // further launch).  A sequence with more splits than slots then runs two
  // partitions back to back, which pays only while the (sequence, kv head)
  // pairs alone fill the GPU twice over: measured, the ragged batch of 512
  // sequences gains 2 % and its 128-sequence cut loses 22 %.
  const int fold = g_split_fold.load(std::memory_order_relaxed);
  if (num_kv_splits && is_fp8_cache(args->kv_cache_dtype) && w == 2 && max_num_partitions >= 2 &&
      fold != 0) {
    const size_t cta_smem = smem_for(args->dtype, args->kv_cache_dtype, args->head_size,
                                     args->block_size, w) + 1024;  // 1 KiB system reserve
    const int64_t resident = int64_t(sm_count()) * int64_t(size_t(smem_per_sm()) / cta_smem);
    if (fold == 2 || int64_t(args->num_seqs) * grid.y >= 2 * resident) {
      p.fold = 1;
      grid.x = unsigned((max_num_partitions + 1) / 2);
    }
  }
  return pkv::launch_attention(args->dtype, pkv_kv_cache_dtype_t(args->kv_cache_dtype), p,
                               args->head_size, args->block_size, w, grid,
                               reinterpret_cast<cudaStream_t>(stream));
}

pkv_status_t paged_attention_v2_reduce(void *out, const int64_t out_stride[3],
                                       const float *tmp_out, const float *exp_sums,
                                       const float *max_logits, const int32_t *seq_lens,
                                       const int32_t *num_kv_splits, int32_t num_seqs,
                                       int32_t num_heads, int32_t head_size, int32_t block_size,
                                       int32_t max_num_partitions, int32_t partition_size,
                                       pkv_dtype_t out_dtype, int32_t *err_flag,
                                       pkv_stream_t stream) {
  if (num_seqs < 0 || num_heads < 1 || elem_size(out_dtype) == 0) return PKV_ERR_INVALID_ARG;
  if (head_size != 64 && head_size != 128 && head_size != 256) return PKV_ERR_UNSUPPORTED;
  if (max_num_partitions < 1) return PKV_ERR_INVALID_ARG;
  if (num_kv_splits == nullptr ? partition_size < 1 : block_size < 1) return PKV_ERR_INVALID_ARG;
  if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !out_stride || !tmp_out || !exp_sums || !max_logits || !seq_lens)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(tmp_out)) return PKV_ERR_INVALID_ARG;
  pkv::ReduceParams p{};
  p.out = out;
  p.o_s0 = out_stride[0];
  p.o_s1 = out_stride[1];
  p.o_s2 = out_stride[2];
  p.tmp = tmp_out;
  p.es = exp_sums;
  p.ml = max_logits;
  p.seq_lens = seq_lens;
  p.splits = num_kv_splits;
  p.err = err_flag;
  p.num_seqs = num_seqs;
  p.num_heads = num_heads;
  p.head_size = head_size;
  p.block_size = block_size;
  p.max_parts = max_num_partitions;
  p.partition_size = partition_size;
  return pkv::launch_reduce(p, out_dtype, reinterpret_cast<cudaStream_t>(stream));
}

pkv_status_t copy_page_indices(int32_t *page_indices, int64_t page_indices_capacity,
                               const int32_t *block_table, int32_t num_cols, int64_t bt_stride0,
                               int64_t bt_stride1, const int32_t *cu_num_blocks, int32_t num_reqs,
                               int32_t *err_flag, pkv_stream_t stream) {
  if (num_reqs < 0 || num_cols < 0 || page_indices_capacity < 0) return PKV_ERR_INVALID_ARG;
  if (num_reqs == 0) return PKV_OK;
  if (!page_indices || !block_table || !cu_num_blocks) return PKV_ERR_INVALID_ARG;
  return pkv::launch_copy_page_indices(page_indices, page_indices_capacity, block_table, num_cols,
                                       bt_stride0, bt_stride1, cu_num_blocks, num_reqs, err_flag,
                                       reinterpret_cast<cudaStream_t>(stream));
}

pkv_status_t compute_num_kv_splits(int32_t *num_kv_splits, const int32_t *seq_lens, int32_t num_seq,
                                   int32_t num_group, int32_t num_head, int32_t num_kv_head,
                                   int32_t max_kv_splits, int32_t device_core_count,
                                   pkv_stream_t stream) {
  if (!num_kv_splits || !seq_lens) return PKV_ERR_INVALID_ARG;
  if (num_seq < 1 || num_group < 1 || num_head < 1 || num_kv_head < 1) return PKV_ERR_INVALID_ARG;
  if (num_head < num_kv_head || max_kv_splits < 1 || device_core_count < 1)
    return PKV_ERR_INVALID_ARG;
  return pkv::launch_num_kv_splits(num_kv_splits, seq_lens, num_seq, num_group, num_head,
                                   num_kv_head, max_kv_splits, device_core_count,
                                   reinterpret_cast<cudaStream_t>(stream));
}

pkv_status_t prepare_decode_metadata(int32_t *page_indices, int64_t page_indices_capacity,
                                     const int32_t *block_table, int32_t num_cols,
                                     int64_t bt_stride0, int64_t bt_stride1,
                                     const int32_t *cu_num_blocks, int32_t num_reqs,
                                     int32_t *num_kv_splits, const int32_t *seq_lens,
                                     int32_t num_group, int32_t num_head, int32_t num_kv_head,
                                     int32_t max_kv_splits, int32_t device_core_count,
                                     int32_t *err_flag, pkv_stream_t stream) {
  if (num_reqs < 1 || num_cols < 0 || page_indices_capacity < 0) return PKV_ERR_INVALID_ARG;
  if (!page_indices || !block_table || !cu_num_blocks || !num_kv_splits || !seq_lens)
    return PKV_ERR_INVALID_ARG;
  if (num_group < 1 || num_head < 1 || num_kv_head < 1 || num_head < num_kv_head ||
      max_kv_splits < 1 || device_core_count < 1)
    return PKV_ERR_INVALID_ARG;
  return pkv::launch_decode_metadata(page_indices, page_indices_capacity, block_table, num_cols,
                                     bt_stride0, bt_stride1, cu_num_blocks, num_reqs,
                                     num_kv_splits, seq_lens, num_group, num_head, num_kv_head,
                                     max_kv_splits, device_core_count, err_flag,
                                     reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace pkv {

pkv_status_t check_partition_args(const pkv_decode_args_t *args, int32_t max_num_partitions,
                                  int32_t partition_size, const int32_t *num_kv_splits) {
  pkv_status_t st = check_decode_args(args);
  if (st != PKV_OK) return st;
  if (max_num_partitions < 1) return PKV_ERR_INVALID_ARG;
  if (num_kv_splits == nullptr) {
    if (partition_size < args->block_size || partition_size % args->block_size != 0)
      return PKV_ERR_INVALID_ARG;
    const int64_t need =
        (int64_t(args->max_blocks_per_seq) * args->block_size + partition_size - 1) /
        partition_size;
    if (args->kv_indptr == nullptr && need > max_num_partitions) return PKV_ERR_INVALID_ARG;
  }
  return PKV_OK;
}

pkv_status_t launch_attention(pkv_dtype_t dtype, pkv_kv_cache_dtype_t kv, const AttnParams &p,
                              int head_size, int block_size, int warps, dim3 grid,
                              cudaStream_t stream) {
  const int D = head_size, BS = block_size, W = warps;
  if (kv == PKV_KV_AUTO) {
    switch (dtype) {
      case PKV_F32: return launch_attention_f32(p, D, BS, W, grid, stream);
      case PKV_F16: return launch_attention_f16(p, D, BS, W, grid, stream);
      case PKV_BF16: return launch_attention_bf16(p, D, BS, W, grid, stream);
      default: return PKV_ERR_UNSUPPORTED;
    }
  }
  const bool e4m3 = kv == PKV_KV_FP8_E4M3;
  switch (dtype) {
    case PKV_F16:
      return e4m3 ? launch_attention_f16_e4m3(p, D, BS, W, grid, stream)
                  : launch_attention_f16_e5m2(p, D, BS, W, grid, stream);
    case PKV_BF16:
      return e4m3 ? launch_attention_bf16_e4m3(p, D, BS, W, grid, stream)
                  : launch_attention_bf16_e5m2(p, D, BS, W, grid, stream);
    default: return PKV_ERR_UNSUPPORTED;
  }
}

}  // namespace pkv
