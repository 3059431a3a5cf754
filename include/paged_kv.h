/*
 * paged_kv.h - C ABI of the GB300 (sm_103a) paged-KV decode library.
 *
 * Five operations make up the decode hot path:
 *
 *   paged_attention_decode        single-pass decode (one partition per sequence)
 *   paged_attention_v2_partition  split-KV partition pass
 *   paged_attention_v2_reduce     log-sum-exp combination of the partitions
 *   copy_page_indices             block-table rows -> flat page list, through an indptr
 *   compute_num_kv_splits         per-sequence split count
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 * - Every pointer argument is DEVICE memory owned and allocated by the caller.
 *   The library never allocates, frees, copies to the host or synchronises; each
 *   call enqueues its kernel(s) on `stream` and returns.  `stream == NULL` is the
 *   legacy default stream.
 * - Strides are in ELEMENTS (not bytes), int64.
 * - Arguments are checked on the host before anything is launched; a rejected
 *   call returns PKV_ERR_INVALID_ARG or PKV_ERR_UNSUPPORTED and enqueues nothing.
 *   A launch failure reported by the CUDA runtime returns PKV_ERR_CUDA.
 * - Device data the host cannot see (seq_lens, block ids, indptr entries, split
 *   counts) is checked inside the kernels.  A bad value never faults or hangs:
 *   the kernel clamps it, OR-s a PKV_ERRF_* bit into the optional `err_flag`
 *   (a caller-zeroed device int32, may be NULL) and carries on; results that
 *   depend on the bad value are then unspecified.
 * - Arithmetic: fp32 accumulation for every input dtype; softmax statistics and
 *   split-KV partials are fp32.  Products: fp16/bf16 operands are exact in
 *   fp32; fp8 codes are widened exactly to f16 (a bf16 query is scaled by a
 *   power of two into f16's range without rounding); the probabilities enter
 *   the value product as a hi + lo pair of 16-bit values.  fp32 operands are
 *   split into two tf32 terms each, and a product takes three of the four term
 *   pairs (all four when a kv head serves at most 4 query heads), about 2^-21
 *   relative per product; the fp32 output stays within 1e-5 of the exact
 *   result on the tested inputs.
 *
 * Cache layouts (vLLM's, as restated on the page "paged_attention_v2_triton.py",
 * argument comments of _paged_attn_v2_partition_kernel):
 *   query        [num_seqs, num_heads, head_size]
 *   key_cache    [num_blocks, num_kv_heads, head_size / x, block_size, x],  x = 16 / sizeof(elem)
 *   value_cache  [num_blocks, num_kv_heads, head_size, block_size]
 *   block_tables [num_seqs, max_blocks_per_seq] int32, any strides
 * The (block, kv_head) page of each cache must be contiguous:
 *   k_stride[2..4] == {block_size*x, x, 1} and v_stride[2..3] == {block_size, 1};
 * the block and head strides are free (multiples of 16 bytes).
 */
#ifndef PAGED_KV_H
#define PAGED_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* Same type as cudaStream_t. */
typedef struct CUstream_st *pkv_stream_t;

typedef enum { PKV_F32 = 0, PKV_F16 = 1, PKV_BF16 = 2 } pkv_dtype_t;

/*
 * Element format of key_cache / value_cache (pkv_decode_args_t.kv_cache_dtype).
 * The page "paged_attention_v2_triton.py" (wrapper paged_attention_v2_triton,
 * arguments kv_cache_dtype, k_scale, v_scale) names these without defining
 * them; this library takes vLLM's reading:
 *   PKV_KV_AUTO      caches hold `dtype` elements; k_scale / v_scale ignored.
 *   PKV_KV_FP8_E4M3  caches hold one-byte OCP E4M3 codes ("fp8", "fp8_e4m3"):
 *   PKV_KV_FP8_E5M2  or E5M2 codes ("fp8_e5m2"); x = 16 and a key element
 *                    stands for decode(code) * k_scale, a value element for
 *                    decode(code) * v_scale.  Queries and the output stay in
 *                    `dtype`, which must then be PKV_F16 or PKV_BF16.
 */
typedef enum { PKV_KV_AUTO = 0, PKV_KV_FP8_E4M3 = 1, PKV_KV_FP8_E5M2 = 2 } pkv_kv_cache_dtype_t;

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1, /* null pointer, bad size, inconsistent strides */
  PKV_ERR_UNSUPPORTED = 2, /* valid but not built: head_size, block_size, group, layout */
  PKV_ERR_CUDA = 3,        /* the CUDA runtime refused the launch */
  PKV_ERR_SCRATCH_TOO_SMALL = 4 /* request exceeds paged_attention_v2_noalloc's fixed scratch */
} pkv_status_t;

/* Bits OR-ed into *err_flag by kernels that meet bad device data. */
#define PKV_ERRF_BLOCK_ID 1u /* block id outside [0, num_blocks): block 0 was read instead */
#define PKV_ERRF_SEQ_LEN 2u  /* seq_len < 0 or above the row's capacity: clamped */
#define PKV_ERRF_SPLITS 4u   /* num_kv_splits[s] outside [1, max_num_partitions]: clamped */
#define PKV_ERRF_INDPTR 8u   /* indptr row negative, longer than the table, or past the output */
#define PKV_ERRF_TIMEOUT 16u /* a wait for a copy into shared memory exceeded its time limit */
#define PKV_ERRF_ORDER 32u   /* seq_order entry outside [0, num_seqs): the identity was used */

/*
 * Inputs shared by paged_attention_decode and paged_attention_v2_partition.
 *
 *   num_seqs, num_heads, num_kv_heads, head_size, block_size, x: shapes above;
 *       num_heads % num_kv_heads == 0; query head h reads kv head
 *       h / (num_heads / num_kv_heads) (contiguous groups).
 *   max_blocks_per_seq: columns of block_tables; seq_len may not exceed
 *       max_blocks_per_seq * block_size.
 *   num_blocks: valid physical block ids are [0, num_blocks).
 *   dtype: element type of query, key_cache, value_cache and the output.
 *   scale: logit = scale * (q . k).
 *   kv_indptr: optional.  NULL: sequence s's logical page j is
 *       block_tables[s*bt_stride[0] + j*bt_stride[1]].  Non-NULL (num_seqs+1
 *       int32): block_tables is a flat page list (e.g. the output of
 *       copy_page_indices) and page j of sequence s is
 *       block_tables[kv_indptr[s] + j*bt_stride[1]], with
 *       kv_indptr[s+1]-kv_indptr[s] pages available to it.
 *   seq_lens: [num_seqs] int32 context lengths.
 *   err_flag: optional device int32 receiving PKV_ERRF_* bits.
 *   kv_cache_dtype, k_scale, v_scale: cache element format (pkv_kv_cache_dtype_t
 *       above); a zero-initialised struct means PKV_KV_AUTO.  With fp8 the
 *       scales must be finite; x, the key/value strides and the 16-byte rules
 *       count one-byte elements.
 *   alibi_slopes: optional [num_heads] fp32 device array (4-byte aligned).
 *       Non-NULL adds slope[h] * (t - seq_len + 1) to the scaled score of
 *       query head h and token t: ALiBi ("Train Short, Test Long", Press et
 *       al.) with the decode query at position seq_len - 1, the reading of the
 *       alibi_slopes argument the page "paged_attention_v2_triton.py" names.
 *       It enters max_logits of the split-KV pass like any logit.
 *   seq_order: optional [num_seqs] int32 device array, a permutation of
 *       0..num_seqs-1 (NULL: identity).  paged_attention_decode launches the
 *       units of sequence seq_order[z] in the z-th place of its grid, e.g.
 *       longest first from pkv_order_by_length; results do not depend on it.
 *       An entry outside 0..num_seqs-1 is replaced by z and sets
 *       PKV_ERRF_ORDER; duplicate entries leave sequences unprocessed.  The
 *       split-KV entry points and the tensor-memory fp8 kernel ignore it.
 */
typedef struct {
  int32_t num_seqs;
  int32_t num_heads;
  int32_t num_kv_heads;
  int32_t head_size;
  int32_t block_size;
  int32_t x;
  int32_t max_blocks_per_seq;
  int32_t num_blocks;
  pkv_dtype_t dtype;
  float scale;
  const void *query;
  int64_t q_stride[3];
  const void *key_cache;
  int64_t k_stride[5];
  const void *value_cache;
  int64_t v_stride[4];
  const int32_t *block_tables;
  int64_t bt_stride[2];
  const int32_t *kv_indptr;
  const int32_t *seq_lens;
  int32_t *err_flag;
  int32_t kv_cache_dtype; /* pkv_kv_cache_dtype_t */
  float k_scale;
  float v_scale;
  const float *alibi_slopes;
  const int32_t *seq_order;
} pkv_decode_args_t;

/* Library version string, e.g. "paged_kv 0.2.0 sm_103a". */
const char *pkv_version(void);
/* Static description of a status code. */
const char *pkv_status_string(pkv_status_t status);
/* sizeof(pkv_decode_args_t), for bindings that mirror the struct. */
size_t pkv_decode_args_size(void);

/*
 * Tuning override for benchmarks and tests, not for serving: warps per CTA of
 * paged_attention_decode / paged_attention_v2_partition, i.e. how many warps
 * split one (sequence, kv head, partition) unit.  0 (default) lets every call
 * pick from its own pass (single or split), number of units and SM count (the
 * measured rule in the launcher); 1, 2 or 4 forces that value, where the
 * instance exists, on every later call of every thread until it is set back
 * to 0.  A serving process leaves it at 0.  Returns PKV_ERR_INVALID_ARG for
 * any other value.
 */
pkv_status_t pkv_set_attention_warps(int32_t warps);

/*
 * Kernel for fp8 caches (kv_cache_dtype E4M3 / E5M2) with head_size 128,
 * block_size 16 and fp16/bf16 queries, process-wide:
 *   0 (default): the mma.sync kernel (codes widened to f16 in registers);
 *   1: the tensor-memory kernel: persistent CTAs that take unstarted CTAs'
 *      work from the launch queue (cluster launch control), both products as
 *      tcgen05 kind::f8f6f4 MMAs on the cache codes in shared memory, the
 *      query as an exact sum of E4M3 terms, probabilities as four E4M3 terms
 *      (about 16 significant bits), accumulators in tensor memory.  Same
 *      results within the tolerances of the mma.sync kernel; slower on the
 *      measured batches.  A forced warp count (pkv_set_attention_warps)
 *      selects the mma.sync kernel.
 * Other shapes always use the mma.sync kernel.  Returns PKV_ERR_INVALID_ARG
 * for any other value.
 */
pkv_status_t pkv_set_fp8_kernel(int32_t which);

/*
 * Split-KV partition pass (paged_attention_v2_partition with num_kv_splits)
 * over an fp8 cache on two warps per CTA (block size below 32, the mma.sync
 * kernel), process-wide; a tuning and test override:
 *   1 (default): when the (sequence, kv head x head sub-group) pairs number
 *      at least twice the GPU's resident CTAs, launch
 *      ceil(max_num_partitions / 2) partition slots per pair, the CTA of
 *      slot x also running partition x + that count of its sequence when
 *      there is one; otherwise one CTA per partition slot;
 *   2: always the halved grid;  0: always one CTA per partition slot.
 * Every setting gives bit-identical outputs.  A sequence fills
 * num_kv_splits[seq] of the slots (on the ragged serving batch 1206 of
 * 8192); an empty slot's CTA still holds a residency slot while it reads the
 * sequence's length and split count, about 0.6 ns of launch time each for the
 * latency-bound fp8 kernel.  A sequence with more splits than slots runs two
 * partitions back to back, which costs more than it saves on small batches.
 * Returns PKV_ERR_INVALID_ARG for any value outside 0..2.
 */
pkv_status_t pkv_set_split_fold(int32_t mode);

/*
 * Limit, in nanoseconds, of every wait of the attention kernels for a stage's
 * copies into shared memory (default 2 s; 0 restores it; at most 60 s).  A
 * wait that runs out sets PKV_ERRF_TIMEOUT, waits (again bounded) for the
 * warp's other copies and finishes the CTA with unspecified results for it;
 * no kernel ever waits without a limit.  Process-wide.
 */
pkv_status_t pkv_set_wait_limit_ns(uint64_t ns);

/*
 * Test hook for the timeout path above, one-shot: every stage of the NEXT
 * attention launch (paged_attention_decode or paged_attention_v2_partition, in
 * any thread) expects `bytes` (a multiple of 16, at most 65536) more than its
 * copies deliver, so each of its waits runs into the limit.  That launch
 * clears the hook; later launches are unaffected.  0 clears it without a
 * launch.  Only for exercising failure detection.
 */
pkv_status_t pkv_test_set_unarrived_bytes(uint32_t bytes);

/*
 * Single-pass paged decode.
 *
 * For every sequence s and query head h:
 *   out[s, h, :] = sum_t softmax_t(scale * q[s,h] . k_t) * v_t   over t < seq_lens[s],
 * where k_t / v_t are gathered through block = table[s, t / block_size],
 * slot = t % block_size (page "Needs help on performance optimization",
 * triton-lang/triton issue 2522, worked example; page
 * "paged_attention_v2_triton.py", module docstring "Algorithm per instance").
 * This is the split-KV computation with a single partition covering the whole
 * sequence.
 *
 *   out: [num_seqs, num_heads, head_size] in args->dtype with strides out_stride.
 *   A sequence with seq_len == 0 gets a zero output row.
 * Supported: fp16/bf16 with head_size in {64, 128, 256}; fp32 with head_size in
 * {64, 128}; block_size in {8, 16, 32}; any num_heads/num_kv_heads (a kv head's
 * query heads are served 8 at a time; above 8 its pages are read once per 8
 * heads, mostly from L2), with num_kv_heads * ceil(group / 8) <= 65535.
 * fp8 caches (kv_cache_dtype != PKV_KV_AUTO): fp16/bf16 queries, the same head
 * and block sizes.  With alibi_slopes the logit of token t gains the ALiBi
 * term described at pkv_decode_args_t.
 */
pkv_status_t paged_attention_decode(void *out, const int64_t out_stride[3],
                                    const pkv_decode_args_t *args, pkv_stream_t stream);

/*
 * Split-KV partition pass (page "paged_attention_v2_triton.py",
 * _paged_attn_v2_partition_kernel and "Algorithm per instance").
 *
 * Partition p of sequence s covers tokens [p*P, min((p+1)*P, seq_len)) where
 *   P = partition_size                      when num_kv_splits == NULL, or
 *   P = roundup(cdiv(seq_len, n), block_size), n = num_kv_splits[s], otherwise
 *       (partitions p >= n are empty; this chunking is a reading: the split
 *       heuristic only gives the count).
 * For every (s, h, p) it writes, over the logits z of the partition's tokens:
 *   max_logits[s,h,p] = max z                       (natural-log units)
 *   exp_sums[s,h,p]   = sum exp(z - max z)
 *   tmp_out[s,h,p,:]  = sum exp(z - max z) v / exp_sums[s,h,p]   (normalised)
 * An empty partition (start >= seq_len, or p >= n) writes max_logits = -inf,
 * exp_sums = 0 and leaves tmp_out untouched.
 *
 *   tmp_out:    [num_seqs, num_heads, max_num_partitions, head_size] fp32, contiguous.
 *   exp_sums, max_logits: [num_seqs, num_heads, max_num_partitions] fp32, contiguous.
 *   partition_size: multiple of block_size (ignored when num_kv_splits != NULL);
 *       max_num_partitions >= cdiv(max_blocks_per_seq*block_size, partition_size).
 *   num_kv_splits: optional [num_seqs] int32 (e.g. from compute_num_kv_splits).
 * Same dtype/shape support as paged_attention_decode.
 */
pkv_status_t paged_attention_v2_partition(float *tmp_out, float *exp_sums, float *max_logits,
                                          int32_t max_num_partitions, int32_t partition_size,
                                          const int32_t *num_kv_splits,
                                          const pkv_decode_args_t *args, pkv_stream_t stream);

/*
 * Log-sum-exp reduce (page "paged_attention_v2_triton.py",
 * _paged_attn_v2_reduce_kernel: global max, rescale, weighted sum).
 *
 * With num_parts the number of non-empty partitions of sequence s (computed
 * from seq_lens and partition_size / num_kv_splits / block_size exactly as the
 * partition pass does):
 *   M = max_p max_logits[p],  w_p = exp(max_logits[p] - M) * exp_sums[p],
 *   out[s,h,:] = sum_p w_p * tmp_out[s,h,p,:] / sum_p w_p     (p < num_parts).
 * A sequence with seq_len == 0 gets a zero row.
 *
 *   out: [num_seqs, num_heads, head_size] in out_dtype with strides out_stride.
 *   tmp_out / exp_sums / max_logits: as written by paged_attention_v2_partition.
 *   head_size in {64, 128, 256}.
 */
pkv_status_t paged_attention_v2_reduce(void *out, const int64_t out_stride[3],
                                       const float *tmp_out, const float *exp_sums,
                                       const float *max_logits, const int32_t *seq_lens,
                                       const int32_t *num_kv_splits, int32_t num_seqs,
                                       int32_t num_heads, int32_t head_size, int32_t block_size,
                                       int32_t max_num_partitions, int32_t partition_size,
                                       pkv_dtype_t out_dtype, int32_t *err_flag,
                                       pkv_stream_t stream);

/*
 * Page-index copy (vLLM PR 35765, "AITER MLA backend: Avoid CPU sync in
 * _build_decode", _copy_page_indices_kernel with the review's stride_1 change):
 *   page_indices[cu_num_blocks[i] + j] = block_table[i*bt_stride0 + j*bt_stride1]
 *   for 0 <= j < cu_num_blocks[i+1] - cu_num_blocks[i],  0 <= i < num_reqs.
 * It replaces block_table[mask] (data-dependent size, hence a host sync) with a
 * fixed-size launch.  Bit-exact.
 *
 *   page_indices: int32 output, page_indices_capacity entries; positions no row
 *       covers are left untouched.  Writes past the capacity are skipped and flagged.
 *   block_table: int32, num_cols columns per row, any strides.
 *   cu_num_blocks: [num_reqs + 1] int32 indptr (non-decreasing).  A row longer
 *       than num_cols is clamped and flagged (PKV_ERRF_INDPTR).
 */
pkv_status_t copy_page_indices(int32_t *page_indices, int64_t page_indices_capacity,
                               const int32_t *block_table, int32_t num_cols, int64_t bt_stride0,
                               int64_t bt_stride1, const int32_t *cu_num_blocks, int32_t num_reqs,
                               int32_t *err_flag, pkv_stream_t stream);

/*
 * Per-sequence split count (sglang python/sglang/kernels/ops/attention/metadata.py,
 * get_num_kv_splits_triton), one CTA, no host sync:
 *   mx = max len, mn = min len (both over max(len, 1)); if mx*8 < mn*10: mn = mx
 *   s1 = min(cdiv(mx, mn), max_kv_splits); c1 = cdiv(mx, s1)
 *   ext = int32(float32(device_core_count) * max(log2_f32(float32(mx) / 64), 1))
 *         (float32 product, log2 correctly rounded to float32, truncation)
 *   G = num_head / num_kv_head
 *   token_grid = num_seq*num_group*num_head                 if G == 1
 *              = num_seq*num_group*cdiv(num_head, min(16, G)) otherwise
 *   s2 = min(cdiv(ext, token_grid), max_kv_splits); c2 = cdiv(mx, s2)
 *   num_kv_splits[s*num_group + i] = max(cdiv(len_s, c1), cdiv(len_s, c2)),  i < num_group
 * Bit-exact.  A zero-length sequence gets 0.
 *
 *   num_kv_splits: [num_seq * num_group] int32 output.
 *   seq_lens: [num_seq] int32.  num_seq >= 1, max_kv_splits >= 1,
 *   device_core_count >= 1 (an argument, not queried).
 */
pkv_status_t compute_num_kv_splits(int32_t *num_kv_splits, const int32_t *seq_lens, int32_t num_seq,
                                   int32_t num_group, int32_t num_head, int32_t num_kv_head,
                                   int32_t max_kv_splits, int32_t device_core_count,
                                   pkv_stream_t stream);

/*
 * Both metadata steps in one launch: exactly copy_page_indices(page_indices,
 * page_indices_capacity, block_table, num_cols, bt_stride0, bt_stride1,
 * cu_num_blocks, num_reqs, err_flag) followed by
 * compute_num_kv_splits(num_kv_splits, seq_lens, num_reqs, num_group, num_head,
 * num_kv_head, max_kv_splits, device_core_count), with the same arguments,
 * outputs and errors (one sequence per request row).  The split heuristic runs
 * on one CTA while the others copy table rows (a warp per row), so the decode
 * step's metadata costs a single launch and no host sync (vLLM PR 35765 and
 * sglang's get_num_kv_splits_triton are separate kernels on their pages).
 */
pkv_status_t prepare_decode_metadata(int32_t *page_indices, int64_t page_indices_capacity,
                                     const int32_t *block_table, int32_t num_cols,
                                     int64_t bt_stride0, int64_t bt_stride1,
                                     const int32_t *cu_num_blocks, int32_t num_reqs,
                                     int32_t *num_kv_splits, const int32_t *seq_lens,
                                     int32_t num_group, int32_t num_head, int32_t num_kv_head,
                                     int32_t max_kv_splits, int32_t device_core_count,
                                     int32_t *err_flag, pkv_stream_t stream);

/*
 * Fused decode metadata (sglang python/sglang/kernels/ops/attention/metadata.py,
 * normal_decode_set_metadata with _fused_metadata_kernel_general and
 * _fused_metadata_kernel_ps1_no_swa), one launch, no host sync.  With
 * SHIFT = log2(page_size) and B = batch_size:
 *   cache_seqlens[i]      = int32(seq_lens[i] + seq_len_delta)
 *   cu_seqlens_k[i]       = cache_seqlens[0] + ... + cache_seqlens[i-1]  (int32, i <= B)
 *   page_index            = req_to_token[req_pool_indices[i], c << SHIFT],  c < max_seq_pages
 *   page_table[i, c]      = page_index >> SHIFT
 *   swa_page_table[i, c]  = int32(full_to_swa_mapping[page_index] >> SHIFT)   (if given)
 *   cu_num_pages[i]       = pages[0] + ... + pages[i-1]  (int32, i <= B; if given),
 *                           pages[j] = ceil(cache_seqlens[j] / page_size), 0 if <= 0:
 *                           the page-count indptr that copy_page_indices and
 *                           prepare_decode_metadata take as cu_num_blocks, built on
 *                           the device in the same launch
 * Bit-exact.  Every column c < max_seq_pages of every row is written, as on
 * the page.  All strides are in elements.  A pool row or column outside
 * [0, req_to_token_rows) x [0, req_to_token_cols), or a page index outside
 * [0, full_to_swa_len), writes 0 there and sets PKV_ERRF_INDPTR in err_flag.
 * page_size must be a power of two; batch_size >= 1.
 */
typedef struct {
  int32_t batch_size;
  int32_t max_seq_pages;
  int32_t seq_len_delta;
  int32_t page_size;
  const int64_t *seq_lens;
  int64_t seq_lens_stride;
  const int32_t *req_to_token;
  int64_t req_to_token_stride[2];
  int64_t req_to_token_rows;
  int64_t req_to_token_cols;
  const int64_t *req_pool_indices;
  int64_t req_pool_indices_stride;
  int32_t *cache_seqlens;
  int64_t cache_seqlens_stride;
  int32_t *cu_seqlens_k;
  int64_t cu_seqlens_k_stride;
  int32_t *page_table;
  int64_t page_table_stride[2];
  int32_t *swa_page_table;            /* optional (NULL: no sliding-window table) */
  int64_t swa_page_table_stride[2];
  const int64_t *full_to_swa_mapping; /* required with swa_page_table */
  int64_t full_to_swa_stride;
  int64_t full_to_swa_len;
  int32_t *err_flag;                  /* optional */
  int32_t *cu_num_pages;              /* optional (NULL: not written) */
  int64_t cu_num_pages_stride;
} pkv_decode_metadata_args_t;

pkv_status_t normal_decode_set_metadata(const pkv_decode_metadata_args_t *args,
                                        pkv_stream_t stream);
/* sizeof(pkv_decode_metadata_args_t), for bindings that mirror the struct. */
size_t pkv_decode_metadata_args_size(void);

/*
 * Sliding-window page table for speculative decoding (sglang
 * python/sglang/kernels/ops/attention/metadata.py, prepare_swa_spec_page_table_triton
 * and _prepare_swa_spec_page_table_kernel).  With R = num_draft_tokens,
 * la = seq_len_a[m / R], lb = seq_len_b[m], for every output row
 * m < bs * R and column n < min(la + lb, len_a + len_b):
 *   dst[m, n] = n < la ? (n < len_a ? page_table_a[m / R, n] : 0)
 *                      : (n - la < len_b ? page_table_b[m, n - la] : 0)
 * Columns at or past min(la + lb, len_a + len_b) are left untouched (reading:
 * the page's grid covers the combined width of the two tables).  Bit-exact.
 *   page_table_a: [bs, len_a] int32; page_table_b: [bs * R, len_b] int32;
 *   seq_len_a: [bs] int32; seq_len_b: [bs * R] int32;
 *   dst: [bs * R, >= len_a + len_b] int32.  Strides in elements.
 * A negative length counts as 0 and sets PKV_ERRF_SEQ_LEN.
 */
typedef struct {
  int32_t bs;
  int32_t num_draft_tokens;
  int32_t len_a;
  int32_t len_b;
  const int32_t *page_table_a;
  int64_t a_stride[2];
  const int32_t *page_table_b;
  int64_t b_stride[2];
  const int32_t *seq_len_a;
  int64_t seq_len_a_stride;
  const int32_t *seq_len_b;
  int64_t seq_len_b_stride;
  int32_t *dst;
  int64_t dst_stride[2];
  int32_t *err_flag; /* optional */
} pkv_swa_spec_args_t;

pkv_status_t prepare_swa_spec_page_table(const pkv_swa_spec_args_t *args, pkv_stream_t stream);
/* sizeof(pkv_swa_spec_args_t), for bindings that mirror the struct. */
size_t pkv_swa_spec_args_size(void);

/*
 * Split-KV decode (partition pass + reduce) that allocates nothing.
 *
 * The pages have no counterpart of this entry point; it exists for callers
 * that cannot call cudaMalloc: an engine that reserves all device memory up
 * front and allows no allocation while serving, a plugin inside a host
 * application that owns the CUDA allocator, or a latency-critical path where
 * cudaMalloc/cudaFree would add an implicit synchronisation.
 *
 * Same result as paged_attention_v2_partition followed by
 * paged_attention_v2_reduce (same arguments, same kernels), but the
 * per-partition scratch lives in a fixed array inside the library: 32 MiB
 * (pkv_noalloc_scratch_bytes()) of device memory that every GPU loading the
 * library holds until the process exits.  A call needs
 *   num_seqs * num_heads * max_num_partitions * (head_size + 2) * 4 bytes
 * (each of the three regions rounded up to 256 B) and returns
 * PKV_ERR_SCRATCH_TOO_SMALL, enqueuing nothing, when that exceeds the array.
 *
 *   out: [num_seqs, num_heads, head_size] in args->dtype with strides out_stride.
 *   max_num_partitions, partition_size, num_kv_splits, args: as for
 *       paged_attention_v2_partition.
 *
 * Arguments are checked exactly as paged_attention_v2_partition checks them
 * (PKV_ERR_INVALID_ARG / PKV_ERR_UNSUPPORTED) before the scratch size is; the
 * size check cannot overflow, whatever the head and partition counts.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it for the life
 * of the process; make that first call before any stream capture.  A
 * cudaDeviceReset reloads the library's module and leaves that cached address
 * stale: a process that resets a device must not call this entry point
 * afterwards.  All calls share the one array and it
 * keeps the last call's contents (every value a call reads is written by the
 * same call first): calls that overlap on the GPU, on different streams,
 * race on it.
 */
pkv_status_t paged_attention_v2_noalloc(void *out, const int64_t out_stride[3],
                                        int32_t max_num_partitions, int32_t partition_size,
                                        const int32_t *num_kv_splits,
                                        const pkv_decode_args_t *args, pkv_stream_t stream);
/* Size in bytes of paged_attention_v2_noalloc's fixed scratch array. */
size_t pkv_noalloc_scratch_bytes(void);

/*
 * Launch order for paged_attention_decode's seq_order, longest sequence first:
 * a single pass starts one CTA per (sequence, kv head group) in grid order, so
 * starting the longest units first shortens the grid's tail (longest
 * processing time first).  One CTA sorts the lengths into 256 buckets by
 * (max_len - len) * 256 / (max_len + 1); within a bucket the order is
 * unspecified.  Negative lengths count as 0.
 *   order:    [num_seqs] int32 device output, a permutation of 0..num_seqs-1.
 *   seq_lens: [num_seqs] int32 device input.
 * No host sync; PKV_ERR_INVALID_ARG for num_seqs < 0 or NULL pointers (with
 * num_seqs > 0).
 */
pkv_status_t pkv_order_by_length(int32_t *order, const int32_t *seq_lens, int32_t num_seqs,
                                 pkv_stream_t stream);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* PAGED_KV_H */
