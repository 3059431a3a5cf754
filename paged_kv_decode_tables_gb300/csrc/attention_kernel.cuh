// Paged decode attention kernel: single-pass (v1) and split-KV partition (v2).
//
// One CTA per (partition, kv_head x query-head sub-group, sequence).  The CTA
// serves up to 8 query heads of the kv head's GQA group at once (all of them
// for groups of 8 or fewer), so each K/V byte crosses HBM once (page
// "paged_attention_v2_triton.py": per instance, load Q, gather K/V of the
// partition's tokens, QK^T, online softmax, weighted V; for GQA the group of
// query heads shares the kv head).
//
// Data movement.  A (block, kv_head) page of either cache is one contiguous
// run of head_size*block_size elements (4 KiB at bf16/128/16).  Each warp runs
// its own pipeline of two stages (three in one instance family, see AttnCfg):
// its lane 0 issues cp.async.bulk copies of whole K and V pages into the
// warp's shared-memory stages, tracked by one mbarrier per stage, and the warp
// computes on one stage while the next ones are in flight.
// Warp w of the CTA takes chunks w, w+WARPS, ... of the partition's tokens (a
// chunk is 16 tokens, 32 for one-byte caches in some instances, or one page,
// whichever is larger).
// Block ids are resolved once per 32 chunks: each lane loads the id of one
// upcoming chunk from the block table and the issuing lane picks it up by
// shuffle (the per-token global scratch of the Triton prototype on page
// "Needs help on performance optimization" is not needed).  Whole pages are
// copied, so no load carries a per-token mask; tokens past the end only get a
// -inf logit.
//
// Arithmetic (fp16/bf16).  Scores are S^T = K Q^T on mma.sync m16n8k16: M =
// 16 tokens (ldmatrix reads the x-packed key page directly, 16 B = 8 dims of
// one token per row), N = 8 query heads of the group, K = head dims, fp32
// accumulate.  The output is O^T = V^T P^T: M = 16 head dims (ldmatrix reads
// the value page, whose rows are one dim's tokens), N = 8 heads, K = 16
// tokens; the probabilities go in as a hi + lo pair of 16-bit values
// (movmatrix turns the score accumulator layout into the B-operand layout),
// which keeps their rounding error near fp32.  Softmax runs in the log2
// domain with ex2; row maxima use warp shuffles; a chunk in which no running
// max grew skips the accumulator rescale (its factor would be exactly 1).
//
// fp32 runs the same pipeline with both products on tf32 MMAs, each operand
// split into two tf32 terms (three MMAs per tile), which keeps the products
// close to fp32 rounding.
//
// fp8 caches (E4M3 / E5M2 codes, one byte per element; page
// "paged_attention_v2_triton.py" names kv_cache_dtype, k_scale and v_scale in
// its wrapper, read here as vLLM's dequantisation): the pages move as bytes,
// half the traffic of a 16-bit cache, and each lane widens the codes it needs
// to f16 in registers for the same f16 MMAs.  ldmatrix hands each lane 32-bit
// words of 4 codes, so both products run on permuted index orders: the key row gives
// dims 4j..4j+3 to the MMA's k-slots {2j, 2j+1, 2j+8, 2j+9} (the query
// fragments use the same order), and the score rows hold the tile's tokens in
// the order that puts tokens 4j..4j+3 on the value product's k-slots
// {2j, 2j+1, 2j+8, 2j+9}.  bf16 queries go to f16 with a power-of-two scale
// per head (max |q| lands in [2^14, 2^15)), taken back out of the logit
// scale; k_scale joins the logit scale and v_scale the epilogue; the
// probabilities enter the value product x 256 (exact), keeping small ones
// out of f16 subnormals.
//
// ALiBi (optional slopes): the logit of token t gains slope_h * (t - L + 1),
// added in the log2 domain as slope_h * log2(e) * (t - L + 1).
#pragma once

#include <type_traits>

#include "pkv_ptx.cuh"

namespace pkv {

enum AttnMode : int { kModeV1 = 0, kModeFixed = 1, kModeSplits = 2 };

struct AttnParams {
  const void *q;
  int64_t q_s0, q_s1, q_s2;
  const void *k;
  int64_t k_s0, k_s1;
  const void *v;
  int64_t v_s0, v_s1;
  const int32_t *bt;
  int64_t bt_s0, bt_s1;
  const int32_t *indptr;
  const int32_t *seq_lens;
  int32_t *err;
  int32_t num_heads, num_kv_heads, group, num_blocks, max_blocks_per_seq;
  int32_t head_groups;  // ceil(group / kMaxGroup): CTAs per kv head along grid y
  float scale_log2;  // scale * log2(e)
  int32_t mode;
  void *out;  // v1 output
  int64_t o_s0, o_s1, o_s2;
  float *tmp, *es, *ml;  // v2 outputs
  int32_t max_parts, partition_size;
  const int32_t *splits;
  uint64_t wait_limit_ns;    // limit of every wait for a stage's copies
  uint32_t extra_expect_tx;  // test hook: bytes a stage expects that never arrive (0)
  const float *alibi;        // [num_heads] ALiBi slopes, or null
  float out_scale;           // multiplies the normalised output (v_scale for fp8 caches, else 1)
  const int32_t *order;      // single pass: grid z -> sequence (a permutation), or null
  // Split-KV, two-warp fp8 instances: the CTA of partition slot x also runs
  // partition x + gridDim.x of its sequence when there is one (grid x is
  // about half of max_parts); 0: one partition per CTA.
  int32_t fold;
};

constexpr int kMaxGroup = 8;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

__host__ __device__ constexpr int clamp_int(int v, int lo, int hi) {
  return v < lo ? lo : (v > hi ? hi : v);
}

// KV is the cache element type: T itself, or an fp8 tag.
template <typename KV, int D, int BS, int WARPS>
struct AttnCfg {
  static constexpr int kElem = int(sizeof(KV));
  static constexpr int kX = 16 / kElem;
  // Tokens per pipeline stage: at least 16 (one MMA tile).  One-byte caches
  // with one warp per CTA take 32 up to head size 128, so that a stage's
  // serial softmax step covers as many bytes as a 16-bit cache's; with more
  // warps per CTA the smaller ring keeps more warps resident, which measured
  // faster (at head size 256 a 16-token stage already holds 8 KiB).
  static constexpr int kMinChunk = (kElem == 1 && D <= 128 && WARPS == 1) ? 32 : 16;
  static constexpr int kChunk = BS >= kMinChunk ? BS : kMinChunk;
  static constexpr int kPagesPerChunk = kChunk / BS;
  static constexpr int kMTiles = kChunk / 16;
  static constexpr int kPageBytes = D * BS * kElem;    // one K (or V) page
  static constexpr int kHalfStage = kChunk * D * kElem;  // K (or V) part of a stage
  static constexpr int kStageBytes = 2 * kHalfStage;
  // Two stages per warp: measured, more resident warps beat deeper per-warp
  // rings at every head size (a 16 KiB ring of 4 KiB stages at head size 64
  // loses 2-25 % to two stages).  One exception, also measured: one-byte
  // caches with two warps per CTA and 16-token pages (a chunk is one page:
  // 4 KiB at head size 128) take three stages, whose second chunk of
  // look-ahead covers the copy latency that the shorter column-pair chunk no
  // longer hides (ragged batch 309 -> 305 us).  With 32-token pages three
  // 8 KiB stages cost residency (ragged batch 312 -> 388 us), and one warp
  // with 32-token chunks loses 4 % with three.
  static constexpr int kStages = (kElem == 1 && D <= 128 && WARPS == 2 && BS == 16) ? 3 : 2;
  static constexpr int kWarpBytes = kStages * kStageBytes;
  static constexpr int kEpiFloats = kMaxGroup * D + 2 * kMaxGroup;
  // fp32 caches: per-warp probabilities of one chunk, [head][token] with rows
  // of kChunk + 4 floats (the padding spreads a row's stores over the banks).
  static constexpr int kPRow = kChunk + 4;
  static constexpr int kPBytes = kElem == 4 ? kMaxGroup * kPRow * 4 : 0;
  static constexpr int kBarOffset = WARPS * (kWarpBytes + kPBytes);
  static constexpr int kSmemBytes = kBarOffset + WARPS * kStages * 8;
  static constexpr int kThreads = WARPS * 32;
  static_assert((kEpiFloats + (WARPS + 1) * kMaxGroup) * 4 <= kWarpBytes,
                "epilogue does not fit the warp's stages");
  static_assert(D % 32 == 0 && BS % 8 == 0, "unsupported shape");
  static_assert(kHalfStage % 16 == 0 && kPageBytes % 16 == 0, "bulk copies need 16 B");
  static_assert(kPBytes % 16 == 0 && (kPRow * 4) % 16 == 0, "16-byte probability rows");
};

// CTAs per SM an instance is compiled to keep resident (0: no floor), all
// measured on fp8 caches (elsewhere floors lose):
// - head size 128, two warps per CTA: 10 CTAs (96 registers, a few bytes of
//   spill) beat the 8 that 127 registers allow (ragged batch 360 -> 347 us);
//   9 CTAs gain nothing, and one or four warps per CTA lose;
// - head size 64: 14 two-warp CTAs (ragged 480 -> 459 us) and 6 four-warp
//   CTAs (GQA single pass 128 -> 124 us).
template <typename KV, int D, int WARPS>
constexpr int resident_ctas() {
  if constexpr (!is_fp8<KV>::value) return 0;
  if constexpr (D == 64) return WARPS == 2 ? 14 : (WARPS == 4 ? 6 : 0);
  if constexpr (D == 128) return WARPS == 2 ? 10 : 0;
  return 0;
}

// PAIR (groups of at most 4 query heads): the MMA columns carry two terms
// per head, so one MMA does the work of two (see each body).
template <typename T, typename KV, int D, int BS, int WARPS, bool PAIR>
__global__ void __launch_bounds__(WARPS * 32, (resident_ctas<KV, D, WARPS>()))
    paged_attention_kernel(const AttnParams p) {
  using Cfg = AttnCfg<KV, D, BS, WARPS>;
  constexpr bool kFp8 = is_fp8<KV>::value;
  constexpr bool kMma = !std::is_same<T, float>::value && !kFp8;
  static_assert(kFp8 || std::is_same<T, KV>::value, "a 16/32-bit cache has the query's type");
  static_assert(!kFp8 || !std::is_same<T, float>::value, "fp8 caches take f16/bf16 queries");
  constexpr int PPC = Cfg::kPagesPerChunk;
  constexpr int CH = Cfg::kChunk;
  constexpr int NST = Cfg::kStages;
  constexpr unsigned FULL = 0xffffffffu;

  // Grid y enumerates (kv head, sub-group): a kv head with more than kMaxGroup
  // query heads is served by several CTAs, each taking up to kMaxGroup of them
  // (their page reads after the first mostly hit L2).
  const int kvh = int(blockIdx.y) / p.head_groups;
  const int hsub = int(blockIdx.y) - kvh * p.head_groups;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = min(kMaxGroup, p.group - hsub * kMaxGroup);  // query heads of this CTA
  const bool leader = threadIdx.x == 0;
  grid_dependency_wait();
  allow_dependent_launch();
  int seq = blockIdx.z;
  if (p.order != nullptr) {
    // Caller-given launch order (e.g. longest first); an entry out of range
    // falls back to the identity and is flagged.
    const int s = p.order[blockIdx.z];
    if (s >= 0 && s < int(gridDim.z)) {
      seq = s;
    } else if (leader) {
      flag_error(p.err, 32u);
    }
  }

  // Split-KV over an fp8 cache: most partition slots of a sequence are empty
  // (it fills num_kv_splits of them), and an empty slot's CTA still holds a
  // residency slot while it reads the length and split count, which the
  // latency-bound fp8 kernel feels.  Its two-warp instances therefore can run
  // two partitions per CTA (slots x and x + gridDim.x, grid x about half of
  // max_parts; p.fold, which the launcher sets for batches whose (sequence,
  // kv head) pairs fill the GPU twice), the second one's emptiness known
  // without a further launch.
  constexpr bool kTwoUnits = kFp8 && WARPS == 2;
  int unit_r = 0;
  {
    const int part = blockIdx.x;
    constexpr bool kSecond = false;
    const bool again = false;
#define PKV_UNIT_EXIT(r)   \
  do {                     \
    unit_r = (r);          \
    goto first_unit_done;  \
  } while (0)
#include "attention_unit.inc"
#undef PKV_UNIT_EXIT
  }
first_unit_done:
  if constexpr (kTwoUnits) {
    if (unit_r != 0 && p.fold != 0 && int(blockIdx.x) + int(gridDim.x) < p.max_parts) {
      __syncthreads();  // every thread is done with the ring and the epilogue rows
      const int part = int(blockIdx.x) + int(gridDim.x);
      constexpr bool kSecond = true;
      const bool again = unit_r == 2;
#define PKV_UNIT_EXIT(r) return
#include "attention_unit.inc"
#undef PKV_UNIT_EXIT
    }
  }
}

}  // namespace pkv
