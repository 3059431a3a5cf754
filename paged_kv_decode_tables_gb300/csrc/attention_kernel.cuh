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
  const int part = blockIdx.x;
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

  // ---------------------------------------------------- work decomposition --
  int L = p.seq_lens[seq];
  int64_t row_base;
  int64_t cap_pages;
  if (p.indptr != nullptr) {
    const int a = p.indptr[seq];
    const int b = p.indptr[seq + 1];
    row_base = a;
    cap_pages = int64_t(b) - a;
    if (a < 0 || cap_pages < 0) {
      if (leader) flag_error(p.err, 8u);
      row_base = 0;
      cap_pages = 0;
    }
  } else {
    row_base = int64_t(seq) * p.bt_s0;
    cap_pages = p.max_blocks_per_seq;
  }
  if (L < 0 || int64_t(L) > cap_pages * BS) {
    if (leader) flag_error(p.err, 2u);
    L = L < 0 ? 0 : int(cap_pages * BS);
  }

  int64_t t0, t1;
  if (p.mode == kModeV1) {
    t0 = 0;
    t1 = L;
  } else if (p.mode == kModeFixed) {
    if (int64_t(L) > int64_t(p.max_parts) * p.partition_size) {
      if (leader) flag_error(p.err, 2u);
      L = int(int64_t(p.max_parts) * p.partition_size);
    }
    t0 = int64_t(part) * p.partition_size;
    t1 = min(t0 + p.partition_size, int64_t(L));
  } else {
    int n = p.splits[seq];
    if (L > 0 && (n < 1 || n > p.max_parts)) {
      if (leader) flag_error(p.err, 4u);
      n = clamp_int(n, 1, p.max_parts);
    }
    // chunk = roundup(cdiv(L, n), BS); 32-bit is exact since 0 < L < 2^31
    int64_t c = BS;
    if (L > 0 && n > 0) c = ((unsigned(L) - 1u) / unsigned(n) + BS) / BS * BS;
    t0 = int64_t(part) * c;
    t1 = part < n ? min(t0 + c, int64_t(L)) : t0;
  }

  const int h0 = kvh * p.group + hsub * kMaxGroup;
  if (t0 >= t1) {
    if (p.mode == kModeV1) {
      T *out = static_cast<T *>(p.out);
      for (int i = threadIdx.x; i < g * D; i += blockDim.x) {
        const int h = i / D, d = i % D;
        out[int64_t(seq) * p.o_s0 + int64_t(h0 + h) * p.o_s1 + int64_t(d) * p.o_s2] =
            from_f32<T>(0.f);
      }
    } else {
      for (int h = threadIdx.x; h < g; h += blockDim.x) {
        const int64_t idx = (int64_t(seq) * p.num_heads + h0 + h) * p.max_parts + part;
        p.es[idx] = 0.f;
        p.ml[idx] = -INFINITY;
      }
    }
    return;
  }

  // -------------------------------------------------------------- pipeline --
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *wbase = smem + warp * Cfg::kWarpBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kBarOffset) + warp * NST;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NST; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  const int ntok = int(t1 - t0);
  const int t0i = int(t0), t1i = int(t1);  // token bounds (below 2^31)
  const int nchunks = (ntok + CH - 1) / CH;
  const int my_n = nchunks > warp ? (nchunks - warp + WARPS - 1) / WARPS : 0;
  const int64_t page0 = t0 / BS;
  const uint8_t *kbase =
      static_cast<const uint8_t *>(p.k) + int64_t(kvh) * p.k_s1 * Cfg::kElem;
  const uint8_t *vbase =
      static_cast<const uint8_t *>(p.v) + int64_t(kvh) * p.v_s1 * Cfg::kElem;
  const int64_t kblk = p.k_s0 * Cfg::kElem;
  const int64_t vblk = p.v_s0 * Cfg::kElem;
  const uint64_t policy = l2_policy_evict_first();

  // Lane l holds the block ids of this warp's chunk (32*batch + l).
  int ids_cur[PPC], ids_nxt[PPC];
  auto load_ids = [&](int batch, int (&ids)[PPC]) {
    const int i = batch * 32 + lane;
    const int64_t c = warp + int64_t(WARPS) * i;
#pragma unroll
    for (int j = 0; j < PPC; ++j) {
      int id = -1;
      const int64_t lp = page0 + c * PPC + j;
      if (i < my_n && lp * BS < t1) {
        id = __ldg(p.bt + row_base + lp * p.bt_s1);
        if (id < 0 || id >= p.num_blocks) {
          flag_error(p.err, 1u);
          id = 0;
        }
      }
      ids[j] = id;
    }
  };
  load_ids(0, ids_cur);
  if (my_n > 32) load_ids(1, ids_nxt);
  int batch_cur = 0;
  int issued = 0;

  auto issue_next = [&]() {
    const int i = issued;
    const int b = i >> 5;
    if (b != batch_cur) {
#pragma unroll
      for (int j = 0; j < PPC; ++j) ids_cur[j] = ids_nxt[j];
      batch_cur = b;
      if (my_n > (b + 1) * 32) load_ids(b + 1, ids_nxt);
    }
    int id[PPC];
#pragma unroll
    for (int j = 0; j < PPC; ++j) id[j] = __shfl_sync(FULL, ids_cur[j], i & 31);
    const int st = i % NST;
    if (lane == 0) {
      uint8_t *ks = wbase + st * Cfg::kStageBytes;
      uint8_t *vs = ks + Cfg::kHalfStage;
      uint32_t np = 0;
#pragma unroll
      for (int j = 0; j < PPC; ++j) np += id[j] >= 0 ? 1u : 0u;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&bars[st], np * 2u * Cfg::kPageBytes + p.extra_expect_tx);
#pragma unroll
      for (int j = 0; j < PPC; ++j) {
        if (id[j] >= 0) {
          bulk_copy_g2s(ks + j * Cfg::kPageBytes, kbase + int64_t(id[j]) * kblk, Cfg::kPageBytes,
                        &bars[st], policy);
          bulk_copy_g2s(vs + j * Cfg::kPageBytes, vbase + int64_t(id[j]) * vblk, Cfg::kPageBytes,
                        &bars[st], policy);
        }
      }
    }
    ++issued;
  };

  const int prologue = my_n < NST ? my_n : NST;
  for (int i = 0; i < prologue; ++i) issue_next();

  // Per-warp softmax state and accumulators.
  float *epi = reinterpret_cast<float *>(wbase);  // reused after the pipeline drains
  bool ok = true;
  int waited = 0;

  if constexpr (kMma) {
    constexpr int DT = D / 16;  // 16-dim tiles
    // Column pairs (groups of at most 4 heads): head h takes column 2h of the
    // score product (column 2h + 1 has a zero query) and columns 2h, 2h + 1
    // of the value product carry the hi and lo parts of its probabilities, so
    // one MMA does the work of the hi and lo MMAs; a lane holds head lane%4.
    constexpr bool pair = PAIR;
    // Q^T fragments (B operand): dims 16ks + 2(lane%4) (+1), (+8); column lane/4.
    uint32_t qf[DT][2];
    {
      const int h = pair ? (((lane >> 2) & 1) ? kMaxGroup : (lane >> 3)) : (lane >> 2);
      const uint16_t *qb = static_cast<const uint16_t *>(p.q) + int64_t(seq) * p.q_s0 +
                           int64_t(h0 + min(h, g - 1)) * p.q_s1;
#pragma unroll
      for (int ks = 0; ks < DT; ++ks) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int d = 16 * ks + 2 * (lane & 3) + 8 * half;
          uint32_t lo = 0, hi = 0;
          if (h < g) {
            lo = qb[int64_t(d) * p.q_s2];
            hi = qb[int64_t(d + 1) * p.q_s2];
          }
          qf[ks][half] = lo | (hi << 16);
        }
      }
    }
    // ALiBi slopes (log2 units) of this lane's two score columns: heads
    // 2*(lane%4) and 2*(lane%4)+1 of the CTA (with column pairs: head lane%4).
    float sl2[2] = {0.f, 0.f};
    if (p.alibi != nullptr) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int h = pair ? (j ? kMaxGroup : (lane & 3)) : 2 * (lane & 3) + j;
        if (h < g) sl2[j] = p.alibi[h0 + h] * kLog2e;
      }
    }
    float acc[DT][4];
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) acc[dt][0] = acc[dt][1] = acc[dt][2] = acc[dt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float muse[2] = {0.f, 0.f};  // m_run, or 0 while it is -inf
    float l_run[2] = {0.f, 0.f};

    const int jm = lane >> 3, rr = lane & 7;
    for (int i = 0; i < my_n; ++i) {
      const int st = i % NST;
      const bool got = mbar_wait_bounded(&bars[st], uint32_t(i / NST) & 1u, p.wait_limit_ns);
      if (!__all_sync(FULL, got)) {
        ok = false;
        break;
      }
      waited = i + 1;
      const int tok0 = t0i + (warp + WARPS * i) * CH;  // the chunk's first token
      const int nv = min(CH, t1i - tok0);
      const int pb = tok0 - L + 1;  // ALiBi position of the chunk's token 0
      uint8_t *ks = wbase + st * Cfg::kStageBytes;
      uint8_t *vs = ks + Cfg::kHalfStage;
      if (nv < CH) {
        // Zero the value columns of tokens past the end: their probability
        // is 0, but 0 * (stale or NaN) must not reach the accumulator.
        T *vt = reinterpret_cast<T *>(vs);
        const int ntail = CH - nv;
        for (int e = lane; e < D * ntail; e += 32) {
          const int d = e / ntail;
          const int tau = nv + e % ntail;
          vt[(tau / BS) * (D * BS) + d * BS + (tau % BS)] = from_f32<T>(0.f);
        }
        __syncwarp();
      }
      const uint32_t ks_a = smem_addr(ks);
      const uint32_t vs_a = smem_addr(vs);

      float x[Cfg::kMTiles][4];
#pragma unroll
      for (int mt = 0; mt < Cfg::kMTiles; ++mt) {
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        const int tok = 16 * mt + rr + 8 * (jm & 1);
        const uint32_t rowa =
            ks_a + (tok / BS) * Cfg::kPageBytes + ((jm >> 1) * BS + (tok % BS)) * 16;
#pragma unroll
        for (int k2 = 0; k2 < DT; ++k2) {
          uint32_t a[4];
          ldsm_x4(rowa + k2 * (2 * BS * 16), a[0], a[1], a[2], a[3]);
          if (k2 & 1)
            Mma16816<T>::run(s1, a, qf[k2][0], qf[k2][1]);
          else
            Mma16816<T>::run(s0, a, qf[k2][0], qf[k2][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = 16 * mt + (lane >> 2) + 8 * (e >> 1);
          float v = (s0[e] + s1[e]) * p.scale_log2;
          if (p.alibi != nullptr) v = fmaf(sl2[e & 1], float(pb + t), v);
          x[mt][e] = (t < nv && !(pair && (e & 1))) ? v : -INFINITY;
        }
      }
      // The running max moves only where some lane's score exceeds it: then
      // the column maxima are reduced over the 8 lanes that hold a head's
      // tokens and sums and accumulators are rescaled.  Otherwise every
      // rescale factor would be exactly 1, and the chunk skips the reduction,
      // its shuffle latency and the rescale (same results either way).
      float alpha[2] = {1.f, 1.f};
      bool grow = false;
#pragma unroll
      for (int mt = 0; mt < Cfg::kMTiles; ++mt)
        grow |= fmaxf(x[mt][0], x[mt][2]) > m_run[0] || fmaxf(x[mt][1], x[mt][3]) > m_run[1];
      if (__any_sync(FULL, grow)) {
        float mloc[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int mt = 0; mt < Cfg::kMTiles; ++mt) {
          mloc[0] = fmaxf(mloc[0], fmaxf(x[mt][0], x[mt][2]));
          mloc[1] = fmaxf(mloc[1], fmaxf(x[mt][1], x[mt][3]));
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          mloc[0] = fmaxf(mloc[0], __shfl_xor_sync(FULL, mloc[0], o));
          mloc[1] = fmaxf(mloc[1], __shfl_xor_sync(FULL, mloc[1], o));
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float mn = fmaxf(m_run[j], mloc[j]);
          muse[j] = mn == -INFINITY ? 0.f : mn;
          alpha[j] = ex2(m_run[j] - muse[j]);
          m_run[j] = mn;
        }
        if (pair) alpha[1] = alpha[0];  // both columns hold head lane%4's sums
        if (__any_sync(FULL, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
          for (int dt = 0; dt < DT; ++dt) {
            acc[dt][0] *= alpha[0];
            acc[dt][1] *= alpha[1];
            acc[dt][2] *= alpha[0];
            acc[dt][3] *= alpha[1];
          }
        }
      }
      float pr[Cfg::kMTiles][4];
#pragma unroll
      for (int mt = 0; mt < Cfg::kMTiles; ++mt) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          pr[mt][e] = (pair && (e & 1)) ? 0.f : ex2(x[mt][e] - muse[e & 1]);
      }
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int mt = 0; mt < Cfg::kMTiles; ++mt) {
        ls0 += pr[mt][0] + pr[mt][2];
        ls1 += pr[mt][1] + pr[mt][3];
      }
      l_run[0] = l_run[0] * alpha[0] + ls0;
      l_run[1] = l_run[1] * alpha[1] + ls1;
#pragma unroll
      for (int mt = 0; mt < Cfg::kMTiles; ++mt) {
        uint32_t bh0, bh1, bl0 = 0u, bl1 = 0u;
        if (pair) {
          // Columns 2(lane%4), 2(lane%4)+1: head lane%4's hi and lo parts.
          const float2 f0 = unpack2<T>(pack2<T>(pr[mt][0], 0.f));
          const float2 f1 = unpack2<T>(pack2<T>(pr[mt][2], 0.f));
          bh0 = movmatrix_trans(pack2<T>(pr[mt][0], pr[mt][0] - f0.x));
          bh1 = movmatrix_trans(pack2<T>(pr[mt][2], pr[mt][2] - f1.x));
        } else {
          const uint32_t hi0 = pack2<T>(pr[mt][0], pr[mt][1]);
          const uint32_t hi1 = pack2<T>(pr[mt][2], pr[mt][3]);
          const float2 f0 = unpack2<T>(hi0), f1 = unpack2<T>(hi1);
          const uint32_t lo0 = pack2<T>(pr[mt][0] - f0.x, pr[mt][1] - f0.y);
          const uint32_t lo1 = pack2<T>(pr[mt][2] - f1.x, pr[mt][3] - f1.y);
          bh0 = movmatrix_trans(hi0);
          bh1 = movmatrix_trans(hi1);
          bl0 = movmatrix_trans(lo0);
          bl1 = movmatrix_trans(lo1);
        }
        const int tok0 = 16 * mt + 8 * (jm >> 1);
        const uint32_t rowv = vs_a + (tok0 / BS) * Cfg::kPageBytes + (tok0 % BS) * 2 +
                              (rr + 8 * (jm & 1)) * (BS * 2);
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
          uint32_t a[4];
          ldsm_x4(rowv + dt * (16 * BS * 2), a[0], a[1], a[2], a[3]);
          Mma16816<T>::run(acc[dt], a, bh0, bh1);
          if (!pair) Mma16816<T>::run(acc[dt], a, bl0, bl1);
        }
      }
      __syncwarp();
      if (issued < my_n) issue_next();
    }

    // Full per-head sums: lanes sharing lane%4 hold the same two heads.
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l_run[0] += __shfl_xor_sync(FULL, l_run[0], o);
      l_run[1] += __shfl_xor_sync(FULL, l_run[1], o);
    }
    if (!ok) {
      if (lane == 0) flag_error(p.err, 16u);
      for (int i = waited; i < issued; ++i)
        mbar_wait_bounded(&bars[i % NST], uint32_t(i / NST) & 1u,
                          min(p.wait_limit_ns, uint64_t(100000000ull)));
      __syncwarp();
    }
    // Stage memory of this warp is free now: store O (as [head][dim]), m, l.
    if (pair) {
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
#pragma unroll
        for (int r = 0; r < 2; ++r)
          epi[(lane & 3) * D + 16 * dt + (lane >> 2) + 8 * r] = acc[dt][2 * r] + acc[dt][2 * r + 1];
      }
      if (lane < 4) {
        epi[kMaxGroup * D + lane] = m_run[0];
        epi[kMaxGroup * D + kMaxGroup + lane] = l_run[0];
      }
    } else {
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int d = 16 * dt + (lane >> 2) + 8 * (e >> 1);
          const int h = 2 * (lane & 3) + (e & 1);
          epi[h * D + d] = acc[dt][e];
        }
      }
      if (lane < 4) {
        epi[kMaxGroup * D + 2 * lane] = m_run[0];
        epi[kMaxGroup * D + 2 * lane + 1] = m_run[1];
        epi[kMaxGroup * D + kMaxGroup + 2 * lane] = l_run[0];
        epi[kMaxGroup * D + kMaxGroup + 2 * lane + 1] = l_run[1];
      }
    }
  } else if constexpr (kFp8) {
    // ------------------------------------- fp8 cache, f16 tensor-core body --
    constexpr int DT = D / 16;
    const int gid = lane >> 2, tig = lane & 3;
    // Column pairs: with at most 4 heads in the CTA, head h takes MMA column
    // 2h of the score product (column 2h + 1 has a zero query), and in the
    // value product columns 2h and 2h + 1 carry the hi and lo parts of head
    // h's probabilities, so one MMA does what the hi and lo MMAs do otherwise.
    // A lane then holds one head (tig) instead of two.
    constexpr bool pair = PAIR;
    // Query fragments (B operand, f16) of column gid: dims 16ks + 4tig + {0, 1}
    // on k-slots 2tig, 2tig+1 and dims 16ks + 4tig + {2, 3} on 2tig+8, 2tig+9.
    uint32_t qf[DT][2];
    float head_unscale;  // 2^-k: undoes the f16 range scale 2^k of column gid's query
    {
      const int qh = pair ? ((gid & 1) ? kMaxGroup : (gid >> 1)) : gid;  // head of column gid
      const T *qb = static_cast<const T *>(p.q) + int64_t(seq) * p.q_s0 +
                    int64_t(h0 + min(qh, g - 1)) * p.q_s1;
      float qv[DT][4];
      float amax = 0.f;
#pragma unroll
      for (int ks = 0; ks < DT; ++ks) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int d = 16 * ks + 4 * tig + j;
          qv[ks][j] = qh < g ? to_f32<T>(qb[int64_t(d) * p.q_s2]) : 0.f;
          amax = fmaxf(amax, fabsf(qv[ks][j]));
        }
      }
      int k = 0;
      if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        // bf16 has f32's exponent range: bring max |q| into [2^14, 2^15) so
        // every query element keeps its 8 significant bits in f16.
        amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 2));
        if (amax > 0.f && amax < INFINITY)
          k = clamp_int(141 - int(__float_as_uint(amax) >> 23), -120, 120);
      }
      const float up = __uint_as_float(uint32_t(127 + k) << 23);
      head_unscale = __uint_as_float(uint32_t(127 - k) << 23);
#pragma unroll
      for (int ks = 0; ks < DT; ++ks) {
        qf[ks][0] = pack2<__half>(qv[ks][0] * up, qv[ks][1] * up);
        qf[ks][1] = pack2<__half>(qv[ks][2] * up, qv[ks][3] * up);
      }
    }
    // Logit factor and ALiBi slope (log2 units) of this lane's two score
    // columns 2tig and 2tig+1 (column c's query is on lanes 4c..4c+3): heads
    // 2tig and 2tig+1, or with column pairs head tig and a column not used.
    float xs2[2], sl2[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int c = 2 * tig + j;
      const int h = pair ? (j ? kMaxGroup : tig) : c;
      xs2[j] = p.scale_log2 * __shfl_sync(FULL, head_unscale, 4 * c);
      if (p.alibi != nullptr && h < g) sl2[j] = p.alibi[h0 + h] * kLog2e;
    }
    float acc[DT][4];
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) acc[dt][0] = acc[dt][1] = acc[dt][2] = acc[dt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float muse[2] = {0.f, 0.f};  // m_run, or 0 while it is -inf
    float l_run[2] = {0.f, 0.f};

    // Score row gid holds token rA of each 16-token tile, row gid+8 token rA+2,
    // so that k-slots {2j, 2j+1, 2j+8, 2j+9} of the value product are tokens
    // 4j..4j+3.
    const int rA = 4 * (gid >> 1) + (gid & 1);
    for (int i = 0; i < my_n; ++i) {
      const int st = i % NST;
      const bool got = mbar_wait_bounded(&bars[st], uint32_t(i / NST) & 1u, p.wait_limit_ns);
      if (!__all_sync(FULL, got)) {
        ok = false;
        break;
      }
      waited = i + 1;
      const int tok0 = t0i + (warp + WARPS * i) * CH;  // the chunk's first token
      const int nv = min(CH, t1i - tok0);
      const int pb = tok0 - L + 1;  // ALiBi position of the chunk's token 0
      uint8_t *ks = wbase + st * Cfg::kStageBytes;
      uint8_t *vs = ks + Cfg::kHalfStage;
      if (nv < CH) {
        // Zero the value codes of tokens past the end (code 0 is +0).
        const int ntail = CH - nv;
        for (int e = lane; e < D * ntail; e += 32) {
          const int d = e / ntail;
          const int tau = nv + e % ntail;
          vs[(tau / BS) * (D * BS) + d * BS + (tau % BS)] = 0;
        }
        __syncwarp();
      }

      float x[Cfg::kMTiles][4];
#pragma unroll
      for (int mt = 0; mt < Cfg::kMTiles; ++mt) {
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        // One ldmatrix.x4 returns, per lane, the code words (bytes 4tig..4tig+3
        // of a 16-byte key row) of rows gid (token rA) and gid+8 (token rA+2)
        // for two 16-dim groups: lane l addresses row l%8 of matrix l/8, i.e.
        // token rA(l%8) + 2*((l/8)&1) of group k2 + l/16.
        const int lt = 16 * mt + 4 * ((lane & 7) >> 1) + (lane & 1) + 2 * ((lane >> 3) & 1);
        const uint32_t krow = smem_addr(ks) + (lt / BS) * Cfg::kPageBytes +
                              ((lane >> 4) * BS + (lt % BS)) * 16;
#pragma unroll
        for (int k2 = 0; k2 < DT; k2 += 2) {
          uint32_t w[4];
          ldsm_x4(krow + k2 * (BS * 16), w[0], w[1], w[2], w[3]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t a[4];
            fp8x4_to_f16x2<KV>(w[2 * h], a[0], a[2]);
            fp8x4_to_f16x2<KV>(w[2 * h + 1], a[1], a[3]);
            if (h)
              Mma16816<__half>::run(s1, a, qf[k2 + h][0], qf[k2 + h][1]);
            else
              Mma16816<__half>::run(s0, a, qf[k2 + h][0], qf[k2 + h][1]);
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = 16 * mt + rA + 2 * (e >> 1);
          float v = (s0[e] + s1[e]) * xs2[e & 1];
          if (p.alibi != nullptr) v = fmaf(sl2[e & 1], float(pb + t), v);
          x[mt][e] = (t < nv && !(pair && (e & 1))) ? v : -INFINITY;
        }
      }
      // The running max moves only where some lane's score exceeds it: then
      // the column maxima are reduced over the 8 lanes that hold a head's
      // tokens and sums and accumulators are rescaled.  Otherwise every
      // rescale factor would be exactly 1, and the chunk skips the reduction,
      // its shuffle latency and the rescale (same results either way).
      float alpha[2] = {1.f, 1.f};
      bool grow = false;
#pragma unroll
      for (int mt = 0; mt < Cfg::kMTiles; ++mt)
        grow |= fmaxf(x[mt][0], x[mt][2]) > m_run[0] || fmaxf(x[mt][1], x[mt][3]) > m_run[1];
      if (__any_sync(FULL, grow)) {
        float mloc[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int mt = 0; mt < Cfg::kMTiles; ++mt) {
          mloc[0] = fmaxf(mloc[0], fmaxf(x[mt][0], x[mt][2]));
          mloc[1] = fmaxf(mloc[1], fmaxf(x[mt][1], x[mt][3]));
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          mloc[0] = fmaxf(mloc[0], __shfl_xor_sync(FULL, mloc[0], o));
          mloc[1] = fmaxf(mloc[1], __shfl_xor_sync(FULL, mloc[1], o));
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float mn = fmaxf(m_run[j], mloc[j]);
          muse[j] = mn == -INFINITY ? 0.f : mn;
          alpha[j] = ex2(m_run[j] - muse[j]);
          m_run[j] = mn;
        }
        if (pair) alpha[1] = alpha[0];  // both columns hold head tig's sums
        if (__any_sync(FULL, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
          for (int dt = 0; dt < DT; ++dt) {
            acc[dt][0] *= alpha[0];
            acc[dt][1] *= alpha[1];
            acc[dt][2] *= alpha[0];
            acc[dt][3] *= alpha[1];
          }
        }
      }
      float pr[Cfg::kMTiles][4];
      if (pair) {
#pragma unroll
        for (int mt = 0; mt < Cfg::kMTiles; ++mt) {
          pr[mt][0] = ex2(x[mt][0] - muse[0]);
          pr[mt][2] = ex2(x[mt][2] - muse[0]);
          pr[mt][1] = pr[mt][3] = 0.f;
        }
      } else {
#pragma unroll
        for (int mt = 0; mt < Cfg::kMTiles; ++mt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) pr[mt][e] = ex2(x[mt][e] - muse[e & 1]);
        }
      }
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int mt = 0; mt < Cfg::kMTiles; ++mt) {
        ls0 += pr[mt][0] + pr[mt][2];
        ls1 += pr[mt][1] + pr[mt][3];
      }
      l_run[0] = l_run[0] * alpha[0] + ls0;
      l_run[1] = l_run[1] * alpha[1] + ls1;
#pragma unroll
      for (int mt = 0; mt < Cfg::kMTiles; ++mt) {
        // Probabilities x 256 (exact) keep small ones out of f16 subnormals;
        // the epilogue takes the factor back out.
        uint32_t bh0, bh1, bl0 = 0u, bl1 = 0u;
        if (pair) {
          // Columns 2tig, 2tig+1 of rows gid and gid+8: head tig's hi and lo.
          const float q0 = pr[mt][0] * 256.f, q2 = pr[mt][2] * 256.f;
          const float h0f = __half2float(__float2half_rn(q0));
          const float h2f = __half2float(__float2half_rn(q2));
          bh0 = movmatrix_trans(pack2<__half>(q0, q0 - h0f));
          bh1 = movmatrix_trans(pack2<__half>(q2, q2 - h2f));
        } else {
          const float q0 = pr[mt][0] * 256.f, q1 = pr[mt][1] * 256.f;
          const float q2 = pr[mt][2] * 256.f, q3 = pr[mt][3] * 256.f;
          const uint32_t hi0 = pack2<__half>(q0, q1);
          const uint32_t hi1 = pack2<__half>(q2, q3);
          const float2 f0 = unpack2<__half>(hi0), f1 = unpack2<__half>(hi1);
          const uint32_t lo0 = pack2<__half>(q0 - f0.x, q1 - f0.y);
          const uint32_t lo1 = pack2<__half>(q2 - f1.x, q3 - f1.y);
          bh0 = movmatrix_trans(hi0);
          bh1 = movmatrix_trans(hi1);
          bl0 = movmatrix_trans(lo0);
          bl1 = movmatrix_trans(lo1);
        }
        if constexpr (BS >= 16) {
          // A value row holds a dim's 16 tokens of the tile in 16 bytes: one
          // ldmatrix.x4 gives the words of dims gid, gid+8 for two dim tiles
          // (lane l addresses dim 16*(l/16) + 8*((l/8)&1) + l%8).
          const int ld = 16 * (lane >> 4) + 8 * ((lane >> 3) & 1) + (lane & 7);
          const uint32_t vrow = smem_addr(vs) + ((16 * mt) / BS) * Cfg::kPageBytes +
                                (16 * mt) % BS + ld * BS;
#pragma unroll
          for (int dt = 0; dt < DT; dt += 2) {
            uint32_t w[4];
            ldsm_x4(vrow + (16 * dt) * BS, w[0], w[1], w[2], w[3]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t a[4];
              fp8x4_to_f16x2<KV>(w[2 * h], a[0], a[2]);
              fp8x4_to_f16x2<KV>(w[2 * h + 1], a[1], a[3]);
              Mma16816<__half>::run(acc[dt + h], a, bh0, bh1);
              if (!pair) Mma16816<__half>::run(acc[dt + h], a, bl0, bl1);
            }
          }
        } else {
          // 8-token pages: the tile's 16 tokens of a dim sit in two pages.
          const int tok0 = 16 * mt + 4 * tig;
          const uint8_t *va = vs + (tok0 / BS) * Cfg::kPageBytes + (tok0 % BS) + gid * BS;
#pragma unroll
          for (int dt = 0; dt < DT; ++dt) {
            const uint32_t wa = *reinterpret_cast<const uint32_t *>(va + (16 * dt) * BS);
            const uint32_t wb = *reinterpret_cast<const uint32_t *>(va + (16 * dt + 8) * BS);
            uint32_t a[4];
            fp8x4_to_f16x2<KV>(wa, a[0], a[2]);
            fp8x4_to_f16x2<KV>(wb, a[1], a[3]);
            Mma16816<__half>::run(acc[dt], a, bh0, bh1);
            if (!pair) Mma16816<__half>::run(acc[dt], a, bl0, bl1);
          }
        }
      }
      __syncwarp();
      if (issued < my_n) issue_next();
    }

#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l_run[0] += __shfl_xor_sync(FULL, l_run[0], o);
      l_run[1] += __shfl_xor_sync(FULL, l_run[1], o);
    }
    if (!ok) {
      if (lane == 0) flag_error(p.err, 16u);
      for (int i = waited; i < issued; ++i)
        mbar_wait_bounded(&bars[i % NST], uint32_t(i / NST) & 1u,
                          min(p.wait_limit_ns, uint64_t(100000000ull)));
      __syncwarp();
    }
    if (pair) {
      // Head tig: the hi and lo columns' sums add up.
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int d = 16 * dt + gid + 8 * r;
          epi[tig * D + d] = (acc[dt][2 * r] + acc[dt][2 * r + 1]) * (1.f / 256.f);
        }
      }
      if (lane < 4) {
        epi[kMaxGroup * D + lane] = m_run[0];
        epi[kMaxGroup * D + kMaxGroup + lane] = l_run[0];
      }
    } else {
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int d = 16 * dt + gid + 8 * (e >> 1);
          const int h = 2 * tig + (e & 1);
          epi[h * D + d] = acc[dt][e] * (1.f / 256.f);
        }
      }
      if (lane < 4) {
        epi[kMaxGroup * D + 2 * lane] = m_run[0];
        epi[kMaxGroup * D + 2 * lane + 1] = m_run[1];
        epi[kMaxGroup * D + kMaxGroup + 2 * lane] = l_run[0];
        epi[kMaxGroup * D + kMaxGroup + 2 * lane + 1] = l_run[1];
      }
    }
  } else {
    // ------------------------------------------- fp32, 3xTF32 tensor body --
    // Both products on mma.sync m16n8k8 tf32.  Every operand x is split as
    // hi + lo (split_tf32: two tf32 values, |x - hi - lo| <= 2^-22 |x|) and
    // a product ab is taken as hi_a hi_b + hi_a lo_b + lo_a hi_b, leaving out
    // lo_a lo_b (<= 2^-22 |ab|): close to fp32 rounding at three MMAs per tile.
    // Scores S^T = K Q^T: M = 16 tokens, N = 8 heads, K = 8 dims; ldmatrix
    // reads the key page (16-byte rows = 4 dims of one token): matrices
    // (tokens 0-7 | 8-15) x (dims 8kk..8kk+3 | 8kk+4..8kk+7) are exactly the
    // tf32 A fragment, k-slot c = dim 8kk + c.  Output O^T = V^T P^T: M = 16
    // head dims, N = 8 heads, K = 8 tokens; each lane reads 4 consecutive
    // tokens 4tig..4tig+3 of one dim row of the value page in 16 bytes and
    // puts them on k-slots (tig, tig+4) of two MMAs: k-step 0 takes tokens
    // 4tig and 4tig+1, k-step 1 tokens 4tig+2 and 4tig+3.  The probabilities
    // reach that order through a per-warp [head][token] array in shared
    // memory.
    // Column pairs (at most 4 heads in the CTA): columns 2h and 2h + 1 of
    // both products carry the hi and lo terms of head h's query (probabilities),
    // so one MMA per A term covers both B terms: two MMAs per tile instead of
    // three (and the small lo lo term comes along).  A lane then holds one
    // head (tig), its score the sum of its two columns.
    constexpr int DK = D / 8;   // 8-dim k-steps of the key product
    constexpr int DT = D / 16;  // 16-dim tiles of the value product
    const int gid = lane >> 2, tig = lane & 3;
    constexpr bool pair = PAIR;
    // Query fragments (B operand): column gid, dims 8kk + tig and 8kk + tig + 4;
    // with column pairs qh holds column gid's term (hi of head gid/2 for even
    // gid, lo for odd) and ql is not used.
    uint32_t qh[DK][2], ql[DK][2];
    {
      const int qhd = pair ? (gid >> 1) : gid;  // head of column gid
      const float *qb = static_cast<const float *>(p.q) + int64_t(seq) * p.q_s0 +
                        int64_t(h0 + min(qhd, g - 1)) * p.q_s1;
#pragma unroll
      for (int kk = 0; kk < DK; ++kk) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float v = qhd < g ? qb[int64_t(8 * kk + tig + 4 * j) * p.q_s2] : 0.f;
          split_tf32(v, qh[kk][j], ql[kk][j]);
          if (pair && (gid & 1)) qh[kk][j] = ql[kk][j];
        }
      }
    }
    float sl2[2] = {0.f, 0.f};  // ALiBi slopes (log2 units) of this lane's heads
    if (p.alibi != nullptr) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int h = pair ? (j ? kMaxGroup : tig) : 2 * tig + j;
        if (h < g) sl2[j] = p.alibi[h0 + h] * kLog2e;
      }
    }
    float acc[DT][4];
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) acc[dt][0] = acc[dt][1] = acc[dt][2] = acc[dt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float muse[2] = {0.f, 0.f};  // m_run, or 0 while it is -inf
    float l_run[2] = {0.f, 0.f};
    // Compensation terms of l_run (Kahan summation).  Once one token holds
    // most of a head's mass, l_run sits near its final value while a chunk
    // adds far less than half an ulp of it; plain fp32 adds would drop every
    // such addition, always in the same direction, so the loss would grow
    // with the chunks a warp walks (2.4e-5 after 9000 peaky tokens).
    float l_c[2] = {0.f, 0.f};
    float *pw = reinterpret_cast<float *>(smem + WARPS * Cfg::kWarpBytes + warp * Cfg::kPBytes);

    const int jm = lane >> 3, rr = lane & 7;
    for (int i = 0; i < my_n; ++i) {
      const int st = i % NST;
      const bool got = mbar_wait_bounded(&bars[st], uint32_t(i / NST) & 1u, p.wait_limit_ns);
      if (!__all_sync(FULL, got)) {
        ok = false;
        break;
      }
      waited = i + 1;
      const int tok0 = t0i + (warp + WARPS * i) * CH;  // the chunk's first token
      const int nv = min(CH, t1i - tok0);
      const int pb = tok0 - L + 1;  // ALiBi position of the chunk's token 0
      uint8_t *ks = wbase + st * Cfg::kStageBytes;
      uint8_t *vs = ks + Cfg::kHalfStage;
      if (nv < CH) {
        // Zero the value columns of tokens past the end: their probability
        // is 0, but 0 * (stale or NaN) must not reach the accumulator.
        float *vt = reinterpret_cast<float *>(vs);
        const int ntail = CH - nv;
        for (int e = lane; e < D * ntail; e += 32) {
          const int d = e / ntail;
          const int tau = nv + e % ntail;
          vt[(tau / BS) * (D * BS) + d * BS + (tau % BS)] = 0.f;
        }
        __syncwarp();
      }
      const uint32_t ks_a = smem_addr(ks);

      float x[Cfg::kMTiles][4];
#pragma unroll
      for (int mt = 0; mt < Cfg::kMTiles; ++mt) {
        // Two accumulators for the leading terms, two for the corrections
        // (even / odd k-steps), summed small-first.
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
        const int tok = 16 * mt + rr + 8 * (jm & 1);
        const uint32_t rowa =
            ks_a + (tok / BS) * Cfg::kPageBytes + ((jm >> 1) * BS + (tok % BS)) * 16;
#pragma unroll
        for (int kk = 0; kk < DK; ++kk) {
          uint32_t a[4], ah[4], al[4];
          ldsm_x4(rowa + kk * (2 * BS * 16), a[0], a[1], a[2], a[3]);
#pragma unroll
          for (int e = 0; e < 4; ++e) split_tf32_fast(__uint_as_float(a[e]), ah[e], al[e]);
          float(&sa)[4] = (kk & 1) ? s1 : s0;
          float(&ca)[4] = (kk & 1) ? c1 : c0;
          mma_tf32_16808(ca, al[0], al[1], al[2], al[3], qh[kk][0], qh[kk][1]);
          if (!pair) mma_tf32_16808(ca, ah[0], ah[1], ah[2], ah[3], ql[kk][0], ql[kk][1]);
          mma_tf32_16808(sa, ah[0], ah[1], ah[2], ah[3], qh[kk][0], qh[kk][1]);
        }
        if (pair) {
          // Column 2tig: hi K x hi q (s) and lo K x hi q (c); column 2tig+1:
          // the same with lo q.
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int t = 16 * mt + gid + 8 * r;
            const float small =
                ((c0[2 * r + 1] + c1[2 * r + 1]) + (c0[2 * r] + c1[2 * r])) +
                (s0[2 * r + 1] + s1[2 * r + 1]);
            float v = (small + (s0[2 * r] + s1[2 * r])) * p.scale_log2;
            if (p.alibi != nullptr) v = fmaf(sl2[0], float(pb + t), v);
            x[mt][2 * r] = t < nv ? v : -INFINITY;
            x[mt][2 * r + 1] = -INFINITY;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int t = 16 * mt + gid + 8 * (e >> 1);
            float v = ((c0[e] + c1[e]) + (s0[e] + s1[e])) * p.scale_log2;
            if (p.alibi != nullptr) v = fmaf(sl2[e & 1], float(pb + t), v);
            x[mt][e] = t < nv ? v : -INFINITY;
          }
        }
      }
      // Running max and probabilities as in the 16-bit body; the rescale
      // joins the chunk's sums below.
      float alpha[2] = {1.f, 1.f};
      bool grow = false;
#pragma unroll
      for (int mt = 0; mt < Cfg::kMTiles; ++mt)
        grow |= fmaxf(x[mt][0], x[mt][2]) > m_run[0] || fmaxf(x[mt][1], x[mt][3]) > m_run[1];
      if (__any_sync(FULL, grow)) {
        float mloc[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int mt = 0; mt < Cfg::kMTiles; ++mt) {
          mloc[0] = fmaxf(mloc[0], fmaxf(x[mt][0], x[mt][2]));
          mloc[1] = fmaxf(mloc[1], fmaxf(x[mt][1], x[mt][3]));
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          mloc[0] = fmaxf(mloc[0], __shfl_xor_sync(FULL, mloc[0], o));
          mloc[1] = fmaxf(mloc[1], __shfl_xor_sync(FULL, mloc[1], o));
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float mn = fmaxf(m_run[j], mloc[j]);
          muse[j] = mn == -INFINITY ? 0.f : mn;
          alpha[j] = ex2(m_run[j] - muse[j]);
          m_run[j] = mn;
        }
        if (pair) alpha[1] = alpha[0];  // both columns hold head tig's sums
      }
      float ls0 = 0.f, ls1 = 0.f;
      if (pair) {
#pragma unroll
        for (int mt = 0; mt < Cfg::kMTiles; ++mt) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const float pr = ex2(x[mt][2 * r] - muse[0]);
            ls0 += pr;
            pw[tig * Cfg::kPRow + 16 * mt + gid + 8 * r] = pr;
          }
        }
      } else {
#pragma unroll
        for (int mt = 0; mt < Cfg::kMTiles; ++mt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float pr = ex2(x[mt][e] - muse[e & 1]);
            if (e & 1)
              ls1 += pr;
            else
              ls0 += pr;
            pw[(2 * tig + (e & 1)) * Cfg::kPRow + 16 * mt + gid + 8 * (e >> 1)] = pr;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float lsj = j ? ls1 : ls0;
        const float lr = __fmul_rn(l_run[j], alpha[j]);
        const float y = lsj - __fmul_rn(l_c[j], alpha[j]);
        const float t = __fadd_rn(lr, y);
        l_c[j] = __fsub_rn(__fsub_rn(t, lr), y);
        l_run[j] = t;
      }
      __syncwarp();
      // The chunk's value products accumulate from zero and join the running
      // sums with one fp32 FMA each (acc * alpha + chunk): the tensor core's
      // accumulation does not round to nearest, so adding every MMA into a
      // long-lived accumulator would let its rounding grow with the length.
      float cacc[DT][4];
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) cacc[dt][0] = cacc[dt][1] = cacc[dt][2] = cacc[dt][3] = 0.f;
#pragma unroll
      for (int mt = 0; mt < Cfg::kMTiles; ++mt) {
        // B fragments: column gid, tokens 16mt + 4tig + {0, 1} (k-step 0) and
        // + {2, 3} (k-step 1); with column pairs ph holds column gid's term
        // of head gid/2 (hi for even gid, lo for odd).
        const int prow = pair ? (gid >> 1) : gid;
        const float4 pq = *reinterpret_cast<const float4 *>(pw + prow * Cfg::kPRow + 16 * mt +
                                                            4 * tig);
        uint32_t ph[4], pl[4];
        split_tf32_fast(pq.x, ph[0], pl[0]);
        split_tf32_fast(pq.y, ph[1], pl[1]);
        split_tf32_fast(pq.z, ph[2], pl[2]);
        split_tf32_fast(pq.w, ph[3], pl[3]);
        if (pair && (gid & 1)) {
#pragma unroll
          for (int e = 0; e < 4; ++e) ph[e] = pl[e];
        }
        const int tv = 16 * mt + 4 * tig;
        const float *vrow = reinterpret_cast<const float *>(vs + (tv / BS) * Cfg::kPageBytes) +
                            gid * BS + (tv % BS);
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
          const float4 va = *reinterpret_cast<const float4 *>(vrow + (16 * dt) * BS);
          const float4 vb = *reinterpret_cast<const float4 *>(vrow + (16 * dt + 8) * BS);
          uint32_t ah[8], al[8];
          split_tf32_fast(va.x, ah[0], al[0]);
          split_tf32_fast(vb.x, ah[1], al[1]);
          split_tf32_fast(va.y, ah[2], al[2]);
          split_tf32_fast(vb.y, ah[3], al[3]);
          split_tf32_fast(va.z, ah[4], al[4]);
          split_tf32_fast(vb.z, ah[5], al[5]);
          split_tf32_fast(va.w, ah[6], al[6]);
          split_tf32_fast(vb.w, ah[7], al[7]);
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int o = 4 * k;
            mma_tf32_16808(cacc[dt], al[o], al[o + 1], al[o + 2], al[o + 3], ph[2 * k],
                           ph[2 * k + 1]);
            if (!pair)
              mma_tf32_16808(cacc[dt], ah[o], ah[o + 1], ah[o + 2], ah[o + 3], pl[2 * k],
                             pl[2 * k + 1]);
            mma_tf32_16808(cacc[dt], ah[o], ah[o + 1], ah[o + 2], ah[o + 3], ph[2 * k],
                           ph[2 * k + 1]);
          }
        }
      }
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[dt][e] = fmaf(acc[dt][e], alpha[e & 1], cacc[dt][e]);
      }
      __syncwarp();
      if (issued < my_n) issue_next();
    }

    // Full per-head sums: lanes sharing lane%4 hold the same two heads.
    l_run[0] -= l_c[0];
    l_run[1] -= l_c[1];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l_run[0] += __shfl_xor_sync(FULL, l_run[0], o);
      l_run[1] += __shfl_xor_sync(FULL, l_run[1], o);
    }
    if (!ok) {
      if (lane == 0) flag_error(p.err, 16u);
      for (int i = waited; i < issued; ++i)
        mbar_wait_bounded(&bars[i % NST], uint32_t(i / NST) & 1u,
                          min(p.wait_limit_ns, uint64_t(100000000ull)));
      __syncwarp();
    }
    if (pair) {
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
#pragma unroll
        for (int r = 0; r < 2; ++r)
          epi[tig * D + 16 * dt + gid + 8 * r] = acc[dt][2 * r] + acc[dt][2 * r + 1];
      }
      if (lane < 4) {
        epi[kMaxGroup * D + lane] = m_run[0];
        epi[kMaxGroup * D + kMaxGroup + lane] = l_run[0];
      }
    } else {
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int d = 16 * dt + gid + 8 * (e >> 1);
          const int h = 2 * tig + (e & 1);
          epi[h * D + d] = acc[dt][e];
        }
      }
      if (lane < 4) {
        epi[kMaxGroup * D + 2 * lane] = m_run[0];
        epi[kMaxGroup * D + 2 * lane + 1] = m_run[1];
        epi[kMaxGroup * D + kMaxGroup + 2 * lane] = l_run[0];
        epi[kMaxGroup * D + kMaxGroup + 2 * lane + 1] = l_run[1];
      }
    }
  }

  // ---------------------------------------------- combine warps, write out --
  // Per head, once: the warps' weights 2^(m_w - M), the total L and the
  // output factor out_scale / L (and the split-KV statistics); then every
  // element is a weighted sum of the warps' rows and one multiply.
  // They sit in warp 0's ring after its epilogue rows (every copy has landed).
  float(*head_w)[kMaxGroup] =
      reinterpret_cast<float(*)[kMaxGroup]>(smem + Cfg::kEpiFloats * 4);
  float *head_fac = reinterpret_cast<float *>(smem + Cfg::kEpiFloats * 4) + WARPS * kMaxGroup;
  if constexpr (WARPS > 1) {
    __syncthreads();
  } else {
    __syncwarp();
  }
  if (threadIdx.x < g) {
    const int h = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
      const float *ew = reinterpret_cast<const float *>(smem + w * Cfg::kWarpBytes);
      M = fmaxf(M, ew[kMaxGroup * D + h]);
    }
    float Ls = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
      const float *ew = reinterpret_cast<const float *>(smem + w * Cfg::kWarpBytes);
      const float f = ex2(ew[kMaxGroup * D + h] - M);
      head_w[w][h] = f;
      Ls = fmaf(f, ew[kMaxGroup * D + kMaxGroup + h], Ls);
    }
    head_fac[h] = __fdiv_rn(p.out_scale, Ls);
    if (p.mode != kModeV1) {
      const int64_t row = (int64_t(seq) * p.num_heads + h0 + h) * p.max_parts + part;
      p.es[row] = Ls;
      p.ml[row] = M * kLn2;
    }
  }
  if constexpr (WARPS > 1) {
    __syncthreads();
  } else {
    __syncwarp();
  }
  for (int idx = threadIdx.x; idx < g * D; idx += WARPS * 32) {
    const int h = idx / D, d = idx % D;
    float O = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
      const float *ew = reinterpret_cast<const float *>(smem + w * Cfg::kWarpBytes);
      O = fmaf(head_w[w][h], ew[h * D + d], O);
    }
    const float r = O * head_fac[h];
    if (p.mode == kModeV1) {
      T *out = static_cast<T *>(p.out);
      out[int64_t(seq) * p.o_s0 + int64_t(h0 + h) * p.o_s1 + int64_t(d) * p.o_s2] = from_f32<T>(r);
    } else {
      const int64_t row = (int64_t(seq) * p.num_heads + h0 + h) * p.max_parts + part;
      p.tmp[row * D + d] = r;
    }
  }
}

}  // namespace pkv
