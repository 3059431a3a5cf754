// Paged decode over fp8 (E4M3 / E5M2) caches on the 5th-generation tensor
// cores: tcgen05 MMAs with both operands read from shared memory and the
// accumulators in tensor memory (TMEM).  Head size 128, block size 16.
//
// Same computation and outputs as paged_attention_kernel (page
// "paged_attention_v2_triton.py": per instance, gather K/V of the partition's
// tokens through the block table, QK^T, softmax, weighted V; the split-KV
// outputs are the normalised partial output, the exp sum and the max logit),
// with the cache dequantisation of the wrapper's kv_cache_dtype / k_scale /
// v_scale arguments (a key element is decode(code) * k_scale, a value element
// decode(code) * v_scale).
//
// Work.  The grid is the usual one (partition, kv head x head sub-group,
// sequence), but CTAs are persistent: a CTA starts on its own unit and then
// takes units that have not started yet from the hardware's launch queue
// (cluster launch control, try_cancel), in launch order, until the queue is
// empty.  Empty units (partitions past a sequence's end) cost one such
// request and a few stores; the pipeline of a CTA runs on across units.
//
// Roles (256 threads):
//   warp 6 (scheduler): launch-queue requests, two in flight; the unit's
//     token range from the lengths, split counts or indptr and its first 32
//     block ids; empty units' outputs; non-empty units into a ring of 4
//     descriptors;
//   warp 4 (copies): per tile of 128 tokens (8 pages), the key and value
//     pages by whole-page bulk copies;
//   warp 7 (key layout): a tile's key pages arrive as [page][16-dim group]
//     [16 tokens][16 B]; swapping the 256-byte blocks (page, group) and
//     (group, page) in place makes them the canonical K-major layout of an
//     MMA operand with the tile's 128 tokens as rows.  (A value page [128
//     dims][16 tokens] already is such an operand, dims as rows.)
//   warp 5 (MMA issue, one thread): S = K Q^T (M = 128 tokens, N = query
//     terms x heads, K = 128 dims, 4 MMAs) into one of two TMEM score
//     buffers; O^T += V^T P^T (M = 128 dims, N = probability terms x heads,
//     K = 128 tokens, 4 MMAs) into the unit's TMEM output buffer (two, one
//     per unit in flight);
//   warps 0-3 (softmax, one token per thread): the unit's query operand (the
//     next unit's query is loaded a unit ahead); per tile the logits, the
//     running max, the probabilities as MMA operand; per unit the epilogue
//     (normalised output, exp sums, max logits), run after the next unit's
//     first tile so that the last value product's latency is hidden.
// Both products run kind::f8f6f4 on the cache codes as stored: no widening.
// The query enters as an exact sum of E4M3 terms (bf16: 2, f16: 3) with a
// power-of-two scale per head; a probability p in [0, 256] enters as four
// E4M3 terms p = c0 + c1/16 + c2/256 + c3/4096 (each the residual of the
// previous ones, rounded to nearest), which keeps about 16 significant bits.
// The running max is lazy: it moves only when a logit exceeds it by more than
// 2^8 (log2 units), and then the output accumulator in TMEM is rescaled; the
// true max is tracked apart for the max_logits output.
//
// Every wait is bounded; a wait that runs out raises a CTA-wide abort flag,
// every role winds down (waiting, bounded, for its own copies and MMAs in
// flight), TMEM is freed and the error flag gets PKV_ERRF_TIMEOUT.
#pragma once

#include <type_traits>

#include "attention_kernel.cuh"
#include "tc_ptx.cuh"

namespace pkv {

constexpr int kTcD = 128;          // head size
constexpr int kTcBS = 16;          // block size (tokens per page)
constexpr int kTcTokens = 128;     // tokens per tile
constexpr int kTcPages = kTcTokens / kTcBS;
constexpr int kTcPageBytes = kTcD * kTcBS;     // one key (or value) page of codes
constexpr int kTcHalf = kTcTokens * kTcD;      // bytes of a tile's key (or value) codes
constexpr int kTcStage = 2 * kTcHalf;
constexpr int kTcWarpCopy = 4, kTcWarpMma = 5, kTcWarpSched = 6, kTcWarpLayout = 7;
constexpr int kTcThreads = 256;
constexpr int kTcRing = 4;         // unit descriptors in flight
constexpr float kTcRescale = 8.f;  // log2 units the running max may lag behind

// One non-empty unit (a partition of one sequence for one kv head's query
// head sub-group), or the end mark.
struct TcUnit {
  int32_t end, seq, part, kvh, hsub, L;
  int64_t t0, t1, row_base;
  int32_t ids[32];  // block ids of the unit's first 32 pages (checked, clamped)
};

// Where a unit's output goes (kept for its deferred epilogue).
struct TcOut {
  int32_t seq, part, kvh, hsub;
};

// GP: query heads per CTA rounded up (4 or 8).
template <typename T, int GP>
struct TcCfg {
  static constexpr int kTerms = std::is_same<T, __nv_bfloat16>::value ? 2 : 3;
  static constexpr int kNK = (kTerms * GP + 15) / 16 * 16;  // N of the key product
  static constexpr int kNV = 4 * GP;                          // N of the value product
  static constexpr int kQBytes = kNK * kTcD;
  static constexpr int kPBytes = kNV * kTcTokens;
  static constexpr int kMiscBytes = 2048;
  // Three stages when two CTAs still fit on an SM (228 KB, 1 KB of it
  // reserved per CTA), else two.
  static constexpr int kFixed = 2 * kQBytes + 2 * kPBytes + kMiscBytes;
  static constexpr int NS = 2 * (kFixed + 3 * kTcStage + 1024) <= 233472 ? 3 : 2;
  static constexpr int kQOff = NS * kTcStage;
  static constexpr int kPOff = kQOff + 2 * kQBytes;
  static constexpr int kMiscOff = kPOff + 2 * kPBytes;
  static constexpr int kSmemBytes = kMiscOff + kMiscBytes;
  static constexpr uint32_t kTmemCols = 128;
  static constexpr int kOCol = 2 * kNK;  // output buffer u at kOCol + u * kNV
  // K-major query operand: row n = term * GP + head, 128 dims; core matrices
  // adjacent along K (16 dims) kQLbo apart, along N 128 bytes apart.
  static constexpr uint32_t kQLbo = (kNK / 8) * 128;
  // MN-major probability operand: token t, column n = term * GP + head at
  // (t / 8) * kPKStride + (n / 16) * 128 + (t % 8) * 16 + n % 16; as for
  // K-major operands, the descriptor's LBO is the K-direction stride
  // (kPKStride, 8 tokens) and SBO the N-direction one (128, 16 columns).
  static constexpr uint32_t kPKStride = (kNV / 16) * 128;
  static_assert(kOCol + 2 * kNV <= int(kTmemCols), "TMEM columns");
  static_assert(GP == 4 || GP == 8, "heads per CTA");
};

// Bounded wait on an mbarrier phase that also gives up as soon as another
// role of the CTA has (shared `abort` flag); a wait that runs out sets it.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                        volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0; i < (1u << 28); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort = 1;
        return false;
      }
    }
  }
  *abort = 1;
  return false;
}

// Token range of unit (part, seq) and the row of its block ids, from the
// decomposition of paged_attention_kernel (v1: the whole sequence; fixed
// partitions; or chunks of roundup(cdiv(L, n), block_size) for n splits).
// Bad lengths, split counts and indptr rows are clamped and flagged.
__device__ __forceinline__ void tc_unit_range(const AttnParams &p, int part, int seq, bool flag,
                                              int &L_out, int64_t &t0, int64_t &t1,
                                              int64_t &row_base) {
  int L = p.seq_lens[seq];
  int64_t cap_pages;
  if (p.indptr != nullptr) {
    const int a = p.indptr[seq];
    const int b = p.indptr[seq + 1];
    row_base = a;
    cap_pages = int64_t(b) - a;
    if (a < 0 || cap_pages < 0) {
      if (flag) flag_error(p.err, 8u);
      row_base = 0;
      cap_pages = 0;
    }
  } else {
    row_base = int64_t(seq) * p.bt_s0;
    cap_pages = p.max_blocks_per_seq;
  }
  if (L < 0 || int64_t(L) > cap_pages * kTcBS) {
    if (flag) flag_error(p.err, 2u);
    L = L < 0 ? 0 : int(cap_pages * kTcBS);
  }
  if (p.mode == kModeV1) {
    t0 = 0;
    t1 = L;
  } else if (p.mode == kModeFixed) {
    if (int64_t(L) > int64_t(p.max_parts) * p.partition_size) {
      if (flag) flag_error(p.err, 2u);
      L = int(int64_t(p.max_parts) * p.partition_size);
    }
    t0 = int64_t(part) * p.partition_size;
    t1 = min(t0 + p.partition_size, int64_t(L));
  } else {
    int n = p.splits[seq];
    if (L > 0 && (n < 1 || n > p.max_parts)) {
      if (flag) flag_error(p.err, 4u);
      n = clamp_int(n, 1, p.max_parts);
    }
    int64_t c = kTcBS;
    if (L > 0 && n > 0) c = ((unsigned(L) - 1u) / unsigned(n) + kTcBS) / kTcBS * kTcBS;
    t0 = int64_t(part) * c;
    t1 = part < n ? min(t0 + c, int64_t(L)) : t0;
  }
  L_out = L;
}

// Block id of page `lp` of a unit (lane-parallel); out-of-range ids are
// flagged and read as block 0; pages past the unit give -1.
__device__ __forceinline__ int tc_block_id(const AttnParams &p, int64_t row_base, int64_t page0,
                                           int64_t npages, int64_t lp) {
  int id = -1;
  if (lp < npages) {
    id = __ldg(p.bt + row_base + (page0 + lp) * p.bt_s1);
    if (id < 0 || id >= p.num_blocks) {
      flag_error(p.err, 1u);
      id = 0;
    }
  }
  return id;
}

template <typename T, typename KV, int GP>
__global__ void __launch_bounds__(kTcThreads, 2)
    paged_attention_fp8_tc_kernel(const AttnParams p) {
  using Cfg = TcCfg<T, GP>;
  constexpr int NK = Cfg::kNK, NV = Cfg::kNV, TQ = Cfg::kTerms, NS = Cfg::NS;
  constexpr uint32_t kFmt = std::is_same<KV, fp8_e5m2_t>::value ? tc::kFmtE5M2 : tc::kFmtE4M3;
  constexpr unsigned FULL = 0xffffffffu;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  grid_dependency_wait();
  allow_dependent_launch();

  // ------------------------------------------------------- shared memory --
  extern __shared__ __align__(1024) uint8_t tc_smem[];
  uint8_t *smem = tc_smem;
  uint8_t *qs = smem + Cfg::kQOff;  // [2] query operands (one per unit in flight)
  uint8_t *ps = smem + Cfg::kPOff;  // [2] probability operands (by tile parity)
  uint8_t *misc = smem + Cfg::kMiscOff;
  uint64_t *bars = reinterpret_cast<uint64_t *>(misc);
  uint64_t *k_raw = bars + 0;        // [NS] key pages landed (tx bytes)
  uint64_t *k_full = bars + 4;       // [NS] key tile in operand layout (layout warp)
  uint64_t *v_full = bars + 8;       // [NS] value pages landed (tx bytes)
  uint64_t *stage_free = bars + 12;  // [NS] value product of the stage's tile done (commit)
  uint64_t *p_full = bars + 16;      // [2] probabilities written (4 warp arrivals)
  uint64_t *s_full = bars + 18;      // [2] scores in TMEM (commit)
  uint64_t *s_free = bars + 20;      // [2] scores read (4 warp arrivals)
  uint64_t *q_ready = bars + 22;     // [2] query operand written (4 warp arrivals)
  uint64_t *o_free = bars + 24;      // [2] output buffer read (4 warp arrivals)
  uint64_t *unit_full = bars + 26;   // [kTcRing] descriptor written (scheduler)
  uint64_t *unit_free = bars + 30;   // [kTcRing] descriptor read (7 consumer warps)
  uint64_t *clc_bar = bars + 34;     // [2] launch-queue responses (16 tx bytes)
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc + 288);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 292);
  // votes of the softmax warps: [2][4] per tile, per query, per unit end and
  // per next unit, [4] at the start
  int *flags = reinterpret_cast<int *>(misc + 304);  // 36 ints, to 448
  int *votes_tile = flags, *votes_query = flags + 8, *votes_end = flags + 16,
      *votes_next = flags + 24, *votes_start = flags + 32;
  float *red_t = reinterpret_cast<float *>(misc + 448);   // [4][8] tile maxima
  float *red_q = reinterpret_cast<float *>(misc + 576);   // [4][8] query maxima
  float *red_l = reinterpret_cast<float *>(misc + 704);   // [2][4][8] exp sums per unit parity
  float *red_m = reinterpret_cast<float *>(misc + 960);   // [2][4][8] max logits
  float *red_r = reinterpret_cast<float *>(misc + 1216);  // [2][8] running max at unit end
  uint4 *clc_resp = reinterpret_cast<uint4 *>(misc + 1280);  // [2]
  TcUnit *ring = reinterpret_cast<TcUnit *>(misc + 1312);    // [kTcRing] (176 B each)
  static_assert(1312 + kTcRing * sizeof(TcUnit) <= Cfg::kMiscBytes, "misc layout");

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      mbar_init(&k_raw[s], 1);
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&stage_free[s], 1);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      mbar_init(&p_full[j], 4);
      mbar_init(&s_full[j], 1);
      mbar_init(&s_free[j], 4);
      mbar_init(&q_ready[j], 4);
      mbar_init(&o_free[j], 4);
      mbar_init(&clc_bar[j], 1);
    }
#pragma unroll
    for (int r = 0; r < kTcRing; ++r) {
      mbar_init(&unit_full[r], 1);
      mbar_init(&unit_free[r], 7);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kTcWarpMma) tc::tmem_alloc(tmem_slot, Cfg::kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint64_t wait_ns = p.wait_limit_ns;
  const uint64_t drain_ns = min(wait_ns, uint64_t(100000000ull));
  bool failed = false;

  // A consumer warp's view of ring slot `u`: wait for it, copy the header
  // (and this lane's block id), free it (lane 0 arrives for the warp).
  auto take_unit = [&](int u, TcUnit &d, int &id0) -> bool {
    const int r = u % kTcRing;
    const bool ok =
        __all_sync(FULL, tc_wait(&unit_full[r], uint32_t(u / kTcRing) & 1u, wait_ns, abort_flag));
    if (ok) {
      const TcUnit &src = ring[r];
      d.end = src.end;
      d.seq = src.seq;
      d.part = src.part;
      d.kvh = src.kvh;
      d.hsub = src.hsub;
      d.L = src.L;
      d.t0 = src.t0;
      d.t1 = src.t1;
      d.row_base = src.row_base;
      id0 = src.ids[lane];
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&unit_free[r]);
    }
    return ok;
  };

  if (warp == kTcWarpSched) {
    // --------------------------------------------------------- scheduler --
    auto clc_request = [&](int slot) {
      if (lane == 0) {
        mbar_arrive_expect_tx(&clc_bar[slot], 16u);
        tc::clc_try_cancel(&clc_resp[slot], &clc_bar[slot]);
      }
    };
    int cx = blockIdx.x, cy = blockIdx.y, cz = blockIdx.z;
    clc_request(0);
    clc_request(1);
    int requested = 2, answered = 0;
    int U = 0;
    while (true) {
      // The candidate unit (cx, cy, cz).
      const int kvh = cy / p.head_groups;
      const int hsub = cy - kvh * p.head_groups;
      const int g = min(kMaxGroup, p.group - hsub * kMaxGroup);
      int L;
      int64_t t0, t1, row_base;
      tc_unit_range(p, cx, cz, lane == 0, L, t0, t1, row_base);
      if (t0 < t1) {
        // its first 32 block ids, loaded while the unit waits in the ring
        const int id = tc_block_id(p, row_base, t0 / kTcBS, (t1 - t0 + kTcBS - 1) / kTcBS, lane);
        if (U >= kTcRing &&
            !__all_sync(FULL, tc_wait(&unit_free[U % kTcRing], uint32_t(U / kTcRing - 1) & 1u,
                                      wait_ns, abort_flag))) {
          failed = true;
          break;
        }
        TcUnit &d = ring[U % kTcRing];
        d.ids[lane] = id;
        if (lane == 0) {
          d.end = 0;
          d.seq = cz;
          d.part = cx;
          d.kvh = kvh;
          d.hsub = hsub;
          d.L = L;
          d.t0 = t0;
          d.t1 = t1;
          d.row_base = row_base;
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&unit_full[U % kTcRing]);
        ++U;
      } else {
        // Empty unit: its outputs directly.
        const int h0 = kvh * p.group + hsub * kMaxGroup;
        if (p.mode == kModeV1) {
          T *out = static_cast<T *>(p.out);
          for (int i = lane; i < g * kTcD; i += 32) {
            const int h = i / kTcD, d = i % kTcD;
            out[int64_t(cz) * p.o_s0 + int64_t(h0 + h) * p.o_s1 + int64_t(d) * p.o_s2] =
                from_f32<T>(0.f);
          }
        } else if (lane < g) {
          const int64_t idx = (int64_t(cz) * p.num_heads + h0 + lane) * p.max_parts + cx;
          p.es[idx] = 0.f;
          p.ml[idx] = -INFINITY;
        }
      }
      // The next unit from the launch queue (the answer to the oldest request).
      const int slot = answered & 1;
      if (!__all_sync(FULL, tc_wait(&clc_bar[slot], uint32_t(answered >> 1) & 1u, wait_ns,
                                    abort_flag))) {
        failed = true;
        break;
      }
      uint32_t got = 0, nx = 0, ny = 0, nz = 0;
      if (lane == 0) tc::clc_read(&clc_resp[slot], got, nx, ny, nz);
      got = __shfl_sync(FULL, got, 0);
      nx = __shfl_sync(FULL, nx, 0);
      ny = __shfl_sync(FULL, ny, 0);
      nz = __shfl_sync(FULL, nz, 0);
      ++answered;
      // An empty queue ends the loop: no further request (the other one in
      // flight answers the same).
      if (!got) break;
      clc_request(slot);
      ++requested;
      cx = int(nx);
      cy = int(ny);
      cz = int(nz);
    }
    // End mark, then wait (bounded) for the requests still in flight.
    if (!failed && !*abort_flag) {
      if (U >= kTcRing &&
          !__all_sync(FULL, tc_wait(&unit_free[U % kTcRing], uint32_t(U / kTcRing - 1) & 1u,
                                    wait_ns, abort_flag))) {
        failed = true;
      } else if (lane == 0) {
        ring[U % kTcRing].end = 1;
        tc::mbar_arrive(&unit_full[U % kTcRing]);
      }
    }
    if (lane == 0)
      for (int i = answered; i < requested; ++i)
        mbar_wait_bounded(&clc_bar[i & 1], uint32_t(i >> 1) & 1u, drain_ns);
    __syncwarp();
  } else if (warp == kTcWarpCopy) {
    // ------------------------------------------------------------ copies --
    const uint64_t policy = l2_policy_evict_first();
    int64_t gt = 0;  // tiles issued by this CTA
    for (int U = 0;; ++U) {
      TcUnit d;
      int ids_cur;
      if (!take_unit(U, d, ids_cur)) {
        failed = true;
        break;
      }
      if (d.end) break;
      const int64_t page0 = d.t0 / kTcBS;
      const int64_t npages = (d.t1 - d.t0 + kTcBS - 1) / kTcBS;
      const int nb = int((d.t1 - d.t0 + kTcTokens - 1) / kTcTokens);
      const uint8_t *kbase = static_cast<const uint8_t *>(p.k) + int64_t(d.kvh) * p.k_s1;
      const uint8_t *vbase = static_cast<const uint8_t *>(p.v) + int64_t(d.kvh) * p.v_s1;
      int ids_nxt = npages > 32 ? tc_block_id(p, d.row_base, page0, npages, 32 + lane) : -1;
      int batch_cur = 0;
      for (int b = 0; b < nb; ++b, ++gt) {
        const int s = int(gt % NS);
        if (gt >= NS && !__all_sync(FULL, tc_wait(&stage_free[s], uint32_t(gt / NS - 1) & 1u,
                                                  wait_ns, abort_flag))) {
          failed = true;
          break;
        }
        const int bt = (b * kTcPages) >> 5;
        if (bt != batch_cur) {
          ids_cur = ids_nxt;
          batch_cur = bt;
          ids_nxt = npages > int64_t(bt + 1) * 32
                        ? tc_block_id(p, d.row_base, page0, npages, int64_t(bt + 1) * 32 + lane)
                        : -1;
        }
        const int base_lane = (b * kTcPages) & 31;
        int id[kTcPages];
#pragma unroll
        for (int i = 0; i < kTcPages; ++i) id[i] = __shfl_sync(FULL, ids_cur, base_lane + i);
        const int npv = int(min(int64_t(kTcPages), npages - int64_t(b) * kTcPages));
        if (lane == 0) {
          uint8_t *kst = smem + s * kTcStage;
          uint8_t *vst = kst + kTcHalf;
          mbar_arrive_expect_tx(&k_raw[s], uint32_t(npv * kTcPageBytes) + p.extra_expect_tx);
#pragma unroll
          for (int i = 0; i < kTcPages; ++i)
            if (i < npv)
              bulk_copy_g2s(kst + i * kTcPageBytes, kbase + int64_t(id[i]) * p.k_s0,
                            uint32_t(kTcPageBytes), &k_raw[s], policy);
          mbar_arrive_expect_tx(&v_full[s], uint32_t(npv * kTcPageBytes));
#pragma unroll
          for (int i = 0; i < kTcPages; ++i)
            if (i < npv)
              bulk_copy_g2s(vst + i * kTcPageBytes, vbase + int64_t(id[i]) * p.v_s0,
                            uint32_t(kTcPageBytes), &v_full[s], policy);
        }
        __syncwarp();
      }
      if (failed) break;
    }
    // No copy may still be in flight when the CTA exits: wait (bounded) for
    // the last stages issued (already complete unless a role gave up).
    if (lane == 0)
      for (int64_t t = gt > NS ? gt - NS : 0; t < gt; ++t) {
        const int s = int(t % NS);
        mbar_wait_bounded(&k_raw[s], uint32_t(t / NS) & 1u, drain_ns);
        mbar_wait_bounded(&v_full[s], uint32_t(t / NS) & 1u, drain_ns);
      }
    __syncwarp();
  } else if (warp == kTcWarpLayout) {
    // -------------------------------------------------------- key layout --
    int64_t gt = 0;
    for (int U = 0;; ++U) {
      TcUnit d;
      int unused;
      if (!take_unit(U, d, unused)) {
        failed = true;
        break;
      }
      if (d.end) break;
      const int nb = int((d.t1 - d.t0 + kTcTokens - 1) / kTcTokens);
      for (int b = 0; b < nb; ++b, ++gt) {
        const int s = int(gt % NS);
        if (!__all_sync(FULL, tc_wait(&k_raw[s], uint32_t(gt / NS) & 1u, wait_ns, abort_flag))) {
          failed = true;
          break;
        }
        // Swap blocks (page p, group q) <-> (page q, group p) for p < q: half
        // a warp per pair of 256-byte blocks, 16 bytes per lane.
        uint8_t *kst = smem + s * kTcStage + (lane & 15) * 16;
        int k = 0;
#pragma unroll
        for (int pp = 0; pp < kTcPages; ++pp) {
#pragma unroll
          for (int qq = pp + 1; qq < kTcPages; ++qq, ++k) {
            if ((k & 1) == (lane >> 4)) {
              uint4 *a = reinterpret_cast<uint4 *>(kst + pp * kTcPageBytes + qq * 256);
              uint4 *c = reinterpret_cast<uint4 *>(kst + qq * kTcPageBytes + pp * 256);
              const uint4 x = *a, y = *c;
              *a = y;
              *c = x;
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&k_full[s]);
      }
      if (failed) break;
    }
  } else if (warp == kTcWarpMma) {
    // ---------------------------------------------------------- MMA issue --
    if (lane == 0) {
      constexpr uint32_t idesc_k = tc::idesc_f8f6f4(kFmt, tc::kFmtE4M3, false, NK, 128);
      constexpr uint32_t idesc_v = tc::idesc_f8f6f4(kFmt, tc::kFmtE4M3, true, NV, 128);
      uint64_t *last_commit = nullptr;
      uint32_t last_parity = 0;
      bool ok = true;
      // The value product of a tile is issued after the key product of the
      // next one (or at the end), so the softmax of a tile overlaps the next
      // key product.
      int64_t pv_T = -1;  // tile whose value product is pending
      int pv_U = 0;
      bool pv_first = false;
      auto issue_pv = [&]() -> bool {
        const int s = int(pv_T % NS), j = int(pv_T & 1);
        if (!tc_wait(&p_full[j], uint32_t(pv_T >> 1) & 1u, wait_ns, abort_flag) ||
            !tc_wait(&v_full[s], uint32_t(pv_T / NS) & 1u, wait_ns, abort_flag))
          return false;
        if (pv_first && pv_U >= 2 &&
            !tc_wait(&o_free[pv_U & 1], uint32_t((pv_U >> 1) - 1) & 1u, wait_ns, abort_flag))
          return false;
        tc::fence_after_sync();
        const uint64_t vdesc =
            tc::smem_desc(smem_addr(smem + s * kTcStage + kTcHalf), 2048, 128);
        const uint64_t pdesc =
            tc::smem_desc(smem_addr(ps + j * Cfg::kPBytes), Cfg::kPKStride, 128);
        const uint32_t ocol = tmem + uint32_t(Cfg::kOCol + (pv_U & 1) * NV);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_f8f6f4(ocol, vdesc + uint64_t(kk * 4096 >> 4),
                         pdesc + uint64_t(kk * 4 * Cfg::kPKStride >> 4), idesc_v,
                         !(pv_first && kk == 0));
        tc::commit(&stage_free[s]);
        last_commit = &stage_free[s];
        last_parity = uint32_t(pv_T / NS) & 1u;
        return true;
      };
      int64_t gt = 0;
      for (int U = 0; ok; ++U) {
        const int r = U % kTcRing;
        if (!tc_wait(&unit_full[r], uint32_t(U / kTcRing) & 1u, wait_ns, abort_flag)) {
          ok = false;
          break;
        }
        const int end = ring[r].end;
        const int64_t ntok = ring[r].t1 - ring[r].t0;
        tc::mbar_arrive(&unit_free[r]);
        if (end) break;
        const int nb = int((ntok + kTcTokens - 1) / kTcTokens);
        if (!tc_wait(&q_ready[U & 1], uint32_t(U >> 1) & 1u, wait_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint64_t qdesc =
            tc::smem_desc(smem_addr(qs + (U & 1) * Cfg::kQBytes), Cfg::kQLbo, 128);
        for (int b = 0; b < nb; ++b, ++gt) {
          const int s = int(gt % NS), j = int(gt & 1);
          if (!tc_wait(&k_full[s], uint32_t(gt / NS) & 1u, wait_ns, abort_flag) ||
              (gt >= 2 &&
               !tc_wait(&s_free[j], uint32_t((gt >> 1) - 1) & 1u, wait_ns, abort_flag))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint64_t kdesc = tc::smem_desc(smem_addr(smem + s * kTcStage), 2048, 128);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_f8f6f4(tmem + uint32_t(j * NK), kdesc + uint64_t(kk * 4096 >> 4),
                           qdesc + uint64_t(kk * 2 * Cfg::kQLbo >> 4), idesc_k, kk > 0);
          tc::commit(&s_full[j]);
          last_commit = &s_full[j];
          last_parity = uint32_t(gt >> 1) & 1u;
          if (pv_T >= 0 && !issue_pv()) {
            ok = false;
            break;
          }
          pv_T = gt;
          pv_U = U;
          pv_first = b == 0;
        }
      }
      if (ok && pv_T >= 0 && !issue_pv()) ok = false;
      if (!ok) failed = true;
      // Every MMA issued must have finished before TMEM is freed (the last
      // commit covers all of them).
      if (last_commit != nullptr && !mbar_wait_bounded(last_commit, last_parity, drain_ns))
        failed = true;
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- softmax --
    const int tid = threadIdx.x;  // 0..127: the token of a tile, the dim of a query or output
    const uint32_t lane_base = uint32_t(32 * warp) << 16;
    // A collective decision of the four softmax warps: each votes `mine`
    // before a named barrier, all read the same four votes after it.
    auto vote_all = [&](int *slot4, int mine) -> int {
      if (lane == 0) slot4[warp] = mine;
      tc::named_bar_sync(1, 128);
      return slot4[0] | slot4[1] | slot4[2] | slot4[3];
    };
    // Dim `tid` of the query of every head of unit d (loaded a unit ahead).
    auto load_query = [&](const TcUnit &d, float (&qv)[GP]) {
      const int g = min(kMaxGroup, p.group - d.hsub * kMaxGroup);
      const int h0 = d.kvh * p.group + d.hsub * kMaxGroup;
      const T *qbase =
          static_cast<const T *>(p.q) + int64_t(d.seq) * p.q_s0 + int64_t(tid) * p.q_s2;
#pragma unroll
      for (int h = 0; h < GP; ++h)
        qv[h] = h < g ? to_f32<T>(qbase[int64_t(h0 + h) * p.q_s1]) : 0.f;
    };
    // Query operand of unit d into buffer qb; the logit factors (log2 units,
    // the query's power of two taken back out) and ALiBi slopes.
    auto prepare_query = [&](const TcUnit &d, int qb, const float (&qv)[GP], float (&xs)[GP],
                             float (&sl2)[GP]) -> bool {
      uint8_t *q = qs + qb * Cfg::kQBytes;
      const int g = min(kMaxGroup, p.group - d.hsub * kMaxGroup);
      const int h0 = d.kvh * p.group + d.hsub * kMaxGroup;
      for (int i = tid; i < Cfg::kQBytes / 16; i += 128)
        reinterpret_cast<uint4 *>(q)[i] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        float a = fabsf(qv[h]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(FULL, a, o));
        if (lane == 0) red_q[warp * 8 + h] = a;
        sl2[h] = (p.alibi != nullptr && h < g) ? p.alibi[h0 + h] * kLog2e : 0.f;
      }
      // (the zeroing above and the maxima are complete past this barrier)
      if (vote_all(votes_query + 4 * qb, (failed || *abort_flag) ? 1 : 0)) return false;
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        const float amax =
            fmaxf(fmaxf(red_q[h], red_q[8 + h]), fmaxf(red_q[16 + h], red_q[24 + h]));
        // Bring max |q| of the head into [2^7, 2^8): every term stays inside
        // the E4M3 range and the bf16 (f16) query is an exact sum of 2 (3)
        // terms.
        int k = 0;
        if (amax > 0.f && amax < INFINITY)
          k = clamp_int(134 - int(__float_as_uint(amax) >> 23), -120, 120);
        const float up = __uint_as_float(uint32_t(127 + k) << 23);
        xs[h] = p.scale_log2 * __uint_as_float(uint32_t(127 - k) << 23);
        float v = qv[h] * up;
#pragma unroll
        for (int t = 0; t < TQ; ++t) {
          const uint32_t c = tc::f32x2_to_e4m3x2(v, 0.f) & 0xFFu;
          const int n = t * GP + h;
          q[(tid / 16) * Cfg::kQLbo + (n / 8) * 128 + (n % 8) * 16 + (tid % 16)] = uint8_t(c);
          v = (v - tc::e4m3x2_to_f32x2(c).x) * 16.f;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&q_ready[qb]);
      return true;
    };
    // Output of unit d (parity u): wait for its last value product (tile
    // `last`), read the accumulator, normalise, write.  The exp sums, maxima
    // and running maxima were reduced into red_l / red_m / red_r at the unit's
    // end.  Returns false if the wait ran out.
    auto epilogue = [&](const TcOut &d, int u, int64_t last) -> bool {
      if (!__all_sync(FULL, tc_wait(&stage_free[last % NS], uint32_t(last / NS) & 1u, wait_ns,
                                    abort_flag)))
        return false;
      tc::fence_after_sync();
      float o[NV];
      const uint32_t ocol = tmem + lane_base + uint32_t(Cfg::kOCol + (u & 1) * NV);
#pragma unroll
      for (int c = 0; c < NV; c += 16) {
        float o16[16];
        tc::ld_x16(ocol + uint32_t(c), o16);
#pragma unroll
        for (int e = 0; e < 16; ++e) o[c + e] = o16[e];
      }
      tc::wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&o_free[u & 1]);
      const int g = min(kMaxGroup, p.group - d.hsub * kMaxGroup);
      const int h0 = d.kvh * p.group + d.hsub * kMaxGroup;
      const float *rl = red_l + (u & 1) * 32, *rm = red_m + (u & 1) * 32;
      const float *rr = red_r + (u & 1) * 8;
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        if (h < g) {
          const float Ls = rl[h] + rl[8 + h] + rl[16 + h] + rl[24 + h];
          const float M = fmaxf(fmaxf(rm[h], rm[8 + h]), fmaxf(rm[16 + h], rm[24 + h]));
          float acc = o[3 * GP + h] * 0.000244140625f;
          acc = fmaf(o[2 * GP + h], 0.00390625f, acc);
          acc = fmaf(o[GP + h], 0.0625f, acc);
          acc += o[h];
          const float r = __fdiv_rn(acc * p.out_scale, Ls);
          if (p.mode == kModeV1) {
            T *out = static_cast<T *>(p.out);
            out[int64_t(d.seq) * p.o_s0 + int64_t(h0 + h) * p.o_s1 + int64_t(tid) * p.o_s2] =
                from_f32<T>(r);
          } else {
            const int64_t rowi = (int64_t(d.seq) * p.num_heads + h0 + h) * p.max_parts + d.part;
            p.tmp[rowi * kTcD + tid] = r;
            if (tid == 0) {
              // exp sums relative to the true max; max logits in natural units
              p.es[rowi] = Ls * ex2(rr[h] - M);
              p.ml[rowi] = M * kLn2;
            }
          }
        }
      }
      return true;
    };

    TcUnit cur, nxt;
    TcOut prev;
    int unused;
    float xs[GP], sl2[GP], qn[GP];
    bool live = take_unit(0, cur, unused);
    if (!live) failed = true;
    // A failed take leaves `cur` unread: decide together.
    live = vote_all(votes_start, live ? 0 : 1) == 0 && !cur.end;
    if (live) {
      float q0[GP];
      load_query(cur, q0);
      if (!prepare_query(cur, 0, q0, xs, sl2)) {
        failed = true;
        live = false;
      }
    }
    int64_t gt = 0, prev_last = -1;
    int prev_u = 0;
    bool have_prev = false, more = false;
    for (int U = 0; live; ++U) {
      const int g = min(kMaxGroup, p.group - cur.hsub * kMaxGroup);
      const int ntok = int(cur.t1 - cur.t0);
      const int nb = (ntok + kTcTokens - 1) / kTcTokens;
      float mref[GP], tmax[GP], lsum[GP];
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        mref[h] = -INFINITY;
        tmax[h] = -INFINITY;
        lsum[h] = 0.f;
      }
      for (int b = 0; b < nb; ++b, ++gt) {
        const int s = int(gt % NS), j = int(gt & 1);
        const bool ok =
            __all_sync(FULL, tc_wait(&s_full[j], uint32_t(gt >> 1) & 1u, wait_ns, abort_flag));
        float sc[NK];
#pragma unroll
        for (int c = 0; c < NK; ++c) sc[c] = 0.f;
        if (ok) {
          tc::fence_after_sync();
#pragma unroll
          for (int c = 0; c < NK; c += 16) {
            float v16[16];
            tc::ld_x16(tmem + lane_base + uint32_t(j * NK + c), v16);
#pragma unroll
            for (int e = 0; e < 16; ++e) sc[c + e] = v16[e];
          }
          tc::wait_ld();
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&s_free[j]);
        }
        const int64_t tok = cur.t0 + int64_t(b) * kTcTokens + tid;
        const bool valid = tok < cur.t1;
        const float pos = float(tok - cur.L + 1);
        float x[GP];
        bool need = false;
#pragma unroll
        for (int h = 0; h < GP; ++h) {
          float sv = sc[h];
#pragma unroll
          for (int t = 1; t < TQ; ++t)
            sv = fmaf(sc[t * GP + h], t == 1 ? 0.0625f : 0.00390625f, sv);
          float v = sv * xs[h];
          if (p.alibi != nullptr) v = fmaf(sl2[h], pos, v);
          x[h] = (valid && h < g) ? v : -INFINITY;
          tmax[h] = fmaxf(tmax[h], x[h]);
          need |= x[h] > mref[h] + kTcRescale;
        }
        // Failures are collective: every warp sees them in this exchange and
        // all four leave together (none may be left waiting at a barrier).
        const int votes = vote_all(votes_tile + 4 * int(gt & 1),
                                   (__any_sync(FULL, need) ? 1 : 0) | ((ok && !failed) ? 0 : 2));
        if (votes & 2) {
          failed = true;
          break;
        }
        if (votes & 1) {
          // Move the running max of every head to the tile's max (if larger).
#pragma unroll
          for (int h = 0; h < GP; ++h) {
            float m = x[h];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
            if (lane == 0) red_t[warp * 8 + h] = m;
          }
          tc::named_bar_sync(1, 128);
          float mnew[GP];
          bool grow = false;
#pragma unroll
          for (int h = 0; h < GP; ++h) {
            const float bm =
                fmaxf(fmaxf(red_t[h], red_t[8 + h]), fmaxf(red_t[16 + h], red_t[24 + h]));
            mnew[h] = fmaxf(mref[h], bm);
            grow |= mnew[h] > mref[h] && mref[h] != -INFINITY;
          }
          tc::named_bar_sync(1, 128);  // red_t is free again
          if (grow && b > 0) {
            // The accumulator holds the unit's earlier tiles: wait for their
            // value product, then rescale its columns head by head.  A wait
            // that runs out skips the rescale; the next vote ends the loop.
            const int64_t pt = gt - 1;
            if (__all_sync(FULL, tc_wait(&stage_free[pt % NS], uint32_t(pt / NS) & 1u, wait_ns,
                                         abort_flag))) {
              tc::fence_after_sync();
              float alpha[GP];
#pragma unroll
              for (int h = 0; h < GP; ++h)
                alpha[h] = mref[h] == -INFINITY ? 0.f : ex2(mref[h] - mnew[h]);
              const uint32_t ocol = tmem + lane_base + uint32_t(Cfg::kOCol + (U & 1) * NV);
#pragma unroll
              for (int c = 0; c < NV; c += 16) {
                float o16[16];
                tc::ld_x16(ocol + uint32_t(c), o16);
                tc::wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) o16[e] *= alpha[(c + e) % GP];
                tc::st_x16(ocol + uint32_t(c), o16);
              }
              tc::wait_st();
              tc::fence_before_sync();
            } else {
              failed = true;
            }
          }
#pragma unroll
          for (int h = 0; h < GP; ++h) {
            const float a = mref[h] == -INFINITY ? 0.f : ex2(mref[h] - mnew[h]);
            lsum[h] *= a;
            mref[h] = mnew[h];
          }
        }
        // Probabilities (<= 2^8) as four E4M3 terms each: word t holds term t
        // of heads 0-3, word t + 4 (GP = 8) heads 4-7.
        uint32_t w[NV / 4];
#pragma unroll
        for (int hp = 0; hp < GP; hp += 2) {
          float a = ex2(x[hp] - mref[hp]);
          float c2 = ex2(x[hp + 1] - mref[hp + 1]);
          if (mref[hp] == -INFINITY) a = 0.f;
          if (mref[hp + 1] == -INFINITY) c2 = 0.f;
          lsum[hp] += a;
          lsum[hp + 1] += c2;
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint32_t code = tc::f32x2_to_e4m3x2(a, c2);
            const int wi = t * (GP / 4) + hp / 4;
            if ((hp & 2) == 0)
              w[wi] = code;
            else
              w[wi] |= code << 16;
            if (t < 3) {
              const float2 dd = tc::e4m3x2_to_f32x2(code);
              a = (a - dd.x) * 16.f;
              c2 = (c2 - dd.y) * 16.f;
            }
          }
        }
        // The probability buffer of this tile parity is free once the value
        // product of tile gt - 2 (the CTA's tile count) is done.
        bool okp = !failed;
        if (okp && gt >= 2)
          okp = __all_sync(FULL, tc_wait(&stage_free[(gt - 2) % NS], uint32_t((gt - 2) / NS) & 1u,
                                         wait_ns, abort_flag));
        if (okp) {
          uint8_t *row = ps + j * Cfg::kPBytes + (tid / 8) * Cfg::kPKStride + (tid % 8) * 16;
#pragma unroll
          for (int c = 0; c < NV / 16; ++c)
            *reinterpret_cast<uint4 *>(row + c * 128) =
                make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        }
        if (okp && b == nb - 1 && ntok - b * kTcTokens < kTcTokens) {
          // Last, partial tile: zero the value codes of the tokens past the
          // end (their probability is 0, but 0 * NaN must not reach the sum).
          okp = __all_sync(FULL, tc_wait(&v_full[s], uint32_t(gt / NS) & 1u, wait_ns, abort_flag));
          if (okp) {
            const int nv = ntok - b * kTcTokens;
            uint8_t *vst = smem + s * kTcStage + kTcHalf;
            for (int e = tid; e < (kTcTokens - nv) * kTcD; e += 128) {
              const int tau = nv + e / kTcD;
              const int dd = e % kTcD;
              vst[(tau / kTcBS) * kTcPageBytes + dd * kTcBS + (tau % kTcBS)] = 0;
            }
          }
        }
        if (!okp) failed = true;
        fence_proxy_async_smem();
        __syncwarp();
        if (okp && lane == 0) tc::mbar_arrive(&p_full[j]);
        if (b == 0) {
          // The previous unit's output, now that its last value product has
          // had this tile's time to finish.
          if (have_prev && !failed && !epilogue(prev, prev_u, prev_last)) failed = true;
          have_prev = false;
          // The next unit's descriptor and query, a unit ahead (decided
          // together: a warp may have failed alone).
          const bool have = !failed && take_unit(U + 1, nxt, unused);
          const int vn = vote_all(votes_next + 4 * (U & 1), !have ? 1 : (nxt.end ? 2 : 0));
          if (vn & 1) {
            failed = true;
            break;
          }
          more = (vn & 2) == 0;
          if (more) load_query(nxt, qn);
        }
      }
      // This unit's exp sums, maxima and running maxima, for its epilogue.
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        float l = lsum[h], m = tmax[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          l += __shfl_xor_sync(FULL, l, o);
          m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
        }
        if (lane == 0) {
          red_l[(U & 1) * 32 + warp * 8 + h] = l;
          red_m[(U & 1) * 32 + warp * 8 + h] = m;
        }
        if (tid == 0) red_r[(U & 1) * 8 + h] = mref[h];
      }
      if (vote_all(votes_end + 4 * (U & 1), (failed || *abort_flag) ? 1 : 0)) {
        failed = true;
        break;
      }
      prev = TcOut{cur.seq, cur.part, cur.kvh, cur.hsub};
      prev_u = U;
      prev_last = gt - 1;
      have_prev = true;
      if (!more) break;
      // Query operand of the next unit (lets the MMA issue go on), then on.
      if (!prepare_query(nxt, (U + 1) & 1, qn, xs, sl2)) {
        failed = true;
        break;
      }
      cur = nxt;
    }
    // The last unit's output.
    if (have_prev && !failed && !epilogue(prev, prev_u, prev_last)) failed = true;
  }

  // ------------------------------------------------------------ teardown --
  if (failed && lane == 0) flag_error(p.err, 16u);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kTcWarpMma) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

}  // namespace pkv
