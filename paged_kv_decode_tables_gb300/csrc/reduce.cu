// Split-KV log-sum-exp reduce (page "paged_attention_v2_triton.py",
// _paged_attn_v2_reduce_kernel): global max of the partitions' max logits,
// weights w_p = exp(m_p - M) * s_p, output = sum_p w_p tmp_p / sum_p w_p.
//
// Lane l of a warp owns head dims [l*D/32, (l+1)*D/32) of the output.  The
// maximum goes round by shuffles; partitions are then taken 32 at a time:
// each lane computes one partition's weight, the weights are broadcast by
// shuffle and every lane accumulates its slice of the fp32 partial rows (one
// coalesced row read per partition).  Up to 32 partitions: each warp takes
// two (sequence, head) pairs, no shared memory.  More: one CTA per
// (sequence, head) whose eight warps take the groups of 32 in turn and add up
// in shared memory.  No host sync and no inter-CTA waiting either way.
#include "pkv_launch.cuh"
#include "reduce.cuh"

namespace pkv {

namespace {

constexpr int kReduceWarps = 8;
constexpr float kLog2e = 1.44269504088896340736f;
constexpr unsigned kFull = 0xffffffffu;

template <int V>
struct Row;  // V consecutive floats of a partial row
template <>
struct Row<2> {
  static __device__ __forceinline__ void load(const float *p, float (&v)[2]) {
    const float2 t = __ldg(reinterpret_cast<const float2 *>(p));
    v[0] = t.x;
    v[1] = t.y;
  }
};
template <>
struct Row<4> {
  static __device__ __forceinline__ void load(const float *p, float (&v)[4]) {
    const float4 t = __ldg(reinterpret_cast<const float4 *>(p));
    v[0] = t.x;
    v[1] = t.y;
    v[2] = t.z;
    v[3] = t.w;
  }
};
template <>
struct Row<8> {
  static __device__ __forceinline__ void load(const float *p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x;
    v[1] = a.y;
    v[2] = a.z;
    v[3] = a.w;
    v[4] = b.x;
    v[5] = b.y;
    v[6] = b.z;
    v[7] = b.w;
  }
};

// Non-empty partitions of a sequence of length L (split count n, when the
// split mode is on), computed exactly as the partition pass splits it: fixed
// size, or roundup(cdiv(L, n), block_size) tokens.
__device__ __forceinline__ int count_parts(const ReduceParams &p, int L, int n, bool report) {
  if (L < 0) {
    if (report) flag_error(p.err, 2u);
    L = 0;
  }
  int num_parts;
  if (L == 0) {
    num_parts = 0;
  } else if (p.splits == nullptr) {
    num_parts = int((unsigned(L) - 1u) / unsigned(p.partition_size)) + 1;
  } else {
    if (n < 1 || n > p.max_parts) {
      if (report) flag_error(p.err, 4u);
      n = n < 1 ? 1 : p.max_parts;
    }
    // chunk = roundup(cdiv(L, n), block_size); 32-bit is exact since L < 2^31
    const unsigned bs = unsigned(p.block_size);
    const unsigned c = ((unsigned(L) - 1u) / unsigned(n) + bs) / bs * bs;
    num_parts = int((unsigned(L) - 1u) / c) + 1;
  }
  if (num_parts > p.max_parts) {
    if (report) flag_error(p.err, 2u);
    num_parts = p.max_parts;
  }
  return num_parts;
}

// Accumulate partitions [c_begin, c_end) in steps of 32 (c_stride apart):
// each lane weighs one partition of the group, the weights go round by
// shuffle, every lane adds its V dims of each partial row.
template <int D>
__device__ __forceinline__ void accumulate_parts(const float *ml, const float *es,
                                                 const float *tmp_lane, int num_parts, float M,
                                                 int c_begin, int c_step, float (&acc)[D / 32],
                                                 float &S) {
  constexpr int V = D / 32;
  const int lane = threadIdx.x & 31;
  for (int c0 = c_begin; c0 < num_parts; c0 += c_step) {
    const int i = c0 + lane;
    float w = 0.f;
    if (i < num_parts) w = ex2((__ldg(ml + i) - M) * kLog2e) * __ldg(es + i);
    S += w;
    const int n = min(32, num_parts - c0);
    const float *t = tmp_lane + int64_t(c0) * D;
#pragma unroll 4
    for (int j = 0; j < n; ++j) {
      const float wj = __shfl_sync(kFull, w, j);
      float v[V];
      Row<V>::load(t + int64_t(j) * D, v);
#pragma unroll
      for (int k = 0; k < V; ++k) acc[k] = fmaf(wj, v[k], acc[k]);
    }
  }
}

// Two (sequence, head) units per warp: for up to a few dozen partitions.
// Every load that does not depend on another (length, split count and the
// first partial row, which is the whole answer for a one-partition sequence)
// is issued before any result is used.
constexpr int kUnitsPerWarp = 2;
constexpr int kPrefetch = 8;  // partial rows fetched together with the statistics

template <typename TO, int D>
__global__ void __launch_bounds__(kReduceWarps * 32) reduce_kernel(const ReduceParams p) {
  constexpr int V = D / 32;
  constexpr int U = kUnitsPerWarp;
  const int lane = threadIdx.x & 31;
  // (sequence, head) units number below 2^31 (checked at launch): 32-bit math.
  grid_dependency_wait();
  allow_dependent_launch();
  const unsigned total = unsigned(p.num_seqs) * unsigned(p.num_heads);
  const unsigned H = unsigned(p.num_heads);
  const unsigned first = (blockIdx.x * kReduceWarps + (threadIdx.x >> 5)) * U;
  int Ls[U], ns[U];
  float row0[U][V];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const unsigned unit = min(first + u, total - 1);
    const int s = int(unit / H);
    Ls[u] = __ldg(p.seq_lens + s);
    ns[u] = p.splits != nullptr ? __ldg(p.splits + s) : 0;
    Row<V>::load(p.tmp + int64_t(unit) * p.max_parts * D + lane * V, row0[u]);
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const unsigned unit = first + u;
    if (unit >= total) break;
    const int s = int(unit / H);
    const int h = int(unit - unsigned(s) * H);
    const int num_parts = count_parts(p, Ls[u], ns[u], lane == 0);
    TO *out = static_cast<TO *>(p.out) + int64_t(s) * p.o_s0 + int64_t(h) * p.o_s1;
    if (num_parts <= 1) {
      // One partition is already normalised: the output is its row.
#pragma unroll
      for (int k = 0; k < V; ++k)
        out[int64_t(lane * V + k) * p.o_s2] = from_f32<TO>(num_parts == 1 ? row0[u][k] : 0.f);
      continue;
    }
    // At most 32 partitions here: lane i holds partition i's statistics, and
    // the first kPrefetch partial rows are fetched in the same round.
    const int64_t row = int64_t(unit) * p.max_parts;  // == (s * num_heads + h) * max_parts
    const bool mine = lane < num_parts;
    const float mlv = mine ? __ldg(p.ml + row + lane) : -INFINITY;
    const float esv = mine ? __ldg(p.es + row + lane) : 0.f;
    const float *tmp = p.tmp + row * D + lane * V;
    float rows[kPrefetch][V];
#pragma unroll
    for (int j = 1; j < kPrefetch; ++j) {
      if (j < num_parts) Row<V>::load(tmp + int64_t(j) * D, rows[j]);
    }
    float M = mlv;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    const float w = mine ? ex2((mlv - M) * kLog2e) * esv : 0.f;
    float S = w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(kFull, S, o);
    float acc[V];
    {
      const float w0 = __shfl_sync(kFull, w, 0);
#pragma unroll
      for (int k = 0; k < V; ++k) acc[k] = w0 * row0[u][k];
    }
#pragma unroll
    for (int j = 1; j < kPrefetch; ++j) {
      const float wj = __shfl_sync(kFull, w, j);
      if (j < num_parts) {
#pragma unroll
        for (int k = 0; k < V; ++k) acc[k] = fmaf(wj, rows[j][k], acc[k]);
      }
    }
    for (int j = kPrefetch; j < num_parts; ++j) {
      const float wj = __shfl_sync(kFull, w, j);
      float v[V];
      Row<V>::load(tmp + int64_t(j) * D, v);
#pragma unroll
      for (int k = 0; k < V; ++k) acc[k] = fmaf(wj, v[k], acc[k]);
    }
    const float inv = __fdiv_rn(1.f, S);
#pragma unroll
    for (int k = 0; k < V; ++k) out[int64_t(lane * V + k) * p.o_s2] = from_f32<TO>(acc[k] * inv);
  }
}

// One CTA per (sequence, head), the eight warps taking groups of 32
// partitions in turn: for long sequences cut into many partitions.
template <typename TO, int D>
__global__ void __launch_bounds__(kReduceWarps * 32) reduce_wide_kernel(const ReduceParams p) {
  constexpr int V = D / 32;
  __shared__ float red[kReduceWarps];
  __shared__ float part_S[kReduceWarps];
  __shared__ __align__(16) float part_acc[kReduceWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dependency_wait();
  allow_dependent_launch();
  const int64_t unit = blockIdx.x;
  const int s = int(unit / p.num_heads);
  const int h = int(unit % p.num_heads);
  const int num_parts = count_parts(p, p.seq_lens[s], p.splits != nullptr ? p.splits[s] : 0,
                                    threadIdx.x == 0);
  TO *out = static_cast<TO *>(p.out) + int64_t(s) * p.o_s0 + int64_t(h) * p.o_s1;
  if (num_parts == 0) {
    for (int d = threadIdx.x; d < D; d += kReduceWarps * 32) out[int64_t(d) * p.o_s2] = from_f32<TO>(0.f);
    return;
  }
  const int64_t row = unit * p.max_parts;
  const float *ml = p.ml + row;
  const float *es = p.es + row;
  float M = -INFINITY;
  for (int i = threadIdx.x; i < num_parts; i += kReduceWarps * 32) M = fmaxf(M, __ldg(ml + i));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  if (lane == 0) red[warp] = M;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kReduceWarps; ++w) M = fmaxf(M, red[w]);
  float S = 0.f;
  float acc[V];
#pragma unroll
  for (int k = 0; k < V; ++k) acc[k] = 0.f;
  accumulate_parts<D>(ml, es, p.tmp + row * D + lane * V, num_parts, M, 32 * warp,
                      32 * kReduceWarps, acc, S);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(kFull, S, o);
#pragma unroll
  for (int k = 0; k < V; ++k) part_acc[warp][lane * V + k] = acc[k];
  if (lane == 0) part_S[warp] = S;
  __syncthreads();
  float St = 0.f;
#pragma unroll
  for (int w = 0; w < kReduceWarps; ++w) St += part_S[w];
  const float inv = __fdiv_rn(1.f, St);
  for (int d = threadIdx.x; d < D; d += kReduceWarps * 32) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kReduceWarps; ++w) t += part_acc[w][d];
    out[int64_t(d) * p.o_s2] = from_f32<TO>(t * inv);
  }
}

template <typename TO, int D>
pkv_status_t launch_d(const ReduceParams &p, cudaStream_t stream) {
  const int64_t units = int64_t(p.num_seqs) * p.num_heads;
  if (units >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
  if (p.max_parts > 32) {
    if (units > 0x7fffffff) return PKV_ERR_UNSUPPORTED;
    if (launch_programmatic(reduce_wide_kernel<TO, D>, dim3(unsigned(units)),
                            dim3(kReduceWarps * 32), 0, stream, p) != cudaSuccess)
      return PKV_ERR_CUDA;
  } else {
    const int64_t per_block = int64_t(kReduceWarps) * kUnitsPerWarp;
    const int64_t blocks = (units + per_block - 1) / per_block;
    if (blocks > 0x7fffffff) return PKV_ERR_UNSUPPORTED;
    if (launch_programmatic(reduce_kernel<TO, D>, dim3(unsigned(blocks)), dim3(kReduceWarps * 32),
                            0, stream, p) != cudaSuccess)
      return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

template <typename TO>
pkv_status_t launch_t(const ReduceParams &p, cudaStream_t stream) {
  switch (p.head_size) {
    case 64: return launch_d<TO, 64>(p, stream);
    case 128: return launch_d<TO, 128>(p, stream);
    case 256: return launch_d<TO, 256>(p, stream);
    default: return PKV_ERR_UNSUPPORTED;
  }
}

}  // namespace

pkv_status_t launch_reduce(const ReduceParams &p, pkv_dtype_t out_dtype, cudaStream_t stream) {
  switch (out_dtype) {
    case PKV_F32: return launch_t<float>(p, stream);
    case PKV_F16: return launch_t<__half>(p, stream);
    case PKV_BF16: return launch_t<__nv_bfloat16>(p, stream);
    default: return PKV_ERR_UNSUPPORTED;
  }
}

}  // namespace pkv
