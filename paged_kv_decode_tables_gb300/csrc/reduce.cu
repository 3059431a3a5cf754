// Split-KV log-sum-exp reduce (page "paged_attention_v2_triton.py",
// _paged_attn_v2_reduce_kernel): global max of the partitions' max logits,
// weights w_p = exp(m_p - M) * s_p, output = sum_p w_p tmp_p / sum_p w_p.
//
// One CTA per (query head, sequence); no host sync, no inter-CTA waiting.
// Pass 1 finds M with warp shuffles; pass 2 stores the weights in shared
// memory and sums them; pass 3 streams the fp32 partial outputs with float4
// loads, the CTA's warps splitting the partitions, and combines the warps'
// sums in shared memory.
#include "reduce.cuh"

namespace pkv {

namespace {

constexpr int kReduceThreads = 256;
constexpr float kLog2e = 1.44269504088896340736f;

__device__ __forceinline__ float block_reduce_max(float v, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = -INFINITY;
  for (int w = 0; w < kReduceThreads / 32; ++w) r = fmaxf(r, red[w]);
  return r;
}

__device__ __forceinline__ float block_reduce_sum(float v, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = 0.f;
  for (int w = 0; w < kReduceThreads / 32; ++w) r += red[w];
  return r;
}

template <typename TO, int D>
__global__ void __launch_bounds__(kReduceThreads) reduce_kernel(const ReduceParams p) {
  constexpr int D4 = D / 4;                     // float4 columns per row
  constexpr int ROWS = kReduceThreads / D4;     // partitions read in parallel
  static_assert(kReduceThreads % D4 == 0, "bad D");
  extern __shared__ float sh[];
  float *w = sh;                                // [max_parts]
  float *red = sh + p.max_parts;                // [8]
  float4 *part_acc = reinterpret_cast<float4 *>(sh + p.smem_head_floats);  // [ROWS][D4]

  const int h = blockIdx.x;
  const int s = blockIdx.y;
  const int tid = threadIdx.x;

  int L = p.seq_lens[s];
  if (L < 0) {
    if (tid == 0) flag_error(p.err, 2u);
    L = 0;
  }
  int num_parts;
  if (p.splits == nullptr) {
    num_parts = int((int64_t(L) + p.partition_size - 1) / p.partition_size);
  } else {
    int n = p.splits[s];
    if (L > 0 && (n < 1 || n > p.max_parts)) {
      if (tid == 0) flag_error(p.err, 4u);
      n = n < 1 ? 1 : p.max_parts;
    }
    if (L > 0) {
      int64_t c = (int64_t(L) + n - 1) / n;
      c = (c + p.block_size - 1) / p.block_size * p.block_size;
      num_parts = int((L + c - 1) / c);
    } else {
      num_parts = 0;
    }
  }
  if (num_parts > p.max_parts) {
    if (tid == 0) flag_error(p.err, 2u);
    num_parts = p.max_parts;
  }
  TO *out = static_cast<TO *>(p.out) + int64_t(s) * p.o_s0 + int64_t(h) * p.o_s1;
  if (num_parts == 0) {
    for (int d = tid; d < D; d += kReduceThreads) out[int64_t(d) * p.o_s2] = from_f32<TO>(0.f);
    return;
  }

  const int64_t row = (int64_t(s) * p.num_heads + h) * p.max_parts;
  const float *ml = p.ml + row;
  const float *es = p.es + row;

  float m = -INFINITY;
  for (int i = tid; i < num_parts; i += kReduceThreads) m = fmaxf(m, ml[i]);
  const float M = block_reduce_max(m, red);

  float sum = 0.f;
  for (int i = tid; i < num_parts; i += kReduceThreads) {
    const float wi = ex2((ml[i] - M) * kLog2e) * es[i];
    w[i] = wi;
    sum += wi;
  }
  const float S = block_reduce_sum(sum, red);  // also orders the w[] stores
  const float inv = __fdiv_rn(1.f, S);

  const int r = tid / D4, c4 = tid % D4;
  const float4 *tmp = reinterpret_cast<const float4 *>(p.tmp + row * D);
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = r; i < num_parts; i += ROWS) {
    const float4 t = __ldg(tmp + int64_t(i) * D4 + c4);
    const float wi = w[i];
    a.x = fmaf(wi, t.x, a.x);
    a.y = fmaf(wi, t.y, a.y);
    a.z = fmaf(wi, t.z, a.z);
    a.w = fmaf(wi, t.w, a.w);
  }
  part_acc[r * D4 + c4] = a;
  __syncthreads();
  if (r == 0) {
    float4 t = part_acc[c4];
    for (int rr = 1; rr < ROWS; ++rr) {
      const float4 u = part_acc[rr * D4 + c4];
      t.x += u.x;
      t.y += u.y;
      t.z += u.z;
      t.w += u.w;
    }
    const int d = 4 * c4;
    out[int64_t(d + 0) * p.o_s2] = from_f32<TO>(t.x * inv);
    out[int64_t(d + 1) * p.o_s2] = from_f32<TO>(t.y * inv);
    out[int64_t(d + 2) * p.o_s2] = from_f32<TO>(t.z * inv);
    out[int64_t(d + 3) * p.o_s2] = from_f32<TO>(t.w * inv);
  }
}

template <typename TO, int D>
pkv_status_t launch_d(const ReduceParams &p, cudaStream_t stream) {
  constexpr int D4 = D / 4;
  constexpr int ROWS = kReduceThreads / D4;
  // w[max_parts] + red[8], rounded to 16 B, then ROWS*D4 float4
  size_t head = (size_t(p.max_parts) + 8) * sizeof(float);
  head = (head + 15) / 16 * 16;
  const size_t smem = head + size_t(ROWS) * D4 * sizeof(float4);
  ReduceParams q = p;
  q.smem_head_floats = int(head / sizeof(float));
  dim3 grid(p.num_heads, p.num_seqs);
  reduce_kernel<TO, D><<<grid, kReduceThreads, smem, stream>>>(q);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
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
