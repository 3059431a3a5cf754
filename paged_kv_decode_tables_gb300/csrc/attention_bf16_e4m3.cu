// Paged decode attention instances for bf16 queries over an E4M3 cache.
#include "attention_launch.cuh"

namespace pkv {

PKV_DEFINE_ATTENTION(bf16_e4m3, __nv_bfloat16, fp8_e4m3_t)

}  // namespace pkv
