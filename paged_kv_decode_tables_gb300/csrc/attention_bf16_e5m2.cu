// Paged decode attention instances for bf16 queries over an E5M2 cache.
#include "attention_launch.cuh"

namespace pkv {

PKV_DEFINE_ATTENTION(bf16_e5m2, __nv_bfloat16, fp8_e5m2_t)

}  // namespace pkv
