// Paged decode attention instances for element type __nv_bfloat16.
#include "attention_launch.cuh"

namespace pkv {

PKV_DEFINE_ATTENTION(bf16, __nv_bfloat16, __nv_bfloat16)

}  // namespace pkv
