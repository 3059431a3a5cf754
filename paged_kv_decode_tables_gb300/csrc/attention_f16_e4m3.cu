// Paged decode attention instances for f16 queries over an E4M3 cache.
#include "attention_launch.cuh"

namespace pkv {

PKV_DEFINE_ATTENTION(f16_e4m3, __half, fp8_e4m3_t)

}  // namespace pkv
