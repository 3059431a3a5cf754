// Paged decode attention instances for f16 queries over an E5M2 cache.
#include "attention_launch.cuh"

namespace pkv {

PKV_DEFINE_ATTENTION(f16_e5m2, __half, fp8_e5m2_t)

}  // namespace pkv
