// Paged decode attention instances for element type __half.
#include "attention_launch.cuh"

namespace pkv {

PKV_DEFINE_ATTENTION(f16, __half, __half)

}  // namespace pkv
