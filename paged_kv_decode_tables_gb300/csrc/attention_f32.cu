// Paged decode attention instances for element type float.
#include "attention_launch.cuh"

namespace pkv {

PKV_DEFINE_ATTENTION(f32, float, float)

}  // namespace pkv
