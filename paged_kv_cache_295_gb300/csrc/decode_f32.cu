// Decode instantiations for float32 KV caches (head_dim 64 and 128).
#include "decode_launch.cuh"

namespace pkv {
PKV_INSTANTIATE_DECODE(F32, 64)
PKV_INSTANTIATE_DECODE(F32, 128)
}  // namespace pkv
