// Decode instantiations for INT8 KV caches (head_dim 64, 128 and 256).
#include "decode_launch.cuh"

namespace pkv {
PKV_INSTANTIATE_DECODE(INT8, 64)
PKV_INSTANTIATE_DECODE(INT8, 128)
PKV_INSTANTIATE_DECODE(INT8, 256)
}  // namespace pkv
