// Decode instantiations for bfloat16 KV caches (head_dim 64, 128 and 256).
#include "decode_launch.cuh"

namespace pkv {
PKV_INSTANTIATE_DECODE(BF16, 64)
PKV_INSTANTIATE_DECODE(BF16, 128)
PKV_INSTANTIATE_DECODE(BF16, 256)
}  // namespace pkv
