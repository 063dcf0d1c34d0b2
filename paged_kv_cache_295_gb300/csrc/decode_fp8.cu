// Decode instantiations for FP8 E4M3 KV caches (head_dim 64, 128 and 256).
#include "decode_launch.cuh"

namespace pkv {
PKV_INSTANTIATE_DECODE(FP8, 64)
PKV_INSTANTIATE_DECODE(FP8, 128)
PKV_INSTANTIATE_DECODE(FP8, 256)
}  // namespace pkv
