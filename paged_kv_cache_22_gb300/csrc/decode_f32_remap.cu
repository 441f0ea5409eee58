// fp32-cache decode kernel instances (fp32 q and out), CUDA cores;
// the instances that may skip blocks (sliding window, cascade prefix).
#include "decode_launch.cuh"

namespace pkv {
bool find_decode_f32_remap(int head_dim, int block_size, int heads, bool balanced, DecodeKernel* out) {
  return find_shape<CacheF32, false, true>(head_dim, block_size, heads, balanced, out);
}
}  // namespace pkv
