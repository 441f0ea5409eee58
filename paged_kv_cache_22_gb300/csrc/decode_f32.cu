// fp32-cache decode kernel instances (fp32 q and out), CUDA cores.
#include "decode_launch.cuh"

namespace pkv {
bool find_decode_f32(int head_dim, int block_size, int heads, bool balanced, DecodeKernel* out) {
  if (block_size != 16) return false;
  if (head_dim == 64) return find_for<CacheF32, 64, 16, false>(heads, balanced, out);
  if (head_dim == 128) return find_for<CacheF32, 128, 16, false>(heads, balanced, out);
  return false;
}
}  // namespace pkv
