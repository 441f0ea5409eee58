// fp8-e4m3-cache shared-prefix kernel instances of cascade decode.
#include "decode_launch.cuh"

namespace pkv {
bool find_prefix_fp8(int head_dim, int block_size, PrefixKernel* out) {
  if (block_size != 16) return false;
  if (head_dim == 128) { *out = prefix_kernel_info<CacheFP8, 128, 16, false>(); return true; }
  if (head_dim == 64) { *out = prefix_kernel_info<CacheFP8, 64, 16, false>(); return true; }
  return false;
}
}  // namespace pkv
