// bf16-cache shared-prefix kernel instances of cascade decode.
#include "decode_launch.cuh"

namespace pkv {
bool find_prefix_bf16(int head_dim, int block_size, PrefixKernel* out) {
  if (head_dim == 128) {
    if (block_size == 16) { *out = prefix_kernel_info<CacheBF16, 128, 16, false>(); return true; }
    if (block_size == 8) { *out = prefix_kernel_info<CacheBF16, 128, 8, false>(); return true; }
    if (block_size == 32) { *out = prefix_kernel_info<CacheBF16, 128, 32, false>(); return true; }
  }
  if (head_dim == 64 && block_size == 16) { *out = prefix_kernel_info<CacheBF16, 64, 16, false>(); return true; }
  return false;
}
}  // namespace pkv
