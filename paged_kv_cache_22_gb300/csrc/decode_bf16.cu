// bf16-cache decode kernel instances (bf16 q and out), tensor cores; block sizes 8,
// 16, 32.
#include "decode_launch.cuh"

namespace pkv {
bool find_decode_bf16_tc(int head_dim, int block_size, int heads, bool balanced, DecodeKernel* out) {
  if (head_dim == 128) {
    if (block_size == 16) return find_for<CacheBF16, 128, 16, true>(heads, balanced, out);
    if (block_size == 8) return find_for<CacheBF16, 128, 8, true>(heads, balanced, out);
    if (block_size == 32) return find_for<CacheBF16, 128, 32, true>(heads, balanced, out);
  }
  if (head_dim == 64 && block_size == 16) return find_for<CacheBF16, 64, 16, true>(heads, balanced, out);
  return false;
}
}  // namespace pkv
