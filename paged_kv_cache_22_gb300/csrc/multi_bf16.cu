// bf16-cache kernel instances of paged attention for several query tokens per sequence.
#include "decode_launch.cuh"

namespace pkv {
namespace {
template <int D, int BS>
bool pick(bool one_warp, PrefixKernel* out) {
  *out = one_warp ? prefix_kernel_info<CacheBF16, D, BS, true, 1>() : prefix_kernel_info<CacheBF16, D, BS, true, 4>();
  return true;
}
}  // namespace

bool find_multi_bf16(int head_dim, int block_size, bool one_warp, PrefixKernel* out) {
  if (head_dim == 128) {
    if (block_size == 16) return pick<128, 16>(one_warp, out);
    if (block_size == 8) return pick<128, 8>(one_warp, out);
    if (block_size == 32) return pick<128, 32>(one_warp, out);
  }
  if (head_dim == 64 && block_size == 16) return pick<64, 16>(one_warp, out);
  return false;
}
}  // namespace pkv
