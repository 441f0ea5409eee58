// fp8-e4m3-cache kernel instances of paged attention for several query tokens per sequence.
#include "decode_launch.cuh"

namespace pkv {
namespace {
template <int D>
bool pick(bool one_warp, PrefixKernel* out) {
  *out = one_warp ? prefix_kernel_info<CacheFP8, D, 16, true, 1>() : prefix_kernel_info<CacheFP8, D, 16, true, 4>();
  return true;
}
}  // namespace

bool find_multi_fp8(int head_dim, int block_size, bool one_warp, PrefixKernel* out) {
  if (block_size != 16) return false;
  if (head_dim == 128) return pick<128>(one_warp, out);
  if (head_dim == 64) return pick<64>(one_warp, out);
  return false;
}
}  // namespace pkv
