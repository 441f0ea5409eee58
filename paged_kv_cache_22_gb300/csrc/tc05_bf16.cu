// tcgen05 kernel instances for bf16 caches (several query tokens per sequence; cascade prefix pass).
#include "decode_launch.cuh"

namespace pkv {
namespace {
template <int D, int BS>
bool pick(bool prefix, Tc05Kernel* out) {
  *out = prefix ? tc05_kernel_info<D, BS, false, true>() : tc05_kernel_info<D, BS, false, false>();
  return true;
}
}  // namespace

bool find_tc05_bf16(int head_dim, int block_size, bool prefix, Tc05Kernel* out) {
  if (head_dim == 128) {
    if (block_size == 16) return pick<128, 16>(prefix, out);
    if (block_size == 8) return pick<128, 8>(prefix, out);
    if (block_size == 32) return pick<128, 32>(prefix, out);
  }
  if (head_dim == 64 && block_size == 16) return pick<64, 16>(prefix, out);
  return false;
}
}  // namespace pkv
