// tcgen05 kernel instances for fp8-e4m3 caches (several query tokens per sequence; cascade prefix pass).
#include "decode_launch.cuh"

namespace pkv {
namespace {
template <int BS>
bool pick(bool prefix, Tc05Kernel* out) {
  *out = prefix ? tc05_kernel_info<128, BS, true, true>() : tc05_kernel_info<128, BS, true, false>();
  return true;
}
}  // namespace

bool find_tc05_fp8(int head_dim, int block_size, bool prefix, Tc05Kernel* out) {
  if (head_dim != 128) return false;
  if (block_size == 16) return pick<16>(prefix, out);
  if (block_size == 8) return pick<8>(prefix, out);
  if (block_size == 32) return pick<32>(prefix, out);
  return false;
}
}  // namespace pkv
