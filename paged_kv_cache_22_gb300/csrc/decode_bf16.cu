// bf16-cache decode kernel instances (bf16 q and out), tensor cores; block sizes 8,
// 16, 32.
#include "decode_launch.cuh"

namespace pkv {
bool find_decode_bf16_tc(int head_dim, int block_size, int heads, bool balanced, DecodeKernel* out) {
  return find_shape<CacheBF16, true, false>(head_dim, block_size, heads, balanced, out);
}
}  // namespace pkv
