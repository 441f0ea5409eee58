// bf16-cache decode kernel instances (bf16 q and out), CUDA cores; block sizes 8,
// 16, 32;
// the instances that may skip blocks (sliding window, cascade prefix).
#include "decode_launch.cuh"

namespace pkv {
bool find_decode_bf16_cc_remap(int head_dim, int block_size, int heads, bool balanced, DecodeKernel* out) {
  return find_shape<CacheBF16, false, true>(head_dim, block_size, heads, balanced, out);
}
}  // namespace pkv
