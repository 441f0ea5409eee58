// fp8-e4m3-cache decode kernel instances (bf16 q and out), tensor cores;
// the instances that may skip blocks (sliding window, cascade prefix).
#include "decode_launch.cuh"

namespace pkv {
bool find_decode_fp8_tc_remap(int head_dim, int block_size, int heads, bool balanced, DecodeKernel* out) {
  return find_shape<CacheFP8, true, true>(head_dim, block_size, heads, balanced, out);
}
}  // namespace pkv
