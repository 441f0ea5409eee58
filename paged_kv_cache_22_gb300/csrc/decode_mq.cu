// Multi-query decode kernel instances (several query tokens per sequence), tensor cores.
#include "decode_launch.cuh"

namespace pkv {
bool find_decode_mq(pkv_dtype dt, int head_dim, int block_size, DecodeKernel* out) {
  if (dt == PKV_BF16) {
    if (head_dim == 128) {
      if (block_size == 16) { *out = decode_mq_kernel_info<CacheBF16, 128, 16>(); return true; }
      if (block_size == 8) { *out = decode_mq_kernel_info<CacheBF16, 128, 8>(); return true; }
      if (block_size == 32) { *out = decode_mq_kernel_info<CacheBF16, 128, 32>(); return true; }
    }
    if (head_dim == 64 && block_size == 16) { *out = decode_mq_kernel_info<CacheBF16, 64, 16>(); return true; }
    return false;
  }
  if (dt == PKV_FP8_E4M3 && block_size == 16) {
    if (head_dim == 128) { *out = decode_mq_kernel_info<CacheFP8, 128, 16>(); return true; }
    if (head_dim == 64) { *out = decode_mq_kernel_info<CacheFP8, 64, 16>(); return true; }
  }
  return false;
}
}  // namespace pkv
