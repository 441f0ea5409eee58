// copy_blocks.cu -- whole-block copies between block pools: the copy of a
// shared block for the branch that is about to write it (copy-on-write,
// "PagedAttention por dentro", section "Copy-on-write para sampling
// paralelo"; "La despensa por casilleros", section "Prefix caching: compartir
// casilleros con copy-on-write"), and the move of a preempted sequence's
// blocks to host memory and back ("PagedAttention por dentro", section
// "Evicción y preemption: qué hace cuando el pool se agota", the swap
// strategy).
//
// A block of one cache is Hkv * BS * D contiguous elements in the
// [num_blocks, Hkv, BS, D] layout, so a pair is two contiguous runs (K and V)
// of block_bytes each.  Each CTA moves one 16 KiB chunk of one run: 256
// threads, 4 independent 16-byte loads in flight per thread, then 4 stores.
// Both ends are streamed past L2 (evict-first); either end may be pinned
// host memory that the device addresses directly.
#include "kernels.h"
#include "pkv_device.cuh"

namespace pkv {

namespace {
constexpr int kThreads = 256;
constexpr int kVecPerThread = 4;
constexpr int64_t kChunk = (int64_t)kThreads * kVecPerThread * 16;  // bytes per CTA
}  // namespace

__global__ void __launch_bounds__(kThreads) copy_blocks_kernel(const CopyBlocksArgs a) {
  const int64_t chunks = (a.block_bytes + kChunk - 1) / kChunk;
  const int64_t job = blockIdx.x / chunks;  // (pair, cache)
  const int64_t chunk = blockIdx.x % chunks;
  const int64_t pair = job >> 1;
  const bool is_v = job & 1;
  if (pair >= a.num_pairs) return;
  const int64_t src = a.pairs[2 * pair], dst = a.pairs[2 * pair + 1];
  if (src < 0 || src >= a.src_blocks || dst < 0 || dst >= a.dst_blocks) {
    if (threadIdx.x == 0 && chunk == 0 && !is_v) raise_error(a.err, PKV_DEVERR_BAD_BLOCK_ID);
    return;
  }
  const uint4* from = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(is_v ? a.v_src : a.k_src) +
                                                     src * a.block_bytes + chunk * kChunk);
  uint4* to = reinterpret_cast<uint4*>(static_cast<uint8_t*>(is_v ? a.v_dst : a.k_dst) + dst * a.block_bytes +
                                       chunk * kChunk);
  const int64_t left = a.block_bytes - chunk * kChunk;  // bytes of this run from the chunk start
  const int nvec = (int)((left < kChunk ? left : kChunk) / 16);
  uint4 v[kVecPerThread];
#pragma unroll
  for (int i = 0; i < kVecPerThread; ++i) {
    const int e = threadIdx.x + i * kThreads;
    if (e < nvec) v[i] = __ldcs(from + e);
  }
#pragma unroll
  for (int i = 0; i < kVecPerThread; ++i) {
    const int e = threadIdx.x + i * kThreads;
    if (e < nvec) __stcs(to + e, v[i]);
  }
}

cudaError_t launch_copy_blocks(const CopyBlocksArgs& a, cudaStream_t stream) {
  if (a.num_pairs <= 0) return cudaSuccess;
  const int64_t chunks = (a.block_bytes + kChunk - 1) / kChunk;
  const int64_t ctas = a.num_pairs * 2 * chunks;
  if (ctas > 0x7FFFFFFF) return cudaErrorInvalidValue;
  copy_blocks_kernel<<<(unsigned)ctas, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pkv
