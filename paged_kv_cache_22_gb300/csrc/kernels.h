// kernels.h -- argument blocks and launchers of the non-attention kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pkv.h"

namespace pkv {

struct ReshapeArgs {
  unsigned int* err;
  const void* k;
  const void* v;
  int num_tokens, num_kv_heads, head_dim;
  void* k_cache;
  void* v_cache;
  int num_blocks, block_size;
  pkv_dtype cache_dtype;
  int cache_bytes;
  const int64_t* slot_mapping;
  float kv_scale;
};

struct GatherArgs {
  unsigned int* err;
  void* k_out;
  void* v_out;
  const void* k_cache;
  const void* v_cache;
  int num_blocks, block_size, num_kv_heads, head_dim, cache_bytes;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* seq_lens;
  const int64_t* cu_seq_lens;
  int num_seqs;
};

struct ReduceArgs {
  unsigned int* err;
  void* out;
  const float* o_part;
  const float* m_part;
  const float* l_part;
  const int32_t* seq_lens;
  int num_seqs, num_q_heads, head_dim, partition_tokens, max_partitions;
  // sliding window (window > 0): partitions cover the blocks the decode read
  int block_size, window, sinks;
};

struct CopyBlocksArgs {
  unsigned int* err;
  void* k_dst;
  void* v_dst;
  const void* k_src;
  const void* v_src;
  int64_t src_blocks, dst_blocks;
  int64_t block_bytes;   // Hkv * bs * d * e: one block of one cache, a multiple of 16
  const int64_t* pairs;  // [num_pairs][2] = (source block, destination block)
  int64_t num_pairs;
};

cudaError_t launch_copy_blocks(const CopyBlocksArgs& a, cudaStream_t stream);
cudaError_t launch_reshape_and_cache(const ReshapeArgs& a, int src_is_bf16, cudaStream_t stream);
cudaError_t launch_gather_kv(const GatherArgs& a, int max_seq_len, cudaStream_t stream);
cudaError_t launch_split_kv_reduce(const ReduceArgs& a, int out_is_bf16, cudaStream_t stream);
cudaError_t launch_wait_timeout_selftest(unsigned int* err, cudaStream_t stream);

}  // namespace pkv
