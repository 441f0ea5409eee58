// kernels.cu -- the cache write, the block-table gather and the split-KV
// reduce.  All three are short, bandwidth-bound element loops.
#include <math_constants.h>

#include "kernels.h"
#include "pkv_device.cuh"

namespace pkv {

constexpr int kReduceThreads = 256;  // split-KV reduce: threads per (sequence, query head)

// ----------------------------------------------------------------------------
// reshape_and_cache: "PagedAttention por dentro" (section "La tabla de páginas
// (block table)") -- the new token of a sequence goes to the free position of
// its last block.  One thread writes 8 consecutive elements of one (token,
// kv head) row of K or V into slot_mapping[token].
// ----------------------------------------------------------------------------
__device__ __forceinline__ void load8(const float* s, float (&x)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(s);
  const float4 b = *reinterpret_cast<const float4*>(s + 4);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* s, float (&x)[8]) {
  const uint4 v = *reinterpret_cast<const uint4*>(s);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = bf16x2_to_f2(w[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

template <class Src>
__device__ __forceinline__ void store8(const Src* s, uint8_t* d, pkv_dtype dt, float kv_scale) {
  if (dt == PKV_BF16 && sizeof(Src) == 2) {  // bit copy
    *reinterpret_cast<uint4*>(d) = *reinterpret_cast<const uint4*>(s);
    return;
  }
  float x[8];
  load8(s, x);
  if (dt == PKV_F32) {
    *reinterpret_cast<float4*>(d) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4*>(d + 16) = make_float4(x[4], x[5], x[6], x[7]);
  } else if (dt == PKV_BF16) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(d) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {  // fp8 e4m3: x / kv_scale in binary32, round to nearest even, saturate
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = make_float2(__fdiv_rn(x[2 * i], kv_scale), __fdiv_rn(x[2 * i + 1], kv_scale));
      const uint32_t two = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      w[i / 2] |= (two & 0xFFFFu) << (16 * (i % 2));
    }
    *reinterpret_cast<uint2*>(d) = make_uint2(w[0], w[1]);
  }
}

template <class Src>
__global__ void reshape_and_cache_kernel(ReshapeArgs a) {
  // A decode launched as this grid's programmatic dependent may start its
  // prologue now; it waits for this grid's writes before reading any K/V.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int chunks = a.head_dim / 8;
  const int64_t per_token = (int64_t)a.num_kv_heads * chunks * 2;
  const int64_t total = (int64_t)a.num_tokens * per_token;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / per_token);
    int rem = (int)(i % per_token);
    const int kv = rem / (a.num_kv_heads * chunks);
    rem %= a.num_kv_heads * chunks;
    const int h = rem / chunks, ch = rem % chunks;
    const int64_t slot = a.slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= (int64_t)a.num_blocks * a.block_size) {
      raise_error(a.err, PKV_DEVERR_BAD_SLOT);
      continue;
    }
    const int64_t blk = slot / a.block_size, off = slot % a.block_size;
    const Src* src = reinterpret_cast<const Src*>(kv ? a.v : a.k) +
                     ((int64_t)t * a.num_kv_heads + h) * a.head_dim + ch * 8;
    const int64_t elem = ((blk * a.num_kv_heads + h) * a.block_size + off) * a.head_dim + ch * 8;
    uint8_t* dst = reinterpret_cast<uint8_t*>(kv ? a.v_cache : a.k_cache) + elem * a.cache_bytes;
    store8<Src>(src, dst, a.cache_dtype, a.kv_scale);
  }
}

cudaError_t launch_reshape_and_cache(const ReshapeArgs& a, int src_is_bf16, cudaStream_t stream) {
  const int64_t total = (int64_t)a.num_tokens * a.num_kv_heads * (a.head_dim / 8) * 2;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks64 = (total + threads - 1) / threads;
  const int blocks = (int)(blocks64 < 65535 * 8 ? blocks64 : 65535 * 8);
  if (src_is_bf16)
    reshape_and_cache_kernel<__nv_bfloat16><<<blocks, threads, 0, stream>>>(a);
  else
    reshape_and_cache_kernel<float><<<blocks, threads, 0, stream>>>(a);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------
// gather: "La despensa por casilleros" (section "El mecanismo: bloques, block
// table y el gather del kernel") -- walk a sequence's physical blocks in
// logical order and read them as if contiguous.  One thread moves 16 bytes.
// ----------------------------------------------------------------------------
__global__ void gather_kv_kernel(GatherArgs a) {
  const int s = blockIdx.y;
  const int L = a.seq_lens[s];
  const int row16 = a.head_dim * a.cache_bytes / 16;  // 16-byte units per (token, head)
  const int64_t per_token = (int64_t)a.num_kv_heads * row16;
  const int64_t total = (int64_t)(L < 0 ? 0 : L) * per_token;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int p = (int)(i / per_token);
    const int rem = (int)(i % per_token);
    const int h = rem / row16, u = rem % row16;
    const int j = p / a.block_size, off = p % a.block_size;
    if (j >= a.max_blocks_per_seq) {
      raise_error(a.err, PKV_DEVERR_BAD_SEQ_LEN);
      continue;
    }
    const int32_t blk = a.block_tables[(int64_t)s * a.max_blocks_per_seq + j];
    if (blk < 0 || blk >= a.num_blocks) {
      raise_error(a.err, PKV_DEVERR_BAD_BLOCK_ID);
      continue;
    }
    const int64_t src = (((int64_t)blk * a.num_kv_heads + h) * a.block_size + off) * row16 + u;
    const int64_t dst = ((a.cu_seq_lens[s] + p) * a.num_kv_heads + h) * row16 + u;
    reinterpret_cast<uint4*>(a.k_out)[dst] = reinterpret_cast<const uint4*>(a.k_cache)[src];
    reinterpret_cast<uint4*>(a.v_out)[dst] = reinterpret_cast<const uint4*>(a.v_cache)[src];
  }
}

cudaError_t launch_gather_kv(const GatherArgs& a, int max_seq_len, cudaStream_t stream) {
  if (a.num_seqs == 0 || max_seq_len <= 0) return cudaSuccess;
  const int threads = 256;
  const int64_t per_seq = (int64_t)max_seq_len * a.num_kv_heads * (a.head_dim * a.cache_bytes / 16);
  int64_t bx = (per_seq + threads - 1) / threads;
  if (bx > 4096) bx = 4096;
  dim3 grid((unsigned)bx, (unsigned)a.num_seqs);
  gather_kv_kernel<<<grid, threads, 0, stream>>>(a);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------
// split-KV reduce: log-sum-exp merge of per-partition partials.  One CTA per
// (sequence, query head) of 256 threads: 256 / head_dim groups of one
// thread per head dimension, each group summing every groups-th partition
// with four independent chains (a row has up to hundreds of partitions, and
// a single chain per thread left the reduce bound by load latency).
// ----------------------------------------------------------------------------
template <class OT>
__global__ void __launch_bounds__(kReduceThreads) split_kv_reduce_kernel(ReduceArgs a) {
  const int row = blockIdx.x;  // s * Hq + qh
  const int s = row / a.num_q_heads;
  const int tid = threadIdx.x, D = a.head_dim;
  const int groups = kReduceThreads / D, grp = tid / D, d = tid % D;
  const int L = a.seq_lens[s];
  int np = L <= 0 ? 0 : (L + a.partition_tokens - 1) / a.partition_tokens;
  if (a.window > 0 && L > a.window) {
    // partitions of the blocks read: the sink blocks, then the window's
    const int bs = a.block_size, ws = L - a.window, sk = a.sinks < ws ? a.sinks : ws;
    const int nsb = (sk + bs - 1) / bs, wsb = ws / bs;
    const int nb = (L + bs - 1) / bs - (wsb > nsb ? wsb - nsb : 0);
    const int pb = a.partition_tokens / bs;
    np = (nb + pb - 1) / pb;
  }
  OT* out = reinterpret_cast<OT*>(a.out) + (int64_t)row * D;
  if (np > a.max_partitions && tid == 0) raise_error(a.err, PKV_DEVERR_BAD_SEQ_LEN);
  const int n = np < a.max_partitions ? np : a.max_partitions;
  const float* m = a.m_part + (int64_t)row * a.max_partitions;
  const float* l = a.l_part + (int64_t)row * a.max_partitions;
  const float* o = a.o_part + (int64_t)row * a.max_partitions * D;
  __shared__ float red[kReduceThreads / 32];
  __shared__ float part[kReduceThreads];  // [group][dim] numerators, then [group] denominators
  // the largest partition maximum, over all threads
  float M = -CUDART_INF_F;
  for (int p = tid; p < n; p += kReduceThreads) M = fmaxf(M, m[p]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if ((tid & 31) == 0) red[tid >> 5] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int i = 1; i < kReduceThreads / 32; ++i) M = fmaxf(M, red[i]);
  // group grp sums the partitions p = grp (mod groups), four independent
  // chains so that several partitions' loads are in flight at once
  float num[4] = {0.f, 0.f, 0.f, 0.f}, den[4] = {0.f, 0.f, 0.f, 0.f};
  int p = grp;
  for (; p + 3 * groups < n; p += 4 * groups) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int q = p + k * groups;
      const float wgt = l[q] * expf(m[q] - M);
      den[k] += wgt;
      num[k] += wgt * o[(int64_t)q * D + d];
    }
  }
  for (; p < n; p += groups) {
    const float wgt = l[p] * expf(m[p] - M);
    den[0] += wgt;
    num[0] += wgt * o[(int64_t)p * D + d];
  }
  __syncthreads();  // red[] is read by every thread above
  part[tid] = (num[0] + num[1]) + (num[2] + num[3]);
  if (d == 0) red[grp] = (den[0] + den[1]) + (den[2] + den[3]);
  __syncthreads();
  if (grp == 0) {
    float nu = 0.f, de = 0.f;
    for (int g2 = 0; g2 < groups; ++g2) {
      nu += part[g2 * D + d];
      de += red[g2];
    }
    out[d] = from_f32<OT>(de > 0.f ? nu / de : 0.f);
  }
}

cudaError_t launch_split_kv_reduce(const ReduceArgs& a, int out_is_bf16, cudaStream_t stream) {
  if (a.num_seqs == 0) return cudaSuccess;
  const unsigned rows = (unsigned)a.num_seqs * a.num_q_heads;
  if (out_is_bf16)
    split_kv_reduce_kernel<__nv_bfloat16><<<rows, kReduceThreads, 0, stream>>>(a);
  else
    split_kv_reduce_kernel<float><<<rows, kReduceThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------
// Self-test of the failure path every pipelined kernel shares: one thread
// arms an mbarrier for 16 bytes of transactions that no copy will ever
// deliver (none is issued, so nothing is in flight), then waits on it with
// the same bounded wait the attention kernels use.  The wait gives up after
// its probe limit, raises PKV_DEVERR_WAIT_TIMEOUT and the kernel returns.
// ----------------------------------------------------------------------------
__global__ void wait_timeout_selftest_kernel(unsigned int* err) {
  __shared__ __align__(8) uint64_t bar;
  mbar_init(&bar, 1);
  fence_mbar_init();
  mbar_arrive_expect_tx(&bar, 16);
  mbar_wait_bounded(&bar, 0, err);
}

cudaError_t launch_wait_timeout_selftest(unsigned int* err, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 1, 0, stream>>>(err);
  return cudaGetLastError();
}

}  // namespace pkv
