// decode_launch.cuh -- registry of the compiled decode kernel instances.
#pragma once

#include "decode.cuh"
#include "decode_tc.cuh"
#include "decode_prefix.cuh"
#include "attn_tc05.cuh"

namespace pkv {

constexpr int kDecodeWarps = 1;  // warps per CTA: each warp is an independent worker

struct DecodeKernel {
  const void* fn = nullptr;  // __global__ entry, parameters (DecodeArgs, TmaMaps)
  int threads = 0;
  size_t smem = 0;           // dynamic shared memory bytes
  int heads_per_unit = 0;    // G
  bool tensor_maps = false;  // reads the caches through the TmaMaps parameter
  // the deferred-merge grid that follows it (merge_cut_kernel: parameters
  // (DecodeArgs, int64_t warps of the decode grid), one CTA of merge_threads
  // threads per decode warp), if any
  const void* merge_fn = nullptr;
  size_t merge_smem = 0;
  int merge_threads = 0;
};

// TC: the q.K and P.V contractions on the tensor cores (decode_tc.cuh, bf16
// and fp8 caches); otherwise on the CUDA cores (decode.cuh, every cache type).
// REMAP: the instance that may skip blocks (a sliding window, a cascade's
// prefix); plain decode runs the instance without that code.
template <class CT, int D, int BS, int G, bool BAL, bool TC, bool REMAP>
DecodeKernel decode_kernel_info() {
  DecodeKernel k;
  if constexpr (TC) {
    static_assert(CT::kBytes != 4, "fp32 caches run on the CUDA cores");
    k.fn = reinterpret_cast<const void*>(&decode_tc_kernel<CT, D, BS, G, kDecodeWarps, BAL, REMAP>);
    k.smem = TcSmem<CT, D, BS, G, kDecodeWarps, REMAP>::kBytes;
    k.tensor_maps = true;
    if constexpr (BAL) {
      // pieces staged per round of a merge (per warp): 16 for one-warp merges
      // (long segments, ~66 pieces on 32k-token sequences, need fewer round
      // trips: +0.6 to +1.8 % on long_split_kv and its window; 32 slots cost
      // the Llama-3-8B decode 5 %: fewer merge CTAs resident), 8 otherwise
      constexpr int kMergeSlots = MergeGeo<G, D, 1>::kWarps > 1 ? 8 : 16;
      k.merge_fn = reinterpret_cast<const void*>(&merge_cut_kernel<__nv_bfloat16, G, D, BS, kMergeSlots>);
      k.merge_smem = MergeGeo<G, D, kMergeSlots>::kSmem;
      k.merge_threads = 32 * MergeGeo<G, D, kMergeSlots>::kWarps;
    }
  } else {
    k.fn = reinterpret_cast<const void*>(&decode_kernel<CT, D, BS, G, kDecodeWarps, BAL, REMAP>);
    k.smem = Smem<CT, D, BS, G, kDecodeWarps>::kBytes;
  }
  k.threads = kDecodeWarps * 32;
  k.heads_per_unit = G;
  return k;
}

// The multi-query instance (several query tokens per sequence; balanced,
// no remap, 16 rows per unit) on the tensor cores.
constexpr int kMqRows = 16;
template <class CT, int D, int BS>
DecodeKernel decode_mq_kernel_info() {
  DecodeKernel k;
  k.fn = reinterpret_cast<const void*>(&decode_tc_kernel<CT, D, BS, kMqRows, kDecodeWarps, true, false, true>);
  k.smem = TcSmem<CT, D, BS, kMqRows, kDecodeWarps, false>::kBytes;
  k.tensor_maps = true;
  k.threads = kDecodeWarps * 32;
  k.heads_per_unit = kMqRows;
  constexpr int kMergeSlots = 4;  // pieces staged per round of a merge (per warp)
  k.merge_fn = reinterpret_cast<const void*>(&merge_cut_kernel<__nv_bfloat16, kMqRows, D, BS, kMergeSlots>);
  k.merge_smem = MergeGeo<kMqRows, D, kMergeSlots>::kSmem;
  k.merge_threads = 32 * MergeGeo<kMqRows, D, kMergeSlots>::kWarps;
  return k;
}
// bf16 caches: head_dim 128 with blocks of 8, 16, 32, head_dim 64 with 16;
// fp8 caches: head_dim 64 or 128 with blocks of 16.
bool find_decode_mq(pkv_dtype dt, int head_dim, int block_size, DecodeKernel* out);

// Fill the tensor maps a kernel reads the caches through (pkv_api.cu); true
// when the kernel needs none or both were encoded.
bool encode_cache_maps(const DecodeKernel& k, const pkv_cache_desc* cache, const void* k_cache,
                       const void* v_cache, TmaMaps* maps);

// Fill `out` with the instance for (D, BS, G, balanced); false if not built.
// One finder per cache type, engine and REMAP, each in its own translation
// unit (they compile in parallel).
#define PKV_DECLARE_FINDER(NAME) \
  bool NAME(int head_dim, int block_size, int heads, bool balanced, DecodeKernel* out);

PKV_DECLARE_FINDER(find_decode_f32)
PKV_DECLARE_FINDER(find_decode_bf16_tc)
PKV_DECLARE_FINDER(find_decode_bf16_cc)
PKV_DECLARE_FINDER(find_decode_fp8_tc)
PKV_DECLARE_FINDER(find_decode_fp8_cc)
PKV_DECLARE_FINDER(find_decode_f32_remap)
PKV_DECLARE_FINDER(find_decode_bf16_tc_remap)
PKV_DECLARE_FINDER(find_decode_bf16_cc_remap)
PKV_DECLARE_FINDER(find_decode_fp8_tc_remap)
PKV_DECLARE_FINDER(find_decode_fp8_cc_remap)

// Shared body of the finders: the heads-per-unit switch for one (D, BS).
template <class CT, int D, int BS, bool TC, bool REMAP>
bool find_for(int heads, bool balanced, DecodeKernel* out) {
  switch (heads) {
    case 1: *out = balanced ? decode_kernel_info<CT, D, BS, 1, true, TC, REMAP>() : decode_kernel_info<CT, D, BS, 1, false, TC, REMAP>(); return true;
    case 2: *out = balanced ? decode_kernel_info<CT, D, BS, 2, true, TC, REMAP>() : decode_kernel_info<CT, D, BS, 2, false, TC, REMAP>(); return true;
    case 4: *out = balanced ? decode_kernel_info<CT, D, BS, 4, true, TC, REMAP>() : decode_kernel_info<CT, D, BS, 4, false, TC, REMAP>(); return true;
    case 8: *out = balanced ? decode_kernel_info<CT, D, BS, 8, true, TC, REMAP>() : decode_kernel_info<CT, D, BS, 8, false, TC, REMAP>(); return true;
    default: return false;
  }
}

// The compiled (D, BS) sets: fp32 and fp8 caches block size 16, head dim 64
// or 128; bf16 caches also block sizes 8 and 32 at head dim 128.
template <class CT, bool TC, bool REMAP>
bool find_shape(int head_dim, int block_size, int heads, bool balanced, DecodeKernel* out) {
  if constexpr (CT::kBytes == 2) {
    if (head_dim == 128) {
      if (block_size == 16) return find_for<CT, 128, 16, TC, REMAP>(heads, balanced, out);
      if (block_size == 8) return find_for<CT, 128, 8, TC, REMAP>(heads, balanced, out);
      if (block_size == 32) return find_for<CT, 128, 32, TC, REMAP>(heads, balanced, out);
    }
    if (head_dim == 64 && block_size == 16) return find_for<CT, 64, 16, TC, REMAP>(heads, balanced, out);
    return false;
  } else {
    if (block_size != 16) return false;
    if (head_dim == 64) return find_for<CT, 64, 16, TC, REMAP>(heads, balanced, out);
    if (head_dim == 128) return find_for<CT, 128, 16, TC, REMAP>(heads, balanced, out);
    return false;
  }
}

// The decode kernel for a cache type, shape, engine and REMAP (fp32 caches
// always take the CUDA cores).
inline bool find_decode(pkv_dtype dt, int D, int BS, int G, bool balanced, bool tensor_cores, bool remap,
                        DecodeKernel* k) {
  switch (dt) {
    case PKV_F32: return remap ? find_decode_f32_remap(D, BS, G, balanced, k) : find_decode_f32(D, BS, G, balanced, k);
    case PKV_BF16:
      if (tensor_cores)
        return remap ? find_decode_bf16_tc_remap(D, BS, G, balanced, k) : find_decode_bf16_tc(D, BS, G, balanced, k);
      return remap ? find_decode_bf16_cc_remap(D, BS, G, balanced, k) : find_decode_bf16_cc(D, BS, G, balanced, k);
    case PKV_FP8_E4M3:
      if (tensor_cores)
        return remap ? find_decode_fp8_tc_remap(D, BS, G, balanced, k) : find_decode_fp8_tc(D, BS, G, balanced, k);
      return remap ? find_decode_fp8_cc_remap(D, BS, G, balanced, k) : find_decode_fp8_cc(D, BS, G, balanced, k);
  }
  return false;
}

// The shared-prefix kernel of cascade decode (bf16 and fp8 caches).
struct PrefixKernel {
  const void* fn = nullptr;  // __global__ entry, parameters (PrefixArgs, TmaMaps)
  size_t smem = 0;
  int warps = kPrefixWarps;  // warps per CTA
};

// MULTI: the same kernel for several query tokens per sequence
// (pkv_paged_attention_multi).
template <class CT, int D, int BS, bool MULTI, int PW = kPrefixWarps>
PrefixKernel prefix_kernel_info() {
  PrefixKernel k;
  k.fn = reinterpret_cast<const void*>(&prefix_attention_kernel<CT, D, BS, MULTI, PW>);
  k.smem = PrefixSmem<CT, D, BS>::kBytes;
  k.warps = PW;
  return k;
}

bool find_prefix_bf16(int head_dim, int block_size, PrefixKernel* out);
bool find_prefix_fp8(int head_dim, int block_size, PrefixKernel* out);
// one_warp: the one-warp-per-CTA instance (at most 16 rows per sequence and kv head)
bool find_multi_bf16(int head_dim, int block_size, bool one_warp, PrefixKernel* out);
bool find_multi_fp8(int head_dim, int block_size, bool one_warp, PrefixKernel* out);

// The tcgen05 kernels (attn_tc05.cuh): 128 query rows per CTA, parameters
// (Tc05Args, TmaMaps). bf16 caches: the maps view each cache as (D, Hkv * BS,
// num_blocks) with a box of one 128-byte span (64, BS, 1); fp8 caches
// (head_dim 128): the decode kernels' map, a box of whole rows (128, BS, 1).
struct Tc05Kernel {
  const void* fn = nullptr;
  size_t smem = 0;
  int threads = 0;
};
template <int D, int BS, bool F8, bool PREFIX>
Tc05Kernel tc05_kernel_info() {
  Tc05Kernel k;
  k.fn = reinterpret_cast<const void*>(&attn_tc05_kernel<D, BS, F8, PREFIX>);
  k.smem = tc05::Layout<D, F8>::kBytes;
  k.threads = tc05::threads(F8);
  return k;
}
// prefix: the cascade's shared-prefix pass; otherwise several query tokens per sequence
bool find_tc05_bf16(int head_dim, int block_size, bool prefix, Tc05Kernel* out);
bool find_tc05_fp8(int head_dim, int block_size, bool prefix, Tc05Kernel* out);

// The engine set by pkv_set_decode_engine (pkv_api.cu).
bool decode_on_tensor_cores();

}  // namespace pkv
