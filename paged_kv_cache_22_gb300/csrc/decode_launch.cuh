// decode_launch.cuh -- registry of the compiled decode kernel instances.
#pragma once

#include "decode.cuh"
#include "decode_tc.cuh"
#include "decode_prefix.cuh"

namespace pkv {

constexpr int kDecodeWarps = 1;  // warps per CTA: each warp is an independent worker

struct DecodeKernel {
  const void* fn = nullptr;  // __global__ entry, parameters (DecodeArgs, TmaMaps)
  int threads = 0;
  size_t smem = 0;           // dynamic shared memory bytes
  int heads_per_unit = 0;    // G
  bool tensor_maps = false;  // reads the caches through the TmaMaps parameter
};

// TC: the q.K and P.V contractions on the tensor cores (decode_tc.cuh, bf16
// and fp8 caches); otherwise on the CUDA cores (decode.cuh, every cache type).
template <class CT, int D, int BS, int G, bool BAL, bool TC>
DecodeKernel decode_kernel_info() {
  DecodeKernel k;
  if constexpr (TC) {
    static_assert(CT::kBytes != 4, "fp32 caches run on the CUDA cores");
    k.fn = reinterpret_cast<const void*>(&decode_tc_kernel<CT, D, BS, G, kDecodeWarps, BAL>);
    k.smem = TcSmem<CT, D, BS, G, kDecodeWarps>::kBytes;
    k.tensor_maps = true;
  } else {
    k.fn = reinterpret_cast<const void*>(&decode_kernel<CT, D, BS, G, kDecodeWarps, BAL>);
    k.smem = Smem<CT, D, BS, G, kDecodeWarps>::kBytes;
  }
  k.threads = kDecodeWarps * 32;
  k.heads_per_unit = G;
  return k;
}

// Fill the tensor maps a kernel reads the caches through (pkv_api.cu); true
// when the kernel needs none or both were encoded.
bool encode_cache_maps(const DecodeKernel& k, const pkv_cache_desc* cache, const void* k_cache,
                       const void* v_cache, TmaMaps* maps);

// Fill `out` with the instance for (D, BS, G, balanced); false if not built.
// One finder per cache type and engine, each in its own translation unit.
#define PKV_DECLARE_FINDER(NAME) \
  bool NAME(int head_dim, int block_size, int heads, bool balanced, DecodeKernel* out);

PKV_DECLARE_FINDER(find_decode_f32)
PKV_DECLARE_FINDER(find_decode_bf16_tc)
PKV_DECLARE_FINDER(find_decode_bf16_cc)
PKV_DECLARE_FINDER(find_decode_fp8_tc)
PKV_DECLARE_FINDER(find_decode_fp8_cc)

// Shared body of the finders: the compiled (D, BS) set is passed as a list.
template <class CT, int D, int BS, bool TC>
bool find_for(int heads, bool balanced, DecodeKernel* out) {
  switch (heads) {
    case 1: *out = balanced ? decode_kernel_info<CT, D, BS, 1, true, TC>() : decode_kernel_info<CT, D, BS, 1, false, TC>(); return true;
    case 2: *out = balanced ? decode_kernel_info<CT, D, BS, 2, true, TC>() : decode_kernel_info<CT, D, BS, 2, false, TC>(); return true;
    case 4: *out = balanced ? decode_kernel_info<CT, D, BS, 4, true, TC>() : decode_kernel_info<CT, D, BS, 4, false, TC>(); return true;
    case 8: *out = balanced ? decode_kernel_info<CT, D, BS, 8, true, TC>() : decode_kernel_info<CT, D, BS, 8, false, TC>(); return true;
    default: return false;
  }
}

// The decode kernel for a cache type, shape and engine (fp32 caches always
// take the CUDA cores).
inline bool find_decode(pkv_dtype dt, int D, int BS, int G, bool balanced, bool tensor_cores, DecodeKernel* k) {
  switch (dt) {
    case PKV_F32: return find_decode_f32(D, BS, G, balanced, k);
    case PKV_BF16:
      return tensor_cores ? find_decode_bf16_tc(D, BS, G, balanced, k) : find_decode_bf16_cc(D, BS, G, balanced, k);
    case PKV_FP8_E4M3:
      return tensor_cores ? find_decode_fp8_tc(D, BS, G, balanced, k) : find_decode_fp8_cc(D, BS, G, balanced, k);
  }
  return false;
}

// The shared-prefix kernel of cascade decode (bf16 and fp8 caches).
struct PrefixKernel {
  const void* fn = nullptr;  // __global__ entry, parameters (PrefixArgs, TmaMaps)
  size_t smem = 0;
};

template <class CT, int D, int BS>
PrefixKernel prefix_kernel_info() {
  PrefixKernel k;
  k.fn = reinterpret_cast<const void*>(&prefix_attention_kernel<CT, D, BS>);
  k.smem = PrefixSmem<CT, D, BS>::kBytes;
  return k;
}

bool find_prefix_bf16(int head_dim, int block_size, PrefixKernel* out);
bool find_prefix_fp8(int head_dim, int block_size, PrefixKernel* out);

// The engine set by pkv_set_decode_engine (pkv_api.cu).
bool decode_on_tensor_cores();

}  // namespace pkv
