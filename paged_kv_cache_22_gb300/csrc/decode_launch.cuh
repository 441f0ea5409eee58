// decode_launch.cuh -- registry of the compiled decode kernel instances.
#pragma once

#include "decode.cuh"
#include "decode_tc.cuh"

namespace pkv {

constexpr int kDecodeWarps = 1;  // warps per CTA: each warp is an independent worker

struct DecodeKernel {
  const void* fn = nullptr;  // __global__ entry, parameters (DecodeArgs, TmaMaps)
  int threads = 0;
  size_t smem = 0;           // dynamic shared memory bytes
  int heads_per_unit = 0;    // G
  bool tensor_maps = false;  // reads the caches through the TmaMaps parameter
};

// fp32 caches run on the CUDA cores, bf16 and fp8 caches on the tensor cores.
template <class CT, int D, int BS, int G, bool BAL>
DecodeKernel decode_kernel_info() {
  DecodeKernel k;
  if constexpr (CT::kBytes == 4) {
    k.fn = reinterpret_cast<const void*>(&decode_kernel<CT, D, BS, G, kDecodeWarps, BAL>);
    k.smem = Smem<CT, D, BS, G, kDecodeWarps>::kBytes;
  } else {
    k.fn = reinterpret_cast<const void*>(&decode_tc_kernel<CT, D, BS, G, kDecodeWarps, BAL>);
    k.smem = TcSmem<CT, D, BS, G, kDecodeWarps>::kBytes;
    k.tensor_maps = true;
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
#define PKV_DECLARE_FINDER(NAME) \
  bool NAME(int head_dim, int block_size, int heads, bool balanced, DecodeKernel* out);

PKV_DECLARE_FINDER(find_decode_f32)
PKV_DECLARE_FINDER(find_decode_bf16)
PKV_DECLARE_FINDER(find_decode_fp8)

// Shared body of the finders: the compiled (D, BS) set is passed as a list.
template <class CT, int D, int BS>
bool find_for(int heads, bool balanced, DecodeKernel* out) {
  switch (heads) {
    case 1: *out = balanced ? decode_kernel_info<CT, D, BS, 1, true>() : decode_kernel_info<CT, D, BS, 1, false>(); return true;
    case 2: *out = balanced ? decode_kernel_info<CT, D, BS, 2, true>() : decode_kernel_info<CT, D, BS, 2, false>(); return true;
    case 4: *out = balanced ? decode_kernel_info<CT, D, BS, 4, true>() : decode_kernel_info<CT, D, BS, 4, false>(); return true;
    case 8: *out = balanced ? decode_kernel_info<CT, D, BS, 8, true>() : decode_kernel_info<CT, D, BS, 8, false>(); return true;
    default: return false;
  }
}

}  // namespace pkv
