// pkv_device.cuh -- device-side building blocks shared by the kernels of
// libpkv.so: cache element types, the 1-D bulk-copy (TMA) and mbarrier
// wrappers, and the per-device error word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pkv.h"

namespace pkv {

// The per-device error word (PKV_DEVERR_* bits) lives in pkv_api.cu; every
// kernel receives its address as an argument.
__device__ __forceinline__ void raise_error(unsigned int* err, unsigned int bits) { atomicOr(err, bits); }

// ----------------------------------------------------------------------------
// Cache element types.  Each type says how many bytes one element takes and
// how a 16-byte (or narrower) shared-memory vector of elements widens to
// fp32 pairs, the operand form of the packed fp32 FMA.
// ----------------------------------------------------------------------------
struct CacheF32 {
  static constexpr int kBytes = 4;
  static constexpr pkv_dtype kDtype = PKV_F32;
  using QType = float;  // q and out type that goes with this cache
};
struct CacheBF16 {
  static constexpr int kBytes = 2;
  static constexpr pkv_dtype kDtype = PKV_BF16;
  using QType = __nv_bfloat16;
};
struct CacheFP8 {
  static constexpr int kBytes = 1;
  static constexpr pkv_dtype kDtype = PKV_FP8_E4M3;
  using QType = __nv_bfloat16;
};

__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
  // bf16 is the top half of a binary32: widening is a shift / mask.
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t two_codes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_codes & 0xFFFFu), __NV_E4M3);
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// Widen kVB bytes at `p` (shared memory, kVB-aligned) into kVB / bytes
// elements, as float2 pairs of consecutive elements.
template <class CT, int kVB>
struct VecLoad;

template <>
struct VecLoad<CacheF32, 16> {
  static constexpr int kPairs = 2;
  __device__ __forceinline__ static void run(const uint8_t* p, float2 (&o)[kPairs]) {
    float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = make_float2(v.x, v.y);
    o[1] = make_float2(v.z, v.w);
  }
};
template <>
struct VecLoad<CacheBF16, 16> {
  static constexpr int kPairs = 4;
  __device__ __forceinline__ static void run(const uint8_t* p, float2 (&o)[kPairs]) {
    uint4 v = *reinterpret_cast<const uint4*>(p);
    o[0] = bf16x2_to_f2(v.x);
    o[1] = bf16x2_to_f2(v.y);
    o[2] = bf16x2_to_f2(v.z);
    o[3] = bf16x2_to_f2(v.w);
  }
};
template <>
struct VecLoad<CacheFP8, 16> {
  static constexpr int kPairs = 8;
  __device__ __forceinline__ static void run(const uint8_t* p, float2 (&o)[kPairs]) {
    uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = e4m3x2_to_f2(w[i]);
      o[2 * i + 1] = e4m3x2_to_f2(w[i] >> 16);
    }
  }
};
template <>
struct VecLoad<CacheFP8, 8> {
  static constexpr int kPairs = 4;
  __device__ __forceinline__ static void run(const uint8_t* p, float2 (&o)[kPairs]) {
    uint2 v = *reinterpret_cast<const uint2*>(p);
    o[0] = e4m3x2_to_f2(v.x);
    o[1] = e4m3x2_to_f2(v.x >> 16);
    o[2] = e4m3x2_to_f2(v.y);
    o[3] = e4m3x2_to_f2(v.y >> 16);
  }
};

// Widen 4 consecutive elements at `p` (shared memory, aligned to 4 elements).
template <class CT>
struct Vec4Load;
template <>
struct Vec4Load<CacheF32> {
  __device__ __forceinline__ static void run(const uint8_t* p, float (&o)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
};
template <>
struct Vec4Load<CacheBF16> {
  __device__ __forceinline__ static void run(const uint8_t* p, float (&o)[4]) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    const float2 a = bf16x2_to_f2(v.x), b = bf16x2_to_f2(v.y);
    o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
  }
};
template <>
struct Vec4Load<CacheFP8> {
  __device__ __forceinline__ static void run(const uint8_t* p, float (&o)[4]) {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
    const float2 a = e4m3x2_to_f2(v), b = e4m3x2_to_f2(v >> 16);
    o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
  }
};

// q / out element access.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <class T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// ----------------------------------------------------------------------------
// mbarrier and 1-D bulk copy (TMA) wrappers, shared::cta addresses.
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One bounded probe of phase `parity`; true once that phase has completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(200000u)
      : "memory");
  return done != 0;
}

// Wait for phase `parity` with an iteration limit.  Returns false (and
// raises PKV_DEVERR_WAIT_TIMEOUT) if the limit runs out.  Each probe may
// suspend the thread for up to the hinted 0.2 ms, so 4096 probes bound the
// wait to about a second; a healthy copy completes in microseconds.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, unsigned int* err) {
#pragma unroll 1
  for (int i = 0; i < 4096; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  raise_error(err, PKV_DEVERR_WAIT_TIMEOUT);
  return false;
}

// One lane of a converged warp (the lowest active one), chosen by the hardware.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses
// 16-byte aligned) completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 2^x on the SFU (flushes subnormal results to zero; 2^-inf = +0).  Relative
// error is a few ulp, far below every tolerance the outputs are held to.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

template <class T>
__device__ __forceinline__ T ld_cg(const T* p) {
  return __ldcg(p);
}

}  // namespace pkv
