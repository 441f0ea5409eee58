// pkv_noalloc.cu -- paged decode attention for callers that cannot allocate
// device memory.
//
// pkv_paged_attention_decode needs a caller-provided workspace for the merge
// counters and partial results of the balanced split.  Some callers cannot
// obtain one: code running where device allocation is forbidden or
// unavailable -- a plugin inside a serving runtime that has reserved all
// device memory for its own pool, a caller without access to any allocator
// (plain C that only receives tensor pointers), or a latency-critical loop
// that must not touch the allocator.  This entry point instead uses scratch
// that the library holds itself: a fixed array in device global memory,
// reserved on every GPU that loads the library for as long as the process
// lives.  It allocates nothing.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/pkv.h"
#include "decode_launch.cuh"

// 16 MiB holds the merge counters (4 bytes per (sequence, kv-head unit)
// segment) and two partial-result slots per warp of the balanced grid.  On a
// 152-SM GB300 the grids these kernels run at need at most ~10 MB of slots
// (8 query heads per unit, head_dim 128: 1216 one-warp CTAs x 2 x 4160 bytes),
// which leaves room for about a million segments.  Where the slots of a full
// grid do not fit beside the counters, the grid is cut to what fits (the
// balanced split works with any grid); a call whose counters leave no room
// for even one warp's slots is refused.
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20)

static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace pkv {
unsigned int* device_error_word(int dev);  // pkv_api.cu

namespace {

constexpr int kMaxCtasPerSmNoAlloc = 16;

std::mutex g_mu;
std::map<int, unsigned char*> g_scratch;             // device -> scratch address
std::map<std::pair<const void*, int>, int> g_occ;    // (kernel, device) -> CTAs/SM

// Device address of the scratch array on `dev` (the current device).  The
// array's name in host code is only a handle; the address must come from the
// runtime, once per device.
unsigned char* scratch_on(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_scratch.find(dev);
  if (it != g_scratch.end()) return it->second;
  unsigned char* ptr = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_scratch) != cudaSuccess) return nullptr;
  g_scratch[dev] = ptr;
  return ptr;
}

int occupancy(const DecodeKernel& k, int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_pair(k.fn, dev);
  auto it = g_occ.find(key);
  if (it != g_occ.end()) return it->second;
  if (cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k.smem) != cudaSuccess) return 0;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k.fn, k.threads, k.smem) != cudaSuccess) return 0;
  g_occ[key] = occ;
  return occ;
}


bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_paged_attention_decode_noalloc(
    void* out, const void* q, pkv_dtype q_dtype, int32_t num_seqs, int32_t num_q_heads, const void* k_cache,
    const void* v_cache, const pkv_cache_desc* cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* seq_lens, int32_t max_seq_len, float scale, float kv_scale, pkv_stream_t stream) {
  if (num_seqs < 0 || !cache || max_blocks_per_seq <= 0 || max_seq_len < 0) return PKV_ERR_INVALID_ARG;
  if (cache->num_blocks <= 0 || cache->num_kv_heads <= 0) return PKV_ERR_INVALID_ARG;
  if (cache->head_dim != 64 && cache->head_dim != 128) return PKV_ERR_INVALID_ARG;
  if (cache->block_size != 8 && cache->block_size != 16 && cache->block_size != 32) return PKV_ERR_INVALID_ARG;
  if (cache->dtype != PKV_F32 && cache->dtype != PKV_BF16 && cache->dtype != PKV_FP8_E4M3)
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return PKV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (cache->dtype == PKV_FP8_E4M3 && !(kv_scale > 0.f && std::isfinite(kv_scale))) return PKV_ERR_INVALID_ARG;
  if (q_dtype != (cache->dtype == PKV_F32 ? PKV_F32 : PKV_BF16)) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_INVALID_ARG;

  const int D = cache->head_dim, BS = cache->block_size;
  const int g = num_q_heads / cache->num_kv_heads;
  int G = 1;
  for (int cand : {8, 4, 2, 1})
    if (g % cand == 0) { G = cand; break; }
  DecodeKernel k;
  if (!find_decode(cache->dtype, D, BS, G, true, decode_on_tensor_cores(), false, &k)) return PKV_ERR_UNSUPPORTED;

  int dev = -1, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PKV_ERR_CUDA;
  unsigned int* err = device_error_word(dev);
  unsigned char* scratch = scratch_on(dev);
  const int occ = occupancy(k, dev);
  if (!err || !scratch || occ <= 0) return PKV_ERR_CUDA;

  DecodeArgs a{};
  a.err = err;
  a.out = out;
  a.q = q;
  a.k_cache = static_cast<const uint8_t*>(k_cache);
  a.v_cache = static_cast<const uint8_t*>(v_cache);
  a.block_tables = block_tables;
  a.table_stride = max_blocks_per_seq;
  a.seq_lens = seq_lens;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = cache->num_kv_heads;
  a.num_blocks = cache->num_blocks;
  a.group = g;
  a.units_per_kv = g / G;
  a.units = cache->num_kv_heads * a.units_per_kv;
  const int64_t table_tokens = (int64_t)max_blocks_per_seq * BS;
  a.len_clip = (int)(table_tokens < max_seq_len ? table_tokens : max_seq_len);
  const bool fp8 = cache->dtype == PKV_FP8_E4M3;
  a.qk_scale = scale * 1.4426950408889634f * (fp8 ? kv_scale : 1.f);
  a.out_scale = fp8 ? kv_scale : 1.f;

  int64_t grid = (int64_t)sms * (occ < kMaxCtasPerSmNoAlloc ? occ : kMaxCtasPerSmNoAlloc);
  const int64_t tiles_hint = (int64_t)num_seqs * a.units * ((a.len_clip + BS - 1) / BS);
  if (tiles_hint < grid) grid = tiles_hint > 0 ? tiles_hint : 1;

  // scratch layout: [merge counters][two partial slots per warp]
  const size_t counter_bytes = round256((size_t)num_seqs * a.units * sizeof(int));
  const size_t cta_bytes = (size_t)2 * kDecodeWarps * partial_slot_floats(G, D) * sizeof(float);
  if (counter_bytes + cta_bytes > PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;  // beyond the fixed scratch
  const int64_t grid_fit = (int64_t)((PKV_NOALLOC_SCRATCH_BYTES - counter_bytes) / cta_bytes);
  if (grid > grid_fit) grid = grid_fit;

  TmaMaps maps{};
  if (!encode_cache_maps(k, cache, k_cache, v_cache, &maps)) return PKV_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the scratch keeps whatever the previous call left: the counters must
  // start at zero
  if (cudaMemsetAsync(scratch, 0, counter_bytes, st) != cudaSuccess) return PKV_ERR_CUDA;
  a.counters = reinterpret_cast<int*>(scratch);
  a.partials = reinterpret_cast<float*>(scratch + counter_bytes);
  void* args[] = {&a, &maps};
  return cudaLaunchKernel(k.fn, dim3((unsigned)grid), dim3(k.threads), args, k.smem, st) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}
