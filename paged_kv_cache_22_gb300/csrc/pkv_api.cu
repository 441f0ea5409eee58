// pkv_api.cu -- host side of libpkv.so: argument validation, workspace
// layout and kernel dispatch for the entry points declared in pkv.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/pkv.h"
#include "decode_launch.cuh"
#include "kernels.h"

namespace pkv {

// One error word per device (a __device__ variable exists once per device
// that loads the module).
__device__ unsigned int g_device_error_word;

namespace {

constexpr int kMaxCtasPerSm = 16;  // upper bound of the balanced grid, per SM
// The tensor-core decode kernel on bf16 caches fits 8 one-warp CTAs per SM;
// 7 measured faster on the Llama-3-8B-shaped, 70B-shaped and long batches
// (fewer tile copies queue at once).  fp8 caches keep every resident CTA:
// their tile loop is compute-bound, and 7 measured 12 % slower.
constexpr int kBf16TcDecodeCtasPerSm = 7;
// Balanced decode on the tensor cores: merge the segments cut between warps
// in a dependent grid (true) or inside the decode grid by tickets (false).
constexpr bool kDeferDecodeMerges = true;
constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(pkv_dtype d) {
  switch (d) {
    case PKV_F32: return 4;
    case PKV_BF16: return 2;
    case PKV_FP8_E4M3: return 1;
  }
  return 0;
}

std::mutex g_mu;
std::map<int, unsigned int*> g_err_addr;                 // device -> error word
std::map<int, int> g_sm_count;                           // device -> SMs
std::map<std::pair<const void*, int>, int> g_occupancy;  // (kernel, device) -> CTAs/SM

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

unsigned int* error_word(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_err_addr.find(dev);
  if (it != g_err_addr.end()) return it->second;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) return nullptr;
  g_err_addr[dev] = static_cast<unsigned int*>(p);
  return static_cast<unsigned int*>(p);
}

int sm_count(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_sm_count.find(dev);
  if (it != g_sm_count.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  g_sm_count[dev] = n;
  return n;
}

// Opt the kernel into its dynamic shared memory and report CTAs per SM.
int prepare_kernel(const DecodeKernel& k, int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_pair(k.fn, dev);
  auto it = g_occupancy.find(key);
  if (it != g_occupancy.end()) return it->second;
  if (cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k.smem) != cudaSuccess)
    return 0;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k.fn, k.threads, k.smem) != cudaSuccess) return 0;
  g_occupancy[key] = occ;
  return occ;
}

// Query heads served per kernel unit: the largest of 8, 4, 2, 1 dividing g.
int heads_per_unit(int g) {
  for (int G : {8, 4, 2, 1})
    if (g % G == 0) return G;
  return 1;
}

std::atomic<int> g_engine{PKV_ENGINE_TENSOR_CORES};

bool valid_cache_desc(const pkv_cache_desc* c) {
  if (!c) return false;
  if (c->num_blocks <= 0 || c->num_kv_heads <= 0) return false;
  if (c->head_dim != 64 && c->head_dim != 128) return false;
  if (c->block_size != 8 && c->block_size != 16 && c->block_size != 32) return false;
  return elem_bytes(c->dtype) != 0;
}

pkv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

// Workspace layout, both modes: [merge counters][mode-specific partials].
// The counter region has a fixed minimum size, so partials of any call never
// land where another (smaller or larger) balanced call keeps its counters.
constexpr size_t kCounterRegionMin = size_t(1) << 20;  // 262144 segments

size_t counter_region(int B, int units) {
  const size_t need = align_up((size_t)B * units * sizeof(int));
  return need > kCounterRegionMin ? need : kCounterRegionMin;
}

// Two partial-result slots per warp of the largest balanced grid.
size_t balanced_workspace(int B, int units, int G, int D, int grid_max) {
  return counter_region(B, units) + (size_t)2 * grid_max * kDecodeWarps * partial_slot_floats(G, D) * sizeof(float);
}

size_t partition_workspace(int B, int Hq, int units, int D, int P) {
  const size_t rows = (size_t)B * Hq * P;
  return counter_region(B, units) + align_up(rows * D * sizeof(float)) + 2 * align_up(rows * sizeof(float));
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (the library links only the runtime).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// The cache [num_blocks, Hkv, BS, D] as the 3-D tensor (D, Hkv * BS,
// num_blocks), one (block, kv head) tile per box, swizzled over the box row.
bool encode_cache_map(const pkv_cache_desc* c, const void* base, TmaMap* out) {
  // the last map encoded by this thread, reused while the cache is the same
  struct Memo {
    const void* base = nullptr;
    pkv_cache_desc desc{};
    TmaMap map{};
  };
  thread_local Memo memo[2];
  thread_local int next = 0;
  for (Memo& m : memo)
    if (m.base == base && std::memcmp(&m.desc, c, sizeof *c) == 0) {
      *out = m.map;
      return true;
    }
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  const int E = elem_bytes(c->dtype);
  const int row = c->head_dim * E;
  const int ib = tma_box_bytes(row);
  const cuuint64_t rows = (cuuint64_t)c->num_kv_heads * c->block_size;
  const CUtensorMapDataType dt = c->dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapSwizzle sw = ib == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  static_assert(sizeof(TmaMap) == sizeof(CUtensorMap), "opaque tensor map size");
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult rc;
  if (row == ib) {
    // (elements of a row, rows of a block, blocks): one box per tile
    const cuuint64_t dims[3] = {(cuuint64_t)c->head_dim, rows, (cuuint64_t)c->num_blocks};
    const cuuint64_t strides[2] = {(cuuint64_t)row, (cuuint64_t)row * rows};
    const cuuint32_t box[3] = {(cuuint32_t)(ib / E), (cuuint32_t)c->block_size, 1};
    rc = fn(reinterpret_cast<CUtensorMap*>(out), dt, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    // rows wider than the swizzle span: (elements of a span, rows of a block,
    // spans of a row, blocks), so that one copy brings a whole tile, laid
    // out span by span (the span stride is smaller than the row stride)
    const cuuint64_t dims[4] = {(cuuint64_t)(ib / E), rows, (cuuint64_t)(row / ib), (cuuint64_t)c->num_blocks};
    const cuuint64_t strides[3] = {(cuuint64_t)row, (cuuint64_t)ib, (cuuint64_t)row * rows};
    const cuuint32_t box[4] = {(cuuint32_t)(ib / E), (cuuint32_t)c->block_size, (cuuint32_t)(row / ib), 1};
    rc = fn(reinterpret_cast<CUtensorMap*>(out), dt, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (rc != CUDA_SUCCESS) return false;
  Memo& m = memo[next];
  next ^= 1;
  m.base = base;
  m.desc = *c;
  m.map = *out;
  return true;
}

// The cache [num_blocks, Hkv, BS, D] (bf16) as the 3-D tensor (D, Hkv * BS,
// num_blocks) with a box of one 128-byte span of one (block, kv head) tile:
// (64, BS, 1), swizzled over the span. The tcgen05 kernel for several query
// tokens stacks the spans of 64 / BS blocks into one operand per span.
bool encode_span_map(const pkv_cache_desc* c, const void* base, TmaMap* out) {
  auto fn = tensor_map_encoder();
  if (!fn || c->dtype != PKV_BF16 || c->head_dim % 64) return false;
  const cuuint64_t rows = (cuuint64_t)c->num_kv_heads * c->block_size;
  const cuuint64_t dims[3] = {(cuuint64_t)c->head_dim, rows, (cuuint64_t)c->num_blocks};
  const cuuint64_t strides[2] = {(cuuint64_t)c->head_dim * 2, (cuuint64_t)c->head_dim * 2 * rows};
  const cuuint32_t box[3] = {64, (cuuint32_t)c->block_size, 1}, estr[3] = {1, 1, 1};
  return fn(reinterpret_cast<CUtensorMap*>(out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor maps of the tcgen05 kernels: bf16, one span box per copy;
// fp8 (rows of one span), the decode kernels' whole-row box.
bool encode_tc05_maps(const pkv_cache_desc* c, const void* k, const void* v, TmaMaps* maps) {
  if (c->dtype == PKV_BF16) return encode_span_map(c, k, &maps->k) && encode_span_map(c, v, &maps->v);
  return encode_cache_map(c, k, &maps->k) && encode_cache_map(c, v, &maps->v);
}

int prepare_tc05(const Tc05Kernel& k, int dev) {
  DecodeKernel kd;
  kd.fn = k.fn;
  kd.threads = k.threads;
  kd.smem = k.smem;
  return prepare_kernel(kd, dev);
}

// Whether pkv_paged_attention_multi and the cascade's prefix pass may take
// the tcgen05 kernels (the default); tests switch them off to compare with
// the mma.sync kernels.
std::atomic<int> g_tc05{1};

}  // namespace

// The current device's error word, for entry points defined in other
// translation units of this library.
unsigned int* device_error_word(int dev) { return error_word(dev); }

bool decode_on_tensor_cores() { return g_engine.load(std::memory_order_relaxed) == PKV_ENGINE_TENSOR_CORES; }

bool encode_cache_maps(const DecodeKernel& k, const pkv_cache_desc* cache, const void* k_cache, const void* v_cache,
                       TmaMaps* maps) {
  if (!k.tensor_maps) return true;
  return encode_cache_map(cache, k_cache, &maps->k) && encode_cache_map(cache, v_cache, &maps->v);
}

}  // namespace pkv

using namespace pkv;

extern "C" {

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
  }
  return "PKV_ERR_UNKNOWN";
}

pkv_status pkv_set_decode_engine(pkv_decode_engine engine) {
  if (engine != PKV_ENGINE_TENSOR_CORES && engine != PKV_ENGINE_CUDA_CORES) return PKV_ERR_INVALID_ARG;
  g_engine.store(engine, std::memory_order_relaxed);
  return PKV_OK;
}

pkv_decode_engine pkv_get_decode_engine(void) {
  return static_cast<pkv_decode_engine>(g_engine.load(std::memory_order_relaxed));
}

void pkv_set_tcgen05(int32_t enable) { g_tc05.store(enable != 0, std::memory_order_relaxed); }

int32_t pkv_get_tcgen05(void) { return g_tc05.load(std::memory_order_relaxed); }

int32_t pkv_device_sm_count(void) {
  const int dev = current_device();
  return dev < 0 ? 0 : sm_count(dev);
}

pkv_status pkv_kv_reshape_and_cache(const void* k, const void* v, pkv_dtype src_dtype, int32_t num_tokens,
                                    void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                                    const int64_t* slot_mapping, float kv_scale, pkv_stream_t stream) {
  if (num_tokens < 0 || !valid_cache_desc(cache)) return PKV_ERR_INVALID_ARG;
  if (src_dtype != PKV_F32 && src_dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_INVALID_ARG;
  if (cache->dtype == PKV_FP8_E4M3 && !(kv_scale > 0.f && std::isfinite(kv_scale))) return PKV_ERR_INVALID_ARG;
  const int dev = current_device();
  unsigned int* err = dev < 0 ? nullptr : error_word(dev);
  if (!err) return PKV_ERR_CUDA;
  ReshapeArgs a;
  a.err = err;
  a.k = k;
  a.v = v;
  a.num_tokens = num_tokens;
  a.num_kv_heads = cache->num_kv_heads;
  a.head_dim = cache->head_dim;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.num_blocks = cache->num_blocks;
  a.block_size = cache->block_size;
  a.cache_dtype = cache->dtype;
  a.cache_bytes = elem_bytes(cache->dtype);
  a.slot_mapping = slot_mapping;
  a.kv_scale = kv_scale;
  return from_cuda(launch_reshape_and_cache(a, src_dtype == PKV_BF16, reinterpret_cast<cudaStream_t>(stream)));
}

size_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t max_seq_len, int32_t partition_tokens) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return 0;
  if (head_dim != 64 && head_dim != 128) return 0;
  if (max_seq_len < 0 || partition_tokens < 0) return 0;
  const int g = num_q_heads / num_kv_heads;
  const int G = heads_per_unit(g);
  const int units = num_kv_heads * (g / G);
  if (partition_tokens == 0) {
    const int dev = current_device();
    const int sms = dev < 0 ? 0 : sm_count(dev);
    if (sms <= 0) return 0;
    return balanced_workspace(num_seqs, units, G, head_dim, sms * kMaxCtasPerSm);
  }
  const int P = max_seq_len == 0 ? 1 : (max_seq_len + partition_tokens - 1) / partition_tokens;
  return partition_workspace(num_seqs, num_q_heads, units, head_dim, P);
}

pkv_status pkv_split_kv_reduce(void* out, pkv_dtype out_dtype, const float* o_part, const float* m_part,
                               const float* l_part, const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads,
                               int32_t head_dim, int32_t partition_tokens, int32_t max_partitions,
                               pkv_stream_t stream) {
  if (num_seqs < 0 || num_q_heads <= 0 || partition_tokens <= 0 || max_partitions <= 0) return PKV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (out_dtype != PKV_F32 && out_dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !o_part || !m_part || !l_part || !seq_lens) return PKV_ERR_INVALID_ARG;
  const int dev = current_device();
  unsigned int* err = dev < 0 ? nullptr : error_word(dev);
  if (!err) return PKV_ERR_CUDA;
  ReduceArgs a{};
  a.err = err;
  a.out = out;
  a.o_part = o_part;
  a.m_part = m_part;
  a.l_part = l_part;
  a.seq_lens = seq_lens;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.head_dim = head_dim;
  a.partition_tokens = partition_tokens;
  a.max_partitions = max_partitions;
  return from_cuda(launch_split_kv_reduce(a, out_dtype == PKV_BF16, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace pkv {
namespace {

// Options of a decode beyond the plain call: the sliding window, and the
// suffix half of cascade decode (blocks past a shared prefix, the prefix's
// partial folded in, always on the tensor cores).
struct DecodeExtras {
  int32_t window = 0, sinks = 0;
  int32_t skip_blocks = 0;
  const float* pre = nullptr;
  bool force_tc = false;
};

// Launch one decode grid; as a programmatic dependent of the previous grid on
// the stream when `programmatic` is set (its prologue then overlaps that grid).
cudaError_t launch_decode_grid(const DecodeKernel& k, dim3 grid, void** args, cudaStream_t st, bool programmatic) {
  if (!programmatic) return cudaLaunchKernel(k.fn, grid, dim3(k.threads), args, k.smem, st);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(k.threads);
  cfg.dynamicSmemBytes = k.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, k.fn, args);
}

pkv_status decode_impl(void* out, const void* q, pkv_dtype q_dtype, int32_t num_seqs, int32_t num_q_heads,
                       const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                       const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                       int32_t max_seq_len, float scale, float kv_scale, int32_t partition_tokens, void* workspace,
                       size_t workspace_bytes, pkv_stream_t stream, bool programmatic, bool dry_run = false,
                       const DecodeExtras& ex = DecodeExtras()) {
  if (num_seqs < 0 || !valid_cache_desc(cache)) return PKV_ERR_INVALID_ARG;
  if (ex.window < 0 || ex.sinks < 0 || ex.skip_blocks < 0) return PKV_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return PKV_ERR_INVALID_ARG;
  if (max_blocks_per_seq <= 0 || max_seq_len < 0 || partition_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (partition_tokens % cache->block_size) return PKV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (cache->dtype == PKV_FP8_E4M3 && !(kv_scale > 0.f && std::isfinite(kv_scale))) return PKV_ERR_INVALID_ARG;
  const pkv_dtype want_q = cache->dtype == PKV_F32 ? PKV_F32 : PKV_BF16;
  if (q_dtype != want_q) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_INVALID_ARG;

  const int D = cache->head_dim, BS = cache->block_size;
  const int g = num_q_heads / cache->num_kv_heads;
  const int G = heads_per_unit(g);
  const bool balanced = partition_tokens == 0;
  DecodeKernel k;
  if (!find_decode(cache->dtype, D, BS, G, balanced, ex.force_tc || decode_on_tensor_cores(),
                   remaps_blocks(ex.window, ex.skip_blocks), &k))
    return PKV_ERR_UNSUPPORTED;

  const int dev = current_device();
  if (dev < 0) return PKV_ERR_CUDA;
  unsigned int* err = error_word(dev);
  const int sms = sm_count(dev);
  const int occ = prepare_kernel(k, dev);
  if (!err || sms <= 0 || occ <= 0) return PKV_ERR_CUDA;

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
  a.window = ex.window;
  a.sinks = ex.window > 0 ? ex.sinks : 0;
  a.skip_blocks = ex.skip_blocks;
  a.pre = ex.pre;
  const bool fp8 = cache->dtype == PKV_FP8_E4M3;
  a.qk_scale = scale * 1.4426950408889634f * (fp8 ? kv_scale : 1.f);
  a.out_scale = fp8 ? kv_scale : 1.f;

  TmaMaps maps{};
  if (!encode_cache_maps(k, cache, k_cache, v_cache, &maps)) return PKV_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  void* args[] = {&a, &maps};
  if (balanced) {
    const int grid_max = sms * kMaxCtasPerSm;
    const size_t need = balanced_workspace(num_seqs, a.units, G, D, grid_max);
    if (!workspace || workspace_bytes < need) return PKV_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return PKV_ERR_INVALID_ARG;
    a.counters = static_cast<int*>(workspace);
    a.partials = reinterpret_cast<float*>(static_cast<char*>(workspace) + counter_region(num_seqs, a.units));
    const int cap = (k.tensor_maps && cache->dtype == PKV_BF16) ? kBf16TcDecodeCtasPerSm : kMaxCtasPerSm;
    int64_t grid = (int64_t)sms * (occ < cap ? occ : cap);
    // never more CTAs than tiles (upper bound from the host hint)
    const int64_t tiles_hint = (int64_t)num_seqs * a.units * ((a.len_clip + BS - 1) / BS);
    if (tiles_hint < grid) grid = tiles_hint > 0 ? tiles_hint : 1;
    if (dry_run) return PKV_OK;
    // A counter region beyond the fixed minimum may cover bytes that an
    // earlier call with fewer segments used for partials: clear it here, so
    // that a workspace zero-filled once serves any sequence of calls.
    const size_t region = counter_region(num_seqs, a.units);
    DecodeKernel merge;
    merge.fn = k.merge_fn;
    merge.threads = k.merge_threads;
    merge.smem = k.merge_smem;
    if (kDeferDecodeMerges && merge.fn) {
      // segments cut between warps are merged by a dependent grid once the
      // streaming is done; no merge counter is taken
      if (prepare_kernel(merge, dev) <= 0) return PKV_ERR_CUDA;
      a.defer_merge = 1;
      cudaError_t e = launch_decode_grid(k, dim3((unsigned)grid), args, st, programmatic);
      if (e != cudaSuccess) return from_cuda(e);
      int64_t nw = grid * kDecodeWarps;
      void* margs[] = {&a, &nw};
      return from_cuda(launch_decode_grid(merge, dim3((unsigned)nw), margs, st, true));
    }
    if (region > kCounterRegionMin && cudaMemsetAsync(workspace, 0, region, st) != cudaSuccess) return PKV_ERR_CUDA;
    return from_cuda(launch_decode_grid(k, dim3((unsigned)grid), args, st, programmatic));
  }
  // fixed partitions, then the log-sum-exp reduce
  const int P = max_seq_len == 0 ? 1 : (max_seq_len + partition_tokens - 1) / partition_tokens;
  const size_t need = partition_workspace(num_seqs, num_q_heads, a.units, D, P);
  if (!workspace || workspace_bytes < need) return PKV_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return PKV_ERR_INVALID_ARG;
  const size_t rows = (size_t)num_seqs * num_q_heads * P;
  char* ws = static_cast<char*>(workspace) + counter_region(num_seqs, a.units);
  a.o_part = reinterpret_cast<float*>(ws);
  a.m_part = reinterpret_cast<float*>(ws + align_up(rows * D * sizeof(float)));
  a.l_part = reinterpret_cast<float*>(ws + align_up(rows * D * sizeof(float)) + align_up(rows * sizeof(float)));
  a.partition_blocks = partition_tokens / BS;
  a.max_partitions = P;
  // one warp per (segment, partition)
  const int64_t pieces = (int64_t)num_seqs * a.units * P;
  const int64_t ctas = (pieces + kDecodeWarps - 1) / kDecodeWarps;
  if (ctas > 0x7FFFFFFF) return PKV_ERR_UNSUPPORTED;
  if (dry_run) return PKV_OK;
  cudaError_t e = launch_decode_grid(k, dim3((unsigned)ctas), args, st, programmatic);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  ReduceArgs r{};
  r.err = err;
  r.out = out;
  r.o_part = a.o_part;
  r.m_part = a.m_part;
  r.l_part = a.l_part;
  r.seq_lens = seq_lens;
  r.num_seqs = num_seqs;
  r.num_q_heads = num_q_heads;
  r.head_dim = D;
  r.partition_tokens = partition_tokens;
  r.max_partitions = P;
  r.block_size = BS;
  r.window = a.window;
  r.sinks = a.sinks;
  return from_cuda(launch_split_kv_reduce(r, q_dtype == PKV_BF16, st));
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status pkv_paged_attention_decode(void* out, const void* q, pkv_dtype q_dtype, int32_t num_seqs,
                                      int32_t num_q_heads, const void* k_cache, const void* v_cache,
                                      const pkv_cache_desc* cache, const int32_t* block_tables,
                                      int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t max_seq_len,
                                      float scale, float kv_scale, int32_t partition_tokens, void* workspace,
                                      size_t workspace_bytes, pkv_stream_t stream) {
  return decode_impl(out, q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache, cache, block_tables,
                     max_blocks_per_seq, seq_lens, max_seq_len, scale, kv_scale, partition_tokens, workspace,
                     workspace_bytes, stream, false);
}

pkv_status pkv_paged_attention_decode_window(void* out, const void* q, pkv_dtype q_dtype, int32_t num_seqs,
                                             int32_t num_q_heads, const void* k_cache, const void* v_cache,
                                             const pkv_cache_desc* cache, const int32_t* block_tables,
                                             int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                             int32_t max_seq_len, float scale, float kv_scale, int32_t window_tokens,
                                             int32_t sink_tokens, int32_t partition_tokens, void* workspace,
                                             size_t workspace_bytes, pkv_stream_t stream) {
  return decode_impl(out, q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache, cache, block_tables,
                     max_blocks_per_seq, seq_lens, max_seq_len, scale, kv_scale, partition_tokens, workspace,
                     workspace_bytes, stream, false, false, DecodeExtras{window_tokens, sink_tokens});
}

}  // extern "C"

namespace pkv {

// Pieces the cascade's prefix pass cuts the prefix into: enough warps (kv
// heads x blocks of 16 query rows x pieces) for one resident wave of
// kPrefixWarpsPerSm per SM, each piece at least kMinPieceBlocks blocks long.
constexpr int kPrefixWarpsPerSm = 12, kMinPieceBlocks = 4, kMaxPieces = 32, kMultiItemsPerSlot = 1;

int prefix_pieces(int sms, int num_seqs, int group, int num_kv_heads, int prefix_blocks) {
  const int64_t pairs = (int64_t)num_kv_heads * (((int64_t)num_seqs * group + 15) / 16);
  int64_t S = pairs > 0 ? (int64_t)sms * kPrefixWarpsPerSm / pairs : 1;
  if (prefix_blocks >= 0) S = std::min<int64_t>(S, prefix_blocks / kMinPieceBlocks);
  return (int)std::max<int64_t>(1, std::min<int64_t>(S, kMaxPieces));
}

// Byte offsets of a cascade's workspace: the balanced decode's workspace,
// then the prefix partial the decode reads, then one partial per piece when
// the prefix is cut (as many pieces as the longest prefix may get).  The
// prefix pass's merge counters (one per kv head and 16-row block) sit at the
// top of the decode's zeroed counter region, whose bottom holds the decode's:
// both fit while num_seqs * units + pairs <= 262144.
struct CascadeLayout {
  size_t counters, pre, scratch, total;
};

bool cascade_layout(int num_seqs, int num_q_heads, int num_kv_heads, int D, int max_seq_len, CascadeLayout* L) {
  const size_t dec = pkv_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, D, max_seq_len, 0);
  if (dec == 0) return false;
  const int dev = current_device();
  const int sms = dev < 0 ? 0 : sm_count(dev);
  if (sms <= 0) return false;
  const int group = num_q_heads / num_kv_heads;
  const size_t pairs = (size_t)num_kv_heads * (((size_t)num_seqs * group + 15) / 16);
  const size_t row_bytes = (size_t)num_seqs * num_q_heads * pre_row_floats(D) * sizeof(float);
  const int pieces = prefix_pieces(sms, num_seqs, group, num_kv_heads, -1);
  const size_t units = (size_t)num_kv_heads * (group / heads_per_unit(group));
  if (((size_t)num_seqs * units + pairs) * sizeof(int) > kCounterRegionMin) return false;
  L->counters = kCounterRegionMin - pairs * sizeof(int);
  L->pre = align_up(dec);
  L->scratch = L->pre + align_up(row_bytes);
  L->total = L->scratch + (pieces > 1 ? align_up(pieces * row_bytes) : 0);
  return true;
}

// Multi-token queries: pieces of the K/V range.  Each sequence's own range
// is cut into S equal pieces (in the kernel), S chosen so that the
// (sequence, kv head, 16-row block, piece) work items number about
// kMultiItemsPerSlot times the resident warps (kPrefixWarpsPerSm per SM):
// on speculative verify one item per slot measured faster than two, three
// or four (every extra piece is one more partial to write and merge).
// nb_max < 0 gives the bound the workspace is sized by.
int multi_pieces(int sms, int num_seqs, int num_kv_heads, int max_rb, int nb_max) {
  const int64_t units = (int64_t)num_seqs * num_kv_heads * max_rb;
  if (units <= 0) return 1;
  const int64_t slots = (int64_t)sms * kPrefixWarpsPerSm * kMultiItemsPerSlot;
  int64_t S = (slots + units - 1) / units;
  if (nb_max >= 0) S = std::min<int64_t>(S, nb_max / kMinPieceBlocks);
  return (int)std::max<int64_t>(1, std::min<int64_t>(S, kMaxPieces));
}

// Workspace of pkv_paged_attention_multi: merge counters (one per sequence,
// kv head and 16-row block) at the bottom of the zeroed 1 MiB counter region,
// then one partial row per (query row, query head) and piece when the K/V
// range is cut.
struct MultiLayout {
  size_t scratch, total;
  int max_rb, pieces;
  int mq_units;  // > 0: the multi-query decode serves the call, with this many units per sequence
};

// Multi-query decode: 16 rows per unit, a unit holding 16 / g tokens of one
// kv head (g a power of two up to 16); used while a (sequence, kv head) has
// at most kMqMaxRows rows, i.e. its K/V is streamed at most twice (the
// repeat, by the second unit, mostly from L2 right after the first).
constexpr int kMqMaxRows = 2 * kMqRows;
int mq_tokens_per_unit(int group) {
  return (group > 0 && group <= kMqRows && (group & (group - 1)) == 0) ? kMqRows / group : 0;
}

bool multi_layout(int num_seqs, int total_q, int max_q, int num_q_heads, int num_kv_heads, int D, MultiLayout* L) {
  if (num_seqs < 0 || total_q < 0 || max_q < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_q_heads % num_kv_heads || (D != 64 && D != 128))
    return false;
  const int dev = current_device();
  const int sms = dev < 0 ? 0 : sm_count(dev);
  if (sms <= 0) return false;
  const int group = num_q_heads / num_kv_heads;
  L->max_rb = (int)(((int64_t)max_q * group + 15) / 16);
  if ((int64_t)num_seqs * num_kv_heads * L->max_rb * sizeof(int) > kCounterRegionMin) return false;
  L->pieces = multi_pieces(sms, num_seqs, num_kv_heads, L->max_rb, -1);
  const size_t row_bytes = (size_t)total_q * num_q_heads * pre_row_floats(D) * sizeof(float);
  L->scratch = kCounterRegionMin;
  L->total = L->scratch + (L->pieces > 1 ? align_up(L->pieces * row_bytes) : 0);
  // the multi-query decode (few tokens per sequence): its merge counters and
  // two partial slots of kMqRows rows per warp of its balanced grid
  L->mq_units = 0;
  if (mq_tokens_per_unit(group) > 0 && (int64_t)max_q * group <= kMqMaxRows) {
    L->mq_units = num_kv_heads * ((max_q + mq_tokens_per_unit(group) - 1) / mq_tokens_per_unit(group));
    const size_t mq = balanced_workspace(num_seqs, L->mq_units, kMqRows, D, sms * kMaxCtasPerSm);
    if (mq > L->total) L->total = mq;
  }
  return true;
}

// The kernel pkv_paged_attention_multi runs for a call of this shape (host
// only): the tcgen05 kernel once a (sequence, kv head) fills a 128-row tile,
// or where the mma.sync kernel has no instance for the cache shape; else the
// multi-query decode for at most kMqMaxRows rows per (sequence, kv head);
// else the mma.sync multi-token kernel.  Fills the chosen kernel's entry.
struct MultiChoice {
  pkv_multi_kernel path = PKV_MULTI_NONE;
  Tc05Kernel tk;
  DecodeKernel mk;
  PrefixKernel pk;
};

MultiChoice choose_multi(int num_seqs, int max_q, int group, const pkv_cache_desc* cache) {
  MultiChoice c;
  const int D = cache->head_dim, BS = cache->block_size;
  const bool fp8 = cache->dtype == PKV_FP8_E4M3;
  if (cache->dtype == PKV_F32 || group <= 0) return c;
  const int64_t rows_max = (int64_t)max_q * group;  // rows of the largest (sequence, kv head)
  const bool one_warp = (rows_max + 15) / 16 == 1;
  const bool have_pk = fp8 ? find_multi_fp8(D, BS, one_warp, &c.pk) : find_multi_bf16(D, BS, one_warp, &c.pk);
  if (g_tc05.load(std::memory_order_relaxed) && (rows_max >= tc05::kRows || !have_pk) && num_seqs <= 65535 &&
      cache->num_kv_heads <= 65535 &&
      (fp8 ? find_tc05_fp8(D, BS, false, &c.tk) : find_tc05_bf16(D, BS, false, &c.tk))) {
    c.path = PKV_MULTI_TCGEN05;
  } else if (mq_tokens_per_unit(group) > 0 && rows_max <= kMqMaxRows && find_decode_mq(cache->dtype, D, BS, &c.mk)) {
    c.path = PKV_MULTI_QUERY_DECODE;
  } else if (have_pk) {
    c.path = PKV_MULTI_MMA_SYNC;
  }
  return c;
}

}  // namespace pkv

extern "C" {

size_t pkv_cascade_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t max_seq_len) {
  CascadeLayout L;
  return cascade_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len, &L) ? L.total : 0;
}

pkv_status pkv_cascade_decode(void* out, const void* q, pkv_dtype q_dtype, int32_t num_seqs, int32_t num_q_heads,
                              const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                              const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                              int32_t max_seq_len, int32_t prefix_blocks, float scale, float kv_scale,
                              void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
  if (prefix_blocks < 0 || prefix_blocks > max_blocks_per_seq) return PKV_ERR_INVALID_ARG;
  if (!valid_cache_desc(cache)) return PKV_ERR_INVALID_ARG;
  if (cache->dtype == PKV_F32) return PKV_ERR_UNSUPPORTED;  // the prefix kernel runs on the tensor cores
  const int D = cache->head_dim, BS = cache->block_size;
  const size_t dec = pkv_decode_workspace_bytes(num_seqs, num_q_heads, cache->num_kv_heads, D, max_seq_len, 0);
  if (prefix_blocks == 0 || num_seqs == 0)
    return decode_impl(out, q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache, cache, block_tables,
                       max_blocks_per_seq, seq_lens, max_seq_len, scale, kv_scale, 0, workspace,
                       workspace_bytes < dec ? workspace_bytes : dec, stream, false);
  CascadeLayout lay;
  if (!cascade_layout(num_seqs, num_q_heads, cache->num_kv_heads, D, max_seq_len, &lay))
    return dec == 0 ? PKV_ERR_INVALID_ARG : PKV_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < lay.total) return PKV_ERR_WORKSPACE;
  const int dev = current_device();
  const int sms = dev < 0 ? 0 : sm_count(dev);
  unsigned int* err = dev < 0 ? nullptr : error_word(dev);
  if (!err || sms <= 0) return PKV_ERR_CUDA;
  const int group = num_q_heads / cache->num_kv_heads;
  int S = prefix_pieces(sms, num_seqs, group, cache->num_kv_heads, prefix_blocks);
  const int SB = (prefix_blocks + S - 1) / S;
  S = (prefix_blocks + SB - 1) / SB;  // no empty piece
  char* ws = static_cast<char*>(workspace);
  float* pre = reinterpret_cast<float*>(ws + lay.pre);
  DecodeExtras ex;
  ex.skip_blocks = prefix_blocks;
  ex.pre = pre;
  ex.force_tc = true;
  // every argument is checked before anything is enqueued
  pkv_status st = decode_impl(out, q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache, cache, block_tables,
                              max_blocks_per_seq, seq_lens, max_seq_len, scale, kv_scale, 0, workspace, dec, stream,
                              false, /*dry_run=*/true, ex);
  if (st != PKV_OK) return st;
  const int64_t prefix_rows = (int64_t)num_seqs * group;
  Tc05Kernel t5;
  const bool fp8c = cache->dtype == PKV_FP8_E4M3;
  PrefixKernel pk;
  const bool have_pk = fp8c ? find_prefix_fp8(D, BS, &pk) : find_prefix_bf16(D, BS, &pk);
  // the tcgen05 kernel once a kv head has a full 128-row tile, or where the
  // mma.sync kernel has no instance for this cache shape
  if (g_tc05.load(std::memory_order_relaxed) && (prefix_rows >= tc05::kRows || !have_pk) &&
      cache->num_kv_heads <= 65535 && (fp8c ? find_tc05_fp8(D, BS, true, &t5) : find_tc05_bf16(D, BS, true, &t5))) {
    // the prefix pass on the tcgen05 kernel: 128 rows per CTA, the prefix cut
    // into as many pieces as fill one wave (bounded by the pieces the
    // workspace holds)
    const int64_t tiles = (prefix_rows + tc05::kRows - 1) / tc05::kRows;
    if (tiles > 65535) return PKV_ERR_UNSUPPORTED;
    int64_t S = std::max<int64_t>(1, sms / (tiles * cache->num_kv_heads));
    S = std::min<int64_t>(S, std::max(1, prefix_blocks / kMinPieceBlocks));
    S = std::min<int64_t>(S, prefix_pieces(sms, num_seqs, group, cache->num_kv_heads, -1));
    const int SB = (int)((prefix_blocks + S - 1) / S);
    S = (prefix_blocks + SB - 1) / SB;  // no empty piece
    TmaMaps tmaps{};
    if (!encode_tc05_maps(cache, k_cache, v_cache, &tmaps)) return PKV_ERR_CUDA;
    if (prepare_tc05(t5, dev) <= 0) return PKV_ERR_CUDA;
    Tc05Args ta{};
    ta.err = err;
    ta.q = static_cast<const __nv_bfloat16*>(q);
    ta.block_tables = block_tables;
    ta.table_stride = max_blocks_per_seq;
    ta.seq_lens = seq_lens;
    ta.num_seqs = num_seqs;
    ta.num_q_heads = num_q_heads;
    ta.num_kv_heads = cache->num_kv_heads;
    ta.group = group;
    ta.num_blocks = cache->num_blocks;
    const int64_t tt = (int64_t)max_blocks_per_seq * BS;
    ta.len_clip = (int)(tt < max_seq_len ? tt : max_seq_len);
    ta.prefix_blocks = prefix_blocks;
    ta.row_tiles = (int)tiles;
    ta.splits = (int)S;
    ta.split_blocks = SB;
    ta.qk_scale = scale * 1.4426950408889634f * (fp8c ? kv_scale : 1.f);
    ta.out_scale = 1.f;
    ta.pre = pre;
    ta.scratch = reinterpret_cast<float*>(ws + lay.scratch);
    ta.counters = reinterpret_cast<int*>(ws + lay.counters);
    void* targs[] = {&ta, &tmaps};
    if (cudaLaunchKernel(t5.fn, dim3((unsigned)S, (unsigned)tiles, (unsigned)cache->num_kv_heads), dim3(t5.threads),
                         targs, t5.smem, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
      return PKV_ERR_CUDA;
    return decode_impl(out, q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache, cache, block_tables,
                       max_blocks_per_seq, seq_lens, max_seq_len, scale, kv_scale, 0, workspace, dec, stream, true,
                       false, ex);
  }
  if (!have_pk) return PKV_ERR_UNSUPPORTED;
  {  // opt into the dynamic shared memory once per kernel and device
    DecodeKernel pkd;
    pkd.fn = pk.fn;
    pkd.threads = 32 * pk.warps;
    pkd.smem = pk.smem;
    if (prepare_kernel(pkd, dev) <= 0) return PKV_ERR_CUDA;
  }
  DecodeKernel tk;  // the tensor maps both kernels read the caches through
  tk.tensor_maps = true;
  TmaMaps maps{};
  if (!encode_cache_maps(tk, cache, k_cache, v_cache, &maps)) return PKV_ERR_CUDA;
  PrefixArgs pa{};
  pa.err = err;
  pa.q = q;
  pa.block_tables = block_tables;
  pa.table_stride = max_blocks_per_seq;
  pa.seq_lens = seq_lens;
  pa.num_seqs = num_seqs;
  pa.num_q_heads = num_q_heads;
  pa.num_kv_heads = cache->num_kv_heads;
  pa.group = num_q_heads / cache->num_kv_heads;
  pa.num_blocks = cache->num_blocks;
  const int64_t table_tokens = (int64_t)max_blocks_per_seq * BS;
  pa.len_clip = (int)(table_tokens < max_seq_len ? table_tokens : max_seq_len);
  pa.prefix_blocks = prefix_blocks;
  pa.row_blocks = (int)(((int64_t)num_seqs * pa.group + 15) / 16);
  pa.splits = S;
  pa.split_blocks = SB;
  const bool fp8 = cache->dtype == PKV_FP8_E4M3;
  pa.qk_scale = scale * 1.4426950408889634f * (fp8 ? kv_scale : 1.f);
  pa.pre = pre;
  pa.scratch = reinterpret_cast<float*>(ws + lay.scratch);
  pa.counters = reinterpret_cast<int*>(ws + lay.counters);
  const int64_t ctas = (int64_t)cache->num_kv_heads * ((pa.row_blocks + kPrefixWarps - 1) / kPrefixWarps) * S;
  if (ctas > 0x7FFFFFFF) return PKV_ERR_UNSUPPORTED;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  void* args[] = {&pa, &maps};
  if (cudaLaunchKernel(pk.fn, dim3((unsigned)ctas), dim3(32 * kPrefixWarps), args, pk.smem, cs) != cudaSuccess)
    return PKV_ERR_CUDA;
  // the suffix decode is the prefix pass's programmatic dependent: its
  // prologue overlaps the pass's tail, and it waits for the pass before it
  // reads a partial
  return decode_impl(out, q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache, cache, block_tables,
                     max_blocks_per_seq, seq_lens, max_seq_len, scale, kv_scale, 0, workspace, dec, stream, true,
                     false, ex);
}

size_t pkv_multi_workspace_bytes(int32_t num_seqs, int32_t total_q, int32_t max_q, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim) {
  MultiLayout L;
  return multi_layout(num_seqs, total_q, max_q, num_q_heads, num_kv_heads, head_dim, &L) ? L.total : 0;
}

pkv_multi_kernel pkv_multi_kernel_for(int32_t num_seqs, int32_t max_q, int32_t num_q_heads,
                                      const pkv_cache_desc* cache) {
  if (num_seqs < 0 || max_q <= 0 || !valid_cache_desc(cache) || num_q_heads <= 0 ||
      num_q_heads % cache->num_kv_heads)
    return PKV_MULTI_NONE;
  return choose_multi(num_seqs, max_q, num_q_heads / cache->num_kv_heads, cache).path;
}

pkv_status pkv_paged_attention_multi(void* out, const void* q, pkv_dtype q_dtype, const int32_t* q_start,
                                     int32_t num_seqs, int32_t total_q, int32_t max_q, int32_t num_q_heads,
                                     const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* seq_lens, int32_t max_seq_len, float scale, float kv_scale,
                                     void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
  if (num_seqs < 0 || total_q < 0 || max_q < 0 || !valid_cache_desc(cache)) return PKV_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return PKV_ERR_INVALID_ARG;
  if (max_blocks_per_seq <= 0 || max_seq_len < 0 || !std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (cache->dtype == PKV_FP8_E4M3 && !(kv_scale > 0.f && std::isfinite(kv_scale))) return PKV_ERR_INVALID_ARG;
  if (cache->dtype == PKV_F32 || q_dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;  // tensor cores: bf16 / fp8
  if (num_seqs == 0 || total_q == 0) return PKV_OK;
  if (max_q == 0) return PKV_ERR_INVALID_ARG;
  if (!out || !q || !q_start || !k_cache || !v_cache || !block_tables || !seq_lens) return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_INVALID_ARG;
  const int D = cache->head_dim, BS = cache->block_size;
  MultiLayout lay;
  if (!multi_layout(num_seqs, total_q, max_q, num_q_heads, cache->num_kv_heads, D, &lay)) return PKV_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < lay.total) return PKV_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return PKV_ERR_INVALID_ARG;
  const int64_t table_tokens = (int64_t)max_blocks_per_seq * BS;
  const int len_clip = (int)(table_tokens < max_seq_len ? table_tokens : max_seq_len);
  const int group = num_q_heads / cache->num_kv_heads;
  const int64_t rows_max = (int64_t)max_q * group;  // rows of the largest (sequence, kv head)
  const bool fp8 = cache->dtype == PKV_FP8_E4M3;
  const MultiChoice choice = choose_multi(num_seqs, max_q, group, cache);
  if (choice.path == PKV_MULTI_NONE) return PKV_ERR_UNSUPPORTED;
  if (choice.path == PKV_MULTI_TCGEN05) {
    const Tc05Kernel& tk = choice.tk;
    {
      const int dev = current_device();
      unsigned int* err = dev < 0 ? nullptr : error_word(dev);
      if (!err) return PKV_ERR_CUDA;
      TmaMaps maps{};
      if (!encode_tc05_maps(cache, k_cache, v_cache, &maps)) return PKV_ERR_CUDA;
      if (prepare_tc05(tk, dev) <= 0) return PKV_ERR_CUDA;
      Tc05Args ta{};
      ta.err = err;
      ta.q = static_cast<const __nv_bfloat16*>(q);
      ta.q_start = q_start;
      ta.block_tables = block_tables;
      ta.table_stride = max_blocks_per_seq;
      ta.seq_lens = seq_lens;
      ta.num_seqs = num_seqs;
      ta.total_q = total_q;
      ta.num_q_heads = num_q_heads;
      ta.num_kv_heads = cache->num_kv_heads;
      ta.group = group;
      ta.num_blocks = cache->num_blocks;
      ta.len_clip = len_clip;
      ta.max_q = max_q;
      ta.qk_scale = scale * 1.4426950408889634f * (fp8 ? kv_scale : 1.f);
      ta.out_scale = fp8 ? kv_scale : 1.f;
      ta.out = static_cast<__nv_bfloat16*>(out);
      const dim3 grid((unsigned)((rows_max + tc05::kRows - 1) / tc05::kRows), (unsigned)cache->num_kv_heads,
                      (unsigned)num_seqs);
      void* args[] = {&ta, &maps};
      return from_cuda(cudaLaunchKernel(tk.fn, grid, dim3(tk.threads), args, tk.smem,
                                        reinterpret_cast<cudaStream_t>(stream)));
    }
  }
  // few tokens per (sequence, kv head): the balanced decode kernel in its
  // multi-query form (the K/V of a sequence streamed by consecutive warps,
  // the whole batch cut into equal ranges)
  if (choice.path == PKV_MULTI_QUERY_DECODE) {
    const DecodeKernel& mk = choice.mk;
    const int dev = current_device();
    unsigned int* err = dev < 0 ? nullptr : error_word(dev);
    const int sms = dev < 0 ? 0 : sm_count(dev);
    const int occ = dev < 0 ? 0 : prepare_kernel(mk, dev);
    if (!err || sms <= 0 || occ <= 0) return PKV_ERR_CUDA;
    DecodeKernel merge;
    merge.fn = mk.merge_fn;
    merge.threads = mk.merge_threads;
    merge.smem = mk.merge_smem;
    if (!merge.fn || prepare_kernel(merge, dev) <= 0) return PKV_ERR_CUDA;
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
    a.group = group;
    a.units = lay.mq_units;
    a.units_per_kv = lay.mq_units / cache->num_kv_heads;
    a.len_clip = len_clip;
    a.q_start = q_start;
    a.mq_tpu = mq_tokens_per_unit(group);
    a.max_q = max_q;
    a.total_q = total_q;
    a.qk_scale = scale * 1.4426950408889634f * (fp8 ? kv_scale : 1.f);
    a.out_scale = fp8 ? kv_scale : 1.f;
    // segments cut between warps are merged by a dependent grid once the
    // streaming is done (merges inside the grid would queue behind the
    // SMs' tile copies at its tail)
    a.defer_merge = 1;
    const size_t region = counter_region(num_seqs, a.units);
    a.counters = static_cast<int*>(workspace);
    a.partials = reinterpret_cast<float*>(static_cast<char*>(workspace) + region);
    int64_t grid = (int64_t)sms * (occ < kMaxCtasPerSm ? occ : kMaxCtasPerSm);
    const int64_t tiles_hint = (int64_t)num_seqs * a.units * ((len_clip + BS - 1) / BS);
    if (tiles_hint < grid) grid = tiles_hint > 0 ? tiles_hint : 1;
    TmaMaps maps{};
    if (!encode_cache_maps(mk, cache, k_cache, v_cache, &maps)) return PKV_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // (no merge counters are taken: the counter region is left as it is)
    void* args[] = {&a, &maps};
    cudaError_t e = launch_decode_grid(mk, dim3((unsigned)grid), args, st, false);
    if (e != cudaSuccess) return from_cuda(e);
    int64_t nw = grid * kDecodeWarps;
    void* margs[] = {&a, &nw};
    return from_cuda(launch_decode_grid(merge, dim3((unsigned)nw), margs, st, true));
  }
  const PrefixKernel& pk = choice.pk;
  const int dev = current_device();
  const int sms = dev < 0 ? 0 : sm_count(dev);
  unsigned int* err = dev < 0 ? nullptr : error_word(dev);
  if (!err || sms <= 0) return PKV_ERR_CUDA;
  const int nb_max = (len_clip + BS - 1) / BS;
  int S = multi_pieces(sms, num_seqs, cache->num_kv_heads, lay.max_rb, nb_max);
  const int SB = nb_max > 0 ? (nb_max + S - 1) / S : 1;
  S = nb_max > 0 ? (nb_max + SB - 1) / SB : 1;  // no empty piece
  const int groups = (lay.max_rb + pk.warps - 1) / pk.warps;
  const int64_t ctas = (int64_t)num_seqs * cache->num_kv_heads * groups * S;
  if (ctas > 0x7FFFFFFF) return PKV_ERR_UNSUPPORTED;
  {  // opt into the dynamic shared memory once per kernel and device
    DecodeKernel pkd;
    pkd.fn = pk.fn;
    pkd.threads = 32 * pk.warps;
    pkd.smem = pk.smem;
    if (prepare_kernel(pkd, dev) <= 0) return PKV_ERR_CUDA;
  }
  DecodeKernel tk;
  tk.tensor_maps = true;
  TmaMaps maps{};
  if (!encode_cache_maps(tk, cache, k_cache, v_cache, &maps)) return PKV_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  PrefixArgs pa{};
  pa.err = err;
  pa.q = q;
  pa.block_tables = block_tables;
  pa.table_stride = max_blocks_per_seq;
  pa.seq_lens = seq_lens;
  pa.num_seqs = num_seqs;
  pa.num_q_heads = num_q_heads;
  pa.num_kv_heads = cache->num_kv_heads;
  pa.group = num_q_heads / cache->num_kv_heads;
  pa.num_blocks = cache->num_blocks;
  pa.len_clip = len_clip;
  pa.splits = S;
  pa.split_blocks = SB;
  pa.qk_scale = scale * 1.4426950408889634f * (fp8 ? kv_scale : 1.f);
  pa.scratch = reinterpret_cast<float*>(ws + lay.scratch);
  pa.counters = reinterpret_cast<int*>(ws);
  pa.q_start = q_start;
  pa.total_q = total_q;
  pa.max_rb = lay.max_rb;
  pa.out = out;
  pa.out_scale = fp8 ? kv_scale : 1.f;
  void* args[] = {&pa, &maps};
  if (cudaLaunchKernel(pk.fn, dim3((unsigned)ctas), dim3(32 * pk.warps), args, pk.smem,
                       reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

pkv_status pkv_decode_step(const void* k, const void* v, pkv_dtype src_dtype, int32_t num_new_tokens,
                           const int64_t* slot_mapping, void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                           void* out, const void* q, pkv_dtype q_dtype, int32_t num_seqs, int32_t num_q_heads,
                           const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                           int32_t max_seq_len, float scale, float kv_scale, int32_t partition_tokens,
                           void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
  // every argument is checked before anything is enqueued
  pkv_status st = decode_impl(out, q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache, cache, block_tables,
                              max_blocks_per_seq, seq_lens, max_seq_len, scale, kv_scale, partition_tokens,
                              workspace, workspace_bytes, stream, false, /*dry_run=*/true);
  if (st != PKV_OK) return st;
  st = pkv_kv_reshape_and_cache(k, v, src_dtype, num_new_tokens, k_cache, v_cache, cache, slot_mapping, kv_scale,
                                stream);
  if (st != PKV_OK) return st;
  // the decode is the cache write's programmatic dependent only if that grid
  // was launched (an empty write enqueues nothing)
  return decode_impl(out, q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache, cache, block_tables,
                     max_blocks_per_seq, seq_lens, max_seq_len, scale, kv_scale, partition_tokens, workspace,
                     workspace_bytes, stream, num_new_tokens > 0);
}

pkv_status pkv_gather_kv(void* k_out, void* v_out, const void* k_cache, const void* v_cache,
                         const pkv_cache_desc* cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* seq_lens, const int64_t* cu_seq_lens, int32_t num_seqs, int32_t max_seq_len,
                         pkv_stream_t stream) {
  if (num_seqs < 0 || max_seq_len < 0 || max_blocks_per_seq <= 0 || !valid_cache_desc(cache))
    return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0 || max_seq_len == 0) return PKV_OK;
  if (!k_out || !v_out || !k_cache || !v_cache || !block_tables || !seq_lens || !cu_seq_lens)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_out) || !aligned16(v_out) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  const int dev = current_device();
  unsigned int* err = dev < 0 ? nullptr : error_word(dev);
  if (!err) return PKV_ERR_CUDA;
  GatherArgs a;
  a.err = err;
  a.k_out = k_out;
  a.v_out = v_out;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.num_blocks = cache->num_blocks;
  a.block_size = cache->block_size;
  a.num_kv_heads = cache->num_kv_heads;
  a.head_dim = cache->head_dim;
  a.cache_bytes = elem_bytes(cache->dtype);
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.seq_lens = seq_lens;
  a.cu_seq_lens = cu_seq_lens;
  a.num_seqs = num_seqs;
  return from_cuda(launch_gather_kv(a, max_seq_len, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_copy_blocks(void* k_dst, void* v_dst, const pkv_cache_desc* dst, const void* k_src,
                           const void* v_src, const pkv_cache_desc* src, const int64_t* block_pairs,
                           int32_t num_pairs, pkv_stream_t stream) {
  if (num_pairs < 0 || !valid_cache_desc(dst) || !valid_cache_desc(src)) return PKV_ERR_INVALID_ARG;
  if (dst->block_size != src->block_size || dst->num_kv_heads != src->num_kv_heads ||
      dst->head_dim != src->head_dim || dst->dtype != src->dtype)
    return PKV_ERR_INVALID_ARG;
  if (num_pairs == 0) return PKV_OK;
  if (!k_dst || !v_dst || !k_src || !v_src || !block_pairs) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_dst) || !aligned16(v_dst) || !aligned16(k_src) || !aligned16(v_src) ||
      (reinterpret_cast<uintptr_t>(block_pairs) & 7u))
    return PKV_ERR_INVALID_ARG;
  const int dev = current_device();
  unsigned int* err = dev < 0 ? nullptr : error_word(dev);
  if (!err) return PKV_ERR_CUDA;
  CopyBlocksArgs a;
  a.err = err;
  a.k_dst = k_dst;
  a.v_dst = v_dst;
  a.k_src = k_src;
  a.v_src = v_src;
  a.src_blocks = src->num_blocks;
  a.dst_blocks = dst->num_blocks;
  a.block_bytes = (int64_t)src->num_kv_heads * src->block_size * src->head_dim * elem_bytes(src->dtype);
  a.pairs = block_pairs;
  a.num_pairs = num_pairs;
  return from_cuda(launch_copy_blocks(a, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_selftest_wait_timeout(pkv_stream_t stream) {
  const int dev = current_device();
  unsigned int* err = dev < 0 ? nullptr : error_word(dev);
  if (!err) return PKV_ERR_CUDA;
  return from_cuda(launch_wait_timeout_selftest(err, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_get_device_error(uint32_t* code_out, pkv_stream_t stream) {
  if (!code_out) return PKV_ERR_INVALID_ARG;
  const int dev = current_device();
  unsigned int* err = dev < 0 ? nullptr : error_word(dev);
  if (!err) return PKV_ERR_CUDA;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return PKV_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return PKV_ERR_CUDA;
  if (cudaMemset(err, 0, sizeof v) != cudaSuccess) return PKV_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return PKV_ERR_CUDA;
  *code_out = v;
  return PKV_OK;
}

}  // extern "C"
