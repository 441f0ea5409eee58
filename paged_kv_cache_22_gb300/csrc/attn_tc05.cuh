// attn_tc05.cuh -- paged attention of 128-row query tiles on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in tensor memory),
// in two modes:
//
//  - MULTI: several query tokens per sequence (pkv_paged_attention_multi: a
//    prefill chunk, speculative verification). Query token i of a chunk of T
//    tokens ending at position L - 1 attends positions 0 .. L - T + i through
//    the block table, causal inside the chunk ("PagedAttention por dentro",
//    section "Chunked prefill integrado con paged KV"; "Componentes Internos
//    de Servicio de vLLM", section "Chunked prefill protege la cola del
//    TTFT"). A CTA takes 128 rows of one (sequence, kv head): row r is query
//    token r / g and query head kvh * g + r % g.
//  - PREFIX: the shared-prefix pass of cascade decode (pkv_cascade_decode).
//    Every sequence of the batch starts with the same prefix blocks ("La
//    despensa por casilleros", section "Prefix caching: compartir casilleros
//    con copy-on-write"); the rows are (sequence, query head) pairs of one kv
//    head, row R being sequence R / g, and each attends the prefix positions
//    below its length. A CTA takes 128 rows and one piece of the prefix; it
//    writes the unnormalised partial (o, m in log2 units, l) that the suffix
//    decode starts each sequence's online softmax from, the last piece of a
//    tile to finish merging the pieces by log-sum-exp.
//
// Per step of 64 positions:
//   S = Q K^T        M 128, N 64, K = D      TMEM columns 0..63 / 64..127
//   P = 2^(S - m)    eight softmax warps, two threads per row (32 columns
//                    each), into shared memory
//   O += P V         M 128, N = D, K = 64    TMEM columns 128 .. 128 + D
// Producer warps start the tile copies (tensor maps, 128-byte swizzle) into
// a ring of as many stages as shared memory holds, reading the block table
// 32 entries at a time one chunk ahead; one warp issues the MMAs, S of step
// j + 1
// while the softmax warps work on step j, and P.V of step j while they write
// P of step j + 1 (P is double-buffered).  The two threads of a row swap
// their half's maximum through shared memory each step, so that two softmax
// warps share every SM sub-partition.  O is rescaled lazily: only when a
// row's running maximum grows by more than 2^8 (probabilities stay below
// 2^8).  The score scale is folded into the exponent's FMA; only the steps
// that cross a row's causal limit or a bad block are masked.
//
// bf16 caches: the tiles land in the operand layout and P is one bf16
// operand (8 significant bits, each probability rounded once; the sums stay
// fp32).  fp8-e4m3 caches: the codes land raw and two converter warps
// widen them exactly to fp16 operand tiles; q is fp16, scaled by a
// power of two per CTA so that it cannot overflow (the factor moves to the
// fp32 score scale); P is one fp16 operand (11 significant bits).
#pragma once

#include <math_constants.h>

#include <type_traits>

#include "decode_tc.cuh"

namespace pkv {

struct Tc05Args {
  unsigned int* err;
  const __nv_bfloat16* q;  // MULTI [total_q, Hq, D]; PREFIX [B, Hq, D]
  const int32_t* q_start;  // MULTI [B + 1]
  const int32_t* block_tables;
  int64_t table_stride;
  const int32_t* seq_lens;
  int num_seqs, total_q, num_q_heads, num_kv_heads, group, num_blocks, len_clip, max_q;
  int prefix_blocks;       // PREFIX: blocks of the shared prefix, read through sequence 0's table
  int row_tiles;           // PREFIX: 128-row tiles per kv head
  int splits;              // PREFIX: pieces of the prefix range
  int split_blocks;        // PREFIX: blocks per piece
  float qk_scale;          // scale * log2(e) (* kv_scale for fp8 caches)
  float out_scale;         // MULTI: 1, or kv_scale for fp8 caches
  __nv_bfloat16* out;      // MULTI [total_q, Hq, D]
  float* pre;              // PREFIX [B * Hq][pre_row_floats(D)]: o, m, l
  float* scratch;          // PREFIX, splits > 1: [splits][B * Hq][pre_row_floats(D)]
  int* counters;           // PREFIX, splits > 1: [Hkv * row_tiles], zero between calls
};

namespace tc05 {

constexpr int kRows = 128;     // query rows per CTA (TMEM lanes)
// Positions per step: 128 for bf16 caches (fewer steps, so the fixed costs of
// a step -- barrier waits, table ids, the row-maximum exchange -- are spread
// over more work), 64 for fp8 caches (whose raw and operand rings would not
// fit shared memory at 128).
__host__ __device__ constexpr int step_tok(bool f8) { return f8 ? 64 : 128; }
constexpr int kSpan = 128;     // bytes of one 128-byte swizzle span
// S buffers in tensor memory: S(j) is computed while the softmax warps still
// work on S(j - 1) and S(j - 2), so that the issue and the latency of its
// MMAs stay off their critical path; O follows the S buffers.
constexpr int kSBuf = 3;
constexpr float kRescaleSlack = 8.f;

// Warps: 0-7 softmax (two per row of the tile); then the tensor-copy
// producers: two for bf16 caches (K and V: a copy costs its issuing thread
// about a hundred cycles, and a step needs up to 32 of them), one for fp8
// caches (half the copies); then the MMA issuers: for bf16 caches one for
// S = Q K^T and one for O += P V (an MMA costs its issuing thread tens of
// cycles, and a step has twelve), one for both with fp8 caches; then, for
// fp8 caches, two converter warps.  Twelve warps either way: at most three
// share an SM sub-partition, so that each thread may hold 168 registers.
constexpr int kConvWarps = 2;
__host__ __device__ constexpr int prod_warps(bool f8) { return f8 ? 1 : 2; }
__host__ __device__ constexpr int mma_warps(bool f8) { return f8 ? 1 : 2; }
__host__ __device__ constexpr int mma_warp(bool f8) { return 8 + prod_warps(f8); }
__host__ __device__ constexpr int conv_warp(bool f8) { return mma_warp(f8) + mma_warps(f8); }
__host__ __device__ constexpr int threads(bool f8) { return (conv_warp(f8) + (f8 ? kConvWarps : 0)) * 32; }

// Shared memory per CTA: one CTA per SM (the 320-448 threads' registers
// fill the SM's file), which keeps 1 KiB of the SM's 228 KiB for the system;
// less the barriers, the row-maximum exchange and a few words.
constexpr int kSmemPerSm = 233472;
constexpr int kSmemReserve = 2560;
__host__ __device__ constexpr int smem_budget(int) { return kSmemPerSm - 1024 - kSmemReserve; }

template <int D, bool F8>
struct Layout {
  static constexpr int kStepTok = step_tok(F8);
  static constexpr int kOCol = kSBuf * kStepTok;                 // TMEM column of O
  static constexpr int kSpans = D / 64;                          // 64 16-bit elements per span
  static constexpr int kQBytes = kSpans * kRows * kSpan;
  static constexpr int kPBuf = kRows * kStepTok * 2;             // one P buffer: [pos span][128 rows][128 B]
  static constexpr int kPBytes = 2 * kPBuf;
  static constexpr int kTile = kSpans * kStepTok * kSpan;        // one cache's operand tile of a step
  static constexpr int kRawTile = F8 ? kStepTok * D : 0;         // fp8: [step pos][D B] as copied
  // The copies must run several steps ahead of the MMAs (a tensor copy
  // takes microseconds; a step a few hundred cycles): as many K/V stages as
  // shared memory holds.  fp8: two operand stages and a deep ring of raw
  // codes (half the bytes), which the converter warps widen just in time.
  static constexpr int kFree = smem_budget(D) - kQBytes - kPBytes;
  static constexpr int kOpStagesFit = F8 ? 2 : kFree / (2 * kTile);
  static constexpr int kOpStages = kOpStagesFit > 6 ? 6 : kOpStagesFit;
  static constexpr int kRawStagesFit = F8 ? (kFree - 2 * kOpStages * kTile) / (2 * kRawTile) : 0;
  static constexpr int kRawStages = kRawStagesFit > 8 ? 8 : kRawStagesFit;
  static constexpr int kLandStages = F8 ? kRawStages : kOpStages;  // stages the tensor copies fill
  static constexpr int kQ = 0;                                   // [span][128 rows][128 B]
  static constexpr int kK = kQ + kQBytes;                        // [stage][span][step pos][128 B]
  static constexpr int kV = kK + kOpStages * kTile;
  static constexpr int kRawK = kV + kOpStages * kTile;
  static constexpr int kRawV = kRawK + kRawStages * kRawTile;
  static constexpr int kP = kRawV + kRawStages * kRawTile;       // [2][pos span][128 rows][64 pos], 16-bit
  static constexpr int kBar = kP + kPBytes;
  static constexpr int kNumBars = 2 * kLandStages + 2 * kOpStages + 2 * kSBuf + 5;
  static constexpr int kXch = (kBar + 8 * kNumBars + 15) / 16 * 16;  // [2][2][128] floats: row maxima, sums
  static constexpr int kMisc = kXch + 4 * kRows * 4;             // int max_lim, int merge flag, float max|q|
  static constexpr int kTmemSlot = kMisc + 16;
  static constexpr int kBytes = kTmemSlot + 16;
  static constexpr uint32_t kTmemCols = 512;                     // S buffers + O, a power of two
  static_assert(kTmemCols >= kSBuf * kStepTok + D, "TMEM columns");
  static_assert(!F8 || D == 128, "fp8 rows of one swizzle span");
  static_assert(kOpStages >= 2 && (!F8 || kRawStages >= 2), "at least double buffering");
  static_assert(kBytes <= smem_budget(D) + kSmemReserve, "shared memory");
};

// Table ids of the blocks of a step, read 32 entries at a time across a
// warp (lane i holds entry 32c + i of the range) with the next 32 already in
// flight, so that no step waits on a table read.
template <int NB>
struct StepIds {
  const int32_t* table;
  int jb, nblk, lane, chunk;
  int32_t cur, nxt;
  __device__ __forceinline__ int32_t load(int c) const {
    const int i = 32 * c + lane;
    return i < nblk ? __ldg(table + jb + i) : -1;
  }
  __device__ __forceinline__ void init(const int32_t* t, int jb_, int je_, int lane_) {
    table = t;
    jb = jb_;
    nblk = je_ - jb_;
    lane = lane_;
    chunk = 0;
    cur = load(0);
    nxt = load(1);
  }
  // The same bits without the ids (the softmax warps need only these): one
  // ballot per chunk of 32 entries.  Called by every lane, steps in order.
  uint32_t valid = 0;
  int valid_chunk = -1;
  __device__ __forceinline__ uint32_t bits(int j, int num_blocks) {
    const int first = j * NB;
    if (first / 32 != valid_chunk) {
      if (first / 32 != chunk) {
        cur = nxt;
        ++chunk;
        nxt = load(chunk + 1);
      }
      valid_chunk = chunk;
      valid = __ballot_sync(0xffffffffu, 32 * chunk + lane < nblk && cur >= 0 && cur < num_blocks);
    }
    return (valid >> (first % 32)) & ((1u << NB) - 1);
  }
  // bit b set when block j * NB + b of the range exists and its id is in the
  // pool; ids[b] the id.  Called by every lane of the warp, steps in order.
  __device__ __forceinline__ uint32_t step(int j, int num_blocks, int (&ids)[NB]) {
    const int first = j * NB;
    if (first / 32 != chunk) {
      cur = nxt;
      ++chunk;
      nxt = load(chunk + 1);
    }
    uint32_t ok = 0;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      ids[b] = __shfl_sync(0xffffffffu, cur, (first % 32) + b);
      if (first + b < nblk && ids[b] >= 0 && ids[b] < num_blocks) ok |= 1u << b;
    }
    return ok;
  }
};

// Shared-memory matrix descriptor, 128-byte swizzle: start >> 4, leading
// byte offset >> 4 at bit 16, stride byte offset >> 4 at bit 32, version 1
// at bit 46, swizzle mode 2 at bit 61.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// kind::f16 instruction descriptor: f32 accumulator (bit 4), A and B both
// bf16 (bits 7 and 10 set) or both fp16 (clear), A K-major, B K-major or
// MN-major (bit 16), N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_f16kind(int m, int n, bool bf16, bool b_mn) {
  return (1u << 4) | (bf16 ? (1u << 7) | (1u << 10) : 0u) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n"
               ::"r"(d_tmem), "l"(a), "l"(b), "r"(id), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive f32 columns of this thread's TMEM lane (warp w of the
// softmax group reads lanes 32w .. 32w + 31); the wait is in the same
// statement, so no use of the registers can be scheduled before it.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])),
        "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
        "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
        "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])),
        "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
        "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
        "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
        "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])),
        "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// One box of a (block, kv head) tile: BS rows of one 128-byte swizzle span,
// from the cache viewed as (D, Hkv * BS, num_blocks); x is the span's first
// element.
__device__ __forceinline__ void tma_span_tile(void* dst, const void* map, int x, int y, int blk, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(blk), "r"(smem_addr(bar))
      : "memory");
}

// Widen 16 e4m3 codes of a raw row chunk into 16 fp16 (two 16-byte chunks).
__device__ __forceinline__ void e4m3x16_to_f16(uint4 raw, uint4& lo, uint4& hi) {
  e4m3x4_to_f16x2x2(raw.x, lo.x, lo.y);
  e4m3x4_to_f16x2x2(raw.y, lo.z, lo.w);
  e4m3x4_to_f16x2x2(raw.z, hi.x, hi.y);
  e4m3x4_to_f16x2x2(raw.w, hi.z, hi.w);
}

}  // namespace tc05

template <int D, int BS, bool F8, bool PREFIX>
__global__ void __launch_bounds__(tc05::threads(F8), 1)
    attn_tc05_kernel(const __grid_constant__ Tc05Args a, const __grid_constant__ TmaMaps maps) {
  using namespace tc05;
  using SM = Layout<D, F8>;
  constexpr int kStepTok = SM::kStepTok, kOCol = SM::kOCol;
  constexpr int NB = kStepTok / BS;  // blocks per step
  constexpr int SPANS = SM::kSpans;
  constexpr int NT = threads(F8);
  extern __shared__ __align__(1024) uint8_t sm[];
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int g = a.group;

  // ---- CTA -> rows and K/V range
  int kvh, row0, rows, jb, je_cap, piece = 0, tile;
  int q0 = 0, T = 0, L = 0;
  const int32_t* table;
  if constexpr (!PREFIX) {
    const int s = blockIdx.z;
    kvh = blockIdx.y;
    tile = blockIdx.x;
    q0 = __ldg(a.q_start + s);
    T = __ldg(a.q_start + s + 1) - q0;
    L = __ldg(a.seq_lens + s);
    const bool bad = L < 0 || L > a.len_clip || T < 0 || T > L || q0 < 0 || q0 + T > a.total_q || T > a.max_q;
    if (bad) {  // flagged once per sequence; its rows are left alone
      if (tid == 0 && kvh == 0 && tile == 0) raise_error(a.err, PKV_DEVERR_BAD_SEQ_LEN);
      return;
    }
    rows = T * g;
    table = a.block_tables + (size_t)s * a.table_stride;
    jb = 0;
    je_cap = (L + BS - 1) / BS;
  } else {
    piece = blockIdx.x;
    tile = blockIdx.y;
    kvh = blockIdx.z;
    rows = a.num_seqs * g;
    table = a.block_tables;  // the prefix through sequence 0's table
    jb = piece * a.split_blocks;
    je_cap = min(a.prefix_blocks, jb + a.split_blocks);
  }
  row0 = tile * kRows;
  if (row0 >= rows) return;
  if (smem_addr(sm) & 1023u) {
    if (tid == 0) raise_error(a.err, PKV_DEVERR_SMEM_ALIGN);
    return;
  }
  constexpr int OPS = SM::kOpStages, LS = SM::kLandStages;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + SM::kBar);  // [LS] tiles (bf16) / raw codes (fp8) landed
  uint64_t* raw_free = full + LS;                               // [LS] fp8: raw codes read
  uint64_t* empty = raw_free + LS;                              // [OPS] operand tiles free (P.V done)
  uint64_t* op_full = empty + OPS;                              // [OPS] fp8: operand tiles written
  uint64_t* s_ready = op_full + OPS;                            // [kSBuf] S computed
  uint64_t* s_free = s_ready + kSBuf;                           // [kSBuf] S read by the softmax warps
  uint64_t* p_ready = s_free + kSBuf;                           // [2] P buffers written
  uint64_t* pv_done = p_ready + 2;                              // [2] P.V of a P buffer done
  uint64_t* drain = pv_done + 2;
  int* max_lim_s = reinterpret_cast<int*>(sm + SM::kMisc);
  int* last_s = max_lim_s + 1;
  unsigned* maxq_s = reinterpret_cast<unsigned*>(max_lim_s + 2);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SM::kTmemSlot);

  if (tid == 0) {
    for (int i = 0; i < LS; ++i) {
      mbar_init(&full[i], prod_warps(F8));  // every producer warp arrives
      mbar_init(&raw_free[i], kConvWarps);  // lane 0 of every converter warp
    }
    for (int i = 0; i < OPS; ++i) {
      mbar_init(&empty[i], 1);
      mbar_init(&op_full[i], kConvWarps);
    }
    for (int i = 0; i < kSBuf; ++i) {
      mbar_init(&s_ready[i], 1);
      mbar_init(&s_free[i], 8);  // lane 0 of every softmax warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_ready[i], 8);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(drain, mma_warps(F8));
    *max_lim_s = 0;
    *last_s = 0;
    *maxq_s = 0u;
    fence_mbar_init();
  }
  if (w == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tslot)),
                 "r"(SM::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  __syncthreads();

  // Row of query tile row r: valid, the q / out row, its query head, the
  // positions it attends (below lim).
  auto row_of = [&](int r, int& qrow, int& qhead, int& lim) -> bool {
    const int R = row0 + r;
    qhead = kvh * g + R % g;
    if constexpr (!PREFIX) {
      const int tok = R / g;
      qrow = q0 + tok;
      lim = L - T + tok + 1;
    } else {
      qrow = R / g;
      int Ls = R < rows ? __ldg(a.seq_lens + qrow) : 0;
      if (Ls < 0 || Ls > a.len_clip) {  // plain decode of this batch flags it too
        Ls = Ls < 0 ? 0 : a.len_clip;
      }
      lim = min(Ls, a.prefix_blocks * BS);
    }
    if (R >= rows) {
      qrow = 0;
      lim = 0;
      return false;
    }
    return true;
  };
  int my_qrow = 0, my_qhead = 0, my_lim = 0;
  bool my_valid = false;
  if (tid < 2 * kRows) {  // the softmax threads: row tid % 128
    my_valid = row_of(tid & (kRows - 1), my_qrow, my_qhead, my_lim);
    if (tid < kRows) atomicMax(max_lim_s, my_lim);
  }
  // the query tile, K-major with the 128-byte swizzle: 16-byte chunk c of row
  // r at r * 128 + ((c ^ (r % 8)) * 16) of its span; padding rows zero. fp8
  // caches: fp16 q scaled by 2^-sh, sh from the tile's largest |q|.
  auto q_chunk = [&](int i, int& r, int& c) -> uint4 {
    r = i / (D / 8);
    c = i % (D / 8);
    int qrow, qhead, lim;
    if (!row_of(r, qrow, qhead, lim)) return make_uint4(0, 0, 0, 0);
    return __ldg(reinterpret_cast<const uint4*>(a.q + ((size_t)qrow * a.num_q_heads + qhead) * D) + c);
  };
  float q_down = 1.f;
  if constexpr (F8) {
    float mq = 0.f;
    for (int i = tid; i < kRows * (D / 8); i += NT) {
      int r, c;
      const uint4 v = q_chunk(i, r, c);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = bf16x2_to_f2(u[k]);
        mq = fmaxf(mq, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
    atomicMax(maxq_s, __float_as_uint(mq));  // non-negative floats order as their bits
    __syncthreads();
    int e = 0;
    frexpf(__uint_as_float(*maxq_s), &e);
    const int sh = e > 15 ? (e - 15 < 100 ? e - 15 : 100) : 0;
    q_down = ldexpf(1.f, -sh);
  }
  // a negative scale moves its sign into q (exact), so that the largest raw
  // score is also the largest scaled one
  const uint32_t q_sign = a.qk_scale < 0.f ? 0x80008000u : 0u;
  for (int i = tid; i < kRows * (D / 8); i += NT) {
    int r, c;
    uint4 v = q_chunk(i, r, c);
    if constexpr (F8) {
      const float2 f0 = bf16x2_to_f2(v.x), f1 = bf16x2_to_f2(v.y), f2 = bf16x2_to_f2(v.z), f3 = bf16x2_to_f2(v.w);
      v = make_uint4(pack_f16x2(f0.x * q_down, f0.y * q_down), pack_f16x2(f1.x * q_down, f1.y * q_down),
                     pack_f16x2(f2.x * q_down, f2.y * q_down), pack_f16x2(f3.x * q_down, f3.y * q_down));
    }
    v.x ^= q_sign;
    v.y ^= q_sign;
    v.z ^= q_sign;
    v.w ^= q_sign;
    const int sp = c / 8, cc = c % 8;
    *reinterpret_cast<uint4*>(sm + SM::kQ + sp * (kRows * kSpan) + r * kSpan + ((cc ^ (r & 7)) << 4)) = v;
  }
  // the operand ring (and the raw ring) start zeroed: a slot no block fills
  // holds finite values, which zero probabilities then multiply
  for (int i = tid; i < (SM::kP - SM::kK) / 16; i += NT) reinterpret_cast<uint4*>(sm + SM::kK)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tslot;
  const float qk_mul = fabsf(a.qk_scale) / q_down;
  // positions at or past max_lim are attended by no row of the tile: their V
  // rows are zeroed before P.V (they may be unwritten)
  const int max_lim = *max_lim_s;
  const int je = min(je_cap, (max_lim + BS - 1) / BS);
  const int steps = je > jb ? (je - jb + NB - 1) / NB : 0;
  // the cascade's suffix decode may start its prologue on SMs this grid
  // frees (it waits for the whole grid before it reads a partial)
  if constexpr (PREFIX) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (w >= 8 && w < mma_warp(F8)) {
    // ---- producers (K then V, or both from one warp): per block of a
    // step, one tensor copy per span (bf16: into the operand tiles; fp8: one
    // 128-byte row box into the raw ring).  The whole warp reads the table;
    // lane 0 waits and copies.
    constexpr int PW = prod_warps(F8);
    const int c_lo = (w - 8) * 2 / PW, c_hi = (w - 8 + 1) * 2 / PW;  // caches of this warp: 0 K, 1 V
    uint64_t* freed = F8 ? raw_free : empty;
    StepIds<NB> sid;
    sid.init(table, jb, je, lane);
    int armed = 0;
    for (int j = 0; j < steps; ++j) {
      const int st = j % LS;
      int ids[NB];
      const uint32_t ok = sid.step(j, a.num_blocks, ids);
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&freed[st], ((j / LS) & 1) ^ 1, a.err))) break;
      armed = j + 1;
      const int left = je - jb - j * NB;
      const uint32_t want = left >= NB ? (1u << NB) - 1 : (1u << left) - 1;
      // every value above is the same on all lanes: one elected lane issues
      if (elect_one()) {
        if (ok != want && c_lo == 0) raise_error(a.err, PKV_DEVERR_BAD_BLOCK_ID);
        mbar_arrive_expect_tx(&full[st], (uint32_t)(__popc(ok) * (c_hi - c_lo) * BS * D * (F8 ? 1 : 2)));
        for (int c = c_lo; c < c_hi; ++c) {
          const TmaMap* map = c ? &maps.v : &maps.k;
          for (int b = 0; b < NB; ++b) {
            if (!(ok >> b & 1)) continue;
            if constexpr (F8) {
              const int off = st * SM::kRawTile + b * (BS * D);
              tma_span_tile(sm + (c ? SM::kRawV : SM::kRawK) + off, map, 0, kvh * BS, ids[b], &full[st]);
            } else {
              for (int sp = 0; sp < SPANS; ++sp) {
                const int off = st * SM::kTile + sp * (kStepTok * kSpan) + b * (BS * kSpan);
                tma_span_tile(sm + (c ? SM::kV : SM::kK) + off, map, sp * 64, kvh * BS, ids[b], &full[st]);
              }
            }
          }
        }
      }
      __syncwarp();
    }
    // no copy may land after the CTA is gone: wait (bounded) for the last
    // copies of every stage, consumed or not
    for (int j = max(0, armed - LS); j < armed; ++j)
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[j % LS], (j / LS) & 1, a.err))) break;
  } else if (F8 && w >= conv_warp(F8)) {
    // ---- converters (fp8): raw e4m3 rows -> fp16 operand tiles, exact; V
    // rows at positions no row attends become zero
    const int ct = tid - conv_warp(F8) * 32;
    for (int j = 0; j < steps; ++j) {
      const int rs = j % LS, st = j % OPS;
      const bool got = mbar_wait_bounded(&full[rs], (j / LS) & 1, a.err) &&
                       mbar_wait_bounded(&empty[st], ((j / OPS) & 1) ^ 1, a.err);
      if (!__all_sync(0xffffffffu, got)) break;
      const int t0 = (jb + j * NB) * BS;  // first position of the step
      // 16-byte raw chunk k of a row: codes 16k .. 16k + 15 -> operand span k / 4, chunks 2 (k % 4), + 1
#pragma unroll 2
      for (int i = ct; i < 2 * kStepTok * (D / 16); i += kConvWarps * 32) {
        const int cache = i / (kStepTok * (D / 16)), rem = i % (kStepTok * (D / 16));
        const int p = rem / (D / 16), k = rem % (D / 16);
        const uint8_t* raw = sm + (cache ? SM::kRawV : SM::kRawK) + rs * SM::kRawTile;
        uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
        if (!cache || t0 + p < max_lim)
          e4m3x16_to_f16(*reinterpret_cast<const uint4*>(raw + p * D + ((k ^ (p & 7)) << 4)), lo, hi);
        uint8_t* op = sm + (cache ? SM::kV : SM::kK) + st * SM::kTile + (k / 4) * (kStepTok * kSpan) + p * kSpan;
        const int c0 = 2 * (k % 4);
        *reinterpret_cast<uint4*>(op + ((c0 ^ (p & 7)) << 4)) = lo;
        *reinterpret_cast<uint4*>(op + (((c0 + 1) ^ (p & 7)) << 4)) = hi;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&raw_free[rs]);
        mbar_arrive(&op_full[st]);
      }
    }
  } else if (w >= mma_warp(F8) && w < conv_warp(F8)) {
    // ---- MMA issue: S(j) = Q K(j)^T into S buffer j % kSBuf ahead of the
    // softmax warps, O += P(j) V(j) once they have written P(j).  The whole
    // warp runs the loop (its values stay warp-uniform); one elected lane
    // issues each group of MMAs and their commit.
    constexpr uint32_t id_s = idesc_f16kind(kRows, kStepTok, !F8, false);
    constexpr uint32_t id_o = idesc_f16kind(kRows, D, !F8, true);
    uint64_t* ready = F8 ? op_full : full;
    // Descriptors of the operand bases; an operand at byte offset x from
    // its base adds x >> 4 to the start-address field (shared addresses
    // stay below 256 KiB, so the 14-bit field never carries).
    const uint64_t dq = sw128_desc(smem_addr(sm + SM::kQ), 16, 1024);
    const uint64_t dk = sw128_desc(smem_addr(sm + SM::kK), 16, 1024);
    const uint64_t dp = sw128_desc(smem_addr(sm + SM::kP), 16, 1024);
    // V is MN-major: 64-element spans of D kStepTok rows apart, 8-row groups 1024 B apart
    const uint64_t dv = sw128_desc(smem_addr(sm + SM::kV), kStepTok * kSpan, 1024);
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, a.err));
    };
    // S(j): its buffer is free once the softmax warps have read S(j - kSBuf)
    auto issue_s = [&](int j) -> bool {
      const int sb = j % kSBuf, st = j % OPS;
      if (j >= kSBuf && !wait_all(&s_free[sb], ((j / kSBuf) - 1) & 1)) return false;
      if (!wait_all(&ready[st], (j / OPS) & 1)) return false;
      fence_after_sync();
      const uint32_t dst = tmem + (uint32_t)(sb * kStepTok);
      const uint64_t dks = dk + (uint64_t)((st * SM::kTile) >> 4);
      if (elect_one()) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {  // 16 dims per MMA: +32 B inside a span
          const int sp = k / 4, ko = (k % 4) * 32;
          mma_bf16(dst, dq + (uint64_t)((sp * (kRows * kSpan) + ko) >> 4),
                   dks + (uint64_t)((sp * (kStepTok * kSpan) + ko) >> 4), id_s, k > 0);
        }
        mma_commit(&s_ready[sb]);
      }
      __syncwarp();
      return true;
    };
    // O += P(j) V(j) once the softmax warps have written P(j); the K/V
    // stage is free after it (S(j) completed before P(j) could be written)
    auto issue_pv = [&](int j) -> bool {
      const int pb = j & 1;  // P buffer of this step
      if (!wait_all(&p_ready[pb], (j >> 1) & 1)) return false;
      fence_after_sync();
      const int st = j % OPS;
      const uint64_t dps = dp + (uint64_t)((pb * SM::kPBuf) >> 4);
      const uint64_t dvs = dv + (uint64_t)((st * SM::kTile) >> 4);
      if (elect_one()) {
#pragma unroll
        for (int k = 0; k < kStepTok / 16; ++k)  // 16 positions per MMA: +32 B in P, +16 rows in V
          mma_bf16(tmem + kOCol, dps + (uint64_t)(((k / 4) * (kRows * kSpan) + (k % 4) * 32) >> 4),
                   dvs + (uint64_t)((k * 16 * kSpan) >> 4), id_o, (j > 0 || k > 0) ? 1u : 0u);
        mma_commit(&empty[st]);
        mma_commit(&pv_done[pb]);
      }
      __syncwarp();
      return true;
    };
    bool ok = true;
    if constexpr (mma_warps(F8) == 1) {
      // S runs LA steps ahead of P.V, no further than the S buffers allow
      // nor than the operand stages: S(j) needs stage j % OPS, which only
      // P.V(j - OPS) frees, and this loop issues that after S(j - OPS + LA)
      constexpr int LA = (kSBuf < OPS ? kSBuf : OPS) - 1;
      for (int j = 0; ok && j < steps + LA; ++j) {
        if (j < steps) ok = issue_s(j);
        if (ok && j >= LA) ok = issue_pv(j - LA);
      }
    } else if (w == mma_warp(F8)) {
      for (int j = 0; ok && j < steps; ++j) ok = issue_s(j);
    } else {
      for (int j = 0; ok && j < steps; ++j) ok = issue_pv(j);
    }
    // every MMA issued has completed before TMEM is released
    if (elect_one()) mma_commit(drain);
    __syncwarp();
    wait_all(drain, 0);
  } else if (w < 8) {
    // ---- softmax: two threads per row of the tile (TMEM lane r).  Warp w
    // takes the column half h = w / 4 of every step's S and the same half of
    // O's columns, so that two warps share each SM sub-partition; the two
    // threads of a row exchange their half's maximum in shared memory.
    const int r = tid & (kRows - 1), h = w >> 2;
    const uint32_t lane_base = tmem + ((uint32_t)((w & 3) * 32) << 16);
    float* xch = reinterpret_cast<float*>(sm + SM::kXch);  // [2 steps][2 halves][128 rows]
    constexpr int HC = kStepTok / 2;                       // columns of a half
    constexpr int HB = HC / BS;                            // blocks of a half
    constexpr int OC = D / 64;                             // 32-column chunks of O per half
    const uint32_t half_blocks = ((1u << HB) - 1) << (h * HB);
    float m_used = -CUDART_INF_F, l = 0.f;
    bool ok = true;
    StepIds<NB> sid;
    sid.init(table, jb, je, lane);
    for (int j = 0; j < steps; ++j) {
      const int st = j % OPS, pb = j & 1;
      const uint32_t okb = sid.bits(j, a.num_blocks);
      const int t0 = (jb + j * NB) * BS, th = t0 + h * HC;  // first position of the step, of this half
      // a half-step where every position of every row of this warp is kept needs no mask
      const bool interior = __all_sync(0xffffffffu, th + HC <= my_lim && (okb & half_blocks) == half_blocks);
      const int sb = j % kSBuf;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(&s_ready[sb], (j / kSBuf) & 1, a.err)))) break;
      fence_after_sync();
      // S is read twice, 32 columns at a time: once for the maximum, once
      // for the exponentials, so that only 32 scores are live at a time
      const uint32_t s_col = lane_base + (uint32_t)(sb * kStepTok + h * HC);
      // the largest raw score of this half (qk_mul >= 0), four independent
      // chains; on a boundary step `keep` marks the positions the row attends
      float mx[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
      uint64_t keep = ~0ull;
      if (!interior) {
        const int lim = min(max(my_lim - th, 0), HC);
        keep = lim >= 64 ? ~0ull : ((1ull << lim) - 1);
#pragma unroll
        for (int b = 0; b < HB; ++b)
          if (!(okb >> (h * HB + b) & 1)) keep &= ~(((1ull << BS) - 1) << (b * BS));
      }
#pragma unroll
      for (int cc = 0; cc < HC / 32; ++cc) {
        float sc[32];
        tmem_ld32(s_col + 32 * cc, sc);
        if (interior) {
#pragma unroll
          for (int c = 0; c < 32; ++c) mx[c & 3] = fmaxf(mx[c & 3], sc[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (keep >> (32 * cc + c) & 1) mx[c & 3] = fmaxf(mx[c & 3], sc[c]);
        }
      }
      const float mine = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      xch[(j & 1) * 2 * kRows + h * kRows + r] = mine;
      asm volatile("bar.sync 2, 256;" ::: "memory");
      const float mraw = fmaxf(mine, xch[(j & 1) * 2 * kRows + (h ^ 1) * kRows + r]);
      const float mt = mraw == -CUDART_INF_F ? -CUDART_INF_F : mraw * qk_mul;
      float factor = 1.f;
      if (mt > m_used + kRescaleSlack) {
        factor = m_used == -CUDART_INF_F ? 0.f : fast_exp2(m_used - mt);
        m_used = mt;
        l *= factor;
      }
      // P buffer pb is free once the P.V of two steps ago is done; a rescale
      // of O needs the previous step's P.V done as well (rare: the maximum
      // must grow by more than the slack)
      const bool rescale = j > 0 && __any_sync(0xffffffffu, factor != 1.f);
      if (j >= 2 && !(ok = __all_sync(0xffffffffu, mbar_wait_bounded(&pv_done[pb], ((j - 2) >> 1) & 1, a.err))))
        break;
      if (rescale &&
          !(ok = __all_sync(0xffffffffu, mbar_wait_bounded(&pv_done[pb ^ 1], ((j - 1) >> 1) & 1, a.err))))
        break;
      fence_after_sync();
      if (rescale) {  // a warp rescales its rows' half of O together (tcgen05.ld / st are warp-wide)
#pragma unroll
        for (int c = 0; c < OC; ++c) {
          float o[32];
          const uint32_t col = kOCol + (uint32_t)((h * OC + c) * 32);
          tmem_ld32(lane_base + col, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= factor;
          tmem_st32(lane_base + col, o);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      // p = 2^(s * qk_mul - m): a row with nothing kept yet (m = -inf) has
      // only masked scores, which give 0
      const float nm = m_used == -CUDART_INF_F ? 0.f : -m_used;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
      // this half's positions within P: span (h * HC) / 64, 16-byte chunks
      // from ((h * HC) % 64) / 8 on
      uint8_t* prow = sm + SM::kP + pb * SM::kPBuf + ((h * HC) / 64) * (kRows * kSpan) + r * kSpan;
      const int c0 = ((h * HC) % 64) / 8;
      auto emit_p = [&](auto masked) {
#pragma unroll
        for (int cc = 0; cc < HC / 32; ++cc) {
          float sc[32];
          tmem_ld32(s_col + 32 * cc, sc);
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = c4 * 8 + 2 * e;
              float p0 = fast_exp2(fmaf(sc[c], qk_mul, nm));
              float p1 = fast_exp2(fmaf(sc[c + 1], qk_mul, nm));
              if constexpr (decltype(masked)::value) {
                p0 = keep >> (32 * cc + c) & 1 ? p0 : 0.f;
                p1 = keep >> (32 * cc + c + 1) & 1 ? p1 : 0.f;
              }
              ls[e] += p0 + p1;
              pk[e] = F8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
            }
            *reinterpret_cast<uint4*>(prow + (((c0 + 4 * cc + c4) ^ (r & 7)) << 4)) =
                make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
      };
      if (interior)
        emit_p(std::false_type{});
      else
        emit_p(std::true_type{});
      // S buffer sb may take S(j + kSBuf) now
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[sb]);
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      if constexpr (!F8) {
        // V rows of positions no row attends (the tile's last step) become zero
        const int z0 = max(0, max_lim - t0);
        if (z0 < kStepTok) {
          for (int i = tid; i < (kStepTok - z0) * SPANS * 8; i += 2 * kRows) {
            const int p = z0 + i / (SPANS * 8), sp = (i / 8) % SPANS, c = i % 8;
            *reinterpret_cast<uint4*>(sm + SM::kV + st * SM::kTile + sp * (kStepTok * kSpan) + p * kSpan + (c << 4)) =
                make_uint4(0, 0, 0, 0);
          }
        }
      }
      fence_proxy_async_smem();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_ready[pb]);
    }
    // every P.V issued has completed before O is read
    if (ok && steps > 0)
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&pv_done[(steps - 1) & 1], ((steps - 1) >> 1) & 1, a.err));
    if (ok && steps > 1)
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&pv_done[(steps - 2) & 1], ((steps - 2) >> 1) & 1, a.err));
    fence_after_sync();
    // the row's sum: both halves' shares, through the exchange area (every
    // read of the last step's maxima is done once all 256 threads are here)
    asm volatile("bar.sync 2, 256;" ::: "memory");
    xch[h * kRows + r] = l;
    asm volatile("bar.sync 2, 256;" ::: "memory");
    l += xch[(h ^ 1) * kRows + r];
    // ---- epilogue: each thread its half of the row's columns
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    if constexpr (!PREFIX) {
      if (ok) {
        __nv_bfloat16* orow = a.out + ((size_t)my_qrow * a.num_q_heads + my_qhead) * D;
        const float sc_out = inv_l * a.out_scale;
#pragma unroll
        for (int c = 0; c < OC; ++c) {
          float o[32];
          const int cc = h * OC + c;
          tmem_ld32(lane_base + kOCol + cc * 32, o);
          if (my_valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(pack_bf16x2(o[8 * v] * sc_out, o[8 * v + 1] * sc_out),
                                  pack_bf16x2(o[8 * v + 2] * sc_out, o[8 * v + 3] * sc_out),
                                  pack_bf16x2(o[8 * v + 4] * sc_out, o[8 * v + 5] * sc_out),
                                  pack_bf16x2(o[8 * v + 6] * sc_out, o[8 * v + 7] * sc_out));
          }
        }
      }
    } else {
      // this piece's partial (o relative to m, m in log2 units, l); an empty
      // piece (or one that gave up) writes o = 0, m = -inf, l = 0
      constexpr int PRF = pre_row_floats(D);
      const size_t all_rows = (size_t)a.num_seqs * a.num_q_heads;
      const size_t orow = (size_t)my_qrow * a.num_q_heads + my_qhead;
      const bool have = ok && steps > 0;
      float* dst = (a.splits == 1 ? a.pre : a.scratch + (size_t)piece * all_rows * PRF) + orow * PRF;
#pragma unroll
      for (int c = 0; c < OC; ++c) {
        float o[32];
        const int cc = h * OC + c;
        if (have) {
          tmem_ld32(lane_base + kOCol + cc * 32, o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0.f;
        }
        if (my_valid) {
#pragma unroll
          for (int v = 0; v < 8; ++v)
            reinterpret_cast<float4*>(dst + cc * 32)[v] = make_float4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
        }
      }
      if (my_valid && h == 0) {
        dst[D] = have ? m_used : -CUDART_INF_F;
        dst[D + 1] = have ? l : 0.f;
      }
      if (a.splits > 1) {
        // the last piece of this (kv head, tile) to finish merges them all,
        // each thread its half of the row's columns
        __threadfence();
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (tid == 0) {
          int* ctr = a.counters + (size_t)kvh * a.row_tiles + tile;
          const int last = atomicAdd(ctr, 1) == a.splits - 1;
          if (last) *ctr = 0;  // ready for the next call
          *last_s = last;
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (*last_s && my_valid) {
          __threadfence();
          float M = -CUDART_INF_F;
          for (int k = 0; k < a.splits; ++k) M = fmaxf(M, __ldcg(a.scratch + ((size_t)k * all_rows + orow) * PRF + D));
          const float Mc = M == -CUDART_INF_F ? 0.f : M;
          float den = 0.f;
          for (int k = 0; k < a.splits; ++k) {
            const float* pk = a.scratch + ((size_t)k * all_rows + orow) * PRF;
            den += fast_exp2(__ldcg(pk + D) - Mc) * __ldcg(pk + D + 1);
          }
          float* out = a.pre + orow * PRF;
#pragma unroll 1
          for (int c = 0; c < OC; ++c) {  // 32 dims at a time
            const int cc = h * OC + c;
            float4 acc[8];
#pragma unroll
            for (int v = 0; v < 8; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int k = 0; k < a.splits; ++k) {
              const float* pk = a.scratch + ((size_t)k * all_rows + orow) * PRF;
              const float wk = fast_exp2(__ldcg(pk + D) - Mc);
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                const float4 x = __ldcg(reinterpret_cast<const float4*>(pk + cc * 32) + v);
                acc[v].x += wk * x.x;
                acc[v].y += wk * x.y;
                acc[v].z += wk * x.z;
                acc[v].w += wk * x.w;
              }
            }
#pragma unroll
            for (int v = 0; v < 8; ++v) reinterpret_cast<float4*>(out + cc * 32)[v] = acc[v];
          }
          if (h == 0) {
            out[D] = M;
            out[D + 1] = den;
          }
        }
      }
      // the prefix blocks a sequence attends must be those of sequence 0's
      // table: kv head 0's CTAs check the sequences of their rows over their
      // piece, one (sequence, block) pair per thread at a time (entries past
      // a short sequence's end are not read by plain decode either)
      if (kvh == 0) {
        const int s_lo = row0 / g, s_hi = min(a.num_seqs, (min(row0 + kRows, rows) - 1) / g + 1);
        const int nblk = je_cap - jb;
        for (int i = tid; i < (s_hi - s_lo) * nblk; i += 2 * kRows) {
          const int sq = s_lo + i / nblk, jj = jb + i % nblk;
          int Ls = __ldg(a.seq_lens + sq);
          Ls = Ls < 0 ? 0 : (Ls > a.len_clip ? a.len_clip : Ls);
          if (jj < (Ls + BS - 1) / BS &&
              __ldg(a.block_tables + (size_t)sq * a.table_stride + jj) != __ldg(a.block_tables + jj))
            raise_error(a.err, PKV_DEVERR_BAD_BLOCK_ID);
        }
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  if (w == 0) {
    fence_after_sync();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(SM::kTmemCols) : "memory");
  }
}

}  // namespace pkv
