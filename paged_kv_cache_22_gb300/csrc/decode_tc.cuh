// decode_tc.cuh -- paged decode attention on the tensor cores (bf16 and
// fp8-e4m3 caches).
//
// Computes what decode_common.cuh states.  The two contractions of a decode
// step are dense once grouped-query heads are stacked: the G query heads of a
// kv head against one tile of K (G x D times D x 16 tokens) and their
// probabilities against the tile of V (G x 16 times 16 x D).  On the CUDA
// cores each element of K and V costs a widening and a fused multiply-add per
// query head, which makes decode issue-bound long before HBM is saturated;
// here both contractions run as mma.sync m16n8k16 with fp32 accumulation, so
// a 16-token tile costs about a hundred warp instructions.
//
// Design (GB300):
//  * Tiles arrive by TMA tensor copies (cp.async.bulk.tensor.3d) of one
//    (block, kv head) tile of K and of V, the cache viewed as the tensor
//    (D, Hkv * BS, num_blocks) with a 128-byte (64-byte for 64-byte rows)
//    swizzle, so that the 8 rows an ldmatrix phase reads fall in 8 distinct
//    bank groups.  Each warp is an independent worker with its own ring of
//    NSW stages and mbarriers, exactly as in the CUDA-core kernel; the
//    balanced split and the ticket merge are shared with it.
//  * Rows of the m16 operand of q.K are the G query heads (G <= 8; rows
//    G..15 are zero and their results dropped).  Lane (g, t) = (lane / 4,
//    lane % 4) owns head g: its running max, its share of the row sum and
//    its 4 x D / 8 accumulators.
//  * q.K: A = q (registers, loaded once per piece), B = K tile through
//    ldmatrix (K rows are the n index, head dims the k index).  Scores are
//    scaled in fp32, masked past the sequence end, and enter an online
//    softmax in log2 units; the rescale of the accumulators is a warp-uniform
//    branch taken only when some row's max grew.
//  * P.V: the probabilities leave the q.K accumulators already in the A
//    operand layout of the next contraction (row g, tokens 2t, 2t+1, 2t+8,
//    2t+9).  P is split into a head and a remainder of the operand type (bf16
//    or fp16), so each weight keeps ~16 or more significant bits: the head
//    fills rows 0..7 of the m16 operand, the remainder rows 8..15, one MMA
//    per n-tile serves both, and the two row halves of the accumulator are
//    summed when the piece ends.
//  * Several query tokens per sequence (speculative verify, short chunks):
//    a unit is 16 rows, (token, head) pairs of one kv head, so that rows g
//    and g + 8 of both m16 operands are query rows.  A lane then keeps two
//    rows' softmax state, P is one operand of the MMA type (its weights keep
//    8 significant bits for bf16, 11 for fp16), and each row attends the
//    positions up to its own token.
//  * bf16 caches: V arrives through ldmatrix.trans.  fp8 caches: K and V
//    codes widen exactly to fp16 (cvt e4m3x2 -> f16x2); q is fp16,
//    pre-scaled by a power of two chosen per piece so that it cannot
//    overflow, the factor moved to the fp32 score scale.  For fp8 V the n
//    index is permuted so that a lane's four token rows are read as 16
//    contiguous bytes each: output column n of n-tile j is head dim
//    (D / 8) * n + j.
#pragma once

#include "decode_common.cuh"

namespace pkv {

// ----------------------------------------------------------------------------
// Instruction wrappers.
// ----------------------------------------------------------------------------

// One box of a 3-D tensor map into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const TmaMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const TmaMap* map, int x, int y, int z, int w, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// c[16x8] += A[16x16] . B[16x8] with rows 8..15 of A zero: a0 / a2 are the
// row-g halves (k 2t..2t+1 / 2t+8..2t+9), c0 / c1 columns 2t, 2t+1 of row g.
template <bool F16>
__device__ __forceinline__ void mma_k16(float& c0, float& c1, uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  float x2, x3;
  if constexpr (F16) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %5}, {%7, %8}, "
        "{%0, %1, %9, %9};"
        : "+f"(c0), "+f"(c1), "=f"(x2), "=f"(x3)
        : "r"(a0), "r"(0u), "r"(a2), "r"(b0), "r"(b1), "f"(0.f));
    (void)x2, (void)x3;
  } else {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %5}, {%7, %8}, "
        "{%0, %1, %9, %9};"
        : "+f"(c0), "+f"(c1), "=f"(x2), "=f"(x3)
        : "r"(a0), "r"(0u), "r"(a2), "r"(b0), "r"(b1), "f"(0.f));
    (void)x2, (void)x3;
  }
}

// c[16x8] += A[16x16] . B[16x8], all 16 rows: c0 / c1 row g, c2 / c3 row g+8.
template <bool F16>
__device__ __forceinline__ void mma_k16_rows16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  if constexpr (F16) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// c[16x8] += A[16x8] . B[8x8] (bf16), all 16 rows.
__device__ __forceinline__ void mma_k8_bf16_rows16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, "
               "{%0, %1, %2, %3};"
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
               : "r"(a0), "r"(a1), "r"(b0));
}

// (lo, hi) -> packed pair, lo in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float2 f16x2_to_f2(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// Four e4m3 codes -> two exact fp16 pairs: bytes (0, 1) -> lo, (2, 3) -> hi.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// ----------------------------------------------------------------------------
// Geometry.
// ----------------------------------------------------------------------------
template <class CT, int D, int BS, int G>
struct TcGeo {
  static constexpr bool F8 = CT::kBytes == 1;
  static constexpr int E = CT::kBytes;
  static constexpr int ROW = D * E;              // bytes of one token row
  static constexpr int IB = tma_box_bytes(ROW);  // bytes of a box row = swizzle span
  static constexpr int NBX = ROW / IB;           // boxes per tile
  static constexpr int BOX = BS * IB;            // bytes of one box
  static constexpr int TILE = BS * ROW;          // bytes of one (block, kv head) tile
  static constexpr int STAGE = 2 * TILE;         // K tile then V tile
  static constexpr int TB = BS < 16 ? BS : 16;   // tokens per compute step
  static constexpr int STEPS = BS / TB;
  static constexpr int NTS = TB / 8;             // score n-tiles per step
  static constexpr int KS = D / 16;              // k-steps of q.K
  static constexpr int NTO = D / 8;              // output n-tiles
  static constexpr int VPL = D / 8;              // fp8 V: bytes of a token row per lane
  static constexpr int NSW0 = 16384 / STAGE;
  static constexpr int NSW = NSW0 < 2 ? 2 : (NSW0 > 8 ? 8 : NSW0);  // stages per warp
  static_assert((G >= 1 && G <= 8) || G == 16, "up to 8 query rows (P head + remainder) or 16");
  static_assert(IB == 128 || IB == 64, "swizzle span");
  static_assert(ROW % IB == 0 && KS % 2 == 0, "tile shape");
  static_assert(!F8 || TB == 16, "fp8 caches: 16-token steps");
  static_assert(TB == 8 || TB == 16, "compute step");
  static_assert(STAGE % 1024 == 0 && BOX % 512 == 0, "stages and boxes keep the swizzle phase");
};

template <class CT, int D, int BS, int G, int W, bool REMAP>
struct TcSmem {
  using GE = TcGeo<CT, D, BS, G>;
  static constexpr size_t kStages = 0;  // 1024-byte aligned
  static constexpr size_t kQBuf = kStages + (size_t)W * GE::NSW * GE::STAGE;
  static constexpr size_t kBars = (kQBuf + (size_t)W * 2 * G * D * sizeof(__nv_bfloat16) + 7) / 8 * 8;
  static constexpr size_t kQBars = kBars + (size_t)W * GE::NSW * 8;
  static constexpr size_t kOk = kQBars + (size_t)W * 2 * 8;
  // cascade (REMAP kernels): one warp's next prefix partial (G rows), and its barrier
  static constexpr size_t kPBuf = (kOk + (size_t)W * GE::NSW * 4 + 15) / 16 * 16;
  static constexpr size_t kPBar = kPBuf + (REMAP ? (size_t)W * G * pre_row_floats(D) * sizeof(float) : 0);
  static constexpr size_t kMBar = kPBar + (size_t)W * 8;  // the merges' bulk copies
  static constexpr size_t kBytes = kMBar + (size_t)W * 8;
  // partial slots a one-warp CTA's stage ring and q buffers (contiguous) hold
  // once its range is done; its merges stage slots there
  static constexpr int kMergeCap =
      W == 1 ? (int)((kBars - kStages) / (partial_slot_floats(G, D) * sizeof(float))) : 0;
};

// One (block, kv head) tile of a cache into `dst`: row-wide boxes with one
// copy each (3-D map), or, for rows wider than the swizzle span, every span
// of the tile in one copy (4-D map); the layout is the same, span by span.
template <class GE>
__device__ __forceinline__ void tma_load_tile(void* dst, const TmaMap* map, int row0, int block, uint64_t* bar) {
  if constexpr (GE::NBX == 1) {
    tma_load_3d(dst, map, 0, row0, block, bar);
  } else {
    tma_load_4d(dst, map, 0, row0, 0, block, bar);
  }
}

// Byte offset, within a tile, of 16-byte chunk c of token row `row` as the
// swizzled tensor copy lays it out: chunk index XOR the 128-byte line index
// (bits 4..6 ^= bits 7..9; for 64-byte spans bits 4..5 ^= bits 7..8).
template <class GE>
__device__ __forceinline__ uint32_t swz(int row, int c) {
  constexpr int CPB = GE::IB / 16;
  const uint32_t off = (uint32_t)((c / CPB) * GE::BOX + row * GE::IB + (c % CPB) * 16);
  constexpr uint32_t M = GE::IB == 128 ? 7u : 3u;
  return off ^ (((off >> 7) & M) << 4);
}

// ----------------------------------------------------------------------------
// The kernel.
// ----------------------------------------------------------------------------
// MQ: several query tokens per sequence (balanced split, no remap): a unit
// is (kv head, group of a.mq_tpu tokens) and its G = a.mq_tpu * group rows
// are (token, head) pairs, each with its own causal limit (G = 16: two rows
// per lane).
template <class CT, int D, int BS, int G, int W, bool BALANCED, bool REMAP, bool MQ = false>
__global__ void __launch_bounds__(W * 32, 8 / W)
    decode_tc_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ TmaMaps maps) {
  static_assert(!MQ || (BALANCED && !REMAP), "multi-query: balanced split, no remap");
  // 16-row units (multi-query): rows g and g + 8 of the m16 operands are both
  // query rows, and P is a single operand of the MMA type (no remainder)
  constexpr bool R16 = G == 16;
  constexpr int RPL = R16 ? 2 : 1;  // query rows per lane: g (and g + 8)
  constexpr int RE = 2 * RPL;       // score / accumulator entries per n-tile and lane
  static_assert(!R16 || MQ, "16-row units: multi-query only");
  using GE = TcGeo<CT, D, BS, G>;
  using SM = TcSmem<CT, D, BS, G, W, REMAP>;
  using QT = typename CT::QType;
  constexpr bool F8 = GE::F8;
  constexpr int NSW = GE::NSW, TB = GE::TB, KS = GE::KS, NTO = GE::NTO, TILE = GE::TILE, STAGE = GE::STAGE;

  extern __shared__ __align__(1024) uint8_t tc_smem[];
  uint8_t* const smem = tc_smem;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  if (smem_addr(smem) & 1023u) {  // the swizzle phase needs 1024-byte aligned stages
    if (threadIdx.x == 0) raise_error(a.err, PKV_DEVERR_SMEM_ALIGN);
    return;
  }
  uint8_t* stages = smem + SM::kStages + (size_t)w * NSW * STAGE;
  const uint32_t stages_s = smem_addr(stages);
  QT* qbuf = reinterpret_cast<QT*>(smem + SM::kQBuf) + (size_t)w * 2 * G * D;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kBars) + w * NSW;
  uint64_t* qbars = reinterpret_cast<uint64_t*>(smem + SM::kQBars) + w * 2;
  int* stage_ok = reinterpret_cast<int*>(smem + SM::kOk) + w * NSW;
  float* pbuf = reinterpret_cast<float*>(smem + SM::kPBuf) + (size_t)w * G * pre_row_floats(D);
  uint64_t* pbar = reinterpret_cast<uint64_t*>(smem + SM::kPBar) + w;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + SM::kMBar) + w;

  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < NSW; ++i) mbar_init(&bars[i], 1);
    mbar_init(&qbars[0], 1);
    mbar_init(&qbars[1], 1);
    mbar_init(pbar, 1);
    mbar_init(mbar, 1);
    fence_mbar_init();
  }
  __syncthreads();  // the only block-wide barrier: warps are independent from here on

  const int64_t gw = (int64_t)blockIdx.x * W + w;
  const int64_t NW = (int64_t)gridDim.x * W;
  int64_t u0 = 0, u1 = 0, T = 0;
  Walker wk0;
  if (!plan_warp<QT, D, BS, BALANCED>(a, gw, NW, lane, wk0, u0, u1, T)) return;

  // ---------------------------------------------------------------- issue side
  Walker cw = wk0;
  int cj = wk0.jb;
  // table entry of the j-th block a walker's sequence reads (the logical
  // block, past the blocks a sliding window leaves out)
  auto table_id = [&](const Walker& wk_, int j) -> int32_t {
    const int jl = REMAP ? logical_block<BS>(a, seq_len_clipped(a, wk_.s), j) : j;
    return __ldg(a.block_tables + (size_t)wk_.s * a.table_stride + jl);
  };
  int32_t next_id = table_id(cw, cj);
  int issued = 0;

  auto issue_next = [&]() {
    if (cw.done) return;
    const int st = issued % NSW;
    {
      // every value here is the same on all lanes of the (converged) warp:
      // one elected lane starts the copies
      const int kvh = cw.unit / a.units_per_kv;
      uint8_t* dst = stages + (size_t)st * STAGE;
      uint64_t* bar = &bars[st];
      const bool valid = next_id >= 0 && next_id < a.num_blocks;
      if (elect_one()) {
        if (valid) {
          stage_ok[st] = 1;
          mbar_arrive_expect_tx(bar, STAGE);
          tma_load_tile<GE>(dst, &maps.k, kvh * BS, next_id, bar);
          tma_load_tile<GE>(dst + TILE, &maps.v, kvh * BS, next_id, bar);
        } else {
          raise_error(a.err, PKV_DEVERR_BAD_BLOCK_ID);
          stage_ok[st] = 0;
          mbar_arrive(bar);
        }
      }
      __syncwarp();
    }
    ++issued;
    if (++cj >= cw.je) {
      walker_next_piece<BS>(cw, a, u1);
      cj = cw.jb;
    }
    if (!cw.done) next_id = table_id(cw, cj);
  };

  auto issue_q = [&](const Walker& pw, int slot) {
    if constexpr (MQ) {
      // the group's heads of each of the unit's tokens: one contiguous run per token
      const MqRows mr = mq_rows(a, pw.s);
      const int kvh = pw.unit / a.units_per_kv, tok0 = (pw.unit % a.units_per_kv) * a.mq_tpu;
      const int nt = max(0, min(a.mq_tpu, mr.T - tok0));
      const uint32_t run = (uint32_t)(a.group * D * sizeof(QT));
      mbar_arrive_expect_tx(&qbars[slot], nt * run);
      for (int i = 0; i < nt; ++i)
        bulk_g2s(qbuf + (size_t)slot * G * D + (size_t)i * a.group * D,
                 reinterpret_cast<const QT*>(a.q) + ((size_t)(mr.q0 + tok0 + i) * a.num_q_heads + kvh * a.group) * D,
                 run, &qbars[slot]);
    } else {
      const QT* src = reinterpret_cast<const QT*>(a.q) + ((size_t)pw.s * a.num_q_heads + unit_first_head(a, pw, G)) * D;
      mbar_arrive_expect_tx(&qbars[slot], G * D * sizeof(QT));
      bulk_g2s(qbuf + (size_t)slot * G * D, src, G * D * sizeof(QT), &qbars[slot]);
    }
  };

  // cascade: the prefix partial of the G rows of a piece that starts a
  // segment (one buffer: the next piece's copy starts once this piece has
  // read its own)
  constexpr uint32_t kPreBytes = (uint32_t)(G * pre_row_floats(D) * sizeof(float));
  auto issue_pre = [&](const Walker& pw) {
    const float* src = a.pre + ((size_t)pw.s * a.num_q_heads + unit_first_head(a, pw, G)) * pre_row_floats(D);
    mbar_arrive_expect_tx(pbar, kPreBytes);
    bulk_g2s(pbuf, src, kPreBytes, pbar);
  };
  int pre_issued = 0, pre_waited = 0;

  // a dependent merge grid may start its own planning now; it waits for
  // this grid to finish before it reads a partial
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  Walker qlook = wk0;
  if (lane == 0) issue_q(wk0, 0);
  // Everything above reads only the step's inputs (lengths, tables, q).  When
  // this grid is the programmatic dependent of the cache write (or of a
  // cascade's prefix pass), the K/V tiles and the prefix partials must wait
  // for that grid; on an ordinary launch this returns at once.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if constexpr (REMAP) {
    if (a.pre && wk0.jb == 0) {
      if (lane == 0) issue_pre(wk0);
      ++pre_issued;
    }
  }
#pragma unroll 1
  for (int i = 0; i < NSW; ++i) issue_next();

  // Per-lane fragment addresses.  A lane reads 16-byte chunk C + h of token
  // row `row`, C a compile-time multiple of the lane part h's range, so the
  // swizzled offset is (lane base) XOR ((C % CPB) << 4) plus the box of C:
  // only the base is kept in a register.
  //  q.K, bf16, 16-token steps: rows (0-7 | 8-15) x chunks (2kk | 2kk+1);
  //  q.K, bf16, 8-token steps: rows 0-7 x chunks 4kq..4kq+3;
  //  q.K, fp8: rows (0-7 | 8-15) x chunks (2kq | 2kq+1), a chunk = 16 dims;
  //  P.V, bf16 (ldmatrix.trans): rows (0-7 | 8-15) x chunks (2j | 2j+1), or
  //  rows 0-7 x chunks 4j..4j+3 for 8-token steps;
  //  P.V, fp8: rows 2t, 2t+1, 2t+8, 2t+9 at this lane's VPL bytes.
  auto lane_base = [](int row, int h) -> uint32_t { return swz<GE>(row, h); };
  uint32_t kx, vx = 0;
  if constexpr (F8) {
    kx = lane_base((lane & 7) + 8 * ((lane >> 3) & 1), lane >> 4);
  } else if constexpr (TB == 16) {
    kx = lane_base((lane & 7) + 8 * (lane >> 4), (lane >> 3) & 1);
    vx = lane_base((lane & 7) + 8 * ((lane >> 3) & 1), lane >> 4);
  } else {
    kx = lane_base(lane & 7, lane >> 3);
    vx = lane_base(lane & 7, lane >> 3);
  }
  // head dim of accumulator o[n][e]
  auto odim = [&](int n, int e) -> int { return F8 ? GE::VPL * (2 * t + e) + n : 8 * n + 2 * t + e; };
  constexpr int CPB = GE::IB / 16;  // chunks per box row
  // address of chunk C (+ the lane part) relative to a 1024-byte aligned tile base
  auto frag = [](uint32_t base, int C) -> uint32_t {
    return (base ^ (uint32_t)((C % CPB) << 4)) + (uint32_t)((C / CPB) * GE::BOX);
  };
  uint32_t voff8[4] = {0, 0, 0, 0};
  if constexpr (F8) {
    const int c = (g * GE::VPL) / 16, b = (g * GE::VPL) % 16;
    voff8[0] = swz<GE>(2 * t, c) + b;
    voff8[1] = swz<GE>(2 * t + 1, c) + b;
    voff8[2] = swz<GE>(2 * t + 8, c) + b;
    voff8[3] = swz<GE>(2 * t + 9, c) + b;
  }

  // q.K of one k-step into one n-tile's score entries of this lane's rows
  auto qk_mma = [](float (&c)[RE], const uint32_t (&qk)[RE], uint32_t b0, uint32_t b1) {
    if constexpr (R16) {
      mma_k16_rows16<F8>(c, qk[0], qk[1], qk[2], qk[3], b0, b1);
    } else {
      mma_k16<F8>(c[0], c[1], qk[0], qk[1], b0, b1);
    }
  };

  // ---------------------------------------------------------------- consume side
  Walker wk = wk0;
  int consumed = 0, waited = 0, piece = 0;
  CutPiece cut0{}, cut1{};  // this warp's cut pieces (its first and last at most)
  int ncut = 0;
  // a first cut piece that ends before the range does has its ticket drawn
  // one tile later (after tile `early_at` is consumed), so that this warp
  // merges at most the segment its range ends in
  int early_at = -1, pre0 = -1;
  bool drawn0 = false;
  bool alive = true;
  uint32_t qa[KS][RE];    // q.K A operand per k-step: (a0, a2) of row g, or (a0, a1, a2, a3)
                          // of rows g and g + 8 (16-row units)
  float o[NTO][4];        // accumulators, columns 2t, 2t+1 of each n-tile: [0..1] row g,
                          // [2..3] row g + 8 (16-row units) or the P-remainder part of row g
  float m_run[RPL], l_run[RPL];  // running max (log2 units) and this lane's share of the sum

#pragma unroll 1
  while (!wk.done) {
    const int qslot = piece & 1;
    {  // prefetch the next piece's q while this one runs
      Walker nx = qlook;
      walker_next_piece<BS>(nx, a, u1);
      if (!nx.done && lane == 0) {
        fence_proxy_async_smem();
        issue_q(nx, qslot ^ 1);
      }
      qlook = nx;
    }
    if (!mbar_wait_bounded(&qbars[qslot], (piece >> 1) & 1, a.err)) alive = false;
    float qk_mul = a.qk_scale;
    // this lane's rows g (+ 8): valid, and (MQ) the positions each attends (below row_lim)
    bool row_ok[RPL];
    int row_lim[RPL];
    MqRows mr{0, 0};
    if constexpr (MQ) mr = mq_rows(a, wk.s);
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
      row_ok[i] = g + 8 * i < G;
      row_lim[i] = 0x7FFFFFFF;
      if constexpr (MQ) {
        const int tok = (wk.unit % a.units_per_kv) * a.mq_tpu + (g + 8 * i) / a.group;
        row_ok[i] = row_ok[i] && tok < mr.T;
        row_lim[i] = seq_len_clipped(a, wk.s) - mr.T + tok + 1;
      }
    }
    {
      // operand slot of row i's k pair h (h = 0: k 2t.., h = 1: k 2t + 8..)
      auto qslot_of = [](int i, int h) { return R16 ? 2 * h + i : h; };
      if constexpr (!F8) {
#pragma unroll
        for (int i = 0; i < RPL; ++i) {
          const QT* qs = qbuf + (size_t)qslot * G * D + (size_t)(row_ok[i] ? g + 8 * i : 0) * D;
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            qa[kk][qslot_of(i, 0)] = row_ok[i] ? *reinterpret_cast<const uint32_t*>(qs + 16 * kk + 2 * t) : 0u;
            qa[kk][qslot_of(i, 1)] = row_ok[i] ? *reinterpret_cast<const uint32_t*>(qs + 16 * kk + 2 * t + 8) : 0u;
          }
        }
      } else {
        // k-step kk holds dims 16kk + 4t + (0, 1) in the first pair and
        // + (2, 3) in the second, the order in which a K chunk reaches the
        // lane through ldmatrix
        float qv[RPL][KS][4];
        float mq = 0.f;
#pragma unroll
        for (int i = 0; i < RPL; ++i) {
          const QT* qs = qbuf + (size_t)qslot * G * D + (size_t)(row_ok[i] ? g + 8 * i : 0) * D;
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            const uint2 raw = *reinterpret_cast<const uint2*>(qs + 16 * kk + 4 * t);
            const float2 lo = bf16x2_to_f2(raw.x), hi = bf16x2_to_f2(raw.y);
            qv[i][kk][0] = row_ok[i] ? lo.x : 0.f;
            qv[i][kk][1] = row_ok[i] ? lo.y : 0.f;
            qv[i][kk][2] = row_ok[i] ? hi.x : 0.f;
            qv[i][kk][3] = row_ok[i] ? hi.y : 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) mq = fmaxf(mq, fabsf(qv[i][kk][e]));
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, off));
        // fp16 tops out at 65504: scale q by 2^-sh so that |q| < 2^15
        int e = 0;
        frexpf(mq, &e);
        const int sh = e > 15 ? (e - 15 < 100 ? e - 15 : 100) : 0;
        const float down = ldexpf(1.f, -sh);
        qk_mul = a.qk_scale * ldexpf(1.f, sh);
#pragma unroll
        for (int i = 0; i < RPL; ++i)
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            qa[kk][qslot_of(i, 0)] = pack_f16x2(qv[i][kk][0] * down, qv[i][kk][1] * down);
            qa[kk][qslot_of(i, 1)] = pack_f16x2(qv[i][kk][2] * down, qv[i][kk][3] * down);
          }
      }
    }
#pragma unroll
    for (int n = 0; n < NTO; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
      m_run[i] = -CUDART_INF_F;
      l_run[i] = 0.f;
    }
    if constexpr (REMAP) {
      if (a.pre && wk.jb == 0) {
        // cascade: a segment's online softmax starts from the shared prefix's
        // partial (o relative to m, l), so no later merge step sees the prefix
        if (alive && !mbar_wait_bounded(pbar, pre_waited & 1, a.err)) alive = false;
        ++pre_waited;
        if (g < G) {
          const float* pr = pbuf + (size_t)g * pre_row_floats(D);
#pragma unroll
          for (int n = 0; n < NTO; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) o[n][e] = pr[odim(n, e)];
          m_run[0] = pr[D];
          l_run[0] = t == 0 ? pr[D + 1] : 0.f;
        }
      }
      if (a.pre && !qlook.done && qlook.jb == 0) {  // the next piece starts a segment
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) issue_pre(qlook);
        ++pre_issued;
      }
    }
    const int L = seq_len_clipped(a, wk.s);

#pragma unroll 1
    for (int j = wk.jb; j < wk.je; ++j) {
      const int st = consumed % NSW;
      bool ok = false;
      if (alive && consumed < issued) {
        ok = mbar_wait_bounded(&bars[st], (consumed / NSW) & 1, a.err);
        waited = consumed + 1;
        if (!ok) alive = false;
      }
      ok = ok && stage_ok[st];
      TileMask tm = tile_mask<BS, REMAP>(a, L, REMAP ? logical_block<BS>(a, L, j) : j);
      if (!ok) tm.clear();  // a skipped tile: nothing is kept

#pragma unroll
      for (int step = 0; step < GE::STEPS; ++step) {
        const uint32_t kt = stages_s + (uint32_t)(st * STAGE + step * TB * GE::IB);
        const uint32_t vt = kt + TILE;
        const int t0 = step * TB;  // first token of this step within the tile

        // ---- scores: s[n][2i + e] = q_(g + 8i) . K[8n + 2t + e]
        float s[GE::NTS][RE];
        if constexpr (TB == 16) {
          float s2[2][2][RE] = {};  // even / odd k-steps, two independent chains
          if constexpr (F8) {
#pragma unroll
            for (int kq = 0; kq < KS / 2; ++kq) {
              uint32_t r[4];
              ldsm_x4(frag(kt + kx, 2 * kq), r);
              uint32_t b[4][2];
#pragma unroll
              for (int m = 0; m < 4; ++m) e4m3x4_to_f16x2x2(r[m], b[m][0], b[m][1]);
              // r[0]: rows 0-7, k-step 2kq; r[1]: rows 8-15, 2kq; r[2], r[3]: k-step 2kq + 1
              qk_mma(s2[0][0], qa[2 * kq], b[0][0], b[0][1]);
              qk_mma(s2[0][1], qa[2 * kq], b[1][0], b[1][1]);
              qk_mma(s2[1][0], qa[2 * kq + 1], b[2][0], b[2][1]);
              qk_mma(s2[1][1], qa[2 * kq + 1], b[3][0], b[3][1]);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
              uint32_t r[4];
              ldsm_x4(frag(kt + kx, 2 * kk), r);
              // r[0], r[1]: rows 0-7 (b0, b1); r[2], r[3]: rows 8-15
              qk_mma(s2[kk & 1][0], qa[kk], r[0], r[1]);
              qk_mma(s2[kk & 1][1], qa[kk], r[2], r[3]);
            }
          }
#pragma unroll
          for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < RE; ++e) s[n][e] = s2[0][n][e] + s2[1][n][e];
        } else {
          float s2[2][RE] = {};
#pragma unroll
          for (int kq = 0; kq < KS / 2; ++kq) {
            uint32_t r[4];
            ldsm_x4(frag(kt + kx, 4 * kq), r);
            // rows 0-7; r[0], r[1]: k-step 2kq; r[2], r[3]: k-step 2kq + 1
            qk_mma(s2[0], qa[2 * kq], r[0], r[1]);
            qk_mma(s2[1], qa[2 * kq + 1], r[2], r[3]);
          }
#pragma unroll
          for (int e = 0; e < RE; ++e) s[0][e] = s2[0][e] + s2[1][e];
        }

        // ---- online softmax of rows g (+ 8) (log2 units)
        float mx[RPL];
        bool grow = false;
#pragma unroll
        for (int i = 0; i < RPL; ++i) {
          const int rl = MQ ? row_lim[i] - j * BS : BS;  // (MQ) the row's positions kept in the tile
          mx[i] = -CUDART_INF_F;
#pragma unroll
          for (int n = 0; n < GE::NTS; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int tok = 8 * n + 2 * t + e;
              float& v = s[n][2 * i + e];
              v = tm.keep(t0 + tok) && (!MQ || t0 + tok < rl) ? v * qk_mul : -CUDART_INF_F;
              mx[i] = fmaxf(mx[i], v);
            }
          mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
          mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
          grow = grow || mx[i] > m_run[i];
        }
        if (__any_sync(0xffffffffu, grow)) {
          float alpha[RPL];
#pragma unroll
          for (int i = 0; i < RPL; ++i) {
            const float m_new = fmaxf(m_run[i], mx[i]);
            alpha[i] = m_new > m_run[i] ? fast_exp2(m_run[i] - m_new) : 1.f;
            l_run[i] *= alpha[i];
            m_run[i] = m_new;
          }
          // o[n][2..3] belong to row g + 8 (16-row units) or to row g's P remainder
          const float2 a0 = make_float2(alpha[0], alpha[0]), a1 = make_float2(alpha[RPL - 1], alpha[RPL - 1]);
#pragma unroll
          for (int n = 0; n < NTO; ++n) {
            const float2 v = __fmul2_rn(make_float2(o[n][0], o[n][1]), a0);
            const float2 u = __fmul2_rn(make_float2(o[n][2], o[n][3]), a1);
            o[n][0] = v.x;
            o[n][1] = v.y;
            o[n][2] = u.x;
            o[n][3] = u.y;
          }
        }
        float p[GE::NTS][RE];
#pragma unroll
        for (int i = 0; i < RPL; ++i) {
          const float m_use = m_run[i] == -CUDART_INF_F ? 0.f : m_run[i];
#pragma unroll
          for (int n = 0; n < GE::NTS; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              p[n][2 * i + e] = fast_exp2(s[n][2 * i + e] - m_use);
              l_run[i] += p[n][2 * i + e];
            }
        }

        // ---- P . V
        const bool full = tm.all(t0, t0 + TB);
        if constexpr (F8) {
          // A rows 0-7 / 8-15: P of rows g / g + 8 (16-row units), or row g's
          // P as head + remainder, all fp16
          uint32_t ph[2], pl[2];
#pragma unroll
          for (int n = 0; n < 2; ++n) {
            ph[n] = pack_f16x2(p[n][0], p[n][1]);
            if constexpr (R16) {
              pl[n] = pack_f16x2(p[n][RE - 2], p[n][RE - 1]);
            } else {
              const float2 h = f16x2_to_f2(ph[n]);
              pl[n] = pack_f16x2(p[n][0] - h.x, p[n][1] - h.y);
            }
          }
          static_assert(GE::VPL == 16 || GE::VPL == 8, "fp8 V slice");
          uint32_t X[4][GE::VPL / 4];  // rows 2t, 2t+1, 2t+8, 2t+9
#pragma unroll
          for (int ri = 0; ri < 4; ++ri) {
            const uint8_t* src = stages + (vt - stages_s) + voff8[ri];
            if constexpr (GE::VPL == 16) {
              const uint4 v = *reinterpret_cast<const uint4*>(src);
              X[ri][0] = v.x; X[ri][1] = v.y; X[ri][2] = v.z; X[ri][3] = v.w;
            } else {
              const uint2 v = *reinterpret_cast<const uint2*>(src);
              X[ri][0] = v.x; X[ri][1] = v.y;
            }
          }
          if (!full) {  // rows not attended may hold NaN codes: their weight is 0, drop them too
            const int rows[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
            for (int ri = 0; ri < 4; ++ri)
#pragma unroll
              for (int q = 0; q < GE::VPL / 4; ++q) X[ri][q] = tm.keep(t0 + rows[ri]) ? X[ri][q] : 0u;
          }
#pragma unroll
          for (int q = 0; q < GE::VPL / 4; ++q) {
            // byte k of the lane's slice is n-tile k: pair the two rows of each
            // B register byte by byte, then widen
            uint32_t b0[4], b1[4];
            e4m3x4_to_f16x2x2(__byte_perm(X[0][q], X[1][q], 0x5140), b0[0], b0[1]);
            e4m3x4_to_f16x2x2(__byte_perm(X[0][q], X[1][q], 0x7362), b0[2], b0[3]);
            e4m3x4_to_f16x2x2(__byte_perm(X[2][q], X[3][q], 0x5140), b1[0], b1[1]);
            e4m3x4_to_f16x2x2(__byte_perm(X[2][q], X[3][q], 0x7362), b1[2], b1[3]);
#pragma unroll
            for (int k = 0; k < 4; ++k) mma_k16_rows16<true>(o[4 * q + k], ph[0], pl[0], ph[1], pl[1], b0[k], b1[k]);
          }
        } else {
          // A rows 0-7 / 8-15: P of rows g / g + 8 (16-row units), or row g's
          // P as head + remainder, all bf16
          uint32_t ph[GE::NTS], pl[GE::NTS];
#pragma unroll
          for (int n = 0; n < GE::NTS; ++n) {
            ph[n] = pack_bf16x2(p[n][0], p[n][1]);
            if constexpr (R16) {
              pl[n] = pack_bf16x2(p[n][RE - 2], p[n][RE - 1]);
            } else {
              const float2 h = bf16x2_to_f2(ph[n]);
              pl[n] = pack_bf16x2(p[n][0] - h.x, p[n][1] - h.y);
            }
          }
          // keep-masks of this lane's token pairs (2t, 2t+1) and (2t+8, 2t+9)
          uint32_t keep0 = 0xFFFFFFFFu, keep1 = 0xFFFFFFFFu;
          if (!full) {
            keep0 = (tm.keep(t0 + 2 * t) ? 0x0000FFFFu : 0u) | (tm.keep(t0 + 2 * t + 1) ? 0xFFFF0000u : 0u);
            keep1 = (tm.keep(t0 + 2 * t + 8) ? 0x0000FFFFu : 0u) | (tm.keep(t0 + 2 * t + 9) ? 0xFFFF0000u : 0u);
          }
          if constexpr (TB == 16) {
#pragma unroll
            for (int jv = 0; jv < NTO / 2; ++jv) {
              uint32_t r[4];
              ldsm_x4_t(frag(vt + vx, 2 * jv), r);
              // r[0], r[1]: n-tile 2jv (tokens 2t.. | 2t+8..); r[2], r[3]: n-tile 2jv + 1
              r[0] &= keep0; r[1] &= keep1; r[2] &= keep0; r[3] &= keep1;
              mma_k16_rows16<false>(o[2 * jv], ph[0], pl[0], ph[1], pl[1], r[0], r[1]);
              mma_k16_rows16<false>(o[2 * jv + 1], ph[0], pl[0], ph[1], pl[1], r[2], r[3]);
            }
          } else {
#pragma unroll
            for (int jv = 0; jv < NTO / 4; ++jv) {
              uint32_t r[4];
              ldsm_x4_t(frag(vt + vx, 4 * jv), r);
              // r[m]: n-tile 4jv + m, tokens 2t, 2t+1
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                r[m] &= keep0;
                mma_k8_bf16_rows16(o[4 * jv + m], ph[0], pl[0], r[m]);
              }
            }
          }
        }
      }
      __syncwarp();  // every lane is done with this stage before it is refilled
      ++consumed;
      if (alive) issue_next();
      if constexpr (BALANCED) {
        if (consumed == early_at) {
          pre0 = draw_ticket(a, cut0, lane, SM::kMergeCap > 0);
          drawn0 = true;
        }
      }
    }

    // ------------------------------------------------------------ piece end
    // row g + 8i's accumulator: o[n][2i + e]; with one row per lane the P
    // remainder's half is added to the head's
    if constexpr (!R16) {
#pragma unroll
      for (int n = 0; n < NTO; ++n) {
        o[n][0] += o[n][2];
        o[n][1] += o[n][3];
      }
    }
    float l_row[RPL];
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
      l_row[i] = l_run[i] + __shfl_xor_sync(0xffffffffu, l_run[i], 1);
      l_row[i] += __shfl_xor_sync(0xffffffffu, l_row[i], 2);
    }
    const int qh0 = unit_first_head(a, wk, G);
    const bool whole = (wk.jb == 0 && wk.je == wk.nb);

    if constexpr (!BALANCED) {
      if (g < G) {
        const int p = (int)(gw % a.max_partitions);
        const size_t row = ((size_t)wk.s * a.num_q_heads + qh0 + g) * a.max_partitions + p;
        const float inv = l_row[0] > 0.f ? a.out_scale / l_row[0] : 0.f;
        float* dst = a.o_part + row * D;
#pragma unroll
        for (int n = 0; n < NTO; ++n)
#pragma unroll
          for (int e = 0; e < 2; ++e) dst[odim(n, e)] = o[n][e] * inv;
        if (t == 0) {
          a.m_part[row] = m_run[0] * 0.69314718055994531f;
          a.l_part[row] = l_row[0];
        }
      }
    } else if (whole) {
#pragma unroll
      for (int i = 0; i < RPL; ++i) {
        if (!row_ok[i]) continue;
        const int r = g + 8 * i;
        QT* dst = reinterpret_cast<QT*>(a.out) +
                  (MQ ? ((size_t)(mr.q0 + (wk.unit % a.units_per_kv) * a.mq_tpu + r / a.group) * a.num_q_heads +
                         (wk.unit / a.units_per_kv) * a.group + r % a.group) * D
                      : ((size_t)wk.s * a.num_q_heads + qh0 + r) * D);
        const float inv = l_row[i] > 0.f ? a.out_scale / l_row[i] : 0.f;
        if constexpr (F8) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            uint32_t pk[NTO / 2];
#pragma unroll
            for (int n = 0; n < NTO / 2; ++n)
              pk[n] = pack_bf16x2(o[2 * n][2 * i + e] * inv, o[2 * n + 1][2 * i + e] * inv);
#pragma unroll
            for (int n = 0; n < NTO / 2; n += 4)
              *reinterpret_cast<uint4*>(dst + odim(2 * n, e)) = make_uint4(pk[n], pk[n + 1], pk[n + 2], pk[n + 3]);
          }
        } else {
#pragma unroll
          for (int n = 0; n < NTO; ++n)
            *reinterpret_cast<uint32_t*>(dst + odim(n, 0)) =
                pack_bf16x2(o[n][2 * i] * inv, o[n][2 * i + 1] * inv);
        }
      }
    } else {
      // segment cut between warps: publish (acc, m, l) now
      float* pslot = partial_slot<G, D>(a, wk, gw, u0);
#pragma unroll
      for (int i = 0; i < RPL; ++i) {
        const int r = g + 8 * i;
        if (r < G) {
#pragma unroll
          for (int n = 0; n < NTO; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) pslot[r * D + odim(n, e)] = o[n][2 * i + e];
          if (t == 0) {
            pslot[G * D + r] = m_run[i];
            pslot[G * D + G + r] = l_row[i];
          }
        }
      }
      // the ticket is taken when this warp's whole range is done
      if (ncut == 0) {
        cut0 = cut_piece_of(wk, mr.q0, mr.T);
        if (wk.seg_u + wk.je < u1 && !a.defer_merge) early_at = consumed + 1;
      } else {
        cut1 = cut_piece_of(wk, mr.q0, mr.T);
      }
      ++ncut;
    }
    ++piece;
    walker_next_piece<BS>(wk, a, u1);
  }

  // Leave no copy in flight: wait (bounded) for every stage this warp filled
  // but did not wait for (only possible after a timeout).
  for (int k = waited; k < issued; ++k) mbar_wait_bounded(&bars[k % NSW], (k / NSW) & 1, a.err);
  for (int k = pre_waited; k < pre_issued; ++k) mbar_wait_bounded(pbar, k & 1, a.err);

  if (BALANCED && !a.defer_merge) {
    // the merges stage partial slots in the stage ring and q buffers, free
    // now (no copy is in flight there unless a wait timed out: then this
    // warp merges nothing, its error already raised)
    MergeStage ms;
    if (SM::kMergeCap > 0 && alive) {
      ms.buf = reinterpret_cast<float*>(smem + SM::kStages);
      ms.cap = SM::kMergeCap;
      ms.bar = mbar;
    }
    finish_cut_pieces<QT, G, D>(a, cut0, cut1, ncut, T, NW, lane, SM::kMergeCap > 0 ? &ms : nullptr, drawn0,
                                pre0);
  }
}

// ----------------------------------------------------------------------------
// Deferred merges.  CTA gw of this grid replays the plan of warp gw of a
// balanced decode grid of NW warps that ran with defer_merge: when that
// warp's range starts inside a segment begun by earlier warps and the
// segment ends within the range, the warp held the segment's last piece, and
// this CTA merges the segment's pieces (accumulators, maxima and sums from
// their partial slots) into its output rows.  Each cut segment has one such
// CTA.  The planning runs while the decode grid is still streaming; the
// merge waits for that grid (programmatic dependent launch).
// ----------------------------------------------------------------------------
// Geometry of a merge: segments of 8 or more rows are merged by G / 4 warps,
// four rows each (a 16-row merge by one warp spent 4-9 us combining and
// writing its rows one after the other); smaller ones by one warp.  Each
// warp stages MC pieces of its rows.
template <int G, int D, int MC>
struct MergeGeo {
  static constexpr int kWarps = G >= 8 ? G / 4 : 1;
  static constexpr int kRows = G / kWarps;  // rows per warp
  static constexpr int kPiece = kWarps > 1 ? kRows * D + 2 * kRows : partial_slot_floats(G, D);  // floats
  static constexpr size_t kSmem = (size_t)kWarps * MC * kPiece * sizeof(float) + (size_t)kWarps * 8;
};

template <class QT, int G, int D, int BS, int MC>
__global__ void __launch_bounds__(32 * MergeGeo<G, D, MC>::kWarps)
    merge_cut_kernel(const __grid_constant__ DecodeArgs a, int64_t NW) {
  using MG = MergeGeo<G, D, MC>;
  extern __shared__ __align__(16) uint8_t merge_smem[];
  const int lane = threadIdx.x & 31, mw = threadIdx.x >> 5;
  const int64_t gw = blockIdx.x;
  float* buf = reinterpret_cast<float*>(merge_smem) + (size_t)mw * MC * MG::kPiece;
  uint64_t* bar = reinterpret_cast<uint64_t*>(merge_smem + (size_t)MG::kWarps * MC * MG::kPiece * sizeof(float)) + mw;
  int64_t u0 = 0, u1 = 0, T = 0;
  Walker wk0;
  const bool mine = plan_warp<QT, D, BS, true, false>(a, gw, NW, lane, wk0, u0, u1, T) && wk0.jb > 0 &&
                    wk0.seg_u + wk0.nb <= u1;
  if (!mine) return;
  MqRows mr{0, 0};
  if (a.q_start) mr = mq_rows(a, wk0.s);
  if (lane == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if constexpr (MG::kWarps > 1) {
    merge_rows_staged<QT, G, D, MG::kRows>(a, cut_piece_of(wk0, mr.q0, mr.T), T, NW, lane, buf, MC, bar,
                                           mw * MG::kRows);
  } else {
    MergeStage ms;
    ms.buf = buf;
    ms.cap = MC;
    ms.bar = bar;
    merge_segment_staged<QT, G, D>(a, cut_piece_of(wk0, mr.q0, mr.T), T, NW, lane, ms);
  }
}

}  // namespace pkv
