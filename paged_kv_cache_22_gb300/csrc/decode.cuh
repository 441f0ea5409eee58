// decode.cuh -- paged decode attention on the CUDA cores (fp32 caches).
//
// Computes what decode_common.cuh states, with every product and sum in
// fp32: the path for fp32 caches, whose results are held to fp32 accuracy.
// bf16 and fp8 caches take the tensor-core kernel of decode_tc.cuh.
//
// Design (GB300):
//  * Work unit = one (block, kv head) tile of K and one of V, each BS * D
//    contiguous elements in the [num_blocks, Hkv, BS, D] cache, fetched whole
//    by one 1-D bulk copy (TMA) into shared memory.  Every tile is read from
//    HBM exactly once and serves all G query heads of its kv head.
//  * Every warp is an independent worker: its own ring of NSW shared-memory
//    stages with their mbarriers, its own double-buffered query, its own
//    online-softmax state.  It consumes stage k and refills it with its tile
//    k + NSW; the block id of the next tile is loaded one tile ahead.  After
//    the one barrier that publishes the mbarrier inits, warps never wait for
//    each other.
//  * Inside a tile: C lanes share a token row, each holding DL = D / C head
//    dims of all G queries in registers; R = 32 / C rows run in parallel.  The
//    partial dot products are finished by recursive halving over the C lanes,
//    after which each lane owns distinct (head, token) scores; the running max
//    is warp-uniform per head, so accumulator rescales are uniform branches.
//    Probabilities go through a small shared buffer to the P.V layout, where
//    each lane owns DV = 4 dims of every token and accumulates token pairs
//    with packed fp32 FMA.
//  * Balanced split: the tiles of all (sequence, kv-head unit) segments are
//    laid end to end and cut into one equal range per warp of the grid, so
//    every SM streams the same bytes whatever the length skew.  A segment cut
//    between warps is merged by the last warp to finish a piece of it (atomic
//    ticket, no waiting): unnormalised partials (acc, m, l) go through the
//    workspace and are combined by log-sum-exp.  Fixed-partition mode gives
//    each warp one partition of one segment and leaves the merge to the
//    reduce kernel.
#pragma once

#include "decode_common.cuh"

namespace pkv {

// Compile-time geometry of one kernel instance.
template <class CT, int D, int BS, int G>
struct Geo {
  static constexpr int E = CT::kBytes;
  static constexpr int TB = BS < 16 ? BS : 16;      // tokens per compute step
  static constexpr int DL0 = 64 / G;                 // keep G * DL = 64 query registers
  static constexpr int DLMAX = D * TB / 32;          // at least one token row per lane
  static constexpr int DL = DL0 < DLMAX ? DL0 : DLMAX;
  static constexpr int C = D / DL;                   // lanes per token row
  static constexpr int R = 32 / C;                   // token rows in flight per warp
  static constexpr int TL = TB / R;                  // tokens per lane per step
  static constexpr int VB = DL * E >= 16 ? 16 : DL * E;  // bytes per shared-memory vector
  static constexpr int VE = VB / E;                  // elements per vector
  static constexpr int NV = DL / VE;                 // vectors per token row per lane
  static constexpr int PV = VE / 2;                  // fp32 pairs per vector
  static constexpr int NP = DL / 2;                  // fp32 pairs per lane
  static constexpr int TILE = BS * D * E;            // bytes of one (block, head) tile
  static constexpr int STEPS = BS / TB;
  // score reduction: N0 partial scores per lane, halved NT times over the C lanes
  static constexpr int N0 = TL * G;
  static constexpr int LC = C == 1 ? 0 : C == 2 ? 1 : C == 4 ? 2 : C == 8 ? 3 : C == 16 ? 4 : 5;
  static constexpr int LN = N0 == 1 ? 0 : N0 == 2 ? 1 : N0 == 4 ? 2 : N0 == 8 ? 3 : N0 == 16 ? 4 : N0 == 32 ? 5 : N0 == 64 ? 6 : 7;
  static constexpr int NT = LC < LN ? LC : LN;
  static constexpr int NF = N0 >> NT;                   // scores owned per lane
  static constexpr int DUP = NT < LC ? (C >> NT) : 1;   // lanes holding the same score
  // P.V: each lane owns DV consecutive dims; SL dim slices, TG token groups
  static constexpr int DV = 4;
  static constexpr int SL = D / DV;
  static constexpr int TG = 32 / SL;
  static constexpr int PPL = (TB / 2) / TG;            // token pairs per lane per step
  static constexpr int NSW0 = 16384 / (2 * TILE);
  static constexpr int NSW = NSW0 < 2 ? 2 : (NSW0 > 8 ? 8 : NSW0);  // stages per warp
  static constexpr int SLOT = partial_slot_floats(G, D);  // floats of one partial result
  static_assert(D % DL == 0 && 32 % C == 0 && R <= TB && TB % R == 0, "lane layout");
  static_assert(DL % VE == 0 && VE % 2 == 0, "vector layout");
  static_assert(TILE % 16 == 0, "bulk copies move multiples of 16 bytes");
  static_assert(SL <= 32 && 32 % SL == 0 && (TB / 2) % TG == 0 && PPL >= 1, "P.V layout");
  static_assert(C >= G && NF <= TL, "each lane owns scores of one head");
};

// Shared memory: per-warp regions, laid out type by type.
template <class CT, int D, int BS, int G, int W>
struct Smem {
  using GE = Geo<CT, D, BS, G>;
  using QT = typename CT::QType;
  static constexpr int kStageBytes = 2 * GE::TILE;  // K tile then V tile
  static constexpr size_t kStages = 0;
  static constexpr size_t kQBuf = kStages + (size_t)W * GE::NSW * kStageBytes;
  static constexpr size_t kP = kQBuf + (size_t)W * 2 * G * D * sizeof(QT);
  static constexpr size_t kBars = (kP + (size_t)W * G * GE::TB * 4 + 7) / 8 * 8;
  static constexpr size_t kQBars = kBars + (size_t)W * GE::NSW * 8;
  static constexpr size_t kOk = kQBars + (size_t)W * 2 * 8;
  static constexpr size_t kBytes = kOk + (size_t)W * GE::NSW * 4;
};

// ----------------------------------------------------------------------------
// The kernel.
// ----------------------------------------------------------------------------
template <class CT, int D, int BS, int G, int W, bool BALANCED, bool REMAP>
__global__ void __launch_bounds__(W * 32, (G >= 8 ? 8 : 12) / W)
    decode_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ TmaMaps) {
  using GE = Geo<CT, D, BS, G>;
  using SM = Smem<CT, D, BS, G, W>;
  using QT = typename CT::QType;
  constexpr int NSW = GE::NSW, C = GE::C, R = GE::R, TL = GE::TL, NV = GE::NV, PV = GE::PV,
                NP = GE::NP, VE = GE::VE, VB = GE::VB, TB = GE::TB, TILE = GE::TILE, DV = GE::DV,
                SL = GE::SL;
  constexpr int E = GE::E;

  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int r = lane / C, c = lane % C;
  uint8_t* stages = smem + SM::kStages + (size_t)w * NSW * SM::kStageBytes;
  QT* qbuf = reinterpret_cast<QT*>(smem + SM::kQBuf) + (size_t)w * 2 * G * D;
  float* ps = reinterpret_cast<float*>(smem + SM::kP) + (size_t)w * G * TB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kBars) + w * NSW;
  uint64_t* qbars = reinterpret_cast<uint64_t*>(smem + SM::kQBars) + w * 2;
  int* stage_ok = reinterpret_cast<int*>(smem + SM::kOk) + w * NSW;

  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < NSW; ++i) mbar_init(&bars[i], 1);
    mbar_init(&qbars[0], 1);
    mbar_init(&qbars[1], 1);
    fence_mbar_init();
  }
  __syncthreads();  // the only block-wide barrier: warps are independent from here on

  const int64_t gw = (int64_t)blockIdx.x * W + w;  // this warp's index in the grid
  const int64_t NW = (int64_t)gridDim.x * W;
  int64_t u0 = 0, u1 = 0, T = 0;
  Walker wk0;
  if (!plan_warp<QT, D, BS, BALANCED>(a, gw, NW, lane, wk0, u0, u1, T)) return;

  const size_t head_stride = (size_t)BS * D * E;  // one kv head's tile
  const size_t block_stride = (size_t)a.num_kv_heads * head_stride;

  // ---------------------------------------------------------------- issue side
  Walker cw = wk0;  // issue cursor: segment of the next tile to fetch
  int cj = wk0.jb;  // its block index
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
    if (lane == 0) {
      const int kvh = cw.unit / a.units_per_kv;
      uint8_t* dst = stages + (size_t)st * SM::kStageBytes;
      uint64_t* bar = &bars[st];
      if (next_id >= 0 && next_id < a.num_blocks) {
        stage_ok[st] = 1;
        const size_t off = (size_t)next_id * block_stride + (size_t)kvh * head_stride;
        mbar_arrive_expect_tx(bar, 2 * TILE);
        bulk_g2s(dst, a.k_cache + off, TILE, bar);
        bulk_g2s(dst + TILE, a.v_cache + off, TILE, bar);
      } else {
        raise_error(a.err, PKV_DEVERR_BAD_BLOCK_ID);
        stage_ok[st] = 0;
        mbar_arrive(bar);
      }
    }
    ++issued;
    if (++cj >= cw.je) {
      walker_next_piece<BS>(cw, a, u1);
      cj = cw.jb;
    }
    // one tile ahead: the id is needed only at the next issue
    if (!cw.done) next_id = table_id(cw, cj);
  };

  // q of the piece a walker stands on: bulk copy into this warp's q slot
  auto issue_q = [&](const Walker& pw, int slot) {
    const int kvh = pw.unit / a.units_per_kv, chunk = pw.unit % a.units_per_kv;
    const int qh0 = kvh * a.group + chunk * G;
    const QT* src = reinterpret_cast<const QT*>(a.q) + ((size_t)pw.s * a.num_q_heads + qh0) * D;
    mbar_arrive_expect_tx(&qbars[slot], G * D * sizeof(QT));
    bulk_g2s(qbuf + (size_t)slot * G * D, src, G * D * sizeof(QT), &qbars[slot]);
  };

  Walker qlook = wk0;  // look-ahead for the q prefetch
  if (lane == 0) issue_q(wk0, 0);
  // Everything above reads only the step's inputs (lengths, tables, q).  When
  // this grid is the programmatic dependent of the cache write, the K/V tiles
  // must wait for that grid; on an ordinary launch this returns at once.
  asm volatile("griddepcontrol.wait;" ::: "memory");
#pragma unroll 1
  for (int i = 0; i < NSW; ++i) issue_next();

  // ---------------------------------------------------------------- consume side
  Walker wk = wk0;
  int consumed = 0, waited = 0, piece = 0;
  CutPiece cut0{}, cut1{};  // this warp's cut pieces (its first and last at most)
  int ncut = 0;
  bool alive = true;
  float2 q2[G][NP];          // this lane's query dims, pre-scaled by scale*log2(e)
  float2 acc[G][DV];         // P.V accumulators: this lane's DV dims, even/odd token halves
  float m_run[G];            // running max per head (log2 units), warp-uniform
  float m_own, l_own;        // the owned head's running max and this lane's share of its sum
  const int h_own = c / (C / G);              // head of the scores this lane owns
  const bool l_counts = (c % GE::DUP) == 0;   // one copy of each duplicated score counts
  const int tg = lane / SL, d0 = (lane % SL) * DV;

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
    {
      const QT* qs = qbuf + (size_t)qslot * G * D;
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int j = 0; j < NV; ++j)
#pragma unroll
          for (int pv = 0; pv < PV; ++pv) {
            const int dim = (c + C * j) * VE + 2 * pv;
            q2[h][j * PV + pv] = make_float2(to_f32(qs[h * D + dim]) * a.qk_scale,
                                             to_f32(qs[h * D + dim + 1]) * a.qk_scale);
          }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m_run[h] = -CUDART_INF_F;
#pragma unroll
      for (int i = 0; i < DV; ++i) acc[h][i] = make_float2(0.f, 0.f);
    }
    m_own = -CUDART_INF_F;
    l_own = 0.f;
    const int L = seq_len_clipped(a, wk.s);

#pragma unroll 1
    for (int j = wk.jb; j < wk.je; ++j) {
      const int st = consumed % NSW;
      const uint8_t* ktile = stages + (size_t)st * SM::kStageBytes;
      const uint8_t* vtile = ktile + TILE;
      bool ok = false;
      if (alive && consumed < issued) {
        ok = mbar_wait_bounded(&bars[st], (consumed / NSW) & 1, a.err);
        waited = consumed + 1;
        if (!ok) alive = false;
      }
      ok = ok && stage_ok[st];
      TileMask tm = tile_mask<BS, REMAP>(a, L, REMAP ? logical_block<BS>(a, L, j) : j);
      if (!ok) tm.clear();  // a skipped tile: nothing is kept

#pragma unroll 1
      for (int step = 0; step < GE::STEPS; ++step) {
        const int tbase = step * TB;
        // ---- partial scores over this lane's DL dims: sc[h * TL + k], token r + R k
        float sc[GE::N0];
#pragma unroll
        for (int k = 0; k < TL; ++k) {
          const int t = tbase + r + R * k;
          float2 part[G];
#pragma unroll
          for (int h = 0; h < G; ++h) part[h] = make_float2(0.f, 0.f);
#pragma unroll
          for (int jv = 0; jv < NV; ++jv) {
            float2 kv[PV];
            VecLoad<CT, VB>::run(ktile + (size_t)t * D * E + (c + C * jv) * VB, kv);
#pragma unroll
            for (int pv = 0; pv < PV; ++pv)
#pragma unroll
              for (int h = 0; h < G; ++h) part[h] = ffma2(q2[h][jv * PV + pv], kv[pv], part[h]);
          }
#pragma unroll
          for (int h = 0; h < G; ++h) sc[h * TL + k] = part[h].x + part[h].y;
        }
        // ---- recursive halving over the C lanes of the row: each round a lane
        //      keeps half of its values (by its lane bit) and adds the partner's
        //      copy of that half; afterwards it owns NF complete scores.
#pragma unroll
        for (int i = 0; i < GE::NT; ++i) {
          const int msk = C >> (i + 1);
          const bool hi = (c & msk) != 0;
          const int half = GE::N0 >> (i + 1);
#pragma unroll
          for (int jj = 0; jj < (GE::N0 >> 1); ++jj) {
            if (jj < half) {
              const float lo_v = sc[jj], hi_v = sc[jj + half];
              const float send = hi ? lo_v : hi_v;
              const float keep = hi ? hi_v : lo_v;
              sc[jj] = keep + __shfl_xor_sync(0xffffffffu, send, msk);
            }
          }
        }
#pragma unroll
        for (int i = GE::NT; i < GE::LC; ++i) sc[0] += __shfl_xor_sync(0xffffffffu, sc[0], C >> (i + 1));
        // ---- owned scores: value v = vbase + jj -> head h_own, token r + R (v % TL)
        const int vbase = (c >> (GE::LC - GE::NT)) << (GE::LN - GE::NT);
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int jj = 0; jj < GE::NF; ++jj) {
          const int t = r + R * ((vbase + jj) % TL);
          if (!tm.keep(tbase + t)) sc[jj] = -CUDART_INF_F;
          mx = fmaxf(mx, sc[jj]);
        }
        // max over the lanes that own the same head, then every head's max to all
#pragma unroll
        for (int off = 1; off < C / G; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
#pragma unroll
        for (int off = C; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new_own = fmaxf(m_own, mx);
        const float m_use_own = (m_new_own == -CUDART_INF_F) ? 0.f : m_new_own;
        float lsum = 0.f;
#pragma unroll
        for (int jj = 0; jj < GE::NF; ++jj) {
          const float pj = fast_exp2(sc[jj] - m_use_own);
          lsum += pj;
          ps[h_own * TB + r + R * ((vbase + jj) % TL)] = pj;
        }
        l_own = l_own * fast_exp2(m_own - m_use_own) + (l_counts ? lsum : 0.f);
        m_own = m_new_own;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float m_new = fmaxf(m_run[h], __shfl_sync(0xffffffffu, mx, h * (C / G)));
          if (m_new > m_run[h]) {  // warp-uniform
            const float alpha = fast_exp2(m_run[h] - m_new);
            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
            for (int i = 0; i < DV; ++i) acc[h][i] = __fmul2_rn(acc[h][i], a2);
            m_run[h] = m_new;
          }
        }
        __syncwarp();
        // ---- P . V: lane owns DV dims for the token pairs of its group
        const bool full = tm.all(tbase, tbase + TB);
#pragma unroll
        for (int i = 0; i < GE::PPL; ++i) {
          const int t0 = 2 * (tg + GE::TG * i);  // first token of the pair, within the step
          float v0[DV], v1[DV];
          Vec4Load<CT>::run(vtile + (size_t)(tbase + t0) * D * E + d0 * E, v0);
          Vec4Load<CT>::run(vtile + (size_t)(tbase + t0 + 1) * D * E + d0 * E, v1);
          if (!full) {  // tokens past the end may hold NaN: their weight is 0, drop the value too
#pragma unroll
            for (int d = 0; d < DV; ++d) {
              v0[d] = tm.keep(tbase + t0) ? v0[d] : 0.f;
              v1[d] = tm.keep(tbase + t0 + 1) ? v1[d] : 0.f;
            }
          }
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float2 p2 = *reinterpret_cast<const float2*>(ps + h * TB + t0);
#pragma unroll
            for (int d = 0; d < DV; ++d) acc[h][d] = ffma2(p2, make_float2(v0[d], v1[d]), acc[h][d]);
          }
        }
        __syncwarp();
      }
      ++consumed;
      if (alive) issue_next();
    }

    // ------------------------------------------------------------ piece end
    // fold the token halves and token groups; l: sum over the lanes of a head
    float o[G][DV];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int d = 0; d < DV; ++d) {
        float v = acc[h][d].x + acc[h][d].y;
#pragma unroll
        for (int off = SL; off < 32; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        o[h][d] = v;
      }
    float l_h = l_own;
#pragma unroll
    for (int off = 1; off < C / G; off <<= 1) l_h += __shfl_xor_sync(0xffffffffu, l_h, off);
#pragma unroll
    for (int off = C; off < 32; off <<= 1) l_h += __shfl_xor_sync(0xffffffffu, l_h, off);
    float l_all[G];
#pragma unroll
    for (int h = 0; h < G; ++h) l_all[h] = __shfl_sync(0xffffffffu, l_h, h * (C / G));

    const int kvh = wk.unit / a.units_per_kv, chunk = wk.unit % a.units_per_kv;
    const int qh0 = kvh * a.group + chunk * G;
    const bool whole = (wk.jb == 0 && wk.je == wk.nb);

    if constexpr (!BALANCED) {
      // fixed partition: normalised output, natural-log max, sum
      const int p = (int)(gw % a.max_partitions);
      if (lane < SL) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const size_t row = ((size_t)wk.s * a.num_q_heads + qh0 + h) * a.max_partitions + p;
          const float inv = l_all[h] > 0.f ? a.out_scale / l_all[h] : 0.f;
          *reinterpret_cast<float4*>(a.o_part + row * D + d0) =
              make_float4(o[h][0] * inv, o[h][1] * inv, o[h][2] * inv, o[h][3] * inv);
          if (lane == 0) {
            a.m_part[row] = m_run[h] * 0.69314718055994531f;
            a.l_part[row] = l_all[h];
          }
        }
      }
    } else if (whole) {
      QT* out = reinterpret_cast<QT*>(a.out) + ((size_t)wk.s * a.num_q_heads + qh0) * D;
      if (lane < SL) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float inv = l_all[h] > 0.f ? a.out_scale / l_all[h] : 0.f;
#pragma unroll
          for (int d = 0; d < DV; ++d) out[h * D + d0 + d] = from_f32<QT>(o[h][d] * inv);
        }
      }
    } else {
      // segment cut between warps: publish (acc, m, l) now; the
      // last warp to arrive combines every piece and writes the output
      float* pslot = partial_slot<G, D>(a, wk, gw, u0);
      if (lane < SL) {
#pragma unroll
        for (int h = 0; h < G; ++h)
          *reinterpret_cast<float4*>(pslot + h * D + d0) = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
      }
#pragma unroll
      for (int h = 0; h < G; ++h)
        if (lane == h) {
          pslot[G * D + h] = m_run[h];
          pslot[G * D + G + h] = l_all[h];
        }
      // the ticket is taken when this warp's whole range is done
      if (ncut == 0) cut0 = cut_piece_of(wk); else cut1 = cut_piece_of(wk);
      ++ncut;
    }
    ++piece;
    walker_next_piece<BS>(wk, a, u1);
  }

  if constexpr (BALANCED) finish_cut_pieces<QT, G, D>(a, cut0, cut1, ncut, T, NW, lane);

  // Leave no copy in flight: wait (bounded) for every stage this warp filled
  // but did not wait for (only possible after a timeout).
  for (int k = waited; k < issued; ++k) mbar_wait_bounded(&bars[k % NSW], (k / NSW) & 1, a.err);
}

}  // namespace pkv
