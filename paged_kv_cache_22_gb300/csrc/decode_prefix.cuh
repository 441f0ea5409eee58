// decode_prefix.cuh -- attention of blocks of 16 query rows over paged K/V
// on the tensor cores, in two modes:
//
//  - the shared-prefix half of cascade decode (MULTI false), below;
//  - several query tokens per sequence (MULTI true): a prefill chunk, or the
//    tokens a speculative step verifies ("PagedAttention por dentro",
//    section "Chunked prefill integrado con paged KV"; "Componentes Internos
//    de Servicio de vLLM", section "Chunked prefill protege la cola del
//    TTFT").  The rows of a warp are (query token, query head) pairs of one
//    sequence and kv head; query token i of a chunk of T sits at position
//    L - T + i and attends positions 0 .. L - T + i (causal inside the
//    chunk), so each row has its own token limit, as the prefix rows do.
//
// When every sequence of a batch starts with the same prefix blocks (a
// shared system prompt: "La despensa por casilleros", section "Prefix
// caching: compartir casilleros con copy-on-write"), decode reads the
// prefix's K and V once per sequence although the tiles are the same.  The
// cascade splits the work: this kernel attends every query row of the batch
// to the prefix once per 16 rows, and the decode kernel then walks each
// sequence's own blocks past the prefix and starts each segment's online
// softmax from this partial result.  The output is that of plain decode.
//
// Design (GB300): one warp per (kv head [, sequence], block of 16 query
// rows, piece of the K/V range); the 16 rows are (sequence or query token,
// query head) pairs of that kv head, so all 16 rows of the m16n8k16 operand
// are real and each tile feeds 16 rows instead of G.  The PW warps of a CTA
// share one ring of tiles: lane 0 of warp 0 starts each TMA tensor copy
// (swizzled for ldmatrix, as in the decode kernel) and refills a stage once
// every warp has arrived on its "empty" barrier.  The range is cut into
// pieces so that the grid fills every SM; the last warp of a row block to
// finish merges the pieces' partials by log-sum-exp.  P keeps a head and a
// remainder of the operand type (two MMAs per n-tile).  Partials are
// unnormalised: o = sum_t 2^(s_t - m) v_t, m = max_t s_t (log2 units of the
// scaled score), l = sum_t 2^(s_t - m), over the tokens t below the row's
// limit.
#pragma once

#include "decode_tc.cuh"

namespace pkv {

struct PrefixArgs {
  unsigned int* err;
  const void* q;                 // [B, Hq, D]; MULTI: [total_q, Hq, D]
  const int32_t* block_tables;   // the first prefix_blocks entries of every row are the prefix
  int64_t table_stride;
  const int32_t* seq_lens;
  int num_seqs, num_q_heads, num_kv_heads, group, num_blocks, len_clip;
  int prefix_blocks;
  int row_blocks;                // ceil(num_seqs * group / 16)
  int splits;                    // the prefix is cut into this many pieces (<= 32) ...
  int split_blocks;              // ... of this many blocks (the last may be shorter)
  float qk_scale;                // scale * log2(e) (* kv_scale for fp8 caches)
  float* pre;                    // [B * Hq] rows of pre_row_floats(D): o, m, l (the result)
  float* scratch;                // [splits, B * Hq] rows of the same: one per piece (splits > 1)
  int* counters;                 // [Hkv * row_blocks], zero between calls (splits > 1)
  // MULTI only
  const int32_t* q_start;        // [B + 1]: sequence s owns query rows q_start[s] .. q_start[s+1]-1
  int total_q;                   // query rows in all
  int max_rb;                    // 16-row blocks per (sequence, kv head) the grid covers
  void* out;                     // [total_q, Hq, D] in the query type, normalised
  float out_scale;               // 1 (kv_scale for fp8 caches)
};

// Warps per CTA (PW): the PW warps of a CTA take 16 rows each of the same kv
// head [and sequence] and piece, and share one ring of tiles (one tensor
// copy per tile for all of them).  Four for the prefix pass and for
// multi-token queries with more than 16 rows per (sequence, kv head); one
// for at most 16 (a speculative step's few tokens), so that no warp slot
// idles.  Either way 12 warps fit per SM (168 registers).
constexpr int kPrefixWarps = 4;

template <class CT, int D, int BS>
struct PrefixSmem {
  using GE = TcGeo<CT, D, BS, 1>;
  static constexpr size_t kStages = 0;  // 1024-byte aligned
  static constexpr size_t kFull = (size_t)GE::NSW * GE::STAGE;  // tile landed
  static constexpr size_t kEmpty = kFull + (size_t)GE::NSW * 8;  // every warp done with it
  static constexpr size_t kOk = kEmpty + (size_t)GE::NSW * 8;     // the stage's block id was valid
  static constexpr size_t kBytes = kOk + (size_t)GE::NSW * 4;
};

template <class CT, int D, int BS, bool MULTI, int PW>
__global__ void __launch_bounds__(32 * PW, 12 / PW)
    prefix_attention_kernel(const __grid_constant__ PrefixArgs a, const __grid_constant__ TmaMaps maps) {
  using GE = TcGeo<CT, D, BS, 1>;
  using SM = PrefixSmem<CT, D, BS>;
  using QT = typename CT::QType;
  constexpr bool F8 = GE::F8;
  constexpr int NSW = GE::NSW, TB = GE::TB, KS = GE::KS, NTO = GE::NTO, TILE = GE::TILE, STAGE = GE::STAGE;
  static_assert(TB == 16 || !F8, "fp8 caches: 16-token steps");

  extern __shared__ __align__(1024) uint8_t pf_smem[];
  uint8_t* const stages = pf_smem + SM::kStages;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  if (smem_addr(stages) & 1023u) {
    if (threadIdx.x == 0) raise_error(a.err, PKV_DEVERR_SMEM_ALIGN);
    return;
  }
  const uint32_t stages_s = smem_addr(stages);
  uint64_t* bars = reinterpret_cast<uint64_t*>(pf_smem + SM::kFull);
  uint64_t* empty = reinterpret_cast<uint64_t*>(pf_smem + SM::kEmpty);
  int* stage_ok = reinterpret_cast<int*>(pf_smem + SM::kOk);

  // CTA -> (piece of the K/V range, kv head [, sequence], PW blocks of 16
  // rows); warp -> one of those blocks
  const int piece = blockIdx.x % a.splits, cg = blockIdx.x / a.splits;
  int h, rb, nrb;             // kv head, this warp's row block, row blocks in all
  int ms = 0, mq0 = 0, mT = 0, mL = 0;  // MULTI: sequence, its first query row, T, its length
  if constexpr (!MULTI) {
    const int groups = (a.row_blocks + PW - 1) / PW;
    h = cg / groups;
    rb = (cg % groups) * PW + w;
    nrb = a.row_blocks;
  } else {
    const int groups = (a.max_rb + PW - 1) / PW;
    const int sh = cg / groups;
    ms = sh / a.num_kv_heads;
    h = sh % a.num_kv_heads;
    rb = (cg % groups) * PW + w;
    mq0 = __ldg(a.q_start + ms);
    mT = __ldg(a.q_start + ms + 1) - mq0;
    mL = __ldg(a.seq_lens + ms);
    const bool bad = mL < 0 || mL > a.len_clip || mT < 0 || mT > mL || mq0 < 0 || mq0 + mT > a.total_q ||
                     mT * a.group > a.max_rb * 16;
    if (bad) {  // flagged once per sequence; its rows are left alone
      if (threadIdx.x == 0 && h == 0 && piece == 0 && cg % groups == 0) raise_error(a.err, PKV_DEVERR_BAD_SEQ_LEN);
      mT = 0;
    }
    nrb = (mT * a.group + 15) / 16;
  }
  // warps past the last row block have nothing to do: they leave before the
  // ring starts, and the "empty" barriers count only the warps that stay
  const int nact = min(PW, max(0, nrb - (rb - w)));
  if (nact == 0) return;  // the whole CTA (uniform)
  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < NSW; ++i) {
      mbar_init(&bars[i], 1);
      mbar_init(&empty[i], nact);
    }
    fence_mbar_init();
  }
  __syncthreads();
  // the cascade's suffix decode may start its prologue on SMs this grid frees
  // (it waits for the whole grid before it reads any partial)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (w >= nact) return;
  const int hr = MULTI ? (ms * a.num_kv_heads + h) * a.max_rb + rb : h * a.row_blocks + rb;
  // the lane's two rows (g, g + 8): the query row they read (the sequence's
  // row for the prefix; the token's row of q for MULTI), query head, tokens
  // attended (positions below rlim), validity
  int rrow[2], rq[2], rlim[2];
  bool rv[2];
  const int ptok = a.prefix_blocks * BS;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int R = rb * 16 + g + 8 * r;
    rq[r] = h * a.group + R % a.group;
    if constexpr (!MULTI) {
      rrow[r] = R / a.group;
      rv[r] = rrow[r] < a.num_seqs;
      int L = rv[r] ? __ldg(a.seq_lens + rrow[r]) : 0;
      L = L < 0 ? 0 : (L > a.len_clip ? a.len_clip : L);
      rlim[r] = L < ptok ? L : ptok;
    } else {
      const int i = R / a.group;  // query token of the chunk
      rv[r] = R < mT * a.group;
      rrow[r] = mq0 + (rv[r] ? i : 0);
      rlim[r] = rv[r] ? mL - mT + i + 1 : 0;
    }
  }
  // tokens no row of this warp attends are zeroed in V (they may be unwritten)
  int lim_all = rlim[0] > rlim[1] ? rlim[0] : rlim[1];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lim_all = max(lim_all, __shfl_xor_sync(0xffffffffu, lim_all, off));

  // blocks of this piece: the prefix's, or (MULTI) the sequence's up to the
  // last position any row of the CTA attends; the table row they are read from
  const int32_t* table = a.block_tables;
  int nb_all = a.prefix_blocks;
  if constexpr (MULTI) {
    table = a.block_tables + (size_t)ms * a.table_stride;
    const int last_row = min(mT * a.group, (rb - w + nact) * 16) - 1;  // the CTA's last row
    nb_all = (mL - mT + last_row / a.group + 1 + BS - 1) / BS;
  }
  // MULTI: each sequence's own range is cut into `splits` equal pieces
  // (lengths differ, so pieces sized by the longest would leave the short
  // sequences' pieces empty and the long ones' long)
  const int sb = MULTI ? (nb_all + a.splits - 1) / a.splits : a.split_blocks;
  const int jb = piece * sb;
  const int je = min(nb_all, jb + sb);

  // the prefix blocks a sequence attends must be those of sequence 0's table
  // (checked once, by kv head 0; entries past a short sequence's end are not
  // read by plain decode either, so they are not compared)
  if (!MULTI && h == 0 && piece == 0) {
    const int s_lo = rb * 16 / a.group, s_hi = min(a.num_seqs, (rb * 16 + 15) / a.group + 1);
    for (int s = s_lo; s < s_hi; ++s) {
      int L = __ldg(a.seq_lens + s);
      L = L < 0 ? 0 : (L > a.len_clip ? a.len_clip : L);
      const int nb = min(a.prefix_blocks, (L + BS - 1) / BS);
      for (int j = lane; j < nb; j += 32)
        if (__ldg(a.block_tables + (size_t)s * a.table_stride + j) != __ldg(a.block_tables + j))
          raise_error(a.err, PKV_DEVERR_BAD_BLOCK_ID);
    }
  }

  // q.K A operand, all 16 rows: (a0, a1, a2, a3) per k-step
  uint32_t qa[KS][4];
  float qk_mul = a.qk_scale;
  {
    const QT* qrow[2];
#pragma unroll
    for (int r = 0; r < 2; ++r)
      qrow[r] = reinterpret_cast<const QT*>(a.q) + ((size_t)(rv[r] ? rrow[r] : 0) * a.num_q_heads + rq[r]) * D;
    if constexpr (!F8) {
#pragma unroll
      for (int kk = 0; kk < KS; ++kk)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const bool live = rv[r];
          qa[kk][r] = live ? *reinterpret_cast<const uint32_t*>(qrow[r] + 16 * kk + 2 * t) : 0u;
          qa[kk][2 + r] = live ? *reinterpret_cast<const uint32_t*>(qrow[r] + 16 * kk + 2 * t + 8) : 0u;
        }
    } else {
      // fp16 operands in the order a K chunk reaches the lane (dims 4t..4t+3
      // of each 16-dim chunk), scaled by a power of two so that |q| < 2^15
      float qv[KS][2][4];
      float mq = 0.f;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const bool live = rv[r];
          const uint2 raw = live ? *reinterpret_cast<const uint2*>(qrow[r] + 16 * kk + 4 * t) : make_uint2(0u, 0u);
          const float2 lo = bf16x2_to_f2(raw.x), hi = bf16x2_to_f2(raw.y);
          qv[kk][r][0] = lo.x;
          qv[kk][r][1] = lo.y;
          qv[kk][r][2] = hi.x;
          qv[kk][r][3] = hi.y;
#pragma unroll
          for (int i = 0; i < 4; ++i) mq = fmaxf(mq, fabsf(qv[kk][r][i]));
        }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, off));
      int e = 0;
      frexpf(mq, &e);
      const int sh = e > 15 ? (e - 15 < 100 ? e - 15 : 100) : 0;
      const float down = ldexpf(1.f, -sh);
      qk_mul = a.qk_scale * ldexpf(1.f, sh);
#pragma unroll
      for (int kk = 0; kk < KS; ++kk)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          qa[kk][r] = pack_f16x2(qv[kk][r][0] * down, qv[kk][r][1] * down);
          qa[kk][2 + r] = pack_f16x2(qv[kk][r][2] * down, qv[kk][r][3] * down);
        }
    }
  }

  // ---------------------------------------------------------------- issue side
  // Producer: lane 0 of warp 0 starts every tile copy of the CTA.
  int issued = 0;  // blocks of this piece whose copy was started
  // The producer warp reads the piece's block ids 32 at a time (one
  // coalesced load) and hands each to lane 0 by shuffle; whether a stage's
  // id was valid goes to shared memory with the stage, so that no warp waits
  // on a global load per block.
  int id_chunk = -1;
  int32_t id_reg = 0;
  auto issue_next = [&]() {
    if (jb + issued >= je) return;
    const int st = issued % NSW;
    if (w == 0) {
      if ((issued >> 5) != id_chunk) {
        id_chunk = issued >> 5;
        const int jj = jb + (id_chunk << 5) + lane;
        id_reg = jj < je ? __ldg(table + jj) : -1;
      }
      const int32_t id = __shfl_sync(0xffffffffu, id_reg, issued & 31);
      uint8_t* dst = stages + (size_t)st * STAGE;
      const bool valid = id >= 0 && id < a.num_blocks;
      if (lane == 0) {
        if (valid) {
          stage_ok[st] = 1;
          mbar_arrive_expect_tx(&bars[st], STAGE);
          tma_load_tile<GE>(dst, &maps.k, h * BS, id, &bars[st]);
          tma_load_tile<GE>(dst + TILE, &maps.v, h * BS, id, &bars[st]);
        } else {
          raise_error(a.err, PKV_DEVERR_BAD_BLOCK_ID);
          stage_ok[st] = 0;
          mbar_arrive(&bars[st]);
        }
      }
    }
    ++issued;
  };
  // the cascade's decode runs after this grid on the stream; the cache write
  // of the step (if any) ran before both
  if (w == 0) {
#pragma unroll 1
    for (int i = 0; i < NSW; ++i) issue_next();
  }

  // fragment addresses (as in the decode kernel)
  auto lane_base = [](int row, int hh) -> uint32_t { return swz<GE>(row, hh); };
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
  constexpr int CPB = GE::IB / 16;
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

  // ---------------------------------------------------------------- consume side
  float o[NTO][4];  // columns 2t, 2t+1 of each n-tile: [0..1] row g, [2..3] row g + 8
#pragma unroll
  for (int n = 0; n < NTO; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F}, l_run[2] = {0.f, 0.f};
  int waited = 0;
  bool alive = true;

#pragma unroll 1
  for (int j = jb; j < je; ++j) {
    const int i = j - jb;  // position in this piece's ring
    const int st = i % NSW;
    if (alive) {
      if (!mbar_wait_bounded(&bars[st], (i / NSW) & 1, a.err)) alive = false;
      waited = i + 1;
    }
    const bool ok = alive && stage_ok[st] != 0;
#pragma unroll
    for (int step = 0; step < GE::STEPS; ++step) {
      const uint32_t kt = stages_s + (uint32_t)(st * STAGE + step * TB * GE::IB);
      const uint32_t vt = kt + TILE;
      const int p0 = j * BS + step * TB;  // prefix position of the step's first token
      // ---- scores of both rows: c[n] = (row g: cols 2t, 2t+1 | row g + 8: same)
      float sc[GE::NTS][4];
      {
        float s2[2][GE::NTS][4] = {};
        if constexpr (F8) {
#pragma unroll
          for (int kq = 0; kq < KS / 2; ++kq) {
            uint32_t r[4];
            ldsm_x4(frag(kt + kx, 2 * kq), r);
            uint32_t b[4][2];
#pragma unroll
            for (int m = 0; m < 4; ++m) e4m3x4_to_f16x2x2(r[m], b[m][0], b[m][1]);
            mma_k16_rows16<true>(s2[0][0], qa[2 * kq][0], qa[2 * kq][1], qa[2 * kq][2], qa[2 * kq][3], b[0][0], b[0][1]);
            mma_k16_rows16<true>(s2[0][1], qa[2 * kq][0], qa[2 * kq][1], qa[2 * kq][2], qa[2 * kq][3], b[1][0], b[1][1]);
            mma_k16_rows16<true>(s2[1][0], qa[2 * kq + 1][0], qa[2 * kq + 1][1], qa[2 * kq + 1][2], qa[2 * kq + 1][3],
                                 b[2][0], b[2][1]);
            mma_k16_rows16<true>(s2[1][1], qa[2 * kq + 1][0], qa[2 * kq + 1][1], qa[2 * kq + 1][2], qa[2 * kq + 1][3],
                                 b[3][0], b[3][1]);
          }
        } else if constexpr (TB == 16) {
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            uint32_t r[4];
            ldsm_x4(frag(kt + kx, 2 * kk), r);
            mma_k16_rows16<false>(s2[kk & 1][0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], r[0], r[1]);
            mma_k16_rows16<false>(s2[kk & 1][1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], r[2], r[3]);
          }
        } else {
#pragma unroll
          for (int kq = 0; kq < KS / 2; ++kq) {
            uint32_t r[4];
            ldsm_x4(frag(kt + kx, 4 * kq), r);
            mma_k16_rows16<false>(s2[0][0], qa[2 * kq][0], qa[2 * kq][1], qa[2 * kq][2], qa[2 * kq][3], r[0], r[1]);
            mma_k16_rows16<false>(s2[1][0], qa[2 * kq + 1][0], qa[2 * kq + 1][1], qa[2 * kq + 1][2],
                                  qa[2 * kq + 1][3], r[2], r[3]);
          }
        }
#pragma unroll
        for (int n = 0; n < GE::NTS; ++n)
#pragma unroll
          for (int c = 0; c < 4; ++c) sc[n][c] = s2[0][n][c] + s2[1][n][c];
      }
      // ---- online softmax, row by row (c = 2r + e: row g + 8r, column 2t + e)
      float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
      for (int n = 0; n < GE::NTS; ++n)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int r = c >> 1, tok = p0 + 8 * n + 2 * t + (c & 1);
          sc[n][c] = (ok && tok < rlim[r]) ? sc[n][c] * qk_mul : -CUDART_INF_F;
          mx[r] = fmaxf(mx[r], sc[n][c]);
        }
      float alpha[2];
      bool grow = false;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        const float m_new = fmaxf(m_run[r], mx[r]);
        alpha[r] = m_new > m_run[r] ? fast_exp2(m_run[r] - m_new) : 1.f;
        grow |= m_new > m_run[r];
        m_run[r] = m_new;
      }
      if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int n = 0; n < NTO; ++n) {
          o[n][0] *= alpha[0];
          o[n][1] *= alpha[0];
          o[n][2] *= alpha[1];
          o[n][3] *= alpha[1];
        }
        l_run[0] *= alpha[0];
        l_run[1] *= alpha[1];
      }
      float p[GE::NTS][4];
#pragma unroll
      for (int n = 0; n < GE::NTS; ++n)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int r = c >> 1;
          const float mu = m_run[r] == -CUDART_INF_F ? 0.f : m_run[r];
          p[n][c] = fast_exp2(sc[n][c] - mu);
          l_run[r] += p[n][c];
        }
      // ---- P . V: P as a head and a remainder, both rows real
      const bool full = ok && p0 + TB <= lim_all;
      uint32_t ph[2][4], pl[2][4];  // [0]: k-step tokens 0-7 (a0 row g, a1 row g+8) ...
      // A operand (m16 x k16 tokens): a0 = row g, tokens 2t..; a1 = row g+8, tokens 2t..;
      // a2 = row g, tokens 2t+8..; a3 = row g+8, tokens 2t+8..
#pragma unroll
      for (int n = 0; n < GE::NTS; ++n)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float x0 = p[n][2 * r], x1 = p[n][2 * r + 1];
          uint32_t hh, ll;
          if constexpr (F8) {
            hh = pack_f16x2(x0, x1);
            const float2 hv = f16x2_to_f2(hh);
            ll = pack_f16x2(x0 - hv.x, x1 - hv.y);
          } else {
            hh = pack_bf16x2(x0, x1);
            const float2 hv = bf16x2_to_f2(hh);
            ll = pack_bf16x2(x0 - hv.x, x1 - hv.y);
          }
          ph[n][r] = hh;
          pl[n][r] = ll;
        }
      if constexpr (F8) {
        uint32_t X[4][GE::VPL / 4];
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
        if (!full) {
          const int rows[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
          for (int ri = 0; ri < 4; ++ri)
#pragma unroll
            for (int qq = 0; qq < GE::VPL / 4; ++qq) X[ri][qq] = (ok && p0 + rows[ri] < lim_all) ? X[ri][qq] : 0u;
        }
#pragma unroll
        for (int qq = 0; qq < GE::VPL / 4; ++qq) {
          uint32_t b0[4], b1[4];
          e4m3x4_to_f16x2x2(__byte_perm(X[0][qq], X[1][qq], 0x5140), b0[0], b0[1]);
          e4m3x4_to_f16x2x2(__byte_perm(X[0][qq], X[1][qq], 0x7362), b0[2], b0[3]);
          e4m3x4_to_f16x2x2(__byte_perm(X[2][qq], X[3][qq], 0x5140), b1[0], b1[1]);
          e4m3x4_to_f16x2x2(__byte_perm(X[2][qq], X[3][qq], 0x7362), b1[2], b1[3]);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            mma_k16_rows16<true>(o[4 * qq + k], ph[0][0], ph[0][1], ph[1][0], ph[1][1], b0[k], b1[k]);
            mma_k16_rows16<true>(o[4 * qq + k], pl[0][0], pl[0][1], pl[1][0], pl[1][1], b0[k], b1[k]);
          }
        }
      } else {
        uint32_t keep0 = 0xFFFFFFFFu, keep1 = 0xFFFFFFFFu;
        if (!full) {
          auto kept = [&](int tok) { return ok && p0 + tok < lim_all; };
          keep0 = (kept(2 * t) ? 0x0000FFFFu : 0u) | (kept(2 * t + 1) ? 0xFFFF0000u : 0u);
          keep1 = (kept(2 * t + 8) ? 0x0000FFFFu : 0u) | (kept(2 * t + 9) ? 0xFFFF0000u : 0u);
        }
        if constexpr (TB == 16) {
#pragma unroll
          for (int jv = 0; jv < NTO / 2; ++jv) {
            uint32_t r[4];
            ldsm_x4_t(frag(vt + vx, 2 * jv), r);
            r[0] &= keep0; r[1] &= keep1; r[2] &= keep0; r[3] &= keep1;
            mma_k16_rows16<false>(o[2 * jv], ph[0][0], ph[0][1], ph[1][0], ph[1][1], r[0], r[1]);
            mma_k16_rows16<false>(o[2 * jv + 1], ph[0][0], ph[0][1], ph[1][0], ph[1][1], r[2], r[3]);
            mma_k16_rows16<false>(o[2 * jv], pl[0][0], pl[0][1], pl[1][0], pl[1][1], r[0], r[1]);
            mma_k16_rows16<false>(o[2 * jv + 1], pl[0][0], pl[0][1], pl[1][0], pl[1][1], r[2], r[3]);
          }
        } else {
#pragma unroll
          for (int jv = 0; jv < NTO / 4; ++jv) {
            uint32_t r[4];
            ldsm_x4_t(frag(vt + vx, 4 * jv), r);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              r[m] &= keep0;
              mma_k8_bf16_rows16(o[4 * jv + m], ph[0][0], ph[0][1], r[m]);
              mma_k8_bf16_rows16(o[4 * jv + m], pl[0][0], pl[0][1], r[m]);
            }
          }
        }
      }
    }
    __syncwarp();  // every lane is done with this stage ...
    if (lane == 0) mbar_arrive(&empty[st]);  // ... and so is this warp
    // The producer refills the stage of the previous block once every warp
    // is done with it (a block later, so the wait seldom blocks).
    if (w == 0 && i >= 1 && jb + issued < je) {
      const int ip = i - 1;
      if (alive && !mbar_wait_bounded(&empty[ip % NSW], (ip / NSW) & 1, a.err)) alive = false;
      if (alive) issue_next();
    }
  }

  // ---------------------------------------------------------------- partials
  // One piece: the result (the prefix partial, or MULTI's normalised
  // output).  Several: this piece's partial, merged below.
  constexpr int PRF = pre_row_floats(D);
  const size_t rows = MULTI ? (size_t)a.total_q * a.num_q_heads : (size_t)a.num_seqs * a.num_q_heads;
  float* base = a.splits == 1 ? a.pre : a.scratch + (size_t)piece * rows * PRF;
  auto odim = [&](int n, int e) -> int { return F8 ? GE::VPL * (2 * t + e) + n : 8 * n + 2 * t + e; };
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float l_row = l_run[r] + __shfl_xor_sync(0xffffffffu, l_run[r], 1);
    l_row += __shfl_xor_sync(0xffffffffu, l_row, 2);
    if (!rv[r]) continue;
    const size_t orow = (size_t)rrow[r] * a.num_q_heads + rq[r];
    if (MULTI && a.splits == 1) {
      QT* dst = reinterpret_cast<QT*>(a.out) + orow * D;
      const float inv = l_row > 0.f ? a.out_scale / l_row : 0.f;
      if constexpr (F8) {  // dims n, n + 1 of column 2t + e are adjacent
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
          for (int n = 0; n < NTO; n += 2)
            *reinterpret_cast<uint32_t*>(dst + odim(n, e)) =
                pack_bf16x2(o[n][2 * r + e] * inv, o[n + 1][2 * r + e] * inv);
      } else {
#pragma unroll
        for (int n = 0; n < NTO; ++n)
          *reinterpret_cast<uint32_t*>(dst + odim(n, 0)) = pack_bf16x2(o[n][2 * r] * inv, o[n][2 * r + 1] * inv);
      }
      continue;
    }
    float* dst = base + orow * PRF;
#pragma unroll
    for (int n = 0; n < NTO; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) dst[odim(n, e)] = o[n][2 * r + e];
    if (t == 0) {
      dst[D] = m_run[r];
      dst[D + 1] = l_row;
    }
  }
  if (a.splits > 1) {
    // the last piece of this (kv head, row block) to finish merges them all
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      last = atomicAdd(a.counters + hr, 1) == a.splits - 1;
      if (last) a.counters[hr] = 0;  // ready for the next call
    }
    if (__shfl_sync(0xffffffffu, last, 0)) {
      __threadfence();
      // four rows at a time, every load of the four issued before any use:
      // lane k < splits reads piece k's (m, l); lane i covers dims 4i..4i+3
#pragma unroll 1
      for (int r0 = 0; r0 < 16; r0 += 4) {
        size_t row[4];
        bool live[4];
        float mk[4], lk[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int R = rb * 16 + r0 + u;
          if constexpr (!MULTI) {
            const int s = R / a.group;
            live[u] = s < a.num_seqs;
            row[u] = live[u] ? (size_t)s * a.num_q_heads + h * a.group + R % a.group : 0;
          } else {
            live[u] = R < mT * a.group;
            row[u] = live[u] ? (size_t)(mq0 + R / a.group) * a.num_q_heads + h * a.group + R % a.group : 0;
          }
          mk[u] = -CUDART_INF_F;
          lk[u] = 0.f;
          if (live[u] && lane < a.splits) {
            const float* p = a.scratch + ((size_t)lane * rows + row[u]) * PRF;
            mk[u] = __ldcg(p + D);
            lk[u] = __ldcg(p + D + 1);
          }
        }
        float M[4], wk[4], den[4];
        float4 acc[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          M[u] = mk[u];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) M[u] = fmaxf(M[u], __shfl_xor_sync(0xffffffffu, M[u], off));
          const float Mc = M[u] == -CUDART_INF_F ? 0.f : M[u];
          wk[u] = lane < a.splits ? fast_exp2(mk[u] - Mc) : 0.f;
          den[u] = lk[u] * wk[u];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) den[u] += __shfl_xor_sync(0xffffffffu, den[u], off);
          acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int k = 0; k < a.splits; ++k) {
          float4 v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            v[u] = (live[u] && 4 * lane < D)
                       ? __ldcg(reinterpret_cast<const float4*>(a.scratch + ((size_t)k * rows + row[u]) * PRF) + lane)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float wkk = __shfl_sync(0xffffffffu, wk[u], k);
            acc[u].x += v[u].x * wkk;
            acc[u].y += v[u].y * wkk;
            acc[u].z += v[u].z * wkk;
            acc[u].w += v[u].w * wkk;
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (!live[u]) continue;
          if constexpr (MULTI) {  // the normalised output row
            const float inv = den[u] > 0.f ? a.out_scale / den[u] : 0.f;
            QT* dst = reinterpret_cast<QT*>(a.out) + row[u] * D;
            if (4 * lane < D)
              *reinterpret_cast<uint2*>(dst + 4 * lane) =
                  make_uint2(pack_bf16x2(acc[u].x * inv, acc[u].y * inv), pack_bf16x2(acc[u].z * inv, acc[u].w * inv));
          } else {
            float* dst = a.pre + row[u] * PRF;
            if (4 * lane < D) reinterpret_cast<float4*>(dst)[lane] = acc[u];
            if (lane == 0) {
              dst[D] = M[u];
              dst[D + 1] = den[u];
            }
          }
        }
      }
    }
  }
  for (int k = waited; k < issued; ++k) mbar_wait_bounded(&bars[k % NSW], (k / NSW) & 1, a.err);
}

}  // namespace pkv
