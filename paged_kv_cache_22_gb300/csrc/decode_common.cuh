// decode_common.cuh -- what both paged decode kernels share: the argument
// block, the tensor-map pair, the balanced split of the tile stream over the
// warps of the grid, the walk over (sequence, kv-head unit) segments, and the
// log-sum-exp merge of a segment that was cut between warps.
//
// The operation (per sequence s, query head qh, kv head h = qh / g):
//   out[s][qh] = softmax_t(scale * q[s][qh] . K_s[t]) . V_s[t],  t < seq_len[s]
// with K_s[t] = k_cache[block_tables[s][t / BS]][h][t % BS] -- the decode
// attention of "Optimización de Inferencia LLM" (section "El Cuello de
// Botella de Atención del que Nadie Habla"), read block by block through the
// block table as "La despensa por casilleros" describes (section "El
// mecanismo: bloques, block table y el gather del kernel"), accumulated with
// an online softmax as the kernel sketch of "Optimización de Inferencia LLM"
// (section "PagedAttention: Conceptos de SO se Encuentran con Memoria GPU")
// prescribes, and split over the key axis with a log-sum-exp merge of the
// partial results.
#pragma once

#include <math_constants.h>

#include "pkv_device.cuh"

namespace pkv {

struct DecodeArgs {
  unsigned int* err;  // device error word
  void* out;
  const void* q;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const int32_t* block_tables;
  int64_t table_stride;  // max_blocks_per_seq
  const int32_t* seq_lens;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int num_blocks;
  int group;         // g = Hq / Hkv
  int units_per_kv;  // g / G: query-head chunks per kv head
  int units;         // num_kv_heads * units_per_kv (segments per sequence)
  int len_clip;      // longest admissible seq_len
  int window;        // > 0: attend only the last `window` tokens and the first `sinks`
  int sinks;
  // cascade: the first skip_blocks blocks of every sequence are a shared
  // prefix already attended; its partial result per output row, [B * Hq]
  // rows of pre_row_floats(D) floats (o unnormalised, then m in log2 units,
  // then l), is where each segment's online softmax starts
  int skip_blocks;
  const float* pre;
  float qk_scale;    // scale * log2(e) (* kv_scale for fp8 caches)
  float out_scale;   // 1 (kv_scale for fp8 caches)
  // several query tokens per sequence (the multi-query instances): sequence
  // s owns query rows q_start[s] .. q_start[s + 1] - 1 of q and out ([rows,
  // Hq, D]), its last positions; a unit is (kv head, group of mq_tpu
  // tokens), its G rows (token, head) = (r / group, r % group) of the group
  const int32_t* q_start;
  int mq_tpu;        // tokens per unit (G / group); 0 for one token per sequence
  int max_q;         // host bound of the query rows per sequence
  int total_q;       // query rows in all
  // balanced split: 1 = cut pieces only publish their partials; a dependent
  // grid (merge_cut_kernel) merges the segments once this grid is done
  int defer_merge;
  // balanced split
  int* counters;     // [num_seqs * units], zero between calls
  float* partials;   // [2 * warps][partial_slot_floats(G, D)]
  // fixed partitions
  int partition_blocks;
  int max_partitions;
  float* o_part;     // [B, Hq, P, D]
  float* m_part;     // [B, Hq, P]
  float* l_part;     // [B, Hq, P]
};

// Opaque TMA tensor maps of the K and V caches (the layout of CUtensorMap:
// 128 bytes, 64-byte aligned), filled on the host by cuTensorMapEncodeTiled.
// Each views a cache [num_blocks, Hkv, BS, D] as the 3-D tensor
// (D, Hkv * BS, num_blocks), innermost first, with a box of one
// (block, kv head) tile: (tma_box_bytes(D * E) / E, BS, 1).
struct alignas(64) TmaMap {
  uint64_t opaque[16];
};
struct TmaMaps {
  TmaMap k, v;
};

// Bytes of the innermost box extent for cache rows of `row_bytes`: the
// 128-byte swizzle span when the row is at least that long, else the row.
__host__ __device__ constexpr int tma_box_bytes(int row_bytes) { return row_bytes >= 128 ? 128 : row_bytes; }

// ----------------------------------------------------------------------------
// Balanced split of T tiles over N workers.  With T >= N every worker gets
// floor((c+1)T/N) - floor(cT/N) >= 1 tiles; with T < N the first T workers
// get one tile each and the rest none, so a segment's tiles always lie on
// consecutive non-empty workers (the merge counts its pieces as
// last - first + 1).
// ----------------------------------------------------------------------------
__device__ __forceinline__ int64_t range_start(int64_t c, int64_t T, int64_t N) {
  return T >= N ? c * T / N : (c < T ? c : T);
}

// The worker whose range holds tile u (0 <= u < T).
__device__ __forceinline__ int64_t owner_of(int64_t u, int64_t T, int64_t N) {
  return T >= N ? ((u + 1) * N - 1) / T : u;
}

// ----------------------------------------------------------------------------
// Walk over the (sequence, unit) segments that intersect a tile range.  All
// lanes of a warp hold the same state.
// ----------------------------------------------------------------------------
struct Walker {
  int s, unit, nb;
  int64_t base;    // linear index of sequence s's first tile
  int64_t seg_u;   // linear index of segment (s, unit)'s first tile
  int jb, je;      // piece = blocks [jb, je) of the segment
  bool done;
};

// ----------------------------------------------------------------------------
// Sliding window with attention sinks ("PagedAttention por dentro", sections
// "Sliding window attention" and "StreamingLLM (Xiao et al., 2024): los
// attention sinks"): a sequence of length L > window attends only its first
// `sinks` tokens and its last `window` tokens.  Its blocks are read as the
// blocks holding sink tokens, then the window's blocks; the whole blocks in
// between (an engine may have freed them) are never touched.  BlockMap:
// blocks [0, nsb) and [wsb, nb) are read, nsb == wsb when nothing is left out.
// ----------------------------------------------------------------------------
struct BlockMap {
  int nsb, wsb;
};

template <int BS>
__device__ __forceinline__ BlockMap block_map(const DecodeArgs& a, int L) {
  BlockMap m{0, 0};
  if (a.skip_blocks > 0) {  // cascade: the blocks past the shared prefix
    const int nb = (L + BS - 1) / BS;
    m.wsb = a.skip_blocks < nb ? a.skip_blocks : nb;
    return m;
  }
  if (a.window > 0 && L > a.window) {
    const int ws = L - a.window;                 // first window token
    const int sk = a.sinks < ws ? a.sinks : ws;  // sink tokens before it
    const int nsb = (sk + BS - 1) / BS, wsb = ws / BS;
    if (wsb > nsb) {
      m.nsb = nsb;
      m.wsb = wsb;
    }
  }
  return m;
}

// Whether some sequence may skip blocks (a window, or a cascade's prefix),
// so that the j-th block read is not logical block j.  The decode kernels
// take this as a compile-time REMAP parameter: a per-tile runtime branch on
// it costs ~10 % of the fp8 decode, whose tile loop is latency bound.
inline bool remaps_blocks(int window, int skip_blocks) { return window > 0 || skip_blocks > 0; }

// Floats per row of a cascade's prefix partial: D of o, m, l, two of padding
// (rows stay 16-byte aligned for bulk copies).
__host__ __device__ constexpr int pre_row_floats(int D) { return D + 4; }

// Floats of one balanced-split partial result: acc[G][D], m[G], l[G], padded
// to a multiple of four so that every slot starts 16-byte aligned (the merge
// reads the accumulators as float4).
__host__ __device__ constexpr int partial_slot_floats(int G, int D) { return (G * D + 2 * G + 3) / 4 * 4; }

// Logical block of the j-th block a sequence of length L reads.
template <int BS>
__device__ __forceinline__ int logical_block(const DecodeArgs& a, int L, int j) {
  const BlockMap m = block_map<BS>(a, L);
  return j < m.nsb ? j : j + (m.wsb - m.nsb);
}

// Tokens of logical block jl that are attended, one bit per token (bit t:
// token t of the block, t < 32): t < hi and, under a window, (t < s_hi or
// t >= w_lo).  Computed once per tile, so that every per-token test in the
// score and V masks is a single bit test.
__device__ __forceinline__ uint32_t low_bits(int n) { return n <= 0 ? 0u : (n >= 32 ? 0xFFFFFFFFu : (1u << n) - 1u); }

struct TileMask {
  uint32_t bits;
  __device__ __forceinline__ bool keep(int tok) const { return (bits >> tok) & 1u; }
  // every token of [t0, t1) kept
  __device__ __forceinline__ bool all(int t0, int t1) const {
    const uint32_t m = low_bits(t1) & ~low_bits(t0);
    return (bits & m) == m;
  }
  __device__ __forceinline__ void clear() { bits = 0u; }
};

template <int BS, bool REMAP>
__device__ __forceinline__ TileMask tile_mask(const DecodeArgs& a, int L, int jl) {
  static_assert(BS <= 32, "one bit per token of a block");
  const int base = jl * BS;
  TileMask m;
  m.bits = low_bits(L - base < BS ? L - base : BS);
  if constexpr (REMAP)
    if (a.window > 0 && L > a.window) m.bits &= low_bits(a.sinks - base) | ~low_bits(L - a.window - base);
  return m;
}

// Blocks a sequence reads (all of its blocks unless a window leaves some out).
template <int BS>
__device__ __forceinline__ int seq_blocks(const DecodeArgs& a, int s) {
  int L = __ldg(a.seq_lens + s);
  if (L < 0 || L > a.len_clip) {
    raise_error(a.err, PKV_DEVERR_BAD_SEQ_LEN);
    L = L < 0 ? 0 : a.len_clip;
  }
  const BlockMap m = block_map<BS>(a, L);
  return (L + BS - 1) / BS - (m.wsb - m.nsb);
}

__device__ __forceinline__ int seq_len_clipped(const DecodeArgs& a, int s) {
  int L = __ldg(a.seq_lens + s);
  return L < 0 ? 0 : (L > a.len_clip ? a.len_clip : L);
}

template <int BS>
__device__ __forceinline__ void walker_settle(Walker& wk, const DecodeArgs& a, int64_t u1) {
  // Move forward to the first segment with blocks left before u1.
  while (!wk.done) {
    if (wk.nb > 0) {
      wk.seg_u = wk.base + (int64_t)wk.unit * wk.nb;
      if (wk.seg_u >= u1) { wk.done = true; break; }
      int64_t left = u1 - wk.seg_u;
      wk.je = (int64_t)wk.nb < left ? wk.nb : (int)left;
      if (wk.jb < wk.je) break;
    }
    wk.jb = 0;
    if (wk.nb > 0 && ++wk.unit < a.units) continue;
    wk.base += (int64_t)wk.nb * a.units;
    wk.unit = 0;
    if (++wk.s >= a.num_seqs) { wk.done = true; break; }
    wk.nb = seq_blocks<BS>(a, wk.s);
  }
}

template <int BS>
__device__ __forceinline__ void walker_next_piece(Walker& wk, const DecodeArgs& a, int64_t u1) {
  wk.jb = wk.je;  // past the current piece
  if (wk.je < wk.nb) { wk.done = true; return; }  // the range ended inside this segment
  wk.jb = 0;
  if (++wk.unit >= a.units) {
    wk.unit = 0;
    wk.base += (int64_t)wk.nb * a.units;
    if (++wk.s >= a.num_seqs) { wk.done = true; return; }
    wk.nb = seq_blocks<BS>(a, wk.s);
  }
  walker_settle<BS>(wk, a, u1);
}

// ----------------------------------------------------------------------------
// This warp's work.  Balanced mode: the warp's range [u0, u1) of the linear
// tile stream (T tiles in all) and the walker on its first piece; rows of
// empty sequences are zeroed on the way.  Fixed-partition mode: warp gw takes
// partition gw % P of segment gw / P.  False when the warp has nothing to do.
// ----------------------------------------------------------------------------
template <class QT, int D, int BS, bool BALANCED, bool ZERO_EMPTY = true>
__device__ __forceinline__ bool plan_warp(const DecodeArgs& a, int64_t gw, int64_t NW, int lane, Walker& wk0,
                                          int64_t& u0, int64_t& u1, int64_t& T) {
  T = 0;
  if constexpr (BALANCED) {
    // sequences with no block to read get their row here (spread over the
    // warps): zero, or in a cascade the shared prefix's result alone
    for (int64_t s = gw; ZERO_EMPTY && s < a.num_seqs && !a.q_start; s += NW) {
      if (seq_blocks<BS>(a, (int)s) == 0) {
        // a cascade's prefix partial comes from the grid this one may depend on
        if (a.pre) asm volatile("griddepcontrol.wait;" ::: "memory");
        QT* o = reinterpret_cast<QT*>(a.out) + (size_t)s * a.num_q_heads * D;
        for (int i = lane; i < a.num_q_heads * D; i += 32) {
          float v = 0.f;
          if (a.pre) {
            const float* pr = a.pre + ((size_t)s * a.num_q_heads + i / D) * pre_row_floats(D);
            const float l = pr[D + 1];
            v = l > 0.f ? pr[i % D] * (a.out_scale / l) : 0.f;
          }
          o[i] = from_f32<QT>(v);
        }
      }
    }
    // total tiles, this warp's range, and the sequence holding its first tile
    int64_t mine = 0;
    for (int s = lane; s < a.num_seqs; s += 32) mine += seq_blocks<BS>(a, s);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, off);
    T = mine * a.units;
    u0 = range_start(gw, T, NW);
    u1 = range_start(gw + 1, T, NW);
    if (u0 >= u1) return false;
    int s0 = a.num_seqs;
    int64_t p0 = 0, run = 0;  // tiles before the current chunk of 32 sequences
    for (int s = 0; s < a.num_seqs; s += 32) {
      const int64_t n = (s + lane < a.num_seqs) ? (int64_t)seq_blocks<BS>(a, s + lane) * a.units : 0;
      int64_t incl = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int64_t t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
      }
      const int64_t excl = incl - n;
      const unsigned hit = __ballot_sync(0xffffffffu, n > 0 && run + excl <= u0 && u0 < run + incl);
      if (hit) {
        const int src = __ffs(hit) - 1;
        s0 = s + src;
        p0 = __shfl_sync(0xffffffffu, run + excl, src);
        break;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (s0 >= a.num_seqs) return false;  // cannot happen for u0 < T
    wk0.s = s0;
    wk0.base = p0;
    wk0.nb = seq_blocks<BS>(a, s0);
    const int64_t off = u0 - p0;
    wk0.unit = (int)(off / wk0.nb);
    wk0.jb = (int)(off % wk0.nb);
    wk0.done = false;
    walker_settle<BS>(wk0, a, u1);
    return true;
  } else {
    // fixed partition p of segment seg, one per warp
    const int64_t segs = (int64_t)a.num_seqs * a.units;
    if (gw >= segs * a.max_partitions) return false;
    const int64_t seg = gw / a.max_partitions;
    const int p = (int)(gw % a.max_partitions);
    const int s = (int)(seg / a.units), unit = (int)(seg % a.units);
    const int nb = seq_blocks<BS>(a, s);
    const int jb = p * a.partition_blocks;
    const int je = min(nb, jb + a.partition_blocks);
    if (jb >= je) return false;
    wk0.s = s;
    wk0.unit = unit;
    wk0.nb = nb;
    wk0.base = 0;
    wk0.seg_u = (int64_t)unit * nb;
    wk0.jb = jb;
    wk0.je = je;
    wk0.done = false;
    u0 = wk0.seg_u + jb;
    u1 = wk0.seg_u + je;
    return true;
  }
}

// First query head of the unit a walker stands on.
__device__ __forceinline__ int unit_first_head(const DecodeArgs& a, const Walker& wk, int G) {
  const int kvh = wk.unit / a.units_per_kv, chunk = wk.unit % a.units_per_kv;
  return kvh * a.group + chunk * G;
}

// Multi-query: the query rows of sequence s (first row of q, token count);
// a count beyond the sequence, the host bound or the rows given is flagged
// and taken as 0 (the sequence's rows are left alone).
struct MqRows {
  int q0, T;
};
__device__ __forceinline__ MqRows mq_rows(const DecodeArgs& a, int s) {
  MqRows r;
  r.q0 = __ldg(a.q_start + s);
  r.T = __ldg(a.q_start + s + 1) - r.q0;
  const int L = seq_len_clipped(a, s);
  if (r.T < 0 || r.T > L || r.T > a.max_q || r.q0 < 0 || r.q0 + r.T > a.total_q) {
    raise_error(a.err, PKV_DEVERR_BAD_SEQ_LEN);
    r.T = 0;
  }
  return r;
}

// The partial-result slot of the piece a walker stands on: two per warp, the
// first for a piece that starts exactly at the warp's range (the tail of a
// segment begun by earlier warps), the second for any later piece.
template <int G, int D>
__device__ __forceinline__ float* partial_slot(const DecodeArgs& a, const Walker& wk, int64_t gw, int64_t u0) {
  const int64_t slot = (wk.seg_u + wk.jb == u0) ? 2 * gw : 2 * gw + 1;
  return a.partials + (size_t)slot * partial_slot_floats(G, D);
}

// ----------------------------------------------------------------------------
// Segments cut between warps.  A warp's cut pieces are at most its first
// piece (when its range starts inside a segment) and its last (when the range
// ends inside one).  The warp writes a cut piece's unnormalised
// (acc[G][D], m[G] in log2 units, l[G]) to its slot as soon as the piece ends
// -- plain stores, no wait -- and takes the segments' tickets only when its
// whole range is done, behind one fence; the last piece of a segment to take
// its ticket merges every piece by log-sum-exp and writes the output rows.
// Nothing waits for another warp.
// ----------------------------------------------------------------------------
struct CutPiece {
  int s, unit, nb;
  int64_t seg_u;  // linear index of the segment's first tile
  int q0, qT;     // multi-query: the sequence's first query row and row count
};

__device__ __forceinline__ CutPiece cut_piece_of(const Walker& wk, int q0 = 0, int qT = 0) {
  return CutPiece{wk.s, wk.unit, wk.nb, wk.seg_u, q0, qT};
}

// Draw the ticket of cut piece `cp` ahead of the range's end, behind a fence
// over this warp's partial-slot stores (issued a tile earlier, so the fence
// finds them landed).  The atomic's result is read only when the range is
// done: lane 0 holds it, the other lanes get -1.
__device__ __forceinline__ int draw_ticket(const DecodeArgs& a, const CutPiece& cp, int lane, bool async_readers) {
  if (async_readers) asm volatile("fence.proxy.async.global;" ::: "memory");
  __threadfence();
  __syncwarp();
  int t = -1;
  if (lane == 0) t = atomicAdd(a.counters + ((int64_t)cp.s * a.units + cp.unit), 1);
  return t;
}

// The output rows of a merged segment: lanes < D / 4 write dims 4 * lane ..
// 4 * lane + 3 of every row, num / den scaled by out_scale: rows h0 .. h0 +
// GW - 1 of the segment's G rows (held as den[hh], num[hh] for row h0 + hh).
template <class QT>
__device__ __forceinline__ void store4(QT* p, float x0, float x1, float x2, float x3);
template <>
__device__ __forceinline__ void store4<float>(float* p, float x0, float x1, float x2, float x3) {
  *reinterpret_cast<float4*>(p) = make_float4(x0, x1, x2, x3);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float x0, float x1, float x2, float x3) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(x0, x1), hi = __floats2bfloat162_rn(x2, x3);
  uint2 v;
  v.x = *reinterpret_cast<const uint32_t*>(&lo);
  v.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = v;
}

template <class QT, int G, int D, int GW = G>
__device__ __forceinline__ void write_merged(const DecodeArgs& a, const CutPiece& cp, int lane, const float (&den)[GW],
                                             const float (&num)[GW][4], int h0 = 0) {
  constexpr int DV = 4, SL = D / DV;
  const int d0 = (lane % SL) * DV;
  const int kvh = cp.unit / a.units_per_kv, chunk = cp.unit % a.units_per_kv;
#pragma unroll
  for (int hh = 0; hh < GW; ++hh) {
    const int h = h0 + hh;
    QT* out;
    if (a.q_start) {  // multi-query: row h is (token chunk * tpu + h / group, head h % group)
      const int tok = chunk * a.mq_tpu + h / a.group;
      if (tok >= cp.qT) continue;
      out = reinterpret_cast<QT*>(a.out) + ((size_t)(cp.q0 + tok) * a.num_q_heads + kvh * a.group + h % a.group) * D;
    } else {
      out = reinterpret_cast<QT*>(a.out) + ((size_t)cp.s * a.num_q_heads + kvh * a.group + chunk * G + h) * D;
    }
    if (lane < SL) {
      const float inv = den[hh] > 0.f ? a.out_scale / den[hh] : 0.f;
      store4<QT>(out + d0, num[hh][0] * inv, num[hh][1] * inv, num[hh][2] * inv, num[hh][3] * inv);
    }
  }
}

// Shared memory a warp lends to its merges once its own range is done: room
// for `cap` partial slots at `buf`, filled by bulk copies that complete on
// `bar` (`phase` = its completed phases).  buf == nullptr: merge through
// registers.
struct MergeStage {
  float* buf = nullptr;
  int cap = 0;
  uint64_t* bar = nullptr;
  uint32_t phase = 0;
};

// Merge all pieces of segment `cp` through shared memory: rounds of up to
// `cap` slots, each slot one bulk copy (accumulators, maxima and sums
// together), the rows combined online by log-sum-exp across rounds.  Every
// lane reads every piece (lanes < D / 4 own 4 dims, the maxima and sums are
// broadcast reads), so no cross-lane reduction follows.  False when a copy
// did not land in time (the error word is set; nothing is written).
template <class QT, int G, int D>
__device__ __forceinline__ bool merge_segment_staged(const DecodeArgs& a, const CutPiece& cp, int64_t T, int64_t NW,
                                                     int lane, MergeStage& ms) {
  constexpr int SLOT = partial_slot_floats(G, D), DV = 4, SL = D / DV;
  const int d0 = (lane % SL) * DV;
  const int64_t w_first = owner_of(cp.seg_u, T, NW), w_last = owner_of(cp.seg_u + cp.nb - 1, T, NW);
  const int64_t n = w_last - w_first + 1;
  const int64_t first_slot = (cp.seg_u != range_start(w_first, T, NW)) ? 2 * w_first + 1 : 2 * w_first;
  auto slot_of = [&](int64_t i) -> const float* {
    return a.partials + (size_t)(i == 0 ? first_slot : 2 * (w_first + i)) * SLOT;
  };
  float M[G], den[G], num[G][DV];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    M[h] = -CUDART_INF_F;
    den[h] = 0.f;
#pragma unroll
    for (int d = 0; d < DV; ++d) num[h][d] = 0.f;
  }
  for (int64_t i0 = 0; i0 < n; i0 += ms.cap) {
    const int cnt = (int)(n - i0 < ms.cap ? n - i0 : ms.cap);
    // the other pieces' slots were written by plain stores of other warps
    // (ordered before this warp's ticket); the copies read them through the
    // async proxy
    asm volatile("fence.proxy.async.global;" ::: "memory");
    fence_proxy_async_smem();  // earlier reads of the buffer before the copies overwrite it
    __syncwarp();
    if (lane == 0) {
      mbar_arrive_expect_tx(ms.bar, (uint32_t)(cnt * SLOT * sizeof(float)));
      for (int i = 0; i < cnt; ++i) bulk_g2s(ms.buf + (size_t)i * SLOT, slot_of(i0 + i), SLOT * sizeof(float), ms.bar);
    }
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(ms.bar, ms.phase & 1, a.err));
    ++ms.phase;
    if (!ok) {
      // leave no copy in flight: one more bounded wait for this round
      mbar_wait_bounded(ms.bar, (ms.phase - 1) & 1, a.err);
      ms.buf = nullptr;  // the buffer is no longer trusted
      return false;
    }
    for (int i = 0; i < cnt; ++i) {
      const float* pp = ms.buf + (size_t)i * SLOT;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float m = pp[G * D + h];
        const float Mn = fmaxf(M[h], m);
        if (Mn == -CUDART_INF_F) continue;  // nothing kept in this row yet
        const float f_old = fast_exp2(M[h] - Mn), f_new = fast_exp2(m - Mn);
        const float4 acc = *reinterpret_cast<const float4*>(pp + h * D + d0);
        den[h] = fmaf(den[h], f_old, f_new * pp[G * D + G + h]);
        num[h][0] = fmaf(num[h][0], f_old, f_new * acc.x);
        num[h][1] = fmaf(num[h][1], f_old, f_new * acc.y);
        num[h][2] = fmaf(num[h][2], f_old, f_new * acc.z);
        num[h][3] = fmaf(num[h][3], f_old, f_new * acc.w);
        M[h] = Mn;
      }
    }
  }
  write_merged<QT, G, D>(a, cp, lane, den, num);
  return true;
}

// A warp's share of a merge split over G / GW warps: rows h0 .. h0 + GW - 1
// of segment `cp`.  Per piece, three bulk copies land the rows' accumulators
// (GW x D floats) and their maxima and sums (GW floats each; GW a multiple of
// 4 keeps every copy a multiple of 16 bytes, 16-byte aligned) in this warp's
// buffer of `cap` pieces, completing on its own barrier `bar`; rows are
// combined online as in merge_segment_staged.  The warps of a merge share
// nothing.  False when a copy did not land in time (nothing is written).
template <class QT, int G, int D, int GW>
__device__ __forceinline__ bool merge_rows_staged(const DecodeArgs& a, const CutPiece& cp, int64_t T, int64_t NW,
                                                  int lane, float* buf, int cap, uint64_t* bar, int h0) {
  static_assert(GW % 4 == 0 && G % GW == 0, "row share");
  constexpr int SLOT = partial_slot_floats(G, D), DV = 4, SL = D / DV, PIECE = GW * D + 2 * GW;
  const int d0 = (lane % SL) * DV;
  const int64_t w_first = owner_of(cp.seg_u, T, NW), w_last = owner_of(cp.seg_u + cp.nb - 1, T, NW);
  const int64_t n = w_last - w_first + 1;
  const int64_t first_slot = (cp.seg_u != range_start(w_first, T, NW)) ? 2 * w_first + 1 : 2 * w_first;
  auto slot_of = [&](int64_t i) -> const float* {
    return a.partials + (size_t)(i == 0 ? first_slot : 2 * (w_first + i)) * SLOT;
  };
  float M[GW], den[GW], num[GW][DV];
#pragma unroll
  for (int hh = 0; hh < GW; ++hh) {
    M[hh] = -CUDART_INF_F;
    den[hh] = 0.f;
#pragma unroll
    for (int d = 0; d < DV; ++d) num[hh][d] = 0.f;
  }
  uint32_t phase = 0;
  for (int64_t i0 = 0; i0 < n; i0 += cap) {
    const int cnt = (int)(n - i0 < cap ? n - i0 : cap);
    // the slots were written by plain stores of the decode grid; the copies
    // read them through the async proxy
    asm volatile("fence.proxy.async.global;" ::: "memory");
    fence_proxy_async_smem();  // earlier reads of the buffer before the copies overwrite it
    __syncwarp();
    if (lane == 0) {
      mbar_arrive_expect_tx(bar, (uint32_t)(cnt * PIECE * sizeof(float)));
      for (int i = 0; i < cnt; ++i) {
        const float* src = slot_of(i0 + i);
        float* dst = buf + (size_t)i * PIECE;
        bulk_g2s(dst, src + h0 * D, GW * D * sizeof(float), bar);
        bulk_g2s(dst + GW * D, src + G * D + h0, GW * sizeof(float), bar);
        bulk_g2s(dst + GW * D + GW, src + G * D + G + h0, GW * sizeof(float), bar);
      }
    }
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar, phase & 1, a.err));
    ++phase;
    if (!ok) {
      mbar_wait_bounded(bar, (phase - 1) & 1, a.err);  // leave no copy in flight
      return false;
    }
    for (int i = 0; i < cnt; ++i) {
      const float* pp = buf + (size_t)i * PIECE;
#pragma unroll
      for (int hh = 0; hh < GW; ++hh) {
        const float m = pp[GW * D + hh];
        const float Mn = fmaxf(M[hh], m);
        if (Mn == -CUDART_INF_F) continue;  // nothing kept in this row yet
        const float f_old = fast_exp2(M[hh] - Mn), f_new = fast_exp2(m - Mn);
        const float4 acc = *reinterpret_cast<const float4*>(pp + hh * D + d0);
        den[hh] = fmaf(den[hh], f_old, f_new * pp[GW * D + GW + hh]);
        num[hh][0] = fmaf(num[hh][0], f_old, f_new * acc.x);
        num[hh][1] = fmaf(num[hh][1], f_old, f_new * acc.y);
        num[hh][2] = fmaf(num[hh][2], f_old, f_new * acc.z);
        num[hh][3] = fmaf(num[hh][3], f_old, f_new * acc.w);
        M[hh] = Mn;
      }
    }
  }
  write_merged<QT, G, D, GW>(a, cp, lane, den, num, h0);
  return true;
}

// Merge all pieces of segment `cp` (lane-parallel; lanes < D / 4 own 4 dims).
template <class QT, int G, int D>
__device__ __forceinline__ void merge_segment(const DecodeArgs& a, const CutPiece& cp, int64_t T, int64_t NW,
                                              int lane) {
  constexpr int SLOT = partial_slot_floats(G, D), DV = 4, SL = D / DV;
  constexpr int NB = G <= 2 ? 8 : (G == 4 ? 4 : (G <= 8 ? 2 : 1));  // pieces loaded per round trip
  const int d0 = (lane % SL) * DV;
  // pieces sit on warps w_first..w_last; the first one's slot depends on
  // whether the segment starts exactly at that warp's range
  const int64_t w_first = owner_of(cp.seg_u, T, NW), w_last = owner_of(cp.seg_u + cp.nb - 1, T, NW);
  const int64_t n = w_last - w_first + 1;
  const int64_t first_slot = (cp.seg_u != range_start(w_first, T, NW)) ? 2 * w_first + 1 : 2 * w_first;
  auto slot_of = [&](int64_t i) -> const float* {
    return a.partials + (size_t)(i == 0 ? first_slot : 2 * (w_first + i)) * SLOT;
  };
  float den[G], num[G][DV];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    den[h] = 0.f;
#pragma unroll
    for (int d = 0; d < DV; ++d) num[h][d] = 0.f;
  }
  if (n <= NB) {
    // the common case: every piece's (m, l, acc) in one round of loads
    float mm[NB][G], ll[NB][G];
    float4 oo[NB][G];
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const float* pp = slot_of(i < n ? i : 0);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        mm[i][h] = i < n ? ld_cg(pp + G * D + h) : -CUDART_INF_F;
        ll[i][h] = i < n ? ld_cg(pp + G * D + G + h) : 0.f;
        oo[i][h] = (i < n && lane < SL) ? ld_cg(reinterpret_cast<const float4*>(pp + h * D + d0))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float M = -CUDART_INF_F;
#pragma unroll
      for (int i = 0; i < NB; ++i) M = fmaxf(M, mm[i][h]);
      if (M == -CUDART_INF_F) M = 0.f;
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        const float f = fast_exp2(mm[i][h] - M);
        den[h] += f * ll[i][h];
        num[h][0] += f * oo[i][h].x;
        num[h][1] += f * oo[i][h].y;
        num[h][2] += f * oo[i][h].z;
        num[h][3] += f * oo[i][h].w;
      }
    }
  } else {
    // many pieces: lanes take slots for the maxima and weights, then the
    // accumulators stream in rounds of NB slots
    float M[G];
#pragma unroll
    for (int h = 0; h < G; ++h) M[h] = -CUDART_INF_F;
    for (int64_t i = lane; i < n; i += 32) {
      const float* pp = slot_of(i);
#pragma unroll
      for (int h = 0; h < G; ++h) M[h] = fmaxf(M[h], ld_cg(pp + G * D + h));
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) M[h] = fmaxf(M[h], __shfl_xor_sync(0xffffffffu, M[h], off));
      if (M[h] == -CUDART_INF_F) M[h] = 0.f;
    }
    for (int64_t base = 0; base < n; base += 32) {
      // lane i holds the weights of slot base + i
      float f[G];
      if (base + lane < n) {
        const float* pp = slot_of(base + lane);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          f[h] = fast_exp2(ld_cg(pp + G * D + h) - M[h]);
          den[h] += f[h] * ld_cg(pp + G * D + G + h);
        }
      } else {
#pragma unroll
        for (int h = 0; h < G; ++h) f[h] = 0.f;
      }
      const int cnt = (int)(n - base < 32 ? n - base : 32);
#pragma unroll 1
      for (int jj = 0; jj < cnt; jj += NB) {
        float4 oo[NB][G];
#pragma unroll
        for (int i = 0; i < NB; ++i) {
          const float* pp = slot_of(base + (jj + i < cnt ? jj + i : jj));
#pragma unroll
          for (int h = 0; h < G; ++h)
            oo[i][h] = (jj + i < cnt && lane < SL) ? ld_cg(reinterpret_cast<const float4*>(pp + h * D + d0))
                                                    : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < NB; ++i)
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float fj = __shfl_sync(0xffffffffu, f[h], (jj + i) & 31);
            const float w = jj + i < cnt ? fj : 0.f;
            num[h][0] += w * oo[i][h].x;
            num[h][1] += w * oo[i][h].y;
            num[h][2] += w * oo[i][h].z;
            num[h][3] += w * oo[i][h].w;
          }
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) den[h] += __shfl_xor_sync(0xffffffffu, den[h], off);
  }
  write_merged<QT, G, D>(a, cp, lane, den, num);
}

// Take the tickets of this warp's cut pieces (n of them, 0..2) behind one
// fence, then merge the segments whose last ticket this warp drew.
// drawn0: c0's ticket was drawn ahead (draw_ticket), its value in pre0 (lane 0).
template <class QT, int G, int D>
__device__ __forceinline__ void finish_cut_pieces(const DecodeArgs& a, const CutPiece& c0, const CutPiece& c1,
                                                  int n, int64_t T, int64_t NW, int lane,
                                                  MergeStage* ms = nullptr, bool drawn0 = false, int pre0 = -1) {
  if (n == 0) return;
  if (!drawn0 || n > 1) {
    // this warp's partial slots before its tickets (a merging warp may read
    // them through the async proxy)
    if (ms) asm volatile("fence.proxy.async.global;" ::: "memory");
    __threadfence();
  }
  __syncwarp();
  int last0 = 0, last1 = 0;
  if (lane == 0) {
    auto take = [&](const CutPiece& cp) -> int* {
      return a.counters + ((int64_t)cp.s * a.units + cp.unit);
    };
    auto pieces = [&](const CutPiece& cp) -> int {
      return (int)(owner_of(cp.seg_u + cp.nb - 1, T, NW) - owner_of(cp.seg_u, T, NW));
    };
    // both atomics in flight before either result is used
    const int t0 = drawn0 ? pre0 : atomicAdd(take(c0), 1);
    const int t1 = n > 1 ? atomicAdd(take(c1), 1) : -1;
    last0 = t0 == pieces(c0);
    last1 = n > 1 && t1 == pieces(c1);
    if (last0) *take(c0) = 0;  // ready for the next call
    if (last1) *take(c1) = 0;
  }
  last0 = __shfl_sync(0xffffffffu, last0, 0);
  last1 = __shfl_sync(0xffffffffu, last1, 0);
  if (last0 | last1) __threadfence();  // every other piece's slot before the reads
  auto merge = [&](const CutPiece& cp) {
    if (ms && ms->buf) {
      merge_segment_staged<QT, G, D>(a, cp, T, NW, lane, *ms);
    } else if (!ms) {
      merge_segment<QT, G, D>(a, cp, T, NW, lane);
    }
  };
  if (last0) merge(c0);
  if (last1) merge(c1);
}

}  // namespace pkv
