// Incremental attention (Q_S = 1..16 new tokens) over a paged or contiguous
// KV cache.
//
// Operation: npu_fused_infer_attention_score_v2 / aclnnFusedInferAttentionScoreV5
// in the IncreFlashAttention case: out = softmax(scale * q K^T) V for the new
// token(s) of each (batch, head), with GQA (query head h reads kv head
// h / (Q_N/KV_N)), per-batch actual_seq_kvlen, and PageAttention (token j of
// batch b lives in block block_table[b][j / block_size], row j % block_size).
//
// Layout of the work:
//   * a unit is (batch, kv head) with its rows = g query heads x Q_S tokens.
//     Every unit's keys are cut into 128-token stages; the host deals the
//     stages of all units to one CTA per SM with a fixed charge for every unit
//     piece a CTA starts (a "segment"), so every CTA streams about the same
//     number of KV bytes.  The plan rides in the kernel parameters;
//   * the products are transposed so the 128 keys of a stage, not the few
//     query rows, fill the 128 rows of the tensor-core tile:
//         S^T = K Q^T   (M = 128 keys, N = G >= rows, K = D), Q in smem
//         O^T = V^T P^T (M = D,        N = G,         K = 32 keys) per warp
//     A softmax thread owns one key (a row of S^T) and, for O^T, one element
//     d of every row;
//   * no exchange between the softmax warps: each warp exponentiates its 32
//     keys against their own maximum, and the P V of its keys goes to an O^T
//     tile of its own (the MMA issuer splits the stage's 128 keys into four
//     K = 32 products).  The warps leave their (maximum, sum) per row in
//     shared memory; one stage later every thread folds the four tiles into
//     its running output with the exact LSE weights, and computes the same
//     running maximum and sum as every other thread.  K and V stream side by
//     side: a ring slot is held only for its copy and a short softmax;
//   * each segment leaves one partial (O / l, lse) per row; the CTA that
//     completes a unit (a per-unit counter tagged with the call's epoch)
//     merges the unit's partials in a fixed order -- deterministic, no float
//     atomics -- on its merge warp, off the softmax warps' path.  A unit held
//     by one segment is written directly.
// Warps: 0..3 softmax (thread r: key r of a stage, element d = r of O^T),
// 4 K producer and Q loader, 5 MMA issuer and TMEM owner, 6 V producer,
// 7 merge.
// TMEM: S^T slots [G s, G (s + 1)) for s < NS, then O^T slots of 4 G
// columns (one G-wide tile per softmax warp) from column NS G.
//
// The kernel may be launched with programmatic stream serialisation: it lets
// the next kernel start launching at once, and every read of the inputs and
// every write of an output or the workspace follows grid_dep_wait().
#pragma once
#include "internal.h"
#include "ptx.cuh"

namespace fia {

constexpr int kDecodeSmemMax = 227 * 1024;
constexpr int kDecodeThreads = 256;

// GL: TMEM columns a softmax thread loads (>= rows); G: MMA N (>= 16).
template <int D, int GL>
struct DecodeCfg {
  static constexpr int G = GL < 16 ? 16 : GL;
  static constexpr int kChunks = D / 64;
  static constexpr int kBoxBytes = 128 * 128;             // one 64-column box of 128 rows
  static constexpr int kTileBytes = kChunks * kBoxBytes;  // K (or V) of one 128-token stage
  static constexpr int kQBytes = kChunks * G * 128;       // Q tile: G rows x D, K-major
  static constexpr int kPBytes = 2 * G * 128;             // P^T tile: G rows x 128 keys, K-major
  static constexpr int kNQ = G <= 16 ? 4 : 2;             // Q tiles (segments) in flight
  static constexpr int kNS = G <= 32 ? 4 : 2;             // S^T slots
  static constexpr int kNO = G <= 32 ? 3 : 1;             // O^T slots (4 G columns each)
  static constexpr int kColO = kNS * G;
  static constexpr uint32_t kTmemCols = (kNS * G + kNO * 4 * G) <= 256 ? 256 : 512;
  // per O slot: the maxima of 4 warps x G rows; then two buffers of the
  // warps' (running max, sum) per row for the segment epilogues
  static constexpr int kMLBytes = kNO * 4 * G * 4 + 2 * 4 * G * 8;
  static constexpr int kBarBytes = 512;
  // V^T spans M = 128 = two 64-wide boxes; with D = 64 a stage holds one, and
  // the second half of M reads the following box: a spare tile after the V
  // ring keeps that read inside the ring (those O^T rows are never used).
  static constexpr int kVPad = D == 64 ? kTileBytes : 0;
  static constexpr int kFixed = kNQ * kQBytes + kMLBytes + kBarBytes + 1024 + kVPad;
  static constexpr int kPerStage = 2 * kTileBytes + kPBytes;   // a K tile, a V tile and its P^T tile
  static constexpr int kFit = (kDecodeSmemMax - kFixed) / kPerStage;
  static constexpr int kVS = kFit > 4 ? 4 : kFit;
  static constexpr int kKSExtra = (kDecodeSmemMax - kFixed - kVS * kPerStage) / kTileBytes;
  // K slots <= S^T slots: a K slot is refilled on the S^T barrier of the
  // stage KS back, which must not have moved on by a whole turn of NS
  static constexpr int kKSMax = kNS < 6 ? kNS : 6;
  static constexpr int kKS = kVS + kKSExtra > kKSMax ? kKSMax : kVS + kKSExtra;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKS * kTileBytes;
  static constexpr int kOffQ = kOffV + kVS * kTileBytes + kVPad;
  static constexpr int kOffP = kOffQ + kNQ * kQBytes;
  static constexpr int kOffML = kOffP + kVS * kPBytes;
  static constexpr int kOffBar = kOffML + kMLBytes;
  static constexpr int kSmem = kOffBar + kBarBytes + 1024;
  static_assert(kVS >= 2 && kKS >= 2, "rings too shallow");
  static_assert(kNS * G + kNO * 4 * G <= 512, "TMEM columns");
  static_assert(kSmem <= kDecodeSmemMax, "shared memory budget");
  static_assert((kOffQ % 1024) == 0 && (kOffP % 1024) == 0, "swizzled tiles need 1024-byte alignment");
};

// Each group of MMAs (one Q K^T, one P V) ends with ONE tcgen05.commit -- a
// second commit straight after the first does not wait for the MMAs -- so its
// barrier serves every party that waits on it:
//   s_full[j % NS]:  S^T_j is in TMEM (softmax) and K slot j % KS is free
//                    (K producer);
//   pv_done[j % VS]: the P V products of stage j have finished: V slot and
//                    P^T tile j % VS are free, and O^T slot j % NO holds the
//                    stage's four tiles.
// p_full[j % VS]: the four softmax warps' P^T_j and (max, sum) of stage j are
// in shared memory, and S^T_j has been read (its slot may take stage j + NS).
// o_free[j % NO]: the four warps have folded stage j (its O^T slot and its
// (max, sum) slot may take stage j + NO).
// q_full / q_free[s % NQ]: Q of segment s is in its tile / all Q K^T products
// of segment s have finished.
struct DecodeBars {
  uint64_t k_full[6], v_full[4], pv_done[4], p_full[4];
  uint64_t s_full[4], o_free[3];
  uint64_t esync[2], efree[2];   // a segment's per-warp row sums published / consumed (by parity)
  uint64_t q_full[4], q_free[4];
  uint64_t part_done[4], part_free[4];   // softmax -> merge warp hand-off ring
  uint32_t tmem_holder;
  int abort_flag;
};

// The plan: 16-bit words in the kernel parameters, or 32-bit words in the
// workspace (layout in internal.h).
struct DecodePlanRef {
  const int16_t* w16;
  const int32_t* w32;
  int seg, unit, len;
  __device__ __forceinline__ int word(int i) const { return w32 != nullptr ? w32[i] : int(w16[i]); }
  __device__ __forceinline__ int cta_seg(int c) const { return word(c); }
  __device__ __forceinline__ DecodeSeg seg_at(int i) const {
    return DecodeSeg{word(seg + 4 * i), word(seg + 4 * i + 1), word(seg + 4 * i + 2), word(seg + 4 * i + 3)};
  }
  __device__ __forceinline__ int2 unit_parts(int u) const { return make_int2(word(unit + 2 * u), word(unit + 2 * u + 1)); }
  __device__ __forceinline__ int kv_len(int b) const {
    if (w32 != nullptr) return w32[len + b];
    return int(uint32_t(uint16_t(w16[len + 2 * b])) | (uint32_t(uint16_t(w16[len + 2 * b + 1])) << 16));
  }
};

__device__ __forceinline__ DecodePlanRef decode_plan(const DecodeParams& p) {
  DecodePlanRef r;
  r.w32 = p.plan_ws;
  r.w16 = p.plan_inline;
  r.seg = p.plan_seg;
  r.unit = p.plan_unit;
  r.len = p.plan_len;
  return r;
}

// Every lane waits; true only if all of them saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, const DevStatus st) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, st));
}

// Walks the CTA's stages in order and issues the TMA copies of one operand
// (K or V) into a ring of NS stages.  Stage j may refill its slot once the
// product that read stage j - NS has finished: barrier free[(j - NS) % FN],
// phase (j - NS) / FN.  The whole warp runs it: the lanes cache 32
// block_table entries of the current sequence so that a page lookup is a
// register shuffle, and lane 0 issues the copies.  With l2_ahead > 0 each
// stage's copy is followed by an L2 prefetch of the stage l2_ahead further on
// in the same segment, so a slot that frees up is refilled from L2.
//
// ql: the K producer's Q loader -- ql.issue(si, sg) starts the global loads
// of segment si's Q rows right after its first copies, ql.commit(si, sg)
// lands them in their tile (false: give up); the V producer passes a
// loader that does nothing.  Returns the number of stages whose copies it
// issued.
template <int TileBytes, int BoxBytes, int Chunks, int NS, int FN, typename QLoader>
__device__ __forceinline__ int decode_producer(const DecodeParams& p, const DecodePlanRef& pl, const CUtensorMap* tm,
                                               uint8_t* ring, uint64_t* full, uint64_t* free_bars,
                                               volatile int* abort_flag, int seg_begin, int seg_end, QLoader& ql) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) tma_prefetch_desc(tm);
  int j = 0;
  bool ok = true;
  int pf_base = -64;          // page ids of the next segment, loaded one segment early
  int32_t pf_blk = 0;
  for (int si = seg_begin; si < seg_end && ok; ++si) {
    const DecodeSeg sg = pl.seg_at(si);
    const int kvh = sg.unit % p.num_kv_heads;
    const int b = sg.unit / p.num_kv_heads;
    const int L = pl.kv_len(b);
    int cache_base = pf_base;   // first page index held by the lanes' cache
    int32_t cache_blk = pf_blk; // lane i holds block_table[b][cache_base + i]
    pf_base = -64;
    if (p.block_table != nullptr && si + 1 < seg_end) {
      const DecodeSeg sn = pl.seg_at(si + 1);
      pf_base = (sn.stage_begin * 128) / p.block_size;
      const int e = pf_base + lane;
      pf_blk = e < p.table_stride ? p.block_table[int64_t(sn.unit / p.num_kv_heads) * p.table_stride + e] : 0;
    }
    // map row of token tok of this sequence (the cache may be reloaded)
    auto row_of = [&](int tok) -> int64_t {
      if (p.block_table == nullptr) return int64_t(b) * p.row_per_blk + int64_t(kvh) * p.row_per_head + tok;
      const int page = tok / p.block_size;
      if (page < cache_base || page >= cache_base + 32) {
        cache_base = page;
        const int e = cache_base + lane;
        cache_blk = e < p.table_stride ? p.block_table[int64_t(b) * p.table_stride + e] : 0;
      }
      const int64_t blk = __shfl_sync(0xffffffffu, cache_blk, page - cache_base);
      return blk * p.row_per_blk + int64_t(kvh) * p.row_per_head + (tok % p.block_size);
    };
    for (int st = sg.stage_begin; st < sg.stage_end; ++st, ++j) {
      const int s = j % NS;
      if (j >= NS && !warp_wait(&free_bars[(j - NS) % FN], ((j - NS) / FN) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      const int t0 = st * 128;
      const int nvalid = min(128, L - t0);
      const int nbox = (nvalid + p.box_rows - 1) / p.box_rows;
      uint8_t* dst = ring + s * TileBytes;
      const bool first = st == sg.stage_begin;
      const int64_t row0 = row_of(t0);
      if (lane == 0) mbar_arrive_expect_tx(&full[s], uint32_t(Chunks * nbox * p.box_rows * 128));
      for (int k = 0; k < nbox; ++k) {
        const int64_t row = k == 0 ? row0 : row_of(t0 + k * p.box_rows);
        if (lane == 0) {
#pragma unroll
          for (int c = 0; c < Chunks; ++c)
            tma_load_2d(dst + c * BoxBytes + k * p.box_rows * 128, tm, &full[s], kvh * p.col_per_head + c * 64,
                        int(row));
        }
      }
      if (first) ql.issue(si - seg_begin, sg);   // Q's loads in flight behind the stage's copies
      // warm L2 with a later stage of this segment (pages outside the lanes'
      // cached window are skipped rather than reloaded)
      const int st2 = st + p.l2_ahead;
      if (p.l2_ahead > 0 && st2 < sg.stage_end) {
        const int u0 = st2 * 128;
        const int nbox2 = (min(128, L - u0) + p.box_rows - 1) / p.box_rows;
        for (int k = 0; k < nbox2; ++k) {
          const int tok = u0 + k * p.box_rows;
          int64_t row;
          if (p.block_table == nullptr) {
            row = int64_t(b) * p.row_per_blk + int64_t(kvh) * p.row_per_head + tok;
          } else {
            const int page = tok / p.block_size;
            if (page < cache_base || page >= cache_base + 32) break;
            const int64_t blk = __shfl_sync(0xffffffffu, cache_blk, page - cache_base);
            row = blk * p.row_per_blk + int64_t(kvh) * p.row_per_head + (tok % p.block_size);
          }
          if (lane == 0) {
#pragma unroll
            for (int c = 0; c < Chunks; ++c) tma_prefetch_l2_2d(tm, kvh * p.col_per_head + c * 64, int(row));
          }
        }
      }
      if (first && !ql.commit(si - seg_begin, sg)) {
        ok = false;
        ++j;   // this stage's copies are in flight
        break;
      }
    }
  }
  return j;
}

// Warms L2 with the K (or V) boxes of the first `nst` stages of segment sg.
// Run before griddepcontrol.wait, while the previous kernel on the stream may
// still be running on other SMs: a prefetch hands nothing to the kernel, so a
// block-table entry read here that the previous kernel later rewrites only
// wastes the prefetch (the copies after the wait read the table again), and
// L2 keeps lines that kernel writes coherent.  Coordinates past the pool are
// not fetched (the tensor map bounds them).  The whole warp runs it.
template <int Chunks>
__device__ __forceinline__ void l2_warm_segment(const DecodeParams& p, const DecodePlanRef& pl, const CUtensorMap* tm,
                                                const DecodeSeg& sg, int nst) {
  const int lane = threadIdx.x & 31;
  const int kvh = sg.unit % p.num_kv_heads;
  const int b = sg.unit / p.num_kv_heads;
  const int L = pl.kv_len(b);
  const int st_end = min(sg.stage_end, sg.stage_begin + nst);
  int page0 = 0;
  int32_t blk_lane = 0;   // lane i: block_table[b][page0 + i]
  if (p.block_table != nullptr) {
    page0 = (sg.stage_begin * 128) / p.block_size;
    const int e = page0 + lane;
    // through L2 only: a line of the table left in L1 here could be stale
    // for the reads after the wait
    blk_lane = e < p.table_stride ? __ldcg(p.block_table + int64_t(b) * p.table_stride + e) : 0;
  }
  for (int st = sg.stage_begin; st < st_end; ++st) {
    const int t0 = st * 128;
    const int nbox = (min(128, L - t0) + p.box_rows - 1) / p.box_rows;
    for (int k = 0; k < nbox; ++k) {
      const int tok = t0 + k * p.box_rows;
      int64_t row;
      if (p.block_table == nullptr) {
        row = int64_t(b) * p.row_per_blk + int64_t(kvh) * p.row_per_head + tok;
      } else {
        const int page = tok / p.block_size;
        if (page - page0 >= 32) return;   // past the lanes' window of table entries
        const int64_t blk = __shfl_sync(0xffffffffu, blk_lane, page - page0);
        row = blk * p.row_per_blk + int64_t(kvh) * p.row_per_head + (tok % p.block_size);
      }
      if (lane == 0) {
#pragma unroll
        for (int c = 0; c < Chunks; ++c) tma_prefetch_l2_2d(tm, kvh * p.col_per_head + c * 64, int(row));
      }
    }
  }
}

// After an abort, lets the copies of the first `issued` stages land before the
// CTA goes away (run once every role has stopped: a producer that finished
// its walk before another role gave up still has copies in flight).
template <int NS>
__device__ __forceinline__ void drain_ring(uint64_t* full, int issued, const DevStatus& st) {
  for (int s = 0; s < NS && s < issued; ++s) {
    const int last = issued - 1 - ((issued - 1 - s) % NS);
    mbar_wait(&full[s], (last / NS) & 1, nullptr, st);
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Maximum over the warp with one integer reduction: the float's bits mapped
// to an integer of the same order (negative values flip their magnitude bits).
__device__ __forceinline__ float warp_max_redux(float v) {
  const int u = __float_as_int(v);
  const int key = u ^ ((u >> 31) & 0x7fffffff);
  const int mk = __reduce_max_sync(0xffffffffu, key);
  return __int_as_float(mk ^ ((mk >> 31) & 0x7fffffff));
}

// Byte offset of element (row, col) in a K-major tile of 128-byte rows with
// the 128-byte swizzle, rows = `rows` per 64-column chunk (the layout TMA
// writes and the tcgen05 descriptors read).
__device__ __forceinline__ uint32_t sw128_offset(int row, int col, int rows) {
  const int chunk = col >> 6, c = col & 63;
  return uint32_t(chunk * rows * 128 + row * 128 + ((((c >> 3) ^ (row & 7))) << 4) + (c & 7) * 2);
}

// One warp merges the partials of a finished unit, in part order:
// lse = log sum_k exp(lse_k), out = sum_k exp(lse_k - lse) O_k.  Four rows at
// a time, lanes over D / 4 float4 columns; the O rows of four parts are loaded
// together, so a merge costs few L2 round trips.  Every lane reads the parts'
// lse words of its four rows itself (the same words in all lanes: one
// transaction each) and weighs the parts locally: no cross-lane reductions on
// the merge's critical path.
template <int D, bool BF16>
__device__ __forceinline__ void merge_unit(const DecodeParams& p, int unit, int2 up, int lane) {
  constexpr int KB = 4;   // parts per batch of loads
  const int g = p.rows;   // rows of the unit: heads x query tokens
  const int kvh = unit % p.num_kv_heads, b = unit / p.num_kv_heads;
  const int64_t s0 = up.x;
  const int ns = up.y;
  const bool col = lane < D / 4;
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  for (int h0 = 0; h0 < g; h0 += 4) {
    float M[4], Ls[4];
    float4 acc[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      M[t] = -INFINITY;
      Ls[t] = 0.f;
      acc[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int k0 = 0; k0 < ns; k0 += KB) {
      const int kn = ns - k0 < KB ? ns - k0 : KB;
      float lk[KB][4];
      float4 o[KB][4];
#pragma unroll
      for (int k = 0; k < KB; ++k)
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const bool v = k < kn && h0 + t < g;
          lk[k][t] = v ? __ldcg(p.part_lse + (s0 + k0 + k) * g + h0 + t) : -INFINITY;
          o[k][t] = (v && col) ? __ldcg(reinterpret_cast<const float4*>(p.part_o + ((s0 + k0 + k) * g + h0 + t) * D) + lane)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        float mb = lk[0][t];
#pragma unroll
        for (int k = 1; k < KB; ++k) mb = fmaxf(mb, lk[k][t]);
        const float m_new = fmaxf(M[t], mb);
        // rescale what is accumulated so far to the new maximum
        const float a = (m_new == -INFINITY) ? 1.f : __expf(M[t] - m_new);
        acc[t].x *= a; acc[t].y *= a; acc[t].z *= a; acc[t].w *= a;
        Ls[t] *= a;
#pragma unroll
        for (int k = 0; k < KB; ++k) {
          const float w = (lk[k][t] == -INFINITY) ? 0.f : __expf(lk[k][t] - m_new);
          Ls[t] += w;
          acc[t].x += w * o[k][t].x; acc[t].y += w * o[k][t].y; acc[t].z += w * o[k][t].z; acc[t].w += w * o[k][t].w;
        }
        M[t] = m_new;
      }
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int hh = h0 + t;
      if (hh >= g) break;
      const int head = kvh * p.group + hh / p.q_tokens, tok = hh % p.q_tokens;
      if (col) {
        const float inv = Ls[t] > 0.f ? 1.f / Ls[t] : 0.f;
        T* orow = reinterpret_cast<T*>(p.out) + int64_t(b) * p.out_sb + int64_t(head) * p.out_sn +
                  int64_t(tok) * p.out_ss + 4 * lane;
        uint2 w2;
        w2.x = pack2(acc[t].x * inv, acc[t].y * inv, BF16);
        w2.y = pack2(acc[t].z * inv, acc[t].w * inv, BF16);
        *reinterpret_cast<uint2*>(orow) = w2;
      }
      if (lane == 0 && p.lse != nullptr)
        p.lse[int64_t(b) * p.lse_sb + int64_t(head) * p.lse_sn + int64_t(tok) * p.lse_ss] =
            Ls[t] > 0.f ? M[t] + __logf(Ls[t]) : INFINITY;
    }
  }
}

template <int N>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 4) {
    tmem_ld4(taddr, r);
    tmem_wait_ld(r);
  } else if constexpr (N == 8) {
    tmem_ld8(taddr, r);
    tmem_wait_ld(r);
  } else if constexpr (N == 16) {
    tmem_ld16(taddr, r);
    tmem_wait_ld(r);
  } else if constexpr (N == 32) {
    tmem_ld32(taddr, r);
    tmem_wait_ld(r);
  } else {
    static_assert(N == 64, "column count");
    uint32_t a[32], b[32];
    tmem_ld32(taddr, a);
    tmem_ld32(taddr + 32, b);
    tmem_wait_ld(a);
    tmem_regs_after_wait(b);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      r[i] = a[i];
      r[32 + i] = b[i];
    }
  }
}

// Q rows of one unit (rows x D) into a swizzled K-major smem tile, by one
// warp.  issue() starts the global loads of the first 16 pieces (16 bytes)
// per lane; commit() waits for the tile to be free, stores them, copies any
// further pieces and publishes the tile.
template <int D, int G, int NQ>
struct DecodeQLoader {
  static constexpr int kPieceRow = D / 8;   // 16-byte pieces per row
  const DecodeParams& p;
  uint8_t* tiles;
  int qbytes;
  uint64_t* q_full;
  uint64_t* q_free;
  volatile int* abort_flag;
  uint4 v[16];

  __device__ __forceinline__ const uint4* src(int unit, int piece) const {
    const int kvh = unit % p.num_kv_heads, b = unit / p.num_kv_heads;
    const int row = piece / kPieceRow;   // head kvh * group + row / Q_S, token row % Q_S
    const int head = kvh * p.group + row / p.q_tokens, tok = row % p.q_tokens;
    const uint16_t* qb = static_cast<const uint16_t*>(p.q) + int64_t(b) * p.q_sb;
    return reinterpret_cast<const uint4*>(qb + int64_t(head) * p.q_sn + int64_t(tok) * p.q_ss +
                                          (piece % kPieceRow) * 8);
  }

  __device__ __forceinline__ void issue(int si, const DecodeSeg& sg) {
    const int lane = threadIdx.x & 31, n = p.rows * kPieceRow;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int piece = lane + 32 * i;
      if (piece < n) v[i] = *src(sg.unit, piece);
    }
  }

  __device__ __forceinline__ bool commit(int si, const DecodeSeg& sg) {
    const int lane = threadIdx.x & 31, n = p.rows * kPieceRow;
    const int slot = si % NQ;
    if (si >= NQ && !warp_wait(&q_free[slot], ((si / NQ) - 1) & 1, abort_flag, p.status)) return false;
    uint8_t* tile = tiles + slot * qbytes;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int piece = lane + 32 * i;
      if (piece < n)
        *reinterpret_cast<uint4*>(tile + sw128_offset(piece / kPieceRow, (piece % kPieceRow) * 8, G)) = v[i];
    }
    for (int base = 16 * 32; base < n; base += 16 * 32) {   // rows beyond the first 16 pieces per lane
      uint4 w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int piece = base + lane + 32 * i;
        if (piece < n) w[i] = *src(sg.unit, piece);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int piece = base + lane + 32 * i;
        if (piece < n)
          *reinterpret_cast<uint4*>(tile + sw128_offset(piece / kPieceRow, (piece % kPieceRow) * 8, G)) = w[i];
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&q_full[slot]);
    return true;
  }
};

struct NoQLoader {
  __device__ __forceinline__ void issue(int, const DecodeSeg&) {}
  __device__ __forceinline__ bool commit(int, const DecodeSeg&) { return true; }
};

// Units without any key (kv length 0): attention_out = 0, lse = +inf, by
// one warp per CTA.  Spread over the CTAs: a serial walk over every unit's
// plan entry in one CTA would hold the whole launch back.
template <int D, bool BF16>
__device__ __forceinline__ void write_empty_units(const DecodeParams& p, const DecodePlanRef& pl, int lane) {
  const int g = p.rows;
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
    if (pl.unit_parts(u).y != 0) continue;
    const int kvh = u % p.num_kv_heads, b = u / p.num_kv_heads;
    for (int hh = 0; hh < g; ++hh) {
      const int head = kvh * p.group + hh / p.q_tokens, tok = hh % p.q_tokens;
      if (lane < D / 4) {
        T* orow = reinterpret_cast<T*>(p.out) + int64_t(b) * p.out_sb + int64_t(head) * p.out_sn +
                  int64_t(tok) * p.out_ss + 4 * lane;
        *reinterpret_cast<uint2*>(orow) = make_uint2(0u, 0u);
      }
      if (lane == 0 && p.lse != nullptr)
        p.lse[int64_t(b) * p.lse_sb + int64_t(head) * p.lse_sn + int64_t(tok) * p.lse_ss] = INFINITY;
    }
  }
}

// The merge warp: after each segment's partials are out (part_done, one
// arrival per softmax warp), bump the unit's counter; the CTA that finishes
// a unit merges it, off the softmax warps' path.  Then writes the units
// without any key.
template <int D, bool BF16>
__device__ __forceinline__ void merge_warp(const DecodeParams& p, const DecodePlanRef& pl, uint64_t* part_done,
                                           uint64_t* part_free, volatile int* abort_flag, int seg_begin, int nseg,
                                           int lane) {
  bool ok = true;
  for (int segi = 0; segi < nseg && ok; ++segi) {
    const DecodeSeg sg = pl.seg_at(seg_begin + segi);
    if (!warp_wait(&part_done[segi & 3], (segi >> 2) & 1, abort_flag, p.status)) {
      ok = false;
      break;
    }
    if (lane == 0) mbar_arrive(&part_free[segi & 3]);   // the slot may take segment segi + 4
    const int2 up = pl.unit_parts(sg.unit);
    if (up.y == 1) continue;   // written directly by the softmax warps
    __threadfence();
    int last = 0;
    if (lane == 0) last = int(tagged_increment(p.unit_counter + sg.unit, unit_tag(p.status.epoch))) == up.y;
    if (__shfl_sync(0xffffffffu, last, 0)) {
      __threadfence();
      merge_unit<D, BF16>(p, sg.unit, up, lane);
    }
  }
  if (ok) write_empty_units<D, BF16>(p, pl, lane);
}

constexpr int kDecodeWarmStages = 4;   // stages warmed in L2 before the grid dependency resolves

template <int D, bool BF16, int GL>
__global__ void __launch_bounds__(kDecodeThreads, 1) decode_kernel(const __grid_constant__ DecodeParams p) {
  using C = DecodeCfg<D, GL>;
  constexpr int G = C::G;
  constexpr int KS = C::kKS, VS = C::kVS, NQ = C::kNQ, NS = C::kNS, NO = C::kNO;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  DecodeBars* bar = reinterpret_cast<DecodeBars*>(smem + C::kOffBar);
  float2* ml = reinterpret_cast<float2*>(smem + C::kOffML);   // maxima, then the sums buffers
  volatile int* abort_flag = &bar->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const DecodePlanRef pl = decode_plan(p);
  const int g = p.rows;   // rows of a unit (of S^T's N): heads x query tokens

  grid_dep_launch();
  if (threadIdx.x == 0) {
    for (int s = 0; s < KS; ++s) mbar_init(&bar->k_full[s], 1);
    for (int s = 0; s < VS; ++s) {
      mbar_init(&bar->v_full[s], 1);
      mbar_init(&bar->pv_done[s], 1);
      mbar_init(&bar->p_full[s], 4);
    }
    for (int s = 0; s < NS; ++s) mbar_init(&bar->s_full[s], 1);
    for (int s = 0; s < NO; ++s) mbar_init(&bar->o_free[s], 4);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar->esync[s], 4);
      mbar_init(&bar->efree[s], 4);
    }
    for (int s = 0; s < NQ; ++s) {
      mbar_init(&bar->q_full[s], 1);
      mbar_init(&bar->q_free[s], 1);
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bar->part_done[s], 4);
      mbar_init(&bar->part_free[s], 1);
    }
    bar->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp < 4) {
    // Q rows past the unit's and every P^T row: zero once (rows >= g are
    // never written again; their products land in unread columns)
    for (int i = threadIdx.x; i < (NQ * C::kQBytes + VS * C::kPBytes) / 16; i += 128)
      *reinterpret_cast<uint4*>(smem + C::kOffQ + i * 16) = make_uint4(0, 0, 0, 0);
  }
  if (warp == 5) {
    tmem_alloc(&bar->tmem_holder, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_holder;
  // L2 warm-up of the CTA's first stages while the previous kernel may still
  // run (a plan carried in the parameters only)
  if ((warp == 4 || warp == 6) && p.n_cta > 0 && p.plan_ws == nullptr) {
    const int sb = pl.cta_seg(blockIdx.x);
    if (sb < pl.cta_seg(blockIdx.x + 1))
      l2_warm_segment<C::kChunks>(p, pl, warp == 4 ? &p.tm_k : &p.tm_v, pl.seg_at(sb), kDecodeWarmStages);
  }
  grid_dep_wait();   // the previous kernel on the stream is complete from here on
  if (threadIdx.x == 0 && blockIdx.x == 0) status_stamp(p.status);
  // (a plan in the workspace was copied there on the stream: read it only now)
  const int seg_begin = p.n_cta > 0 ? pl.cta_seg(blockIdx.x) : 0;
  const int seg_end = p.n_cta > 0 ? pl.cta_seg(blockIdx.x + 1) : 0;
  const int nseg = seg_end - seg_begin;

  int issued = 0;   // producers: stages whose copies are in flight or landed
  if (warp == 4) {
    // K producer; it also loads each segment's Q rows into Q tile si % NQ
    // (free once the Q K^T products of segment si - NQ have finished)
    DecodeQLoader<D, G, NQ> ql{p, smem + C::kOffQ, C::kQBytes, bar->q_full, bar->q_free, abort_flag};
    issued = decode_producer<C::kTileBytes, C::kBoxBytes, C::kChunks, KS, NS>(
        p, pl, &p.tm_k, smem + C::kOffK, bar->k_full, bar->s_full, abort_flag, seg_begin, seg_end, ql);
  } else if (warp == 6) {
    NoQLoader nq;
    issued = decode_producer<C::kTileBytes, C::kBoxBytes, C::kChunks, VS, VS>(
        p, pl, &p.tm_v, smem + C::kOffV, bar->v_full, bar->pv_done, abort_flag, seg_begin, seg_end, nq);
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    // Lane 0 issues the tcgen05 work; the whole warp runs the loop so that,
    // before a ragged stage's P V, it can clear the V rows past the sequence
    // (a pool's unused rows may hold NaN, and P = 0 times NaN is not 0).
    constexpr uint32_t idesc_qk = idesc_f16(128, G, BF16 ? 1 : 0, 0, 0);   // K (M) and Q (N) K-major
    constexpr uint32_t idesc_pv = idesc_f16(128, G, BF16 ? 1 : 0, 1, 0);   // V^T MN-major, P^T K-major
    // V^T as the A operand: M = d runs along a V row, the second 64-wide half
    // of M is one box further (for D = 64: the next slot or the spare tile;
    // rows 64..127 of O^T are then not read).
    constexpr uint32_t v_lbo = C::kBoxBytes;
    const uint32_t k_base = smem_u32(smem + C::kOffK), v_base = smem_u32(smem + C::kOffV);
    const uint32_t q_base = smem_u32(smem + C::kOffQ), p_base = smem_u32(smem + C::kOffP);
    // cursors: Q K^T of stage jq (segment qsi, stage qst), P V of stage jp
    // (segment psi, stage pst); jpf stages have their P^T in (S slots free)
    int jq = 0, jp = 0, jpf = 0;
    int qsi = 0, psi = 0, qst = 0, pst = 0;
    DecodeSeg qsg{0, 0, 0, 0}, psg{0, 0, 0, 0};
    int pL = 0;
    if (nseg > 0) {
      qsg = psg = pl.seg_at(seg_begin);
      qst = pst = qsg.stage_begin;
      pL = pl.kv_len(psg.unit / p.num_kv_heads);
    }
    bool q_ok = false;   // lane 0's view: Q of segment qsi is in
    bool ok = true;
    uint64_t* last_bar = nullptr;   // barrier and phase of the latest commit
    uint32_t last_parity = 0;
    uint64_t t_last = cycles();
    while (ok && (qsi < nseg || psi < nseg)) {
      int ev = 0;
      if (lane == 0) {
        if (qsi < nseg && jq < jpf + NS) {
          if (!q_ok) q_ok = mbar_test_wait(&bar->q_full[qsi % NQ], (qsi / NQ) & 1);
          if (q_ok && mbar_test_wait(&bar->k_full[jq % KS], (jq / KS) & 1)) ev |= 1;
        }
        if (jpf < jq && mbar_test_wait(&bar->p_full[jpf % VS], (jpf / VS) & 1)) ev |= 4;
        if (jp < jpf + ((ev & 4) ? 1 : 0) && mbar_test_wait(&bar->v_full[jp % VS], (jp / VS) & 1) &&
            (jp < NO || mbar_test_wait(&bar->o_free[jp % NO], ((jp / NO) - 1) & 1)))
          ev |= 2;
        if (ev == 0) {
          if (*abort_flag) {
            ev = 8;
          } else if (cycles() - t_last > p.status.limit_ns * kCyclesPerNs) {
            *abort_flag = 1;
            status_raise(p.status, 10u /* FIA_ERR_TIMEOUT */);
            ev = 8;
          }
        }
      }
      ev = __shfl_sync(0xffffffffu, ev, 0);
      if (ev & 8) {
        ok = false;
        break;
      }
      if (ev & 1) {
        if (lane == 0) {
          tc_fence_after();
          const uint32_t kb = k_base + (jq % KS) * C::kTileBytes;
          const uint32_t qb = q_base + (qsi % NQ) * C::kQBytes;
          const uint32_t dcol = tmem + uint32_t(G) * uint32_t(jq % NS);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(dcol, smem_desc_sw128(kb + (kk >> 2) * C::kBoxBytes + (kk & 3) * 32, 16, 1024),
                   smem_desc_sw128(qb + (kk >> 2) * (G * 128) + (kk & 3) * 32, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
          mma_commit(&bar->s_full[jq % NS]);
        }
        last_bar = &bar->s_full[jq % NS];
        last_parity = (jq / NS) & 1;
        ++jq;
        if (++qst == qsg.stage_end) {
          q_ok = false;
          if (++qsi < nseg) {
            qsg = pl.seg_at(seg_begin + qsi);
            qst = qsg.stage_begin;
          }
        }
      }
      if (ev & 4) ++jpf;
      if (ev & 2) {
        const int s = jp % VS;
        const int nvalid = min(128, pL - pst * 128);
        if (nvalid < 128) {
          // every lane acquires the landed tile before clearing its tail rows
          mbar_wait(&bar->v_full[s], (jp / VS) & 1, abort_flag, p.status);
          uint8_t* vs = smem + C::kOffV + s * C::kTileBytes;
          for (int c = 0; c < C::kChunks; ++c)
            for (int u = lane; u < (128 - nvalid) * 8; u += 32)
              *reinterpret_cast<uint4*>(vs + c * C::kBoxBytes + (nvalid + (u >> 3)) * 128 + (u & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t vb = v_base + s * C::kTileBytes;
          const uint32_t pb = p_base + s * C::kPBytes;
          const uint32_t ocol = tmem + uint32_t(C::kColO) + uint32_t(4 * G) * uint32_t(jp % NO);
          // keys 32 w .. 32 w + 31 (softmax warp w) into O^T tile w
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk)
            mma_ss(ocol + uint32_t(G) * uint32_t(kk >> 1), smem_desc_sw128(vb + kk * 2048, v_lbo, 1024),
                   smem_desc_sw128(pb + (kk >> 2) * (G * 128) + (kk & 3) * 32, 16, 1024), idesc_pv,
                   (kk & 1) ? 1u : 0u);
          mma_commit(&bar->pv_done[s]);
        }
        last_bar = &bar->pv_done[s];
        last_parity = (jp / VS) & 1;
        ++jp;
        if (++pst == psg.stage_end) {
          if (++psi < nseg) {
            psg = pl.seg_at(seg_begin + psi);
            pst = psg.stage_begin;
            pL = pl.kv_len(psg.unit / p.num_kv_heads);
          }
        }
      }
      if (ev == 0) {
        __nanosleep(32);   // yield the issue slots to the softmax warp on this scheduler
      } else {
        t_last = cycles();
      }
    }
    // Every MMA issued has finished before TMEM goes: the latest commit
    // tracks them all.
    if (last_bar != nullptr && lane == 0) mbar_wait(last_bar, last_parity, nullptr, p.status);
    __syncwarp();
  } else if (warp == 7) {
    // ------------------------------------------------------------ merge warp
    merge_warp<D, BF16>(p, pl, bar->part_done, bar->part_free, abort_flag, seg_begin, nseg, lane);
  } else {
    // ------------------------------------------------------------ softmax
    // Thread r owns key r of each stage (row r of S^T and of P^T) and element
    // d = r of the unit's rows (row r of every O^T tile).
    const int r = threadIdx.x;
    const uint32_t lane_off = uint32_t(32 * warp) << 16;
    const float sl2 = p.scale_log2;
    uint8_t* p_tiles = smem + C::kOffP;
    bool ok = true;

    // A segment's partials are handed to the merge warp one stage later, so
    // the device-scope fence that makes them visible to other CTAs overlaps
    // work instead of stalling the softmax warps.
    int rel = -1;
    auto release = [&](int sidx) -> bool {
      __threadfence();
      // 4-slot ring: a slot is reused only after the merge warp took its
      // previous segment
      if (sidx >= 4 && !warp_wait(&bar->part_free[sidx & 3], ((sidx >> 2) - 1) & 1, abort_flag, p.status))
        return false;
      warp_arrive(&bar->part_done[sidx & 3]);
      return true;
    };

    // Two running states.  The fold's, for the segment being folded: the
    // maximum m (log2 units) of every row over the stages folded so far (the
    // same in every thread) and this d's output acc relative to it.  The
    // P pass's, for the segment being exponentiated: this warp's running
    // maximum mw_run of every row and this thread's keys' sum of p relative to
    // it; the rows' sums are combined across the warps once, at the
    // segment's end.  Rows h >= g compute on -inf scores (no keys): their
    // values are 0 / -inf and never stored.
    float m[GL], acc[GL], mw_run[GL], lp[GL];
#pragma unroll
    for (int h = 0; h < GL; ++h) {
      m[h] = -INFINITY;
      acc[h] = 0.f;
      mw_run[h] = -INFINITY;
      lp[h] = 0.f;
    }
    float* mls = reinterpret_cast<float*>(ml);   // [NO][4 warps][G] maxima
    float2* wsl = reinterpret_cast<float2*>(mls + NO * 4 * G);   // [2][4 warps][G] (running max, sum)
    // fold cursor: stage jf (segment fsi, stage fst of it)
    int jf = 0, fsi = 0, fst = 0;
    DecodeSeg fsg{0, 0, 0, 0};
    if (nseg > 0) {
      fsg = pl.seg_at(seg_begin);
      fst = fsg.stage_begin;
    }
    // Folds stage jf: the four warps' O^T tiles weighted by 2^(m_w - m_new)
    // into acc; at a segment's last stage also writes the segment's partial
    // (or the output) with the rows' sums exchanged at the end of its P pass.
    auto fold = [&]() -> bool {
      const int x = jf;
      const int os = x % NO;
      // P V of stage x and the warps' maxima of it: this thread has written
      // P up to stage x + 1 at most, so neither barrier can have moved on to
      // stage x + VS (VS >= 2)
      if (!warp_wait(&bar->pv_done[x % VS], (x / VS) & 1, abort_flag, p.status)) return false;
      if (!warp_wait(&bar->p_full[x % VS], (x / VS) & 1, abort_flag, p.status)) return false;
      tc_fence_after();
      const float* mx = mls + os * 4 * G;
      const uint32_t obase = tmem + lane_off + uint32_t(C::kColO) + uint32_t(4 * G) * uint32_t(os);
      if constexpr (GL <= 16) {
        float f0[GL], f1[GL], f2[GL], f3[GL];
#pragma unroll
        for (int h = 0; h < GL; ++h) {
          const float a0 = mx[h], a1 = mx[G + h], a2 = mx[2 * G + h], a3 = mx[3 * G + h];
          const float mn = fmaxf(fmaxf(m[h], fmaxf(a0, a1)), fmaxf(a2, a3));
          const float mo = mn == -INFINITY ? 0.f : mn;
          acc[h] *= fast_exp2(m[h] - mo);   // m = -inf: acc is 0 and the factor 0
          f0[h] = fast_exp2(a0 - mo);
          f1[h] = fast_exp2(a1 - mo);
          f2[h] = fast_exp2(a2 - mo);
          f3[h] = fast_exp2(a3 - mo);
          m[h] = mn;
        }
        // the four warps' tiles: four loads in flight, one wait
        uint32_t o0[GL], o1[GL], o2[GL], o3[GL];
        if constexpr (GL == 4) {
          tmem_ld4(obase, o0); tmem_ld4(obase + G, o1); tmem_ld4(obase + 2 * G, o2); tmem_ld4(obase + 3 * G, o3);
        } else if constexpr (GL == 8) {
          tmem_ld8(obase, o0); tmem_ld8(obase + G, o1); tmem_ld8(obase + 2 * G, o2); tmem_ld8(obase + 3 * G, o3);
        } else {
          tmem_ld16(obase, o0); tmem_ld16(obase + G, o1); tmem_ld16(obase + 2 * G, o2); tmem_ld16(obase + 3 * G, o3);
        }
        tmem_wait_ld(o0);
        tmem_regs_after_wait_n<GL>(o1);
        tmem_regs_after_wait_n<GL>(o2);
        tmem_regs_after_wait_n<GL>(o3);
#pragma unroll
        for (int h = 0; h < GL; ++h)
          acc[h] += (__uint_as_float(o0[h]) * f0[h] + __uint_as_float(o1[h]) * f1[h]) +
                    (__uint_as_float(o2[h]) * f2[h] + __uint_as_float(o3[h]) * f3[h]);
      } else {
        // wide tiles: the new maxima first, then one tile at a time
#pragma unroll
        for (int h = 0; h < GL; ++h) {
          const float mn = fmaxf(fmaxf(m[h], fmaxf(mx[h], mx[G + h])), fmaxf(mx[2 * G + h], mx[3 * G + h]));
          acc[h] *= fast_exp2(m[h] - (mn == -INFINITY ? 0.f : mn));
          m[h] = mn;
        }
#pragma unroll 1
        for (int w = 0; w < 4; ++w) {
          uint32_t ou[GL];
          tmem_load_cols<GL>(obase + uint32_t(G * w), ou);
#pragma unroll
          for (int h = 0; h < GL; ++h)
            acc[h] += __uint_as_float(ou[h]) * fast_exp2(mx[w * G + h] - (m[h] == -INFINITY ? 0.f : m[h]));
        }
      }
      tc_fence_before();   // O^T read before the slot takes stage x + NO
      warp_arrive(&bar->o_free[os]);
      ++jf;
      if (++fst < fsg.stage_end) return true;
      // ---- segment epilogue: one partial (O / l, lse) per row.  The rows'
      // sums (relative to each warp's running maximum) were published at the
      // end of the segment's P pass.
      if (!warp_wait(&bar->esync[fsi & 1], (fsi >> 1) & 1, abort_flag, p.status)) return false;
      const int64_t part = fsg.part;
      // a unit that lies in this one segment is final here: attention_out and
      // softmax_lse directly, no partial and no merge
      const bool whole = pl.unit_parts(fsg.unit).y == 1;
      const int kvh = fsg.unit % p.num_kv_heads, b = fsg.unit / p.num_kv_heads;
      const float2* ws = wsl + (fsi & 1) * 4 * G;
#pragma unroll
      for (int h = 0; h < GL; ++h) {
        if (h < g) {
          const float mo = m[h] == -INFINITY ? 0.f : m[h];
          float l = 0.f;
#pragma unroll
          for (int w = 0; w < 4; ++w) l += ws[w * G + h].y * fast_exp2(ws[w * G + h].x - mo);
          const bool has = l > 0.f;
          const float inv = has ? 1.f / l : 0.f;
          const float lse = has ? (m[h] + __log2f(l)) * 0.69314718055994531f : INFINITY;
          if (whole) {
            const int head = kvh * p.group + h / p.q_tokens, tok = h % p.q_tokens;
            if (r < D) {
              const uint32_t bits = pack2(acc[h] * inv, 0.f, BF16);
              reinterpret_cast<uint16_t*>(p.out)[int64_t(b) * p.out_sb + int64_t(head) * p.out_sn +
                                                 int64_t(tok) * p.out_ss + r] = uint16_t(bits & 0xffffu);
            }
            if (r == h && p.lse != nullptr)
              p.lse[int64_t(b) * p.lse_sb + int64_t(head) * p.lse_sn + int64_t(tok) * p.lse_ss] = lse;
          } else {
            if (r < D) p.part_o[(part * g + h) * D + r] = acc[h] * inv;
            if (r == h) p.part_lse[part * g + h] = has ? lse : -INFINITY;
          }
        }
        m[h] = -INFINITY;
        acc[h] = 0.f;
      }
      // the (max, sum) buffer of this segment's parity may take segment fsi + 2
      warp_arrive(&bar->efree[fsi & 1]);
      if (rel >= 0 && !release(rel)) return false;
      rel = fsi;
      if (++fsi < nseg) {
        fsg = pl.seg_at(seg_begin + fsi);
        fst = fsg.stage_begin;
      }
      return true;
    };
    // the end of a segment's P pass: publish this warp's (running max, sum)
    // of every row for the fold's epilogue
    auto publish_sums = [&](int segi) -> bool {
      // buffer segi & 1 is free once every warp's fold finished segment segi - 2
      if (segi >= 2 && !warp_wait(&bar->efree[segi & 1], ((segi >> 1) - 1) & 1, abort_flag, p.status)) return false;
      float2* dst = wsl + (segi & 1) * 4 * G + warp * G;
#pragma unroll
      for (int h = 0; h < GL; ++h) {
        const float sw = warp_sum(lp[h]);
        if (lane == (h & 31) && h < g) dst[h] = make_float2(mw_run[h], sw);
        mw_run[h] = -INFINITY;
        lp[h] = 0.f;
      }
      warp_arrive(&bar->esync[segi & 1]);
      return true;
    };

    int j = 0;   // stages whose P^T this thread has written
    for (int segi = 0; segi < nseg && ok; ++segi) {
      const DecodeSeg sg = pl.seg_at(seg_begin + segi);
      const int L = pl.kv_len(sg.unit / p.num_kv_heads);
      // several query tokens: row h is token h % Q_S, which sees keys up to
      // klim + h % Q_S (sparse_mode 3: klim = S_kv - Q_S; 2: klim = 0)
      const int klim = p.q_causal == 3 ? L - p.q_tokens : 0;
      const uint8_t* mrow = p.key_mask != nullptr
                                ? p.key_mask + int64_t(sg.unit / p.num_kv_heads) * p.key_mask_sb : nullptr;
      for (int st = sg.stage_begin; st < sg.stage_end; ++st, ++j) {
        const int ps = j % VS, os = j % NO;
        // this thread's key's atten_mask byte, read before the waits
        const bool kmasked = mrow != nullptr && r < L - st * 128 && __ldg(mrow + st * 128 + r) != 0;
        // one O^T slot (64 rows): every stage shares the maxima slot, so the
        // stage before is folded first
        if (NO == 1 && jf < j && !fold()) {
          ok = false;
          break;
        }
        // P^T tile free (P V of stage j - VS done), maxima slot free (all
        // warps folded stage j - NO), S^T_j in
        if ((j >= VS && !warp_wait(&bar->pv_done[ps], ((j / VS) - 1) & 1, abort_flag, p.status)) ||
            (j >= NO && !warp_wait(&bar->o_free[os], ((j / NO) - 1) & 1, abort_flag, p.status)) ||
            !warp_wait(&bar->s_full[j % NS], (j / NS) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t su[GL];
        tmem_load_cols<GL>(tmem + lane_off + uint32_t(G) * uint32_t(j % NS), su);
        // every Q K^T of the segment has finished once its last S^T is in
        if (st + 1 == sg.stage_end && warp == 0 && lane == 0) mbar_arrive(&bar->q_free[segi % NQ]);
        const bool valid = r < L - st * 128 && !kmasked;
        const bool causal = p.q_causal != 0 && st * 128 + 127 > klim;   // a key of this stage is past a limit
        const int kfrom = st * 128 + r - klim;
        uint8_t* pt = p_tiles + ps * C::kPBytes;
        float sv[GL], mw[GL];
#pragma unroll
        for (int h = 0; h < GL; ++h) {
          const bool live = valid && h < g && (!causal || kfrom <= h % p.q_tokens);
          sv[h] = live ? __uint_as_float(su[h]) * sl2 : -INFINITY;
        }
#pragma unroll
        for (int h = 0; h < GL; ++h) mw[h] = warp_max_redux(sv[h]);   // this warp's 32 keys
        float mine = -INFINITY;   // lane h publishes row h's maximum
#pragma unroll
        for (int h = 0; h < GL; ++h) {
          const float mo = mw[h] == -INFINITY ? 0.f : mw[h];
          const float pv = fast_exp2(sv[h] - mo);   // 0 for -inf scores
          const float nm = fmaxf(mw_run[h], mw[h]);
          const float no = nm == -INFINITY ? 0.f : nm;
          lp[h] = lp[h] * fast_exp2(mw_run[h] - no) + pv * fast_exp2(mw[h] - no);
          mw_run[h] = nm;
          if (lane == h) mine = mw[h];
          const uint32_t bits = pack2(pv, 0.f, BF16);
          *reinterpret_cast<uint16_t*>(pt + sw128_offset(h, r, G)) = uint16_t(bits & 0xffffu);
        }
        if (GL > 32) {
#pragma unroll
          for (int h = 32; h < GL; ++h)
            if (lane == h - 32) mls[(os * 4 + warp) * G + h] = mw[h];
        }
        if (lane < GL && lane < 32) mls[(os * 4 + warp) * G + lane] = mine;
        fence_proxy_async_smem();   // P^T for the tensor core
        tc_fence_before();          // and S^T_j read before its slot is reused
        warp_arrive(&bar->p_full[ps]);
        if (st + 1 == sg.stage_end && !publish_sums(segi)) {
          ok = false;
          break;
        }
        if (rel >= 0) {
          if (!release(rel)) {
            ok = false;
            break;
          }
          rel = -1;
        }
        // fold the stage before this one
        if (NO > 1 && jf < j && !fold()) {
          ok = false;
          break;
        }
      }
    }
    while (ok && jf < j) ok = fold();
    if (ok && rel >= 0) release(rel);
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && lane == 0) {
    if (warp == 4) drain_ring<KS>(bar->k_full, issued, p.status);
    if (warp == 6) drain_ring<VS>(bar->v_full, issued, p.status);
  }
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool BF16, int GL>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t s) {
  using C = DecodeCfg<D, GL>;
  cudaError_t e = set_smem_once<decode_kernel<D, BF16, GL>>(C::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_cta > 0 ? p.n_cta : 1);
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<D, BF16, GL>, p);
}

template <int D, bool BF16>
cudaError_t launch_decode_group(const DecodeParams& p, cudaStream_t s) {
  static_assert(sizeof(DecodeBars) <= 512, "barrier area too small");
  if (p.rows <= 4) return launch_decode_t<D, BF16, 4>(p, s);
  if (p.rows <= 8) return launch_decode_t<D, BF16, 8>(p, s);
  if (p.rows <= 16) return launch_decode_t<D, BF16, 16>(p, s);
  if (p.rows <= 32) return launch_decode_t<D, BF16, 32>(p, s);
  if (p.rows <= 64) return launch_decode_t<D, BF16, 64>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace fia
