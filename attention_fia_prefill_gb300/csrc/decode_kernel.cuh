// Incremental (Q_S = 1) attention over a paged or contiguous KV cache.
//
// Operation: npu_fused_infer_attention_score_v2 / aclnnFusedInferAttentionScoreV5
// in the IncreFlashAttention case: out = softmax(scale * q K^T) V for one query
// token per (batch, head), with GQA (query head h reads kv head h / (Q_N/KV_N)),
// per-batch actual_seq_kvlen, and PageAttention (token j of batch b lives in
// block block_table[b][j / block_size], row j % block_size).
//
// Layout of the work:
//   * a unit is (batch, kv head) with its g = Q_N / KV_N query heads.  Every
//     unit's keys are cut into 128-token stages; the stages of all units are
//     dealt out to one CTA per SM with a fixed charge for every unit a CTA
//     starts (a "segment"), so every CTA streams about the same number of KV
//     bytes;
//   * the products are transposed so that the 128 keys of a stage, not the g
//     heads, fill the 128 rows of the tensor-core tile:
//         S^T = K Q^T   (M = 128 keys, N = G >= g heads, K = D), Q in smem
//         O^T = V^T P^T (M = D,        N = G heads,      K = 128 keys)
//     so a stage costs two thin MMAs, and a softmax thread owns one key and
//     all g heads of it;
//   * every P V writes a fresh O^T tile (two alternate in TMEM); the softmax
//     threads (thread = d for O^T) fold it into registers with the running
//     rescale, so O never has to be rescaled in TMEM and a segment boundary
//     does not drain the pipeline;
//   * one max per head is kept across the CTA's 128 keys: each stage the four
//     softmax warps publish their warp maxima and a vote ("does any key raise a
//     head's max by more than 2^8?") and meet at an mbarrier; only a yes
//     triggers a rescale;
//   * each segment leaves one partial (O / l, lse) per head; the CTA that
//     completes a unit (a per-unit counter tagged with the call's epoch)
//     merges the unit's partials in a fixed order -- deterministic, no float
//     atomics -- on its merge warp, off the softmax warps' path.
// Warps: 0..3 softmax, 4 K producer, 5 MMA issuer and TMEM owner, 6 V
// producer, 7 merge (unit counters and merges).
// TMEM columns: S^T buffers [0, G) and [G, 2G), O^T buffers [2G, 3G) and
// [3G, 4G).
#pragma once
#include "internal.h"
#include "ptx.cuh"

namespace fia {

constexpr int kDecodeSmemMax = 227 * 1024;

// GL: TMEM columns a softmax thread loads (>= g); G: MMA N (>= 16).
template <int D, int GL>
struct DecodeCfg {
  static constexpr int G = GL < 16 ? 16 : GL;
  static constexpr int kChunks = D / 64;
  static constexpr int kBoxBytes = 128 * 128;             // one 64-column box of 128 rows
  static constexpr int kTileBytes = kChunks * kBoxBytes;  // K (or V) of one 128-token stage
  static constexpr int kQBytes = kChunks * G * 128;       // Q tile: G rows x D, K-major
  static constexpr int kPBytes = 2 * G * 128;             // P^T tile: G rows x 128 keys, K-major
  static constexpr int kScratchBytes = 3 * G * 4 * 4;     // warp maxima (2 buffers) + warp sums
  static constexpr int kBarBytes = 512;
  // V^T spans M = 128 = two 64-wide boxes; with D = 64 a stage holds one, and
  // the second half of M reads the following box: a spare tile after the V
  // ring keeps that read inside the ring (those O^T rows are never used).
  static constexpr int kVPad = D == 64 ? kTileBytes : 0;
  static constexpr int kFixed = 2 * kQBytes + 2 * kPBytes + kScratchBytes + kBarBytes + 1024 + kVPad;
  static constexpr int kRing = (kDecodeSmemMax - kFixed) / kTileBytes;   // K + V stages that fit
  static constexpr int kKS = kRing / 2 + (kRing & 1) > 4 ? 4 : kRing / 2 + (kRing & 1);
  static constexpr int kVS = kRing / 2 > 4 ? 4 : kRing / 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKS * kTileBytes;
  static constexpr int kOffQ = kOffV + kVS * kTileBytes + kVPad;
  static constexpr int kOffP = kOffQ + 2 * kQBytes;
  static constexpr int kOffScratch = kOffP + 2 * kPBytes;
  static constexpr int kOffBar = kOffScratch + kScratchBytes;
  static constexpr int kSmem = kOffBar + kBarBytes + 1024;
  static constexpr int kThreads = 256;
  static constexpr uint32_t kTmemCols = 4 * G < 32 ? 32 : 4 * G;   // a power of two for G in {16, 32, 64}
  static constexpr uint32_t kColO = 2 * G;
  static_assert(kVS >= 2 && kKS >= 2, "rings too shallow");
  static_assert(kSmem <= kDecodeSmemMax, "shared memory budget");
  static_assert((kOffQ % 1024) == 0 && (kOffP % 1024) == 0, "swizzled tiles need 1024-byte alignment");
};

// Each group of MMAs (one Q K^T, one P V) ends with ONE tcgen05.commit -- a
// second commit straight after the first does not wait for the MMAs -- so its
// barrier serves every party that waits on it:
//   qk_done[j % KS]: S^T_j is in TMEM (softmax) and K slot j % KS is free;
//   pv_done[j % VS]: O^T_j is in TMEM (softmax) and V slot j % VS is free.
// p_full[j & 1]: the softmax warps' P^T_j is in shared memory.
// sync[j & 1]: the four softmax warps' maxima and votes of stage j are in.
// esync[s & 1]: the warps' sums of segment s are in (epilogue).
struct DecodeBars {
  uint64_t k_full[4], qk_done[4], v_full[4], pv_done[4];
  uint64_t p_full[2], q_ready[2], sync[2], esync[2];
  uint64_t part_done[4], part_free[4];   // softmax -> merge warp hand-off ring
  uint32_t tmem_holder;
  int abort_flag;
  int vote[2];
};

__device__ __forceinline__ const DecodeSeg* plan_segs(const DecodeParams& p) { return p.segs; }
__device__ __forceinline__ const int32_t* plan_cta(const DecodeParams& p) { return p.cta_seg; }
__device__ __forceinline__ const int2* plan_units(const DecodeParams& p) { return p.unit_parts; }
__device__ __forceinline__ const int32_t* plan_kvlen(const DecodeParams& p) { return p.kv_len; }

// Walks the CTA's stages in order and issues the TMA copies of one operand
// (K or V) into a ring of NS stages.  The whole warp runs it: the lanes cache
// 32 block_table entries of the current sequence so that a page lookup is a
// register shuffle, and lane 0 issues the copies.
template <int TileBytes, int BoxBytes, int Chunks, int NS>
__device__ __forceinline__ void decode_producer(const DecodeParams& p, const CUtensorMap* tm, uint8_t* ring,
                                                uint64_t* full, uint64_t* empty, volatile int* abort_flag,
                                                int seg_begin, int seg_end) {
  const int lane = threadIdx.x & 31;
  const DecodeSeg* segs = plan_segs(p);
  const int32_t* kvlen = plan_kvlen(p);
  if (lane == 0) tma_prefetch_desc(tm);
  int j = 0;
  bool ok = true;
  int pf_base = -64;          // page ids of the next segment, loaded one segment early
  int32_t pf_blk = 0;
  for (int si = seg_begin; si < seg_end && ok; ++si) {
    const DecodeSeg sg = segs[si];
    const int kvh = sg.unit % p.num_kv_heads;
    const int b = sg.unit / p.num_kv_heads;
    const int L = kvlen[b];
    int cache_base = pf_base;   // first page index held by the lanes' cache
    int32_t cache_blk = pf_blk; // lane i holds block_table[b][cache_base + i]
    pf_base = -64;
    if (p.block_table != nullptr && si + 1 < seg_end) {
      const DecodeSeg sn = segs[si + 1];
      pf_base = (sn.stage_begin * 128) / p.block_size;
      const int e = pf_base + lane;
      pf_blk = e < p.table_stride ? p.block_table[int64_t(sn.unit / p.num_kv_heads) * p.table_stride + e] : 0;
    }
    for (int st = sg.stage_begin; st < sg.stage_end; ++st, ++j) {
      const int s = j % NS;
      if (j >= NS && !__all_sync(0xffffffffu, mbar_wait(&empty[s], ((j / NS) - 1) & 1, abort_flag, p.status))) {
        ok = false;
        break;
      }
      const int t0 = st * 128;
      const int nvalid = min(128, L - t0);
      const int nbox = (nvalid + p.box_rows - 1) / p.box_rows;
      uint8_t* dst = ring + s * TileBytes;
      if (lane == 0) mbar_arrive_expect_tx(&full[s], uint32_t(Chunks * nbox * p.box_rows * 128));
      for (int k = 0; k < nbox; ++k) {
        const int tok = t0 + k * p.box_rows;
        int64_t row;
        if (p.block_table != nullptr) {
          const int page = tok / p.block_size;
          if (page < cache_base || page >= cache_base + 32) {
            cache_base = page;
            const int e = cache_base + lane;
            cache_blk = e < p.table_stride ? p.block_table[int64_t(b) * p.table_stride + e] : 0;
          }
          const int64_t blk = __shfl_sync(0xffffffffu, cache_blk, page - cache_base);
          row = blk * p.row_per_blk + int64_t(kvh) * p.row_per_head + (tok % p.block_size);
        } else {
          row = int64_t(b) * p.row_per_blk + int64_t(kvh) * p.row_per_head + tok;
        }
        if (lane == 0) {
#pragma unroll
          for (int c = 0; c < Chunks; ++c)
            tma_load_2d(dst + c * BoxBytes + k * p.box_rows * 128, tm, &full[s], kvh * p.col_per_head + c * 64,
                        int(row));
        }
      }
    }
  }
  if (lane == 0 && *abort_flag) {
    // let the copies already issued land before the CTA goes away
    for (int s = 0; s < NS && s < j; ++s) {
      const int last = j - 1 - ((j - 1 - s) % NS);
      mbar_wait(&full[s], (last / NS) & 1, nullptr, p.status);
    }
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
// lse = log sum_k exp(lse_k), out = sum_k exp(lse_k - lse) O_k.  Four heads at
// a time, lanes over D / 4 float4 columns; the lse values and the O rows of
// eight parts are loaded together, so a merge costs few L2 round trips.
template <int D, bool BF16>
__device__ __forceinline__ void merge_unit(const DecodeParams& p, int unit, int2 up, int lane) {
  constexpr int KB = 8;   // parts per batch of loads
  const int g = p.rows;   // rows of the unit: heads x query tokens
  const int kvh = unit % p.num_kv_heads, b = unit / p.num_kv_heads;
  const int64_t s0 = up.x;
  const int ns = up.y;
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
      float lk[4];
#pragma unroll
      for (int t = 0; t < 4; ++t)
        lk[t] = (h0 + t < g && lane < kn) ? __ldcg(p.part_lse + (s0 + k0 + lane) * g + h0 + t) : -INFINITY;
      float4 o[KB][4];
#pragma unroll
      for (int k = 0; k < KB; ++k)
#pragma unroll
        for (int t = 0; t < 4; ++t)
          o[k][t] = (k < kn && h0 + t < g && lane < D / 4)
                        ? __ldcg(reinterpret_cast<const float4*>(p.part_o + ((s0 + k0 + k) * g + h0 + t) * D) + lane)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
      // running max over the batches; rescale what is accumulated so far
      float wl[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float m_new = fmaxf(M[t], warp_max(lk[t]));
        const float a = (m_new == -INFINITY) ? 1.f : __expf(M[t] - m_new);
        acc[t].x *= a; acc[t].y *= a; acc[t].z *= a; acc[t].w *= a;
        M[t] = m_new;
        wl[t] = (lk[t] == -INFINITY) ? 0.f : __expf(lk[t] - m_new);
        Ls[t] = Ls[t] * a + warp_sum(wl[t]);
      }
#pragma unroll
      for (int k = 0; k < KB; ++k)
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float w = __shfl_sync(0xffffffffu, wl[t], k);
          acc[t].x += w * o[k][t].x; acc[t].y += w * o[k][t].y; acc[t].z += w * o[k][t].z; acc[t].w += w * o[k][t].w;
        }
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int hh = h0 + t;
      if (hh >= g) break;
      const int head = kvh * p.group + hh / p.q_tokens, tok = hh % p.q_tokens;
      if (lane < D / 4) {
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

// Q rows of one unit (g heads x D) into a swizzled K-major smem tile: the
// softmax threads each move up to QP 16-byte pieces; load and store are split
// so the global-load latency can overlap other work.
template <int D, int GL>
struct QPieces {
  static constexpr int kPer = (GL * D / 8 + 127) / 128;
  uint4 v[kPer];
};

template <int D, int GL>
__device__ __forceinline__ void q_load(const DecodeParams& p, int unit, int t, QPieces<D, GL>& q) {
  const int kvh = unit % p.num_kv_heads, b = unit / p.num_kv_heads;
  const uint16_t* qb = static_cast<const uint16_t*>(p.q) + int64_t(b) * p.q_sb;
#pragma unroll
  for (int i = 0; i < QPieces<D, GL>::kPer; ++i) {
    const int piece = t + 128 * i;
    const int row = piece / (D / 8);   // head kvh * group + row / Q_S, token row % Q_S
    if (row < p.rows) {
      const int head = kvh * p.group + row / p.q_tokens, tok = row % p.q_tokens;
      q.v[i] = *reinterpret_cast<const uint4*>(qb + int64_t(head) * p.q_sn + int64_t(tok) * p.q_ss +
                                               (piece % (D / 8)) * 8);
    }
  }
}

template <int D, int GL>
__device__ __forceinline__ void q_store(uint8_t* qtile, int g, int t, const QPieces<D, GL>& q) {
  constexpr int G = DecodeCfg<D, GL>::G;
#pragma unroll
  for (int i = 0; i < QPieces<D, GL>::kPer; ++i) {
    const int piece = t + 128 * i;
    if (piece < g * (D / 8)) {
      const int h = piece / (D / 8), col = (piece % (D / 8)) * 8;
      *reinterpret_cast<uint4*>(qtile + sw128_offset(h, col, G)) = q.v[i];
    }
  }
}

template <int D, bool BF16, int GL>
__global__ void __launch_bounds__(256, 1) decode_kernel(const __grid_constant__ DecodeParams p) {
  using C = DecodeCfg<D, GL>;
  constexpr int G = C::G;
  constexpr int KS = C::kKS, VS = C::kVS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  DecodeBars* bar = reinterpret_cast<DecodeBars*>(smem + C::kOffBar);
  float* red = reinterpret_cast<float*>(smem + C::kOffScratch);   // [2][G][4] warp maxima
  float* wsum = red + 2 * G * 4;                                   // [G][4] warp sums
  volatile int* abort_flag = &bar->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* cta_seg = plan_cta(p);
  const DecodeSeg* segs = plan_segs(p);
  const int2* unit_parts = plan_units(p);
  const int32_t* kvlen = plan_kvlen(p);
  const int seg_begin = p.n_cta > 0 ? cta_seg[blockIdx.x] : 0;
  const int seg_end = p.n_cta > 0 ? cta_seg[blockIdx.x + 1] : 0;
  const int g = p.rows;   // rows of a unit (of S^T's N): heads x query tokens

  if (threadIdx.x == 0) {
    if (blockIdx.x == 0) status_stamp(p.status);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bar->k_full[s], 1);
      mbar_init(&bar->qk_done[s], 1);
      mbar_init(&bar->v_full[s], 1);
      mbar_init(&bar->pv_done[s], 1);
      mbar_init(&bar->part_done[s], 4);
      mbar_init(&bar->part_free[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar->p_full[s], 4);
      mbar_init(&bar->q_ready[s], 4);
      mbar_init(&bar->sync[s], 4);
      mbar_init(&bar->esync[s], 4);
      bar->vote[s] = -1;
    }
    bar->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp < 4) {
    // rows g..G-1 of both Q tiles are never written again: zero them once
    for (int i = threadIdx.x; i < 2 * C::kQBytes / 16; i += 128) {
      const int off = i * 16;
      const int row = (off % (G * 128)) / 128;
      if (row >= g) *reinterpret_cast<uint4*>(smem + C::kOffQ + off) = make_uint4(0, 0, 0, 0);
    }
  }
  if (warp == 5) {
    tmem_alloc(&bar->tmem_holder, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_holder;

  if (warp == 4) {
    decode_producer<C::kTileBytes, C::kBoxBytes, C::kChunks, KS>(p, &p.tm_k, smem + C::kOffK, bar->k_full,
                                                                 bar->qk_done, abort_flag, seg_begin, seg_end);
  } else if (warp == 6) {
    decode_producer<C::kTileBytes, C::kBoxBytes, C::kChunks, VS>(p, &p.tm_v, smem + C::kOffV, bar->v_full,
                                                                 bar->pv_done, abort_flag, seg_begin, seg_end);
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
    int j = 0, segi = 0;
    bool ok = true;
    uint64_t* last_bar = nullptr;   // barrier and phase of the latest commit
    uint32_t last_parity = 0;
    // P V of stage jj (whose inputs are in); nvalid = its keys (< 128: clear the rest of V first)
    auto do_pv = [&](int jj, int nvalid) {
      const int s = jj % VS;
      if (nvalid < 128) {
        mbar_wait(&bar->v_full[s], (jj / VS) & 1, abort_flag, p.status);   // complete: an acquire per lane
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
        const uint32_t pb = p_base + (jj & 1) * C::kPBytes;
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk)
          mma_ss(tmem + C::kColO + (jj & 1) * G, smem_desc_sw128(vb + kk * 2048, v_lbo, 1024),
                 smem_desc_sw128(pb + (kk >> 2) * (G * 128) + (kk & 3) * 32, 16, 1024), idesc_pv,
                 kk > 0 ? 1u : 0u);
        mma_commit(&bar->pv_done[s]);
      }
      last_bar = &bar->pv_done[s];
      last_parity = (jj / VS) & 1;
    };
    // Each step issues Q K^T_j and P V_{j-1} in whichever order their inputs
    // arrive (the two are independent), so neither waits behind the other:
    // a segment's last P V does not wait for the next unit's first K tile,
    // nor Q K^T_j for a slow P_{j-1}.
    int prev_nvalid = 128;
    for (int si = seg_begin; si < seg_end && ok; ++si, ++segi) {
      const DecodeSeg sg = segs[si];
      const uint32_t qb = q_base + (segi & 1) * C::kQBytes;
      const int L = kvlen[sg.unit / p.num_kv_heads];
      bool q_ok = false;   // lane 0's view
      for (int st = sg.stage_begin; st < sg.stage_end && ok; ++st, ++j) {
        const int s = j % KS;
        bool qk = false, pv = (j == 0);
        const uint64_t t0 = globaltimer();
        while (!(qk && pv)) {
          int ev = 0;
          if (lane == 0) {
            if (!qk) {
              if (!q_ok) q_ok = mbar_test_wait(&bar->q_ready[segi & 1], (segi >> 1) & 1);
              if (q_ok && mbar_test_wait(&bar->k_full[s], (j / KS) & 1)) ev |= 1;
            }
            if (!pv && mbar_test_wait(&bar->p_full[(j - 1) & 1], ((j - 1) >> 1) & 1) &&
                mbar_test_wait(&bar->v_full[(j - 1) % VS], ((j - 1) / VS) & 1))
              ev |= 2;
            if (ev == 0) {
              if (*abort_flag) {
                ev = 4;
              } else if (globaltimer() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                status_raise(p.status, 10u /* FIA_ERR_TIMEOUT */);
                ev = 4;
              }
            }
          }
          ev = __shfl_sync(0xffffffffu, ev, 0);
          if (ev & 4) {
            ok = false;
            break;
          }
          if (ev & 1) {
            if (lane == 0) {
              tc_fence_after();
              const uint32_t kb = k_base + s * C::kTileBytes;
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk)
                mma_ss(tmem + (j & 1) * G, smem_desc_sw128(kb + (kk >> 2) * C::kBoxBytes + (kk & 3) * 32, 16, 1024),
                       smem_desc_sw128(qb + (kk >> 2) * (G * 128) + (kk & 3) * 32, 16, 1024), idesc_qk,
                       kk > 0 ? 1u : 0u);
              mma_commit(&bar->qk_done[s]);
            }
            last_bar = &bar->qk_done[s];
            last_parity = (j / KS) & 1;
            qk = true;
          }
          if (ev & 2) {
            do_pv(j - 1, prev_nvalid);
            pv = true;
          }
          if (ev == 0) __nanosleep(32);   // yield the issue slots: softmax warp 1 shares this scheduler
        }
        prev_nvalid = min(128, L - st * 128);
      }
    }
    if (ok && j > 0) {
      const int jj = j - 1;
      if (__all_sync(0xffffffffu, mbar_wait(&bar->p_full[jj & 1], (jj >> 1) & 1, abort_flag, p.status) &&
                                      mbar_wait(&bar->v_full[jj % VS], (jj / VS) & 1, abort_flag, p.status)))
        do_pv(jj, prev_nvalid);
    }
    // Every MMA issued has finished before TMEM goes: the latest commit
    // tracks them all (the one before it on the same barrier has completed,
    // so the barrier is at most one phase behind).
    if (last_bar != nullptr && lane == 0) mbar_wait(last_bar, last_parity, nullptr, p.status);
    __syncwarp();
  } else if (warp == 7) {
    // ------------------------------------------------------------ merge warp
    // After each segment's partials are out, bump the unit's counter; the CTA
    // that finishes a unit merges it here, off the softmax warps' path.
    bool ok = true;
    const int nseg = seg_end - seg_begin;
    for (int segi = 0; segi < nseg && ok; ++segi) {
      const DecodeSeg sg = segs[seg_begin + segi];
      if (!__all_sync(0xffffffffu, mbar_wait(&bar->part_done[segi & 3], (segi >> 2) & 1, abort_flag, p.status))) {
        ok = false;
        break;
      }
      if (lane == 0) mbar_arrive(&bar->part_free[segi & 3]);   // the slot may take segment segi + 4
      const int2 up = unit_parts[sg.unit];
      if (up.y == 1) continue;   // written directly by the softmax warps
      __threadfence();
      int last = 0;
      if (lane == 0) {
        unsigned long long* ctr = p.unit_counter + sg.unit;
        const unsigned long long tag = unit_tag(p.status.epoch);
        unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(ctr), nxt, prev;
        while (true) {
          nxt = ((cur & 0xffffffff00000000ull) == tag) ? cur + 1 : (tag | 1ull);
          prev = atomicCAS(ctr, cur, nxt);
          if (prev == cur) break;
          cur = prev;
        }
        last = int(nxt & 0xffffffffull) == up.y;
      }
      if (__shfl_sync(0xffffffffu, last, 0)) {
        __threadfence();
        merge_unit<D, BF16>(p, sg.unit, up, lane);
      }
    }
    // Units without any key (kv length 0): attention_out = 0, lse = +inf.
    // Spread over the CTAs: a serial walk over every unit's plan entry in
    // one CTA would hold the whole launch back.
    if (ok) {
      using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
      for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
        if (unit_parts[u].y != 0) continue;
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
  } else {
    // ------------------------------------------------------------ softmax
    // Thread r owns key r of each stage (row r of S^T and of P^T) and element
    // d = r of the head rows (row r of O^T).
    const int r = threadIdx.x;
    const uint32_t lane_off = uint32_t(32 * warp) << 16;
    const float sl2 = p.scale_log2;
    uint8_t* q_tiles = smem + C::kOffQ;
    uint8_t* p_tiles = smem + C::kOffP;
    bool ok = true;
    const int nseg = seg_end - seg_begin;

    // Q of the first two segments (buffers 0 and 1), both loads in flight
    {
      QPieces<D, GL> q0, q1;
      if (nseg > 0) q_load<D, GL>(p, segs[seg_begin].unit, r, q0);
      if (nseg > 1) q_load<D, GL>(p, segs[seg_begin + 1].unit, r, q1);
      if (nseg > 0) {
        q_store<D, GL>(q_tiles, g, r, q0);
        fence_proxy_async_smem();
        warp_arrive(&bar->q_ready[0]);
      }
      if (nseg > 1) {
        q_store<D, GL>(q_tiles + C::kQBytes, g, r, q1);
        fence_proxy_async_smem();
        warp_arrive(&bar->q_ready[1]);
      }
    }

    // A segment's partials are handed to the merge warp one stage later, so
    // the device-scope fence that makes them visible to other CTAs overlaps
    // work instead of stalling the softmax warps.
    int rel = -1;
    auto release = [&](int sidx) -> bool {
      __threadfence();
      // 4-slot ring: a slot is reused only after the merge warp took its
      // previous segment
      if (sidx >= 4 &&
          !__all_sync(0xffffffffu, mbar_wait(&bar->part_free[sidx & 3], ((sidx >> 2) - 1) & 1, abort_flag, p.status)))
        return false;
      warp_arrive(&bar->part_done[sidx & 3]);
      return true;
    };

    float m[GL], lp[GL], acc[GL];   // running max (log2 units), this key's sum of p, this d's O
    int j = 0;
    for (int segi = 0; segi < nseg && ok; ++segi) {
      const DecodeSeg sg = segs[seg_begin + segi];
      const int L = kvlen[sg.unit / p.num_kv_heads];
      const int first = j;
#pragma unroll
      for (int h = 0; h < GL; ++h) {
        m[h] = -INFINITY;
        lp[h] = 0.f;
        acc[h] = 0.f;
      }
      for (int st = sg.stage_begin; st < sg.stage_end; ++st, ++j) {
        // Q for segment segi + 1 goes into the buffer segment segi - 1 used;
        // its Q K^T products are complete once this segment's first S is.
        const bool next_q = (j == first) && segi >= 1 && segi + 1 < nseg;
        QPieces<D, GL> qn;
        if (next_q) q_load<D, GL>(p, segs[seg_begin + segi + 1].unit, r, qn);
        if (!__all_sync(0xffffffffu, mbar_wait(&bar->qk_done[j % KS], (j / KS) & 1, abort_flag, p.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (next_q) {
          q_store<D, GL>(q_tiles + ((segi + 1) & 1) * C::kQBytes, g, r, qn);
          fence_proxy_async_smem();
          warp_arrive(&bar->q_ready[(segi + 1) & 1]);
        }
        uint32_t su[GL];
        tmem_load_cols<GL>(tmem + lane_off + (j & 1) * G, su);
        const int nvalid = min(128, L - st * 128);
        const bool valid = r < nvalid;
        // several query tokens: row h is token h % Q_S, which sees keys up to
        // klim + h % Q_S (sparse_mode 3: klim = S_kv - Q_S; 2: klim = 0)
        const int klim = p.q_causal == 3 ? L - p.q_tokens : 0;
        const bool causal = p.q_causal != 0 && st * 128 + 127 > klim;   // a key of this stage is past a limit
        const int kfrom = st * 128 + r - klim;
        float s[GL];
        bool raise = false;
#pragma unroll
        for (int h = 0; h < GL; ++h) {
          bool live = valid && h < g;
          if (causal) live = live && kfrom <= h % p.q_tokens;
          s[h] = live ? __uint_as_float(su[h]) * sl2 : -INFINITY;
          raise |= s[h] > m[h] + 8.f;
        }
        // publish the warp maxima and the vote; meet the other three warps
        const int bsel = j & 1;
        float* rb = red + bsel * G * 4;
#pragma unroll
        for (int h = 0; h < GL; ++h) {
          if (h < g) {
            const float wm = warp_max_redux(s[h]);
            if (lane == (h & 31)) rb[h * 4 + warp] = wm;
          }
        }
        const bool any_w = __any_sync(0xffffffffu, raise);
        if (lane == 0) atomicMax(&bar->vote[bsel], (j << 1) | (any_w ? 1 : 0));
        warp_arrive(&bar->sync[bsel]);
        if (!__all_sync(0xffffffffu, mbar_wait(&bar->sync[bsel], (j >> 1) & 1, abort_flag, p.status))) {
          ok = false;
          break;
        }
        const bool any = *reinterpret_cast<volatile int*>(&bar->vote[bsel]) == ((j << 1) | 1);
        float alpha[GL];
#pragma unroll
        for (int h = 0; h < GL; ++h) {
          alpha[h] = 1.f;
          if (any && h < g) {
            const float4 w4 = *reinterpret_cast<const float4*>(rb + h * 4);
            const float m_new = fmaxf(m[h], fmaxf(fmaxf(w4.x, w4.y), fmaxf(w4.z, w4.w)));
            alpha[h] = (m_new == m[h]) ? 1.f : fast_exp2(m[h] - m_new);
            m[h] = m_new;
          }
        }
        // P^T row r (this key) of the stage, 16-bit, into tile j & 1
        uint8_t* pt = p_tiles + bsel * C::kPBytes;
#pragma unroll
        for (int h = 0; h < GL; ++h) {
          if (h < g) {
            const float mo = (m[h] == -INFINITY) ? 0.f : m[h];
            const float pv = (s[h] == -INFINITY) ? 0.f : fast_exp2(s[h] - mo);
            lp[h] = lp[h] * alpha[h] + pv;
            const uint32_t bits = pack2(pv, 0.f, BF16);
            *reinterpret_cast<uint16_t*>(pt + sw128_offset(h, r, G)) = uint16_t(bits & 0xffffu);
          }
        }
        fence_proxy_async_smem();   // P^T for the tensor core
        tc_fence_before();
        warp_arrive(&bar->p_full[bsel]);
        // fold O^T_{j-1} (relative to the previous max) into the registers,
        // then move everything to this stage's max
        if (j > first) {
          const int jp = j - 1;
          if (!__all_sync(0xffffffffu, mbar_wait(&bar->pv_done[jp % VS], (jp / VS) & 1, abort_flag, p.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t ou[GL];
          tmem_load_cols<GL>(tmem + lane_off + C::kColO + (jp & 1) * G, ou);
#pragma unroll
          for (int h = 0; h < GL; ++h) acc[h] += __uint_as_float(ou[h]);
        }
#pragma unroll
        for (int h = 0; h < GL; ++h) acc[h] *= alpha[h];
        if (rel >= 0) {
          if (!release(rel)) {
            ok = false;
            break;
          }
          rel = -1;
        }
      }
      if (!ok) break;
      // ---- segment epilogue: one partial (O / l, lse) per head
      {
        const int jp = j - 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&bar->pv_done[jp % VS], (jp / VS) & 1, abort_flag, p.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t ou[GL];
        tmem_load_cols<GL>(tmem + lane_off + C::kColO + (jp & 1) * G, ou);
#pragma unroll
        for (int h = 0; h < GL; ++h) acc[h] += __uint_as_float(ou[h]);
      }
      // l = sum over the 128 keys' partial sums
#pragma unroll
      for (int h = 0; h < GL; ++h) {
        if (h < g) {
          const float wsv = warp_sum(lp[h]);
          if (lane == (h & 31)) wsum[h * 4 + warp] = wsv;
        }
      }
      warp_arrive(&bar->esync[segi & 1]);
      if (!__all_sync(0xffffffffu, mbar_wait(&bar->esync[segi & 1], (segi >> 1) & 1, abort_flag, p.status))) {
        ok = false;
        break;
      }
      const int64_t part = sg.part;
      // a unit that lies in this one segment is final here: attention_out and
      // softmax_lse directly, no partial and no merge
      const bool whole = unit_parts[sg.unit].y == 1;
      const int kvh = sg.unit % p.num_kv_heads, b = sg.unit / p.num_kv_heads;
#pragma unroll
      for (int h = 0; h < GL; ++h) {
        if (h < g) {
          const float4 w4 = *reinterpret_cast<const float4*>(wsum + h * 4);
          const float l = (w4.x + w4.y) + (w4.z + w4.w);
          const bool has = l > 0.f;
          if (whole) {
            const int head = kvh * p.group + h / p.q_tokens, tok = h % p.q_tokens;
            if (r < D) {
              const uint32_t bits = pack2(has ? acc[h] / l : 0.f, 0.f, BF16);
              reinterpret_cast<uint16_t*>(p.out)[int64_t(b) * p.out_sb + int64_t(head) * p.out_sn +
                                                 int64_t(tok) * p.out_ss + r] = uint16_t(bits & 0xffffu);
            }
            if (r == h && p.lse != nullptr)
              p.lse[int64_t(b) * p.lse_sb + int64_t(head) * p.lse_sn + int64_t(tok) * p.lse_ss] =
                  has ? (m[h] + __log2f(l)) * 0.69314718055994531f : INFINITY;
          } else {
            if (r < D) p.part_o[(part * g + h) * D + r] = has ? acc[h] / l : 0.f;
            if (r == h) p.part_lse[part * g + h] = has ? (m[h] + __log2f(l)) * 0.69314718055994531f : -INFINITY;
          }
        }
      }
      if (rel >= 0 && !release(rel)) {
        ok = false;
        break;
      }
      rel = segi;
    }
    if (ok && rel >= 0) release(rel);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool BF16, int GL>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t s) {
  using C = DecodeCfg<D, GL>;
  auto k = decode_kernel<D, BF16, GL>;
  cudaError_t e = set_smem_once<decode_kernel<D, BF16, GL>>(C::kSmem);
  if (e != cudaSuccess) return e;
  k<<<p.n_cta > 0 ? p.n_cta : 1, C::kThreads, C::kSmem, s>>>(p);
  return cudaGetLastError();
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
