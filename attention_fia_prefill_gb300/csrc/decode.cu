// Incremental (Q_S = 1) attention over a paged or contiguous KV cache.
//
// Operation: npu_fused_infer_attention_score_v2 / aclnnFusedInferAttentionScoreV5
// in the IncreFlashAttention case: out = softmax(scale * q K^T) V for one query
// token per (batch, head), with GQA (query head h reads kv head h / (Q_N/KV_N)),
// per-batch actual_seq_kvlen, and PageAttention (token j of batch b lives in
// block block_table[b][j / block_size], row j % block_size).
//
// Layout of the work:
//   * a unit is (batch, kv head).  The g = Q_N / KV_N query heads of the unit
//     are the rows of a 128-row query tile that lives in TMEM, in R = 4
//     (g <= 32) or R = 2 (g <= 64) copies; S = Q K^T and O += P V are tcgen05
//     MMAs with the A operand (Q, then P) read from TMEM;
//   * every unit's keys are cut into 128-token stages; the stages of all units,
//     in unit order, are dealt out to one CTA per SM with a fixed charge for
//     every unit a CTA starts (a "segment"), so every CTA streams about the
//     same number of KV bytes;
//   * copy c of the head rows owns 128 / R of each stage's key columns: the
//     four softmax warps share every stage, and each (segment, copy, head) is
//     an independent partial (O / l, lse) over its keys;
//   * two producer warps stream K (4-deep ring, freed after Q K^T) and V
//     (3-deep ring, freed after P V) with 2-D TMA loads, one per page segment;
//   * the CTA that completes a unit (a per-unit counter tagged with the call's
//     epoch) merges the unit's partials in a fixed order -- deterministic, no
//     float atomics -- on its merge warp, off the softmax warps' path, and
//     writes attention_out and softmax_lse.
// Warps: 0..3 softmax (warp w = TMEM lanes 32w..32w+31), 4 K producer, 5 MMA
// issuer and TMEM owner, 6 V producer, 7 merge (unit counters and merges).
// TMEM columns: S0 [0,128), S1 [128,256), O [256, 256+D), Q buffers
// [384, 384+D/2) and [384+D/2, 384+D).
#include "internal.h"
#include "ptx.cuh"

namespace fia {

template <int D>
struct DecodeCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kBoxBytes = 128 * 128;
  static constexpr int kTileBytes = kChunks * kBoxBytes;   // K (or V) of one 128-token stage
  static constexpr int kKS = 4;
  static constexpr int kVS = 3;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKS * kTileBytes;
  static constexpr int kOffBar = kOffV + kVS * kTileBytes;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmemUsed = kOffBar + kBarBytes + 1024;
  static constexpr int kSmem = kSmemUsed < 122880 ? 122880 : kSmemUsed;   // one CTA (and TMEM owner) per SM
  static constexpr int kThreads = 256;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;
  static constexpr uint32_t kColQ = 384;
};

// Each group of MMAs (one Q K^T, one P V) ends with ONE tcgen05.commit -- a
// second commit straight after the first does not wait for the MMAs -- so its
// barrier serves every party that waits on it:
//   qk_done[j % 4]: S_j is in TMEM (softmax) and K stage slot j % 4 is free
//                   (K producer);
//   pv_done[j % 3]: P_j V_j is accumulated in O (softmax rescale / epilogue)
//                   and V stage slot j % 3 is free (V producer).
// p_full[j & 1] takes the 128 softmax threads' arrivals for stage j.  A warp
// may run one stage ahead of the others (S_{j+1} can be ready before every
// warp has arrived for stage j), so consecutive stages use different
// barriers; two stages ahead is impossible (S_{j+2} needs P_j V_j issued).
struct DecodeBars {
  uint64_t k_full[4], qk_done[4], v_full[3], pv_done[3];
  uint64_t p_full[2], o_free, q_ready[2];
  uint64_t part_done[4], part_free[4];   // softmax -> merge warp hand-off ring
  uint32_t tmem_holder;
  int abort_flag;
};

__device__ __forceinline__ const DecodeSeg* plan_segs(const DecodeParams& p) {
  return p.plan_inline ? p.plan.segs : p.segs;
}
__device__ __forceinline__ const int32_t* plan_cta(const DecodeParams& p) {
  return p.plan_inline ? p.plan.cta_seg : p.cta_seg;
}
__device__ __forceinline__ const int2* plan_units(const DecodeParams& p) {
  return p.plan_inline ? p.plan.unit_parts : p.unit_parts;
}
__device__ __forceinline__ const int32_t* plan_kvlen(const DecodeParams& p) {
  return p.plan_inline ? p.plan.kv_len : p.kv_len;
}

// Walks the CTA's stages in order and issues the TMA copies of one operand
// (K or V) into a ring of NS stages.  The whole warp runs it: the lanes cache
// 32 block_table entries of the current sequence so that a page lookup is a
// register shuffle, and lane 0 issues the copies.
template <int D, int NS>
__device__ __forceinline__ void decode_producer(const DecodeParams& p, const CUtensorMap* tm, uint8_t* ring,
                                                uint64_t* full, uint64_t* empty, volatile int* abort_flag,
                                                int seg_begin, int seg_end) {
  using C = DecodeCfg<D>;
  const int lane = threadIdx.x & 31;
  const DecodeSeg* segs = plan_segs(p);
  const int32_t* kvlen = plan_kvlen(p);
  if (lane == 0) tma_prefetch_desc(tm);
  int j = 0;
  bool ok = true;
  for (int si = seg_begin; si < seg_end && ok; ++si) {
    const DecodeSeg sg = segs[si];
    const int kvh = sg.unit % p.num_kv_heads;
    const int b = sg.unit / p.num_kv_heads;
    const int L = kvlen[b];
    int cache_base = -64;     // first page index held by the lanes' cache
    int32_t cache_blk = 0;    // lane i holds block_table[b][cache_base + i]
    for (int st = sg.stage_begin; st < sg.stage_end; ++st, ++j) {
      const int s = j % NS;
      if (j >= NS && !__all_sync(0xffffffffu, mbar_wait(&empty[s], ((j / NS) - 1) & 1, abort_flag, p.status))) {
        ok = false;
        break;
      }
      const int t0 = st * 128;
      const int nvalid = min(128, L - t0);
      const int nbox = (nvalid + p.box_rows - 1) / p.box_rows;
      uint8_t* dst = ring + s * C::kTileBytes;
      if (lane == 0) mbar_arrive_expect_tx(&full[s], uint32_t(C::kChunks * nbox * p.box_rows * 128));
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
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_2d(dst + c * C::kBoxBytes + k * p.box_rows * 128, tm, &full[s], kvh * p.col_per_head + c * 64,
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

// Softmax threads write the query rows of one segment into a TMEM Q buffer as
// packed pairs: row r = copy r / (32 QD) of head r % (32 QD); rows past the
// group get zeros.  q_load issues the global loads and q_store the TMEM store,
// so the load latency can overlap other work.
template <int D>
struct QRow {
  uint4 v[D / 8];
};

template <int D>
__device__ __forceinline__ void q_load(const DecodeParams& p, int b, int kvh, int h, QRow<D>& q) {
  if (h < p.group) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                      (int64_t(b) * p.num_heads + kvh * p.group + h) * D);
#pragma unroll
    for (int i = 0; i < D / 8; ++i) q.v[i] = src[i];
  } else {
#pragma unroll
    for (int i = 0; i < D / 8; ++i) q.v[i] = make_uint4(0, 0, 0, 0);
  }
}

template <int D>
__device__ __forceinline__ void q_store(uint32_t taddr, const QRow<D>& q) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    uint32_t u[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      u[4 * i + 0] = q.v[c * 8 + i].x;
      u[4 * i + 1] = q.v[c * 8 + i].y;
      u[4 * i + 2] = q.v[c * 8 + i].z;
      u[4 * i + 3] = q.v[c * 8 + i].w;
    }
    tmem_st32(taddr + c * 32, u);
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

// One warp merges the partials of a finished unit, in sub-part order:
// lse = log sum_k exp(lse_k), out = sum_k exp(lse_k - lse) O_k.  Four heads at
// a time, lanes over D / 4 float4 columns; the lse values and the O rows of
// eight sub-parts are loaded together, so a merge costs few L2 round trips.
template <int D, bool BF16, int R>
__device__ __forceinline__ void merge_unit(const DecodeParams& p, int unit, int2 up, int lane) {
  constexpr int KB = 8;   // sub-parts per batch of loads
  const int g = p.group;
  const int kvh = unit % p.num_kv_heads, b = unit / p.num_kv_heads;
  const int64_t s0 = int64_t(up.x) * R;
  const int ns = up.y * R;
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
      const int head = kvh * g + hh;
      if (lane < D / 4) {
        const float inv = Ls[t] > 0.f ? 1.f / Ls[t] : 0.f;
        T* orow = reinterpret_cast<T*>(p.out) + int64_t(b) * p.out_sb + int64_t(head) * p.out_sn + 4 * lane;
        uint2 w2;
        w2.x = pack2(acc[t].x * inv, acc[t].y * inv, BF16);
        w2.y = pack2(acc[t].z * inv, acc[t].w * inv, BF16);
        *reinterpret_cast<uint2*>(orow) = w2;
      }
      if (lane == 0 && p.lse != nullptr)
        p.lse[int64_t(b) * p.lse_sb + int64_t(head) * p.lse_sn] = Ls[t] > 0.f ? M[t] + __logf(Ls[t]) : INFINITY;
    }
  }
}

template <int D, bool BF16, int R>
__global__ void __launch_bounds__(256, 1) decode_kernel(const __grid_constant__ DecodeParams p) {
  using C = DecodeCfg<D>;
  constexpr int KS = C::kKS, VS = C::kVS;
  constexpr int QD = 4 / R;            // TMEM lane quadrants (warps) per copy of the head rows
  constexpr int CW = 128 / R;          // key columns of a stage each copy handles
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  DecodeBars* bar = reinterpret_cast<DecodeBars*>(smem + C::kOffBar);
  volatile int* abort_flag = &bar->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* cta_seg = plan_cta(p);
  const DecodeSeg* segs = plan_segs(p);
  const int2* unit_parts = plan_units(p);
  const int32_t* kvlen = plan_kvlen(p);
  const int seg_begin = p.n_cta > 0 ? cta_seg[blockIdx.x] : 0;
  const int seg_end = p.n_cta > 0 ? cta_seg[blockIdx.x + 1] : 0;
  const int g = p.group;

  if (threadIdx.x == 0) {
    if (blockIdx.x == 0) status_stamp(p.status);
    for (int s = 0; s < KS; ++s) {
      mbar_init(&bar->k_full[s], 1);
      mbar_init(&bar->qk_done[s], 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(&bar->v_full[s], 1);
      mbar_init(&bar->pv_done[s], 1);
    }
    mbar_init(&bar->p_full[0], 128);
    mbar_init(&bar->p_full[1], 128);
    mbar_init(&bar->o_free, 128);
    mbar_init(&bar->q_ready[0], 128);
    mbar_init(&bar->q_ready[1], 128);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bar->part_done[s], 128);
      mbar_init(&bar->part_free[s], 1);
    }
    bar->abort_flag = 0;
    fence_mbar_init();
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
    decode_producer<D, KS>(p, &p.tm_k, smem + C::kOffK, bar->k_full, bar->qk_done, abort_flag, seg_begin, seg_end);
  } else if (warp == 6) {
    decode_producer<D, VS>(p, &p.tm_v, smem + C::kOffV, bar->v_full, bar->pv_done, abort_flag, seg_begin, seg_end);
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16(128, 128, BF16 ? 1 : 0, 0, 0);
      constexpr uint32_t idesc_pv = idesc_f16(128, D, BF16 ? 1 : 0, 0, 1);
      const uint32_t k_base = smem_u32(smem + C::kOffK), v_base = smem_u32(smem + C::kOffV);
      int j = 0, segi = 0;
      bool ok = true;
      uint64_t* last_bar = nullptr;   // barrier and phase of the latest commit
      uint32_t last_parity = 0;
      auto issue_pv = [&](int jj, int first, int seg_index) -> bool {
        const int s = jj % VS;
        if (jj == first && seg_index > 0 && !mbar_wait(&bar->o_free, (seg_index - 1) & 1, abort_flag, p.status))
          return false;
        if (!mbar_wait(&bar->p_full[jj & 1], (jj >> 1) & 1, abort_flag, p.status)) return false;
        if (!mbar_wait(&bar->v_full[s], (jj / VS) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint32_t vb = v_base + s * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk)
          mma_ts(tmem + C::kColO, tmem + (jj & 1) * 128 + kk * 8, smem_desc_sw128(vb + kk * 2048, C::kBoxBytes, 1024),
                 idesc_pv, (jj > first || kk > 0) ? 1u : 0u);
        mma_commit(&bar->pv_done[s]);
        last_bar = &bar->pv_done[s];
        last_parity = (jj / VS) & 1;
        return true;
      };
      for (int si = seg_begin; si < seg_end && ok; ++si, ++segi) {
        const DecodeSeg sg = segs[si];
        if (!mbar_wait(&bar->q_ready[segi & 1], (segi >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t qcol = C::kColQ + (segi & 1) * (D / 2);
        const int first = j;
        for (int st = sg.stage_begin; st < sg.stage_end; ++st, ++j) {
          const int s = j % KS;
          const int sb = j & 1;   // S buffer
          if (!mbar_wait(&bar->k_full[s], (j / KS) & 1, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kb = k_base + s * C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ts(tmem + sb * 128, tmem + qcol + kk * 8,
                   smem_desc_sw128(kb + (kk >> 2) * C::kBoxBytes + (kk & 3) * 32, 16, 1024), idesc_qk,
                   kk > 0 ? 1u : 0u);
          mma_commit(&bar->qk_done[s]);
          last_bar = &bar->qk_done[s];
          last_parity = (j / KS) & 1;
          if (j > first && !issue_pv(j - 1, first, segi)) { ok = false; break; }
        }
        if (!ok) break;
        if (j > first && !issue_pv(j - 1, first, segi)) { ok = false; break; }
      }
      // Every MMA issued has finished before TMEM goes: the latest commit
      // tracks them all (the one before it on the same barrier has completed,
      // so the barrier is at most one phase behind).
      if (last_bar != nullptr) mbar_wait(last_bar, last_parity, nullptr, p.status);
    }
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
      __threadfence();
      const int2 up = unit_parts[sg.unit];
      int last = 0;
      if (lane == 0) {
        unsigned long long* ctr = p.unit_counter + sg.unit;
        const unsigned long long tag = (p.status.epoch & 0xffffffffull) << 32;
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
        merge_unit<D, BF16, R>(p, sg.unit, up, lane);
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
          const int head = kvh * g + hh;
          if (lane < D / 4) {
            T* orow = reinterpret_cast<T*>(p.out) + int64_t(b) * p.out_sb + int64_t(head) * p.out_sn + 4 * lane;
            *reinterpret_cast<uint2*>(orow) = make_uint2(0u, 0u);
          }
          if (lane == 0 && p.lse != nullptr) p.lse[int64_t(b) * p.lse_sb + int64_t(head) * p.lse_sn] = INFINITY;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Warp w reads TMEM lanes 32w..32w+31.  Tile row r holds copy r / (32 QD)
    // of head r % (32 QD); the copy owns key columns [cp * CW, cp * CW + CW)
    // of every stage.
    const int r = 32 * warp + lane;
    const int cp = warp / QD;
    const int h = r - cp * 32 * QD;
    const int c0 = cp * CW;
    const uint32_t lane_off = uint32_t(32 * warp) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    const int nseg = seg_end - seg_begin;

    // Q of the first two segments (buffers 0 and 1)
    for (int k = 0; k < 2 && k < nseg; ++k) {
      const DecodeSeg sg = segs[seg_begin + k];
      QRow<D> q;
      q_load<D>(p, sg.unit / p.num_kv_heads, sg.unit % p.num_kv_heads, h, q);
      q_store<D>(tmem + lane_off + C::kColQ + k * (D / 2), q);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar->q_ready[k]);
    }

    // A segment's epilogue (read O, write the partial) runs after the next
    // segment's first stage: by then the segment's last P V has completed
    // (it was issued before that stage's Q K^T), so nothing waits for it.
    // That stage never touches O, and the next P V waits for o_free.  The
    // partial is handed to the merge warp one stage later again, so the
    // device-scope fence that makes it visible to other CTAs overlaps work.
    struct Pending {
      int segi, part, jlast;
      float m, l;
    };
    Pending epi{-1, 0, 0, 0.f, 0.f};
    int rel = -1;
    auto release = [&](int sidx) -> bool {
      __threadfence();
      // 4-slot ring: a slot is reused only after the merge warp took its
      // previous segment
      if (sidx >= 4 &&
          !__all_sync(0xffffffffu, mbar_wait(&bar->part_free[sidx & 3], ((sidx >> 2) - 1) & 1, abort_flag, p.status)))
        return false;
      mbar_arrive(&bar->part_done[sidx & 3]);
      return true;
    };
    // one partial (O / l, lse) per (copy, head) of segment epi.segi
    auto epilogue = [&]() -> bool {
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&bar->pv_done[epi.jlast % VS], (epi.jlast / VS) & 1, abort_flag, p.status)))
        return false;
      tc_fence_after();
      const bool has = epi.l > 0.f;
      const float inv_l = has ? 1.f / epi.l : 0.f;
      const int64_t sub = int64_t(epi.part) * R + cp;
      float* po = p.part_o + (sub * g + h) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem + lane_off + C::kColO + c * 32, u);
        tmem_wait_ld(u);
        if (c == D / 32 - 1) {
          tc_fence_before();
          mbar_arrive(&bar->o_free);     // the next segment's first P V may overwrite O now
        }
        if (h < g) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(po + c * 32 + 4 * q) =
                has ? make_float4(__uint_as_float(u[4 * q]) * inv_l, __uint_as_float(u[4 * q + 1]) * inv_l,
                                  __uint_as_float(u[4 * q + 2]) * inv_l, __uint_as_float(u[4 * q + 3]) * inv_l)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      if (h < g) p.part_lse[sub * g + h] = has ? (epi.m + __log2f(epi.l)) * 0.69314718055994531f : -INFINITY;
      rel = epi.segi;
      epi.segi = -1;
      return true;
    };
    // work deferred from earlier segments, done after a stage's P is handed over
    auto catch_up = [&]() -> bool {
      if (rel >= 0) {
        if (!release(rel)) return false;
        rel = -1;
      }
      return epi.segi < 0 || epilogue();
    };
    int j = 0;
    for (int segi = 0; segi < nseg && ok; ++segi) {
      const DecodeSeg sg = segs[seg_begin + segi];
      const int L = kvlen[sg.unit / p.num_kv_heads];
      const int first = j;
      float m = -INFINITY, l = 0.f;
      for (int st = sg.stage_begin; st < sg.stage_end; ++st, ++j) {
        const int sb = j & 1;
        // Q for segment segi + 1 goes into the buffer segment segi - 1 used;
        // its Q K^T products are complete once this segment's first S is.
        const bool next_q = (j == first) && segi >= 1 && segi + 1 < nseg;
        QRow<D> qn;
        if (next_q) {
          const DecodeSeg sn = segs[seg_begin + segi + 1];
          q_load<D>(p, sn.unit / p.num_kv_heads, sn.unit % p.num_kv_heads, h, qn);
        }
        if (!__all_sync(0xffffffffu, mbar_wait(&bar->qk_done[j % KS], (j / KS) & 1, abort_flag, p.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (next_q) {
          q_store<D>(tmem + lane_off + C::kColQ + ((segi + 1) & 1) * (D / 2), qn);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bar->q_ready[(segi + 1) & 1]);
        }
        uint32_t su[CW / 32][32];
#pragma unroll
        for (int c = 0; c < CW / 32; ++c) tmem_ld32(tmem + lane_off + sb * 128 + c0 + c * 32, su[c]);
        tmem_wait_ld(su[0]);
#pragma unroll
        for (int c = 1; c < CW / 32; ++c) tmem_regs_after_wait(su[c]);
        float x[CW];
#pragma unroll
        for (int c = 0; c < CW / 32; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(su[c][e]);
        const int nvalid = min(128, L - st * 128);
        if (nvalid < c0 + CW) {
#pragma unroll
          for (int c = 0; c < CW; ++c)
            if (c0 + c >= nvalid) x[c] = -INFINITY;
        }
        const float m_new = fmaxf(m, tree_max<CW>(x) * sl2);
        const float m_use = (m == -INFINITY || m_new > m + 8.f) ? m_new : m;
        const float alpha = (m_use == m) ? 1.f : fast_exp2(m - m_use);
        const float mo = (m_use == -INFINITY) ? 0.f : m_use;
        const float sum = exp2_and_sum<CW>(x, sl2, mo);
        l = l * alpha + sum;
        if (j > first && __any_sync(0xffffffffu, alpha != 1.f)) {
          if (!__all_sync(0xffffffffu,
                          mbar_wait(&bar->pv_done[(j - 1) % VS], ((j - 1) / VS) & 1, abort_flag, p.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t u[32];
            tmem_ld32(tmem + lane_off + C::kColO + c * 32, u);
            tmem_wait_ld(u);
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
            tmem_st32(tmem + lane_off + C::kColO + c * 32, u);
          }
        }
        // P row (packed pairs): this copy's CW keys at packed columns
        // [cp * CW / 2, (cp + 1) * CW / 2), zero in the other copies' columns.
        {
          uint32_t u[CW / 2], z[CW / 2];
#pragma unroll
          for (int e = 0; e < CW / 2; ++e) {
            u[e] = pack2(x[2 * e], x[2 * e + 1], BF16);
            z[e] = 0u;
          }
#pragma unroll
          for (int k = 0; k < R; ++k) {
            const uint32_t col = tmem + lane_off + sb * 128 + k * (CW / 2);
            if constexpr (CW == 32) {
              if (k == cp) tmem_st16(col, u); else tmem_st16(col, z);
            } else {
              if (k == cp) tmem_st32(col, u); else tmem_st32(col, z);
            }
          }
        }
        if (nvalid < 128) {
          // V rows past the sequence may hold anything (a pool's unused rows can
          // be NaN); P is 0 there but 0 * NaN is not, so clear them.
          const int s = j % VS;
          if (!__all_sync(0xffffffffu, mbar_wait(&bar->v_full[s], (j / VS) & 1, abort_flag, p.status))) {
            ok = false;
            break;
          }
          if (r >= nvalid) {
            uint8_t* vs = smem + C::kOffV + s * C::kTileBytes;
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
#pragma unroll
              for (int q = 0; q < 8; ++q)
                *reinterpret_cast<uint4*>(vs + c * C::kBoxBytes + r * 128 + q * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        tmem_wait_st();
        if (nvalid < 128) fence_proxy_async_smem();   // the cleared V rows, for the tensor core
        tc_fence_before();
        mbar_arrive(&bar->p_full[j & 1]);
        m = m_use;
        if (!catch_up()) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
      epi = Pending{segi, sg.part, j - 1, m, l};
    }
    if (ok) ok = catch_up();
    if (ok && rel >= 0) release(rel);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool BF16>
static cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t s) {
  using C = DecodeCfg<D>;
  auto k = p.copies == 2 ? decode_kernel<D, BF16, 2> : decode_kernel<D, BF16, 4>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  k<<<p.n_cta > 0 ? p.n_cta : 1, C::kThreads, C::kSmem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams& p, int head_dim, bool bf16, cudaStream_t s) {
  static_assert(sizeof(DecodeBars) <= DecodeCfg<128>::kBarBytes, "barrier area too small");
  if (head_dim == 128) return bf16 ? launch_decode_t<128, true>(p, s) : launch_decode_t<128, false>(p, s);
  if (head_dim == 64) return bf16 ? launch_decode_t<64, true>(p, s) : launch_decode_t<64, false>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace fia
