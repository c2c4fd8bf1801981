// MLA decode: incremental attention over a paged latent cache.
//
// Operation: npu_fused_infer_attention_score_v2 with query_rope / key_rope
// (the MLA case): the key of token j is [latent_j, rope_j] (512 + 64 = 576
// wide), its value is latent_j, and one kv head serves every query head:
//   out[h] = softmax_j(scale * ([q_h, qr_h] . [latent_j, rope_j])) latent_j.
//
// Layout of the work:
//   * a unit is a batch.  Its keys are cut into 32-token stages; the stages of
//     all units are dealt out to CTA pairs, so every pair streams about the
//     same number of cache bytes;
//   * the two CTAs of a pair run the same segments at the same time: each
//     computes S = Q' K'^T for all heads (M = 128 head rows, N = 32 keys, 576
//     deep; Q' = [q, q_rope] stays in shared memory for the segment) and the
//     softmax, and accumulates half h of the 512-wide output, O_h += P V_h
//     (N = 256), in TMEM.  Both read each cache tile at the same moment, so
//     the second read is served by L2;
//   * each segment leaves one partial (O_h / l, lse) per head; the CTA that
//     completes a (unit, half) merges its partials in a fixed order on its
//     merge warp; a unit held by one segment is written directly.
// Warps: 0..3 softmax (warp w = TMEM lanes 32w..32w+31 = head rows), 4 K'
// producer, 5 MMA issuer and TMEM owner, 6 Q' producer, 7 merge.
// TMEM columns: S buffers [0, 32) and [32, 64) (P overwrites the first 16 of
// its S as packed pairs), O_h [64, 320).
#include "internal.h"
#include "ptx.cuh"

namespace fia {
namespace {

constexpr int kMlaKeys = 32;                 // keys per stage
constexpr int kLatChunks = 8;                // 512 latent columns = 8 boxes of 64
constexpr int kKBox = kMlaKeys * 128;        // one 64-column box of 32 rows
constexpr int kKStage = (kLatChunks + 1) * kKBox;   // latent + rope of one stage: 36 KB
constexpr int kQBox = 128 * 128;             // one 64-column box of 128 head rows
constexpr int kQTile = (kLatChunks + 1) * kQBox;    // Q' = [q, q_rope]: 144 KB
constexpr int kOffK = 0;
constexpr int kOffQ = kOffK + 2 * kKStage;
constexpr int kOffBar = kOffQ + kQTile;
constexpr int kMlaSmem = kOffBar + 512 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 64;
constexpr int kHalf = 256;                   // output columns per CTA
constexpr int kPrefetch = 6;                 // stages ahead warmed in L2

struct MlaBars {
  uint64_t k_full[2], qk_done[2], pv_done[2], p_full[2];
  uint64_t q_full, q_empty, o_free;
  uint64_t part_done[4], part_free[4];
  uint32_t tmem_holder;
  int abort_flag;
};
static_assert(sizeof(MlaBars) <= 512, "barrier area");
static_assert(kMlaSmem <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ const DecodeSeg* mla_segs(const MlaParams& p) { return p.segs; }
__device__ __forceinline__ const int32_t* mla_cta(const MlaParams& p) { return p.cta_seg; }
__device__ __forceinline__ const int2* mla_units(const MlaParams& p) { return p.unit_parts; }
__device__ __forceinline__ const int32_t* mla_kvlen(const MlaParams& p) { return p.kv_len; }

__device__ __forceinline__ float mla_warp_max(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float mla_warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Merges the partials of (unit b, half) in part order (lanes over the 256
// columns, two float4 each; four heads at a time; loads batched by 4 parts).
template <bool BF16>
__device__ void mla_merge(const MlaParams& p, int b, int half, int2 up, int lane) {
  constexpr int KB = 4;
  const int nh = p.num_heads;
  const float* po = p.part_o + half * p.part_stride_o;
  const float* pl = p.part_lse + half * p.part_stride_lse;
  for (int h0 = 0; h0 < nh; h0 += 4) {
    float M[4], Ls[4];
    float4 acc[4][2];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      M[t] = -INFINITY;
      Ls[t] = 0.f;
      acc[t][0] = acc[t][1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int k0 = 0; k0 < up.y; k0 += KB) {
      const int kn = up.y - k0 < KB ? up.y - k0 : KB;
      float lk[4];
#pragma unroll
      for (int t = 0; t < 4; ++t)
        lk[t] = (h0 + t < nh && lane < kn) ? __ldcg(pl + int64_t(up.x + k0 + lane) * nh + h0 + t) : -INFINITY;
      float4 o[KB][4][2];
#pragma unroll
      for (int k = 0; k < KB; ++k)
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
          for (int c = 0; c < 2; ++c)
            o[k][t][c] = (k < kn && h0 + t < nh)
                             ? __ldcg(reinterpret_cast<const float4*>(po + (int64_t(up.x + k0 + k) * nh + h0 + t) * kHalf) +
                                      c * 32 + lane)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      float wl[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float m_new = fmaxf(M[t], mla_warp_max(lk[t]));
        const float a = (m_new == -INFINITY) ? 1.f : __expf(M[t] - m_new);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          acc[t][c].x *= a; acc[t][c].y *= a; acc[t][c].z *= a; acc[t][c].w *= a;
        }
        M[t] = m_new;
        wl[t] = (lk[t] == -INFINITY) ? 0.f : __expf(lk[t] - m_new);
        Ls[t] = Ls[t] * a + mla_warp_sum(wl[t]);
      }
#pragma unroll
      for (int k = 0; k < KB; ++k)
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float w = __shfl_sync(0xffffffffu, wl[t], k);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            acc[t][c].x += w * o[k][t][c].x; acc[t][c].y += w * o[k][t][c].y;
            acc[t][c].z += w * o[k][t][c].z; acc[t][c].w += w * o[k][t][c].w;
          }
        }
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int h = h0 + t;
      if (h >= nh) break;
      const float inv = Ls[t] > 0.f ? 1.f / Ls[t] : 0.f;
      uint16_t* orow = reinterpret_cast<uint16_t*>(p.out) + int64_t(b) * p.out_sb + int64_t(h) * p.out_sn + half * kHalf;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint2 w2;
        w2.x = pack2(acc[t][c].x * inv, acc[t][c].y * inv, BF16);
        w2.y = pack2(acc[t][c].z * inv, acc[t][c].w * inv, BF16);
        *reinterpret_cast<uint2*>(orow + (c * 32 + lane) * 4) = w2;
      }
      if (half == 0 && lane == 0 && p.lse != nullptr)
        p.lse[int64_t(b) * p.lse_sb + int64_t(h) * p.lse_sn] = Ls[t] > 0.f ? M[t] + __logf(Ls[t]) : INFINITY;
    }
  }
}

template <bool BF16>
__global__ void __launch_bounds__(256, 1) mla_kernel(const __grid_constant__ MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  MlaBars* bar = reinterpret_cast<MlaBars*>(smem + kOffBar);
  volatile int* abort_flag = &bar->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = blockIdx.x & 1, pair = blockIdx.x >> 1;
  const DecodeSeg* segs = mla_segs(p);
  const int32_t* cta_seg = mla_cta(p);
  const int2* unit_parts = mla_units(p);
  const int32_t* kvlen = mla_kvlen(p);
  const int seg_begin = p.n_pairs > 0 ? cta_seg[pair] : 0;
  const int seg_end = p.n_pairs > 0 ? cta_seg[pair + 1] : 0;
  const int nseg = seg_end - seg_begin;
  const int nh = p.num_heads;

  if (threadIdx.x == 0) {
    if (blockIdx.x == 0) status_stamp(p.status);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar->k_full[s], 1);
      mbar_init(&bar->qk_done[s], 1);
      mbar_init(&bar->pv_done[s], 1);
      mbar_init(&bar->p_full[s], 4);
    }
    mbar_init(&bar->q_full, 1);
    mbar_init(&bar->q_empty, 1);
    mbar_init(&bar->o_free, 4);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bar->part_done[s], 4);
      mbar_init(&bar->part_free[s], 1);
    }
    bar->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&bar->tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_holder;

  if (warp == 4) {
    // ------------------------------------------------------- K' producer
    // latent (8 boxes) + rope (1 box) of every 32-token stage into a 2-slot
    // ring; a slot is free once the stage's P V is done (it read V = latent).
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_lat);
      tma_prefetch_desc(&p.tm_rope);
    }
    int j = 0;
    bool ok = true;
    for (int si = seg_begin; si < seg_end && ok; ++si) {
      const DecodeSeg sg = segs[si];
      const int b = sg.unit;
      const int L = kvlen[b];
      int cache_base = -64;
      int32_t cache_blk = 0;
      for (int st = sg.stage_begin; st < sg.stage_end; ++st, ++j) {
        const int s = j & 1;
        if (j >= 2 &&
            !__all_sync(0xffffffffu, mbar_wait(&bar->pv_done[s], ((j >> 1) - 1) & 1, abort_flag, p.status))) {
          ok = false;
          break;
        }
        const int t0 = st * kMlaKeys;
        const int nvalid = min(kMlaKeys, L - t0);
        const int nbox = (nvalid + p.box_rows - 1) / p.box_rows;
        uint8_t* dst = smem + kOffK + s * kKStage;
        if (lane == 0) mbar_arrive_expect_tx(&bar->k_full[s], uint32_t((kLatChunks + 1) * nbox * p.box_rows * 128));
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
            row = blk * p.row_per_blk + (tok % p.block_size);
          } else {
            row = int64_t(b) * p.row_per_blk + tok;
          }
          if (lane == 0) {
#pragma unroll
            for (int c = 0; c < kLatChunks; ++c)
              tma_load_2d(dst + c * kKBox + k * p.box_rows * 128, &p.tm_lat, &bar->k_full[s], c * 64, int(row));
            tma_load_2d(dst + kLatChunks * kKBox + k * p.box_rows * 128, &p.tm_rope, &bar->k_full[s], 0, int(row));
          }
        }
        // The ring holds two stages only (Q' takes most of shared memory), so
        // the tiles kPrefetch stages ahead are pulled into L2 now: their loads
        // then wait for L2, not for HBM.
        const int pst = st + kPrefetch;
        if (pst < sg.stage_end) {
          const int ptok = pst * kMlaKeys;
          int64_t prow = -1;
          if (p.block_table != nullptr) {
            const int page = ptok / p.block_size;
            const bool cached = page >= cache_base && page < cache_base + 32;
            const int64_t blk = __shfl_sync(0xffffffffu, cache_blk, cached ? page - cache_base : 0);
            if (cached) prow = blk * p.row_per_blk + (ptok % p.block_size);
          } else {
            prow = int64_t(b) * p.row_per_blk + ptok;
          }
          if (lane == 0 && prow >= 0) {
#pragma unroll
            for (int c = 0; c < kLatChunks; ++c) tma_prefetch_l2_2d(&p.tm_lat, c * 64, int(prow));
            tma_prefetch_l2_2d(&p.tm_rope, 0, int(prow));
          }
        }
      }
    }
    if (lane == 0 && *abort_flag) {
      for (int s = 0; s < 2 && s < j; ++s) {
        const int last = j - 1 - ((j - 1 - s) & 1);
        mbar_wait(&bar->k_full[s], (last >> 1) & 1, nullptr, p.status);
      }
    }
  } else if (warp == 6) {
    // ------------------------------------------------------- Q' producer
    // Q' = [q, q_rope] of the segment's batch (all heads); the tile is reused
    // once the previous segment's last Q K'^T is done (q_empty, one arrival
    // per segment from the MMA warp).
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_qr);
      int issued = 0;
      for (int segi = 0; segi < nseg; ++segi) {
        const DecodeSeg sg = segs[seg_begin + segi];
        if (segi > 0 && !mbar_wait(&bar->q_empty, (segi - 1) & 1, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&bar->q_full, uint32_t(kQTile));
        const int row = sg.unit * nh;
#pragma unroll
        for (int c = 0; c < kLatChunks; ++c) tma_load_2d(smem + kOffQ + c * kQBox, &p.tm_q, &bar->q_full, c * 64, row);
        tma_load_2d(smem + kOffQ + kLatChunks * kQBox, &p.tm_qr, &bar->q_full, 0, row);
        ++issued;
      }
      if (*abort_flag && issued > 0) mbar_wait(&bar->q_full, (issued - 1) & 1, nullptr, p.status);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------- MMA issuer
    // Lane 0 issues; the whole warp clears, before a ragged stage's P V, the
    // latent rows past the sequence in its half (a cache's unused rows may
    // hold NaN, and P = 0 times NaN is not 0).
    constexpr uint32_t idesc_qk = idesc_f16(128, kMlaKeys, BF16 ? 1 : 0, 0, 0);
    constexpr uint32_t idesc_pv = idesc_f16(128, kHalf, BF16 ? 1 : 0, 0, 1);
    const uint32_t k_base = smem_u32(smem + kOffK), q_base = smem_u32(smem + kOffQ);
    int j = 0;
    bool ok = true;
    uint64_t* last_bar = nullptr;
    uint32_t last_parity = 0;
    // seg_last: jj is the segment's last stage.  Its P is in only after the
    // softmax saw S_jj, so every Q K'^T of the segment has completed and the
    // Q' tile may be refilled (q_empty).
    auto issue_pv = [&](int jj, int first, int segi, int nvalid, bool seg_last) -> bool {
      const int s = jj & 1;
      if (jj == first && segi > 0 &&
          !__all_sync(0xffffffffu, mbar_wait(&bar->o_free, (segi - 1) & 1, abort_flag, p.status)))
        return false;
      if (!__all_sync(0xffffffffu, mbar_wait(&bar->p_full[s], (jj >> 1) & 1, abort_flag, p.status))) return false;
      if (seg_last && lane == 0) mbar_arrive(&bar->q_empty);
      if (nvalid < kMlaKeys) {
        uint8_t* vs = smem + kOffK + s * kKStage + 4 * half * kKBox;
        for (int c = 0; c < 4; ++c)
          for (int u = lane; u < (kMlaKeys - nvalid) * 8; u += 32)
            *reinterpret_cast<uint4*>(vs + c * kKBox + (nvalid + (u >> 3)) * 128 + (u & 7) * 16) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        tc_fence_after();
        const uint32_t vb = k_base + s * kKStage + 4 * half * kKBox;
#pragma unroll
        for (int kk = 0; kk < kMlaKeys / 16; ++kk)
          mma_ts(tmem + kColO, tmem + s * 32 + kk * 8, smem_desc_sw128(vb + kk * 2048, kKBox, 1024), idesc_pv,
                 (jj > first || kk > 0) ? 1u : 0u);
        mma_commit(&bar->pv_done[s]);
      }
      last_bar = &bar->pv_done[s];
      last_parity = (jj >> 1) & 1;
      return true;
    };
    for (int segi = 0; segi < nseg && ok; ++segi) {
      const DecodeSeg sg = segs[seg_begin + segi];
      const int L = kvlen[sg.unit];
      if (!__all_sync(0xffffffffu, mbar_wait(&bar->q_full, segi & 1, abort_flag, p.status))) {
        ok = false;
        break;
      }
      const int first = j;
      int prev_nvalid = kMlaKeys;
      for (int st = sg.stage_begin; st < sg.stage_end; ++st, ++j) {
        const int s = j & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&bar->k_full[s], (j >> 1) & 1, abort_flag, p.status))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t kb = k_base + s * kKStage;
#pragma unroll
          for (int kk = 0; kk < (kLatChunks + 1) * 4; ++kk)
            mma_ss(tmem + s * 32, smem_desc_sw128(q_base + (kk >> 2) * kQBox + (kk & 3) * 32, 16, 1024),
                   smem_desc_sw128(kb + (kk >> 2) * kKBox + (kk & 3) * 32, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
          mma_commit(&bar->qk_done[s]);
        }
        last_bar = &bar->qk_done[s];
        last_parity = (j >> 1) & 1;
        if (j > first && !issue_pv(j - 1, first, segi, prev_nvalid, false)) {
          ok = false;
          break;
        }
        prev_nvalid = min(kMlaKeys, L - st * kMlaKeys);
      }
      if (!ok) break;
      if (!issue_pv(j - 1, first, segi, prev_nvalid, true)) ok = false;
    }
    if (last_bar != nullptr && lane == 0) mbar_wait(last_bar, last_parity, nullptr, p.status);
    __syncwarp();
  } else if (warp == 7) {
    // ------------------------------------------------------- merge warp
    bool ok = true;
    for (int segi = 0; segi < nseg && ok; ++segi) {
      const DecodeSeg sg = segs[seg_begin + segi];
      if (!__all_sync(0xffffffffu, mbar_wait(&bar->part_done[segi & 3], (segi >> 2) & 1, abort_flag, p.status))) {
        ok = false;
        break;
      }
      if (lane == 0) mbar_arrive(&bar->part_free[segi & 3]);
      const int2 up = unit_parts[sg.unit];
      if (up.y == 1) continue;   // written directly by the softmax warps
      __threadfence();
      int last = 0;
      if (lane == 0)
        last = int(tagged_increment(p.unit_counter + sg.unit * 2 + half, unit_tag(p.status.epoch))) == up.y;
      if (__shfl_sync(0xffffffffu, last, 0)) {
        __threadfence();
        mla_merge<BF16>(p, sg.unit, half, up, lane);
      }
    }
    // batches without keys: attention_out = 0, lse = +inf (spread over the pairs)
    if (ok) {
      const int npair = p.n_pairs > 0 ? p.n_pairs : 1;
      for (int b = pair; b < p.n_units; b += npair) {
        if (unit_parts[b].y != 0) continue;
        for (int h = 0; h < nh; ++h) {
          uint16_t* orow = reinterpret_cast<uint16_t*>(p.out) + int64_t(b) * p.out_sb + int64_t(h) * p.out_sn + half * kHalf;
          *reinterpret_cast<uint4*>(orow + lane * 8) = make_uint4(0, 0, 0, 0);
          if (half == 0 && lane == 0 && p.lse != nullptr) p.lse[int64_t(b) * p.lse_sb + int64_t(h) * p.lse_sn] = INFINITY;
        }
      }
    }
  } else {
    // ------------------------------------------------------- softmax
    // thread r = head row r of S (TMEM lane r)
    const int r = threadIdx.x;
    const uint32_t lane_off = uint32_t(32 * warp) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    int j = 0;
    for (int segi = 0; segi < nseg && ok; ++segi) {
      const DecodeSeg sg = segs[seg_begin + segi];
      const int L = kvlen[sg.unit];
      const int first = j;
      float m = -INFINITY, l = 0.f;
      for (int st = sg.stage_begin; st < sg.stage_end; ++st, ++j) {
        const int sb = j & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&bar->qk_done[sb], (j >> 1) & 1, abort_flag, p.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t su[32];
        tmem_ld32(tmem + lane_off + sb * 32, su);
        tmem_wait_ld(su);
        float x[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) x[c] = __uint_as_float(su[c]);
        const int nvalid = min(kMlaKeys, L - st * kMlaKeys);
        if (nvalid < kMlaKeys) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c >= nvalid) x[c] = -INFINITY;
        }
        const float m_new = fmaxf(m, tree_max<32>(x) * sl2);
        const float m_use = (m == -INFINITY || m_new > m + 8.f) ? m_new : m;
        const float alpha = (m_use == m) ? 1.f : fast_exp2(m - m_use);
        const float mo = (m_use == -INFINITY) ? 0.f : m_use;
        const float sum = exp2_and_sum<32>(x, sl2, mo);
        l = l * alpha + sum;
        if (j > first && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O_h holds P_{j-1} V_{j-1} once that P V is done; the next one
          // waits for this stage's P
          if (!__all_sync(0xffffffffu, mbar_wait(&bar->pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, p.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < kHalf / 32; ++c) {
            uint32_t u[32];
            tmem_ld32(tmem + lane_off + kColO + c * 32, u);
            tmem_wait_ld(u);
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
            tmem_st32(tmem + lane_off + kColO + c * 32, u);
          }
        }
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack2(x[2 * e], x[2 * e + 1], BF16);
        tmem_st16(tmem + lane_off + sb * 32, pk);
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(&bar->p_full[sb]);
        m = m_use;
      }
      if (!ok) break;
      // ---- segment epilogue: O_h / l and lse, as a partial or final
      if (!__all_sync(0xffffffffu, mbar_wait(&bar->pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, p.status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool has = l > 0.f;
      const float inv_l = has ? 1.f / l : 0.f;
      const int b = sg.unit;
      const bool whole = unit_parts[b].y == 1;
      const bool row = r < nh;
      float* po = p.part_o + half * p.part_stride_o + (int64_t(sg.part) * nh + r) * kHalf;
      uint16_t* orow = reinterpret_cast<uint16_t*>(p.out) + int64_t(b) * p.out_sb + int64_t(r) * p.out_sn + half * kHalf;
#pragma unroll
      for (int c = 0; c < kHalf / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem + lane_off + kColO + c * 32, u);
        tmem_wait_ld(u);
        if (c == kHalf / 32 - 1) {
          tc_fence_before();
          warp_arrive(&bar->o_free);     // the next segment's first P V may overwrite O_h now
        }
        if (row) {
          if (whole) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 w;
              w.x = pack2(__uint_as_float(u[8 * q + 0]) * inv_l, __uint_as_float(u[8 * q + 1]) * inv_l, BF16);
              w.y = pack2(__uint_as_float(u[8 * q + 2]) * inv_l, __uint_as_float(u[8 * q + 3]) * inv_l, BF16);
              w.z = pack2(__uint_as_float(u[8 * q + 4]) * inv_l, __uint_as_float(u[8 * q + 5]) * inv_l, BF16);
              w.w = pack2(__uint_as_float(u[8 * q + 6]) * inv_l, __uint_as_float(u[8 * q + 7]) * inv_l, BF16);
              *reinterpret_cast<uint4*>(orow + c * 32 + 8 * q) = w;
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<float4*>(po + c * 32 + 4 * q) =
                  make_float4(__uint_as_float(u[4 * q]) * inv_l, __uint_as_float(u[4 * q + 1]) * inv_l,
                              __uint_as_float(u[4 * q + 2]) * inv_l, __uint_as_float(u[4 * q + 3]) * inv_l);
          }
        }
      }
      if (row) {
        const float lse_v = has ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        if (whole) {
          if (half == 0 && p.lse != nullptr)
            p.lse[int64_t(b) * p.lse_sb + int64_t(r) * p.lse_sn] = has ? lse_v : INFINITY;
        } else {
          p.part_lse[half * p.part_stride_lse + int64_t(sg.part) * nh + r] = lse_v;
        }
      }
      // hand the segment to the merge warp (4-slot ring)
      __threadfence();
      if (segi >= 4 &&
          !__all_sync(0xffffffffu, mbar_wait(&bar->part_free[segi & 3], ((segi >> 2) - 1) & 1, abort_flag, p.status))) {
        ok = false;
        break;
      }
      warp_arrive(&bar->part_done[segi & 3]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool BF16>
cudaError_t launch_mla_t(const MlaParams& p, cudaStream_t s) {
  auto k = mla_kernel<BF16>;
  cudaError_t e = set_smem_once<mla_kernel<BF16>>(kMlaSmem);
  if (e != cudaSuccess) return e;
  k<<<p.n_pairs > 0 ? 2 * p.n_pairs : 2, 256, kMlaSmem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mla(const MlaParams& p, bool bf16, cudaStream_t s) {
  return bf16 ? launch_mla_t<true>(p, s) : launch_mla_t<false>(p, s);
}

}  // namespace fia
