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
//   * the two CTAs of a pair form a cluster and split the 576-wide key by
//     columns: CTA 0 holds latent columns 0..255, CTA 1 latent 256..511 and
//     the 64 rope columns -- of Q' = [q, q_rope] (kept in shared memory for
//     the segment) and of every cache tile, which it alone reads.  Each
//     computes its part of S = Q' K'^T for all heads (M = 128 head rows,
//     N = 32 keys, 256 or 320 deep), sends the partial rows to the partner's
//     shared memory (distributed shared memory: asynchronous stores that
//     complete on the partner's barrier) and adds the partner's: both CTAs
//     then hold the same scores, run the same softmax, and accumulate
//     O_h += P V_h over their own latent columns (N = 256), which are exactly
//     the V half h needs.  The exchange moves 512 bytes per key each way,
//     about as many as the pair reads from HBM, over a network measured at
//     8-12 bytes per cycle per SM in both directions at once, under half an
//     SM's share of HBM bandwidth: it, not HBM, sets this kernel's rate;
//   * each segment leaves one partial (O_h / l, lse) per head; the CTA that
//     completes a (unit, half) merges its partials in a fixed order on its
//     merge warp; a unit held by one segment is written directly.
// Warps: 0..3 softmax (warp w = TMEM lanes 32w..32w+31 = head rows), 4 K'
// producer, 5 MMA issuer and TMEM owner, 6 Q' producer, 7 merge.
// TMEM columns: S buffers [32 s, 32 s + 32) for s < 4 (P overwrites the first
// 16 of its S as packed pairs), O_h [128, 384).
#include "internal.h"
#include "ptx.cuh"

namespace fia {
namespace {

constexpr int kMlaKeys = 32;                 // keys per stage
constexpr int kLatChunks = 8;                // 512 latent columns = 8 boxes of 64 (box 8: the rope)
constexpr int kKBox = kMlaKeys * 128;        // one 64-column box of 32 rows
constexpr int kNBMax = 5;                    // boxes of a CTA: 4 (half 0) or 5 (half 1)
constexpr int kKStage = kNBMax * kKBox;      // a CTA's columns of one stage: <= 20 KB
constexpr int kKS = 5;                       // K' ring slots
constexpr int kNS = 4;                       // S buffers in TMEM (Q K'^T runs up to 3 stages ahead)
constexpr int kQBox = 128 * 128;             // one 64-column box of 128 head rows
constexpr int kQTile = kNBMax * kQBox;       // a CTA's columns of Q' = [q, q_rope]: <= 80 KB
constexpr int kXStride = 36;                 // floats per row of the exchange buffer (32 + 4: no bank conflicts)
constexpr int kXBytes = 128 * kMlaKeys * 4;  // one stage's partial rows (all 128 head rows)
constexpr int kOffK = 0;
constexpr int kOffQ = kOffK + kKS * kKStage;
constexpr int kOffX = kOffQ + kQTile;                    // [2][128 rows][kXStride] partner's partial scores
constexpr int kOffBar = kOffX + 2 * 128 * kXStride * 4;
constexpr int kMlaSmem = kOffBar + 512 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = kNS * 32;
constexpr int kHalf = 256;                   // output columns per CTA
constexpr int kPrefetch = 8;                 // stages ahead warmed in L2

struct MlaBars {
  uint64_t k_full[kKS], pv_done[kKS];   // per ring slot: tiles landed / the stage's P V done (slot free)
  uint64_t qk_done[kNS], p_full[kNS];   // per S buffer
  uint64_t x_full[2], x_free[2];        // exchange slots: the partner's row is in / this CTA's row was read
  uint64_t q_full, q_empty, o_free;
  uint64_t part_done[4], part_free[4];
  uint32_t tmem_holder;
  int abort_flag;
  // the CTA's last segment completed a unit: merged by every warp once the
  // roles are done (-1: none)
  int final_unit;
};
static_assert(sizeof(MlaBars) <= 512, "barrier area");
static_assert(kMlaSmem <= 227 * 1024, "shared memory budget");
static_assert(kOffQ % 1024 == 0 && kKStage % 1024 == 0, "swizzled tiles need 1024-byte alignment");

__device__ __forceinline__ const DecodeSeg* mla_segs(const MlaParams& p) { return p.segs; }
__device__ __forceinline__ const int32_t* mla_cta(const MlaParams& p) { return p.cta_seg; }
__device__ __forceinline__ const int2* mla_units(const MlaParams& p) { return p.unit_parts; }
__device__ __forceinline__ const int32_t* mla_kvlen(const MlaParams& p) { return p.kv_len; }

// Merges the partials of (unit b, half) in part order: lanes over the 256
// columns (two float4 each), four heads at a time, the O rows of four parts
// loaded together.  Every lane reads the parts' lse words of its four heads
// itself (the same words in all lanes: one transaction each) and weighs the
// parts locally, so no cross-lane reduction sits on the merge's critical
// path.  Head groups g0, g0 + gstep, ... of four heads: one warp takes them
// all, or the CTA's warps share them.
template <bool BF16>
__device__ void mla_merge(const MlaParams& p, int b, int half, int2 up, int lane, int g0, int gstep) {
  constexpr int KB = 4;
  const int nh = p.num_heads;
  const float* po = p.part_o + half * p.part_stride_o;
  const float* pl = p.part_lse + half * p.part_stride_lse;
  for (int h0 = 4 * g0; h0 < nh; h0 += 4 * gstep) {
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
      float lk[KB][4];
      float4 o[KB][4][2];
#pragma unroll
      for (int k = 0; k < KB; ++k)
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const bool v = k < kn && h0 + t < nh;
          lk[k][t] = v ? __ldcg(pl + int64_t(up.x + k0 + k) * nh + h0 + t) : -INFINITY;
#pragma unroll
          for (int c = 0; c < 2; ++c)
            o[k][t][c] = v ? __ldcg(reinterpret_cast<const float4*>(po + (int64_t(up.x + k0 + k) * nh + h0 + t) * kHalf) +
                                    c * 32 + lane)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        float mb = lk[0][t];
#pragma unroll
        for (int k = 1; k < KB; ++k) mb = fmaxf(mb, lk[k][t]);
        const float m_new = fmaxf(M[t], mb);
        const float a = (m_new == -INFINITY) ? 1.f : __expf(M[t] - m_new);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          acc[t][c].x *= a; acc[t][c].y *= a; acc[t][c].z *= a; acc[t][c].w *= a;
        }
        Ls[t] *= a;
#pragma unroll
        for (int k = 0; k < KB; ++k) {
          const float w = (lk[k][t] == -INFINITY) ? 0.f : __expf(lk[k][t] - m_new);
          Ls[t] += w;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            acc[t][c].x += w * o[k][t][c].x; acc[t][c].y += w * o[k][t][c].y;
            acc[t][c].z += w * o[k][t][c].z; acc[t][c].w += w * o[k][t][c].w;
          }
        }
        M[t] = m_new;
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

// ------------------------------------------------------------ cluster helpers
// The two CTAs of a pair form a cluster (ranks 0 and 1 = half).
__device__ __forceinline__ uint32_t cluster_map(uint32_t local_smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem_addr), "r"(rank));
  return r;
}
// An asynchronous store to the partner's shared memory that completes its
// bytes on the partner's barrier (expect-tx): the sender does not wait.
__device__ __forceinline__ void cluster_store4_async(uint32_t addr, float a, float b, float c, float d,
                                                     uint32_t remote_bar_addr) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
               "f"(a), "f"(b), "f"(c), "f"(d), "r"(remote_bar_addr)
               : "memory");
}
// An arrival on the partner's barrier with the default (CTA-scope release)
// semantics.  It tells the partner that this CTA has read an exchange slot:
// the reads' values are consumed before it is issued, and the partner's
// refill is an asynchronous store a network round trip later, so no
// cluster-scope fence (which waits for this thread's own stores to the
// partner still in flight) is needed.
__device__ __forceinline__ void cluster_arrive_remote(uint32_t remote_bar_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(remote_bar_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// mbar_wait_lean with cluster-scope acquire (the phase is completed by the
// partner CTA's stores and arrivals).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                  const DevStatus& status) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t limit_ns = status.limit_ns;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > limit_ns) {
      *abort = 1;
      status_raise(status, 10u /* FIA_ERR_TIMEOUT */);
      return false;
    }
  }
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1) mla_kernel(const __grid_constant__ MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  MlaBars* bar = reinterpret_cast<MlaBars*>(smem + kOffBar);
  volatile int* abort_flag = &bar->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = blockIdx.x & 1, pair = blockIdx.x >> 1;
  const uint32_t partner = uint32_t(half ^ 1);
  // this CTA's 64-column boxes of [latent | rope]: half 0 latent 0..255,
  // half 1 latent 256..511 and the rope (box 8)
  const int c0 = 4 * half, nb = 4 + half;
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
    for (int s = 0; s < kKS; ++s) {
      mbar_init(&bar->k_full[s], 1);
      mbar_init(&bar->pv_done[s], 1);
    }
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&bar->qk_done[s], 1);
      mbar_init(&bar->p_full[s], 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar->x_full[s], 1);   // armed by this CTA, completed by the partner's kXBytes
      mbar_init(&bar->x_free[s], 4);   // the partner's four softmax warps
    }
    mbar_init(&bar->q_full, 1);
    mbar_init(&bar->q_empty, 1);
    mbar_init(&bar->o_free, 4);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bar->part_done[s], 4);
      mbar_init(&bar->part_free[s], 1);
    }
    bar->abort_flag = 0;
    bar->final_unit = -1;
    fence_mbar_init();
    // the exchange slots of stages 0 and 1 expect the partner's rows
    mbar_arrive_expect_tx(&bar->x_full[0], uint32_t(kXBytes));
    mbar_arrive_expect_tx(&bar->x_full[1], uint32_t(kXBytes));
  }
  if (warp == 5) {
    tmem_alloc(&bar->tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // both CTAs' barriers are initialised before either touches the other's
  cluster_sync_all();
  const uint32_t tmem = bar->tmem_holder;

  if (warp == 4) {
    // ------------------------------------------------------- K' producer
    // this CTA's boxes of every 32-token stage into a kKS-slot ring; a slot
    // is free once the stage's P V is done (it read V = latent)
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
      auto row_of = [&](int tok) -> int64_t {
        if (p.block_table == nullptr) return int64_t(b) * p.row_per_blk + tok;
        const int page = tok / p.block_size;
        if (page < cache_base || page >= cache_base + 32) {
          cache_base = page;
          const int e = cache_base + lane;
          cache_blk = e < p.table_stride ? p.block_table[int64_t(b) * p.table_stride + e] : 0;
        }
        const int64_t blk = __shfl_sync(0xffffffffu, cache_blk, page - cache_base);
        return blk * p.row_per_blk + (tok % p.block_size);
      };
      for (int st = sg.stage_begin; st < sg.stage_end; ++st, ++j) {
        const int s = j % kKS;
        if (j >= kKS && !__all_sync(0xffffffffu, mbar_wait_lean(&bar->pv_done[s], uint32_t(j / kKS - 1) & 1u, abort_flag,
                                                           p.status))) {
          ok = false;
          break;
        }
        const int t0 = st * kMlaKeys;
        const int nvalid = min(kMlaKeys, L - t0);
        const int nbox = (nvalid + p.box_rows - 1) / p.box_rows;
        uint8_t* dst = smem + kOffK + s * kKStage;
        if (lane == 0) mbar_arrive_expect_tx(&bar->k_full[s], uint32_t(nb * nbox * p.box_rows * 128));
        for (int k = 0; k < nbox; ++k) {
          const int64_t row = row_of(t0 + k * p.box_rows);
          if (lane == 0) {
            for (int bx = 0; bx < nb; ++bx) {
              const int c = c0 + bx;
              uint8_t* d = dst + bx * kKBox + k * p.box_rows * 128;
              if (c < kLatChunks) tma_load_2d(d, &p.tm_lat, &bar->k_full[s], c * 64, int(row));
              else tma_load_2d(d, &p.tm_rope, &bar->k_full[s], 0, int(row));
            }
          }
        }
        // the tiles kPrefetch stages ahead are pulled into L2 now: their
        // loads then wait for L2, not for HBM
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
            for (int bx = 0; bx < nb; ++bx) {
              const int c = c0 + bx;
              if (c < kLatChunks) tma_prefetch_l2_2d(&p.tm_lat, c * 64, int(prow));
              else tma_prefetch_l2_2d(&p.tm_rope, 0, int(prow));
            }
          }
        }
      }
    }
    if (lane == 0 && *abort_flag) {
      for (int s = 0; s < kKS && s < j; ++s) {
        const int last = j - 1 - ((j - 1 - s) % kKS);
        mbar_wait_lean(&bar->k_full[s], uint32_t(last / kKS) & 1u, nullptr, p.status);
      }
    }
  } else if (warp == 6) {
    // ------------------------------------------------------- Q' producer
    // this CTA's columns of Q' = [q, q_rope] for the segment's batch (all
    // heads); the tile is reused once the previous segment's last Q K'^T is
    // done (q_empty, one arrival per segment from the MMA warp)
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_qr);
      int issued = 0;
      for (int segi = 0; segi < nseg; ++segi) {
        const DecodeSeg sg = segs[seg_begin + segi];
        if (segi > 0 && !mbar_wait_lean(&bar->q_empty, uint32_t(segi - 1) & 1u, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&bar->q_full, uint32_t(nb * kQBox));
        const int row = sg.unit * nh;
        for (int bx = 0; bx < nb; ++bx) {
          const int c = c0 + bx;
          if (c < kLatChunks) tma_load_2d(smem + kOffQ + bx * kQBox, &p.tm_q, &bar->q_full, c * 64, row);
          else tma_load_2d(smem + kOffQ + bx * kQBox, &p.tm_qr, &bar->q_full, 0, row);
        }
        ++issued;
      }
      if (*abort_flag && issued > 0) mbar_wait_lean(&bar->q_full, uint32_t(issued - 1) & 1u, nullptr, p.status);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------- MMA issuer
    // Lane 0 issues; the whole warp clears, before a ragged stage's P V, the
    // latent rows past the sequence (a cache's unused rows may hold NaN, and
    // P = 0 times NaN is not 0).  The Q K'^T products run up to kNS - 1
    // stages ahead of the P V products (an S buffer is rewritten only after
    // the P V that read its P has been issued: MMAs run in issue order).
    constexpr uint32_t idesc_qk = idesc_f16(128, kMlaKeys, BF16 ? 1 : 0, 0, 0);
    constexpr uint32_t idesc_pv = idesc_f16(128, kHalf, BF16 ? 1 : 0, 0, 1);
    const uint32_t k_base = smem_u32(smem + kOffK), q_base = smem_u32(smem + kOffQ);
    int j = 0;
    bool ok = true;
    uint64_t* last_bar = nullptr;
    uint32_t last_parity = 0;
    auto issue_pv = [&](int jj, int first, int segi, int nvalid, bool seg_last) -> bool {
      const int s = jj % kKS, sb = jj % kNS;
      if (jj == first && segi > 0 &&
          !__all_sync(0xffffffffu, mbar_wait_lean(&bar->o_free, uint32_t(segi - 1) & 1u, abort_flag, p.status)))
        return false;
      if (!__all_sync(0xffffffffu, mbar_wait_lean(&bar->p_full[sb], uint32_t(jj / kNS) & 1u, abort_flag, p.status)))
        return false;
      // every Q K'^T of the segment has completed once the softmax has its
      // last P: the Q' tile may be refilled
      if (seg_last && lane == 0) mbar_arrive(&bar->q_empty);
      if (nvalid < kMlaKeys) {
        uint8_t* vs = smem + kOffK + s * kKStage;
        for (int c = 0; c < 4; ++c)
          for (int u = lane; u < (kMlaKeys - nvalid) * 8; u += 32)
            *reinterpret_cast<uint4*>(vs + c * kKBox + (nvalid + (u >> 3)) * 128 + (u & 7) * 16) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        tc_fence_after();
        const uint32_t vb = k_base + s * kKStage;   // local boxes 0..3 = this CTA's 256 latent columns
#pragma unroll
        for (int kk = 0; kk < kMlaKeys / 16; ++kk)
          mma_ts(tmem + kColO, tmem + sb * 32 + kk * 8, smem_desc_sw128(vb + kk * 2048, kKBox, 1024), idesc_pv,
                 (jj > first || kk > 0) ? 1u : 0u);
        mma_commit(&bar->pv_done[s]);
      }
      last_bar = &bar->pv_done[s];
      last_parity = uint32_t(jj / kKS) & 1u;
      return true;
    };
    for (int segi = 0; segi < nseg && ok; ++segi) {
      const DecodeSeg sg = segs[seg_begin + segi];
      const int L = kvlen[sg.unit];
      if (!__all_sync(0xffffffffu, mbar_wait_lean(&bar->q_full, uint32_t(segi) & 1u, abort_flag, p.status))) {
        ok = false;
        break;
      }
      const int first = j;
      int jp = j;   // next P V of this segment to issue
      auto nvalid_of = [&](int jj) { return min(kMlaKeys, L - (sg.stage_begin + jj - first) * kMlaKeys); };
      for (int st = sg.stage_begin; st < sg.stage_end; ++st, ++j) {
        const int s = j % kKS, sb = j % kNS;
        while (ok && jp <= j - kNS) {   // S buffer sb still holds P of stage j - kNS
          ok = issue_pv(jp, first, segi, nvalid_of(jp), false);
          ++jp;
        }
        if (!ok) break;
        if (!__all_sync(0xffffffffu, mbar_wait_lean(&bar->k_full[s], uint32_t(j / kKS) & 1u, abort_flag, p.status))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t kb = k_base + s * kKStage;
          for (int kk = 0; kk < nb * 4; ++kk)
            mma_ss(tmem + sb * 32, smem_desc_sw128(q_base + (kk >> 2) * kQBox + (kk & 3) * 32, 16, 1024),
                   smem_desc_sw128(kb + (kk >> 2) * kKBox + (kk & 3) * 32, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
          mma_commit(&bar->qk_done[sb]);
        }
        last_bar = &bar->qk_done[sb];
        last_parity = uint32_t(j / kNS) & 1u;
      }
      while (ok && jp < j) {
        ok = issue_pv(jp, first, segi, nvalid_of(jp), jp == j - 1);
        ++jp;
      }
    }
    if (last_bar != nullptr && lane == 0) mbar_wait_lean(last_bar, last_parity, nullptr, p.status);
    __syncwarp();
  } else if (warp == 7) {
    // ------------------------------------------------------- merge warp
    bool ok = true;
    for (int segi = 0; segi < nseg && ok; ++segi) {
      const DecodeSeg sg = segs[seg_begin + segi];
      if (!__all_sync(0xffffffffu, mbar_wait_lean(&bar->part_done[segi & 3], uint32_t(segi >> 2) & 1u, abort_flag,
                                             p.status))) {
        ok = false;
        break;
      }
      if (lane == 0) mbar_arrive(&bar->part_free[segi & 3]);
      const int2 up = unit_parts[sg.unit];
      if (up.y == 1) continue;   // written directly by the softmax warps
      // the increment releases this segment's partials (written by the
      // softmax warps before part_done) and, for the last one, acquires the
      // others'; the warp barrier orders every lane's loads after it
      int last = 0;
      if (lane == 0)
        last = int(tagged_increment_acq_rel(p.unit_counter + sg.unit * 2 + half, unit_tag(p.status.epoch))) == up.y;
      if (__shfl_sync(0xffffffffu, last, 0)) {
        __syncwarp();
        if (segi == nseg - 1) {
          // the CTA's last segment: nothing follows it, so all eight warps
          // share this merge after the roles end
          if (lane == 0) bar->final_unit = sg.unit;
        } else {
          mla_merge<BF16>(p, sg.unit, half, up, lane, 0, 1);
        }
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
    // Thread r = head row r of S (TMEM lane r).  Each CTA's Q K'^T covers its
    // share of the 576-deep contraction; the scores are the sum of the two
    // CTAs' partial products.  A stage's partial row goes to the partner's
    // exchange buffer as soon as it is in TMEM (asynchronous stores that
    // complete on the partner's barrier); the softmax of the stage before it
    // runs meanwhile, so the exchange's latency is hidden behind a stage of
    // work.  Both CTAs add the same two fp32 values (in either
    // order, exactly), so their scores, maxima, sums and P agree bit for bit.
    const int r = threadIdx.x;
    const uint32_t lane_off = uint32_t(32 * warp) << 16;
    const float sl2 = p.scale_log2;
    float* xbuf = reinterpret_cast<float*>(smem + kOffX);   // [2][128 rows][kXStride]
    const uint32_t x_local = smem_u32(xbuf);
    const uint32_t x_remote = cluster_map(x_local, partner);
    const uint32_t xfull_remote[2] = {cluster_map(smem_u32(&bar->x_full[0]), partner),
                                      cluster_map(smem_u32(&bar->x_full[1]), partner)};
    const uint32_t xfree_remote[2] = {cluster_map(smem_u32(&bar->x_free[0]), partner),
                                      cluster_map(smem_u32(&bar->x_free[1]), partner)};
    bool ok = true;
    int j = 0;
    float xp[kMlaKeys];   // this CTA's partial scores of the stage waiting for its softmax
    for (int segi = 0; segi < nseg && ok; ++segi) {
      const DecodeSeg sg = segs[seg_begin + segi];
      const int L = kvlen[sg.unit];
      const int first = j;
      float m = -INFINITY, l = 0.f;
      // the softmax of stage js (scores = xp + the partner's row), P into
      // its S buffer
      auto softmax_stage = [&](int js) -> bool {
        const int sb = js % kNS, xs = js & 1;
        if (!__all_sync(0xffffffffu, mbar_wait_cluster(&bar->x_full[xs], uint32_t(js >> 1) & 1u, abort_flag, p.status)))
          return false;
        float x[32];
        const float* xr = xbuf + (xs * 128 + r) * kXStride;
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 v = *reinterpret_cast<const float4*>(xr + c);
          x[c] = xp[c] + v.x;
          x[c + 1] = xp[c + 1] + v.y;
          x[c + 2] = xp[c + 2] + v.z;
          x[c + 3] = xp[c + 3] + v.w;
        }
        // this warp's rows of the buffer are read: re-arm the slot for stage
        // js + 2 (before any "free" reaches the partner, so the arm precedes
        // the partner's next bytes), then let the partner refill it
        __syncwarp();
        if (threadIdx.x == 0) mbar_arrive_expect_tx(&bar->x_full[xs], uint32_t(kXBytes));
        if (lane == 0) cluster_arrive_remote(xfree_remote[xs]);
        const int nvalid = min(kMlaKeys, L - (sg.stage_begin + js - first) * kMlaKeys);
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
        if (js > first && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O_h holds P V up to stage js - 1 once that P V is done; the next
          // one waits for this stage's P
          if (!__all_sync(0xffffffffu, mbar_wait_lean(&bar->pv_done[(js - 1) % kKS], uint32_t((js - 1) / kKS) & 1u,
                                                 abort_flag, p.status)))
            return false;
          tc_fence_after();
#pragma unroll 1
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
        return true;
      };
      for (int st = sg.stage_begin; st < sg.stage_end; ++st, ++j) {
        const int sb = j % kNS, xs = j & 1;
        // ---- this stage's partial row: TMEM -> the partner's buffer
        if (!__all_sync(0xffffffffu, mbar_wait_lean(&bar->qk_done[sb], uint32_t(j / kNS) & 1u, abort_flag, p.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t su[32];
        tmem_ld32(tmem + lane_off + sb * 32, su);
        tmem_wait_ld(su);
        // the partner has read what this CTA sent two stages ago from that slot
        if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait_cluster(&bar->x_free[xs], uint32_t((j >> 1) - 1) & 1u,
                                                                 abort_flag, p.status))) {
          ok = false;
          break;
        }
        const uint32_t dst = x_remote + uint32_t(((xs * 128 + r) * kXStride) * 4);
#pragma unroll
        for (int c = 0; c < 32; c += 4)
          cluster_store4_async(dst + c * 4, __uint_as_float(su[c]), __uint_as_float(su[c + 1]),
                               __uint_as_float(su[c + 2]), __uint_as_float(su[c + 3]), xfull_remote[xs]);
        // ---- the softmax of the stage before, while the exchange runs
        if (j > first && !softmax_stage(j - 1)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) xp[c] = __uint_as_float(su[c]);
      }
      if (!ok) break;
      if (j > first && !softmax_stage(j - 1)) {
        ok = false;
        break;
      }
      // ---- segment epilogue: O_h / l and lse, as a partial or final
      if (!__all_sync(0xffffffffu, mbar_wait_lean(&bar->pv_done[(j - 1) % kKS], uint32_t((j - 1) / kKS) & 1u, abort_flag,
                                             p.status))) {
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
#pragma unroll 1
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
      // hand the segment to the merge warp (4-slot ring); its fence before
      // the unit counter covers these writes (released by the arrival)
      if (segi >= 4 && !__all_sync(0xffffffffu, mbar_wait_lean(&bar->part_free[segi & 3], uint32_t((segi >> 2) - 1) & 1u,
                                                          abort_flag, p.status))) {
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
  // the last segment's merge (its counter's acquire, by the merge warp, is
  // ordered before these loads by the CTA barrier above)
  const int fu = bar->final_unit;
  if (fu >= 0 && !*abort_flag) mla_merge<BF16>(p, fu, half, unit_parts[fu], lane, warp, 8);
  // neither CTA leaves while the other may still write to its shared memory
  cluster_sync_all();
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
