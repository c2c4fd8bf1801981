// Incremental attention for small query groups: units of at most 16 query
// rows (GQA groups of up to 16 heads per kv head with one new token, or 4
// heads with 4 new tokens, and so on) and head_dim 128.
//
// Operation: the IncreFlashAttention case of npu_fused_infer_attention_score
// (as decode_kernel.cuh): out = softmax(scale * q K^T) V per (batch, head)
// over a paged or contiguous cache, per-batch actual_seq_kvlen, GQA, a
// per-batch key mask with one new token, and for several new tokens the
// sparse_mode 2 / 3 limits.
//
// With so few rows the two products of a 128-key stage are thin (at most
// 16 x 128 x 128 multiply-adds each).  The tcgen05 form (decode_kernel.cuh)
// pays a round trip per stage through TMEM and barriers between warps; here
// every compute warp runs its own warp-synchronous mma.sync products, and no
// warp waits on another inside a segment:
//   * the plan is decode_kernel.cuh's: units (batch, kv head), 128-token
//     stages dealt to one CTA per SM in segments, one partial per segment
//     and row, merged in part order by the CTA that completes a unit;
//   * warps 8 and 9 stream the K and V tiles of each stage into rings by TMA
//     (128-byte swizzle, one 64-column box per 128 bytes of a row), warp 10
//     merges finished units, except the unit of a CTA's last segment, which
//     the compute warps count and merge themselves (it ends the CTA's walk);
//   * compute warp w (0..7) owns keys [16 w, 16 w + 16) of every stage and
//     keeps its own running maximum, sum and O^T for every row; the eight
//     warps' states are combined once per segment with the exact LSE
//     weights.  Two compute warps per scheduler hide each other's latency.
// K and V slots are released (one arrival per compute warp) as soon as the
// warp's reads of them are done.
#include "decode_kernel.cuh"

namespace fia {

namespace {

constexpr int kGqaKS = 3;                 // K ring slots
constexpr int kGqaTile = 2 * 128 * 128;   // K (or V) of one 128-token stage, D = 128: two 16 KB boxes
constexpr int kGqaBox = 128 * 128;
constexpr int kGqaW = 8;                  // compute warps, 16 keys of a stage each
constexpr int kGqaThreads = (kGqaW + 3) * 32;   // + K producer, V producer, merge
constexpr int kGqaWarmStages = 4;          // stages warmed in L2 before the grid dependency resolves
constexpr int kGqaBarBytes = 1024;

// Shared memory of the kernel for units of kRows (4 or 16) rows: the K and V
// rings (three slots each), each warp's O of a segment (fp32, kERows x 128:
// 16-row units go through it in two passes of 8 rows, which leaves the room
// for the third V slot) and (max, sum) per row, the barriers.
template <int kRows>
struct GqaCfg {
  static constexpr int kVS = 3;
  static constexpr int kERows = kRows == 16 ? 8 : kRows;   // rows per warp in one pass
  static constexpr int kPasses = kRows / kERows;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kGqaKS * kGqaTile;
  static constexpr int kOffE = kOffV + kVS * kGqaTile;              // [warp][kERows][128]
  static constexpr int kOffML = kOffE + kGqaW * kERows * 128 * 4;   // [warp][kRows] (max, sum)
  static constexpr int kOffBar = kOffML + kGqaW * kRows * 8;
  static constexpr int kSmem = kOffBar + kGqaBarBytes + 1024;
  static_assert(kSmem <= kDecodeSmemMax, "shared memory budget");
};

struct GqaBars {
  uint64_t k_full[kGqaKS], v_full[kGqaKS];   // TMA landed (expect-tx)
  uint64_t k_free[kGqaKS], v_free[kGqaKS];   // every compute warp is done with the slot
  uint64_t esync, efree;                     // the warps' segment states are in / have been read
  uint64_t part_done[4], part_free[4];       // compute -> merge warp hand-off ring
  uint64_t tail_in, tail_count;              // the last segment's partials are out / its unit is counted
  int tail_last;                             // this CTA completed the last segment's unit
  int abort_flag;
};
static_assert(sizeof(GqaBars) <= kGqaBarBytes, "barrier area");

// One m8n8 x4 shared-memory matrix load (ldmatrix): lane i gives the address
// of row i % 8 of matrix i / 8; lane (g, t) receives elements (g, 2t), (g, 2t+1)
// of each matrix -- with .trans, elements (2t, g), (2t+1, g).
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// d += A B for one m16n8k16 tile (A row-major 16 x 16, B column-major 16 x 8,
// 16-bit inputs of the call's type, fp32 accumulators).
template <bool BF16>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// kRows: 4 (row g of a lane's S fragment; rows 4..7 masked) or 16 (rows g
// and g + 8).
template <bool BF16, int kRows>
__global__ void __launch_bounds__(kGqaThreads, 1) decode_gqa_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int D = 128;
  using C = GqaCfg<kRows>;
  constexpr int VS = C::kVS;
  constexpr bool kTwo = kRows == 16;   // two rows per lane, two O^T row tiles
  constexpr int NT = kTwo ? 2 : 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  GqaBars* bar = reinterpret_cast<GqaBars*>(smem + C::kOffBar);
  volatile int* abort_flag = &bar->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const DecodePlanRef pl = decode_plan(p);
  const int g = p.rows;

  grid_dep_launch();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGqaKS; ++s) {
      mbar_init(&bar->k_full[s], 1);
      mbar_init(&bar->k_free[s], kGqaW);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(&bar->v_full[s], 1);
      mbar_init(&bar->v_free[s], kGqaW);
    }
    mbar_init(&bar->esync, kGqaW);
    mbar_init(&bar->efree, kGqaW);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bar->part_done[s], kGqaW);
      mbar_init(&bar->part_free[s], 1);
    }
    mbar_init(&bar->tail_in, kGqaW);
    mbar_init(&bar->tail_count, 1);
    bar->tail_last = 0;
    bar->abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // This CTA may start on an SM the previous kernel's CTA has just left while
  // that kernel's other CTAs still run: the producers warm L2 with the first
  // stages of the CTA's first segment meanwhile (a plan carried in the
  // parameters only; one in the workspace is read after the wait).
  if ((warp == kGqaW || warp == kGqaW + 1) && p.n_cta > 0 && p.plan_ws == nullptr) {
    const int sb = pl.cta_seg(blockIdx.x);
    if (sb < pl.cta_seg(blockIdx.x + 1))
      l2_warm_segment<2>(p, pl, warp == kGqaW ? &p.tm_k : &p.tm_v, pl.seg_at(sb), kGqaWarmStages);
  }
  grid_dep_wait();   // the previous kernel on the stream is complete from here on
  if (threadIdx.x == 0 && blockIdx.x == 0) status_stamp(p.status);
  const int seg_begin = p.n_cta > 0 ? pl.cta_seg(blockIdx.x) : 0;
  const int seg_end = p.n_cta > 0 ? pl.cta_seg(blockIdx.x + 1) : 0;
  const int nseg = seg_end - seg_begin;
  // The CTA's last segment, when its unit is split, is counted and merged by
  // the compute warps themselves (it ends the CTA's walk: a hand-off to the
  // merge warp would only add its latency); the merge warp takes the others.
  const bool tail_split = nseg > 0 && pl.unit_parts(pl.seg_at(seg_end - 1).unit).y > 1;

  int issued = 0;
  if (warp == kGqaW) {
    NoQLoader nq;
    issued = decode_producer<kGqaTile, kGqaBox, 2, kGqaKS, kGqaKS>(p, pl, &p.tm_k, smem + C::kOffK, bar->k_full,
                                                                   bar->k_free, abort_flag, seg_begin, seg_end, nq);
  } else if (warp == kGqaW + 1) {
    NoQLoader nq;
    issued = decode_producer<kGqaTile, kGqaBox, 2, VS, VS>(p, pl, &p.tm_v, smem + C::kOffV, bar->v_full, bar->v_free,
                                                           abort_flag, seg_begin, seg_end, nq);
  } else if (warp == kGqaW + 2) {
    merge_warp<D, BF16>(p, pl, bar->part_done, bar->part_free, abort_flag, seg_begin, nseg - int(tail_split), lane);
  } else {
    // ------------------------------------------------------------ compute
    // Warp-synchronous tensor-core products (mma.sync m16n8k16, fp32
    // accumulate), lane (g = lane / 4, t = lane % 4) in the fragment layouts:
    //   S = Q K^T over the warp's 16 keys: A = Q (rows g and g + 8, from
    //     registers), B = K^T by ldmatrix from the swizzled K tile; lane
    //     (g, t) gets S[rows g, g + 8][keys 2t, 2t+1] and [8 + 2t, 9 + 2t];
    //   O^T = V^T P^T, one product per 8 rows: A = V^T by ldmatrix.trans from
    //     the V tile, B = P^T, whose fragment is exactly lane (g, t)'s
    //     probabilities of row g (or g + 8) at keys 2t, 2t+1 | 8 + 2t, 9 + 2t,
    //     so P never leaves the registers; lane (g, t) holds
    //     O^T[d = 16 m + g (+ 8)][rows 2t, 2t+1 (+ 8)].
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    const int w = warp;
    const int fg = lane >> 2, ft = lane & 3;
    const int lr = lane & 7, lm = lane >> 3;      // ldmatrix: row of a matrix, matrix
    float* ebuf = reinterpret_cast<float*>(smem + C::kOffE);
    float2* mlbuf = reinterpret_cast<float2*>(smem + C::kOffML);
    const float sl2 = p.scale_log2;
    const uint32_t k_base = smem_u32(smem + C::kOffK), v_base = smem_u32(smem + C::kOffV);
    auto sw_off = [](int row, int col8) -> uint32_t {   // col8: 16-byte block of the row (0..15)
      return uint32_t((col8 >> 3) * kGqaBox + row * 128 + (((col8 & 7) ^ (row & 7)) << 4));
    };
    // this lane's rows of S and P: ra = g and (16 rows) rb = g + 8
    const int ra = fg, rb = fg + 8;
    const bool live_a = ra < g, live_b = kTwo && rb < g;
    const int tok_a = ra % p.q_tokens, tok_b = rb % p.q_tokens;
    // this lane's words of the A = Q fragments of segment sq: per 16-element
    // step ks, row r's elements [16 ks + 2t, +1] and [16 ks + 8 + 2t, +1]
    auto q_row = [&](const DecodeSeg& sq, int r) -> const uint32_t* {
      const int kvh_q = sq.unit % p.num_kv_heads, b_q = sq.unit / p.num_kv_heads;
      const int head = kvh_q * p.group + r / p.q_tokens, tok = r % p.q_tokens;
      return reinterpret_cast<const uint32_t*>(reinterpret_cast<const T*>(p.q) + int64_t(b_q) * p.q_sb +
                                               int64_t(head) * p.q_sn + int64_t(tok) * p.q_ss);
    };
    auto load_q = [&](const DecodeSeg& sq, uint32_t (&dst)[8][kTwo ? 4 : 2]) {
      const uint32_t* sa = live_a ? q_row(sq, ra) : nullptr;
      const uint32_t* sb = live_b ? q_row(sq, rb) : nullptr;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        dst[ks][0] = live_a ? __ldg(sa + 8 * ks + ft) : 0u;
        dst[ks][1] = live_a ? __ldg(sa + 8 * ks + 4 + ft) : 0u;
        if constexpr (kTwo) {
          dst[ks][2] = live_b ? __ldg(sb + 8 * ks + ft) : 0u;
          dst[ks][3] = live_b ? __ldg(sb + 8 * ks + 4 + ft) : 0u;
        }
      }
    };
    // 4 rows: the next segment's fragments wait in registers; 16 rows (twice
    // the fragments, twice the O^T): its q rows are warmed in L2 instead
    uint32_t qn[8][kTwo ? 1 : 2];
    bool ok = true;
    int j = 0;   // stages consumed
    for (int segi = 0; segi < nseg && ok; ++segi) {
      const DecodeSeg sg = pl.seg_at(seg_begin + segi);
      const int kvh = sg.unit % p.num_kv_heads, b = sg.unit / p.num_kv_heads;
      const int L = pl.kv_len(b);
      // several query tokens: row h is token h % Q_S and sees keys up to
      // klim + h % Q_S (sparse_mode 3: klim = S_kv - Q_S; 2: klim = 0)
      const int klim = p.q_causal == 3 ? L - p.q_tokens : 0;
      uint32_t qa[8][kTwo ? 4 : 2];
      if constexpr (kTwo) {
        load_q(sg, qa);
        if (segi + 1 < nseg && lane < g) {   // one 256-byte q row per lane
          const uint32_t* nr = q_row(pl.seg_at(seg_begin + segi + 1), lane);
          asm volatile("prefetch.global.L2 [%0];" ::"l"(nr) : "memory");
          asm volatile("prefetch.global.L2 [%0];" ::"l"(nr + 32) : "memory");
        }
      } else {
        if (segi == 0) {
          load_q(sg, qa);
        } else {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            qa[ks][0] = qn[ks][0];
            qa[ks][1] = qn[ks][1];
          }
        }
        if (segi + 1 < nseg) load_q(pl.seg_at(seg_begin + segi + 1), qn);
      }
      // this warp's running state: the maximum m (log2 units) of rows ra, rb
      // and the sums of this lane's p of them relative to m; O^T
      float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
      float o[8][NT][4];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int c = 0; c < 4; ++c) o[mt][n][c] = 0.f;

      for (int st = sg.stage_begin; st < sg.stage_end; ++st, ++j) {
        const int kslot = j % kGqaKS, vslot = j % VS;
        const uint32_t kpar = uint32_t(j / kGqaKS) & 1u, vpar = uint32_t(j / VS) & 1u;
        const int t0 = st * 128;
        const int nvalid = min(128, L - t0);
        const int nvw = nvalid - 16 * w;   // valid keys of this warp (may be <= 0 or >= 16)
        // atten_mask bytes of this lane's four keys (bit e: key e masked),
        // read while the stage's copies land
        uint32_t kmask = 0;
        if (p.key_mask != nullptr) {
          const uint8_t* mrow = p.key_mask + int64_t(b) * p.key_mask_sb + t0 + 16 * w;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int kl = 8 * (e >> 1) + 2 * ft + (e & 1);
            if (kl < nvw && __ldg(mrow + kl) != 0) kmask |= 1u << e;
          }
        }
        if (!warp_wait(&bar->k_full[kslot], kpar, abort_flag, p.status)) {
          ok = false;
          break;
        }
        // ---- S = Q K^T
        const uint32_t kt = k_base + uint32_t(kslot * kGqaTile);
        float sacc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
          for (int c = 0; c < 4; ++c) sacc[nt][c] = 0.f;
          const int row = 16 * w + 8 * nt + lr;
#pragma unroll
          for (int kp = 0; kp < 4; ++kp) {
            uint32_t kb[4];
            ldmatrix_x4(kt + sw_off(row, 4 * kp + lm), kb);
            if constexpr (kTwo) {
              mma_16816<BF16>(sacc[nt], qa[2 * kp][0], qa[2 * kp][2], qa[2 * kp][1], qa[2 * kp][3], kb[0], kb[1]);
              mma_16816<BF16>(sacc[nt], qa[2 * kp + 1][0], qa[2 * kp + 1][2], qa[2 * kp + 1][1], qa[2 * kp + 1][3],
                              kb[2], kb[3]);
            } else {
              mma_16816<BF16>(sacc[nt], qa[2 * kp][0], 0u, qa[2 * kp][1], 0u, kb[0], kb[1]);
              mma_16816<BF16>(sacc[nt], qa[2 * kp + 1][0], 0u, qa[2 * kp + 1][1], 0u, kb[2], kb[3]);
            }
          }
        }
        warp_arrive(&bar->k_free[kslot]);

        // ---- online softmax of rows ra (and rb) over the warp's keys
        const bool causal = p.q_causal != 0 && t0 + 127 > klim;   // a key of this stage is past a limit
        uint32_t pf[NT][2];   // B = P^T fragments: keys 2t, 2t+1 | 8 + 2t, 9 + 2t of row ra (rb)
        float alpha[2];
#pragma unroll
        for (int h = 0; h < NT; ++h) {
          const bool live = h == 0 ? live_a : live_b;
          const int tok = h == 0 ? tok_a : tok_b;
          float sv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int kl = 8 * (e >> 1) + 2 * ft + (e & 1);
            const int key = 16 * w + kl;
            const bool on = live && kl < nvw && (!causal || t0 + key - klim <= tok) && !((kmask >> e) & 1u);
            sv[e] = on ? sacc[e >> 1][2 * h + (e & 1)] * sl2 : -INFINITY;
          }
          float mx = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          const float mn = fmaxf(m_run[h], mx);
          const float mo = mn == -INFINITY ? 0.f : mn;
          alpha[h] = fast_exp2(m_run[h] - mo);   // 0 while m_run = -inf (nothing accumulated)
          float pv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) pv[e] = fast_exp2(sv[e] - mo);   // 0 for masked keys and rows
          l_run[h] = l_run[h] * alpha[h] + ((pv[0] + pv[1]) + (pv[2] + pv[3]));
          m_run[h] = mn;
          pf[h][0] = pack2(pv[0], pv[1], BF16);
          pf[h][1] = pack2(pv[2], pv[3], BF16);
        }
        // O^T's rows 2t, 2t+1 (+ 8) take the factors of those rows (lanes 8t, 8t + 4)
#pragma unroll
        for (int h = 0; h < NT; ++h) {
          const float a_lo = __shfl_sync(0xffffffffu, alpha[h], 8 * ft);
          const float a_hi = __shfl_sync(0xffffffffu, alpha[h], (8 * ft + 4) & 31);
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            o[mt][h][0] *= a_lo;
            o[mt][h][1] *= a_hi;
            o[mt][h][2] *= a_lo;
            o[mt][h][3] *= a_hi;
          }
        }

        // ---- O^T += V^T P^T (a pool's rows past the sequence may hold
        // anything, NaN included: their V elements are cleared, since a
        // weight of 0 alone would not cancel a NaN; a branch per key instead
        // keeps the loads from running ahead, about 3x slower)
        if (!warp_wait(&bar->v_full[vslot], vpar, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const uint32_t keep_lo = (2 * ft < nvw ? 0x0000ffffu : 0u) | (2 * ft + 1 < nvw ? 0xffff0000u : 0u);
        const uint32_t keep_hi = (2 * ft + 8 < nvw ? 0x0000ffffu : 0u) | (2 * ft + 9 < nvw ? 0xffff0000u : 0u);
        const uint32_t vt = v_base + uint32_t(vslot * kGqaTile);
        const int vrow = 16 * w + 8 * (lm >> 1) + lr;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t va[4];
          ldmatrix_x4_trans(vt + sw_off(vrow, 2 * mt + (lm & 1)), va);
          va[0] &= keep_lo;
          va[1] &= keep_lo;
          va[2] &= keep_hi;
          va[3] &= keep_hi;
#pragma unroll
          for (int h = 0; h < NT; ++h) mma_16816<BF16>(o[mt][h], va[0], va[1], va[2], va[3], pf[h][0], pf[h][1]);
        }
        warp_arrive(&bar->v_free[vslot]);
      }
      if (!ok) break;

      // ---- segment end: this warp's sums of rows ra (rb)
      float l[2];
#pragma unroll
      for (int h = 0; h < NT; ++h) {
        l[h] = l_run[h];
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
      }
      // ---- the unit's rows: one partial (O / l, lse) each, or attention_out
      // and softmax_lse when the unit lies in this segment alone.  4 rows:
      // warp w takes row w % 4, elements [64 (w / 4), + 64); 16 rows: rows
      // 2w and 2w + 1, all 128 elements, in the pass (of two, 8 rows each)
      // that holds them.
      const int2 up = pl.unit_parts(sg.unit);
      const bool whole = up.y == 1;
      const bool tail = segi + 1 == nseg && !whole;
      constexpr int kRowsPerWarp = kTwo ? 2 : 1;
      constexpr int kCols = kTwo ? 4 : 2;   // elements per lane
      constexpr int NP = C::kPasses, ER = C::kERows;
      float own_o[kRowsPerWarp][kCols], own_lse[kRowsPerWarp];   // this segment's partial of the warp's slice
      for (int ps = 0; ps < NP; ++ps) {
        const int pidx = segi * NP + ps;   // passes so far: the phase of esync / efree
        // the buffers are free once every warp has read the previous pass's
        if (pidx > 0 && !warp_wait(&bar->efree, uint32_t(pidx - 1) & 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        if (ps == 0 && ft == 0) {
          if (ra < kRows) mlbuf[w * kRows + ra] = make_float2(m_run[0], l[0]);
          if (kTwo) mlbuf[w * kRows + rb] = make_float2(m_run[1], l[1]);
        }
        if (kTwo || ft < 2) {
          // rows 2t, 2t + 1 of the pass (row 2t + 1 is D further); 16 rows:
          // O^T row tile ps
          float* e0 = ebuf + (w * ER + 2 * ft) * D + fg;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const int h = kTwo ? ps : 0;
            e0[16 * mt] = o[mt][h][0];
            e0[D + 16 * mt] = o[mt][h][1];
            e0[16 * mt + 8] = o[mt][h][2];
            e0[D + 16 * mt + 8] = o[mt][h][3];
          }
        }
        warp_arrive(&bar->esync);
        if (!warp_wait(&bar->esync, uint32_t(pidx) & 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
          const int r = kTwo ? 2 * w + i : (w & 3);
          const int dcol = kTwo ? kCols * lane : 64 * (w >> 2) + kCols * lane;
          if (r >= g || (kTwo && (r >> 3) != ps)) continue;
          const int er = r - ER * ps;   // the row's place in this pass
          float M = -INFINITY;
#pragma unroll
          for (int x = 0; x < kGqaW; ++x) M = fmaxf(M, mlbuf[x * kRows + r].x);
          const float Mo = M == -INFINITY ? 0.f : M;
          float Ls = 0.f;
          float acc[kCols] = {};
#pragma unroll
          for (int x = 0; x < kGqaW; ++x) {
            const float2 ml = mlbuf[x * kRows + r];
            const float wt = fast_exp2(ml.x - Mo);
            Ls += ml.y * wt;
            const float* src = ebuf + (x * ER + er) * D + dcol;
            if constexpr (kCols == 4) {
              const float4 ov = *reinterpret_cast<const float4*>(src);
              acc[0] += wt * ov.x; acc[1] += wt * ov.y; acc[2] += wt * ov.z; acc[3] += wt * ov.w;
            } else {
              const float2 ov = *reinterpret_cast<const float2*>(src);
              acc[0] += wt * ov.x; acc[1] += wt * ov.y;
            }
          }
          const bool has = Ls > 0.f;
          const float inv = has ? 1.f / Ls : 0.f;
          const float lse = has ? (M + __log2f(Ls)) * 0.69314718055994531f : INFINITY;
          const bool lse_lane = lane == 0 && (kTwo || w < 4);
          if (whole) {
            const int head = kvh * p.group + r / p.q_tokens, tok = r % p.q_tokens;
            T* orow = reinterpret_cast<T*>(p.out) + int64_t(b) * p.out_sb + int64_t(head) * p.out_sn +
                      int64_t(tok) * p.out_ss + dcol;
            if constexpr (kCols == 4) {
              *reinterpret_cast<uint2*>(orow) =
                  make_uint2(pack2(acc[0] * inv, acc[1] * inv, BF16), pack2(acc[2] * inv, acc[3] * inv, BF16));
            } else {
              *reinterpret_cast<uint32_t*>(orow) = pack2(acc[0] * inv, acc[1] * inv, BF16);
            }
            if (lse_lane && p.lse != nullptr)
              p.lse[int64_t(b) * p.lse_sb + int64_t(head) * p.lse_sn + int64_t(tok) * p.lse_ss] = lse;
          } else {
            const int64_t part = sg.part;
            float* prow = p.part_o + (part * g + r) * D + dcol;
#pragma unroll
            for (int c = 0; c < kCols; ++c) own_o[i][c] = acc[c] * inv;
            own_lse[i] = has ? lse : -INFINITY;
            if constexpr (kCols == 4) {
              *reinterpret_cast<float4*>(prow) = make_float4(own_o[i][0], own_o[i][1], own_o[i][2], own_o[i][3]);
            } else {
              *reinterpret_cast<float2*>(prow) = make_float2(own_o[i][0], own_o[i][1]);
            }
            if (lse_lane) p.part_lse[part * g + r] = own_lse[i];
          }
        }
        warp_arrive(&bar->efree);
      }
      if (!ok) break;
      if (tail) {
        // count the unit's piece: warp 0 waits for every warp's partial
        // (the arrivals release them within the CTA), a device-scope fence
        // publishes them (cumulativity), one lane increments the counter
        warp_arrive(&bar->tail_in);
        if (w == 0) {
          if (!warp_wait(&bar->tail_in, 0u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            __threadfence();
            bar->tail_last = int(tagged_increment(p.unit_counter + sg.unit, unit_tag(p.status.epoch))) == up.y;
            mbar_arrive(&bar->tail_count);
          }
        }
        if (!warp_wait(&bar->tail_count, 0u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        if (*reinterpret_cast<volatile int*>(&bar->tail_last)) {
          // every other piece is done: merge the warp's slice in part order,
          // this piece from registers, with merge_unit's arithmetic (same
          // bits whichever CTA completes the unit)
          __threadfence();
#pragma unroll
          for (int i = 0; i < kRowsPerWarp; ++i) {
            const int r = kTwo ? 2 * w + i : (w & 3);
            const int dcol = kTwo ? kCols * lane : 64 * (w >> 2) + kCols * lane;
            if (r >= g) continue;
            constexpr int KB = 4;
            float M = -INFINITY, Ls = 0.f;
            float a[kCols] = {};
            for (int k0 = 0; k0 < up.y; k0 += KB) {
              float lk[KB], o[KB][kCols];
#pragma unroll
              for (int k = 0; k < KB; ++k) {
                const int part = up.x + k0 + k;
                const bool v = k0 + k < up.y;
                if (v && part == sg.part) {
                  lk[k] = own_lse[i];
#pragma unroll
                  for (int c = 0; c < kCols; ++c) o[k][c] = own_o[i][c];
                } else {
                  lk[k] = v ? __ldcg(p.part_lse + int64_t(part) * g + r) : -INFINITY;
                  const float* src = p.part_o + (int64_t(part) * g + r) * D + dcol;
                  if constexpr (kCols == 4) {
                    const float4 t4 = v ? __ldcg(reinterpret_cast<const float4*>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
                    o[k][0] = t4.x; o[k][1] = t4.y; o[k][2] = t4.z; o[k][3] = t4.w;
                  } else {
                    const float2 t2 = v ? __ldcg(reinterpret_cast<const float2*>(src)) : make_float2(0.f, 0.f);
                    o[k][0] = t2.x; o[k][1] = t2.y;
                  }
                }
              }
              float mb = lk[0];
#pragma unroll
              for (int k = 1; k < KB; ++k) mb = fmaxf(mb, lk[k]);
              const float m_new = fmaxf(M, mb);
              const float sc = (m_new == -INFINITY) ? 1.f : __expf(M - m_new);
#pragma unroll
              for (int c = 0; c < kCols; ++c) a[c] *= sc;
              Ls *= sc;
#pragma unroll
              for (int k = 0; k < KB; ++k) {
                const float wk = (lk[k] == -INFINITY) ? 0.f : __expf(lk[k] - m_new);
                Ls += wk;
#pragma unroll
                for (int c = 0; c < kCols; ++c) a[c] += wk * o[k][c];
              }
              M = m_new;
            }
            const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
            const int head = kvh * p.group + r / p.q_tokens, tok = r % p.q_tokens;
            T* orow = reinterpret_cast<T*>(p.out) + int64_t(b) * p.out_sb + int64_t(head) * p.out_sn +
                      int64_t(tok) * p.out_ss + dcol;
            if constexpr (kCols == 4) {
              *reinterpret_cast<uint2*>(orow) =
                  make_uint2(pack2(a[0] * inv, a[1] * inv, BF16), pack2(a[2] * inv, a[3] * inv, BF16));
            } else {
              *reinterpret_cast<uint32_t*>(orow) = pack2(a[0] * inv, a[1] * inv, BF16);
            }
            if (lane == 0 && (kTwo || w < 4) && p.lse != nullptr)
              p.lse[int64_t(b) * p.lse_sb + int64_t(head) * p.lse_sn + int64_t(tok) * p.lse_ss] =
                  Ls > 0.f ? M + __logf(Ls) : INFINITY;
          }
        }
        continue;   // not handed to the merge warp
      }
      // hand the segment to the merge warp (its 4-slot ring is reused only
      // after the merge warp took the segment 4 back).  No fence here: the
      // barrier arrival releases this warp's partial to the merge warp, whose
      // device-scope fence before the unit counter then covers it for the
      // other CTAs (cumulativity), off the compute warps' path.
      if (segi >= 4 && !warp_wait(&bar->part_free[segi & 3], uint32_t((segi >> 2) - 1) & 1u, abort_flag, p.status)) {
        ok = false;
        break;
      }
      warp_arrive(&bar->part_done[segi & 3]);
    }
  }

  __syncthreads();
  if (*abort_flag && lane == 0) {
    if (warp == kGqaW) drain_ring<kGqaKS>(bar->k_full, issued, p.status);
    if (warp == kGqaW + 1) drain_ring<VS>(bar->v_full, issued, p.status);
  }
}

template <bool BF16, int kRows>
cudaError_t launch_gqa_t(const DecodeParams& p, cudaStream_t s) {
  using C = GqaCfg<kRows>;
  cudaError_t e = set_smem_once<decode_gqa_kernel<BF16, kRows>>(C::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_cta > 0 ? p.n_cta : 1);
  cfg.blockDim = dim3(kGqaThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_gqa_kernel<BF16, kRows>, p);
}

}  // namespace

cudaError_t launch_decode_gqa(const DecodeParams& p, bool bf16, cudaStream_t s) {
  if (p.rows <= 4) return bf16 ? launch_gqa_t<true, 4>(p, s) : launch_gqa_t<false, 4>(p, s);
  if (p.rows <= 16) return bf16 ? launch_gqa_t<true, 16>(p, s) : launch_gqa_t<false, 16>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace fia
