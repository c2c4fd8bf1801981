// Incremental attention for small query groups: units of at most 4 query
// rows (GQA with up to 4 query heads per kv head and one new token, or fewer
// heads with a few new tokens) and head_dim 128.
//
// Operation: the IncreFlashAttention case of npu_fused_infer_attention_score
// (as decode_kernel.cuh): out = softmax(scale * q K^T) V per (batch, head)
// over a paged or contiguous cache, per-batch actual_seq_kvlen, GQA.
//
// With 4 rows the two products of a 128-key stage are matrix-vector products
// (4 x 128 x 128 multiply-adds each), far too little work to keep a tensor
// core pipeline fed without a round trip per stage through TMEM and
// barriers.  Here they run on the CUDA cores (1024 fp32 FMAs per key and
// lane group, about a third of the HBM time of a stage at full bandwidth),
// and no warp waits on another inside a segment:
//   * the plan is decode_kernel.cuh's: units (batch, kv head), 128-token
//     stages dealt to one CTA per SM in segments, one partial per segment
//     and row, merged in part order by the CTA that completes a unit;
//   * warps 8 and 9 stream the K and V tiles of each stage into rings of NS
//     slots with TMA (128-byte swizzle, one 64-column box per 128 bytes of a
//     row), warp 10 merges finished units;
//   * compute warp w (0..7) owns keys [16 w, 16 w + 16) of every stage and
//     keeps its own running maximum, sum and O for all 4 rows; the eight
//     warps' states are combined once per segment with the exact LSE
//     weights.  Two compute warps per scheduler hide each other's latency.
//   Q K^T: lane = (key kk = lane / 8 of a pass of 4 keys, d-slice s = lane % 8
//     of 16 elements); 4 passes cover the warp's keys.  q, scaled by
//     scale * log2(e), stays in registers as fp32; a three-level
//     shuffle reduce-scatter over the 8 d-slices leaves lanes s = 2 r and
//     2 r + 1 with the score of key kk for row r.
//   P V: lane = (key parity kq = lane / 16, d-slice ds = lane % 16 of 8
//     elements); the probabilities of a key's 4 rows come from a per-warp
//     buffer in one 16-byte load.  No branch per key: the V words of keys
//     past the sequence are cleared with a mask (a branch there keeps the
//     compiler from running the loads ahead, about 3x slower).
// K and V slots are released (one arrival per compute warp) as soon as the
// warp's reads of them are done.
#include "decode_kernel.cuh"

namespace fia {

namespace {

constexpr int kGqaNS = 3;                 // K and V ring slots
constexpr int kGqaTile = 2 * 128 * 128;   // K (or V) of one 128-token stage, D = 128: two 16 KB boxes
constexpr int kGqaBox = 128 * 128;
constexpr int kGqaW = 8;                  // compute warps, 16 keys of a stage each
constexpr int kGqaThreads = (kGqaW + 3) * 32;   // + K producer, V producer, merge
constexpr int kGqaOffK = 0;
constexpr int kGqaOffV = kGqaOffK + kGqaNS * kGqaTile;
constexpr int kGqaOffE = kGqaOffV + kGqaNS * kGqaTile;      // [warp][4 rows][128] O of a segment
constexpr int kGqaOffML = kGqaOffE + kGqaW * 4 * 128 * 4;   // [warp][4 rows] (max, sum)
constexpr int kGqaOffBar = kGqaOffML + kGqaW * 4 * 8;
constexpr int kGqaBarBytes = 1024;
constexpr int kGqaSmem = kGqaOffBar + kGqaBarBytes + 1024;
static_assert(kGqaSmem <= kDecodeSmemMax, "shared memory budget");

struct GqaBars {
  uint64_t k_full[kGqaNS], v_full[kGqaNS];   // TMA landed (expect-tx)
  uint64_t k_free[kGqaNS], v_free[kGqaNS];   // every compute warp is done with the slot
  uint64_t esync, efree;                     // the warps' segment states are in / have been read
  uint64_t part_done[4], part_free[4];       // compute -> merge warp hand-off ring
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

template <bool BF16>
__global__ void __launch_bounds__(kGqaThreads, 1) decode_gqa_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  GqaBars* bar = reinterpret_cast<GqaBars*>(smem + kGqaOffBar);
  volatile int* abort_flag = &bar->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const DecodePlanRef pl = decode_plan(p);
  const int g = p.rows;

  grid_dep_launch();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGqaNS; ++s) {
      mbar_init(&bar->k_full[s], 1);
      mbar_init(&bar->v_full[s], 1);
      mbar_init(&bar->k_free[s], kGqaW);
      mbar_init(&bar->v_free[s], kGqaW);
    }
    mbar_init(&bar->esync, kGqaW);
    mbar_init(&bar->efree, kGqaW);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bar->part_done[s], kGqaW);
      mbar_init(&bar->part_free[s], 1);
    }
    bar->abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  grid_dep_wait();   // the previous kernel on the stream is complete from here on
  if (threadIdx.x == 0 && blockIdx.x == 0) status_stamp(p.status);
  const int seg_begin = p.n_cta > 0 ? pl.cta_seg(blockIdx.x) : 0;
  const int seg_end = p.n_cta > 0 ? pl.cta_seg(blockIdx.x + 1) : 0;
  const int nseg = seg_end - seg_begin;

  int issued = 0;
  if (warp == kGqaW) {
    NoQLoader nq;
    issued = decode_producer<kGqaTile, kGqaBox, 2, kGqaNS, kGqaNS>(p, pl, &p.tm_k, smem + kGqaOffK, bar->k_full,
                                                                   bar->k_free, abort_flag, seg_begin, seg_end, nq);
  } else if (warp == kGqaW + 1) {
    NoQLoader nq;
    issued = decode_producer<kGqaTile, kGqaBox, 2, kGqaNS, kGqaNS>(p, pl, &p.tm_v, smem + kGqaOffV, bar->v_full,
                                                                   bar->v_free, abort_flag, seg_begin, seg_end, nq);
  } else if (warp == kGqaW + 2) {
    merge_warp<D, BF16>(p, pl, bar->part_done, bar->part_free, abort_flag, seg_begin, nseg, lane);
  } else {
    // ------------------------------------------------------------ compute
    // Warp-synchronous tensor-core products (mma.sync m16n8k16, fp32
    // accumulate), lane (g = lane / 4, t = lane % 4) in the fragment layouts:
    //   S = Q K^T over the warp's 16 keys: A = Q (rows g < 4 real, from
    //     registers), B = K^T by ldmatrix from the swizzled K tile; lane
    //     (g, t) gets S[row g][keys 2t, 2t+1] and [8 + 2t, 9 + 2t];
    //   O^T = V^T P^T: A = V^T by ldmatrix.trans from the V tile, B = P^T,
    //     whose fragment is exactly lane (g, t)'s probabilities of row g
    //     (keys 2t, 2t+1 | 8 + 2t, 9 + 2t), so P never leaves the registers;
    //     lane (g, t) holds O^T[d = 16 m + g (+ 8)][rows 2t, 2t+1].
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    const int w = warp;
    const int fg = lane >> 2, ft = lane & 3;
    const int lr = lane & 7, lm = lane >> 3;      // ldmatrix: row of a matrix, matrix
    float* ebuf = reinterpret_cast<float*>(smem + kGqaOffE);
    float2* mlbuf = reinterpret_cast<float2*>(smem + kGqaOffML);
    const float sl2 = p.scale_log2;
    const uint32_t k_base = smem_u32(smem + kGqaOffK), v_base = smem_u32(smem + kGqaOffV);
    // byte offsets (within a stage's tile) of this lane's ldmatrix rows:
    // K: key 16 w + 8 nt + lr, element block (8 d) 4 kp + lm;
    // V: key 16 w + 8 (lm >> 1) + lr, element block 2 mt + (lm & 1)
    auto sw_off = [](int row, int col8) -> uint32_t {   // col8: 16-byte block of the row (0..15)
      return uint32_t((col8 >> 3) * kGqaBox + row * 128 + (((col8 & 7) ^ (row & 7)) << 4));
    };
    const bool row_live = fg < g;   // this lane's row g of S
    const int tok_g = fg % p.q_tokens;
    // this lane's words of the A = Q fragments of segment sg
    auto load_q = [&](const DecodeSeg& sq, uint32_t (&dst)[8][2]) {
      const uint32_t* src = nullptr;
      if (row_live) {
        const int kvh_q = sq.unit % p.num_kv_heads, b_q = sq.unit / p.num_kv_heads;
        const int head = kvh_q * p.group + fg / p.q_tokens;
        src = reinterpret_cast<const uint32_t*>(reinterpret_cast<const T*>(p.q) + int64_t(b_q) * p.q_sb +
                                                int64_t(head) * p.q_sn + int64_t(tok_g) * p.q_ss);
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        dst[ks][0] = row_live ? __ldg(src + 8 * ks + ft) : 0u;
        dst[ks][1] = row_live ? __ldg(src + 8 * ks + 4 + ft) : 0u;
      }
    };
    uint32_t qn[8][2];   // the next segment's
    bool ok = true;
    int j = 0;   // stages consumed
    for (int segi = 0; segi < nseg && ok; ++segi) {
      const DecodeSeg sg = pl.seg_at(seg_begin + segi);
      const int kvh = sg.unit % p.num_kv_heads, b = sg.unit / p.num_kv_heads;
      const int L = pl.kv_len(b);
      // several query tokens: row h is token h % Q_S and sees keys up to
      // klim + h % Q_S (sparse_mode 3: klim = S_kv - Q_S; 2: klim = 0)
      const int klim = p.q_causal == 3 ? L - p.q_tokens : 0;

      // A = Q: per 16-element step ks, Q[g][16 ks + 2t, +1] and [16 ks + 8 + 2t, +1].
      // The next segment's are loaded now, a whole segment ahead: a load
      // issued at a segment's start waits microseconds behind the KV stream.
      uint32_t qa[8][2];
      if (segi == 0) load_q(sg, qa);
      else {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          qa[ks][0] = qn[ks][0];
          qa[ks][1] = qn[ks][1];
        }
      }
      if (segi + 1 < nseg) load_q(pl.seg_at(seg_begin + segi + 1), qn);
      // this warp's running state: the maximum m (log2 units) of row g and
      // the sum of this lane's p of it relative to m; O^T
      float m_run = -INFINITY, l_run = 0.f;
      float o[8][4];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c) o[mt][c] = 0.f;

      for (int st = sg.stage_begin; st < sg.stage_end; ++st, ++j) {
        const int slot = j % kGqaNS;
        const uint32_t par = uint32_t(j / kGqaNS) & 1u;
        const int t0 = st * 128;
        const int nvalid = min(128, L - t0);
        const int nvw = nvalid - 16 * w;   // valid keys of this warp (may be <= 0 or >= 16)
        if (!warp_wait(&bar->k_full[slot], par, abort_flag, p.status)) {
          ok = false;
          break;
        }
        // ---- S = Q K^T
        const uint32_t kt = k_base + uint32_t(slot * kGqaTile);
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
            mma_16816<BF16>(sacc[nt], qa[2 * kp][0], 0u, qa[2 * kp][1], 0u, kb[0], kb[1]);
            mma_16816<BF16>(sacc[nt], qa[2 * kp + 1][0], 0u, qa[2 * kp + 1][1], 0u, kb[2], kb[3]);
          }
        }
        warp_arrive(&bar->k_free[slot]);

        // ---- online softmax of row g over the warp's keys
        const bool causal = p.q_causal != 0 && t0 + 127 > klim;   // a key of this stage is past a limit
        float sv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kl = 8 * (e >> 1) + 2 * ft + (e & 1);
          const int key = 16 * w + kl;
          const bool live = row_live && kl < nvw && (!causal || t0 + key - klim <= tok_g);
          sv[e] = live ? sacc[e >> 1][e & 1] * sl2 : -INFINITY;
        }
        float mx = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mn = fmaxf(m_run, mx);
        const float mo = mn == -INFINITY ? 0.f : mn;
        const float alpha = fast_exp2(m_run - mo);   // 0 while m_run = -inf (nothing accumulated)
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) pv[e] = fast_exp2(sv[e] - mo);   // 0 for masked keys and rows
        l_run = l_run * alpha + ((pv[0] + pv[1]) + (pv[2] + pv[3]));
        m_run = mn;
        const uint32_t pb0 = pack2(pv[0], pv[1], BF16), pb1 = pack2(pv[2], pv[3], BF16);
        // O^T's rows 2t, 2t+1 take the factors of rows 2t, 2t+1 (lanes 8t, 8t + 4)
        const float a_lo = __shfl_sync(0xffffffffu, alpha, 8 * ft);
        const float a_hi = __shfl_sync(0xffffffffu, alpha, (8 * ft + 4) & 31);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          o[mt][0] *= a_lo;
          o[mt][1] *= a_hi;
          o[mt][2] *= a_lo;
          o[mt][3] *= a_hi;
        }

        // ---- O^T += V^T P^T (a pool's rows past the sequence may hold
        // anything, NaN included: their V elements are cleared, since a
        // weight of 0 alone would not cancel a NaN)
        if (!warp_wait(&bar->v_full[slot], par, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const uint32_t keep_lo = (2 * ft < nvw ? 0x0000ffffu : 0u) | (2 * ft + 1 < nvw ? 0xffff0000u : 0u);
        const uint32_t keep_hi = (2 * ft + 8 < nvw ? 0x0000ffffu : 0u) | (2 * ft + 9 < nvw ? 0xffff0000u : 0u);
        const uint32_t vt = v_base + uint32_t(slot * kGqaTile);
        const int vrow = 16 * w + 8 * (lm >> 1) + lr;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t va[4];
          ldmatrix_x4_trans(vt + sw_off(vrow, 2 * mt + (lm & 1)), va);
          mma_16816<BF16>(o[mt], va[0] & keep_lo, va[1] & keep_lo, va[2] & keep_hi, va[3] & keep_hi, pb0, pb1);
        }
        warp_arrive(&bar->v_free[slot]);
      }
      if (!ok) break;

      // ---- segment end: this warp's sum of row g
      float l = l_run;
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      // the buffers are free once every warp has read the previous segment's
      if (segi > 0 && !warp_wait(&bar->efree, uint32_t(segi - 1) & 1u, abort_flag, p.status)) {
        ok = false;
        break;
      }
      if (ft == 0 && fg < 4) mlbuf[w * 4 + fg] = make_float2(m_run, l);
      if (ft < 2) {
        float* e0 = ebuf + (w * 4 + 2 * ft) * D + fg;   // row 2t; row 2t + 1 is D further
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          e0[16 * mt] = o[mt][0];
          e0[D + 16 * mt] = o[mt][1];
          e0[16 * mt + 8] = o[mt][2];
          e0[D + 16 * mt + 8] = o[mt][3];
        }
      }
      warp_arrive(&bar->esync);
      if (!warp_wait(&bar->esync, uint32_t(segi) & 1u, abort_flag, p.status)) {
        ok = false;
        break;
      }
      // ---- warp w finishes row w % 4, elements [64 (w / 4), + 64), of the
      // unit: one partial (O / l, lse), or attention_out and softmax_lse when
      // the unit lies in this segment alone
      const int r = w & 3;
      const int dcol = 64 * (w >> 2) + 2 * lane;
      const bool whole = pl.unit_parts(sg.unit).y == 1;
      if (r < g) {
        float M = -INFINITY;
#pragma unroll
        for (int x = 0; x < kGqaW; ++x) M = fmaxf(M, mlbuf[x * 4 + r].x);
        const float Mo = M == -INFINITY ? 0.f : M;
        float Ls = 0.f;
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int x = 0; x < kGqaW; ++x) {
          const float2 ml = mlbuf[x * 4 + r];
          const float wt = fast_exp2(ml.x - Mo);
          Ls += ml.y * wt;
          const float2 ov = *reinterpret_cast<const float2*>(ebuf + (x * 4 + r) * D + dcol);
          acc.x += wt * ov.x;
          acc.y += wt * ov.y;
        }
        const bool has = Ls > 0.f;
        const float inv = has ? 1.f / Ls : 0.f;
        const float lse = has ? (M + __log2f(Ls)) * 0.69314718055994531f : INFINITY;
        if (whole) {
          const int head = kvh * p.group + r / p.q_tokens, tok = r % p.q_tokens;
          T* orow = reinterpret_cast<T*>(p.out) + int64_t(b) * p.out_sb + int64_t(head) * p.out_sn +
                    int64_t(tok) * p.out_ss + dcol;
          *reinterpret_cast<uint32_t*>(orow) = pack2(acc.x * inv, acc.y * inv, BF16);
          if (w < 4 && lane == 0 && p.lse != nullptr)
            p.lse[int64_t(b) * p.lse_sb + int64_t(head) * p.lse_sn + int64_t(tok) * p.lse_ss] = lse;
        } else {
          const int64_t part = sg.part;
          *reinterpret_cast<float2*>(p.part_o + (part * g + r) * D + dcol) = make_float2(acc.x * inv, acc.y * inv);
          if (w < 4 && lane == 0) p.part_lse[part * g + r] = has ? lse : -INFINITY;
        }
      }
      warp_arrive(&bar->efree);
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
    if (warp == kGqaW) drain_ring<kGqaNS>(bar->k_full, issued, p.status);
    if (warp == kGqaW + 1) drain_ring<kGqaNS>(bar->v_full, issued, p.status);
  }
}

template <bool BF16>
cudaError_t launch_gqa_t(const DecodeParams& p, cudaStream_t s) {
  cudaError_t e = set_smem_once<decode_gqa_kernel<BF16>>(kGqaSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_cta > 0 ? p.n_cta : 1);
  cfg.blockDim = dim3(kGqaThreads);
  cfg.dynamicSmemBytes = kGqaSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_gqa_kernel<BF16>, p);
}

}  // namespace

cudaError_t launch_decode_gqa(const DecodeParams& p, bool bf16, cudaStream_t s) {
  if (p.rows > 4) return cudaErrorInvalidValue;
  return bf16 ? launch_gqa_t<true>(p, s) : launch_gqa_t<false>(p, s);
}

}  // namespace fia
