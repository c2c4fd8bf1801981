// Prefill attention with two query tiles per CTA: every sparse_mode, contiguous
// or paged K/V, head dims 64/64, 128/128 and 192/128 (MLA prefill).
//
// Operation: as prefill.cu -- torch_npu.npu_prompt_flash_attention ("功能说明",
// formula) and npu_fused_infer_attention_score_v2 (Q_S > 1, softmax_lse):
// out = softmax(scale * Q K^T + mask) V with sparse_mode 0 (no mask), the
// causal modes 2 / 3 and the band mode 4 computed from indices, or an explicit
// atten_mask (sparse_mode 0 with a mask, 1) read from memory.
//
// One CTA owns 256 query rows of one (batch, query head): tile A (rows
// q0..q0+127) and tile B (q0+128..q0+255).  Both read every K/V tile the CTA
// loads, and the tensor core alternates between them: while warpgroup A
// exponentiates S_A(j), the MMA warp runs P_B(j-1) V and Q_B K(j)^T, and the
// other way round, so the softmax of one tile hides behind the products of the
// other (one tile alone leaves the tensor core idle while its softmax runs).
//   warp 0      TMA producer: Q_A and Q_B once, K and V tiles through rings
//               of their own; after the first tile it warms L2 with the Q of
//               the item that will take this CTA's SM about one item later
//   warp 1      MMA issuer (one thread) and TMEM owner, in the order
//                 P_A(j) V, Q_A K(j+1)^T, P_B(j) V, Q_B K(j+1)^T
//   warps 2..5  softmax of tile A, warps 6..9 softmax of tile B: one thread
//               per query row (= TMEM lane), running max / sum in registers,
//               P written over S in TMEM, O rescaled in TMEM when the max grows
//               by more than 2^8, epilogue O / l and LSE.
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256, 256+DV), O_B [256+DV,
// 256+2DV).  Causal: tile B needs the K/V tiles of tile A plus at most one; the
// CTA walks tile B's range and tile A stops early.
// Paged K/V (chunked prefill against a block table): the producer takes each
// 128-key tile from its block (block_size is a multiple of 128).
// Explicit mask: a summary pass first gives every 128 x 128 tile of the mask
// a code (no key masked / some / all); a CTA walks only from its rows' first
// to their last tile with a visible key.  For a tile with some keys masked
// each softmax thread copies its row's 128 mask bytes into its own 128-byte
// shared slot (cp.async, one tile ahead) and turns them into a 128-bit mask;
// fully visible tiles need no bytes, and for a fully masked one (or a warp
// whose rows are all masked) the warp writes P = 0 and skips its softmax.
#include "internal.h"
#include "ptx.cuh"

namespace fia {
namespace {

// DQK: head dim of the scores (Q and K; 192 = MLA's 128 + 64 rope columns),
// DV: head dim of V and O.  K and V have rings of their own: a K stage is free
// once its last Q K^T is done, a V stage once its last P V is.  kM: the
// explicit-mask layout, whose 32 KB of mask slots take, at DQK 192, one of
// the two K stages.
template <int DQK, int DV, bool kM = false>
struct PairCfg {
  static constexpr int kChunksQK = DQK / 64;
  static constexpr int kChunksV = DV / 64;
  static constexpr int kBoxBytes = 128 * 128;
  static constexpr int kTileQK = kChunksQK * kBoxBytes;
  static constexpr int kTileV = kChunksV * kBoxBytes;
  static constexpr int kKStages = DQK == 64 ? 3 : (DQK == 192 && kM) ? 1 : 2;
  static constexpr int kVStages = DQK == 64 ? 3 : DQK == 128 ? 2 : 1;
  static constexpr int kOffQ = 0;                                   // Q_A, Q_B
  static constexpr int kOffK = kOffQ + 2 * kTileQK;
  static constexpr int kOffV = kOffK + kKStages * kTileQK;
  static constexpr int kOffBar = kOffV + kVStages * kTileV;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmem = kOffBar + kBarBytes + 1024;
  // explicit atten_mask: one 128-byte slot per softmax thread (256 rows),
  // 16-byte chunk q of row r at (q ^ (r & 7)) * 16 (no bank conflicts)
  static constexpr int kOffMask = kOffBar + kBarBytes;
  static constexpr int kSmemMask = kOffMask + 256 * 128 + 1024;
  static constexpr bool kMaskFits = kSmemMask <= 227 * 1024;
  static constexpr int kThreads = 320;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;                            // O_A; O_B at kColO + DV
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  static_assert(kKStages <= 3 && kVStages <= 3, "barrier slots");
};

// Tile codes of an explicit atten_mask: one CTA per 128 x 128 tile of one
// mask slice, code 0 when no byte of the tile is nonzero, 2 when every byte
// is, 1 otherwise (rows and columns past the mask are left out).  Thread t
// reads 64 bytes of row t / 2: four 16-byte loads when rows are 16-byte
// aligned, single bytes otherwise.
__global__ void __launch_bounds__(256) mask_tile_summary_kernel(const uint8_t* __restrict__ mask, int64_t s1,
                                                                int64_t s2, int cs, uint8_t* __restrict__ codes) {
  const int kt = blockIdx.x, qt = blockIdx.y, b = blockIdx.z;
  const int64_t row = int64_t(qt) * kTileM + (threadIdx.x >> 1);
  const int64_t c0 = int64_t(kt) * kTileN + (threadIdx.x & 1) * 64;
  bool any = false, all = true;
  if (row < s1 && c0 < s2) {
    const uint8_t* src = mask + (int64_t(b) * s1 + row) * s2 + c0;
    const int n = int(min(int64_t(64), s2 - c0));
    if (cs == 16 && n == 64) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + q);
        any |= (v.x | v.y | v.z | v.w) != 0u;
        all &= (nonzero_bytes4(v.x) & nonzero_bytes4(v.y) & nonzero_bytes4(v.z) & nonzero_bytes4(v.w)) == 0xfu;
      }
    } else {
      for (int c = 0; c < n; ++c) {
        const bool nz = __ldg(src + c) != 0;
        any |= nz;
        all &= nz;
      }
    }
  }
  const int a = __syncthreads_or(any), l = __syncthreads_and(all);
  if (threadIdx.x == 0) codes[(int64_t(b) * gridDim.y + qt) * gridDim.x + kt] = uint8_t(l ? 2 : (a ? 1 : 0));
}

// Key tiles needed by the query rows [qa, qa + 128) of a batch.
__device__ __forceinline__ int tiles_for_rows(const BatchInfo& bi, int qa, int mode, int diag_off) {
  if (mode != kCausal) return (bi.kv_len + kTileN - 1) / kTileN;
  const int last_row = min(qa + kTileM - 1, bi.q_len - 1);
  const int maxkey = min(bi.kv_len - 1, last_row + diag_off);
  return maxkey >= 0 ? maxkey / kTileN + 1 : 0;
}

template <int DQK, int DV, bool BF16, int MODE>
__global__ void __launch_bounds__(320, 1) prefill_pair_kernel(const __grid_constant__ PrefillParams p) {
  using C = PairCfg<DQK, DV, MODE == kMask>;
  constexpr int KS = C::kKStages, VS = C::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;     // [KS]
  uint64_t* v_full = bars + 4;     // [VS]
  // v_free[s]: P_B V of the tile in V stage s is done (one commit per MMA
  // group): the stage is free, and O_B holds it.
  uint64_t* v_free = bars + 7;     // [VS]
  // s_full[3 t + s]: S_t of the tile in K stage s is in TMEM.  The last one of
  // a tile (S_B, or S_A when the pair has no tile B) also frees the K stage.
  uint64_t* s_full = bars + 10;    // [2][3]
  uint64_t* pa_full = bars + 16;   // [2] by tile parity: warpgroup A's P is in (4 warp arrivals)
  uint64_t* pb_full = bars + 18;   // [2]
  // pva_done: tile A's last P V is done (its epilogue may read O_A).  Earlier
  // P_A V products need no commit of their own: each is followed on the
  // tensor pipe by a Q K^T whose commit covers it.
  uint64_t* pva_done = bars + 20;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 21);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 22);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WorkItem it = p.items[blockIdx.x];
  const BatchInfo bi = p.batches[it.b];
  const int q0 = it.q_tile * 2 * kTileM;
  const int kvh = it.h / p.group;
  const int diag_off = (MODE == kCausal && p.causal_offset_mode == 3) ? (bi.kv_len - bi.q_len) : 0;
  int na = tiles_for_rows(bi, q0, MODE, diag_off);
  // Tile B walks at least tile A's range (its rows past the batch are computed
  // but not written); a pair whose tile B starts past the batch runs tile A
  // alone.  nl = tiles the CTA loads; the last tile product of each K/V tile
  // (tile B's when it has rows, else tile A's) releases the stage.
  const bool has_b = q0 + kTileM < bi.q_len;
  int nb = has_b ? max(na, tiles_for_rows(bi, q0 + kTileM, MODE, diag_off)) : 0;
  // sparse_mode 4 (band) and the explicit mask (band i - pre .. i + next): both
  // tiles walk the K/V tiles of the union of their rows' bands, from tile jt0
  // on; the softmax masks each row's edges.
  int jt0 = 0;
  const int64_t band_d = MODE == kBand ? int64_t(bi.kv_len) - bi.q_len : 0;
  if (MODE == kBand || MODE == kMask) {
    const int64_t last = min(q0 + 2 * kTileM - 1, bi.q_len - 1);
    const int64_t lo = max(int64_t(0), q0 + band_d - p.band_pre);
    const int64_t hi = min(int64_t(bi.kv_len) - 1, last + band_d + p.band_next);
    const int n = hi < lo ? 0 : int(hi / kTileN - lo / kTileN + 1);
    jt0 = hi < lo ? 0 : int(lo / kTileN);
    // tile A's rows end earlier: it stops after its own last key's tile
    const int64_t last_a = min(q0 + kTileM - 1, bi.q_len - 1);
    const int64_t hi_a = min(int64_t(bi.kv_len) - 1, last_a + band_d + p.band_next);
    na = (hi < lo || hi_a < lo) ? 0 : int(hi_a / kTileN - lo / kTileN + 1);
    nb = has_b ? n : 0;
  }
  // explicit mask: walk only from the first to the last tile in which some
  // key of the tile's rows is visible (tile codes from the summary pass);
  // all-masked tiles inside that range take the P = 0 path below
  const uint8_t* mtc = MODE == kMask ? p.mask_tiles + int64_t(it.b) * p.mask_tiles_sb : nullptr;
  const int qta = q0 / kTileM;   // row tile of tile A in the mask (tile B: qta + 1)
  if (MODE == kMask && nb + na > 0) {
    int fa = -1, la = -1, fb = -1, lb = -1;
    for (int j = 0; j < na; ++j)
      if (mtc[int64_t(qta) * p.mask_nkt + jt0 + j] != 2) { fa = fa < 0 ? j : fa; la = j; }
    for (int j = 0; j < nb; ++j)
      if (mtc[int64_t(qta + 1) * p.mask_nkt + jt0 + j] != 2) { fb = fb < 0 ? j : fb; lb = j; }
    const int first = fa < 0 ? fb : (fb < 0 ? fa : min(fa, fb));
    if (first < 0) {
      na = nb = 0;
    } else {
      jt0 += first;
      na = la < 0 ? 0 : la - first + 1;
      // tile B releases every stage the CTA loads: it walks at least tile A's range
      nb = has_b ? max(na, lb < 0 ? 0 : lb - first + 1) : 0;
    }
  }
  const int nl = max(na, nb);

  if (threadIdx.x == 0) {
    if (blockIdx.x == 0) status_stamp(p.status);
    mbar_init(q_full, 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&s_full[3 + s], 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_free[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&pa_full[t], 4);
      mbar_init(&pb_full[t], 4);
    }
    mbar_init(pva_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const bool is_tnd = p.is_tnd != 0;
  const int q_row0 = is_tnd ? bi.q_start + q0 : q0;
  const int kv_row0 = is_tnd && p.block_table == nullptr ? bi.kv_start : 0;
  const int b_coord = is_tnd ? 0 : it.b;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      // 64-column chunks of Q / K: the first 128 columns from tm_q / tm_k, a
      // third (DQK = 192) from tm_qr / tm_kr at column rope_col (a separate
      // rope tensor, or columns 128..191 of the same one)
      auto qk_src = [&](int c, const CUtensorMap* m, const CUtensorMap* mr, int& col) -> const CUtensorMap* {
        col = c < 2 ? c * 64 : p.rope_col;
        return c < 2 ? m : mr;
      };
      mbar_arrive_expect_tx(q_full, 2 * C::kTileQK);
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int c = 0; c < C::kChunksQK; ++c) {
          int col;
          const CUtensorMap* m = qk_src(c, &p.tm_q, &p.tm_qr, col);
          tma_load_4d(smem + C::kOffQ + t * C::kTileQK + c * C::kBoxBytes, m, q_full, col, q_row0 + t * kTileM, it.h,
                      b_coord);
        }
      // the Q K^T that frees a K stage: tile B's, or tile A's without a tile B
      uint64_t* k_rel = s_full + (nb > 0 ? 3 : 0);
      int j = 0, nk = 0, nv = 0;   // tiles loaded; K and V loads issued
      for (; j < nl; ++j) {
        const int sk = j % KS, sv = j % VS;
        // K/V tile coordinates: (row, batch) of a contiguous tensor, or (row in
        // block, block id) of a paged pool (the table read overlaps the wait)
        const int key = (jt0 + j) * kTileN;
        int kv_r = kv_row0 + key, kv_b = b_coord;
        if (p.block_table != nullptr) {
          kv_b = __ldg(p.block_table + int64_t(it.b) * p.table_stride + key / p.block_size);
          kv_r = key % p.block_size;
        }
        if (j >= KS && !mbar_wait_lean(&k_rel[sk], ((j / KS) - 1) & 1, abort_flag, p.status)) break;
        uint8_t* ks = smem + C::kOffK + sk * C::kTileQK;
        mbar_arrive_expect_tx(&k_full[sk], C::kTileQK);
#pragma unroll
        for (int c = 0; c < C::kChunksQK; ++c) {
          int col;
          const CUtensorMap* m = qk_src(c, &p.tm_k, &p.tm_kr, col);
          tma_load_4d(ks + c * C::kBoxBytes, m, &k_full[sk], col, kv_r, kvh, kv_b);
        }
        nk = j + 1;
        if (j >= VS && !mbar_wait_lean(&v_free[sv], ((j / VS) - 1) & 1, abort_flag, p.status)) break;
        uint8_t* vs = smem + C::kOffV + sv * C::kTileV;
        mbar_arrive_expect_tx(&v_full[sv], C::kTileV);
#pragma unroll
        for (int c = 0; c < C::kChunksV; ++c)
          tma_load_4d(vs + c * C::kBoxBytes, &p.tm_v, &v_full[sv], c * 64, kv_r, kvh, kv_b);
        nv = j + 1;
        if (j == 0 && p.prefetch_stride > 0 && int(blockIdx.x) + p.prefetch_stride < p.n_items) {
          // Q of the item that takes this CTA's place about one item from now
          // (CTAs start in index order, one per SM): into L2, so its first
          // loads do not wait on HBM
          const WorkItem nx = p.items[blockIdx.x + p.prefetch_stride];
          const BatchInfo nb_info = p.batches[nx.b];
          const int nq0 = nx.q_tile * 2 * kTileM;
          const int nrow = is_tnd ? nb_info.q_start + nq0 : nq0;
          const int nbc = is_tnd ? 0 : nx.b;
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int c = 0; c < C::kChunksQK; ++c) {
              int col;
              const CUtensorMap* m = qk_src(c, &p.tm_q, &p.tm_qr, col);
              tma_prefetch_l2_4d(m, col, nrow + t * kTileM, nx.h, nbc);
            }
        }
      }
      if (*abort_flag) {
        // let every copy in flight land before the CTA exits
        mbar_wait_lean(q_full, 0, nullptr, p.status);
        for (int s = 0; s < KS && s < nk; ++s) {
          const int last = nk - 1 - ((nk - 1 - s) % KS);
          mbar_wait_lean(&k_full[s], (last / KS) & 1, nullptr, p.status);
        }
        for (int s = 0; s < VS && s < nv; ++s) {
          const int last = nv - 1 - ((nv - 1 - s) % VS);
          mbar_wait_lean(&v_full[s], (last / VS) & 1, nullptr, p.status);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16(128, 128, BF16 ? 1 : 0, 0, 0);
      constexpr uint32_t idesc_pv = idesc_f16(128, DV, BF16 ? 1 : 0, 0, 1);
      // Descriptors of every operand buffer, built once; an MMA's K-slice
      // only moves the start address (bits 0..13, in 16-byte units), which
      // stays below 2^14 here, so a constant added to the whole descriptor
      // selects it.
      const uint64_t qd0 = smem_desc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
      const uint64_t qd1 = smem_desc_sw128(smem_u32(smem + C::kOffQ + C::kTileQK), 16, 1024);
      const uint64_t kd0 = smem_desc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
      const uint64_t vd0 = smem_desc_sw128(smem_u32(smem + C::kOffV), C::kBoxBytes, 1024);
      constexpr uint64_t kStepK = C::kTileQK >> 4, kStepV = C::kTileV >> 4;
      uint64_t* last_bar = nullptr;   // barrier and phase of the latest commit
      uint32_t last_parity = 0;
      bool ok = mbar_wait_lean(q_full, 0, abort_flag, p.status);
      // A K/V stage is waited for once, by the first product that reads it
      // (tile A's, unless the tile is past tile A's range).
      // S_t = Q_t K(j)^T
      auto qk = [&](int t, int j) -> bool {
        const int s = j % KS;
        if ((t == 0 || j >= na) && !mbar_wait_lean(&k_full[s], (j / KS) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint64_t qd = t == 0 ? qd0 : qd1;
        const uint64_t kd = kd0 + uint64_t(s) * kStepK;
        const uint32_t dst = tmem + t * 128;
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint64_t off = uint64_t(((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4);
          mma_ss(dst, qd + off, kd + off, idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[3 * t + s]);
        last_bar = &s_full[3 * t + s];
        last_parity = (j / KS) & 1;
        return true;
      };
      // O_t += P_t(j) V(j): P read from tile t's S columns in TMEM; V is
      // [keys x DV], an MN-major operand (16 keys = 2048 bytes per K-step, the
      // next 64 columns of DV one box further)
      auto pv = [&](int t, int j) -> bool {
        const int s = j % VS;
        if (!mbar_wait_lean(t == 0 ? &pa_full[j & 1] : &pb_full[j & 1], (j >> 1) & 1, abort_flag, p.status)) return false;
        if ((t == 0 || j >= na) && !mbar_wait_lean(&v_full[s], (j / VS) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint64_t vd = vd0 + uint64_t(s) * kStepV;
        const uint32_t dst = tmem + C::kColO + t * DV;
        const uint32_t pt = tmem + t * 128;
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk)
          mma_ts(dst, pt + kk * 8, vd + uint64_t((kk * 2048) >> 4), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        if (t == 0 && nb > 0) {
          if (j == na - 1) {
            mma_commit(pva_done);
            last_bar = pva_done;
            last_parity = 0;
          }
        } else {
          mma_commit(&v_free[s]);
          last_bar = &v_free[s];
          last_parity = (j / VS) & 1;
        }
        return true;
      };
      if (ok && na > 0) ok = qk(0, 0);
      if (ok && nb > 0) ok = qk(1, 0);
      for (int j = 0; j < nl && ok; ++j) {
        if (j < na) {
          ok = pv(0, j);
          if (ok && j + 1 < na) ok = qk(0, j + 1);
        }
        if (ok && j < nb) {
          ok = pv(1, j);
          if (ok && j + 1 < nb) ok = qk(1, j + 1);
        }
      }
      // Every MMA issued has finished before TMEM goes: the latest commit
      // tracks them all (the one before it on the same barrier has completed).
      if (last_bar != nullptr) mbar_wait_lean(last_bar, last_parity, nullptr, p.status);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 2) >> 2;              // 0: tile A, 1: tile B
    const int r = 32 * (warp & 3) + lane;
    const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
    const uint32_t col_s = t * 128;
    const uint32_t col_o = C::kColO + t * DV;
    const int n = t == 0 ? na : nb;
    const int tile_q0 = q0 + t * kTileM;
    const int i = tile_q0 + r;
    const int diag = i + diag_off;
    const float sl2 = p.scale_log2;
    uint64_t* my_pfull = t == 0 ? pa_full : pb_full;
    // explicit mask: this row's bytes of K/V tile jj into the thread's slot
    const bool mrow = MODE == kMask && i < bi.q_len;
    const uint8_t* mask_row = MODE == kMask ? p.attn_mask + int64_t(it.b) * p.mask_sb + int64_t(i) * p.mask_ss : nullptr;
    uint8_t* mslot = smem + C::kOffMask + (t * 128 + r) * 128;
    const int r7 = r & 7;
    auto mask_fetch = [&](int jj) {
      const int kvj = (jt0 + jj) * kTileN;
      const int valid = min(bi.kv_len - kvj, kTileN);   // bytes of the row inside the batch
      const uint8_t* src = mask_row + kvj;
      const uint32_t dst = smem_u32(mslot);
      if (p.mask_cs == 16) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (16 * q < valid) cp_async_zfill<16>(dst + ((q ^ r7) << 4), src + 16 * q, min(16, valid - 16 * q));
      } else if (p.mask_cs == 8) {
#pragma unroll
        for (int h = 0; h < 16; ++h)
          if (8 * h < valid)
            cp_async_zfill<8>(dst + (((h >> 1) ^ r7) << 4) + (h & 1) * 8, src + 8 * h, min(8, valid - 8 * h));
      } else if (p.mask_cs == 4) {
#pragma unroll
        for (int h = 0; h < 32; ++h)
          if (4 * h < valid)
            cp_async_zfill<4>(dst + (((h >> 2) ^ r7) << 4) + (h & 3) * 4, src + 4 * h, min(4, valid - 4 * h));
      } else {
#pragma unroll 4
        for (int c = 0; c < kTileN; ++c)
          if (c < valid) mslot[(((c >> 4) ^ r7) << 4) + (c & 15)] = __ldg(src + c);
      }
      cp_async_commit();
    };
    // tile code of this tile's rows for K/V tile jj (explicit mask)
    auto mcode = [&](int jj) -> int { return MODE == kMask ? mtc[int64_t(qta + t) * p.mask_nkt + jt0 + jj] : 0; };
    if (mrow && n > 0 && mcode(0) == 1) mask_fetch(0);
    // Rows of V past the batch's keys may hold anything (even NaN); P is 0
    // there but 0 * NaN is not, so they are cleared before the first P V that
    // reads tile jj: tile A's if it uses the tile, else tile B's.
    auto clear_v_tail = [&](int jj, int kv0j) -> bool {
      const int s = jj % VS;
      if (!__all_sync(0xffffffffu, mbar_wait_lean(&v_full[s], (jj / VS) & 1, abort_flag, p.status))) return false;
      if (r >= bi.kv_len - kv0j) {
        uint8_t* vs = smem + C::kOffV + s * C::kTileV;
#pragma unroll
        for (int c = 0; c < C::kChunksV; ++c)
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4*>(vs + c * C::kBoxBytes + r * 128 + q * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      return true;
    };
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      // mb: bit c of mb[c >> 5] set when atten_mask masks key kv0 + c
      uint32_t mb[4] = {0u, 0u, 0u, 0u};
      const int code = mcode(j);
      if (MODE == kMask && code == 2) {
        mb[0] = mb[1] = mb[2] = mb[3] = 0xffffffffu;   // every key of the tile masked for every row
        if (mrow && j + 1 < n && mcode(j + 1) == 1) mask_fetch(j + 1);
      } else if (MODE == kMask && code == 0) {
        if (mrow && j + 1 < n && mcode(j + 1) == 1) mask_fetch(j + 1);
      } else if (mrow) {
        cp_async_wait_all();
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint4 a0 = *reinterpret_cast<const uint4*>(mslot + (((2 * w) ^ r7) << 4));
          const uint4 a1 = *reinterpret_cast<const uint4*>(mslot + (((2 * w + 1) ^ r7) << 4));
          mb[w] = nonzero_bytes4(a0.x) | (nonzero_bytes4(a0.y) << 4) | (nonzero_bytes4(a0.z) << 8) |
                  (nonzero_bytes4(a0.w) << 12) | (nonzero_bytes4(a1.x) << 16) | (nonzero_bytes4(a1.y) << 20) |
                  (nonzero_bytes4(a1.z) << 24) | (nonzero_bytes4(a1.w) << 28);
        }
        // the slot is read (mb depends on every byte): refill it with the next tile
        if (j + 1 < n && mcode(j + 1) == 1) mask_fetch(j + 1);
      }
      if (!__all_sync(0xffffffffu, mbar_wait_lean(&s_full[3 * t + j % KS], (j / KS) & 1, abort_flag, p.status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (MODE == kMask && __all_sync(0xffffffffu, (mb[0] & mb[1] & mb[2] & mb[3]) == 0xffffffffu)) {
        // the mask hides every key of this tile from all of the warp's rows:
        // P = 0, and the max, the sum and O stay as they are (what the full
        // path computes, bit for bit, from a row of -inf)
        uint32_t z[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) z[e] = 0u;
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_st16(tmem + lane_off + col_s + c * 16, z);
        const int kv0 = (jt0 + j) * kTileN;
        if (kv0 + kTileN > bi.kv_len && (t == 0 || j >= na) && !clear_v_tail(j, kv0)) {
          ok = false;
          break;
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(&my_pfull[j & 1]);
        continue;
      }
      // S in two halves: the second half's load is in flight while the
      // first half is masked and reduced.
      uint32_t su[4][32];
      tmem_ld32(tmem + lane_off + col_s, su[0]);
      tmem_ld32(tmem + lane_off + col_s + 32, su[1]);
      tmem_wait_ld(su[0]);
      tmem_regs_after_wait(su[1]);
      tmem_ld32(tmem + lane_off + col_s + 64, su[2]);
      tmem_ld32(tmem + lane_off + col_s + 96, su[3]);
      float* x = reinterpret_cast<float*>(&su[0][0]);
      const int kv0 = (jt0 + j) * kTileN;
      const bool ragged = kv0 + kTileN > bi.kv_len;
      // keys allowed for this row: [lim_lo, lim]
      int lim = (MODE == kCausal) ? min(bi.kv_len - 1, diag) : bi.kv_len - 1;
      int lim_lo = 0;
      constexpr bool kBanded = MODE == kBand || MODE == kMask;
      if (kBanded) {
        lim = int(min(int64_t(bi.kv_len) - 1, int64_t(i) + band_d + p.band_next));
        lim_lo = int(max(int64_t(0), int64_t(i) + band_d - p.band_pre));
      }
      const bool need_mask = ragged || (MODE == kCausal && kv0 + kTileN - 1 > tile_q0 + diag_off) ||
                             (kBanded && (kv0 + kTileN - 1 > lim || kv0 < lim_lo)) ||
                             (MODE == kMask && (mb[0] | mb[1] | mb[2] | mb[3]) != 0u);
      float a[8];
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (kv0 + c > lim || (kBanded && kv0 + c < lim_lo) || (MODE == kMask && ((mb[c >> 5] >> (c & 31)) & 1u)))
            su[c >> 5][c & 31] = __float_as_uint(-INFINITY);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k)
        a[k] = fmax3(__uint_as_float(su[0][k]), __uint_as_float(su[0][8 + k]), __uint_as_float(su[0][16 + k]));
#pragma unroll
      for (int k = 0; k < 8; ++k) a[k] = fmax3(a[k], __uint_as_float(su[0][24 + k]), __uint_as_float(su[1][k]));
#pragma unroll
      for (int k = 0; k < 8; ++k)
        a[k] = fmax3(a[k], __uint_as_float(su[1][8 + k]), __uint_as_float(su[1][16 + k]));
#pragma unroll
      for (int k = 0; k < 8; ++k) a[k] = fmaxf(a[k], __uint_as_float(su[1][24 + k]));
      tmem_wait_ld(su[2]);
      tmem_regs_after_wait(su[3]);
      if (need_mask) {
#pragma unroll
        for (int c = 64; c < 128; ++c)
          if (kv0 + c > lim || (kBanded && kv0 + c < lim_lo) || (MODE == kMask && ((mb[c >> 5] >> (c & 31)) & 1u)))
            su[c >> 5][c & 31] = __float_as_uint(-INFINITY);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k)
        a[k] = fmax3(a[k], __uint_as_float(su[2][k]), __uint_as_float(su[2][8 + k]));
#pragma unroll
      for (int k = 0; k < 8; ++k)
        a[k] = fmax3(a[k], __uint_as_float(su[2][16 + k]), __uint_as_float(su[2][24 + k]));
#pragma unroll
      for (int k = 0; k < 8; ++k) a[k] = fmax3(a[k], __uint_as_float(su[3][k]), __uint_as_float(su[3][8 + k]));
#pragma unroll
      for (int k = 0; k < 8; ++k)
        a[k] = fmax3(a[k], __uint_as_float(su[3][16 + k]), __uint_as_float(su[3][24 + k]));
      const float m_tile = fmax3(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
      const float m_new = fmaxf(m, m_tile * sl2);
      // Keep a stale max unless it grows by more than 8 (log2 units): p <= 2^8
      // stays exact in fp32 and representable in bf16/f16.
      const float m_use = (m == -INFINITY || m_new > m + 8.f) ? m_new : m;
      const float alpha = (m_use == m) ? 1.f : fast_exp2(m - m_use);
      const float mo = (m_use == -INFINITY) ? 0.f : m_use;
      // p = 2^(s * scale * log2(e) - m) in packed pairs, written back as P
      // (16-bit pairs over the first 64 columns of S) 32 keys at a time.
      const uint64_t sc2 = f2_pack(sl2, sl2), nmo2 = f2_pack(-mo, -mo);
      uint64_t acc2[2] = {0ull, 0ull};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t u[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float y0, y1;
          f2_unpack(f2_fma(f2_pack(x[32 * c + 2 * e], x[32 * c + 2 * e + 1]), sc2, nmo2), y0, y1);
          y0 = fast_exp2(y0);
          y1 = fast_exp2(y1);
          acc2[e & 1] = f2_add(acc2[e & 1], f2_pack(y0, y1));
          u[e] = pack2(y0, y1, BF16);
        }
        tmem_st16(tmem + lane_off + col_s + c * 16, u);
      }
      float s0, s1;
      f2_unpack(f2_add(acc2[0], acc2[1]), s0, s1);
      l = l * alpha + (s0 + s1);
      // O_t holds P_t(j-1) V already: Q_t K(j)^T, whose S this thread just
      // read, was issued after that P V on the same tensor pipe.
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < DV / 16; ++c) {
          uint32_t u[16];
          tmem_ld16(tmem + lane_off + col_o + c * 16, u);
          tmem_wait_ld(u);
#pragma unroll
          for (int e = 0; e < 16; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
          tmem_st16(tmem + lane_off + col_o + c * 16, u);
        }
      }
      if (ragged && (t == 0 || j >= na) && !clear_v_tail(j, kv0)) {
        ok = false;
        break;
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(&my_pfull[j & 1]);
      m = m_use;
    }
    if (MODE == kMask) cp_async_wait_all();   // no copy into the slot outlives the loop
    // ------------------------------------------------------------ epilogue
    if (ok && n > 0) {
      const int jl = n - 1;
      ok = __all_sync(0xffffffffu, (t == 0 && nb > 0)
                                       ? mbar_wait_lean(pva_done, 0, abort_flag, p.status)
                                       : mbar_wait_lean(&v_free[jl % VS], (jl / VS) & 1, abort_flag, p.status));
      tc_fence_after();
    }
    if (ok) {
      const bool row_valid = i < bi.q_len;
      const bool has = l > 0.f;
      const float inv_l = has ? 1.f / l : 0.f;
      using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
      T* orow = reinterpret_cast<T*>(p.out) + (is_tnd ? int64_t(bi.q_start + i) * p.out_ss
                                                       : int64_t(it.b) * p.out_sb + int64_t(i) * p.out_ss) +
                int64_t(it.h) * p.out_sn;
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t u[32];
        if (n > 0) {
          tmem_ld32(tmem + lane_off + col_o + c * 32, u);
          tmem_wait_ld(u);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = 0u;
        }
        if (row_valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack2(__uint_as_float(u[8 * q + 0]) * inv_l, __uint_as_float(u[8 * q + 1]) * inv_l, BF16);
            w.y = pack2(__uint_as_float(u[8 * q + 2]) * inv_l, __uint_as_float(u[8 * q + 3]) * inv_l, BF16);
            w.z = pack2(__uint_as_float(u[8 * q + 4]) * inv_l, __uint_as_float(u[8 * q + 5]) * inv_l, BF16);
            w.w = pack2(__uint_as_float(u[8 * q + 6]) * inv_l, __uint_as_float(u[8 * q + 7]) * inv_l, BF16);
            if (!has) w = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(orow + c * 32 + q * 8) = w;
          }
        }
      }
      if (row_valid && p.lse != nullptr) {
        const float lse = has ? (m + __log2f(l)) * 0.69314718055994531f : INFINITY;
        float* lp = p.lse + (is_tnd ? int64_t(bi.q_start + i) * p.lse_ss
                                    : int64_t(it.b) * p.lse_sb + int64_t(i) * p.lse_ss) +
                    int64_t(it.h) * p.lse_sn;
        *lp = lse;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int DQK, int DV, bool BF16, int MODE>
cudaError_t launch_pair_one(const PrefillParams& p, cudaStream_t s) {
  using C = PairCfg<DQK, DV, MODE == kMask>;
  static_assert(MODE != kMask || C::kMaskFits, "mask slots do not fit beside the rings");
  auto k = prefill_pair_kernel<DQK, DV, BF16, MODE>;
  constexpr int smem = MODE == kMask ? C::kSmemMask : C::kSmem;
  cudaError_t e = set_smem_once<prefill_pair_kernel<DQK, DV, BF16, MODE>>(smem);
  if (e != cudaSuccess) return e;
  k<<<p.n_items, C::kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mask_tile_summary(const uint8_t* mask, int64_t s1, int64_t s2, int n_mb, int cs, uint8_t* codes,
                                     cudaStream_t s) {
  const int64_t nqt = (s1 + kTileM - 1) / kTileM, nkt = (s2 + kTileN - 1) / kTileN;
  if (nqt == 0 || nkt == 0 || n_mb == 0) return cudaSuccess;
  if (nqt > 65535 || n_mb > 65535 || nkt > 0x7fffffff) return cudaErrorInvalidValue;
  mask_tile_summary_kernel<<<dim3(unsigned(nkt), unsigned(nqt), unsigned(n_mb)), 256, 0, s>>>(mask, s1, s2, cs, codes);
  return cudaGetLastError();
}

cudaError_t launch_prefill_pair(const PrefillParams& p, int head_dim_qk, int head_dim_v, bool bf16, int mode,
                                cudaStream_t s) {
  if (p.n_items == 0) return cudaSuccess;
#define FIA_PAIR_MODES(DQ, DV, BB)                                          \
  switch (mode) {                                                           \
    case kDense: return launch_pair_one<DQ, DV, BB, kDense>(p, s);          \
    case kCausal: return launch_pair_one<DQ, DV, BB, kCausal>(p, s);        \
    case kBand: return launch_pair_one<DQ, DV, BB, kBand>(p, s);            \
    case kMask: return launch_pair_one<DQ, DV, BB, kMask>(p, s);            \
    default: return cudaErrorInvalidValue;                                  \
  }
  if (head_dim_qk == 128 && head_dim_v == 128) {
    if (bf16) { FIA_PAIR_MODES(128, 128, true) } else { FIA_PAIR_MODES(128, 128, false) }
  }
  if (head_dim_qk == 64 && head_dim_v == 64) {
    if (bf16) { FIA_PAIR_MODES(64, 64, true) } else { FIA_PAIR_MODES(64, 64, false) }
  }
  if (head_dim_qk == 192 && head_dim_v == 128) {
    if (bf16) { FIA_PAIR_MODES(192, 128, true) } else { FIA_PAIR_MODES(192, 128, false) }
  }
#undef FIA_PAIR_MODES
  return cudaErrorInvalidValue;
}

}  // namespace fia
