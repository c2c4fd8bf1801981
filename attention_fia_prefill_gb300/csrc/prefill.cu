// Prefill attention on sm_103a: out = softmax(scale * Q K^T + mask) V, plus LSE.
//
// Operation: torch_npu.npu_prompt_flash_attention ("功能说明", formula) and
// npu_fused_infer_attention_score_v2 (Q_S > 1 path, softmax_lse output); the
// block-sparse variant is aclnnBlockSparseAttentionV2 ("计算公式"), where each
// 128-row query tile only visits the KV tiles that blockSparseMask selects.
//
// One CTA owns 128 query rows of one (batch, query head).  Roles:
//   warp 0      TMA producer: Q once, then K/V tiles through a ring of stages
//   warp 1      MMA issuer (one thread) and TMEM owner:
//                 S_j = Q K_j^T   (tcgen05, SS, fp32 accumulator in TMEM)
//                 O  += P_j V_j   (tcgen05, P read from TMEM)
//   warps 2..5  softmax: one thread per query row (= TMEM lane); reads S_j from
//               TMEM, masks, keeps the running max/sum in registers, writes P_j
//               (bf16/f16), rescales O in TMEM when the max grows by more than
//               2^8, and runs the epilogue (O / l, LSE).
// TMEM columns: S0 [0,128), S1 [128,256), O [256, 256 + D); P_j overwrites
// the first 64 columns of S_j as packed 16-bit pairs.
// Shared memory tiles are 128 rows x 128 bytes boxes with the 128-byte swizzle
// that both TMA and the tcgen05 shared-memory descriptors understand.
#include "internal.h"
#include "ptx.cuh"

namespace fia {

template <int D>
struct PrefillCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kBoxBytes = 128 * 128;
  static constexpr int kTileBytes = kChunks * kBoxBytes;
  static constexpr int kStages = 3;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kTileBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemUsed = kOffBar + kBarBytes + 1024;
  // at least ~120 KB so that a second CTA never shares the SM (and its TMEM)
  static constexpr int kSmem = kSmemUsed < 122880 ? 122880 : kSmemUsed;
  static constexpr int kThreads = 192;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;
};

// Iterates the KV tiles one query tile visits, in ascending order.
struct TileIter {
  int n;                       // tiles [0, n) are candidates
  const uint8_t* mrow;         // block-sparse: mask row, else nullptr
  int y;                       // block-sparse: keys per mask column
  __device__ __forceinline__ int next(int t) const {
    for (int u = t + 1; u < n; ++u)
      if (mrow == nullptr || mrow[(u * kTileN) / y] != 0) return u;
    return -1;
  }
};

template <int D, bool BF16, int MODE>
__global__ void __launch_bounds__(192, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
  using C = PrefillCfg<D>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = bars + 4;
  // pv_done[s] completes each time P_t V_t of a tile t in stage s has been
  // accumulated: it frees the stage for the producer and tells the softmax
  // that O is up to date.  One tcgen05.commit per group of MMAs -- a second
  // commit straight after the first does not wait for them.
  uint64_t* pv_done = bars + 7;
  uint64_t* s_full = bars + 10;
  // p_full[t & 1] takes the 128 softmax threads' arrivals for tile t: a warp
  // may run one tile ahead of the others (S_{t+1} can be ready before every
  // warp has arrived for tile t), never two (S_{t+2} needs P_t V_t issued).
  uint64_t* p_full = bars + 12;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 17);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WorkItem it = p.items[blockIdx.x];
  const BatchInfo bi = p.batches[it.b];
  const int q0 = it.q_tile * kTileM;
  const int kvh = it.h / p.group;
  const int diag_off = (MODE == kCausal && p.causal_offset_mode == 3) ? (bi.kv_len - bi.q_len) : 0;

  TileIter iter;
  iter.mrow = nullptr;
  iter.y = kTileN;
  if (MODE == kCausal) {
    const int last_row = min(q0 + kTileM - 1, bi.q_len - 1);
    const int maxkey = min(bi.kv_len - 1, last_row + diag_off);
    iter.n = maxkey >= 0 ? maxkey / kTileN + 1 : 0;
  } else {
    iter.n = (bi.kv_len + kTileN - 1) / kTileN;
  }
  if (MODE == kBlockSparse) {
    const int qb = q0 / p.bsa_x;
    iter.mrow = p.bsa_mask + ((int64_t(it.b) * p.num_heads + it.h) * p.bsa_nqb + qb) * p.bsa_nkb;
    iter.y = p.bsa_y;
  }

  if (threadIdx.x == 0) {
    if (blockIdx.x == 0) status_stamp(p.status);
    mbar_init(q_full, 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(&p_full[0], 128);
    mbar_init(&p_full[1], 128);
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
  const int kv_row0 = is_tnd ? bi.kv_start : 0;
  const int b_coord = is_tnd ? 0 : it.b;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      mbar_arrive_expect_tx(q_full, C::kTileBytes);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_4d(smem + C::kOffQ + c * C::kBoxBytes, &p.tm_q, q_full, c * 64, q_row0, it.h, b_coord);
      int j = 0;
      for (int t = iter.next(-1); t >= 0; t = iter.next(t), ++j) {
        const int s = j % S;
        if (j >= S && !mbar_wait(&pv_done[s], ((j / S) - 1) & 1, abort_flag, p.status)) break;
        uint8_t* ks = smem + C::kOffK + s * C::kTileBytes;
        uint8_t* vs = smem + C::kOffV + s * C::kTileBytes;
        mbar_arrive_expect_tx(&k_full[s], C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(ks + c * C::kBoxBytes, &p.tm_k, &k_full[s], c * 64, kv_row0 + t * kTileN, kvh, b_coord);
        mbar_arrive_expect_tx(&v_full[s], C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(vs + c * C::kBoxBytes, &p.tm_v, &v_full[s], c * 64, kv_row0 + t * kTileN, kvh, b_coord);
      }
      // On an abort, let every copy already issued land before the CTA exits.
      if (*abort_flag) {
        for (int s = 0; s < S && s < j; ++s) {
          const int last = j - 1 - ((j - 1 - s) % S);   // last tile issued into stage s
          mbar_wait(&k_full[s], (last / S) & 1, nullptr, p.status);
          mbar_wait(&v_full[s], (last / S) & 1, nullptr, p.status);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16(128, 128, BF16 ? 1 : 0, 0, 0);
      constexpr uint32_t idesc_pv = idesc_f16(128, D, BF16 ? 1 : 0, 0, 1);
      const uint32_t q_base = smem_u32(smem + C::kOffQ);
      bool ok = mbar_wait(q_full, 0, abort_flag, p.status);
      int j = 0;
      uint64_t* last_bar = nullptr;   // barrier and phase of the latest commit
      uint32_t last_parity = 0;
      auto issue_pv = [&](int jj) -> bool {
        const int s = jj % S;
        if (!mbar_wait(&p_full[jj & 1], (jj >> 1) & 1, abort_flag, p.status)) return false;
        if (!mbar_wait(&v_full[s], (jj / S) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint32_t v_base = smem_u32(smem + C::kOffV + s * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          // V is [keys x D] with D contiguous: an MN-major B operand.  A K-step
          // of 16 keys is 16 rows = 2048 bytes; the next 64 columns of D sit
          // one 16 KB box further (leading byte offset).
          const uint64_t bdesc = smem_desc_sw128(v_base + kk * 2048, C::kBoxBytes, 1024);
          mma_ts(tmem + C::kColO, tmem + (jj & 1) * 128 + kk * 8, bdesc, idesc_pv, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&pv_done[s]);
        last_bar = &pv_done[s];
        last_parity = (jj / S) & 1;
        return true;
      };
      if (ok) {
        for (int t = iter.next(-1); t >= 0; t = iter.next(t), ++j) {
          const int s = j % S;
          const int sb = j & 1;
          if (!mbar_wait(&k_full[s], (j / S) & 1, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t k_base = smem_u32(smem + C::kOffK + s * C::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kBoxBytes + (kk & 3) * 32;
            const uint64_t adesc = smem_desc_sw128(q_base + off, 16, 1024);
            const uint64_t bdesc = smem_desc_sw128(k_base + off, 16, 1024);
            mma_ss(tmem + sb * 128, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
          }
          mma_commit(&s_full[sb]);
          last_bar = &s_full[sb];
          last_parity = (j >> 1) & 1;
          if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
        }
        if (ok && j >= 1) issue_pv(j - 1);
      }
      // Every MMA this thread issued has finished before TMEM goes: the latest
      // commit tracks them all (the one before it has completed, so its barrier
      // is at most one phase behind).
      if (last_bar != nullptr) mbar_wait(last_bar, last_parity, nullptr, p.status);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = 32 * (warp & 3) + lane;
    const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
    const int i = q0 + r;
    const int diag = i + diag_off;
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    int j = 0;
    for (int t = iter.next(-1); t >= 0; t = iter.next(t), ++j) {
      const int sb = j & 1;
      if (!mbar_wait(&s_full[sb], (j >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      uint32_t su[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_off + sb * 128 + c * 32, su[c]);
      tmem_wait_ld(su[0]);
#pragma unroll
      for (int c = 1; c < 4; ++c) tmem_regs_after_wait(su[c]);
      float x[128];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(su[c][e]);
      const int kv0 = t * kTileN;
      const bool ragged = kv0 + kTileN > bi.kv_len;
      const bool need_mask = ragged || (MODE == kCausal && kv0 + kTileN - 1 > q0 + diag_off);
      if (need_mask) {
        const int lim = (MODE == kCausal) ? min(bi.kv_len - 1, diag) : bi.kv_len - 1;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (kv0 + c > lim) x[c] = -INFINITY;
      }
      const float m_tile = tree_max<128>(x) * sl2;
      const float m_new = fmaxf(m, m_tile);
      // Keep a stale max unless it grows by more than 8 (log2 units): p <= 2^8
      // stays exact in fp32 and representable in bf16/f16.
      const float m_use = (m == -INFINITY || m_new > m + 8.f) ? m_new : m;
      const float alpha = (m_use == m) ? 1.f : fast_exp2(m - m_use);
      const float mo = (m_use == -INFINITY) ? 0.f : m_use;
      // p = 2^(s * scale * log2(e) - m) in packed pairs; the row sum in the
      // same order as the two-tile kernel's, so an all-ones block-sparse mask
      // reproduces dense prefill bit for bit.
      {
        const uint64_t sc2 = f2_pack(sl2, sl2), nmo2 = f2_pack(-mo, -mo);
        uint64_t acc2[2] = {0ull, 0ull};
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          float y0, y1;
          f2_unpack(f2_fma(f2_pack(x[2 * e], x[2 * e + 1]), sc2, nmo2), y0, y1);
          y0 = fast_exp2(y0);
          y1 = fast_exp2(y1);
          acc2[e & 1] = f2_add(acc2[e & 1], f2_pack(y0, y1));
          x[2 * e] = y0;
          x[2 * e + 1] = y1;
        }
        float s0, s1;
        f2_unpack(f2_add(acc2[0], acc2[1]), s0, s1);
        l = l * alpha + (s0 + s1);
      }
      // O only has to hold P_{j-1} V_{j-1} when this warp rescales it; the next
      // P V accumulates after it on the tensor pipe anyway.
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[(j - 1) % S], ((j - 1) / S) & 1, abort_flag, p.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        {
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
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t u[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) u[e] = pack2(x[c * 64 + 2 * e], x[c * 64 + 2 * e + 1], BF16);
        tmem_st32(tmem + lane_off + sb * 128 + c * 32, u);
      }
      if (ragged) {
        // Rows of V past the batch's keys may hold anything (even NaN); P is 0
        // there but 0 * NaN is not, so clear them before the PV product.
        const int s = j % S;
        if (!mbar_wait(&v_full[s], (j / S) & 1, abort_flag, p.status)) { ok = false; break; }
        if (r >= bi.kv_len - kv0) {
          uint8_t* vs = smem + C::kOffV + s * C::kTileBytes;
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<uint4*>(vs + c * C::kBoxBytes + r * 128 + q * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[j & 1]);
      m = m_use;
    }
    // ------------------------------------------------------------ epilogue
    if (ok && j > 0) {
      ok = mbar_wait(&pv_done[(j - 1) % S], ((j - 1) / S) & 1, abort_flag, p.status);
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
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        if (j > 0) {
          tmem_ld32(tmem + lane_off + C::kColO + c * 32, u);
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

template <int D, bool BF16, int MODE>
static cudaError_t launch_one(const PrefillParams& p, cudaStream_t s) {
  using C = PrefillCfg<D>;
  auto k = prefill_kernel<D, BF16, MODE>;
  cudaError_t e = set_smem_once<prefill_kernel<D, BF16, MODE>>(C::kSmem);
  if (e != cudaSuccess) return e;
  k<<<p.n_items, C::kThreads, C::kSmem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillParams& p, int head_dim, bool bf16, int mode, cudaStream_t s) {
  if (p.n_items == 0) return cudaSuccess;
#define FIA_DISPATCH_MODE(DD, BB)                                                            \
  switch (mode) {                                                                          \
    case kDense: return launch_one<DD, BB, kDense>(p, s);                        \
    case kCausal: return launch_one<DD, BB, kCausal>(p, s);                      \
    case kBlockSparse: return launch_one<DD, BB, kBlockSparse>(p, s);            \
    default: return cudaErrorInvalidValue;                                                 \
  }
  if (head_dim == 128) {
    if (bf16) { FIA_DISPATCH_MODE(128, true) } else { FIA_DISPATCH_MODE(128, false) }
  } else if (head_dim == 64) {
    if (bf16) { FIA_DISPATCH_MODE(64, true) } else { FIA_DISPATCH_MODE(64, false) }
  }
#undef FIA_DISPATCH_MODE
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------------
// Rows that no prefill CTA writes: padding rows past a batch's actual query
// length (mode 0) or every row (mode 1, e.g. K/V with S2 = 0).  They receive
// attention_out = 0 and softmax_lse = +inf.
// dims = {B, N, S, D}; out_strides/lse_strides = (b, n, s) element strides.
// ------------------------------------------------------------------------
__global__ void fill_rows_kernel(uint16_t* out, float* lse, int64_t B, int64_t N, int64_t Sq, int64_t D,
                                 int64_t osb, int64_t osn, int64_t oss, int64_t lsb, int64_t lsn, int64_t lss,
                                 const BatchInfo* batches, int mode) {
  const int64_t row = int64_t(blockIdx.x) * blockDim.y + threadIdx.y;
  if (row >= B * N * Sq) return;
  const int64_t s = row % Sq, n = (row / Sq) % N, b = row / (Sq * N);
  if (mode == 0 && s < batches[b].q_len) return;
  for (int64_t d = threadIdx.x; d < D; d += blockDim.x) out[b * osb + n * osn + s * oss + d] = 0;
  if (lse != nullptr && threadIdx.x == 0) lse[b * lsb + n * lsn + s * lss] = INFINITY;
}

cudaError_t launch_fill_rows(void* out, bool /*half_type*/, float* lse, const int64_t* dims,
                             const int64_t* os, const int64_t* ls, const BatchInfo* batches, int mode,
                             cudaStream_t st) {
  const int64_t rows = dims[0] * dims[1] * dims[2];
  if (rows == 0) return cudaSuccess;
  dim3 block(32, 8);
  const int64_t grid = (rows + 7) / 8;
  fill_rows_kernel<<<(unsigned)grid, block, 0, st>>>(static_cast<uint16_t*>(out), lse, dims[0], dims[1], dims[2],
                                                    dims[3], os[0], os[1], os[2], ls ? ls[0] : 0, ls ? ls[1] : 0,
                                                    ls ? ls[2] : 0, batches, mode);
  return cudaGetLastError();
}

}  // namespace fia
