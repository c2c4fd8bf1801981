// FP8 block-sparse attention on sm_103a.
//
// Operation: aclnnBlockSparseAttentionV2 ("计算公式", "FP8特性说明"): query,
// key and value hold float8 e4m3 values; row i of query head h is worth
// q[i] * qDequantScale[b, h, i / 128], key / value row j of kv head n is worth
// k[j] * kDequantScale[b, n, j / Y] (v likewise), Y = blockShape[1] (256 or
// 512).  out = softmax(scale * Q K^T over the blocks blockSparseMask keeps) V,
// written in bf16, plus LSE.
//
// Two kernels per call:
//   e4m3_to_f16_kernel   the value tensor, e4m3 -> f16 holding 2^-8 of each
//                        value (exact, by moving bits), into the workspace:
//                        one HBM pass instead of one conversion per CTA that
//                        reads a tile (every tile is read by several query
//                        tiles and by the Q_N / KV_N heads sharing it)
//   bsa_fp8_kernel       one CTA per 128 query rows (one quantisation block,
//                        one mask row) of one (batch, query head), walking the
//                        128-key tiles its mask row keeps:
//     warp 0      TMA producer: Q (fp8) once, then K (fp8, 16 KB) and V (f16,
//                 32 KB) tiles through a three-stage ring
//     warp 1      MMA issuer and TMEM owner:
//                   S_j = Q K_j^T   (tcgen05 kind::f8f6f4, e4m3 x e4m3 -> fp32)
//                   O  += P_j V_j   (tcgen05 kind::f16, P f16 from TMEM, V f16)
//     warps 2..5  softmax, one thread per query row: S_j * (scale * q_scale *
//                 k_scale of the tile) in log2 units, running max / sum, P
//                 times the tile's v_scale (f16) over S in TMEM, O rescaled in
//                 TMEM when the max grows by more than 2^8, epilogue
//                 2^8 O / l and LSE
// The scores use the fp8 tensor-core rate.  A tile's value scale rides on P
// (O += (P v_scale) V: v_scale is one number per tile since a tile lies in one
// quantisation block), so only P is rounded (to f16's 11 bits) and V enters
// exactly; P v_scale must stay below 65504 (v_scale < 255).  The converted V
// is finite whatever the bytes (its f16 exponent field stays below 16), so
// rows past a batch's keys need no clearing: P is 0 there.
#include "internal.h"
#include "ptx.cuh"

namespace fia {
namespace {

struct Fp8Cfg {
  static constexpr int kTile8 = 128 * 128;              // fp8 tile: 128 rows x 128 bytes
  static constexpr int kTileV = 2 * 128 * 128;          // f16 V tile: two 64-column boxes
  static constexpr int kStages = 3;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTile8;
  static constexpr int kOffV = kOffK + kStages * kTile8;
  static constexpr int kOffBar = kOffV + kStages * kTileV;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmem = kOffBar + kBarBytes + 1024;
  static constexpr int kThreads = 192;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor for kind::f8f6f4: fp32 accumulator, A and B e4m3
// (format code 0), both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(uint32_t M, uint32_t N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Two e4m3 values (bytes 0 and 1 of w, or 2 and 3 with hi) as a packed f16
// pair worth 2^-8 of them, by moving bits: e4m3 s.eeee.mmm (bias 7) placed
// as f16 s.0eeee.mmm0000000 (bias 15) reads 2^-8 times the value, normals and
// subnormals alike (an e4m3 subnormal m 2^-9 lands on the f16 subnormal
// m 2^-17).  Exact; the 2^8 goes back in the epilogue.  The e4m3 NaN
// encodings read as +-480 (they carry no number to keep).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_lo8(uint32_t w, bool hi) {
  const uint32_t t = __byte_perm(w, 0u, hi ? 0x4342u : 0x4140u);   // bytes -> low halves of the two lanes
  return ((t << 7) & 0x3f803f80u) | ((t << 8) & 0x80008000u);
}

// Tiles one query tile visits: the mask row's kept 128-key tiles (every
// tile without a mask: dense FP8 attention).
struct MaskIter {
  int n;
  const uint8_t* mrow;
  int y;
  __device__ __forceinline__ int next(int t) const {
    for (int u = t + 1; u < n; ++u)
      if (mrow == nullptr || mrow[(u * kTileN) / y] != 0) return u;
    return -1;
  }
};

// dst[i] (f16, 2^-8 of the value) = src[i] (e4m3), n bytes (a multiple of 16),
// both 16-byte aligned; a grid-stride loop of 16-byte loads and 32-byte stores.
__global__ void e4m3_to_f16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n16) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += int64_t(gridDim.x) * blockDim.x) {
    const uint4 a = __ldg(src + i);
    uint4 lo, hi;
    lo.x = e4m3x2_to_f16x2_lo8(a.x, false);
    lo.y = e4m3x2_to_f16x2_lo8(a.x, true);
    lo.z = e4m3x2_to_f16x2_lo8(a.y, false);
    lo.w = e4m3x2_to_f16x2_lo8(a.y, true);
    hi.x = e4m3x2_to_f16x2_lo8(a.z, false);
    hi.y = e4m3x2_to_f16x2_lo8(a.z, true);
    hi.z = e4m3x2_to_f16x2_lo8(a.w, false);
    hi.w = e4m3x2_to_f16x2_lo8(a.w, true);
    dst[2 * i] = lo;
    dst[2 * i + 1] = hi;
  }
}

__global__ void __launch_bounds__(192, 1) bsa_fp8_kernel(const __grid_constant__ PrefillParams p) {
  using C = Fp8Cfg;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;     // [S]
  uint64_t* v_full = bars + 4;     // [S]
  // pv_done[s]: P V of the tile in stage s is done: the stage is free and O
  // holds the tile.
  uint64_t* pv_done = bars + 7;    // [S]
  uint64_t* s_full = bars + 10;    // [2] by tile parity
  uint64_t* p_full = bars + 12;    // [2] 128 softmax arrivals
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 17);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WorkItem it = p.items[blockIdx.x];
  const BatchInfo bi = p.batches[it.b];
  const int q0 = it.q_tile * kTileM;
  const int kvh = it.h / p.group;

  MaskIter iter;
  iter.n = (bi.kv_len + kTileN - 1) / kTileN;
  iter.mrow = p.bsa_mask != nullptr
                  ? p.bsa_mask + ((int64_t(it.b) * p.num_heads + it.h) * p.bsa_nqb + q0 / p.bsa_x) * p.bsa_nkb
                  : nullptr;
  iter.y = p.bsa_y;
  // dequant scales: the query block of this CTA, the key / value block of tile t
  const float q_scale = p.fp8_qscale[(int64_t(it.b) * p.num_heads + it.h) * p.fp8_nqs + q0 / kTileM];
  const float* k_scales = p.fp8_kscale + (int64_t(it.b) * p.num_kv_heads + kvh) * p.fp8_nks;
  const float* v_scales = p.fp8_vscale + (int64_t(it.b) * p.num_kv_heads + kvh) * p.fp8_nks;

  if (threadIdx.x == 0) {
    if (blockIdx.x == 0) status_stamp(p.status);
    mbar_init(q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&pv_done[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128);
    }
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
      mbar_arrive_expect_tx(q_full, C::kTile8);
      tma_load_4d(smem + C::kOffQ, &p.tm_q, q_full, 0, q_row0, it.h, b_coord);
      int j = 0;
      for (int t = iter.next(-1); t >= 0; t = iter.next(t), ++j) {
        const int s = j % S;
        if (j >= S && !mbar_wait_lean(&pv_done[s], ((j / S) - 1) & 1, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&k_full[s], C::kTile8);
        tma_load_4d(smem + C::kOffK + s * C::kTile8, &p.tm_k, &k_full[s], 0, kv_row0 + t * kTileN, kvh, b_coord);
        mbar_arrive_expect_tx(&v_full[s], C::kTileV);
        tma_load_4d(smem + C::kOffV + s * C::kTileV, &p.tm_v, &v_full[s], 0, kv_row0 + t * kTileN, kvh, b_coord);
        tma_load_4d(smem + C::kOffV + s * C::kTileV + 128 * 128, &p.tm_v, &v_full[s], 64, kv_row0 + t * kTileN, kvh,
                    b_coord);
      }
      // On an abort, let every copy already issued land before the CTA exits.
      if (*abort_flag) {
        mbar_wait_lean(q_full, 0, nullptr, p.status);
        for (int s = 0; s < S && s < j; ++s) {
          const int last = j - 1 - ((j - 1 - s) % S);
          mbar_wait_lean(&k_full[s], (last / S) & 1, nullptr, p.status);
          mbar_wait_lean(&v_full[s], (last / S) & 1, nullptr, p.status);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_e4m3(128, 128);
      constexpr uint32_t idesc_pv = idesc_f16(128, 128, 0, 0, 1);   // f16 P and V
      const uint32_t q_base = smem_u32(smem + C::kOffQ);
      bool ok = mbar_wait_lean(q_full, 0, abort_flag, p.status);
      int j = 0;
      uint64_t* last_bar = nullptr;   // barrier and phase of the latest commit
      uint32_t last_parity = 0;
      auto issue_pv = [&](int jj) -> bool {
        const int s = jj % S;
        if (!mbar_wait_lean(&p_full[jj & 1], (jj >> 1) & 1, abort_flag, p.status)) return false;
        if (!mbar_wait_lean(&v_full[s], (jj / S) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint32_t v_base = smem_u32(smem + C::kOffV + s * C::kTileV);
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          // f16 V [keys x 128]: an MN-major B operand, 16 keys = 2048 bytes
          // per K-step, the second 64 columns one 16 KB box further
          const uint64_t bdesc = smem_desc_sw128(v_base + kk * 2048, 128 * 128, 1024);
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
          if (!mbar_wait_lean(&k_full[s], (j / S) & 1, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t k_base = smem_u32(smem + C::kOffK + s * C::kTile8);
          // 128 fp8 columns = one 128-byte swizzled row; a K-step is 32 of them
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t adesc = smem_desc_sw128(q_base + kk * 32, 16, 1024);
            const uint64_t bdesc = smem_desc_sw128(k_base + kk * 32, 16, 1024);
            mma_ss_f8(tmem + sb * 128, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
          }
          mma_commit(&s_full[sb]);
          last_bar = &s_full[sb];
          last_parity = (j >> 1) & 1;
          if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
        }
        if (ok && j >= 1) issue_pv(j - 1);
      }
      if (last_bar != nullptr) mbar_wait_lean(last_bar, last_parity, nullptr, p.status);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = 32 * (warp & 3) + lane;
    const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
    const int i = q0 + r;
    const float sl2_q = p.scale_log2 * q_scale;
    // dequant scales must be positive: any other value (<= 0, NaN) is
    // reported as FIA_ERR_UNSUPPORTED in the call's status word
    if (r == 0 && !(q_scale > 0.f)) status_raise(p.status, 5u /* FIA_ERR_UNSUPPORTED */);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    int j = 0;
    for (int t = iter.next(-1); t >= 0; t = iter.next(t), ++j) {
      const int sb = j & 1;
      const int kv0 = t * kTileN;
      // a non-positive scale is an error (reported above or here); the
      // factor is still kept above 0 so that masked scores (-inf) times it
      // stay -inf instead of NaN and the kernel runs to its end
      const float ks = k_scales[kv0 / p.bsa_y];
      const float vs = v_scales[kv0 / p.bsa_y];
      if (r == 0 && !(ks > 0.f && vs > 0.f)) status_raise(p.status, 5u /* FIA_ERR_UNSUPPORTED */);
      const float sl2 = fmaxf(sl2_q * ks, 1e-30f);
      if (!mbar_wait_lean(&s_full[sb], (j >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
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
      if (kv0 + kTileN > bi.kv_len) {
        const int lim = bi.kv_len - 1;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (kv0 + c > lim) x[c] = -INFINITY;
      }
      // the scale factor is positive, so the max of x * sl2 is max(x) * sl2
      const float m_tile = tree_max<128>(x) * sl2;
      const float m_new = fmaxf(m, m_tile);
      const float m_use = (m == -INFINITY || m_new > m + 8.f) ? m_new : m;
      const float alpha = (m_use == m) ? 1.f : fast_exp2(m - m_use);
      const float mo = (m_use == -INFINITY) ? 0.f : m_use;
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
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        if (!__all_sync(0xffffffffu, mbar_wait_lean(&pv_done[(j - 1) % S], ((j - 1) / S) & 1, abort_flag, p.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t u[32];
          tmem_ld32(tmem + lane_off + C::kColO + c * 32, u);
          tmem_wait_ld(u);
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
          tmem_st32(tmem + lane_off + C::kColO + c * 32, u);
        }
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t u[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float y0, y1;
          f2_unpack(f2_fma(f2_pack(x[c * 64 + 2 * e], x[c * 64 + 2 * e + 1]), f2_pack(vs, vs), 0ull), y0, y1);
          u[e] = pack2(y0, y1, false);   // P times the tile's value scale
        }
        tmem_st32(tmem + lane_off + sb * 128 + c * 32, u);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[j & 1]);
      m = m_use;
    }
    // ------------------------------------------------------------ epilogue
    if (ok && j > 0) {
      ok = mbar_wait_lean(&pv_done[(j - 1) % S], ((j - 1) / S) & 1, abort_flag, p.status);
      tc_fence_after();
    }
    if (ok) {
      const bool row_valid = i < bi.q_len;
      const bool has = l > 0.f;
      const float inv_l = has ? 256.f / l : 0.f;   // the f16 V tiles hold 2^-8 of V
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) +
                            (is_tnd ? int64_t(bi.q_start + i) * p.out_ss
                                    : int64_t(it.b) * p.out_sb + int64_t(i) * p.out_ss) +
                            int64_t(it.h) * p.out_sn;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
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
            w.x = pack2(__uint_as_float(u[8 * q + 0]) * inv_l, __uint_as_float(u[8 * q + 1]) * inv_l, true);
            w.y = pack2(__uint_as_float(u[8 * q + 2]) * inv_l, __uint_as_float(u[8 * q + 3]) * inv_l, true);
            w.z = pack2(__uint_as_float(u[8 * q + 4]) * inv_l, __uint_as_float(u[8 * q + 5]) * inv_l, true);
            w.w = pack2(__uint_as_float(u[8 * q + 6]) * inv_l, __uint_as_float(u[8 * q + 7]) * inv_l, true);
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

}  // namespace

cudaError_t launch_e4m3_to_f16(const void* src, void* dst, int64_t n_bytes, int n_sm, cudaStream_t s) {
  const int64_t n16 = n_bytes / 16;
  if (n16 == 0) return cudaSuccess;
  const int64_t want = (n16 + 255) / 256;
  const int blocks = int(want < int64_t(n_sm) * 8 ? want : int64_t(n_sm) * 8);
  e4m3_to_f16_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16);
  return cudaGetLastError();
}

cudaError_t launch_bsa_fp8(const PrefillParams& p, cudaStream_t s) {
  if (p.n_items == 0) return cudaSuccess;
  cudaError_t e = set_smem_once<bsa_fp8_kernel>(Fp8Cfg::kSmem);
  if (e != cudaSuccess) return e;
  bsa_fp8_kernel<<<p.n_items, Fp8Cfg::kThreads, Fp8Cfg::kSmem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace fia
