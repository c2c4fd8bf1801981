// Incremental (Q_S = 1) attention over a paged or contiguous KV cache.
//
// Operation: npu_fused_infer_attention_score_v2 / aclnnFusedInferAttentionScoreV5
// in the IncreFlashAttention case: out = softmax(scale * q K^T) V for one query
// token per (batch, head), with GQA (query head h reads kv head h / (Q_N/KV_N)),
// per-batch actual_seq_kvlen, and PageAttention (token j of batch b lives in
// block block_table[b][j / block_size], row j % block_size).
//
// The work is memory bound (about 4 flop per KV byte), so it runs on CUDA
// cores, laid out for HBM streaming:
//   * each unit (batch, kv head, block of up to G query heads) is cut into
//     128-token stages; all stages are dealt out evenly to one CTA per SM;
//   * warp 8 streams the K and V rows of each stage into a 3-deep shared-memory
//     ring with TMA (128-byte swizzle, so row reads are bank-conflict free);
//   * warps 0..7 take 16 tokens each: scores with lanes split over (token,
//     half of D), an online softmax per warp, then P V with lanes split over D;
//     packed fp32x2 FMAs do the arithmetic;
//   * at the end of each unit a CTA merges its 8 warps and writes one partial
//     (O / l, lse); fia_decode_combine merges the partials of every unit in a
//     fixed order (deterministic, no atomics).
#include "internal.h"
#include "ptx.cuh"

namespace fia {

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t ra = *reinterpret_cast<uint64_t*>(&a), rb = *reinterpret_cast<uint64_t*>(&b),
           rc = *reinterpret_cast<uint64_t*>(&c), rd;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  return *reinterpret_cast<float2*>(&rd);
}

template <bool BF16>
__device__ __forceinline__ float2 cvt2(uint32_t w) {
  if constexpr (BF16) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  } else {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
  }
}

template <bool BF16>
__device__ __forceinline__ float to_f32(const void* base, int64_t idx) {
  if constexpr (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
  else return __half2float(reinterpret_cast<const __half*>(base)[idx]);
}

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <int D, int G>
struct DecodeCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kStageBytes = 128 * 128 * kChunks;   // K (or V) of one stage
  static constexpr int kStages = (D == 128 && G == 8) ? 2 : 3;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kStages * kStageBytes;
  static constexpr int kOffQ = kOffV + kStages * kStageBytes;          // f32 [G][D]
  static constexpr int kOffP = kOffQ + G * D * 4;                      // f32 [8][16][G]
  static constexpr int kOffMO = kOffP + 8 * 16 * G * 4;                // f32 [8][G][D]
  static constexpr int kOffML = kOffMO + 8 * G * D * 4;                // f32 [8][G] m, [8][G] l
  static constexpr int kOffBar = kOffML + 2 * 8 * G * 4;
  static constexpr int kSmem = kOffBar + 64 + 1024;
  static constexpr int kThreads = 288;
};

template <int D, bool BF16, int G>
__global__ void __launch_bounds__(288, 1) decode_kernel(const __grid_constant__ DecodeParams p) {
  using C = DecodeCfg<D, G>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* empty = full + 3;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + 6);
  float* q_s = reinterpret_cast<float*>(smem + C::kOffQ);
  float* p_s = reinterpret_cast<float*>(smem + C::kOffP);
  float* mo_s = reinterpret_cast<float*>(smem + C::kOffMO);
  float* mm_s = reinterpret_cast<float*>(smem + C::kOffML);
  float* ml_s = mm_s + 8 * G;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg_begin = p.cta_seg[blockIdx.x], seg_end = p.cta_seg[blockIdx.x + 1];

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 8);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      int j = 0;
      bool ok = true;
      for (int si = seg_begin; si < seg_end && ok; ++si) {
        const DecodeSeg sg = p.segs[si];
        const int hb = sg.unit % p.head_blocks;
        const int kvh = (sg.unit / p.head_blocks) % p.num_kv_heads;
        const int b = sg.unit / (p.head_blocks * p.num_kv_heads);
        (void)hb;
        const int L = p.kv_len[b];
        for (int st = sg.stage_begin; st < sg.stage_end; ++st, ++j) {
          const int s = j % S;
          if (j >= S && !mbar_wait(&empty[s], ((j / S) - 1) & 1, abort_flag, p.status)) { ok = false; break; }
          const int t0 = st * 128;
          const int nvalid = min(128, L - t0);
          const int nbox = (nvalid + p.box_rows - 1) / p.box_rows;
          mbar_arrive_expect_tx(&full[s], 2u * C::kChunks * nbox * p.box_rows * 128u);
          uint8_t* ks = smem + C::kOffK + s * C::kStageBytes;
          uint8_t* vs = smem + C::kOffV + s * C::kStageBytes;
          for (int k = 0; k < nbox; ++k) {
            const int tok = t0 + k * p.box_rows;
            int64_t row;
            if (p.block_table != nullptr) {
              const int64_t blk = p.block_table[int64_t(b) * p.table_stride + tok / p.block_size];
              row = blk * p.row_per_blk + int64_t(kvh) * p.row_per_head + (tok % p.block_size);
            } else {
              row = int64_t(b) * p.row_per_blk + int64_t(kvh) * p.row_per_head + tok;
            }
            const int col0 = kvh * p.col_per_head;
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {
              const int off = c * 128 * 128 + k * p.box_rows * 128;
              tma_load_2d(ks + off, &p.tm_k, &full[s], col0 + c * 64, int(row));
              tma_load_2d(vs + off, &p.tm_v, &full[s], col0 + c * 64, int(row));
            }
          }
        }
      }
      if (*abort_flag) {
        for (int s = 0; s < S && s < j; ++s) {
          const int last = j - 1 - ((j - 1 - s) % S);
          mbar_wait(&full[s], (last / S) & 1, nullptr, p.status);
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int tid = threadIdx.x;          // 0..255
  const int tl = lane & 15, half = lane >> 4;
  const int r_qk = warp * 16 + tl;      // stage row this lane scores
  constexpr int kDPL = D / 32;          // d values per lane in P V
  int j = 0;
  bool ok = true;
  for (int si = seg_begin; si < seg_end; ++si) {
    const DecodeSeg sg = p.segs[si];
    const int hb = sg.unit % p.head_blocks;
    const int kvh = (sg.unit / p.head_blocks) % p.num_kv_heads;
    const int b = sg.unit / (p.head_blocks * p.num_kv_heads);
    const int L = p.kv_len[b];
    const int h0 = kvh * p.group + hb * G;
    const int nh = min(G, p.group - hb * G);

    named_bar(1, 256);   // previous segment fully done with q_s and the merge area
    for (int idx = tid; idx < G * D; idx += 256) {
      const int h = idx / D, d = idx % D;
      q_s[idx] = (h < nh) ? to_f32<BF16>(p.q, int64_t(b) * p.q_sb + int64_t(h0 + h) * p.q_sn + d) * p.scale_log2
                          : 0.f;
    }
    named_bar(1, 256);

    float m[G], l[G];
    float2 o[G][kDPL / 2 > 0 ? kDPL / 2 : 1];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int e = 0; e < (kDPL / 2 > 0 ? kDPL / 2 : 1); ++e) o[h][e] = make_float2(0.f, 0.f);
    }

    for (int st = sg.stage_begin; st < sg.stage_end && ok; ++st, ++j) {
      const int s = j % S;
      ok = mbar_wait(&full[s], (j / S) & 1, abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const uint8_t* ks = smem + C::kOffK + s * C::kStageBytes;
      const uint8_t* vs = smem + C::kOffV + s * C::kStageBytes;
      const int nvalid = min(128, L - st * 128);

      // ---- scores: lane (tl, half) covers row r_qk, half of D
      float2 acc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = make_float2(0.f, 0.f);
#pragma unroll
      for (int cc = 0; cc < D / 16; ++cc) {
        const int c = half * (D / 16) + cc;
        const int box = c >> 3, kc = c & 7;
        const uint4 kw =
            *reinterpret_cast<const uint4*>(ks + box * 16384 + r_qk * 128 + ((kc ^ (r_qk & 7)) << 4));
        const float2 k01 = cvt2<BF16>(kw.x), k23 = cvt2<BF16>(kw.y), k45 = cvt2<BF16>(kw.z),
                     k67 = cvt2<BF16>(kw.w);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 qa = *reinterpret_cast<const float4*>(q_s + h * D + c * 8);
          const float4 qb = *reinterpret_cast<const float4*>(q_s + h * D + c * 8 + 4);
          acc[h] = fma2(k01, make_float2(qa.x, qa.y), acc[h]);
          acc[h] = fma2(k23, make_float2(qa.z, qa.w), acc[h]);
          acc[h] = fma2(k45, make_float2(qb.x, qb.y), acc[h]);
          acc[h] = fma2(k67, make_float2(qb.z, qb.w), acc[h]);
        }
      }
      const bool valid = r_qk < nvalid;
      float pr[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float sc = acc[h].x + acc[h].y;
        sc += __shfl_xor_sync(0xffffffffu, sc, 16);
        sc = valid ? sc : -INFINITY;
        float mx = sc;
#pragma unroll
        for (int o2 = 8; o2 >= 1; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
        const float m_new = fmaxf(m[h], mx);
        const float alpha = (m_new == -INFINITY) ? 1.f : fast_exp2(m[h] - m_new);
        const float pv = (sc == -INFINITY) ? 0.f : fast_exp2(sc - m_new);
        float sum = pv;
#pragma unroll
        for (int o2 = 8; o2 >= 1; o2 >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o2);
        l[h] = l[h] * alpha + sum;
        m[h] = m_new;
#pragma unroll
        for (int e = 0; e < (kDPL / 2 > 0 ? kDPL / 2 : 1); ++e) {
          o[h][e].x *= alpha;
          o[h][e].y *= alpha;
        }
        pr[h] = pv;
      }
      float* pw = p_s + warp * 16 * G;
      if (half == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) pw[tl * G + h] = pr[h];
      }
      __syncwarp();

      // ---- P V: lane covers kDPL consecutive d of every row of this warp
      const int nrows = min(16, nvalid - warp * 16);
      for (int t = 0; t < nrows; ++t) {
        const int r = warp * 16 + t;
        float ph[G];
#pragma unroll
        for (int h = 0; h < G; ++h) ph[h] = pw[t * G + h];
        if constexpr (D == 128) {
          const int box = lane >> 4, kc = (lane & 15) >> 1, hf = lane & 1;
          const uint2 vw =
              *reinterpret_cast<const uint2*>(vs + box * 16384 + r * 128 + ((kc ^ (r & 7)) << 4) + hf * 8);
          const float2 v01 = cvt2<BF16>(vw.x), v23 = cvt2<BF16>(vw.y);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            o[h][0] = fma2(make_float2(ph[h], ph[h]), v01, o[h][0]);
            o[h][1] = fma2(make_float2(ph[h], ph[h]), v23, o[h][1]);
          }
        } else {
          const int kc = lane >> 2, q4 = lane & 3;
          const uint32_t vw = *reinterpret_cast<const uint32_t*>(vs + r * 128 + ((kc ^ (r & 7)) << 4) + q4 * 4);
          const float2 v01 = cvt2<BF16>(vw);
#pragma unroll
          for (int h = 0; h < G; ++h) o[h][0] = fma2(make_float2(ph[h], ph[h]), v01, o[h][0]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ---- merge the 8 warps of this CTA and write one partial for the segment
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        mm_s[warp * G + h] = m[h];
        ml_s[warp * G + h] = l[h];
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int e = 0; e < (kDPL / 2 > 0 ? kDPL / 2 : 1); ++e) {
        const int d = lane * kDPL + 2 * e;
        mo_s[(warp * G + h) * D + d] = o[h][e].x;
        mo_s[(warp * G + h) * D + d + 1] = o[h][e].y;
      }
    }
    named_bar(1, 256);
    for (int idx = tid; idx < G * D; idx += 256) {
      const int h = idx / D, d = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < 8; ++w) M = fmaxf(M, mm_s[w * G + h]);
      float Ls = 0.f, O = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const float f = fast_exp2(mm_s[w * G + h] - M);
          Ls += ml_s[w * G + h] * f;
          O += mo_s[(w * G + h) * D + d] * f;
        }
      }
      const bool has = Ls > 0.f;
      p.part_o[(int64_t(sg.part) * G + h) * D + d] = has ? O / Ls : 0.f;
      if (d == 0) p.part_lse[int64_t(sg.part) * G + h] = has ? (M + __log2f(Ls)) * 0.69314718055994531f : -INFINITY;
    }
  }
}

// Merge the partials of every (batch, query head): one warp each, fixed order.
template <int D, bool BF16, int G>
__global__ void decode_combine_kernel(const __grid_constant__ DecodeParams p) {
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= p.batch * p.num_heads) return;
  const int b = gw / p.num_heads, h = gw % p.num_heads;
  const int kvh = h / p.group, hg = h % p.group, hb = hg / G, hl = hg % G;
  const int unit = (b * p.num_kv_heads + kvh) * p.head_blocks + hb;
  const int2 up = p.unit_parts[unit];
  float M = -INFINITY;
  for (int k = 0; k < up.y; ++k) M = fmaxf(M, p.part_lse[int64_t(up.x + k) * G + hl]);
  constexpr int kDPL = D / 32;
  float acc[kDPL];
#pragma unroll
  for (int e = 0; e < kDPL; ++e) acc[e] = 0.f;
  float Ls = 0.f;
  if (M != -INFINITY) {
    for (int k = 0; k < up.y; ++k) {
      const float lk = p.part_lse[int64_t(up.x + k) * G + hl];
      const float w = __expf(lk - M);
      Ls += w;
      const float* po = p.part_o + (int64_t(up.x + k) * G + hl) * D + lane * kDPL;
#pragma unroll
      for (int e = 0; e < kDPL; ++e) acc[e] += w * po[e];
    }
  }
  const bool has = Ls > 0.f;
  const float inv = has ? 1.f / Ls : 0.f;
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  T* orow = reinterpret_cast<T*>(p.out) + int64_t(b) * p.out_sb + int64_t(h) * p.out_sn + lane * kDPL;
#pragma unroll
  for (int e = 0; e < kDPL; e += 2) {
    const uint32_t w = pack2(acc[e] * inv, acc[e + 1] * inv, BF16);
    *reinterpret_cast<uint32_t*>(orow + e) = w;
  }
  if (lane == 0 && p.lse != nullptr)
    p.lse[int64_t(b) * p.lse_sb + int64_t(h) * p.lse_sn] = has ? M + __logf(Ls) : INFINITY;
}

template <int D, bool BF16, int G>
static cudaError_t launch_decode_t(const DecodeParams& p, int part, cudaStream_t s) {
  using C = DecodeCfg<D, G>;
  if (part == 0) {
    if (p.n_cta == 0) return cudaSuccess;
    auto k = decode_kernel<D, BF16, G>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    k<<<p.n_cta, C::kThreads, C::kSmem, s>>>(p);
    return cudaGetLastError();
  }
  const int warps = p.batch * p.num_heads;
  if (warps > 0) decode_combine_kernel<D, BF16, G><<<(warps + 3) / 4, 128, 0, s>>>(p);
  return cudaGetLastError();
}

// part 0: the split-KV kernel; part 1: the combine kernel.
cudaError_t launch_decode(const DecodeParams& p, int head_dim, bool bf16, int part, cudaStream_t s) {
#define FIA_DEC_G(DD, BB)                                         \
  switch (p.heads_per_unit) {                                     \
    case 1: return launch_decode_t<DD, BB, 1>(p, part, s);        \
    case 2: return launch_decode_t<DD, BB, 2>(p, part, s);        \
    case 4: return launch_decode_t<DD, BB, 4>(p, part, s);        \
    case 8: return launch_decode_t<DD, BB, 8>(p, part, s);        \
    default: return cudaErrorInvalidValue;                        \
  }
  if (head_dim == 128) {
    if (bf16) { FIA_DEC_G(128, true) } else { FIA_DEC_G(128, false) }
  } else if (head_dim == 64) {
    if (bf16) { FIA_DEC_G(64, true) } else { FIA_DEC_G(64, false) }
  }
#undef FIA_DEC_G
  return cudaErrorInvalidValue;
}

}  // namespace fia
