// Single-CTA checks of the tcgen05 building blocks the attention kernels use,
// each against a plain CPU matrix product of the same bf16 inputs:
//   test 0: D[128x128] = A[128x64] . B[128x64]^T, both K-major from TMA tiles
//           (the Q K^T shape of the prefill kernel, 128-byte swizzle)
//   test 1: D[128x128] = P[128x128] . V[128x128], P K-major in shared memory,
//           V row-major = an MN-major B operand (the P V shape)
//   test 2: as test 1 with P read from tensor memory (written by tcgen05.st)
// Built by the test with nvcc into a small shared library; every wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <vector>

#include "../../attention_fia_prefill_gb300/csrc/ptx.cuh"

using namespace fia;

struct Maps {
  CUtensorMap a, b;
};

__global__ void __launch_bounds__(128, 1) selftest_kernel(const __grid_constant__ Maps m, int test,
                                                          const __nv_bfloat16* p_global, float* out,
                                                          unsigned long long* status) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = align_smem_1024(raw);
  uint8_t* sa = smem;            // A: up to 2 boxes of 16 KB
  uint8_t* sb = smem + 32768;    // B: up to 2 boxes
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 65536);
  uint32_t* holder = reinterpret_cast<uint32_t*>(bars + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 5);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(holder, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;
  const int na = test == 0 ? 1 : 2;   // A boxes (64 columns each)
  const int nb = test == 0 ? 1 : 2;   // B boxes
  if (threadIdx.x == 0) {
    const bool load_a = test != 2;
    mbar_arrive_expect_tx(&bars[0], (load_a ? na : 0) * 16384 + nb * 16384);
    if (load_a)
      for (int c = 0; c < na; ++c) tma_load_2d(sa + c * 16384, &m.a, &bars[0], c * 64, 0);
    for (int c = 0; c < nb; ++c) tma_load_2d(sb + c * 16384, &m.b, &bars[0], c * 64, 0);
  }
  if (test == 2) {
    // thread r writes row r of P into TMEM columns [128, 192) as packed pairs
    const int r = threadIdx.x;
    uint32_t u[32];
    for (int half = 0; half < 2; ++half) {
      for (int e = 0; e < 32; ++e) {
        const float lo = __bfloat162float(p_global[r * 128 + half * 64 + 2 * e]);
        const float hi = __bfloat162float(p_global[r * 128 + half * 64 + 2 * e + 1]);
        u[e] = pack2(lo, hi, true);
      }
      tmem_st32(tmem + (uint32_t(32 * warp) << 16) + 128 + half * 32, u);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    tc_fence_after();
    bool ok = mbar_wait(&bars[0], 0, abort_flag, DevStatus{status, 1, kWaitLimitNs});
    if (ok) {
      tc_fence_after();
      const uint32_t a0 = smem_u32(sa), b0 = smem_u32(sb);
      if (test == 0) {
        const uint32_t idesc = idesc_f16(128, 128, 1, 0, 0);
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem, smem_desc_sw128(a0 + kk * 32, 16, 1024), smem_desc_sw128(b0 + kk * 32, 16, 1024), idesc,
                 kk > 0);
      } else {
        const uint32_t idesc = idesc_f16(128, 128, 1, 0, 1);
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bdesc = smem_desc_sw128(b0 + kk * 2048, 16384, 1024);
          if (test == 1)
            mma_ss(tmem, smem_desc_sw128(a0 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024), bdesc, idesc, kk > 0);
          else
            mma_ts(tmem, tmem + 128 + kk * 8, bdesc, idesc, kk > 0);
        }
      }
      mma_commit(&bars[1]);
      mbar_wait(&bars[1], 0, abort_flag, DevStatus{status, 1, kWaitLimitNs});
    }
  }
  __syncthreads();
  tc_fence_after();
  if (*abort_flag == 0) {
    for (int c = 0; c < 4; ++c) {
      uint32_t u[32];
      tmem_ld32(tmem + (uint32_t(32 * warp) << 16) + c * 32, u);
      tmem_wait_ld(u);
      const int r = 32 * warp + lane;
      for (int e = 0; e < 32; ++e) out[r * 128 + c * 32 + e] = __uint_as_float(u[e]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static int encode(EncodeFn fn, CUtensorMap* m, void* p, int cols, int rows) {
  cuuint64_t gd[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  cuuint64_t gs[1] = {cuuint64_t(cols) * 2};
  cuuint32_t box[2] = {64, 128}, es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, p, gd, gs, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

static float bf(uint16_t h) {
  uint32_t u = uint32_t(h) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

// Returns the max abs error of the test (negative on a setup failure), -1e9 on timeout.
extern "C" double fia_selftest_run(int test) {
  void* fnp = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fnp, 12000, cudaEnableDefault, &q) != cudaSuccess)
    return -1;
  EncodeFn fn = reinterpret_cast<EncodeFn>(fnp);
  const int K_a = test == 0 ? 64 : 128;   // A: 128 rows x K_a;  B: 128 rows x K_a (test 0) or V 128 x 128
  std::vector<uint16_t> ha(128 * K_a), hb(128 * 128);
  uint32_t s = 12345u;
  auto rnd = [&]() {
    s = s * 1664525u + 1013904223u;
    const float f = (float(s >> 8) / float(1 << 24)) * 2.f - 1.f;   // [-1, 1)
    uint32_t u;
    memcpy(&u, &f, 4);
    return uint16_t(u >> 16);
  };
  for (auto& x : ha) x = rnd();
  for (auto& x : hb) x = rnd();
  const int b_cols = test == 0 ? 64 : 128;
  void *da, *db, *dout, *dstatus;
  cudaMalloc(&da, ha.size() * 2);
  cudaMalloc(&db, 128 * b_cols * 2);
  cudaMalloc(&dout, 128 * 128 * 4);
  cudaMalloc(&dstatus, 8);
  cudaMemcpy(da, ha.data(), ha.size() * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(db, hb.data(), 128 * b_cols * 2, cudaMemcpyHostToDevice);
  cudaMemset(dout, 0, 128 * 128 * 4);
  cudaMemset(dstatus, 0, 8);
  Maps m;
  if (encode(fn, &m.a, da, K_a, 128) != CUDA_SUCCESS || encode(fn, &m.b, db, b_cols, 128) != CUDA_SUCCESS) return -2;
  const int smem = 65536 + 1024 + 1024;
  cudaFuncSetAttribute(selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  selftest_kernel<<<1, 128, smem>>>(m, test, static_cast<const __nv_bfloat16*>(da), static_cast<float*>(dout),
                                    static_cast<unsigned long long*>(dstatus));
  if (cudaDeviceSynchronize() != cudaSuccess) return -3;
  std::vector<float> out(128 * 128);
  unsigned long long st = 0;
  cudaMemcpy(out.data(), dout, out.size() * 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(&st, dstatus, 8, cudaMemcpyDeviceToHost);
  cudaFree(da); cudaFree(db); cudaFree(dout); cudaFree(dstatus);
  if (st != 0) return -1e9;
  double maxerr = 0;
  for (int i = 0; i < 128; ++i)
    for (int j = 0; j < 128; ++j) {
      double ref = 0;
      if (test == 0) {
        for (int k = 0; k < 64; ++k) ref += double(bf(ha[i * 64 + k])) * double(bf(hb[j * 64 + k]));
      } else {
        for (int k = 0; k < 128; ++k) ref += double(bf(ha[i * 128 + k])) * double(bf(hb[k * 128 + j]));
      }
      maxerr = fmax(maxerr, fabs(ref - double(out[i * 128 + j])));
    }
  return maxerr;
}
