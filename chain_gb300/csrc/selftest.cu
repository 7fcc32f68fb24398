// selftest.cu -- diagnostics of the building blocks every kernel uses:
//  * a single-CTA TMA + tcgen05.mma product checking the shared-memory
//    descriptors (K-major A, K-major or MN-major B) and the tensor-memory
//    load layout;
//  * a bounded wait on a barrier that never completes, checking that the
//    failure path records a timeout and returns instead of hanging.
#include "internal.h"

namespace chain {
namespace {

enum : int { SITE_SELFTEST_WAIT = 0x901, SITE_SELFTEST_UMMA = 0x902 };

__global__ void wait_selftest_kernel(WaitCfg wc) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nobody arrives: the wait must expire and record SITE_SELFTEST_WAIT.
    mbar_wait(&bar, 0, wc, &abort_flag, SITE_SELFTEST_WAIT);
  }
  __syncthreads();
}

// D[128][N] = A[128][K] * op(B); A via map {K, 128}, B via map {K, N}
// (K-major) or {N, K} (MN-major); boxes of 64 elements x rows.
template <int N>
__global__ void __launch_bounds__(128, 1)
    umma_selftest_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB, float *D, int K, int b_mn,
                         const __nv_bfloat16 *A_gmem, int a_tmem, WaitCfg wc) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t a_bytes = 128 * K * 2, b_bytes = N * K * 2;
  uint8_t *sA = smem;
  uint8_t *sB = smem + a_bytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sB + b_bytes);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 3);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  if (a_tmem) {
    // Row r of A (thread r) goes to lane r, columns 256 + k/2 (bf16 pairs,
    // element 2c in the low half of column c).
    const __nv_bfloat16 *arow = A_gmem + (size_t)threadIdx.x * K;
    for (int c0 = 0; c0 < K / 2; c0 += 32) {
      uint32_t r[32];
      for (int k = 0; k < 32; ++k) {
        const uint16_t lo = reinterpret_cast<const uint16_t *>(arow)[2 * (c0 + k)];
        const uint16_t hi = reinterpret_cast<const uint16_t *>(arow)[2 * (c0 + k) + 1];
        r[k] = (uint32_t)lo | ((uint32_t)hi << 16);
      }
      tmem_st32(tmem + lane_off + 256 + c0, r);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  bool ok = true;
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bars[0], a_bytes + b_bytes);
    for (int c = 0; c < K / 64; ++c) tma_load_2d(sA + c * 128 * 128, &tmA, &bars[0], c * 64, 0);
    (void)A_gmem;
    if (!b_mn) {
      for (int c = 0; c < K / 64; ++c) tma_load_2d(sB + c * N * 128, &tmB, &bars[0], c * 64, 0);
    } else {
      for (int c = 0; c < N / 64; ++c) tma_load_2d(sB + c * K * 128, &tmB, &bars[0], c * 64, 0);
    }
    ok = mbar_wait(&bars[0], 0, wc, abort_flag, SITE_SELFTEST_UMMA);
    if (ok) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(128, N, 0, b_mn);
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
      for (int kk = 0; kk < K / 16; ++kk) {
        const uint64_t ad = sdesc_sw128(a0 + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024);
        const uint64_t bd =
            b_mn ? sdesc_sw128(b0 + kk * 2048, K * 128, 1024)
                 : sdesc_sw128(b0 + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024);
        if (a_tmem)
          umma_f16_ts(tmem, tmem + 256 + kk * 8, bd, idesc, kk > 0 ? 1u : 0u);
        else
          umma_f16_ss(tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
      }
    }
    umma_commit(&bars[1]);
  }
  __syncwarp();
  ok = mbar_wait(&bars[1], 0, wc, abort_flag, SITE_SELFTEST_UMMA) && !*abort_flag;
  tc_fence_after();
  const int row = threadIdx.x;
  for (int c = 0; c < N / 32; ++c) {
    uint32_t r[32];
    tmem_ld32(tmem + lane_off + c * 32, r);
    tmem_wait_ld();
    if (ok)
      for (int k = 0; k < 32; ++k) D[row * N + c * 32 + k] = __uint_as_float(r[k]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  (void)lane;
}

}  // namespace

cudaError_t launch_wait_selftest(const WaitCfg &wc, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(wc);
  return cudaGetLastError();
}

cudaError_t launch_umma_selftest(const void *A, const void *B, float *D, int N, int K,
                                 int flags, const WaitCfg &wc, cudaStream_t st) {
  const int b_mn_major = flags & 1, a_tmem = (flags >> 1) & 1;
  if ((N != 64 && N != 128) || K <= 0 || K % 64 != 0 || K > 256) return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  const uint64_t da[2] = {(uint64_t)K, 128};
  const uint64_t sa[1] = {(uint64_t)K * 2};
  const uint32_t boxa[2] = {64, 128};
  cudaError_t e = make_tmap(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, da, sa, boxa);
  if (e != cudaSuccess) return e;
  if (!b_mn_major) {
    const uint64_t db[2] = {(uint64_t)K, (uint64_t)N};
    const uint64_t sb[1] = {(uint64_t)K * 2};
    const uint32_t boxb[2] = {64, (uint32_t)N};
    e = make_tmap(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, db, sb, boxb);
  } else {
    const uint64_t db[2] = {(uint64_t)N, (uint64_t)K};
    const uint64_t sb[1] = {(uint64_t)N * 2};
    const uint32_t boxb[2] = {64, (uint32_t)K};
    e = make_tmap(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, db, sb, boxb);
  }
  if (e != cudaSuccess) return e;
  const size_t smem = 1024 + (size_t)128 * K * 2 + (size_t)N * K * 2 + 64;
  if (N == 64) {
    cudaFuncSetAttribute(umma_selftest_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    umma_selftest_kernel<64><<<1, 128, smem, st>>>(
        ma, mb, D, K, b_mn_major, static_cast<const __nv_bfloat16 *>(A), a_tmem, wc);
  } else {
    cudaFuncSetAttribute(umma_selftest_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    umma_selftest_kernel<128><<<1, 128, smem, st>>>(
        ma, mb, D, K, b_mn_major, static_cast<const __nv_bfloat16 *>(A), a_tmem, wc);
  }
  return cudaGetLastError();
}

}  // namespace chain
