// mlp_bwd.cu -- backward of the MLP instance of O = f(A B) C ("Memory-
// efficient tensor parallelism", FITEE 10.1631/FITEE.2400602, abstract), with
// the intermediate recomputed rather than kept from the forward ("AutoSP",
// section 2.B).  O = f(X W1) W2, f = GeLU (tanh form) or identity:
//   T = X W1,  H = f(T),  dH = dO W2^T,  dT = dH * f'(T)
//   dW2 = H^T dO,   dX = dT W1^T,   dW1 = X^T dT.
//
// Two kernels:
//   mlp_bwd_act_kernel  one CTA per (128 rows, 256 hidden columns): T and dH
//                       on the tensor cores (fp32 in tensor memory), then H
//                       and dT as bf16 into the caller's workspace [M][N] x 2;
//   gemm_kernel         the three products above as one launch of 128 x 256
//                       output tiles, each operand K- or MN-major as stored.
#include "internal.h"

namespace chain {
namespace {

constexpr int BM = 128;
constexpr int KT = 64;  // K-tile of every product
constexpr int NTHREADS = 192;

enum : int {
  SITE_MB_PROD = 0x401,
  SITE_MB_MMA = 0x402,
  SITE_MB_EPI = 0x403,
  SITE_MB_DRAIN = 0x404,
  SITE_GM_PROD = 0x411,
  SITE_GM_MMA = 0x412,
  SITE_GM_EPI = 0x413
};

__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, const WaitCfg &wc) {
  volatile int never = 0;
  mbar_wait(bar, parity, wc, &never, SITE_MB_DRAIN);
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                     ~static_cast<uintptr_t>(1023));
}

// GeLU, tanh form (Hendrycks & Gimpel), and its derivative:
//   g(t)  = 0.5 t (1 + tanh u),  u = k (t + 0.044715 t^3),  k = sqrt(2/pi)
//   g'(t) = 0.5 (1 + tanh u) + 0.5 t (1 - tanh^2 u) k (1 + 3*0.044715 t^2)
// with tanh u = 1 - 2 / (1 + e^{2u}) evaluated through ex2.
__device__ __forceinline__ void gelu_tanh_and_grad(float t, float &g, float &dg) {
  const float k = 0.7978845608028654f;
  const float t2 = t * t;
  const float u = k * fmaf(0.044715f * t, t2, t);
  const float e = ex2(fminf(u * 2.8853900817779268f, 64.0f));  // e^{2u}, capped
  const float th = 1.0f - __fdividef(2.0f, 1.0f + e);
  g = 0.5f * t * (1.0f + th);
  dg = fmaf(0.5f * t * (1.0f - th * th), k * fmaf(0.134145f, t2, 1.0f), 0.5f * (1.0f + th));
}

// ------------------------------------------------------------ H and dT
constexpr int HN = 256;  // hidden columns per CTA of the activation kernel

struct ActLayout {
  static constexpr int NSTAGE = 4;
  static constexpr uint32_t STAGE = 16384 + HN * KT * 2;  // A tile 16 KB, B tile 32 KB
  static constexpr uint32_t OFF_BAR = NSTAGE * STAGE;
  static constexpr uint32_t NBAR = 2 * NSTAGE + 2;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t ALLOC = OFF_MISC + 16 + 1024;
};

struct ActParams {
  int M, K, N, P, gelu;
  __nv_bfloat16 *H, *dT;  // [M][N] each
  WaitCfg wc;
};

// Stage sequence: K/64 tiles of (X rows, W1 columns) for T, then P/64 tiles
// of (dO rows, W2 rows) for dH.
__global__ void __launch_bounds__(NTHREADS, 1)
    mlp_bwd_act_kernel(const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmW1,
                       const __grid_constant__ CUtensorMap tmdO,
                       const __grid_constant__ CUtensorMap tmW2, const ActParams p) {
  using L = ActLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
  uint64_t *full = bars;                // [NSTAGE]
  uint64_t *empty = bars + L::NSTAGE;   // [NSTAGE]
  uint64_t *acc_full = bars + 2 * L::NSTAGE;
  uint64_t *mma_drain = acc_full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = p.N / HN;
  const int rb = blockIdx.x / nb, hb = blockIdx.x % nb;
  const int nk = p.K / KT, np = p.P / KT, nst = nk + np;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 2 * HN);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW1);
    tma_prefetch_desc(&tmdO);
    tma_prefetch_desc(&tmW2);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // T [0,HN), dH [HN,2HN)

  if (warp == 4) {
    // -------------------------------------------------------- producer
    if (lane == 0) {
      int issued = 0;
      for (int st = 0; st < nst; ++st) {
        const int s = st % L::NSTAGE;
        if (st >= L::NSTAGE &&
            !mbar_wait(&empty[s], ((st / L::NSTAGE) - 1) & 1, p.wc, abort_flag, SITE_MB_PROD))
          break;
        uint8_t *dst = smem + s * L::STAGE;
        mbar_arrive_expect_tx(&full[s], L::STAGE);
        if (st < nk) {  // X [rows][k tile] (K-major), W1 [k tile][hidden cols] (MN-major)
          tma_load_2d(dst, &tmX, &full[s], st * KT, rb * BM);
#pragma unroll
          for (int i = 0; i < HN / 64; ++i)
            tma_load_2d(dst + 16384 + i * 8192, &tmW1, &full[s], hb * HN + i * 64, st * KT);
        } else {        // dO [rows][p tile] (K-major), W2 [hidden rows][p tile] (K-major)
          const int pt = st - nk;
          tma_load_2d(dst, &tmdO, &full[s], pt * KT, rb * BM);
#pragma unroll
          for (int i = 0; i < HN / 128; ++i)
            tma_load_2d(dst + 16384 + i * 16384, &tmW2, &full[s], pt * KT, hb * HN + i * 128);
        }
        issued = st + 1;
      }
      if (*abort_flag) {
        for (int j = (issued > L::NSTAGE ? issued - L::NSTAGE : 0); j < issued; ++j)
          drain_wait(&full[j % L::NSTAGE], (j / L::NSTAGE) & 1, p.wc);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------ MMA issuer
    // The whole warp runs the loop; one elected lane issues each group and
    // its commits.
    {
      const uint32_t id_t = idesc_bf16_f32(BM, HN, 0, 1);   // T: W1 MN-major
      const uint32_t id_h = idesc_bf16_f32(BM, HN, 0, 0);   // dH: W2 rows K-major
      bool ok = true;
      for (int st = 0; st < nst; ++st) {
        const int s = st % L::NSTAGE;
        if (!mbar_wait_warp(&full[s], (st / L::NSTAGE) & 1, p.wc, abort_flag, SITE_MB_MMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = smem_u32(smem + s * L::STAGE);
        const SDesc a = sdesc_make(base, 16, 1024);
        const bool is_t = st < nk;
        const SDesc b = is_t ? sdesc_make(base + 16384, 8192, 1024) : sdesc_make(base + 16384, 16, 1024);
        const int first = is_t ? 0 : nk;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < KT / 16; ++kk)
            umma_f16_ss(tmem + (is_t ? 0 : HN), sdesc_at(a, kk * 32),
                        sdesc_at(b, is_t ? kk * 2048 : kk * 32), is_t ? id_t : id_h,
                        (st > first || kk > 0) ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        __syncwarp();
      }
      if (elect_one()) {
        if (ok) umma_commit(acc_full);
        umma_commit(mma_drain);
      }
      __syncwarp();
      if (lane == 0) drain_wait(mma_drain, 0, p.wc);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------- epilogue
    // thread r owns row rb*128 + r (tensor-memory lane r)
    const int row = threadIdx.x;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    if (mbar_wait(acc_full, 0, p.wc, abort_flag, SITE_MB_EPI)) {
      tc_fence_after();
      const int64_t off = (int64_t)(rb * BM + row) * p.N + hb * HN;
      uint4 *hrow = reinterpret_cast<uint4 *>(p.H + off);
      uint4 *drow = reinterpret_cast<uint4 *>(p.dT + off);
#pragma unroll 1
      for (int q = 0; q < HN / 32; ++q) {
        uint32_t t[32], dh[32];
        tmem_ld32(tmem + lane_off + q * 32, t);
        tmem_ld32(tmem + lane_off + HN + q * 32, dh);
        tmem_wait_ld();
        uint32_t hp[16], dp[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          float g0 = __uint_as_float(t[2 * k]), g1 = __uint_as_float(t[2 * k + 1]);
          float d0 = 1.0f, d1 = 1.0f;
          if (p.gelu) {
            gelu_tanh_and_grad(__uint_as_float(t[2 * k]), g0, d0);
            gelu_tanh_and_grad(__uint_as_float(t[2 * k + 1]), g1, d1);
          }
          hp[k] = pack_bf16(g0, g1);
          dp[k] = pack_bf16(__uint_as_float(dh[2 * k]) * d0, __uint_as_float(dh[2 * k + 1]) * d1);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          hrow[q * 4 + k] = make_uint4(hp[4 * k], hp[4 * k + 1], hp[4 * k + 2], hp[4 * k + 3]);
          drow[q * 4 + k] = make_uint4(dp[4 * k], dp[4 * k + 1], dp[4 * k + 2], dp[4 * k + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * HN);
  }
}

// ------------------------------------------------------ generic product
// C [Mc][Nc] (bf16, row stride ldc) = A [Mc][Kc] B [Kc][Nc], fp32 accumulate.
// A is K-major (stored [Mc][Kc]) or MN-major (stored [Kc][Mc]); B is K-major
// (stored [Nc][Kc]) or MN-major (stored [Kc][Nc]).  128 x 256 output tiles.
constexpr int GM = 128, GN = 256, GJOBS = 3;

struct GemmLayout {
  static constexpr int NSTAGE = 4;
  static constexpr uint32_t A_BYTES = GM * KT * 2;  // 16 KB
  static constexpr uint32_t B_BYTES = GN * KT * 2;  // 32 KB
  static constexpr uint32_t STAGE = A_BYTES + B_BYTES;
  static constexpr uint32_t OFF_BAR = NSTAGE * STAGE;
  static constexpr uint32_t NBAR = 2 * NSTAGE + 2;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t ALLOC = OFF_MISC + 16 + 1024;
};

struct GemmJobs {
  CUtensorMap a[GJOBS], b[GJOBS];
  __nv_bfloat16 *c[GJOBS];
  int64_t ldc[GJOBS];
  int tiles_n[GJOBS], ktiles[GJOBS], a_mn[GJOBS], b_mn[GJOBS];
  int tile_begin[GJOBS + 1];
  int njobs;
  WaitCfg wc;
};

__global__ void __launch_bounds__(NTHREADS, 1) gemm_kernel(const __grid_constant__ GemmJobs J) {
  using L = GemmLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
  uint64_t *full = bars;
  uint64_t *empty = bars + L::NSTAGE;
  uint64_t *acc_full = bars + 2 * L::NSTAGE;
  uint64_t *mma_drain = acc_full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int j = 0;
  while (j + 1 < J.njobs && (int)blockIdx.x >= J.tile_begin[j + 1]) ++j;
  const int tile = (int)blockIdx.x - J.tile_begin[j];
  const int tm = tile / J.tiles_n[j], tn = tile % J.tiles_n[j];
  const int nkt = J.ktiles[j];
  const bool a_mn = J.a_mn[j] != 0, b_mn = J.b_mn[j] != 0;
  const CUtensorMap *ma = &J.a[j], *mb = &J.b[j];

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(ma);
    tma_prefetch_desc(mb);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // -------------------------------------------------------- producer
    if (lane == 0) {
      int issued = 0;
      for (int kt = 0; kt < nkt; ++kt) {
        const int s = kt % L::NSTAGE;
        if (kt >= L::NSTAGE &&
            !mbar_wait(&empty[s], ((kt / L::NSTAGE) - 1) & 1, J.wc, abort_flag, SITE_GM_PROD))
          break;
        uint8_t *da = smem + s * L::STAGE, *db = da + L::A_BYTES;
        mbar_arrive_expect_tx(&full[s], L::STAGE);
        if (a_mn) {  // stored [K][M]: two 64-column boxes of 64 rows
          tma_load_2d(da, ma, &full[s], tm * GM, kt * KT);
          tma_load_2d(da + 8192, ma, &full[s], tm * GM + 64, kt * KT);
        } else {     // stored [M][K]: one box of 128 rows
          tma_load_2d(da, ma, &full[s], kt * KT, tm * GM);
        }
        if (b_mn) {  // stored [K][N]: four 64-column boxes of 64 rows
#pragma unroll
          for (int q = 0; q < 4; ++q) tma_load_2d(db + q * 8192, mb, &full[s], tn * GN + 64 * q, kt * KT);
        } else {     // stored [N][K]: one box of 256 rows
          tma_load_2d(db, mb, &full[s], kt * KT, tn * GN);
        }
        issued = kt + 1;
      }
      if (*abort_flag) {
        for (int q = (issued > L::NSTAGE ? issued - L::NSTAGE : 0); q < issued; ++q)
          drain_wait(&full[q % L::NSTAGE], (q / L::NSTAGE) & 1, J.wc);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------ MMA issuer
    {
      const uint32_t id = idesc_bf16_f32(GM, GN, a_mn ? 1 : 0, b_mn ? 1 : 0);
      const uint32_t a_step = a_mn ? 2048u : 32u, b_step = b_mn ? 2048u : 32u;
      bool ok = true;
      for (int kt = 0; kt < nkt; ++kt) {
        const int s = kt % L::NSTAGE;
        if (!mbar_wait_warp(&full[s], (kt / L::NSTAGE) & 1, J.wc, abort_flag, SITE_GM_MMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = smem_u32(smem + s * L::STAGE);
        const SDesc a = sdesc_make(base, a_mn ? 8192u : 16u, 1024);
        const SDesc b = sdesc_make(base + L::A_BYTES, b_mn ? 8192u : 16u, 1024);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < KT / 16; ++kk)
            umma_f16_ss(tmem, sdesc_at(a, kk * a_step), sdesc_at(b, kk * b_step), id,
                        (kt > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        __syncwarp();
      }
      if (elect_one()) {
        if (ok) umma_commit(acc_full);
        umma_commit(mma_drain);
      }
      __syncwarp();
      if (lane == 0) drain_wait(mma_drain, 0, J.wc);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------- epilogue
    const int row = threadIdx.x;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    if (mbar_wait(acc_full, 0, J.wc, abort_flag, SITE_GM_EPI)) {
      tc_fence_after();
      uint4 *crow = reinterpret_cast<uint4 *>(J.c[j] + (int64_t)(tm * GM + row) * J.ldc[j] + tn * GN);
#pragma unroll 1
      for (int q = 0; q < GN / 32; ++q) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + q * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          crow[q * 4 + k] = make_uint4(
              pack_bf16(__uint_as_float(r[8 * k + 0]), __uint_as_float(r[8 * k + 1])),
              pack_bf16(__uint_as_float(r[8 * k + 2]), __uint_as_float(r[8 * k + 3])),
              pack_bf16(__uint_as_float(r[8 * k + 4]), __uint_as_float(r[8 * k + 5])),
              pack_bf16(__uint_as_float(r[8 * k + 6]), __uint_as_float(r[8 * k + 7])));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// A row-major bf16 matrix [rows][cols] as a 2-D tensor map with the given box.
cudaError_t map2d(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, uint32_t box_cols,
                  uint32_t box_rows) {
  const uint64_t d[2] = {(uint64_t)cols, (uint64_t)rows};
  const uint64_t s[1] = {(uint64_t)cols * 2};
  const uint32_t box[2] = {box_cols, box_rows};
  return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, d, s, box);
}

// One product of the batch: C [Mc][Nc] = A B with A stored [Mc][Kc]
// (a_mn = 0) or [Kc][Mc] (a_mn = 1), B stored [Nc][Kc] (b_mn = 0) or
// [Kc][Nc] (b_mn = 1).
cudaError_t add_job(GemmJobs &J, int &tiles, const void *A, int a_mn, const void *B, int b_mn,
                    void *C, int64_t Mc, int64_t Nc, int64_t Kc) {
  const int q = J.njobs;
  cudaError_t e;
  if ((e = a_mn ? map2d(&J.a[q], A, Kc, Mc, 64, 64) : map2d(&J.a[q], A, Mc, Kc, 64, 128))) return e;
  if ((e = b_mn ? map2d(&J.b[q], B, Kc, Nc, 64, 64) : map2d(&J.b[q], B, Nc, Kc, 64, 256))) return e;
  J.c[q] = static_cast<__nv_bfloat16 *>(C);
  J.ldc[q] = Nc;
  J.tiles_n[q] = (int)(Nc / GN);
  J.ktiles[q] = (int)(Kc / KT);
  J.a_mn[q] = a_mn;
  J.b_mn[q] = b_mn;
  J.tile_begin[q] = tiles;
  tiles += (int)((Mc / GM) * (Nc / GN));
  J.tile_begin[q + 1] = tiles;
  J.njobs = q + 1;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_mlp_bwd(const MlpBwdArgs &a, const WaitCfg &wc, cudaStream_t st) {
  // shapes: 128-row blocks of X, 128-wide hidden chunks, 256-wide output
  // tiles of every product, 64-deep K tiles
  if (a.M % 128 || a.K % 256 || a.N % 256 || a.P % 256) return cudaErrorNotSupported;
  cudaError_t e;
  __nv_bfloat16 *H = static_cast<__nv_bfloat16 *>(a.workspace);
  __nv_bfloat16 *dT = H + (int64_t)a.M * a.N;
  {
    CUtensorMap mx, mw1, mdo, mw2;
    if ((e = map2d(&mx, a.X, a.M, a.K, 64, 128))) return e;
    if ((e = map2d(&mw1, a.W1, a.K, a.N, 64, 64))) return e;
    if ((e = map2d(&mdo, a.dO, a.M, a.P, 64, 128))) return e;
    if ((e = map2d(&mw2, a.W2, a.N, a.P, 64, 128))) return e;
    ActParams p;
    p.M = a.M; p.K = a.K; p.N = a.N; p.P = a.P; p.gelu = a.gelu;
    p.H = H; p.dT = dT; p.wc = wc;
    if ((e = cudaFuncSetAttribute(mlp_bwd_act_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  ActLayout::ALLOC)))
      return e;
    const unsigned grid = (unsigned)((a.M / BM) * (a.N / HN));
    timing_mark(st, 0);
    mlp_bwd_act_kernel<<<grid, NTHREADS, ActLayout::ALLOC, st>>>(mx, mw1, mdo, mw2, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  GemmJobs J;
  J.njobs = 0;
  J.wc = wc;
  int tiles = 0;
  // dW2 [N][P] = H^T dO: A = H^T, stored H [M][N] = [K][Mc]; B = dO [M][P] = [K][Nc]
  if ((e = add_job(J, tiles, H, 1, a.dO, 1, a.dW2, a.N, a.P, a.M))) return e;
  // dX [M][K] = dT W1^T: A = dT [M][N] = [Mc][K]; B = W1^T, stored W1 [K][N] = [Nc][K]
  if ((e = add_job(J, tiles, dT, 0, a.W1, 0, a.dX, a.M, a.K, a.N))) return e;
  // dW1 [K][N] = X^T dT: A = X^T, stored X [M][K] = [K][Mc]; B = dT [M][N] = [K][Nc]
  if ((e = add_job(J, tiles, a.X, 1, dT, 1, a.dW1, a.K, a.N, a.M))) return e;
  if ((e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                GemmLayout::ALLOC)))
    return e;
  timing_mark(st, 1);
  gemm_kernel<<<(unsigned)tiles, NTHREADS, GemmLayout::ALLOC, st>>>(J);
  timing_mark(st, 2);
  return cudaGetLastError();
}

}  // namespace chain
