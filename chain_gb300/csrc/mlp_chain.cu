// mlp_chain.cu -- the MLP instance of the unit O = f(A B) C ("Memory-
// efficient tensor parallelism", FITEE 10.1631/FITEE.2400602, abstract):
//   O = f(X W1) W2,  f = GeLU (tanh form) or identity,
// X [M][K], W1 [K][N], W2 [N][P] bf16 row-major, O [M][P] bf16.  The
// [M][N] intermediate is produced 128 columns at a time in tensor memory,
// passed through f in registers and consumed from shared memory by the
// second product; it is never written to global memory (the activation
// the AutoSP write-up, section 2.B, recomputes instead of storing).
//
// One CTA per (128-row block of X, 256-column block of O).  For each
// 128-wide hidden chunk c:
//   GEMM1  T_c = X_blk W1[:, c]           (tcgen05, fp32 in tensor memory)
//   f      H_c = f(T_c) in fp32 registers, split into H_hi = bf16(H_c) and
//          H_lo = bf16(H_c - H_hi), written to 128-byte-swizzled smem
//   GEMM2  O_blk += H_hi W2[c, blk] + H_lo W2[c, blk]
// The split keeps the intermediate's rounding at ~2^-16 relative, so the
// only bf16 rounding left is the output's.  GEMM1 of chunk c+1 runs while
// the epilogue warps process chunk c.
//
// Roles (192 threads): warps 0-3 epilogue (thread t owns row t), warp 4
// TMA producer (one 32 KB stage ring carrying X/W1 K-tiles and W2 tiles in
// consumption order), warp 5 MMA issuer.  Tensor memory: T buffers at
// columns [0,128) and [128,256), O accumulator [256,512).
#include "internal.h"

namespace chain {
namespace {

constexpr int BM = 128;      // rows per CTA
constexpr int BP = 256;      // output columns per CTA
constexpr int HC = 128;      // hidden chunk
constexpr int KT = 64;       // K-tile of GEMM1 and of GEMM2 (hidden rows)
constexpr int NSTAGE = 4;
constexpr uint32_t STAGE_BYTES = 32768;
constexpr int NTHREADS = 192;

struct MlpLayout {
  static constexpr uint32_t OFF_RING = 0;
  static constexpr uint32_t OFF_HHI = OFF_RING + NSTAGE * STAGE_BYTES;
  static constexpr uint32_t OFF_HLO = OFF_HHI + BM * HC * 2;
  static constexpr uint32_t OFF_BAR = OFF_HLO + BM * HC * 2;
  static constexpr uint32_t NBAR = 2 * NSTAGE + 2 + 2 + 1 + 1 + 1 + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  static constexpr uint32_t ALLOC = BYTES + 1024;
};

struct MlpParams {
  int M, K, N, P, gelu;
  __nv_bfloat16 *O;
  WaitCfg wc;
};

enum : int {
  SITE_MLP_PROD = 0x301,
  SITE_MLP_MMA = 0x302,
  SITE_MLP_EPI = 0x303,
  SITE_MLP_DRAIN = 0x304
};

__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, const WaitCfg &wc) {
  volatile int never = 0;
  mbar_wait(bar, parity, wc, &never, SITE_MLP_DRAIN);
}

// GeLU, tanh form (Hendrycks & Gimpel): 0.5 t (1 + tanh(sqrt(2/pi)(t + 0.044715 t^3))),
// with tanh(y) = 1 - 2 / (1 + e^{2y}) evaluated through ex2.
__device__ __forceinline__ float gelu_tanh(float t) {
  const float y = 0.7978845608028654f * fmaf(0.044715f * t, t * t, t);
  const float e = ex2(fminf(y * 2.8853900817779268f, 64.0f));  // e^{2y}, capped
  const float th = 1.0f - __fdividef(2.0f, 1.0f + e);
  return 0.5f * t * (1.0f + th);
}

__global__ void __launch_bounds__(NTHREADS, 1)
    mlp_chain_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmW1,
                     const __grid_constant__ CUtensorMap tmW2, const MlpParams p) {
  using L = MlpLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
  uint64_t *full = bars;                 // [NSTAGE]
  uint64_t *empty = bars + NSTAGE;       // [NSTAGE]
  uint64_t *t_full = bars + 2 * NSTAGE;  // [2]
  uint64_t *t_free = t_full + 2;         // [2]
  uint64_t *h_ready = t_free + 2;
  uint64_t *h_free = h_ready + 1;
  uint64_t *o_done = h_free + 1;
  uint64_t *mma_drain = o_done + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rb = blockIdx.x / (p.P / BP);
  const int pb = blockIdx.x % (p.P / BP);
  const int NC = p.N / HC;      // hidden chunks
  const int NKT = p.K / KT;     // GEMM1 K-tiles per chunk

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&t_full[b], 1);
      mbar_init(&t_free[b], 128);
    }
    mbar_init(h_ready, 128);
    mbar_init(h_free, 1);
    mbar_init(o_done, 1);
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW1);
    tma_prefetch_desc(&tmW2);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // -------------------------------------------------------- producer
    // Consumption order of the MMA warp: GEMM1(c) K-tiles, then the two
    // W2 tiles of chunk c-1.
    if (lane == 0) {
      int st = 0;
      bool ok = true;
      for (int c = 0; c <= NC && ok; ++c) {
        const int n_tiles = (c < NC ? NKT : 0) + (c >= 1 ? HC / KT : 0);
        for (int t = 0; t < n_tiles; ++t, ++st) {
          const int s = st % NSTAGE;
          if (st >= NSTAGE &&
              !mbar_wait(&empty[s], ((st / NSTAGE) - 1) & 1, p.wc, abort_flag, SITE_MLP_PROD)) {
            ok = false;
            break;
          }
          uint8_t *dst = smem + L::OFF_RING + s * STAGE_BYTES;
          mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
          if (c < NC && t < NKT) {
            // X [rows rb*128..][k t*64..] (16 KB) + W1 [k t*64..][n c*128..] (2 boxes)
            tma_load_2d(dst, &tmX, &full[s], t * KT, rb * BM);
            tma_load_2d(dst + 16384, &tmW1, &full[s], c * HC, t * KT);
            tma_load_2d(dst + 24576, &tmW1, &full[s], c * HC + 64, t * KT);
          } else {
            // W2 [hidden (c-1)*128 + h*64 ..][out pb*256 ..] as 4 boxes of 64 cols
            const int h = t - (c < NC ? NKT : 0);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              tma_load_2d(dst + q * 8192, &tmW2, &full[s], pb * BP + q * 64, (c - 1) * HC + h * KT);
          }
        }
      }
      if (*abort_flag) {
        for (int j = (st > NSTAGE ? st - NSTAGE : 0); j < st; ++j)
          drain_wait(&full[j % NSTAGE], (j / NSTAGE) & 1, p.wc);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------ MMA issuer
    // The whole warp runs the loop; one elected lane issues each group of
    // products together with its commits.
    {
      const uint32_t id1 = idesc_bf16_f32(BM, HC, 0, 1);  // T = X W1, W1 MN-major
      const uint32_t id2 = idesc_bf16_f32(BM, BP, 0, 1);  // O += H W2, W2 MN-major
      // ring stage s: X tile (K-major) at 0, W1 (MN-major) at 16 KB; W2 tiles
      // (MN-major) at 0.  Base descriptors built once per stage.
      const uint32_t ring = smem_u32(smem + L::OFF_RING);
      SDesc dX[NSTAGE], dW1[NSTAGE], dW2[NSTAGE];
#pragma unroll
      for (int q = 0; q < NSTAGE; ++q) {
        dX[q] = sdesc_make(ring + q * STAGE_BYTES, 16, 1024);
        dW1[q] = sdesc_make(ring + q * STAGE_BYTES + 16384, 8192, 1024);
        dW2[q] = sdesc_make(ring + q * STAGE_BYTES, 8192, 1024);
      }
      const SDesc dHhi = sdesc_make(smem_u32(smem + L::OFF_HHI), 16, 1024);
      const SDesc dHlo = sdesc_make(smem_u32(smem + L::OFF_HLO), 16, 1024);
      int st = 0;
      bool ok = true;
      for (int c = 0; c <= NC && ok; ++c) {
        if (c < NC) {
          const int b = c & 1;
          if (c >= 2 && !mbar_wait_warp(&t_free[b], ((c >> 1) - 1) & 1, p.wc, abort_flag, SITE_MLP_MMA)) {
            ok = false;
            break;
          }
          for (int t = 0; t < NKT; ++t, ++st) {
            const int s = st % NSTAGE;
            if (!mbar_wait_warp(&full[s], (st / NSTAGE) & 1, p.wc, abort_flag, SITE_MLP_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
            SDesc ax = dX[0], bw = dW1[0];
#pragma unroll
            for (int q = 1; q < NSTAGE; ++q)
              if (s == q) {
                ax = dX[q];
                bw = dW1[q];
              }
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < KT / 16; ++kk)
                umma_f16_ss(tmem + b * HC, sdesc_at(ax, kk * 32), sdesc_at(bw, kk * 2048), id1,
                            (t > 0 || kk > 0) ? 1u : 0u);
              umma_commit(&empty[s]);
            }
            __syncwarp();
          }
          if (!ok) break;
          if (elect_one()) umma_commit(&t_full[b]);
          __syncwarp();
        }
        if (c >= 1) {
          const int cp = c - 1;
          if (!mbar_wait_warp(h_ready, cp & 1, p.wc, abort_flag, SITE_MLP_MMA)) {
            ok = false;
            break;
          }
          for (int h = 0; h < HC / KT; ++h, ++st) {
            const int s = st % NSTAGE;
            if (!mbar_wait_warp(&full[s], (st / NSTAGE) & 1, p.wc, abort_flag, SITE_MLP_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
            SDesc bw = dW2[0];
#pragma unroll
            for (int q = 1; q < NSTAGE; ++q)
              if (s == q) bw = dW2[q];
            if (elect_one()) {
#pragma unroll
              for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int kk = 0; kk < KT / 16; ++kk)
                  umma_f16_ss(tmem + 256, sdesc_at(part ? dHlo : dHhi, h * (BM * 128) + kk * 32),
                              sdesc_at(bw, kk * 2048), id2,
                              (cp > 0 || h > 0 || part > 0 || kk > 0) ? 1u : 0u);
              umma_commit(&empty[s]);
            }
            __syncwarp();
          }
          if (!ok) break;
          if (elect_one()) umma_commit(h_free);
          __syncwarp();
        }
      }
      if (elect_one()) {
        if (ok) umma_commit(o_done);
        umma_commit(mma_drain);
      }
      __syncwarp();
      if (lane == 0) drain_wait(mma_drain, 0, p.wc);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------- epilogue
    const int row = threadIdx.x;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t sHhi = smem_u32(smem + L::OFF_HHI), sHlo = smem_u32(smem + L::OFF_HLO);
    bool ok = true;
    for (int c = 0; c < NC; ++c) {
      const int b = c & 1;
      if (!mbar_wait(&t_full[b], (c >> 1) & 1, p.wc, abort_flag, SITE_MLP_EPI)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v[HC];
#pragma unroll
      for (int q = 0; q < HC / 32; ++q)
        tmem_ld32(tmem + lane_off + b * HC + q * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[q * 32]));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&t_free[b]);
      uint32_t hi[HC / 2], lo[HC / 2];
#pragma unroll
      for (int k = 0; k < HC; k += 2) {
        float h0 = __uint_as_float(v[k]), h1 = __uint_as_float(v[k + 1]);
        if (p.gelu) {
          h0 = gelu_tanh(h0);
          h1 = gelu_tanh(h1);
        }
        const uint32_t ph = pack_bf16(h0, h1);
        hi[k / 2] = ph;
        lo[k / 2] = pack_bf16(h0 - __uint_as_float(ph << 16), h1 - __uint_as_float(ph & 0xffff0000u));
      }
      if (c >= 1 && !mbar_wait(h_free, (c - 1) & 1, p.wc, abort_flag, SITE_MLP_EPI)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const int bb = h * 32 + ch * 4;
          const uint32_t off = h * (BM * 128) + sw128_off(row, ch);
          st_shared_v4(sHhi + off, hi[bb], hi[bb + 1], hi[bb + 2], hi[bb + 3]);
          st_shared_v4(sHlo + off, lo[bb], lo[bb + 1], lo[bb + 2], lo[bb + 3]);
        }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(h_ready);
    }
    if (ok && mbar_wait(o_done, 0, p.wc, abort_flag, SITE_MLP_EPI)) {
      tc_fence_after();
      __nv_bfloat16 *orow = p.O + (int64_t)(rb * BM + row) * p.P + pb * BP;
#pragma unroll 1
      for (int q = 0; q < BP / 32; ++q) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + 256 + q * 32, r);
        tmem_wait_ld();
        uint4 *dst = reinterpret_cast<uint4 *>(orow + q * 32);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint4 o;
          o.x = pack_bf16(__uint_as_float(r[8 * k + 0]), __uint_as_float(r[8 * k + 1]));
          o.y = pack_bf16(__uint_as_float(r[8 * k + 2]), __uint_as_float(r[8 * k + 3]));
          o.z = pack_bf16(__uint_as_float(r[8 * k + 4]), __uint_as_float(r[8 * k + 5]));
          o.w = pack_bf16(__uint_as_float(r[8 * k + 6]), __uint_as_float(r[8 * k + 7]));
          dst[k] = o;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_mlp_chain(const MlpArgs &a, const WaitCfg &wc, cudaStream_t st) {
  if (a.M % BM || a.K % KT || a.N % HC || a.P % BP) return cudaErrorNotSupported;
  CUtensorMap mx, mw1, mw2;
  cudaError_t e;
  {
    const uint64_t d[2] = {(uint64_t)a.K, (uint64_t)a.M};
    const uint64_t s[1] = {(uint64_t)a.K * 2};
    const uint32_t box[2] = {64, 128};
    if ((e = make_tmap(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.X, d, s, box))) return e;
  }
  {
    const uint64_t d[2] = {(uint64_t)a.N, (uint64_t)a.K};
    const uint64_t s[1] = {(uint64_t)a.N * 2};
    const uint32_t box[2] = {64, 64};
    if ((e = make_tmap(&mw1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.W1, d, s, box))) return e;
  }
  {
    const uint64_t d[2] = {(uint64_t)a.P, (uint64_t)a.N};
    const uint64_t s[1] = {(uint64_t)a.P * 2};
    const uint32_t box[2] = {64, 64};
    if ((e = make_tmap(&mw2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.W2, d, s, box))) return e;
  }
  MlpParams p;
  p.M = a.M;
  p.K = a.K;
  p.N = a.N;
  p.P = a.P;
  p.gelu = a.gelu;
  p.O = static_cast<__nv_bfloat16 *>(a.O);
  p.wc = wc;
  if ((e = cudaFuncSetAttribute(mlp_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                MlpLayout::ALLOC)))
    return e;
  const unsigned grid = (unsigned)((a.M / BM) * (a.P / BP));
  timing_mark(st, 0);
  mlp_chain_kernel<<<grid, NTHREADS, MlpLayout::ALLOC, st>>>(mx, mw1, mw2, p);
  timing_mark(st, 1);
  return cudaGetLastError();
}

}  // namespace chain
