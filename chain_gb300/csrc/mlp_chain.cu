// mlp_chain.cu -- the MLP instance of the unit O = f(A B) C ("Memory-
// efficient tensor parallelism", FITEE 10.1631/FITEE.2400602, abstract):
//   O = f(X W1) W2,  f = GeLU (tanh form) or identity,
// X [M][K], W1 [K][N], W2 [N][P] bf16 row-major, O [M][P] bf16.  The
// [M][N] intermediate is produced 128 columns at a time in tensor memory,
// passed through f in registers and consumed from shared memory by the
// second product; it is never written to global memory (the activation
// the AutoSP write-up, section 2.B, recomputes instead of storing).
//
// Two kernels.  The default (mlp_cluster_kernel, P/256 = 2..4) shares the
// intermediate across a cluster so X W1 is formed once per row block; it is
// described where it is defined.  The other, used for the remaining shapes:
// one CTA per (128-row block of X, 256-column block of O).  For each
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


// ------------------------------------------------- cluster variant (default)
// One cluster of CS = P/256 CTAs (2 to 4) per 128-row block; CTA q of the
// cluster owns output columns [256q, 256q+256).  The hidden dimension runs in
// 64-wide chunks c.  Chunk c is computed (GEMM1, f, hi/lo split) once, by CTA
// k = c % CS, into its slot k; CTA k then pushes the 32 KB H_hi/H_lo tile (16
// KB of f16 H in the F16H instance) into slot k of every other CTA with bulk
// copies.  Every CTA runs GEMM2 over all chunks.  X W1 is formed once per row
// block instead of once per output block.
//
// Slot k is written only by CTA k:
//   h_full[k]   in every CTA: the chunk in slot k is present (remote: the
//               owner's copy completes the bytes the local MMA warp expects;
//               own: the epilogue arrives after writing it)
//   h_empty[k]  used in CTA k only: one multicast arrival from every CTA's
//               GEMM2 of the chunk in slot k; CTA k waits for it (phase by
//               phase) before overwriting the slot
// A CTA leaves after its own GEMM2s, its last h_empty phase and its outgoing
// copies have completed: then no peer can still write into its shared memory.
constexpr int HC2 = 64;
constexpr int MAX_CS = 4;

struct ClusterLayout {
  static constexpr int NST = 3;
  static constexpr uint32_t OFF_RING = 0;
  // [MAX_CS] x 32 KB: (hi 16 KB, lo 16 KB), or the f16 H in the first 16 KB
  static constexpr uint32_t OFF_SLOT = OFF_RING + NST * STAGE_BYTES;
  static constexpr uint32_t SLOT_BYTES = 32768;
  static constexpr uint32_t OFF_BAR = OFF_SLOT + MAX_CS * SLOT_BYTES;
  // full[3], empty[3], t_full[2], t_free[2], h_full[4], h_empty[4], o_done, mma_drain
  static constexpr uint32_t NBAR = 2 * NST + 4 + 2 * MAX_CS + 2;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t ALLOC = OFF_MISC + 16 + 1024;
};

struct ClusterParams {
  int M, K, N, P, gelu, CS;
  __nv_bfloat16 *O;
  const float *w_inv;  // F16H: 2^-k undoing the scale of W2's f16 copy
  WaitCfg wc;
};

// F16H: the intermediate enters the second product as ONE f16 tile (11
// significant bits) against an f16 copy of W2, instead of the bf16 pair
// H_hi, H_lo against bf16 W2: one product per chunk instead of two, and half
// the bytes per slot and per copy to the peers.
template <bool F16H>
__global__ void __launch_bounds__(NTHREADS, 1)
    mlp_cluster_kernel(const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmW1,
                       const __grid_constant__ CUtensorMap tmW2, const ClusterParams p) {
  using L = ClusterLayout;
  // bytes of one hidden chunk in a slot: H_hi then H_lo, or the f16 H alone
  constexpr uint32_t HBYTES = F16H ? L::SLOT_BYTES / 2 : L::SLOT_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
  uint64_t *full = bars;                  // [NST]
  uint64_t *empty = bars + L::NST;        // [NST]
  uint64_t *t_full = bars + 2 * L::NST;   // [2]
  uint64_t *t_free = t_full + 2;          // [2], 128 arrivals
  uint64_t *h_full = t_free + 2;          // [MAX_CS]
  uint64_t *h_empty = h_full + MAX_CS;    // [MAX_CS], CS arrivals
  uint64_t *o_done = h_empty + MAX_CS;
  uint64_t *mma_drain = o_done + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int CS = p.CS;
  const int q = (int)cluster_ctarank();
  const int rb = blockIdx.x / CS;
  const int NC = p.N / HC2;   // hidden chunks
  const int NKT = p.K / KT;   // GEMM1 K-tiles per chunk
  const int n_own = (NC - q + CS - 1) / CS;  // chunks q, q+CS, ...
  const int n_pair = (n_own + 1) / 2;        // GEMM1 runs on pairs (q+2jCS, q+(2j+1)CS)
  const uint32_t slot0 = smem_u32(smem + L::OFF_SLOT);

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&t_full[b], 1);
      mbar_init(&t_free[b], 128);
    }
    for (int k = 0; k < MAX_CS; ++k) {
      mbar_init(&h_full[k], 1);
      mbar_init(&h_empty[k], (uint32_t)CS);
    }
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
  // every CTA's barriers exist before any peer signals them
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // T buffers [0,128), [128,256) (a pair each); O [256,512)

  if (warp == 4) {
    // -------------------------------------------------------- producer
    // Consumption order of the MMA warp: GEMM1 of pair 0; then for each
    // chunk c: GEMM1 of the next pair when c opens a pair, then the W2 tile
    // of c.  A pair's W1 tile is two 64-column boxes (chunks c0 and c0+CS);
    // a missing second chunk reads as zeros (past N).
    if (lane == 0) {
      int st = 0;
      bool ok = true;
      auto stage = [&](bool is_g1, int c, int t) -> bool {
        const int s = st % L::NST;
        if (st >= L::NST &&
            !mbar_wait(&empty[s], ((st / L::NST) - 1) & 1, p.wc, abort_flag, SITE_MLP_PROD))
          return false;
        uint8_t *dst = smem + L::OFF_RING + s * STAGE_BYTES;
        if (is_g1) {  // X [rows][k tile] 16 KB + W1 [k tile][chunks c, c+CS] 2 x 8 KB
          mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
          tma_load_2d(dst, &tmX, &full[s], t * KT, rb * BM);
          tma_load_2d(dst + 16384, &tmW1, &full[s], c * HC2, t * KT);
          tma_load_2d(dst + 24576, &tmW1, &full[s], (c + CS) * HC2, t * KT);
        } else {      // W2 [hidden 64][out 256q..] as 4 boxes of 64 columns
          // F16H: W2's f16 copy comes from the pre-pass, which this kernel
          // may overlap (programmatic launch): wait for it before the first
          // W2 tile; GEMM1's operands before it do not depend on it
          if (F16H && c == 0) pdl_wait();
          mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            tma_load_2d(dst + i * 8192, &tmW2, &full[s], q * BP + i * 64, c * HC2);
        }
        ++st;
        return true;
      };
      if (n_pair >= 1)
        for (int t = 0; t < NKT && ok; ++t) ok = stage(true, q, t);
      for (int c = 0; c < NC && ok; ++c) {
        if (c % (2 * CS) == q && c + 2 * CS < NC)
          for (int t = 0; t < NKT && ok; ++t) ok = stage(true, c + 2 * CS, t);
        if (ok) ok = stage(false, c, 0);
      }
      if (*abort_flag) {
        for (int j = (st > L::NST ? st - L::NST : 0); j < st; ++j)
          drain_wait(&full[j % L::NST], (j / L::NST) & 1, p.wc);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------ MMA issuer
    {
      const uint32_t id1 = idesc_bf16_f32(BM, 2 * HC2, 0, 1);  // T = X W1 (a pair), W1 MN-major
      const uint32_t id2 = F16H ? idesc_f16_f32(BM, BP, 0, 1)     // O += H W2, W2 MN-major
                                : idesc_bf16_f32(BM, BP, 0, 1);
      const uint32_t ring = smem_u32(smem + L::OFF_RING);
      int st = 0;
      bool ok = true;
      auto gemm1 = [&](int j) -> bool {  // own pair j into T buffer j & 1
        const int b = j & 1;
        if (j >= 2 && !mbar_wait_warp(&t_free[b], ((j >> 1) - 1) & 1, p.wc, abort_flag, SITE_MLP_MMA))
          return false;
        for (int t = 0; t < NKT; ++t, ++st) {
          const int s = st % L::NST;
          if (!mbar_wait_warp(&full[s], (st / L::NST) & 1, p.wc, abort_flag, SITE_MLP_MMA)) return false;
          tc_fence_after();
          const SDesc ax = sdesc_make(ring + s * STAGE_BYTES, 16, 1024);
          const SDesc bw = sdesc_make(ring + s * STAGE_BYTES + 16384, 8192, 1024);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < KT / 16; ++kk)
              umma_f16_ss(tmem + b * 2 * HC2, sdesc_at(ax, kk * 32), sdesc_at(bw, kk * 2048), id1,
                          (t > 0 || kk > 0) ? 1u : 0u);
            umma_commit(&empty[s]);
          }
          __syncwarp();
        }
        if (elect_one()) umma_commit(&t_full[b]);
        __syncwarp();
        return true;
      };
      int pair = 0;
      if (n_pair >= 1) ok = gemm1(pair++);
      for (int c = 0; c < NC && ok; ++c) {
        if (c % (2 * CS) == q && c + 2 * CS < NC && !(ok = gemm1(pair++))) break;
        // GEMM2 of chunk c from slot k = its owner
        const int k = c % CS, u = c / CS;
        if (k != q && elect_one()) mbar_arrive_expect_tx(&h_full[k], HBYTES);
        __syncwarp();
        if (!mbar_wait_warp(&h_full[k], u & 1, p.wc, abort_flag, SITE_MLP_MMA)) {
          ok = false;
          break;
        }
        const int s = st % L::NST;
        if (!mbar_wait_warp(&full[s], (st / L::NST) & 1, p.wc, abort_flag, SITE_MLP_MMA)) {
          ok = false;
          break;
        }
        ++st;
        tc_fence_after();
        const SDesc bw = sdesc_make(ring + s * STAGE_BYTES, 8192, 1024);
        const SDesc dhi = sdesc_make(slot0 + k * L::SLOT_BYTES, 16, 1024);
        const SDesc dlo = sdesc_make(slot0 + k * L::SLOT_BYTES + 16384, 16, 1024);
        if (elect_one()) {
#pragma unroll
          for (int part = 0; part < (F16H ? 1 : 2); ++part)
#pragma unroll
            for (int kk = 0; kk < HC2 / 16; ++kk)
              umma_f16_ss(tmem + 256, sdesc_at(part ? dlo : dhi, kk * 32), sdesc_at(bw, kk * 2048),
                          id2, (c > 0 || part > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&empty[s]);
          umma_commit_multicast(&h_empty[k], (uint16_t)(1u << k));  // slot k read here
        }
        __syncwarp();
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
    // Every thread passes the same named barriers in every iteration; after
    // a failure (abort flag) the waits and copies are skipped, not the loop.
    const int row = threadIdx.x;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t my_hi = slot0 + q * L::SLOT_BYTES, my_lo = my_hi + 16384;
    const bool issuer = threadIdx.x == 0;
    bool ok = true;
    bool beyond = false;  // F16H: some f(T) outside f16's finite range
    for (int i = 0; i < n_own; ++i) {
      const int j = i >> 1, h = i & 1, b = j & 1;  // pair j, half h, T buffer b
      if (ok && h == 0) ok = mbar_wait(&t_full[b], (j >> 1) & 1, p.wc, abort_flag, SITE_MLP_EPI);
      tc_fence_after();
      uint32_t v[HC2];
      const uint32_t tcol = tmem + lane_off + b * 2 * HC2 + h * HC2;
      tmem_ld32(tcol, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld32(tcol + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tmem_wait_ld();
      tc_fence_before();
      if (h == 1 || i == n_own - 1) mbar_arrive(&t_free[b]);  // both halves of the pair read
      uint32_t hi[HC2 / 2], lo[HC2 / 2];
#pragma unroll
      for (int k = 0; k < HC2; k += 2) {
        float h0 = __uint_as_float(v[k]), h1 = __uint_as_float(v[k + 1]);
        if (p.gelu) {
          h0 = gelu_tanh(h0);
          h1 = gelu_tanh(h1);
        }
        if constexpr (F16H) {
          const uint32_t ph = pack_f16(h0, h1);
          hi[k / 2] = ph;
          // an all-ones exponent field: infinite or NaN
          beyond |= ((ph & 0x7c00u) == 0x7c00u) | ((ph & 0x7c000000u) == 0x7c000000u);
        } else {
          const uint32_t ph = pack_bf16(h0, h1);
          hi[k / 2] = ph;
          lo[k / 2] = pack_bf16(h0 - __uint_as_float(ph << 16), h1 - __uint_as_float(ph & 0xffff0000u));
        }
      }
      // slot q may be overwritten once every CTA has run GEMM2 on the
      // previous own chunk and this CTA's copies of it have read the slot
      if (issuer && ok) {
        if (i >= 1) ok = mbar_wait(&h_empty[q], (i - 1) & 1, p.wc, abort_flag, SITE_MLP_EPI);
        bulk_wait_read_all();
      }
      named_bar_sync(1, 128);
      if (*abort_flag) ok = false;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const uint32_t off = sw128_off(row, ch);
        st_shared_v4(my_hi + off, hi[4 * ch], hi[4 * ch + 1], hi[4 * ch + 2], hi[4 * ch + 3]);
        if constexpr (!F16H)
          st_shared_v4(my_lo + off, lo[4 * ch], lo[4 * ch + 1], lo[4 * ch + 2], lo[4 * ch + 3]);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (issuer && ok) {
        mbar_arrive(&h_full[q]);  // own GEMM2 reads the slot in place
        for (int r = 0; r < CS; ++r)
          if (r != q)
            bulk_copy_to_cluster(mapa_shared(my_hi, (uint32_t)r), my_hi, HBYTES,
                                 mapa_shared(smem_u32(&h_full[q]), (uint32_t)r));
        bulk_commit_group();
      }
    }
    if constexpr (F16H) {
      // reported by the next chain_check (the result is then not valid)
      if (__any_sync(0xffffffffu, beyond) && lane == 0) atomicExch(&p.wc.status->reserved[0], 1);
    }
    // O epilogue
    if (ok && mbar_wait(o_done, 0, p.wc, abort_flag, SITE_MLP_EPI)) {
      tc_fence_after();
      if (F16H) pdl_wait();  // the pre-pass's scale (returns at once by now)
      const float os = F16H ? __ldg(p.w_inv) : 1.0f;
      __nv_bfloat16 *orow = p.O + (int64_t)(rb * BM + row) * p.P + q * BP;
#pragma unroll 1
      for (int j = 0; j < BP / 32; ++j) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + 256 + j * 32, r);
        tmem_wait_ld();
        uint4 *dst = reinterpret_cast<uint4 *>(orow + j * 32);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint4 o;
          o.x = pack_bf16(__uint_as_float(r[8 * k + 0]) * os, __uint_as_float(r[8 * k + 1]) * os);
          o.y = pack_bf16(__uint_as_float(r[8 * k + 2]) * os, __uint_as_float(r[8 * k + 3]) * os);
          o.z = pack_bf16(__uint_as_float(r[8 * k + 4]) * os, __uint_as_float(r[8 * k + 5]) * os);
          o.w = pack_bf16(__uint_as_float(r[8 * k + 6]) * os, __uint_as_float(r[8 * k + 7]) * os);
          dst[k] = o;
        }
      }
    }
    // Before leaving: the outgoing copies have completed, and every CTA has
    // run GEMM2 on this CTA's last chunk (the last h_empty phase, one phase
    // after the one waited for above), so no peer signals this CTA any more.
    if (issuer) {
      bulk_wait_all();
      if (n_own >= 1) {
        volatile int never = 0;
        mbar_wait(&h_empty[q], (n_own - 1) & 1, p.wc, &never, SITE_MLP_DRAIN);
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

// ------------------------------------------------ W2 -> f16 (F16H only)
// One power-of-two scale 2^k for the whole of W2, chosen from its largest
// |w| (bf16 magnitude bits order like the values) so that it lands in
// [2^14, 2^15): every bf16 value is then exact in f16 except values below
// 2^-31 of that maximum (f16 subnormals, absolute error at most 2^-39 of
// it).  Two passes: WPB partial maxima, then each block reduces them,
// converts its share and (block 0) stores 2^-k for the epilogue.
constexpr int WPB = 256;   // blocks of both passes (partial maxima of the first): with the
                           // main kernel all resident at once, so the launches overlap
constexpr int WU = 4;      // 16-byte vectors in flight per thread and round

__device__ __forceinline__ uint32_t block_max256(uint32_t v, uint32_t *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  v = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) v = max(v, red[w]);
  __syncthreads();
  return v;
}

__global__ void __launch_bounds__(256)
    w_absmax_kernel(const uint4 *__restrict__ W, int64_t nvec, uint32_t *__restrict__ part) {
  pdl_launch_dependents();  // the conversion may launch now; it waits for this grid
  __shared__ uint32_t red[8];
  const int64_t stride = (int64_t)gridDim.x * 256;
  uint32_t m = 0;
  for (int64_t base = blockIdx.x * 256 + threadIdx.x; base < nvec; base += WU * stride) {
    uint4 x[WU];
#pragma unroll
    for (int u = 0; u < WU; ++u)
      x[u] = base + u * stride < nvec ? __ldg(W + base + u * stride) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < WU; ++u) {
      const uint32_t w[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) m = max(m, max(w[k] & 0x7fffu, (w[k] >> 16) & 0x7fffu));
    }
  }
  m = block_max256(m, red);
  if (threadIdx.x == 0) part[blockIdx.x] = m;
}

__global__ void __launch_bounds__(256)
    w_to_f16_kernel(const uint4 *__restrict__ W, int64_t nvec, const uint32_t *__restrict__ part,
                    uint4 *__restrict__ out, float *__restrict__ w_inv) {
  // the main kernel may begin launching now; it waits for this grid's
  // completion before it reads the copy or the scale
  pdl_launch_dependents();
  pdl_wait();  // the partial maxima of w_absmax_kernel
  __shared__ uint32_t red[8];
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < WPB / 256; ++i) m = max(m, part[i * 256 + threadIdx.x]);
  m = block_max256(m, red);
  // exponent field e of the largest |w|: k = 141 - e puts it in [2^14, 2^15);
  // zero, infinite or NaN maxima keep k = 0
  const int e = (int)(m >> 7);
  int k = (m == 0 || e == 255) ? 0 : 141 - e;
  k = k < -126 ? -126 : (k > 126 ? 126 : k);
  const float sc = __uint_as_float((uint32_t)(127 + k) << 23);
  if (blockIdx.x == 0 && threadIdx.x == 0) *w_inv = __uint_as_float((uint32_t)(127 - k) << 23);
  const int64_t stride = (int64_t)gridDim.x * 256;
  for (int64_t base = blockIdx.x * 256 + threadIdx.x; base < nvec; base += WU * stride) {
    uint4 x[WU];
#pragma unroll
    for (int u = 0; u < WU; ++u)
      x[u] = base + u * stride < nvec ? __ldg(W + base + u * stride) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < WU; ++u) {
      const uint32_t w[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
      uint32_t y[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        y[q] = pack_f16(__uint_as_float(w[q] << 16) * sc, __uint_as_float(w[q] & 0xffff0000u) * sc);
      if (base + u * stride < nvec) out[base + u * stride] = make_uint4(y[0], y[1], y[2], y[3]);
    }
  }
}

// Tensor maps of X [M][K] (64 x 128 boxes), W1 [K][N] and W2 [N][P] (64 x 64
// boxes); W2 as bf16 or as its f16 copy.
cudaError_t mlp_maps(const MlpArgs &a, const void *w2, CUtensorMapDataType w2_type,
                     CUtensorMap *mx, CUtensorMap *mw1, CUtensorMap *mw2) {
  cudaError_t e;
  {
    const uint64_t d[2] = {(uint64_t)a.K, (uint64_t)a.M};
    const uint64_t s[1] = {(uint64_t)a.K * 2};
    const uint32_t box[2] = {64, 128};
    if ((e = make_tmap(mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.X, d, s, box))) return e;
  }
  {
    const uint64_t d[2] = {(uint64_t)a.N, (uint64_t)a.K};
    const uint64_t s[1] = {(uint64_t)a.N * 2};
    const uint32_t box[2] = {64, 64};
    if ((e = make_tmap(mw1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.W1, d, s, box))) return e;
  }
  {
    const uint64_t d[2] = {(uint64_t)a.P, (uint64_t)a.N};
    const uint64_t s[1] = {(uint64_t)a.P * 2};
    const uint32_t box[2] = {64, 64};
    if ((e = make_tmap(mw2, w2_type, 2, w2, d, s, box))) return e;
  }
  return cudaSuccess;
}

// F16H: launched to overlap the tail of its pre-pass (programmatic stream
// serialization); the kernel waits for the pre-pass where it first needs W2.
template <bool F16H>
cudaError_t launch_cluster(const MlpArgs &a, const CUtensorMap &mx, const CUtensorMap &mw1,
                           const CUtensorMap &mw2, const float *w_inv, const WaitCfg &wc,
                           cudaStream_t st) {
  // X W1 once per row block, shared through the cluster
  const int CS = a.P / BP;
  ClusterParams p;
  p.M = a.M; p.K = a.K; p.N = a.N; p.P = a.P; p.gelu = a.gelu; p.CS = CS;
  p.O = static_cast<__nv_bfloat16 *>(a.O);
  p.w_inv = w_inv;
  p.wc = wc;
  cudaError_t e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((a.M / BM) * CS));
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = ClusterLayout::ALLOC;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = F16H ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, mlp_cluster_kernel<F16H>, mx, mw1, mw2, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

bool cluster_shape(const MlpArgs &a) {
  const int CS = a.P / BP;
  return a.P % BP == 0 && CS >= 2 && CS <= MAX_CS && a.N % HC2 == 0;
}

}  // namespace

cudaError_t launch_mlp_chain(const MlpArgs &a, const WaitCfg &wc, cudaStream_t st) {
  if (a.M % BM || a.K % KT || a.N % HC || a.P % BP) return cudaErrorNotSupported;
  CUtensorMap mx, mw1, mw2;
  cudaError_t e;
  if ((e = mlp_maps(a, a.W2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, &mx, &mw1, &mw2))) return e;
  if (cluster_shape(a)) {
    if ((e = cudaFuncSetAttribute(mlp_cluster_kernel<false>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, ClusterLayout::ALLOC)))
      return e;
    timing_mark(st, 0);
    e = launch_cluster<false>(a, mx, mw1, mw2, nullptr, wc, st);
    timing_mark(st, 1);
    return e;
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

size_t mlp_f16h_workspace(int64_t N, int64_t P) {
  const size_t wb = ((size_t)N * (size_t)P * 2 + 255) & ~(size_t)255;
  return wb + 4 * WPB + 256;
}

cudaError_t launch_mlp_chain_f16h(const MlpArgs &a, void *ws, const WaitCfg &wc,
                                  cudaStream_t st) {
  if (a.M % BM || a.K % KT || !cluster_shape(a)) return cudaErrorNotSupported;
  uint8_t *base = static_cast<uint8_t *>(ws);
  const size_t wb = ((size_t)a.N * (size_t)a.P * 2 + 255) & ~(size_t)255;
  uint4 *w16 = reinterpret_cast<uint4 *>(base);
  uint32_t *part = reinterpret_cast<uint32_t *>(base + wb);
  float *w_inv = reinterpret_cast<float *>(base + wb + 4 * WPB);
  const int64_t nvec = (int64_t)a.N * a.P / 8;  // P is a multiple of 256
  // Host work first, so the main kernel's launch follows the pre-pass's
  // closely enough to overlap its tail.
  CUtensorMap mx, mw1, mw2;
  cudaError_t e;
  if ((e = mlp_maps(a, w16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, &mx, &mw1, &mw2))) return e;
  if ((e = cudaFuncSetAttribute(mlp_cluster_kernel<true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, ClusterLayout::ALLOC)))
    return e;
  timing_mark(st, 0);
  w_absmax_kernel<<<WPB, 256, 0, st>>>(static_cast<const uint4 *>(a.W2), nvec, part);
  {
    // the conversion launches while the maxima are still being taken
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(WPB);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, w_to_f16_kernel, static_cast<const uint4 *>(a.W2), nvec,
                                static_cast<const uint32_t *>(part), w16, w_inv)))
      return e;
  }
  if ((e = cudaGetLastError())) return e;
  // no mark between the pre-pass and the main kernel: a recorded event there
  // would keep them from overlapping
  e = launch_cluster<true>(a, mx, mw1, mw2, w_inv, wc, st);
  timing_mark(st, 1);
  return e;
}

}  // namespace chain
