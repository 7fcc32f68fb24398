// attn_bwd.cu -- backward of softmax attention with recompute.
//
// The forward keeps only O and the row log-sum-exp; the backward rebuilds
// S and P tile by tile from them instead of storing the n x n matrices
// ("AutoSP: Unlocking Long-Context LLM Training Via Compiler-Based Sequence
// Parallelism", section 2.B: discard activations and recompute them in the
// backward pass; the unit itself is the O = f(AB)C of "Memory-efficient
// tensor parallelism", FITEE 10.1631/FITEE.2400602).  With P = softmax(S),
// S = scale Q K^T, dP = dO V^T, D_i = sum_e dO_ie O_ie:
//   dV = P^T dO,  dS = P o (dP - D),  dK = scale dS^T Q,  dQ = scale dS K.
//
// Three kernels:
//   bwd_prep    D_i = sum_e dO_ie O_ie (fp32), zeroes the fp32 dQ accumulator;
//   bwd_main    one CTA per (head, 128-key block j), looping over the query
//               tiles i that see block j (i >= j when causal);
//   bwd_dq_cvt  dQ accumulator (fp32) -> dQ (bf16).
//
// bwd_main roles (448 threads):
//   warps 0-7  compute, two warpgroups: warpgroup w takes queries
//              [64w, 64w+64) of each tile; thread r owns key row j*128 + r
//              (tensor-memory lane r).  P^T = exp2(S^T scale log2e - LSE)
//              is written back as bf16 over the S^T columns it was read from
//              and feeds dV from tensor memory; dS^T = P^T o (dP^T - D) goes
//              to a 128-byte-swizzled shared tile read by dK (K-major) and
//              dQ (MN-major, as dS).
//   warps 8-11 dQ drain: reads dQ_i (lane = query row) and adds it into the
//              fp32 accumulator with red.global.add.v4.f32 while the next
//              tile is computed.
//   warp 12    TMA producer: K_j, V_j once; Q_i (2 stages), dO_i (1 stage).
//   warp 13    MMA issuer.  Per tile:  S^T = K_j Q_i^T,  dP^T = V_j dO_i^T,
//              then  dV += P^T dO_i,  dK += dS^T Q_i,  dQ_i = dS K_j.
// Tensor memory: S^T / P^T [0,128), dP^T and dQ_i [128,256), dV [256,256+d),
// dK [256+d, 256+2d).  CTAs run head by head so the key blocks of a head
// share Q, dO, LSE and D through L2.
#include "internal.h"

namespace chain {
namespace {

constexpr int BM = 128;  // rows per tile (keys and queries)
constexpr int NTHREADS = 448;

template <int D>
struct BwdLayout {
  static constexpr uint32_t T_BYTES = BM * D * 2;   // one [128][D] bf16 tile
  static constexpr uint32_t S_BYTES = BM * BM * 2;  // one [128][128] bf16 tile
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + T_BYTES;
  static constexpr uint32_t OFF_Q = OFF_V + T_BYTES;       // 2 stages
  static constexpr uint32_t OFF_DO = OFF_Q + 2 * T_BYTES;  // 1 stage
  static constexpr uint32_t OFF_DST = OFF_DO + T_BYTES;
  static constexpr uint32_t OFF_LD = OFF_DST + S_BYTES;    // LSE and D staging, 2 KB
  static constexpr uint32_t OFF_BAR = OFF_LD + 2048;
  static constexpr uint32_t NBAR = 15;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  static constexpr uint32_t ALLOC = (BYTES + 1024 > 120 * 1024) ? BYTES + 1024 : 120 * 1024;
};

struct BwdParams {
  int BH, n, nqb, causal;
  float scale, scale_log2;
  const float *LSE;  // [BH][n]
  const float *Dvec; // [BH][n]
  float *dq_acc;     // [BH][n][D]
  __nv_bfloat16 *dK, *dV;
  WaitCfg wc;
};

enum : int {
  SITE_BWD_PROD = 0x201,
  SITE_BWD_MMA = 0x202,
  SITE_BWD_COMPUTE = 0x203,
  SITE_BWD_EPI = 0x204,
  SITE_BWD_DRAIN = 0x205
};

__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, const WaitCfg &wc) {
  volatile int never = 0;
  mbar_wait(bar, parity, wc, &never, SITE_BWD_DRAIN);
}

// ------------------------------------------------------------ preprocess
// 16 threads per row of d = 128 (8 per row of d = 64): each loads 16 bytes
// of O and dO, the partial dot products are reduced with shuffles.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16 *__restrict__ O,
                                                       const __nv_bfloat16 *__restrict__ dO,
                                                       float *__restrict__ Dvec,
                                                       float *__restrict__ dq_acc,
                                                       int64_t rows) {
  constexpr int TPR = D / 8;  // threads per row
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = tid / TPR;
  const int part = (int)(tid % TPR);
  float acc = 0.0f;
  if (row < rows) {
    const uint4 a = *reinterpret_cast<const uint4 *>(O + row * D + part * 8);
    const uint4 b = *reinterpret_cast<const uint4 *>(dO + row * D + part * 8);
    const __nv_bfloat162 *pa = reinterpret_cast<const __nv_bfloat162 *>(&a);
    const __nv_bfloat162 *pb = reinterpret_cast<const __nv_bfloat162 *>(&b);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 fa = __bfloat1622float2(pa[k]);
      const float2 fb = __bfloat1622float2(pb[k]);
      acc = fmaf(fa.x, fb.x, acc);
      acc = fmaf(fa.y, fb.y, acc);
    }
    float4 *z = reinterpret_cast<float4 *>(dq_acc + row * D + part * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && part == 0) Dvec[row] = acc;
}

// ------------------------------------------------------------ dQ convert
__global__ void __launch_bounds__(256) bwd_dq_cvt_kernel(const float *__restrict__ acc,
                                                         __nv_bfloat16 *__restrict__ dq,
                                                         int64_t n8) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4 *>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4 *>(acc)[2 * i + 1];
    uint4 o;
    o.x = pack_bf16(a.x, a.y);
    o.y = pack_bf16(a.z, a.w);
    o.z = pack_bf16(b.x, b.y);
    o.w = pack_bf16(b.z, b.w);
    reinterpret_cast<uint4 *>(dq)[i] = o;
  }
}

// ------------------------------------------------------------ main kernel
template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmdO, const BwdParams p) {
  using L = BwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
  uint64_t *kv_full = bars + 0;
  uint64_t *q_full = bars + 1;   // [2]
  uint64_t *q_empty = bars + 3;  // [2]
  uint64_t *do_full = bars + 5;
  uint64_t *do_empty = bars + 6;
  uint64_t *s_full = bars + 7;
  uint64_t *dp_full = bars + 8;
  uint64_t *p_ready = bars + 9;   // both compute warpgroups (256 arrivals)
  uint64_t *dq_full = bars + 10;
  uint64_t *dq_free = bars + 11;  // drain warpgroup (128 arrivals)
  uint64_t *ds_free = bars + 12;
  uint64_t *fin = bars + 13;
  uint64_t *mma_drain = bars + 14;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);
  // staged LSE (log2 units) and D: [warpgroup][buffer][64 queries]
  float *sL = reinterpret_cast<float *>(smem + L::OFF_LD);
  float *sDv = sL + 2 * 2 * 64;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // head-major order: the key blocks of one head run together and share
  // Q, dO, LSE and D through L2; smallest (heaviest causal) block first
  const int bh = blockIdx.x / p.nqb;
  const int jb = blockIdx.x % p.nqb;
  const int i_begin = p.causal ? jb : 0;
  const int T = p.nqb - i_begin;

  if (threadIdx.x == 0) {
    for (int b = 0; b < (int)L::NBAR; ++b) {
      uint32_t cnt = 1;
      if (&bars[b] == p_ready) cnt = 256;
      if (&bars[b] == dq_free) cnt = 128;
      mbar_init(&bars[b], cnt);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 13) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 12 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 12) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int q_issued = 0, do_issued = 0;
      mbar_arrive_expect_tx(kv_full, 2 * L::T_BYTES);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(smem + L::OFF_K + c * (BM * 128), &tmK, kv_full, c * 64, jb * BM, bh);
        tma_load_3d(smem + L::OFF_V + c * (BM * 128), &tmV, kv_full, c * 64, jb * BM, bh);
      }
      for (int t = 0; t < T; ++t) {
        const int i = i_begin + t, qs = t & 1;
        if (t >= 2 &&
            !mbar_wait(&q_empty[qs], ((t >> 1) - 1) & 1, p.wc, abort_flag, SITE_BWD_PROD))
          break;
        mbar_arrive_expect_tx(&q_full[qs], L::T_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::OFF_Q + qs * L::T_BYTES + c * (BM * 128), &tmQ, &q_full[qs],
                      c * 64, i * BM, bh);
        q_issued = t + 1;
        if (t >= 1 && !mbar_wait(do_empty, (t - 1) & 1, p.wc, abort_flag, SITE_BWD_PROD)) break;
        mbar_arrive_expect_tx(do_full, L::T_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::OFF_DO + c * (BM * 128), &tmdO, do_full, c * 64, i * BM, bh);
        do_issued = t + 1;
      }
      if (*abort_flag) {
        drain_wait(kv_full, 0, p.wc);
        for (int t = (q_issued > 2 ? q_issued - 2 : 0); t < q_issued; ++t)
          drain_wait(&q_full[t & 1], (t >> 1) & 1, p.wc);
        if (do_issued > 0) drain_wait(do_full, (do_issued - 1) & 1, p.wc);
      }
    }
    __syncwarp();
  } else if (warp == 13) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(BM, BM, 0, 0);  // S^T, dP^T
      const uint32_t id_kv = idesc_bf16_f32(BM, D, 0, 1);  // dV (A in TMEM), dK
      const uint32_t id_q = idesc_bf16_f32(BM, D, 1, 1);   // dQ
      const uint32_t sK = smem_u32(smem + L::OFF_K);
      const uint32_t sV = smem_u32(smem + L::OFF_V);
      const uint32_t sQ0 = smem_u32(smem + L::OFF_Q);
      const uint32_t sdO = smem_u32(smem + L::OFF_DO);
      const uint32_t sdST = smem_u32(smem + L::OFF_DST);
      const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;
      auto issue_s = [&](int t) {  // S^T = K_j Q_t^T
        const uint32_t sQ = sQ0 + (t & 1) * L::T_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
          umma_f16_ss(tS, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ + off, 16, 1024), id_s,
                      kk > 0 ? 1u : 0u);
        }
      };
      auto issue_dp = [&]() {  // dP^T = V_j dO_t^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
          umma_f16_ss(tdP, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sdO + off, 16, 1024),
                      id_s, kk > 0 ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(kv_full, 0, p.wc, abort_flag, SITE_BWD_MMA) &&
                mbar_wait(&q_full[0], 0, p.wc, abort_flag, SITE_BWD_MMA);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        umma_commit(s_full);
        ok = mbar_wait(do_full, 0, p.wc, abort_flag, SITE_BWD_MMA);
        if (ok) {
          tc_fence_after();
          issue_dp();
          umma_commit(dp_full);
        }
      }
      for (int t = 0; ok && t < T; ++t) {
        const int qs = t & 1;
        const uint32_t sQ = sQ0 + qs * L::T_BYTES;
        if (!mbar_wait(p_ready, t & 1, p.wc, abort_flag, SITE_BWD_MMA)) break;
        tc_fence_after();
        // dV += P^T dO_t: A = P^T in tensor memory (queries [64w, 64w+64)
        // packed into columns [64w, 64w+32)), B = dO MN-major
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          umma_f16_ts(tdV, tS + (kk >> 2) * 64 + (kk & 3) * 8,
                      sdesc_sw128(sdO + kk * 2048, BM * 128, 1024), id_kv,
                      (t > 0 || kk > 0) ? 1u : 0u);
        umma_commit(do_empty);
        // dK += dS^T Q_t
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk) {
          const uint32_t aoff = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
          umma_f16_ss(tdK, sdesc_sw128(sdST + aoff, 16, 1024),
                      sdesc_sw128(sQ + kk * 2048, BM * 128, 1024), id_kv,
                      (t > 0 || kk > 0) ? 1u : 0u);
        }
        // dQ_t = dS K_j (A: dS read MN-major from the dS^T tile; B: K MN-major)
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          umma_f16_ss(tdP, sdesc_sw128(sdST + kk * 2048, BM * 128, 1024),
                      sdesc_sw128(sK + kk * 2048, BM * 128, 1024), id_q, kk > 0 ? 1u : 0u);
        umma_commit(dq_full);
        umma_commit(&q_empty[qs]);
        umma_commit(ds_free);
        if (t + 1 < T) {
          if (!mbar_wait(&q_full[(t + 1) & 1], ((t + 1) >> 1) & 1, p.wc, abort_flag, SITE_BWD_MMA))
            break;
          tc_fence_after();
          issue_s(t + 1);  // after dV_t in issue order: P^T_t is consumed first
          umma_commit(s_full);
          if (!mbar_wait(do_full, (t + 1) & 1, p.wc, abort_flag, SITE_BWD_MMA)) break;
          if (!mbar_wait(dq_free, t & 1, p.wc, abort_flag, SITE_BWD_MMA)) break;
          tc_fence_after();
          issue_dp();
          umma_commit(dp_full);
        }
      }
      if (ok) umma_commit(fin);
      umma_commit(mma_drain);
      drain_wait(mma_drain, 0, p.wc);
    }
    __syncwarp();
  } else if (warp >= 8) {
    // ----------------------------------------------------- dQ drain (WG2)
    const int r = threadIdx.x - 256;  // tensor-memory lane = query row of dQ_t
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    for (int t = 0; t < T; ++t) {
      if (!mbar_wait(dq_full, t & 1, p.wc, abort_flag, SITE_BWD_DRAIN + 0x10)) break;
      tc_fence_after();
      const int q = (i_begin + t) * BM + r;
      float *dst = p.dq_acc + ((int64_t)bh * p.n + q) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + 128 + c * 32, v);
        tmem_wait_ld();
        if (q < p.n) {
#pragma unroll
          for (int k = 0; k < 32; k += 4)
            red_add_v4(dst + c * 32 + k, __uint_as_float(v[k]) * p.scale,
                       __uint_as_float(v[k + 1]) * p.scale, __uint_as_float(v[k + 2]) * p.scale,
                       __uint_as_float(v[k + 3]) * p.scale);
        }
      }
      tc_fence_before();
      mbar_arrive(dq_free);
    }
  } else {
    // ------------------------------------------- compute (WG0 and WG1)
    // Warpgroup w handles queries [64w, 64w+64) of every tile; thread r
    // owns key row j*128 + r (tensor-memory lane r).
    const int w = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int kv_idx = jb * BM + r;
    const bool kv_ok = kv_idx < p.n;
    const uint32_t sdST = smem_u32(smem + L::OFF_DST);
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      const int i = i_begin + t, buf = t & 1;
      const bool diag = p.causal && (i == jb);
      float *wl = sL + (w * 2 + buf) * 64;
      float *wd = sDv + (w * 2 + buf) * 64;
      if (r < 64) {
        const int q = i * BM + 64 * w + r;
        const bool q_ok = q < p.n;
        wl[r] = q_ok ? p.LSE[(int64_t)bh * p.n + q] * 1.4426950408889634f : INFINITY;
        wd[r] = q_ok ? p.Dvec[(int64_t)bh * p.n + q] : 0.0f;
      }
      named_bar_sync(1 + w, 128);
      if (!mbar_wait(s_full, t & 1, p.wc, abort_flag, SITE_BWD_COMPUTE)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // P^T for the 64 queries: packed bf16 pairs, written over the S^T
      // columns this warpgroup has just read
      uint32_t pk[32];
      {
        uint32_t sv[64];
        tmem_ld32(tmem + lane_off + 64 * w, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_ld32(tmem + lane_off + 64 * w + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float pv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int qq = c + u;
            float pr = ex2(fmaf(__uint_as_float(sv[qq]), p.scale_log2, -wl[qq]));
            if (!kv_ok || (diag && 64 * w + qq < r)) pr = 0.0f;
            pv[u] = pr;
          }
          pk[c / 2] = pack_bf16(pv[0], pv[1]);
        }
      }
      tmem_st32(tmem + lane_off + 64 * w, pk);
      if (!mbar_wait(dp_full, t & 1, p.wc, abort_flag, SITE_BWD_COMPUTE)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (t >= 1 && !mbar_wait(ds_free, (t - 1) & 1, p.wc, abort_flag, SITE_BWD_COMPUTE)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t dp[32];
        tmem_ld32(tmem + lane_off + 128 + 64 * w + 32 * h, dp);
        tmem_wait_ld();
        uint32_t dd[16];
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          const int qq = 32 * h + k;
          const uint32_t pp = pk[qq / 2];
          const float p0 = __uint_as_float(pp << 16), p1 = __uint_as_float(pp & 0xffff0000u);
          dd[k / 2] = pack_bf16(p0 * (__uint_as_float(dp[k]) - wd[qq]),
                                p1 * (__uint_as_float(dp[k + 1]) - wd[qq + 1]));
        }
        // queries [64w + 32h, +32) = chunks 4h..4h+3 of half w of the dS^T tile
#pragma unroll
        for (int u = 0; u < 4; ++u)
          st_shared_v4(sdST + w * (BM * 128) + sw128_off(r, 4 * h + u), dd[4 * u], dd[4 * u + 1],
                       dd[4 * u + 2], dd[4 * u + 3]);
      }
      fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_ready);
    }
    // --------------------------------------------------- dK, dV epilogue
    if (ok && T > 0 && mbar_wait(fin, 0, p.wc, abort_flag, SITE_BWD_EPI)) {
      tc_fence_after();
      // WG0 writes dV, WG1 writes dK (times scale)
      const uint32_t col = 256 + w * D;
      const float mul = w ? p.scale : 1.0f;
      __nv_bfloat16 *row = (w ? p.dK : p.dV) + ((int64_t)bh * p.n + kv_idx) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t a[32];
        tmem_ld32(tmem + lane_off + col + c * 32, a);
        tmem_wait_ld();
        if (kv_ok) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(a[8 * k + 0]) * mul, __uint_as_float(a[8 * k + 1]) * mul);
            v.y = pack_bf16(__uint_as_float(a[8 * k + 2]) * mul, __uint_as_float(a[8 * k + 3]) * mul);
            v.z = pack_bf16(__uint_as_float(a[8 * k + 4]) * mul, __uint_as_float(a[8 * k + 5]) * mul);
            v.w = pack_bf16(__uint_as_float(a[8 * k + 6]) * mul, __uint_as_float(a[8 * k + 7]) * mul);
            reinterpret_cast<uint4 *>(row + c * 32)[k] = v;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_bwd_d(const AttnBwdArgs &a, const WaitCfg &wc, cudaStream_t st) {
  using L = BwdLayout<D>;
  const int64_t rows = (int64_t)a.BH * a.n;
  cudaError_t e;
  {
    const int64_t threads = rows * (D / 8);
    const unsigned grid = (unsigned)((threads + 255) / 256);
    bwd_prep_kernel<D><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(a.O),
                                             static_cast<const __nv_bfloat16 *>(a.dO), a.Dvec,
                                             a.dq_acc, rows);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  CUtensorMap mq, mk, mv, mdo;
  const uint32_t box[3] = {64, 128, 1};
  const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.n, (uint64_t)a.BH};
  const uint64_t str[2] = {(uint64_t)D * 2, (uint64_t)a.n * D * 2};
  if ((e = make_tmap(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.Q, dims, str, box))) return e;
  if ((e = make_tmap(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.K, dims, str, box))) return e;
  if ((e = make_tmap(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.V, dims, str, box))) return e;
  if ((e = make_tmap(&mdo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.dO, dims, str, box))) return e;
  BwdParams p;
  p.BH = a.BH;
  p.n = a.n;
  p.nqb = (a.n + BM - 1) / BM;
  p.causal = a.causal;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.LSE = a.LSE;
  p.Dvec = a.Dvec;
  p.dq_acc = a.dq_acc;
  p.dK = static_cast<__nv_bfloat16 *>(a.dK);
  p.dV = static_cast<__nv_bfloat16 *>(a.dV);
  p.wc = wc;
  auto kern = attn_bwd_kernel<D>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC)))
    return e;
  timing_mark_start(st);
  kern<<<(unsigned)(p.nqb * a.BH), NTHREADS, L::ALLOC, st>>>(mq, mk, mv, mdo, p);
  timing_mark_stop(st);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  {
    const int64_t n8 = rows * D / 8;
    int64_t grid = (n8 + 255) / 256;
    if (grid > 152 * 16) grid = 152 * 16;
    bwd_dq_cvt_kernel<<<(unsigned)grid, 256, 0, st>>>(a.dq_acc, static_cast<__nv_bfloat16 *>(a.dQ),
                                                      n8);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_attn_bwd(const AttnBwdArgs &a, const WaitCfg &wc, cudaStream_t st) {
  if (a.d == 128) return launch_bwd_d<128>(a, wc, st);
  if (a.d == 64) return launch_bwd_d<64>(a, wc, st);
  return cudaErrorInvalidValue;
}

}  // namespace chain
