// attn_fwd.cu -- softmax attention forward, O = softmax(scale Q K^T) V, bf16.
//
// The unit O = f(AB)C of "Memory-efficient tensor parallelism" (FITEE
// 10.1631/FITEE.2400602, abstract) with f = row softmax, computed the way
// the Ulysses write-up ("Contexte Technique") describes FlashAttention:
// tile by tile, never storing the n x n score matrix.  Causal masking keeps
// keys j <= i on global positions (AutoSP, section 2.A item 4).
//
// One CTA per (head, 128-row query block), heaviest causal blocks first.
// Warp roles (192 threads):
//   warps 0-3  softmax: thread t owns query row t of the block.  Reads its
//              row of S from tensor memory, runs the online softmax in fp32
//              registers, and writes P as two bf16 tiles, P_hi = bf16(P)
//              (round-to-nearest-even) and P_lo = bf16(P - P_hi), into
//              128-byte-swizzled shared memory; O accumulates P_hi V + P_lo V,
//              so rounding the intermediate costs ~2^-16 relative instead of
//              2^-9 and the only bf16 rounding left is the output's.  It
//              rescales O in tensor memory when its running max grew by more
//              than 2^8, and finally writes O / l (bf16) and LSE.
//   warp 4     TMA producer: Q once, then K_j and V_j into a 2-stage ring
//              (the on-chip form of METP's double buffer).
//   warp 5     MMA issuer: S_j = Q K_j^T into one of two tensor-memory S
//              buffers, then O += (P_hi + P_lo)_{j-1} V_{j-1}; completion is signalled
//              with tcgen05.commit onto mbarriers.
// Tensor memory: S0 [0,128), S1 [128,256), O [256, 256+d).
#include "internal.h"

namespace chain {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int STAGES = 2;
constexpr int NTHREADS = 192;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units

template <int D>
struct FwdLayout {
  static constexpr uint32_t Q_BYTES = BM * D * 2;
  static constexpr uint32_t KV_BYTES = BN * D * 2;
  static constexpr uint32_t P_TILE = BM * BN * 2;  // one bf16 [128][128] tile
  static constexpr uint32_t P_BYTES = 2 * P_TILE;    // P_hi, P_lo
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr uint32_t OFF_P = OFF_V + STAGES * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_P + P_BYTES;
  static constexpr uint32_t NBAR = 1 + 3 * STAGES + 2 + 2 + 1 + 1 + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  // Dynamic shared memory requested: the layout plus slack to align the
  // base to 1024 bytes, and at least enough to keep one CTA per SM (the
  // kernel allocates all 512 tensor-memory columns).
  static constexpr uint32_t ALLOC = (BYTES + 1024 > 120 * 1024) ? BYTES + 1024 : 120 * 1024;
};

struct FwdParams {
  int BH, n, nqb, nkb, causal;
  float scale_log2;
  __nv_bfloat16 *O;
  int64_t o_sbh, o_srow;
  float *LSE;
  int64_t lse_sbh;
  WaitCfg wc;
};

enum : int {
  SITE_FWD_PROD = 0x101,
  SITE_FWD_MMA = 0x102,
  SITE_FWD_SOFTMAX = 0x103,
  SITE_FWD_EPI = 0x104,
  SITE_FWD_DRAIN = 0x105
};

// Wait that ignores the abort flag: used while draining in-flight copies
// and MMAs before the CTA releases its memory.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, const WaitCfg &wc) {
  volatile int never = 0;
  mbar_wait(bar, parity, wc, &never, SITE_FWD_DRAIN);
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using L = FwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
  uint64_t *q_full = bars;
  uint64_t *k_full = bars + 1;
  uint64_t *v_full = k_full + STAGES;
  uint64_t *kv_empty = v_full + STAGES;
  uint64_t *s_full = kv_empty + STAGES;
  uint64_t *s_free = s_full + 2;
  uint64_t *p_full = s_free + 2;
  uint64_t *pv_done = p_full + 1;
  uint64_t *mma_drain = pv_done + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int blk = blockIdx.x;
  const int qb = p.causal ? (p.nqb - 1 - blk / p.BH) : (blk / p.BH);
  const int bh = blk % p.BH;
  const int nkv = p.causal ? (qb + 1) : p.nkb;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], 128);
    }
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      mbar_arrive_expect_tx(q_full, L::Q_BYTES);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(smem + L::OFF_Q + c * (BM * 128), &tmQ, q_full, c * 64, qb * BM, bh);
      for (int j = 0; j < nkv; ++j) {
        const int st = j % STAGES;
        if (j >= STAGES &&
            !mbar_wait(&kv_empty[st], ((j / STAGES) - 1) & 1, p.wc, abort_flag, SITE_FWD_PROD))
          break;
        mbar_arrive_expect_tx(&k_full[st], L::KV_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::OFF_K + st * L::KV_BYTES + c * (BN * 128), &tmK, &k_full[st],
                      c * 64, j * BN, bh);
        mbar_arrive_expect_tx(&v_full[st], L::KV_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::OFF_V + st * L::KV_BYTES + c * (BN * 128), &tmV, &v_full[st],
                      c * 64, j * BN, bh);
        issued = j + 1;
      }
      if (*abort_flag) {
        // Let every copy still in flight land before shared memory is freed.
        drain_wait(q_full, 0, p.wc);
        for (int j = (issued > STAGES ? issued - STAGES : 0); j < issued; ++j) {
          drain_wait(&k_full[j % STAGES], (j / STAGES) & 1, p.wc);
          drain_wait(&v_full[j % STAGES], (j / STAGES) & 1, p.wc);
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(BM, BN, 0, 0);
      const uint32_t idO = idesc_bf16_f32(BM, D, 0, 1);
      const uint32_t sQ = smem_u32(smem + L::OFF_Q);
      const uint32_t sK = smem_u32(smem + L::OFF_K);
      const uint32_t sV = smem_u32(smem + L::OFF_V);
      const uint32_t sP = smem_u32(smem + L::OFF_P);
      if (mbar_wait(q_full, 0, p.wc, abort_flag, SITE_FWD_MMA)) {
        for (int j = 0; j <= nkv; ++j) {
          if (j < nkv) {
            const int st = j % STAGES, sb = j & 1;
            if (!mbar_wait(&k_full[st], (j / STAGES) & 1, p.wc, abort_flag, SITE_FWD_MMA)) break;
            if (j >= 2 &&
                !mbar_wait(&s_free[sb], ((j >> 1) - 1) & 1, p.wc, abort_flag, SITE_FWD_MMA))
              break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
              const uint64_t a = sdesc_sw128(sQ + off, 16, 1024);
              const uint64_t b =
                  sdesc_sw128(sK + st * L::KV_BYTES + (kk >> 2) * (BN * 128) + (kk & 3) * 32, 16,
                              1024);
              umma_f16_ss(tmem + sb * BN, a, b, idS, kk > 0 ? 1u : 0u);
            }
            umma_commit(&s_full[sb]);
          }
          if (j >= 1) {
            const int jp = j - 1, st = jp % STAGES;
            if (!mbar_wait(p_full, jp & 1, p.wc, abort_flag, SITE_FWD_MMA)) break;
            if (!mbar_wait(&v_full[st], (jp / STAGES) & 1, p.wc, abort_flag, SITE_FWD_MMA))
              break;
            tc_fence_after();
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
              for (int kk = 0; kk < BN / 16; ++kk) {
                const uint64_t a = sdesc_sw128(
                    sP + part * L::P_TILE + (kk >> 2) * (BM * 128) + (kk & 3) * 32, 16, 1024);
                const uint64_t b =
                    sdesc_sw128(sV + st * L::KV_BYTES + kk * 2048, BN * 128, 1024);
                umma_f16_ss(tmem + 2 * BN, a, b, idO, (jp > 0 || part > 0 || kk > 0) ? 1u : 0u);
              }
            umma_commit(pv_done);
            umma_commit(&kv_empty[st]);
          }
        }
      }
      // No MMA may still be running when tensor memory is released.
      umma_commit(mma_drain);
      drain_wait(mma_drain, 0, p.wc);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int row = threadIdx.x;  // 0..127, TMEM lane = row
    const int q_idx = qb * BM + row;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int sb = j & 1;
      if (!mbar_wait(&s_full[sb], (j >> 1) & 1, p.wc, abort_flag, SITE_FWD_SOFTMAX)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
        tmem_ld32(tmem + lane_off + sb * BN + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&s_free[sb]);

      const int kv0 = j * BN;
      const bool diag = p.causal && (j == qb);
      const bool tail = (kv0 + BN > p.n);
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < BN; ++c) {
        float v = __uint_as_float(s[c]) * p.scale_log2;
        if ((diag && kv0 + c > q_idx) || (tail && kv0 + c >= p.n)) v = -INFINITY;
        s[c] = __float_as_uint(v);
        mx = fmaxf(mx, v);
      }
      float alpha = 1.0f;
      bool rescale = false;
      if (j == 0) {
        m = mx;
      } else if (mx > m + RESCALE_THRESHOLD) {
        alpha = ex2(m - mx);
        m = mx;
        rescale = true;
      }
      const float mref = (m == -INFINITY) ? 0.0f : m;
      float rs = 0.0f;
      uint32_t pk[BN / 2], pl[BN / 2];
#pragma unroll
      for (int c = 0; c < BN; c += 2) {
        const float p0 = ex2(__uint_as_float(s[c]) - mref);
        const float p1 = ex2(__uint_as_float(s[c + 1]) - mref);
        rs += p0 + p1;
        const uint32_t h = pack_bf16(p0, p1);
        pk[c / 2] = h;
        pl[c / 2] = pack_bf16(p0 - __uint_as_float(h << 16), p1 - __uint_as_float(h & 0xffff0000u));
      }
      l = l * alpha + rs;

      if (j > 0) {
        if (!mbar_wait(pv_done, (j - 1) & 1, p.wc, abort_flag, SITE_FWD_SOFTMAX)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            const uint32_t ta = tmem + lane_off + 2 * BN + c * 32;
            tmem_ld32(ta, o);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            tmem_st32(ta, o);
          }
          tmem_wait_st();
        }
      }
      // P into the 128-byte-swizzled K-major tile: half h holds keys
      // [64h, 64h+64) of every row, 8 chunks of 16 bytes per row.
      const uint32_t sP = smem_u32(smem + L::OFF_P);
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const int b = h * 32 + ch * 4;
          const uint32_t off = h * (BM * 128) + sw128_off(row, ch);
          st_shared_v4(sP + off, pk[b], pk[b + 1], pk[b + 2], pk[b + 3]);
          st_shared_v4(sP + L::P_TILE + off, pl[b], pl[b + 1], pl[b + 2], pl[b + 3]);
        }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    // ----------------------------------------------------------- epilogue
    if (ok && mbar_wait(pv_done, (nkv - 1) & 1, p.wc, abort_flag, SITE_FWD_EPI)) {
      tc_fence_after();
      const float inv_l = 1.0f / l;
      __nv_bfloat16 *orow = p.O + (int64_t)bh * p.o_sbh + (int64_t)q_idx * p.o_srow;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + 2 * BN + c * 32, o);
        tmem_wait_ld();
        if (q_idx < p.n) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(o[8 * k + 0]) * inv_l, __uint_as_float(o[8 * k + 1]) * inv_l);
            v.y = pack_bf16(__uint_as_float(o[8 * k + 2]) * inv_l, __uint_as_float(o[8 * k + 3]) * inv_l);
            v.z = pack_bf16(__uint_as_float(o[8 * k + 4]) * inv_l, __uint_as_float(o[8 * k + 5]) * inv_l);
            v.w = pack_bf16(__uint_as_float(o[8 * k + 6]) * inv_l, __uint_as_float(o[8 * k + 7]) * inv_l);
            dst[k] = v;
          }
        }
      }
      if (q_idx < p.n)
        p.LSE[(int64_t)bh * p.lse_sbh + q_idx] = (m + lg2(l)) * 0.69314718055994531f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_fwd_d(const AttnFwdArgs &a, const WaitCfg &wc, cudaStream_t st) {
  using L = FwdLayout<D>;
  CUtensorMap mq, mk, mv;
  const uint32_t box[3] = {64, 128, 1};
  const uint64_t dims[3] = {(uint64_t)a.d, (uint64_t)a.n, (uint64_t)a.BH};
  uint64_t sq[2] = {(uint64_t)a.q_srow * 2, (uint64_t)a.q_sbh * 2};
  uint64_t sk[2] = {(uint64_t)a.k_srow * 2, (uint64_t)a.k_sbh * 2};
  uint64_t sv[2] = {(uint64_t)a.v_srow * 2, (uint64_t)a.v_sbh * 2};
  cudaError_t e;
  if ((e = make_tmap(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.Q, dims, sq, box)) != cudaSuccess)
    return e;
  if ((e = make_tmap(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.K, dims, sk, box)) != cudaSuccess)
    return e;
  if ((e = make_tmap(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.V, dims, sv, box)) != cudaSuccess)
    return e;
  FwdParams p;
  p.BH = a.BH;
  p.n = a.n;
  p.nqb = (a.n + BM - 1) / BM;
  p.nkb = (a.n + BN - 1) / BN;
  p.causal = a.causal;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.O = static_cast<__nv_bfloat16 *>(a.O);
  p.o_sbh = a.o_sbh;
  p.o_srow = a.o_srow;
  p.LSE = a.LSE;
  p.lse_sbh = a.lse_sbh;
  p.wc = wc;
  auto kern = attn_fwd_kernel<D>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(p.nqb * a.BH);
  timing_mark_start(st);
  kern<<<grid, NTHREADS, L::ALLOC, st>>>(mq, mk, mv, p);
  timing_mark_stop(st);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd_bf16(const AttnFwdArgs &a, const WaitCfg &wc, cudaStream_t st) {
  if (a.d == 128) return launch_fwd_d<128>(a, wc, st);
  if (a.d == 64) return launch_fwd_d<64>(a, wc, st);
  return cudaErrorInvalidValue;
}

}  // namespace chain
