// attn_fwd_f32.cu -- softmax attention forward for fp32 inputs and output,
// O = softmax(scale Q K^T) V with d = 64 (the small full-precision
// instance of the unit O = f(AB)C, "Memory-efficient tensor parallelism",
// FITEE 10.1631/FITEE.2400602, abstract).
//
// Both products run on the tensor cores as kind::tf32 MMAs with every
// operand split into a tf32 head and an fp32 remainder, x = x_hi + x_lo
// (x_hi keeps the 10 mantissa bits the tensor core reads, x_lo = x - x_hi
// is exact), and a.b ~ a_hi.b_hi + a_hi.b_lo + a_lo.b_hi.  The dropped
// a_lo.b_lo term is ~2^-22 relative, so the result carries fp32 accuracy
// rather than tf32's.
//
// One CTA (128 threads) per (head, 128-row query block).  The work is
// small, so the structure is synchronous: per 64-key tile the threads load
// K and V with plain vector loads, split them into hi/lo tiles (V stored
// transposed so that every MMA operand is K-major), thread 0 issues the
// MMAs, and thread t runs the online softmax of query row t.
#include "internal.h"

namespace chain {
namespace {

constexpr int BM = 128;  // query rows per CTA
constexpr int BN = 64;   // keys per tile
constexpr int D = 64;    // head dimension
constexpr int NT = 128;

// K-major fp32 tiles: rows of 32 floats (128 bytes) per half, two halves.
constexpr uint32_t Q_HALF = BM * 128, K_HALF = BN * 128, VT_HALF = D * 128, P_HALF = BM * 128;
constexpr uint32_t OFF_QH = 0, OFF_QL = OFF_QH + 2 * Q_HALF;
constexpr uint32_t OFF_KH = OFF_QL + 2 * Q_HALF, OFF_KL = OFF_KH + 2 * K_HALF;
constexpr uint32_t OFF_VH = OFF_KL + 2 * K_HALF, OFF_VL = OFF_VH + 2 * VT_HALF;
constexpr uint32_t OFF_PH = OFF_VL + 2 * VT_HALF, OFF_PL = OFF_PH + 2 * P_HALF;
constexpr uint32_t OFF_BAR = OFF_PL + 2 * P_HALF;
constexpr uint32_t SMEM_BYTES = OFF_BAR + 64;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;

struct F32Params {
  const float *Q, *K, *V;
  int64_t q_sbh, q_srow, k_sbh, k_srow, v_sbh, v_srow;
  float *O;
  int64_t o_sbh, o_srow;
  float *LSE;
  int64_t lse_sbh;
  int BH, n, nqb, causal;
  float scale_log2;
  WaitCfg wc;
};

enum : int { SITE_F32_MMA = 0x401 };

__device__ __forceinline__ float tf32_head(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xffffe000u);
}

// byte offset of element (r, c) of a K-major fp32 tile with 128-byte rows
// per 32-column half (half stride hs)
__device__ __forceinline__ uint32_t kmaj_off(uint32_t r, uint32_t c, uint32_t hs) {
  return (c >> 5) * hs + sw128_off(r, (c & 31) >> 2) + (c & 3) * 4;
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Three-term product D (+)= Ah Bh + Ah Bl + Al Bh over K = 64 (8 steps of 8).
__device__ __forceinline__ void mma3(uint32_t d, uint32_t ah, uint32_t al, uint32_t a_hs,
                                     uint32_t bh, uint32_t bl, uint32_t b_hs, uint32_t idesc,
                                     bool accumulate) {
  const uint32_t as[3] = {ah, ah, al}, bs[3] = {bh, bl, bh};
#pragma unroll
  for (int t = 0; t < 3; ++t)
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint64_t a = sdesc_sw128(as[t] + (kk >> 2) * a_hs + (kk & 3) * 32, 16, 1024);
      const uint64_t b = sdesc_sw128(bs[t] + (kk >> 2) * b_hs + (kk & 3) * 32, 16, 1024);
      umma_tf32_ss(d, a, b, idesc, (accumulate || t > 0 || kk > 0) ? 1u : 0u);
    }
}

__global__ void __launch_bounds__(NT, 1) attn_fwd_f32_kernel(const F32Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_BAR + 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_BAR + 12);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int qb = p.causal ? (p.nqb - 1 - (int)blockIdx.x / p.BH) : ((int)blockIdx.x / p.BH);
  const int bh = blockIdx.x % p.BH;
  const int q_idx = qb * BM + tid;
  const int nkv_tiles = p.causal ? ((qb + 1) * BM + BN - 1) / BN : (p.n + BN - 1) / BN;
  const int nkv = min(nkv_tiles, (p.n + BN - 1) / BN);

  if (tid == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  // Q tile -> hi/lo (rows beyond n are zero)
  for (int i = tid; i < BM * D / 4; i += NT) {
    const int r = i / (D / 4), c = (i % (D / 4)) * 4;
    const int q = qb * BM + r;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (q < p.n) x = *reinterpret_cast<const float4 *>(p.Q + bh * p.q_sbh + (int64_t)q * p.q_srow + c);
    const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float h = tf32_head(xs[u]);
      st_shared_f32(sb + OFF_QH + kmaj_off(r, c + u, Q_HALF), h);
      st_shared_f32(sb + OFF_QL + kmaj_off(r, c + u, Q_HALF), xs[u] - h);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 64;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t id = idesc_tf32_f32(BM, 64, 0, 0);
  float m = -INFINITY, l = 0.0f;
  uint32_t phase = 0;
  bool ok = true;

  for (int j = 0; j < nkv && ok; ++j) {
    const int kv0 = j * BN;
    // K -> K-major hi/lo; V -> transposed (d rows, key columns) hi/lo
    for (int i = tid; i < BN * D / 4; i += NT) {
      const int r = i / (D / 4), c = (i % (D / 4)) * 4;
      const int kv = kv0 + r;
      float4 kx = make_float4(0.f, 0.f, 0.f, 0.f), vx = kx;
      if (kv < p.n) {
        kx = *reinterpret_cast<const float4 *>(p.K + bh * p.k_sbh + (int64_t)kv * p.k_srow + c);
        vx = *reinterpret_cast<const float4 *>(p.V + bh * p.v_sbh + (int64_t)kv * p.v_srow + c);
      }
      const float ks[4] = {kx.x, kx.y, kx.z, kx.w}, vs[4] = {vx.x, vx.y, vx.z, vx.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float kh = tf32_head(ks[u]), vh = tf32_head(vs[u]);
        st_shared_f32(sb + OFF_KH + kmaj_off(r, c + u, K_HALF), kh);
        st_shared_f32(sb + OFF_KL + kmaj_off(r, c + u, K_HALF), ks[u] - kh);
        st_shared_f32(sb + OFF_VH + kmaj_off(c + u, r, VT_HALF), vh);
        st_shared_f32(sb + OFF_VL + kmaj_off(c + u, r, VT_HALF), vs[u] - vh);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      mma3(tS, sb + OFF_QH, sb + OFF_QL, Q_HALF, sb + OFF_KH, sb + OFF_KL, K_HALF, id, false);
      umma_commit(bar);
    }
    __syncwarp();
    if (!mbar_wait(bar, phase, p.wc, abort_flag, SITE_F32_MMA)) ok = false;
    phase ^= 1;
    tc_fence_after();
    uint32_t s[64];
    tmem_ld32(tS + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
    tmem_ld32(tS + lane_off + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
    tmem_wait_ld();
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < BN; ++c) {
      const int kv = kv0 + c;
      float v = __uint_as_float(s[c]) * p.scale_log2;
      if (kv >= p.n || (p.causal && kv > q_idx)) v = -INFINITY;
      s[c] = __float_as_uint(v);
      mx = fmaxf(mx, v);
    }
    const float m_new = fmaxf(m, mx);
    const float mref = (m_new == -INFINITY) ? 0.0f : m_new;
    const float alpha = (m == -INFINITY) ? 0.0f : ex2(m - mref);
    m = m_new;
    float rs = 0.0f;
#pragma unroll
    for (int c = 0; c < BN; ++c) {
      const float pv = ex2(__uint_as_float(s[c]) - mref);
      rs += pv;
      const float ph = tf32_head(pv);
      st_shared_f32(sb + OFF_PH + kmaj_off(tid, c, P_HALF), ph);
      st_shared_f32(sb + OFF_PL + kmaj_off(tid, c, P_HALF), pv - ph);
    }
    l = l * alpha + rs;
    if (j > 0) {
      uint32_t o[32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        tmem_ld32(tO + lane_off + h * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
        tmem_st32(tO + lane_off + h * 32, o);
      }
      tmem_wait_st();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      mma3(tO, sb + OFF_PH, sb + OFF_PL, P_HALF, sb + OFF_VH, sb + OFF_VL, VT_HALF, id, j > 0);
      umma_commit(bar);
    }
    __syncwarp();
    if (!mbar_wait(bar, phase, p.wc, abort_flag, SITE_F32_MMA)) ok = false;
    phase ^= 1;
    tc_fence_after();
    __syncthreads();  // smem tiles are rewritten by the next iteration
  }
  if (ok) {
    uint32_t o[32];
    const float inv_l = 1.0f / l;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      tmem_ld32(tO + lane_off + h * 32, o);
      tmem_wait_ld();
      if (q_idx < p.n) {
        float4 *dst = reinterpret_cast<float4 *>(p.O + bh * p.o_sbh + (int64_t)q_idx * p.o_srow + h * 32);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          dst[k] = make_float4(__uint_as_float(o[4 * k]) * inv_l, __uint_as_float(o[4 * k + 1]) * inv_l,
                               __uint_as_float(o[4 * k + 2]) * inv_l, __uint_as_float(o[4 * k + 3]) * inv_l);
      }
    }
    if (q_idx < p.n) p.LSE[bh * p.lse_sbh + q_idx] = (m + lg2(l)) * 0.69314718055994531f;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

}  // namespace

cudaError_t launch_attn_fwd_f32(const AttnFwdArgs &a, const WaitCfg &wc, cudaStream_t st) {
  if (a.d != D) return cudaErrorNotSupported;
  F32Params p;
  p.Q = static_cast<const float *>(a.Q);
  p.K = static_cast<const float *>(a.K);
  p.V = static_cast<const float *>(a.V);
  p.q_sbh = a.q_sbh; p.q_srow = a.q_srow;
  p.k_sbh = a.k_sbh; p.k_srow = a.k_srow;
  p.v_sbh = a.v_sbh; p.v_srow = a.v_srow;
  p.O = static_cast<float *>(a.O);
  p.o_sbh = a.o_sbh; p.o_srow = a.o_srow;
  p.LSE = a.LSE;
  p.lse_sbh = a.lse_sbh;
  p.BH = a.BH;
  p.n = a.n;
  p.nqb = (a.n + BM - 1) / BM;
  p.causal = a.causal;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.wc = wc;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_f32_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  timing_mark(st, 0);
  attn_fwd_f32_kernel<<<(unsigned)(p.nqb * a.BH), NT, SMEM_ALLOC, st>>>(p);
  timing_mark(st, 1);
  return cudaGetLastError();
}

}  // namespace chain
