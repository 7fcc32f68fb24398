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
// Three kernels, no atomics, deterministic:
//   bwd_prep   D_i = sum_e dO_ie O_ie (fp32), into the workspace;
//   bwd_dkdv   one CTA per (head, 128-key block j), looping over the query
//              tiles i that see block j (i >= j when causal):
//                S^T = K_j Q_i^T,  dP^T = V_j dO_i^T      (tensor memory)
//                P^T as a bf16 tile in shared memory, which frees the S^T
//                columns for S^T of the next tile at once;
//                dS^T written back as bf16 over the dP^T columns
//                dV += P^T dO_i (shared A),  dK += dS^T Q_i (tensor-memory A)
//   bwd_dq     one CTA per (head, 128-query tile i), looping over the key
//              tiles j <= i; Q_i and dO_i stay in tensor memory as the A
//              operand of
//                S = Q_i K_j^T,  dP = dO_i V_j^T
//                dS written back as bf16 over the dP columns
//                dQ += dS K_j                               (A from tensor memory)
// bwd_dq recomputes S and dP, 7 products per tile pair instead of 5, in
// exchange for accumulating dQ on chip instead of adding 128 x 128 fp32
// partials per tile pair into global memory.
//
// Roles (320 threads) in both main kernels: warps 0-7 compute, two
// warpgroups splitting the 128 columns of each tile (warpgroup w takes
// columns [64w, 64w+64); thread r owns row r = tensor-memory lane r); warp 8
// TMA producer; warp 9 MMA issuer.  A warpgroup writes the bf16 result of a
// 64-column half into the first 32 columns of that half, which it alone has
// read, so the two warpgroups never overwrite each other's inputs.  The
// MMAs of one thread execute in issue order, so an MMA that overwrites a
// tensor-memory region is issued after the MMAs that read it, and its
// completion tells the compute warps the old contents are consumed.
#include "internal.h"

namespace chain {
namespace {

constexpr int BM = 128;  // rows per tile (keys and queries)
constexpr int NTHREADS = 320;

template <int D>
struct BwdLayout {
  static constexpr uint32_t T_BYTES = BM * D * 2;  // one [128][D] bf16 tile
  // bwd_dkdv: K_j, V_j, Q (2 stages), dO (2 stages), P^T
  static constexpr uint32_t A_K = 0;
  static constexpr uint32_t A_V = A_K + T_BYTES;
  static constexpr uint32_t A_Q = A_V + T_BYTES;
  static constexpr uint32_t A_DO = A_Q + 2 * T_BYTES;
  static constexpr uint32_t A_PT = A_DO + 2 * T_BYTES;  // P^T [128 keys][128 queries] bf16
  static constexpr uint32_t A_LD = A_PT + BM * BM * 2;  // LSE/D staging [2 wg][64] x2
  static constexpr uint32_t A_BAR = A_LD + 1024;
  // bwd_dq: K, V (3 stages each); Q_i, dO_i live in tensor memory
  static constexpr uint32_t B_K = 0;
  static constexpr uint32_t B_V = B_K + 3 * T_BYTES;
  static constexpr uint32_t B_BAR = B_V + 3 * T_BYTES;
  static constexpr uint32_t NBAR = 20;
  static constexpr uint32_t A_MISC = A_BAR + NBAR * 8;
  static constexpr uint32_t B_MISC = B_BAR + NBAR * 8;
  static constexpr uint32_t A_ALLOC =
      (A_MISC + 16 + 1024 > 120 * 1024) ? A_MISC + 16 + 1024 : 120 * 1024;
  static constexpr uint32_t B_ALLOC =
      (B_MISC + 16 + 1024 > 120 * 1024) ? B_MISC + 16 + 1024 : 120 * 1024;
};

struct BwdParams {
  int BH, n, nb, causal;
  int G;  // query heads per K/V head (grouped-query attention; 1 = none)
  // element strides: Q, O, dO, dQ rows / heads; K, V, dK, dV rows / heads;
  // LSE and D heads (their rows are contiguous)
  int64_t q_srow, q_shead, kv_srow, kv_shead, l_shead;
  // Variable-length batch (null cu when not): sequence b is rows
  // [cu[b], cu[b+1]) of the packed tensors; nb counts the blocks of the
  // longest sequence.
  const int *cu;
  int nbatch;
  float scale, scale_log2;
  const float *LSE;   // [BH][n]
  const float *Dvec;  // [BH][n]
  const __nv_bfloat16 *Q, *dO;
  __nv_bfloat16 *dQ, *dK, *dV;
  WaitCfg wc;
};

enum : int {
  SITE_BWD_PROD = 0x201,
  SITE_BWD_MMA = 0x202,
  SITE_BWD_COMPUTE = 0x203,
  SITE_BWD_EPI = 0x204,
  SITE_BWD_DRAIN = 0x205,
  SITE_DQ_PROD = 0x211,
  SITE_DQ_MMA = 0x212,
  SITE_DQ_COMPUTE = 0x213,
  SITE_DQ_EPI = 0x214
};

__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, const WaitCfg &wc) {
  volatile int never = 0;
  mbar_wait(bar, parity, wc, &never, SITE_BWD_DRAIN);
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                     ~static_cast<uintptr_t>(1023));
}

// NC fp32 accumulators of one row (tensor-memory columns from taddr) ->
// bf16 row in global memory, times mul.
template <int NC>
__device__ __forceinline__ void store_row_bf16(uint32_t taddr, __nv_bfloat16 *row, float mul,
                                               bool ok) {
#pragma unroll 1
  for (int c = 0; c < NC / 32; ++c) {
    uint32_t a[32];
    tmem_ld32(taddr + c * 32, a);
    tmem_wait_ld();
    if (ok) {
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

// One sequence of a variable-length batch: bounds clamped to the packed rows
// so a bad cu can never address memory outside the tensors.
__device__ __forceinline__ void seq_bounds(const BwdParams &p, int b, int &row0, int &n) {
  int lo = __ldg(p.cu + b), hi = __ldg(p.cu + b + 1);
  lo = lo < 0 ? 0 : (lo > p.n ? p.n : lo);
  hi = hi < lo ? lo : (hi > p.n ? p.n : hi);
  row0 = lo;
  n = hi - lo;
}

// ------------------------------------------------------------ preprocess
// 16 threads per row of d = 128 (8 per row of d = 64): each loads 16 bytes
// of O and dO; the partial dot products are reduced with shuffles.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16 *__restrict__ O,
                                                       const __nv_bfloat16 *__restrict__ dO,
                                                       float *__restrict__ Dvec, int64_t rows,
                                                       int n, int64_t srow, int64_t shead,
                                                       int64_t l_shead) {
  constexpr int TPR = D / 8;  // threads per row
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = tid / TPR;  // head row / n, position row % n
  const int part = (int)(tid % TPR);
  const int64_t h = row / n, t = row % n;
  const int64_t off = h * shead + t * srow + part * 8;
  float acc = 0.0f;
  if (row < rows) {
    const uint4 a = *reinterpret_cast<const uint4 *>(O + off);
    const uint4 b = *reinterpret_cast<const uint4 *>(dO + off);
    const __nv_bfloat162 *pa = reinterpret_cast<const __nv_bfloat162 *>(&a);
    const __nv_bfloat162 *pb = reinterpret_cast<const __nv_bfloat162 *>(&b);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 fa = __bfloat1622float2(pa[k]);
      const float2 fb = __bfloat1622float2(pb[k]);
      acc = fmaf(fa.x, fb.x, acc);
      acc = fmaf(fa.y, fb.y, acc);
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && part == 0) Dvec[h * l_shead + t] = acc;
}

// ------------------------------------------------------- dK, dV kernel
template <int D, bool VARLEN>
__global__ void __launch_bounds__(NTHREADS, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmdO, const BwdParams p) {
  using L = BwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::A_BAR);
  uint64_t *kv_full = bars + 0;
  uint64_t *q_full = bars + 1;    // [2]
  uint64_t *q_empty = bars + 3;   // [2]
  uint64_t *do_full = bars + 5;   // [2]
  uint64_t *do_empty = bars + 7;  // [2]
  uint64_t *s_full = bars + 9;
  uint64_t *dp_full = bars + 10;
  uint64_t *p_ready = bars + 11;  // P^T in shared memory, dS^T in tensor memory (256 arrivals)
  uint64_t *fin = bars + 12;
  uint64_t *mma_drain = bars + 13;
  uint64_t *s_free = bars + 14;   // S^T read into registers (256 arrivals)
  uint64_t *pt_free = bars + 15;  // dV MMA done with the P^T tile
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::A_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::A_MISC + 4);
  float *sL = reinterpret_cast<float *>(smem + L::A_LD);  // [wg][64], LSE in log2 units
  float *sDv = sL + 2 * 64;                                // [wg][64]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // head-major order: the key blocks of one K/V head run together and share
  // Q, dO, LSE and D through L2; smallest (heaviest causal) block first.
  // Tile t covers query tile i_begin + t % Tq of query head bkv*G + t / Tq
  // (Tq = nb - i_begin):
  // with grouped-query attention dK and dV sum over the group's heads.
  int bkv, jb, n = p.n, nb = p.nb, row0 = 0;
  if constexpr (!VARLEN) {
    bkv = blockIdx.x / p.nb;
    jb = blockIdx.x % p.nb;
  } else {
    // Within a K/V head, key blocks run in decreasing work over all of the
    // batch's sequences: causal key block jb meets nb - jb query tiles, so
    // blocks go by that count, largest first (without a mask, the longest
    // sequences go first).
    const int per_head = p.nbatch * p.nb;
    bkv = blockIdx.x / per_head;
    const int qd = (blockIdx.x % per_head) / p.nbatch;
    seq_bounds(p, blockIdx.x % p.nbatch, row0, n);
    nb = (n + BM - 1) / BM;
    if (nb > p.nb) {  // longer than the stated maximum: reported, not computed
      if (qd == 0 && threadIdx.x == 0 && bkv == 0) atomicExch(&p.wc.status->reserved[0], 1);
      return;
    }
    const int jr = p.nb - 1 - qd;
    jb = p.causal ? nb - 1 - jr : jr;
    if (jb < 0 || jb >= nb) return;  // nothing of this sequence for this CTA
  }
  const int i_begin = p.causal ? jb : 0;
  const int T = (nb - i_begin) * p.G;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 16; ++b)
      mbar_init(&bars[b], (&bars[b] == p_ready || &bars[b] == s_free) ? 256u : 1u);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;

  if (warp == 8) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int q_issued = 0, do_issued = 0;
      mbar_arrive_expect_tx(kv_full, 2 * L::T_BYTES);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(smem + L::A_K + c * (BM * 128), &tmK, kv_full, c * 64, row0 + jb * BM, bkv);
        tma_load_3d(smem + L::A_V + c * (BM * 128), &tmV, kv_full, c * 64, row0 + jb * BM, bkv);
      }
      int i = i_begin, bh = bkv * p.G;  // query tile and head of tile t
      for (int t = 0; t < T; ++t, (++i == nb) ? (i = i_begin, ++bh) : 0) {
        const int s = t & 1;
        if (t >= 2 && !mbar_wait(&q_empty[s], ((t >> 1) - 1) & 1, p.wc, abort_flag, SITE_BWD_PROD))
          break;
        mbar_arrive_expect_tx(&q_full[s], L::T_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::A_Q + s * L::T_BYTES + c * (BM * 128), &tmQ, &q_full[s], c * 64,
                      row0 + i * BM, bh);
        q_issued = t + 1;
        if (t >= 2 && !mbar_wait(&do_empty[s], ((t >> 1) - 1) & 1, p.wc, abort_flag, SITE_BWD_PROD))
          break;
        mbar_arrive_expect_tx(&do_full[s], L::T_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::A_DO + s * L::T_BYTES + c * (BM * 128), &tmdO, &do_full[s], c * 64,
                      row0 + i * BM, bh);
        do_issued = t + 1;
      }
      if (*abort_flag) {
        drain_wait(kv_full, 0, p.wc);
        for (int t = (q_issued > 2 ? q_issued - 2 : 0); t < q_issued; ++t)
          drain_wait(&q_full[t & 1], (t >> 1) & 1, p.wc);
        for (int t = (do_issued > 2 ? do_issued - 2 : 0); t < do_issued; ++t)
          drain_wait(&do_full[t & 1], (t >> 1) & 1, p.wc);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // --------------------------------------------------------- MMA issuer
    // Per query tile t, in issue (= execution) order:
    //   S^T(t+1)                     once the warpgroups have read S^T(t)
    //   dK += dS^T(t) Q_t            A from tensor memory
    //   dV += P^T(t) dO_t            A from shared memory
    //   dP^T(t+1)                    over dS^T(t), after dK(t) read it
    // so the exponentials of tile t+1 overlap the products of tile t.  The
    // whole warp runs the loop; one elected lane issues each group and its
    // commits.
    {
      const uint32_t id_s = idesc_bf16_f32(BM, BM, 0, 0);  // S^T, dP^T
      const uint32_t id_kv = idesc_bf16_f32(BM, D, 0, 1);  // dV, dK (B MN-major)
      // base descriptors, built once (K-major operands, then MN-major views)
      const SDesc kK = sdesc_make(smem_u32(smem + L::A_K), 16, 1024);
      const SDesc kV = sdesc_make(smem_u32(smem + L::A_V), 16, 1024);
      const SDesc kP = sdesc_make(smem_u32(smem + L::A_PT), 16, 1024);
      const SDesc kQ0 = sdesc_make(smem_u32(smem + L::A_Q), 16, 1024);
      const SDesc kQ1 = sdesc_make(smem_u32(smem + L::A_Q + L::T_BYTES), 16, 1024);
      const SDesc kO0 = sdesc_make(smem_u32(smem + L::A_DO), 16, 1024);
      const SDesc kO1 = sdesc_make(smem_u32(smem + L::A_DO + L::T_BYTES), 16, 1024);
      const SDesc mQ0 = sdesc_make(smem_u32(smem + L::A_Q), BM * 128, 1024);
      const SDesc mQ1 = sdesc_make(smem_u32(smem + L::A_Q + L::T_BYTES), BM * 128, 1024);
      const SDesc mO0 = sdesc_make(smem_u32(smem + L::A_DO), BM * 128, 1024);
      const SDesc mO1 = sdesc_make(smem_u32(smem + L::A_DO + L::T_BYTES), BM * 128, 1024);
      auto issue_s = [&](int t) -> bool {  // S^T = K_j Q_t^T
        const int s = t & 1;
        if (!mbar_wait_warp(&q_full[s], (t >> 1) & 1, p.wc, abort_flag, SITE_BWD_MMA)) return false;
        tc_fence_after();
        const SDesc bq = s ? kQ1 : kQ0;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
            umma_f16_ss(tS, sdesc_at(kK, off), sdesc_at(bq, off), id_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(s_full);
        }
        __syncwarp();
        return true;
      };
      auto issue_dp = [&](int t) -> bool {  // dP^T = V_j dO_t^T
        const int s = t & 1;
        if (!mbar_wait_warp(&do_full[s], (t >> 1) & 1, p.wc, abort_flag, SITE_BWD_MMA)) return false;
        tc_fence_after();
        const SDesc bo = s ? kO1 : kO0;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
            umma_f16_ss(tdP, sdesc_at(kV, off), sdesc_at(bo, off), id_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(dp_full);
        }
        __syncwarp();
        return true;
      };
      bool ok = mbar_wait_warp(kv_full, 0, p.wc, abort_flag, SITE_BWD_MMA) &&
                (T == 0 || (issue_s(0) && issue_dp(0)));
      for (int t = 0; ok && t < T; ++t) {
        const int s = t & 1;
        if (t + 1 < T) {
          if (!mbar_wait_warp(s_free, t & 1, p.wc, abort_flag, SITE_BWD_MMA) || !issue_s(t + 1)) {
            ok = false;
            break;
          }
        }
        if (!mbar_wait_warp(p_ready, t & 1, p.wc, abort_flag, SITE_BWD_MMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // dS^T of queries [64w, 64w+64) sits packed in columns [64w, 64w+32)
        // of the dP^T region
        const SDesc bq = s ? mQ1 : mQ0;
        const SDesc bo = s ? mO1 : mO0;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            umma_f16_ts(tdK, tdP + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_at(bq, kk * 2048), id_kv,
                        (t > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&q_empty[s]);
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            umma_f16_ss(tdV, sdesc_at(kP, (kk >> 2) * (BM * 128) + (kk & 3) * 32),
                        sdesc_at(bo, kk * 2048), id_kv, (t > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&do_empty[s]);
          umma_commit(pt_free);
        }
        __syncwarp();
        if (t + 1 < T && !issue_dp(t + 1)) {
          ok = false;
          break;
        }
      }
      if (elect_one()) {
        if (ok) umma_commit(fin);
        umma_commit(mma_drain);
      }
      __syncwarp();
      if (lane == 0) drain_wait(mma_drain, 0, p.wc);
    }
    __syncwarp();
  } else {
    // --------------------------------------------- compute (two warpgroups)
    // Every warp of a warpgroup passes the same named barriers: after a
    // failed wait (ok false) the remaining waits are skipped, not the loop.
    const int w = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int kv_idx = jb * BM + r;
    const bool kv_ok = kv_idx < n;
    // P^T row r, queries [64w, 64w+64): 128 bytes of a 128B-swizzled tile
    const uint32_t pt_row = smem_u32(smem + L::A_PT + w * (BM * 128) + r * 128);
    float *wl = sL + w * 64;
    float *wd = sDv + w * 64;
    // LSE (log2 units) and D of query 64w + r of a tile (r < 64), fetched
    // one tile ahead
    auto fetch = [&](int i, int bh, float &lv, float &dv) {
      const int q = i * BM + 64 * w + r;
      const bool q_ok = r < 64 && q < n;
      const int64_t li = (int64_t)bh * p.l_shead + row0 + q;
      lv = q_ok ? __ldg(p.LSE + li) * 1.4426950408889634f : INFINITY;
      dv = q_ok ? __ldg(p.Dvec + li) : 0.0f;
    };
    float l_next = INFINITY, d_next = 0.0f;
    if (T > 0) fetch(i_begin, bkv * p.G, l_next, d_next);
    bool ok = true;
    int i = i_begin, bh = bkv * p.G;  // query tile and head of tile t
    for (int t = 0; t < T; ++t, (++i == nb) ? (i = i_begin, ++bh) : 0) {
      const bool diag = p.causal && (i == jb);
      if (t > 0) named_bar_sync(1 + w, 128);  // warpgroup done with the staged values of t-1
      if (r < 64) {
        wl[r] = l_next;
        wd[r] = d_next;
      }
      named_bar_sync(1 + w, 128);
      if (t + 1 < T) {
        const bool wrap = i + 1 == nb;
        fetch(wrap ? i_begin : i + 1, wrap ? bh + 1 : bh, l_next, d_next);
      }
      if (ok) ok = mbar_wait(s_full, t & 1, p.wc, abort_flag, SITE_BWD_COMPUTE);
      tc_fence_after();
      // P^T for queries [64w, 64w+64): fp32 exponentials; S^T is released
      // to the next product as soon as it sits in registers
      float pf[64];
      {
        uint32_t sv[64];
        tmem_ld32(tS + lane_off + 64 * w, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_ld32(tS + lane_off + 64 * w + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(s_free);
        const float4 *wl4 = reinterpret_cast<const float4 *>(wl);
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 lv = wl4[c4];
          const float ls[4] = {lv.x, lv.y, lv.z, lv.w};
#pragma unroll
          for (int u = 0; u < 4; ++u)
            pf[4 * c4 + u] = ex2(fmaf(__uint_as_float(sv[4 * c4 + u]), p.scale_log2, -ls[u]));
        }
        // key beyond n, or (diagonal tile) query before the key: one branch
        // around the whole pass, none in the loop above
        if (!kv_ok || diag) {
#pragma unroll
          for (int qq = 0; qq < 64; ++qq)
            if (!kv_ok || 64 * w + qq < r) pf[qq] = 0.0f;
        }
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) pk[c] = pack_bf16(pf[2 * c], pf[2 * c + 1]);
        // the dV product of tile t-1 still reads the P^T tile
        if (ok && t > 0) ok = mbar_wait(pt_free, (t - 1) & 1, p.wc, abort_flag, SITE_BWD_COMPUTE);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_shared_v4(pt_row + ((c ^ (r & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                       pk[4 * c + 3]);
        fence_proxy_async_smem();
      }
      if (ok) ok = mbar_wait(dp_full, t & 1, p.wc, abort_flag, SITE_BWD_COMPUTE);
      tc_fence_after();
      // dS^T = P^T o (dP^T - D) for the same queries, over the dP^T columns
      {
        uint32_t dp[64];
        tmem_ld32(tdP + lane_off + 64 * w, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
        tmem_ld32(tdP + lane_off + 64 * w + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
        tmem_wait_ld();
        const float4 *wd4 = reinterpret_cast<const float4 *>(wd);
        uint32_t dk[32];
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 dv = wd4[c4];
          const float ds[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int qq = 4 * c4 + 2 * h;
            dk[qq / 2] = pack_bf16(pf[qq] * (__uint_as_float(dp[qq]) - ds[2 * h]),
                                   pf[qq + 1] * (__uint_as_float(dp[qq + 1]) - ds[2 * h + 1]));
          }
        }
        tmem_st32(tdP + lane_off + 64 * w, dk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_ready);
    }
    // --------------------------------------------------- dK, dV epilogue
    if (ok && T > 0 && mbar_wait(fin, 0, p.wc, abort_flag, SITE_BWD_EPI)) {
      tc_fence_after();
      // warpgroup 0 writes dV, warpgroup 1 writes dK (times scale)
      __nv_bfloat16 *row =
          (w ? p.dK : p.dV) + (int64_t)bkv * p.kv_shead + (int64_t)(row0 + kv_idx) * p.kv_srow;
      store_row_bf16<D>((w ? tdK : tdV) + lane_off, row, w ? p.scale : 1.0f, kv_ok);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------ dQ kernel
// Q_i and dO_i are the same for every key tile of a CTA, so they sit in
// tensor memory as the A operand of S = Q_i K_j^T and dP = dO_i V_j^T: those
// products then read only K_j or V_j from shared memory.
template <int D, bool VARLEN>
__global__ void __launch_bounds__(NTHREADS, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const BwdParams p) {
  using L = BwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::B_BAR);
  uint64_t *k_full = bars + 0;    // [3]
  uint64_t *k_empty = bars + 3;   // [3]
  uint64_t *v_full = bars + 6;    // [3]
  uint64_t *v_empty = bars + 9;   // [3]
  uint64_t *qd_ready = bars + 12; // Q_i, dO_i in tensor memory (256 arrivals)
  uint64_t *s_full = bars + 13;
  uint64_t *s_free = bars + 14;   // S read into registers (256 arrivals)
  uint64_t *dp_full = bars + 15;
  uint64_t *p_ready = bars + 16;  // dS in tensor memory (256 arrivals)
  uint64_t *fin = bars + 17;
  uint64_t *mma_drain = bars + 18;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::B_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::B_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // head-major, heaviest (last) causal query tile first within a head
  int bh, ib, n = p.n, nb = p.nb, row0 = 0;
  if constexpr (!VARLEN) {
    bh = blockIdx.x / p.nb;
    ib = p.causal ? (p.nb - 1 - (int)(blockIdx.x % p.nb)) : (int)(blockIdx.x % p.nb);
  } else {
    // Within a head, query tiles run in decreasing position over all of the
    // batch's sequences: causal tile ib meets ib + 1 key blocks, so the
    // heaviest go first (without a mask, the longest sequences go first).
    const int per_head = p.nbatch * p.nb;
    bh = blockIdx.x / per_head;
    const int qd = (blockIdx.x % per_head) / p.nbatch;
    seq_bounds(p, blockIdx.x % p.nbatch, row0, n);
    nb = (n + BM - 1) / BM;
    if (nb > p.nb) return;  // longer than the stated maximum: reported by the dK, dV kernel
    ib = p.nb - 1 - qd;
    if (ib >= nb) return;  // nothing of this sequence for this CTA
  }
  const int NJ = p.causal ? ib + 1 : nb;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 19; ++b) {
      const bool wide = &bars[b] == qd_ready || &bars[b] == s_free || &bars[b] == p_ready;
      mbar_init(&bars[b], wide ? 256u : 1u);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // S [0,128), dP / dS [128,256), dQ [256, 256+D), Q_i and dO_i as packed
  // bf16 pairs (D/2 columns each) after it
  const uint32_t tS = tmem, tdP = tmem + 128, tdQ = tmem + 256;
  const uint32_t tQ = tmem + 256 + D, tdO = tmem + 256 + D + D / 2;

  if (warp == 8) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int k_issued = 0, v_issued = 0;
      const int bkv = bh / p.G;  // the group's K/V head
      for (int j = 0; j < NJ; ++j) {
        const int sk = j % 3;
        if (j >= 3 && !mbar_wait(&k_empty[sk], ((j / 3) - 1) & 1, p.wc, abort_flag, SITE_DQ_PROD))
          break;
        mbar_arrive_expect_tx(&k_full[sk], L::T_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::B_K + sk * L::T_BYTES + c * (BM * 128), &tmK, &k_full[sk], c * 64,
                      row0 + j * BM, bkv);
        k_issued = j + 1;
        if (j >= 3 && !mbar_wait(&v_empty[sk], ((j / 3) - 1) & 1, p.wc, abort_flag, SITE_DQ_PROD))
          break;
        mbar_arrive_expect_tx(&v_full[sk], L::T_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::B_V + sk * L::T_BYTES + c * (BM * 128), &tmV, &v_full[sk], c * 64,
                      row0 + j * BM, bkv);
        v_issued = j + 1;
      }
      if (*abort_flag) {
        for (int j = (k_issued > 3 ? k_issued - 3 : 0); j < k_issued; ++j)
          drain_wait(&k_full[j % 3], (j / 3) & 1, p.wc);
        for (int j = (v_issued > 3 ? v_issued - 3 : 0); j < v_issued; ++j)
          drain_wait(&v_full[j % 3], (j / 3) & 1, p.wc);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // --------------------------------------------------------- MMA issuer
    // Per key tile j, in issue (= execution) order:
    //   S(j+1)           once the warpgroups hold S(j) in registers
    //   dQ += dS(j) K_j  A from the dP columns
    //   dP(j+1)          over dS(j), after dQ(j) read it
    // The whole warp runs the loop; one elected lane issues each group and
    // its commits.
    {
      const uint32_t id_s = idesc_bf16_f32(BM, BM, 0, 0);  // S, dP (B K-major)
      const uint32_t id_q = idesc_bf16_f32(BM, D, 0, 1);   // dQ (B MN-major)
      const SDesc kK0 = sdesc_make(smem_u32(smem + L::B_K), 16, 1024);
      const SDesc kK1 = sdesc_make(smem_u32(smem + L::B_K + L::T_BYTES), 16, 1024);
      const SDesc kK2 = sdesc_make(smem_u32(smem + L::B_K + 2 * L::T_BYTES), 16, 1024);
      const SDesc kV0 = sdesc_make(smem_u32(smem + L::B_V), 16, 1024);
      const SDesc kV1 = sdesc_make(smem_u32(smem + L::B_V + L::T_BYTES), 16, 1024);
      const SDesc kV2 = sdesc_make(smem_u32(smem + L::B_V + 2 * L::T_BYTES), 16, 1024);
      const SDesc mK0 = sdesc_make(smem_u32(smem + L::B_K), BM * 128, 1024);
      const SDesc mK1 = sdesc_make(smem_u32(smem + L::B_K + L::T_BYTES), BM * 128, 1024);
      const SDesc mK2 = sdesc_make(smem_u32(smem + L::B_K + 2 * L::T_BYTES), BM * 128, 1024);
      auto issue_s = [&](int j) -> bool {  // S(j) = Q_i K_j^T
        const int sk = j % 3;
        if (!mbar_wait_warp(&k_full[sk], (j / 3) & 1, p.wc, abort_flag, SITE_DQ_MMA)) return false;
        tc_fence_after();
        const SDesc b = sk == 0 ? kK0 : (sk == 1 ? kK1 : kK2);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
            umma_f16_ts(tS, tQ + kk * 8, sdesc_at(b, off), id_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(s_full);
        }
        __syncwarp();
        return true;
      };
      auto issue_dp = [&](int j) -> bool {  // dP(j) = dO_i V_j^T
        const int sv = j % 3;
        if (!mbar_wait_warp(&v_full[sv], (j / 3) & 1, p.wc, abort_flag, SITE_DQ_MMA)) return false;
        tc_fence_after();
        const SDesc b = sv == 0 ? kV0 : (sv == 1 ? kV1 : kV2);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
            umma_f16_ts(tdP, tdO + kk * 8, sdesc_at(b, off), id_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(dp_full);
          umma_commit(&v_empty[sv]);  // V_j is read by dP(j) only
        }
        __syncwarp();
        return true;
      };
      bool ok = mbar_wait_warp(qd_ready, 0, p.wc, abort_flag, SITE_DQ_MMA);
      if (ok) tc_fence_after();
      ok = ok && issue_s(0) && issue_dp(0);
      for (int j = 0; ok && j < NJ; ++j) {
        if (j + 1 < NJ) {
          if (!mbar_wait_warp(s_free, j & 1, p.wc, abort_flag, SITE_DQ_MMA) || !issue_s(j + 1)) {
            ok = false;
            break;
          }
        }
        if (!mbar_wait_warp(p_ready, j & 1, p.wc, abort_flag, SITE_DQ_MMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // dQ += dS(j) K_j: keys [64w, 64w+64) of dS sit packed in columns
        // [64w, 64w+32) of the dP region
        const int sk = j % 3;
        const SDesc bk = sk == 0 ? mK0 : (sk == 1 ? mK1 : mK2);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            umma_f16_ts(tdQ, tdP + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_at(bk, kk * 2048), id_q,
                        (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&k_empty[sk]);
        }
        __syncwarp();
        if (j + 1 < NJ && !issue_dp(j + 1)) {
          ok = false;
          break;
        }
      }
      if (elect_one()) {
        if (ok) umma_commit(fin);
        umma_commit(mma_drain);
      }
      __syncwarp();
      if (lane == 0) drain_wait(mma_drain, 0, p.wc);
    }
    __syncwarp();
  } else {
    // --------------------------------------------- compute (two warpgroups)
    // Warpgroup w takes keys [64w, 64w+64) of each tile; thread r owns query
    // row ib*128 + r (tensor-memory lane r), whose LSE and D are constants.
    const int w = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int q_idx = ib * BM + r;
    const bool q_ok = q_idx < n;
    const int64_t li = (int64_t)bh * p.l_shead + row0 + q_idx;
    const float lse2 = q_ok ? p.LSE[li] * 1.4426950408889634f : INFINITY;
    const float dval = q_ok ? p.Dvec[li] : 0.0f;
    // warpgroup 0 puts row q_idx of Q into tensor memory, warpgroup 1 the
    // same row of dO (zeros past n); the bf16 pairs of a row are already
    // the packed column words
    {
      const uint4 *src = reinterpret_cast<const uint4 *>((w ? p.dO : p.Q) +
                                                         (int64_t)bh * p.q_shead +
                                                         (int64_t)(row0 + q_idx) * p.q_srow);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 u = q_ok ? __ldg(src + c * 8 + k) : make_uint4(0u, 0u, 0u, 0u);
          v[4 * k] = u.x;
          v[4 * k + 1] = u.y;
          v[4 * k + 2] = u.z;
          v[4 * k + 3] = u.w;
        }
        tmem_st32((w ? tdO : tQ) + lane_off + 32 * c, v);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(qd_ready);
    }
    bool ok = true;
    for (int j = 0; j < NJ; ++j) {
      const bool masked = (p.causal && j == ib) || ((j + 1) * BM > n);
      if (!mbar_wait(s_full, j & 1, p.wc, abort_flag, SITE_DQ_COMPUTE)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float pf[64];
      {
        uint32_t sv[64];
        tmem_ld32(tS + lane_off + 64 * w, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_ld32(tS + lane_off + 64 * w + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(s_free);  // S(j+1) may overwrite these columns
        // two keys per packed fp32 fma
        const uint64_t sc2 = f32x2(p.scale_log2, p.scale_log2);
        const uint64_t nl2 = f32x2(-lse2, -lse2);
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float a0, a1;
          f32x2_split(fma_f32x2(f32x2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sc2, nl2),
                      a0, a1);
          pf[c] = ex2(a0);
          pf[c + 1] = ex2(a1);
        }
        // keys after the query (diagonal tile) or beyond n (ragged tile): one
        // branch around the whole pass, none in the loop above
        if (masked) {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int kv = j * BM + 64 * w + c;
            if ((p.causal && kv > q_idx) || kv >= n) pf[c] = 0.0f;
          }
        }
      }
      if (!mbar_wait(dp_full, j & 1, p.wc, abort_flag, SITE_DQ_COMPUTE)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        uint32_t dp[64];
        tmem_ld32(tdP + lane_off + 64 * w, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
        tmem_ld32(tdP + lane_off + 64 * w + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
        tmem_wait_ld();
        uint32_t ds[32];
        const uint64_t dv2 = f32x2(dval, dval);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float a0, a1;
          f32x2_split(mul_f32x2(f32x2(pf[2 * c], pf[2 * c + 1]),
                                sub_f32x2(f32x2(__uint_as_float(dp[2 * c]),
                                                __uint_as_float(dp[2 * c + 1])), dv2)),
                      a0, a1);
          ds[c] = pack_bf16(a0, a1);
        }
        // dS over the first half of the dP columns this warpgroup just read
        tmem_st32(tdP + lane_off + 64 * w, ds);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_ready);
    }
    // -------------------------------------------------------- dQ epilogue
    if (ok && mbar_wait(fin, 0, p.wc, abort_flag, SITE_DQ_EPI)) {
      tc_fence_after();
      // warpgroup w writes columns [w D/2, (w+1) D/2) of dQ row q_idx
      __nv_bfloat16 *row =
          p.dQ + (int64_t)bh * p.q_shead + (int64_t)(row0 + q_idx) * p.q_srow + w * (D / 2);
      store_row_bf16<D / 2>(tdQ + lane_off + w * (D / 2), row, p.scale, q_ok);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_bwd_d(const AttnBwdArgs &a, const WaitCfg &wc, cudaStream_t st) {
  using L = BwdLayout<D>;
  const bool varlen = a.cu_seqlens != nullptr;
  // blocks per head come from the longest sequence of a variable-length batch
  const int nb_max = ((varlen ? a.max_seqlen : a.n) + BM - 1) / BM;
  const int64_t nseq = varlen ? a.nbatch : 1;
  // one CTA per (head, sequence, 128-row block): many short sequences beside
  // one long one can exceed the grid's x extent; refused before any launch
  if ((int64_t)nb_max * a.BH * nseq > 0x7fffffff) return cudaErrorNotSupported;
  cudaError_t e;
  {
    const int64_t rows = (int64_t)a.BH * a.n;  // every (head, position)
    const int64_t threads = rows * (D / 8);
    const unsigned grid = (unsigned)((threads + 255) / 256);
    bwd_prep_kernel<D><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(a.O),
                                             static_cast<const __nv_bfloat16 *>(a.dO), a.Dvec,
                                             rows, a.n, a.q_srow, a.q_shead, a.l_shead);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  CUtensorMap mq, mk, mv, mdo;
  const uint32_t box[3] = {64, 128, 1};
  const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.n, (uint64_t)a.BH};
  const uint64_t dkv[3] = {(uint64_t)D, (uint64_t)a.n, (uint64_t)a.BHkv};
  const uint64_t sq[2] = {(uint64_t)a.q_srow * 2, (uint64_t)a.q_shead * 2};
  const uint64_t skv[2] = {(uint64_t)a.kv_srow * 2, (uint64_t)a.kv_shead * 2};
  if ((e = make_tmap(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.Q, dims, sq, box))) return e;
  if ((e = make_tmap(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.K, dkv, skv, box))) return e;
  if ((e = make_tmap(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.V, dkv, skv, box))) return e;
  if ((e = make_tmap(&mdo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.dO, dims, sq, box))) return e;
  BwdParams p;
  p.BH = a.BH;
  p.n = a.n;
  p.nb = nb_max;
  p.causal = a.causal;
  p.G = a.BH / a.BHkv;
  p.q_srow = a.q_srow;
  p.q_shead = a.q_shead;
  p.kv_srow = a.kv_srow;
  p.kv_shead = a.kv_shead;
  p.l_shead = a.l_shead;
  p.cu = a.cu_seqlens;
  p.nbatch = a.nbatch;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.LSE = a.LSE;
  p.Dvec = a.Dvec;
  p.Q = static_cast<const __nv_bfloat16 *>(a.Q);
  p.dO = static_cast<const __nv_bfloat16 *>(a.dO);
  p.dQ = static_cast<__nv_bfloat16 *>(a.dQ);
  p.dK = static_cast<__nv_bfloat16 *>(a.dK);
  p.dV = static_cast<__nv_bfloat16 *>(a.dV);
  p.wc = wc;
  auto ka = varlen ? bwd_dkdv_kernel<D, true> : bwd_dkdv_kernel<D, false>;
  auto kb = varlen ? bwd_dq_kernel<D, true> : bwd_dq_kernel<D, false>;
  if ((e = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, L::A_ALLOC)))
    return e;
  if ((e = cudaFuncSetAttribute(kb, cudaFuncAttributeMaxDynamicSharedMemorySize, L::B_ALLOC)))
    return e;
  const unsigned grid_kv = (unsigned)((int64_t)p.nb * a.BHkv * nseq);
  const unsigned grid_q = (unsigned)((int64_t)p.nb * a.BH * nseq);
  timing_mark(st, 0);
  ka<<<grid_kv, NTHREADS, L::A_ALLOC, st>>>(mq, mk, mv, mdo, p);
  timing_mark(st, 1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  kb<<<grid_q, NTHREADS, L::B_ALLOC, st>>>(mk, mv, p);
  timing_mark(st, 2);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd(const AttnBwdArgs &a, const WaitCfg &wc, cudaStream_t st) {
  if (a.d == 128) return launch_bwd_d<128>(a, wc, st);
  if (a.d == 64) return launch_bwd_d<64>(a, wc, st);
  return cudaErrorInvalidValue;
}

}  // namespace chain
