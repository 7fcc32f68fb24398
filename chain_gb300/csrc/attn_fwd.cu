// attn_fwd.cu -- softmax attention forward, O = softmax(scale Q K^T) V, bf16.
//
// The unit O = f(AB)C of "Memory-efficient tensor parallelism" (FITEE
// 10.1631/FITEE.2400602, abstract) with f = row softmax, computed the way
// the Ulysses write-up ("Contexte Technique") describes FlashAttention:
// tile by tile, never storing the n x n score matrix.  Causal masking keeps
// keys j <= i on global positions (AutoSP, section 2.A item 4).
//
// One CTA per (head, 256-row query block) = two 128-row query tiles "a" and
// "b" that share every K/V tile; CTAs run head by head (K/V reuse in L2),
// heaviest causal blocks first within a head.
// Warp roles (320 threads; 384 for the f16 P V kernels, warps 10 and 11
// idle):
//   warps 0-3  softmax of tile a, warps 4-7 softmax of tile b: thread t of
//              a warpgroup owns query row t of its tile.  It reads its row
//              of S from tensor memory, runs the online softmax in fp32
//              registers and writes P back into the same tensor-memory
//              columns as a compensated pair, P_hi = bf16(P) (round to
//              nearest even) and P_lo = bf16(P - P_hi): keys [16k, 16k+16)
//              occupy columns [16k, 16k+8) (P_hi) and [16k+8, 16k+16)
//              (P_lo), two keys per 32-bit column.  O then accumulates
//              P_hi V + P_lo V, so the only bf16 rounding left is the
//              output's.  O is rescaled in tensor memory only when the row
//              max grew by more than 2^8 since the last rescale.
//   warp 8     TMA producer: Q_a and Q_b once, then K_j and V_j into 2-stage
//              rings (the on-chip form of METP's double buffer).
//   warp 9     MMA issuer, in the order  PV_a(j), S_a(j+1), PV_b(j), S_b(j+1):
//              while one warpgroup exponentiates, the tensor core multiplies
//              for the other.  The MMAs of one thread execute in issue order,
//              so completion of S_t(j+1) implies PV_t(j) is done and
//              P_t(j+1) may overwrite P_t(j) as soon as S_t(j+1) is read.
// Tensor memory: S_a/P_a [0,128), S_b/P_b [128,256), O_a [256,384),
// O_b [384,512).
//
// f16 P V (attn_fwd_pv16_kernel, attn_fwd_sp_pv16_kernel: bf16 Q, K, V;
// attn_fwd_fp8_kernel: e4m3 Q, K, V): P enters one f16 P V product and V an
// f16 copy made by a pre-pass (bf16: per K/V head scaled by a power of two,
// undone in the epilogue).  8-bit inputs: Q and K in e4m3, S = Q K^T by the
// kind::f8f6f4 tensor-core product (K = 32 per instruction, one 128-byte
// swizzled row per d = 128 row).  P is written back as one f16 per key
// (keys [32g, 32g+32) in columns [16g, 16g+16)): f16 keeps 11 significant
// bits, so no compensating low part is needed.  V arrives as f16 holding
// e4m3 value x 2^-8 (an exact re-encoding made by v_e4m3_to_f16_kernel) and
// the epilogue multiplies by 2^8 times the caller's V scale.
#include "internal.h"

namespace chain {
namespace {

constexpr int BM = 128;  // rows per query tile (two tiles per CTA)
constexpr int BN = 128;  // keys per K/V tile
constexpr int STAGES = 2;
// Threads a CTA: 320 for the compensated bf16 kernel (8 softmax warps, producer, MMA; 168
// registers, three warps per scheduler filling its quarter of the register
// file).  For the f16 P V kernels 384 at 168 registers (384 x 168 = 64,512 of the
// SM's 65,536): the producer/MMA warpgroup (with two idle warps) gives back
// down to 136 and the softmax warpgroups take 184, so that a row of S stays
// in registers next to the packed arithmetic's register pairs:
// 256 x 184 + 128 x 136 = 64,512, and 184 + 184 + 136 <= 512 per scheduler.
// (The same split measured 2-3% slower for the compensated kernel at n = 131072.)
template <bool PV16>
constexpr int fwd_threads() { return PV16 ? 384 : 320; }
constexpr uint32_t REGS_SOFTMAX = 184, REGS_CONTROL = 136;  // f16 P V kernels
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units

template <int D, bool QK8>
struct FwdLayout {
  static constexpr uint32_t QK_ELEM = QK8 ? 1 : 2;            // bytes per Q/K element
  static constexpr uint32_t Q_BYTES = BM * D * QK_ELEM;
  static constexpr uint32_t K_BYTES = BN * D * QK_ELEM;
  static constexpr uint32_t V_BYTES = BN * D * 2;             // bf16 or f16
  static constexpr uint32_t OFF_Q = 0;                        // Q_a, Q_b
  static constexpr uint32_t OFF_K = OFF_Q + 2 * Q_BYTES;      // STAGES
  static constexpr uint32_t OFF_V = OFF_K + STAGES * K_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + STAGES * V_BYTES;
  // q_full, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2],
  // p_ready[2], pv_done[2], mma_drain
  static constexpr uint32_t NBAR = 1 + 4 * STAGES + 2 + 2 + 2 + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  // At least enough shared memory to keep one CTA per SM: the kernel holds
  // all 512 tensor-memory columns.
  static constexpr uint32_t ALLOC = (BYTES + 1024 > 120 * 1024) ? BYTES + 1024 : 120 * 1024;
};

struct FwdParams {
  int BH, n, nqb2, nkb, causal;
  int G;      // query heads per K/V head (grouped-query attention; 1 = none)
  // Variable-length batch (null cu when not): sequence b occupies rows
  // [cu[b], cu[b+1]) of the packed tensors; CTAs run per (head, sequence,
  // 256-row block) over nqb2 blocks of the longest sequence.
  const int *cu;
  int nbatch;
  int n_loc;  // positions per sequence shard (n when unsharded)
  // causal, one sequence per head: the last tail_heads query heads' blocks run
  // interleaved, heaviest first across them (1: strictly head by head)
  int tail_heads;
  float scale_log2;
  float o_scale;  // f16 P V: factor applied with 1/l (8-bit inputs: 2^8 x the V scale)
  const float *v_inv;  // bf16 inputs with f16 P V: per K/V head 2^-k undoing V's scale
  __nv_bfloat16 *O;
  int64_t o_sbh, o_srow, o_sshard;
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

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// Number of key tiles query tile t (0 = a, 1 = b) of 256-row block qb sees.
__device__ __forceinline__ int kv_tiles(const FwdParams &p, int nkb, int qb, int t) {
  if (!p.causal) return nkb;
  const int last = 2 * qb + t + 1;  // tiles 0..2qb+t hold keys <= the tile's rows
  return last < nkb ? last : nkb;
}

// MODE 0: bf16 Q, K, V; P V as the compensated bf16 pair.
// MODE 1: bf16 Q, K; P V as one f16 product with V re-encoded in f16 (a
//         per-head power-of-two scale, undone in the epilogue).
// MODE 2: e4m3 Q, K (8-bit Q K^T); P V as in MODE 1 (V's codes times 2^-8).
template <int D, bool SHARDED, bool VARLEN, int MODE>
__device__ __forceinline__ void attn_fwd_body(const CUtensorMap &tmQ, const CUtensorMap &tmK,
                                              const CUtensorMap &tmV, const FwdParams &p) {
  constexpr bool QK8 = MODE == 2;   // e4m3 Q, K
  constexpr bool PV16 = MODE != 0;  // one f16 P V product
  static_assert(!QK8 || D == 128, "8-bit inputs: d = 128 only");
  static_assert(!QK8 || !SHARDED, "8-bit inputs: head-major layout only");
  using L = FwdLayout<D, QK8>;
  // Q/K boxes: 128-byte rows of 64 bf16 or 128 e4m3 elements
  constexpr int QK_BOX = 128 / L::QK_ELEM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
  uint64_t *q_full = bars;
  uint64_t *k_full = bars + 1;
  uint64_t *k_empty = k_full + STAGES;
  uint64_t *v_full = k_empty + STAGES;
  uint64_t *v_empty = v_full + STAGES;
  uint64_t *s_full = v_empty + STAGES;  // [2]
  uint64_t *p_ready = s_full + 2;       // [2]
  uint64_t *pv_done = p_ready + 2;      // [2]
  uint64_t *mma_drain = pv_done + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int blk = blockIdx.x;
  // Head-major order: the CTAs resident at one time cover one or two heads,
  // whose K and V then stay in L2 for every query block that reads them;
  // within a head the heaviest (last) causal blocks go first.
  int bh, qb, n = p.n, row0 = 0;
  if constexpr (!VARLEN) {
    bh = blk / p.nqb2;
    qb = p.causal ? (p.nqb2 - 1 - blk % p.nqb2) : (blk % p.nqb2);
    // The last heads' heaviest blocks would otherwise start only when their
    // own head comes up, and end the kernel after every other SM has gone
    // idle; interleaving the final few heads starts them together.
    const int first_tail = (p.BH - p.tail_heads) * p.nqb2;
    if (p.causal && p.tail_heads > 1 && blk >= first_tail) {
      const int r = blk - first_tail;
      bh = p.BH - p.tail_heads + r % p.tail_heads;
      qb = p.nqb2 - 1 - r / p.tail_heads;
    }
  } else {
    // one sequence of a variable-length batch; bounds clamped to the packed
    // tensor so a bad cu can never address memory outside it.  Within a
    // head, query-block pairs run in decreasing position over all of the
    // batch's sequences: a causal pair's work grows with its position, so
    // the heaviest pairs go first and the lightest fill the tail (without
    // a mask, the longest sequences go first).
    const int per_head = p.nbatch * p.nqb2;
    bh = blk / per_head;
    const int qd = (blk % per_head) / p.nbatch, b = blk % p.nbatch;
    int lo = __ldg(p.cu + b), hi = __ldg(p.cu + b + 1);
    lo = lo < 0 ? 0 : (lo > p.n ? p.n : lo);
    hi = hi < lo ? lo : (hi > p.n ? p.n : hi);
    row0 = lo;
    n = hi - lo;
    const int nqb2_b = (n + 2 * BM - 1) / (2 * BM);
    if (nqb2_b > p.nqb2) {  // longer than the stated maximum: reported, not computed
      if (qd == 0 && threadIdx.x == 0 && bh == 0) atomicExch(&p.wc.status->reserved[0], 1);
      return;
    }
    qb = p.nqb2 - 1 - qd;
    if (qb >= nqb2_b) return;  // nothing of this sequence for this CTA
  }
  const int nkb = (n + BN - 1) / BN;
  const int nkv_a = kv_tiles(p, nkb, qb, 0);
  const int nkv_b = kv_tiles(p, nkb, qb, 1);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_ready[t], 128);
      mbar_init(&pv_done[t], 1);
    }
    mbar_init(mma_drain, 1);
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The three roles; the f16 P V kernels reallocate registers per warpgroup
  // before running theirs.
  auto role_producer = [&]() {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int k_issued = 0, v_issued = 0;
      // 128-row box starting at sequence position `row`; over sequence
      // shards: shard row / n_loc, row row % n_loc in it (a box never
      // crosses a shard)
      // Q of head bh; K and V of its group's head bh / G
      auto load = [&](uint8_t *dst, const CUtensorMap *map, uint64_t *bar, int c0, int row,
                      int head) {
        if constexpr (SHARDED) {
          const int sh = row / p.n_loc;
          tma_load_4d(dst, map, bar, c0, row - sh * p.n_loc, sh, head);
        } else {
          tma_load_3d(dst, map, bar, c0, row0 + row, head);
        }
      };
      const int bkv = bh / p.G;
      mbar_arrive_expect_tx(q_full, 2 * L::Q_BYTES);
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int c = 0; c < D / QK_BOX; ++c)
          load(smem + L::OFF_Q + t * L::Q_BYTES + c * (BM * 128), &tmQ, q_full, c * QK_BOX,
               (2 * qb + t) * BM, bh);
      for (int j = 0; j < nkv_b; ++j) {
        const int st = j % STAGES;
        if (j >= STAGES &&
            !mbar_wait(&k_empty[st], ((j / STAGES) - 1) & 1, p.wc, abort_flag, SITE_FWD_PROD))
          break;
        mbar_arrive_expect_tx(&k_full[st], L::K_BYTES);
#pragma unroll
        for (int c = 0; c < D / QK_BOX; ++c)
          load(smem + L::OFF_K + st * L::K_BYTES + c * (BN * 128), &tmK, &k_full[st], c * QK_BOX,
               j * BN, bkv);
        k_issued = j + 1;
        if (j >= STAGES &&
            !mbar_wait(&v_empty[st], ((j / STAGES) - 1) & 1, p.wc, abort_flag, SITE_FWD_PROD))
          break;
        mbar_arrive_expect_tx(&v_full[st], L::V_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint8_t *dst = smem + L::OFF_V + st * L::V_BYTES + c * (BN * 128);
          if constexpr (PV16)  // the f16 copy of V is head-major in every layout
            tma_load_3d(dst, &tmV, &v_full[st], c * 64, row0 + j * BN, bkv);
          else
            load(dst, &tmV, &v_full[st], c * 64, j * BN, bkv);
        }
        v_issued = j + 1;
      }
      if (*abort_flag) {
        // Let every copy still in flight land before shared memory is freed.
        drain_wait(q_full, 0, p.wc);
        for (int j = (k_issued > STAGES ? k_issued - STAGES : 0); j < k_issued; ++j)
          drain_wait(&k_full[j % STAGES], (j / STAGES) & 1, p.wc);
        for (int j = (v_issued > STAGES ? v_issued - STAGES : 0); j < v_issued; ++j)
          drain_wait(&v_full[j % STAGES], (j / STAGES) & 1, p.wc);
      }
    }
    __syncwarp();
  };
  auto role_mma = [&]() {
    // --------------------------------------------------------- MMA issuer
    // The whole warp runs the loop; one elected lane issues each group of
    // products together with its commits.
    {
      const uint32_t idS = QK8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN, 0, 0);
      const uint32_t idO = PV16 ? idesc_f16_f32(BM, D, 0, 1) : idesc_bf16_f32(BM, D, 0, 1);
      // Base descriptors built once; every MMA below only adds a
      // compile-time byte offset to the low word.
      const SDesc dQ0 = sdesc_make(smem_u32(smem + L::OFF_Q), 16, 1024);
      const SDesc dQ1 = sdesc_make(smem_u32(smem + L::OFF_Q + L::Q_BYTES), 16, 1024);
      const SDesc dK0 = sdesc_make(smem_u32(smem + L::OFF_K), 16, 1024);
      const SDesc dK1 = sdesc_make(smem_u32(smem + L::OFF_K + L::K_BYTES), 16, 1024);
      const SDesc dV0 = sdesc_make(smem_u32(smem + L::OFF_V), BN * 128, 1024);
      const SDesc dV1 = sdesc_make(smem_u32(smem + L::OFF_V + L::V_BYTES), BN * 128, 1024);
      static_assert(STAGES == 2, "descriptor selection assumes two stages");
      // S_t(j) = Q_t K_j^T into columns [128t, 128t+128); each product
      // takes a 32-byte K slice of the 128-byte rows (16 bf16 or 32 e4m3)
      auto issue_s = [&](int t, int j) {
        const SDesc a = t ? dQ1 : dQ0;
        const SDesc b = (j & 1) ? dK1 : dK0;
#pragma unroll
        for (int kk = 0; kk < D * (int)L::QK_ELEM / 32; ++kk) {
          const uint32_t off = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
          if constexpr (QK8)
            umma_f8_ss(tmem + t * BN, sdesc_at(a, off), sdesc_at(b, off), idS, kk > 0 ? 1u : 0u);
          else
            umma_f16_ss(tmem + t * BN, sdesc_at(a, off), sdesc_at(b, off), idS, kk > 0 ? 1u : 0u);
        }
      };
      // O_t += P_hi V_j + P_lo V_j (f16 P V: O_t += P V_j, one f16 P
      // per key), P read from tensor memory
      auto issue_pv = [&](int t, int j) {
        const SDesc b = (j & 1) ? dV1 : dV0;
        const uint32_t tP = tmem + t * BN;
        if constexpr (PV16) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            umma_f16_ts(tmem + 256 + t * 128, tP + kk * 8, sdesc_at(b, kk * 2048), idO,
                        (j > 0 || kk > 0) ? 1u : 0u);
        } else {
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              umma_f16_ts(tmem + 256 + t * 128, tP + kk * 16 + part * 8, sdesc_at(b, kk * 2048),
                          idO, (j > 0 || part > 0 || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait_warp(q_full, 0, p.wc, abort_flag, SITE_FWD_MMA) &&
                mbar_wait_warp(&k_full[0], 0, p.wc, abort_flag, SITE_FWD_MMA);
      if (ok) {
        tc_fence_after();
        if (elect_one()) {
          issue_s(0, 0);
          umma_commit(&s_full[0]);
          issue_s(1, 0);
          umma_commit(&s_full[1]);
          umma_commit(&k_empty[0]);
        }
        __syncwarp();
      }
      for (int j = 0; ok && j < nkv_b; ++j) {
        const int st = j % STAGES;
        const int jn = j + 1, stn = jn % STAGES;
        if (!mbar_wait_warp(&v_full[st], (j / STAGES) & 1, p.wc, abort_flag, SITE_FWD_MMA)) break;
        if (j < nkv_a) {
          if (!mbar_wait_warp(&p_ready[0], j & 1, p.wc, abort_flag, SITE_FWD_MMA)) break;
          tc_fence_after();
          if (elect_one()) {
            issue_pv(0, j);
            umma_commit(&pv_done[0]);
          }
          __syncwarp();
          if (jn < nkv_a) {
            if (!mbar_wait_warp(&k_full[stn], (jn / STAGES) & 1, p.wc, abort_flag, SITE_FWD_MMA)) break;
            tc_fence_after();
            if (elect_one()) {
              issue_s(0, jn);
              umma_commit(&s_full[0]);
            }
            __syncwarp();
          }
        }
        if (!mbar_wait_warp(&p_ready[1], j & 1, p.wc, abort_flag, SITE_FWD_MMA)) break;
        tc_fence_after();
        if (elect_one()) {
          issue_pv(1, j);
          umma_commit(&pv_done[1]);
          umma_commit(&v_empty[st]);
        }
        __syncwarp();
        if (jn < nkv_b) {
          if (!mbar_wait_warp(&k_full[stn], (jn / STAGES) & 1, p.wc, abort_flag, SITE_FWD_MMA)) break;
          tc_fence_after();
          if (elect_one()) {
            issue_s(1, jn);
            umma_commit(&s_full[1]);
            umma_commit(&k_empty[stn]);
          }
          __syncwarp();
        }
      }
      // No MMA may still be running when tensor memory is released.
      if (elect_one()) umma_commit(mma_drain);
      __syncwarp();
      if (lane == 0) drain_wait(mma_drain, 0, p.wc);
    }
    __syncwarp();
  };
  auto role_softmax = [&]() {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;            // query tile of this warpgroup
    const int row = threadIdx.x & 127;  // tensor-memory lane = row
    const int q_idx = (2 * qb + t) * BM + row;
    const int nkv = t ? nkv_b : nkv_a;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * BN;
    const uint32_t tO = tmem + lane_off + 256 + t * 128;
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      if (!mbar_wait(&s_full[t], j & 1, p.wc, abort_flag, SITE_FWD_SOFTMAX)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int kv0 = j * BN;
      const bool diag = p.causal && (j == 2 * qb + t);
      const bool masked = diag || (kv0 + BN > n);
      // Row of S: one round trip to tensor memory, kept in registers for
      // both passes.  Diagonal and ragged tiles mask keys after the row and
      // keys beyond n.
      uint32_t s[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
        tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));
      tmem_wait_ld();
      if (masked) {
#pragma unroll
        for (int k = 0; k < BN; ++k) {
          const int kv = kv0 + k;
          if ((diag && kv > q_idx) || kv >= n) s[k] = __float_as_uint(-INFINITY);
        }
      }
      // pass 1: row max, eight independent partial maxima (a tree, not a
      // 128-long dependent chain); f16 P V: four, two keys per three-input
      // max
      float mx8[8];
      if constexpr (PV16) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          mx8[u] = fmaxf(__uint_as_float(s[2 * u]), __uint_as_float(s[2 * u + 1]));
#pragma unroll
        for (int k = 8; k < BN; k += 8)
#pragma unroll
          for (int u = 0; u < 4; ++u)
            mx8[u] = fmax3(mx8[u], __uint_as_float(s[k + 2 * u]), __uint_as_float(s[k + 2 * u + 1]));
        mx8[4] = mx8[5] = mx8[6] = mx8[7] = -INFINITY;
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) mx8[u] = __uint_as_float(s[u]);
#pragma unroll
        for (int k = 8; k < BN; ++k) mx8[k & 7] = fmaxf(mx8[k & 7], __uint_as_float(s[k]));
      }
      float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      mx *= p.scale_log2;  // scale > 0: the max commutes with the scaling
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
      // pass 2: P = 2^(s*scale*log2e - m), 16 keys at a time, written back
      // over the columns already read: keys [16g, 16g+16) go to columns
      // [16g, 16g+8) (P_hi) and [16g+8, 16g+16) (P_lo), two keys per column.
      float rs4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if constexpr (PV16) {
        // f16 P: keys [32g, 32g+32) to columns [16g, 16g+16); two keys per
        // packed fp32 instruction for x = s * scale - m and the row sum
        const uint64_t sc2 = f32x2(p.scale_log2, p.scale_log2);
        const uint64_t nm2 = f32x2(-mref, -mref);
        uint64_t rs2[4] = {0, 0, 0, 0};
#pragma unroll
        for (int g = 0; g < BN / 32; ++g) {
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            float x0, x1;
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(s[g * 32 + k]),
                                        __uint_as_float(s[g * 32 + k + 1])), sc2, nm2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            rs2[(k >> 1) & 3] = add_f32x2(rs2[(k >> 1) & 3], f32x2(p0, p1));
            pk[k >> 1] = pack_f16(p0, p1);
          }
          tmem_st16(tS + g * 16, pk);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float a0, a1;
          f32x2_split(rs2[u], a0, a1);
          rs4[u] = a0 + a1;
        }
      }
#pragma unroll
      for (int g = 0; g < (PV16 ? 0 : BN / 16); ++g) {
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; k += 2) {
          const float p0 = ex2(fmaf(__uint_as_float(s[g * 16 + k]), p.scale_log2, -mref));
          const float p1 = ex2(fmaf(__uint_as_float(s[g * 16 + k + 1]), p.scale_log2, -mref));
          rs4[(k >> 1) & 3] += p0 + p1;
          const uint32_t h = pack_bf16(p0, p1);
          pk[k >> 1] = h;
          pk[8 + (k >> 1)] =
              pack_bf16(p0 - __uint_as_float(h << 16), p1 - __uint_as_float(h & 0xffff0000u));
        }
        tmem_st16(tS + g * 16, pk);
      }
      const float rs = (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
      // O_t holds every P_t(j') V_j' with j' < j here: S_t(j) was issued
      // after PV_t(j-1), and PV_t(j) waits for p_ready below.  (Done after
      // pass 2 so the row of S is no longer live.)
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tmem_st32(tO + c * 32, o);
        }
      }
      l = l * alpha + rs;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_ready[t]);
    }
    // ----------------------------------------------------------- epilogue
    if (ok && mbar_wait(&pv_done[t], (nkv - 1) & 1, p.wc, abort_flag, SITE_FWD_EPI)) {
      tc_fence_after();
      float inv_l = 1.0f / l;
      if constexpr (PV16) inv_l *= p.o_scale;
      if constexpr (MODE == 1) inv_l *= __ldg(p.v_inv + bh / p.G);
      const int q_sh = SHARDED ? q_idx / p.n_loc : 0;
      __nv_bfloat16 *orow = p.O + (int64_t)bh * p.o_sbh + (int64_t)q_sh * p.o_sshard +
                            (int64_t)(row0 + q_idx - q_sh * p.n_loc) * p.o_srow;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_wait_ld();
        if (q_idx < n) {
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
      if (q_idx < n)
        p.LSE[(int64_t)bh * p.lse_sbh + row0 + q_idx] = (m + lg2(l)) * 0.69314718055994531f;
    }
  };
  if constexpr (PV16) {
    if (warp >= 8) {  // warps 10 and 11 only hand their registers over
      setmaxnreg_dec<REGS_CONTROL>();
      if (warp == 8)
        role_producer();
      else if (warp == 9)
        role_mma();
    } else {
      setmaxnreg_inc<REGS_SOFTMAX>();
      role_softmax();
    }
  } else {
    if (warp == 8)
      role_producer();
    else if (warp == 9)
      role_mma();
    else
      role_softmax();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool SHARDED, bool VARLEN>
__global__ void __launch_bounds__(fwd_threads<false>(), 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  attn_fwd_body<D, SHARDED, VARLEN, 0>(tmQ, tmK, tmV, p);
}

template <int D>
__global__ void __launch_bounds__(fwd_threads<true>(), 1)
    attn_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  attn_fwd_body<D, false, false, 2>(tmQ, tmK, tmV, p);
}

template <int D>
__global__ void __launch_bounds__(fwd_threads<true>(), 1)
    attn_fwd_pv16_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  attn_fwd_body<D, false, false, 1>(tmQ, tmK, tmV, p);
}

// The same over sequences packed end to end ([total][H][d], cu_seqlens);
// V's f16 copy is [Hkv][total][d].
template <int D>
__global__ void __launch_bounds__(fwd_threads<true>(), 1)
    attn_fwd_varlen_pv16_kernel(const __grid_constant__ CUtensorMap tmQ,
                                const __grid_constant__ CUtensorMap tmK,
                                const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  attn_fwd_body<D, false, true, 1>(tmQ, tmK, tmV, p);
}

// The same over Ulysses sequence shards: Q, K read from and O written to
// [p][n_loc][H][d]; V's f16 copy is head-major (its pre-pass reads the shards).
template <int D>
__global__ void __launch_bounds__(fwd_threads<true>(), 1)
    attn_fwd_sp_pv16_kernel(const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  attn_fwd_body<D, true, false, 1>(tmQ, tmK, tmV, p);
}

// e4m3 V [BHkv][n][128] (strided rows) -> f16 [BHkv][n][128] packed, each
// value times 2^-8, exactly.  An e4m3 byte s.eeee.mmm placed as the f16 bit
// pattern s.0eeee.mmm0000000 is the same number scaled by 2^(7-15): the f16
// exponent bias is 15, e4m3's is 7, and e4m3 subnormals (e = 0) land on f16
// subnormals with the same mantissa.  The NaN codes s.1111.111 become
// +-1.875 (read as 480 after the epilogue's 2^8): inputs are taken finite.
__global__ void __launch_bounds__(256)
    v_e4m3_to_f16_kernel(const uint8_t *__restrict__ V, int64_t s_bh, int64_t s_row, int n,
                         int64_t rows, uint16_t *__restrict__ out) {
  const int64_t chunks = rows * 8;  // 16 e4m3 (16 bytes) per chunk
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < chunks;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i >> 3;
    const int c = (int)(i & 7);
    const int64_t h = r / n, t = r - h * n;
    const uint4 x = __ldg(reinterpret_cast<const uint4 *>(V + h * s_bh + t * s_row + c * 16));
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t y[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // bytes (b0, b1) and (b2, b3) to the high byte of each 16-bit half
      const uint32_t u0 = __byte_perm(w[k], 0, 0x1404);
      const uint32_t u1 = __byte_perm(w[k], 0, 0x3424);
      y[2 * k] = (u0 & 0x80008000u) | ((u0 >> 1) & 0x3F803F80u);
      y[2 * k + 1] = (u1 & 0x80008000u) | ((u1 >> 1) & 0x3F803F80u);
    }
    uint4 *dst = reinterpret_cast<uint4 *>(out + r * 128 + c * 16);
    dst[0] = make_uint4(y[0], y[1], y[2], y[3]);
    dst[1] = make_uint4(y[4], y[5], y[6], y[7]);
  }
}

// bf16 V -> f16 with one power-of-two scale 2^k per K/V head, chosen from the
// head's largest |v| so that it lands in [2^14, 2^15): every value keeps its
// 8 significant bits in f16 exactly, except values smaller than 2^-31 of
// that maximum, which fall into f16's subnormal range and are rounded with an
// absolute error of at most 2^-39 of the maximum.  Two passes over V in row chunks of VCH_ROWS rows:
// v_absmax_kernel writes each chunk's largest |v| (as bf16 magnitude bits,
// which order like the values), v_to_f16_kernel reduces a head's chunk
// maxima, converts its chunk and (chunk 0) stores 2^-k for the epilogue.
constexpr int VCH_ROWS = 256;

__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  v = red[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) v = max(v, red[w]);
  __syncthreads();
  return v;
}

// Row t of head h lives at V + h s_bh + (t / n_loc) s_shard + (t % n_loc) s_row
// (n_loc = n, s_shard = 0 for one contiguous sequence).
__device__ __forceinline__ const __nv_bfloat16 *v_row(const __nv_bfloat16 *V, int64_t s_bh,
                                                      int64_t s_row, int64_t s_shard, int n_loc,
                                                      int h, int t) {
  const int sh = t / n_loc;
  return V + h * s_bh + sh * s_shard + (int64_t)(t - sh * n_loc) * s_row;
}

template <int D>
__global__ void __launch_bounds__(256)
    v_absmax_kernel(const __nv_bfloat16 *__restrict__ V, int64_t s_bh, int64_t s_row,
                    int64_t s_shard, int n_loc, int n, int nch, uint32_t *__restrict__ part) {
  __shared__ uint32_t red[8];
  const int h = blockIdx.y, ch = blockIdx.x;
  const int r0 = ch * VCH_ROWS;
  const int rows = min(VCH_ROWS, n - r0);
  constexpr int VPR = D / 8;  // 16-byte vectors per row
  uint32_t m = 0;
  for (int i = threadIdx.x; i < rows * VPR; i += blockDim.x) {
    const int r = i / VPR, c = i % VPR;
    const uint4 x =
        __ldg(reinterpret_cast<const uint4 *>(v_row(V, s_bh, s_row, s_shard, n_loc, h, r0 + r)) + c);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) m = max(m, max(w[k] & 0x7fffu, (w[k] >> 16) & 0x7fffu));
  }
  m = block_max_u32(m, red);
  if (threadIdx.x == 0) part[(int64_t)h * nch + ch] = m;
}

template <int D>
__global__ void __launch_bounds__(256)
    v_to_f16_kernel(const __nv_bfloat16 *__restrict__ V, int64_t s_bh, int64_t s_row,
                    int64_t s_shard, int n_loc, int n, int nch,
                    const uint32_t *__restrict__ part, uint16_t *__restrict__ out,
                    float *__restrict__ v_inv) {
  __shared__ uint32_t red[8];
  const int h = blockIdx.y, ch = blockIdx.x;
  uint32_t m = 0;
  for (int i = threadIdx.x; i < nch; i += blockDim.x) m = max(m, part[(int64_t)h * nch + i]);
  m = block_max_u32(m, red);
  // m: bf16 bits of the head's largest |v|; its exponent field e gives
  // |v|max in [2^(e-127), 2^(e-126)), so k = 141 - e puts it in [2^14, 2^15).
  // Zero, infinite or NaN maxima keep k = 0.
  const int e = (int)(m >> 7);
  int k = (m == 0 || e == 255) ? 0 : 141 - e;
  k = k < -126 ? -126 : (k > 126 ? 126 : k);
  const float sc = __uint_as_float((uint32_t)(127 + k) << 23);
  if (ch == 0 && threadIdx.x == 0) v_inv[h] = __uint_as_float((uint32_t)(127 - k) << 23);
  const int r0 = ch * VCH_ROWS;
  const int rows = min(VCH_ROWS, n - r0);
  constexpr int VPR = D / 8;
  for (int i = threadIdx.x; i < rows * VPR; i += blockDim.x) {
    const int r = i / VPR, c = i % VPR;
    const uint4 x =
        __ldg(reinterpret_cast<const uint4 *>(v_row(V, s_bh, s_row, s_shard, n_loc, h, r0 + r)) + c);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t y[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      y[q] = pack_f16(__uint_as_float(w[q] << 16) * sc, __uint_as_float(w[q] & 0xffff0000u) * sc);
    reinterpret_cast<uint4 *>(out + ((int64_t)h * n + r0 + r) * D)[c] = make_uint4(y[0], y[1], y[2], y[3]);
  }
}


// Query heads whose blocks interleave at the end of a causal launch of one
// sequence per head: as many as keep their K and V (a 16-bit copy each, at
// most) under 64 MB of L2, in whole K/V-head groups.  Within the kernel, heads
// otherwise run one after the other so each head's K and V stay in L2.
int fwd_tail_heads(int BH, int BHkv, int64_t n, int d, bool causal, bool varlen) {
  if (!causal || varlen || BHkv <= 0) return 1;
  const int64_t kv = (int64_t(64) << 20) / (4 * n * d);
  if (kv < 1) return 1;
  const int64_t t = kv * (BH / BHkv);
  return t < BH ? (int)t : BH;
}

template <int D>
cudaError_t launch_fwd_d(const AttnFwdArgs &a, const WaitCfg &wc, cudaStream_t st) {
  using L = FwdLayout<D, false>;
  // Tensor maps {d, row, head} for one contiguous sequence; {d, row in
  // shard, shard, head} over sequence shards.
  CUtensorMap mq, mk, mv;
  const bool sharded = a.n_loc != a.n;
  const int rank = sharded ? 4 : 3;
  const int nsh = a.n / a.n_loc;
  const uint32_t box[4] = {64, 128, 1, 1};
  uint64_t dims[4] = {(uint64_t)a.d, (uint64_t)a.n_loc, (uint64_t)nsh, (uint64_t)a.BH};
  uint64_t dkv[4] = {(uint64_t)a.d, (uint64_t)a.n_loc, (uint64_t)nsh, (uint64_t)a.BHkv};
  uint64_t sq[3] = {(uint64_t)a.q_srow * 2, (uint64_t)a.q_sshard * 2, (uint64_t)a.q_sbh * 2};
  uint64_t sk[3] = {(uint64_t)a.k_srow * 2, (uint64_t)a.k_sshard * 2, (uint64_t)a.k_sbh * 2};
  uint64_t sv[3] = {(uint64_t)a.v_srow * 2, (uint64_t)a.v_sshard * 2, (uint64_t)a.v_sbh * 2};
  if (!sharded) {  // drop the shard dimension
    dims[2] = dims[3];
    dkv[2] = dkv[3];
    sq[1] = sq[2];
    sk[1] = sk[2];
    sv[1] = sv[2];
  }
  cudaError_t e;
  if ((e = make_tmap(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, a.Q, dims, sq, box)) != cudaSuccess)
    return e;
  if ((e = make_tmap(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, a.K, dkv, sk, box)) != cudaSuccess)
    return e;
  if ((e = make_tmap(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, a.V, dkv, sv, box)) != cudaSuccess)
    return e;
  FwdParams p;
  p.BH = a.BH;
  p.n = a.n;
  p.cu = a.cu_seqlens;
  p.nbatch = a.nbatch;
  // with a variable-length batch, blocks per head come from the longest sequence
  const int nmax = a.cu_seqlens ? a.max_seqlen : a.n;
  p.nqb2 = (nmax + 2 * BM - 1) / (2 * BM);
  p.nkb = (a.n + BN - 1) / BN;
  p.causal = a.causal;
  p.tail_heads = fwd_tail_heads(a.BH, a.BHkv, a.n, D, a.causal, a.cu_seqlens != nullptr);
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.o_scale = 1.0f;
  p.v_inv = nullptr;
  p.O = static_cast<__nv_bfloat16 *>(a.O);
  p.o_sbh = a.o_sbh;
  p.o_srow = a.o_srow;
  p.o_sshard = a.o_sshard;
  p.n_loc = a.n_loc;
  p.G = a.BH / a.BHkv;
  p.LSE = a.LSE;
  p.lse_sbh = a.lse_sbh;
  p.wc = wc;
  auto kern = sharded ? attn_fwd_kernel<D, true, false>
                      : (a.cu_seqlens ? attn_fwd_kernel<D, false, true> : attn_fwd_kernel<D, false, false>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  // one CTA per (head, sequence, query-block pair): many short sequences
  // beside one long one can exceed the grid's x extent
  const int64_t grid64 = (int64_t)p.nqb2 * a.BH * (a.cu_seqlens ? a.nbatch : 1);
  if (grid64 > 0x7fffffff) return cudaErrorNotSupported;
  const unsigned grid = (unsigned)grid64;
  timing_mark(st, 0);
  kern<<<grid, fwd_threads<false>(), L::ALLOC, st>>>(mq, mk, mv, p);
  timing_mark(st, 1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd_bf16(const AttnFwdArgs &a, const WaitCfg &wc, cudaStream_t st) {
  if (a.d == 128) return launch_fwd_d<128>(a, wc, st);
  if (a.d == 64) return launch_fwd_d<64>(a, wc, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_fwd_fp8(const AttnFwdArgs &a, void *v16, const WaitCfg &wc,
                               cudaStream_t st) {
  if (a.d != 128 || a.n_loc != a.n || a.cu_seqlens) return cudaErrorNotSupported;
  using L = FwdLayout<128, true>;
  // V -> f16 (x 2^-8) into the workspace, [BHkv][n][128] packed
  const int64_t rows = (int64_t)a.BHkv * a.n;
  const int64_t blocks = (rows * 8 + 255) / 256;
  timing_mark(st, 0);
  v_e4m3_to_f16_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, st>>>(
      static_cast<const uint8_t *>(a.V), a.v_sbh, a.v_srow, a.n, rows,
      static_cast<uint16_t *>(v16));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // Q, K: e4m3 rows of 128 bytes, one 128 x 128 box per tile; V: f16 boxes
  // of 64 columns as in the bf16 kernel
  CUtensorMap mq, mk, mv;
  const uint32_t box_qk[3] = {128, 128, 1};
  const uint32_t box_v[3] = {64, 128, 1};
  const uint64_t dq[3] = {128, (uint64_t)a.n, (uint64_t)a.BH};
  const uint64_t dkv[3] = {128, (uint64_t)a.n, (uint64_t)a.BHkv};
  const uint64_t sq[2] = {(uint64_t)a.q_srow, (uint64_t)a.q_sbh};
  const uint64_t sk[2] = {(uint64_t)a.k_srow, (uint64_t)a.k_sbh};
  const uint64_t sv[2] = {256, (uint64_t)a.n * 256};
  if ((e = make_tmap(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.Q, dq, sq, box_qk)) != cudaSuccess)
    return e;
  if ((e = make_tmap(&mk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.K, dkv, sk, box_qk)) != cudaSuccess)
    return e;
  if ((e = make_tmap(&mv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, v16, dkv, sv, box_v)) != cudaSuccess)
    return e;
  FwdParams p;
  p.BH = a.BH;
  p.n = a.n;
  p.cu = nullptr;
  p.nbatch = 0;
  p.nqb2 = (a.n + 2 * BM - 1) / (2 * BM);
  p.nkb = (a.n + BN - 1) / BN;
  p.causal = a.causal;
  p.tail_heads = fwd_tail_heads(a.BH, a.BHkv, a.n, 128, a.causal, false);
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.o_scale = 256.0f * a.v_scale;
  p.v_inv = nullptr;
  p.O = static_cast<__nv_bfloat16 *>(a.O);
  p.o_sbh = a.o_sbh;
  p.o_srow = a.o_srow;
  p.o_sshard = 0;
  p.n_loc = a.n;
  p.G = a.BH / a.BHkv;
  p.LSE = a.LSE;
  p.lse_sbh = a.lse_sbh;
  p.wc = wc;
  e = cudaFuncSetAttribute(attn_fwd_fp8_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           L::ALLOC);
  if (e != cudaSuccess) return e;
  timing_mark(st, 1);
  attn_fwd_fp8_kernel<128>
      <<<(unsigned)(p.nqb2 * a.BH), fwd_threads<true>(), L::ALLOC, st>>>(mq, mk, mv, p);
  timing_mark(st, 2);
  return cudaGetLastError();
}

size_t attn_fwd_pv16_workspace(int BHkv, int n, int d) {
  const size_t vb = ((size_t)2 * BHkv * n * d + 255) & ~(size_t)255;
  const size_t nch = (size_t)(n + VCH_ROWS - 1) / VCH_ROWS;
  return vb + ((4 * (size_t)BHkv * nch + 255) & ~(size_t)255) + ((4 * (size_t)BHkv + 255) & ~(size_t)255);
}

template <int D>
static cudaError_t launch_pv16_d(const AttnFwdArgs &a, void *ws, const WaitCfg &wc,
                                 cudaStream_t st) {
  using L = FwdLayout<D, false>;
  // with a variable-length batch, blocks per head come from the longest
  // sequence; one CTA per (head, sequence, query-block pair), refused before
  // any launch when that exceeds the grid's x extent
  const int nqb2 = ((a.cu_seqlens ? a.max_seqlen : a.n) + 2 * BM - 1) / (2 * BM);
  const int64_t grid64 = (int64_t)nqb2 * a.BH * (a.cu_seqlens ? a.nbatch : 1);
  if (grid64 > 0x7fffffff) return cudaErrorNotSupported;
  const int nch = (a.n + VCH_ROWS - 1) / VCH_ROWS;
  uint8_t *base = static_cast<uint8_t *>(ws);
  const size_t vb = ((size_t)2 * a.BHkv * a.n * D + 255) & ~(size_t)255;
  uint16_t *v16 = reinterpret_cast<uint16_t *>(base);
  uint32_t *part = reinterpret_cast<uint32_t *>(base + vb);
  float *v_inv = reinterpret_cast<float *>(base + vb + ((4 * (size_t)a.BHkv * nch + 255) & ~(size_t)255));
  const dim3 vgrid((unsigned)nch, (unsigned)a.BHkv);
  const __nv_bfloat16 *V = static_cast<const __nv_bfloat16 *>(a.V);
  const bool sharded = a.n_loc != a.n;
  const int64_t v_sshard = sharded ? a.v_sshard : 0;
  timing_mark(st, 0);
  v_absmax_kernel<D><<<vgrid, 256, 0, st>>>(V, a.v_sbh, a.v_srow, v_sshard, a.n_loc, a.n, nch,
                                            part);
  v_to_f16_kernel<D><<<vgrid, 256, 0, st>>>(V, a.v_sbh, a.v_srow, v_sshard, a.n_loc, a.n, nch,
                                            part, v16, v_inv);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // Q, K: {d, row, head}, or {d, row in shard, shard, head} over sequence
  // shards; V's f16 copy: {d, row, head}
  CUtensorMap mq, mk, mv;
  const int rank = sharded ? 4 : 3;
  const uint32_t box[4] = {64, 128, 1, 1};
  const int64_t nsh = a.n / a.n_loc;
  uint64_t dq[4] = {(uint64_t)D, (uint64_t)a.n_loc, (uint64_t)nsh, (uint64_t)a.BH};
  uint64_t dk[4] = {(uint64_t)D, (uint64_t)a.n_loc, (uint64_t)nsh, (uint64_t)a.BHkv};
  uint64_t sq[3] = {(uint64_t)a.q_srow * 2, (uint64_t)a.q_sshard * 2, (uint64_t)a.q_sbh * 2};
  uint64_t sk[3] = {(uint64_t)a.k_srow * 2, (uint64_t)a.k_sshard * 2, (uint64_t)a.k_sbh * 2};
  if (!sharded) {  // drop the shard dimension
    dq[2] = dq[3];
    dk[2] = dk[3];
    sq[1] = sq[2];
    sk[1] = sk[2];
  }
  const uint64_t dv[3] = {(uint64_t)D, (uint64_t)a.n, (uint64_t)a.BHkv};
  const uint64_t sv[2] = {(uint64_t)D * 2, (uint64_t)a.n * D * 2};
  if ((e = make_tmap(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, a.Q, dq, sq, box)) != cudaSuccess)
    return e;
  if ((e = make_tmap(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, a.K, dk, sk, box)) != cudaSuccess)
    return e;
  if ((e = make_tmap(&mv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, v16, dv, sv, box)) != cudaSuccess)
    return e;
  FwdParams p;
  p.BH = a.BH;
  p.n = a.n;
  p.cu = a.cu_seqlens;
  p.nbatch = a.cu_seqlens ? a.nbatch : 0;
  p.nqb2 = nqb2;
  p.nkb = (a.n + BN - 1) / BN;
  p.causal = a.causal;
  p.tail_heads = fwd_tail_heads(a.BH, a.BHkv, a.n, D, a.causal, a.cu_seqlens != nullptr);
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.o_scale = 1.0f;
  p.v_inv = v_inv;
  p.O = static_cast<__nv_bfloat16 *>(a.O);
  p.o_sbh = a.o_sbh;
  p.o_srow = a.o_srow;
  p.o_sshard = sharded ? a.o_sshard : 0;
  p.n_loc = a.n_loc;
  p.G = a.BH / a.BHkv;
  p.LSE = a.LSE;
  p.lse_sbh = a.lse_sbh;
  p.wc = wc;
  auto kern = sharded ? attn_fwd_sp_pv16_kernel<D>
                      : (a.cu_seqlens ? attn_fwd_varlen_pv16_kernel<D> : attn_fwd_pv16_kernel<D>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)grid64;
  timing_mark(st, 1);
  kern<<<grid, fwd_threads<true>(), L::ALLOC, st>>>(mq, mk, mv, p);
  timing_mark(st, 2);
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd_pv16(const AttnFwdArgs &a, void *ws, const WaitCfg &wc,
                                 cudaStream_t st) {
  if (a.cu_seqlens && a.n_loc != a.n) return cudaErrorNotSupported;
  if (a.d == 128) return launch_pv16_d<128>(a, ws, wc, st);
  if (a.d == 64) return launch_pv16_d<64>(a, ws, wc, st);
  return cudaErrorInvalidValue;
}

}  // namespace chain
