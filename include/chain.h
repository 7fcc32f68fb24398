/*
 * chain.h -- C ABI of the GB300 (sm_103a) library for the unit
 *            O = f(A . B) . C
 *
 * The unit: two consecutive matrix products with a function between them,
 * as named in the abstract of "Memory-efficient tensor parallelism"
 * (FITEE 10.1631/FITEE.2400602).  Three instances are served:
 *   - f = row softmax of scaled scores (attention: A = Q, B = K^T * scale,
 *     C = V), causal or not, forward and a backward that recomputes the
 *     scores from the saved log-sum-exp instead of storing them ("AutoSP:
 *     Unlocking Long-Context LLM Training Via Compiler-Based Sequence
 *     Parallelism", section 2.B);
 *   - f = GeLU (tanh form), the MLP chain, whose [M][N] intermediate is
 *     never written to memory;
 *   - f = identity, O = (A B) C.
 * plus the Ulysses sequence-shard -> head-major relayout that precedes
 * attention ("Ulysses Sequence Parallelism", "Contexte Technique") and its
 * inverse (the second exchange of "Analyse et Implications").
 *
 * Conventions common to every entry point
 *  - Tensors are described by chain_tensor_t: a DEVICE pointer, an element
 *    type, and shape/strides counted in ELEMENTS (not bytes), outermost
 *    dimension first.  The innermost stride must be 1; every other stride
 *    must describe a row-major layout without overlap.  Base pointers must
 *    be 16-byte aligned and row pitches multiples of 16 bytes.
 *  - Ownership: the caller allocates every buffer, including workspaces.
 *    The library allocates no device memory, keeps no pointer after a call
 *    returns, and does not synchronise: all work is enqueued on `stream`
 *    (a cudaStream_t, NULL = the legacy default stream).
 *  - Errors: 0 (CHAIN_OK) on success, a negative chain_status_t otherwise.
 *    Argument errors are detected on the host before anything is enqueued.
 *    CHAIN_ERR_CUDA keeps the CUDA error code, readable through
 *    chain_last_cuda_error().  Device-side bounded waits that expire (a
 *    pipeline that stopped making progress) do not trap: the kernel stops,
 *    records the event in a device status word, and chain_check() returns
 *    CHAIN_ERR_TIMEOUT after synchronising the stream.
 *  - Thread safety: calls may be issued concurrently from several host
 *    threads; the only global state is a per-device cache of attributes
 *    guarded by a mutex.
 *  - Device resets: the per-device cache holds device addresses of the
 *    library's own status word (and of chain_bwd_noalloc's scratch array),
 *    looked up on the first call on each device.  A device reset
 *    (cudaDeviceReset) makes them stale: do not call the library on a device
 *    after resetting it in the same process.
 */
#ifndef CHAIN_GB300_H
#define CHAIN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CHAIN_OK = 0,
  CHAIN_ERR_ARG = -1,     /* null pointer, shape/stride mismatch, misalignment, bad size */
  CHAIN_ERR_DTYPE = -2,   /* element type not supported for this call */
  CHAIN_ERR_DEVICE = -3,  /* current device is not compute capability 10.3 */
  CHAIN_ERR_CUDA = -4,    /* a CUDA runtime/driver call failed */
  CHAIN_ERR_TIMEOUT = -5, /* a bounded device-side wait expired */
  CHAIN_ERR_UNSUPPORTED = -6, /* valid request this library does not implement */
  CHAIN_ERR_SCRATCH_LIMIT = -7 /* problem needs more than CHAIN_NOALLOC_SCRATCH_BYTES */
} chain_status_t;

/* CHAIN_E4M3: 8-bit float, 1 sign, 4 exponent (bias 7) and 3 mantissa bits,
 * no infinities, S.1111.111 = NaN; largest finite value 448. */
typedef enum { CHAIN_BF16 = 0, CHAIN_F32 = 1, CHAIN_E4M3 = 2 } chain_dtype_t;

typedef enum {
  CHAIN_F_IDENTITY = 0,  /* O = (A B) C */
  CHAIN_F_SOFTMAX = 1,   /* O = softmax_row(scale * A B) C; attention */
  CHAIN_F_GELU_TANH = 2  /* O = gelu_tanh(A B) C; MLP chain */
} chain_f_t;

typedef enum { CHAIN_MASK_NONE = 0, CHAIN_MASK_CAUSAL = 1 } chain_mask_t;

typedef struct {
  void *ptr;          /* device address of element [0, 0, ...] */
  int32_t dtype;      /* chain_dtype_t */
  int32_t ndim;       /* 1..4 */
  int64_t shape[4];   /* elements, outermost first */
  int64_t stride[4];  /* elements; stride[ndim-1] must be 1 */
} chain_tensor_t;

/*
 * chain_fwd -- O = f(A B) C  (FITEE abstract: the unit METP partitions).
 *
 * f = CHAIN_F_SOFTMAX (attention):
 *   A = Q [BH][n][d], B = K [BH][n][d] (passed untransposed; the product is
 *   Q K^T), C = V [BH][n][d]; 3-D, or 4-D [B][H][n][d] (B*H folded).
 *   Grouped-query attention (bf16): K and V may have fewer heads, [BHkv][n][d]
 *   with BH a multiple of BHkv; query head h then attends K/V head
 *   h / (BH / BHkv) (for 4-D, H a multiple of Hkv keeps each group within
 *   one batch entry).
 *   n >= 1.  bf16 in -> O bf16, d in {64, 128}; O is accumulated from the
 *   compensated pair P_hi + P_lo (bf16 head and residual of P) so the only
 *   bf16 rounding is the output's.  f32 in -> O f32, d = 64 only (else
 *   CHAIN_ERR_UNSUPPORTED): a small full-precision variant whose tensor-core
 *   products split every operand into tf32 head + remainder (3 MMAs).
 *   S = scale * Q K^T (scale applied in fp32 to the fp32 product);
 *   mask CAUSAL keeps keys j <= i on global positions (AutoSP 2.A item 4).
 *   LSE [BH][n] f32 (required): LSE_i = ln sum_j exp(S_ij), natural log,
 *   scale included.  O [BH][n][d].
 * f = CHAIN_F_GELU_TANH or CHAIN_F_IDENTITY (MLP chain):
 *   A [M][K], B [K][N], C [N][P] row-major bf16; O [M][P] bf16; LSE NULL;
 *   scale and mask ignored (mask must be NONE).  Requires M and N
 *   multiples of 128, K a multiple of 64, P a multiple of 256 (else
 *   CHAIN_ERR_UNSUPPORTED).  The [M][N] intermediate is held on chip in
 *   128 x 128 chunks and never written to memory.  fp32 accumulation; the
 *   intermediate enters the second product as bf16 H_hi + bf16 residual
 *   H_lo, so its rounding error is ~2^-16 relative.
 */
int chain_fwd(const chain_tensor_t *A, const chain_tensor_t *B,
              const chain_tensor_t *C, int f, int mask, float scale,
              chain_tensor_t *O, chain_tensor_t *LSE, void *stream);

/*
 * chain_fwd_f16h -- the MLP chain O = f(A B) C of chain_fwd (f =
 * CHAIN_F_GELU_TANH or CHAIN_F_IDENTITY; the unit of "Memory-efficient
 * tensor parallelism", FITEE 10.1631/FITEE.2400602, abstract, with the
 * intermediate kept on chip as the AutoSP write-up, section 2.B, requires),
 * with the intermediate H = f(A B) entering the second product as ONE f16
 * tile (11 significant bits) against an f16 copy of C, instead of the bf16
 * pair H_hi + H_lo against bf16 C: one product per hidden chunk instead of
 * two, and half the on-chip traffic of the intermediate.
 *   A [M][K], B [K][N], C [N][P], O [M][P]: 2-D, row-major, contiguous
 *   rows, bf16.  M a multiple of 128, K and N multiples of 64, P = 512, 768
 *   or 1024 (the clusters of 2 to 4 thread blocks that share H), else
 *   CHAIN_ERR_UNSUPPORTED.
 *   workspace  at least chain_fwd_f16h_workspace_size(C) bytes, 16-byte
 *              aligned: C in f16 (2 * N * P bytes) and its scale factor.
 * The copy of C carries one power-of-two scale that puts its largest |c| in
 * [2^14, 2^15); every value is then exact in f16 except values below 2^-31
 * of that maximum (error at most 2^-39 of it).  The epilogue undoes the
 * scale.  H must stay within f16's finite range (|H| <= 65504): a value
 * beyond it is reported by the next chain_check() as CHAIN_ERR_ARG and the
 * result is then not valid.  Values of |H| below 2^-14 are f16 subnormals
 * (absolute error at most 2^-25).  Error otherwise: one bf16 rounding of O
 * plus H's f16 rounding (~2^-12 relative, random over the hidden index).
 * Returns CHAIN_ERR_DTYPE unless bf16, CHAIN_ERR_ARG for a shape, stride,
 * alignment or workspace violation or another f.  Asynchronous on `stream`.
 * chain_fwd_f16h_workspace_size returns 0 for an invalid C.
 */
size_t chain_fwd_f16h_workspace_size(const chain_tensor_t *C);
int chain_fwd_f16h(const chain_tensor_t *A, const chain_tensor_t *B, const chain_tensor_t *C,
                   int f, chain_tensor_t *O, void *workspace, size_t ws_bytes, void *stream);

/*
 * chain_bwd_workspace_size -- bytes of device workspace chain_bwd needs for
 * these shapes, rounded up to 256 bytes.  A and C of one shape mean the
 * softmax chain: the fp32 [BH][n] row term D.  2-D A and C of different
 * shapes mean the MLP chain (A = X [M][K], C = W2 [N][P]): H and dT, [M][N]
 * bf16 each.  Returns 0 for invalid descriptors.
 */
size_t chain_bwd_workspace_size(const chain_tensor_t *A, const chain_tensor_t *C);

/*
 * chain_bwd_workspace_size_f -- the same, with the chain named by f, for the
 * MLP shapes chain_bwd_workspace_size cannot tell apart (X and W2 of one
 * shape).  Returns 0 for invalid descriptors or f.
 */
size_t chain_bwd_workspace_size_f(const chain_tensor_t *A, const chain_tensor_t *C, int f);

/*
 * chain_bwd -- gradients of the softmax chain (attention backward).
 *   Inputs: dO, Q (A), K (B), V (C), O [BH][n][d] bf16 and LSE [BH][n] f32
 *   as produced by chain_fwd (or chain_fwd_f16pv) with the same f, mask and
 *   scale.  Only
 *   f = CHAIN_F_SOFTMAX with bf16 and d in {64, 128} is supported.
 *   Outputs: dQ (dA), dK (dB), dV (dC) [BH][n][d] bf16.  With grouped-query
 *   attention K, V, dK, dV are [BHkv][n][d] and dK, dV sum over the query
 *   heads of each group.
 *   S and P are recomputed per tile from LSE ("recompute, don't store",
 *   AutoSP 2.B); D_i = sum_e dO_ie O_ie.  dK, dV come from one pass over
 *   the key blocks and dQ from a second over the query tiles, each
 *   accumulating on chip: no atomics, results are deterministic.
 *   workspace: device buffer of at least chain_bwd_workspace_size() bytes,
 *   16-byte aligned, contents ignored on entry.
 *
 * f = CHAIN_F_GELU_TANH or CHAIN_F_IDENTITY: gradients of the MLP chain
 *   O = f(X W1) W2 ("Memory-efficient tensor parallelism", abstract), the
 *   intermediate recomputed from X and W1 instead of kept from the forward
 *   (AutoSP, section 2.B):
 *     T = X W1, H = f(T), dH = dO W2^T, dT = dH * f'(T),
 *     dW2 = H^T dO,  dX = dT W1^T,  dW1 = X^T dT.
 *   dO [M][P], A = X [M][K], B = W1 [K][N], C = W2 [N][P] bf16, dense
 *   row-major; O, LSE and scale are ignored (may be NULL / any); mask must be
 *   CHAIN_MASK_NONE.  Outputs dA = dX [M][K], dB = dW1 [K][N], dC = dW2
 *   [N][P] bf16.  H and dT go through the workspace as bf16 (fp32
 *   accumulation everywhere else).  CHAIN_ERR_UNSUPPORTED unless M % 128 ==
 *   0 and K, N, P are multiples of 256.
 */
int chain_bwd(const chain_tensor_t *dO, const chain_tensor_t *A,
              const chain_tensor_t *B, const chain_tensor_t *C,
              const chain_tensor_t *O, const chain_tensor_t *LSE, int f,
              int mask, float scale, chain_tensor_t *dA, chain_tensor_t *dB,
              chain_tensor_t *dC, void *workspace, size_t ws_bytes,
              void *stream);

/*
 * chain_bwd_noalloc -- chain_bwd for callers that cannot allocate device
 * memory.  (An addition of this library: the method's write-ups have no
 * counterpart.)
 *
 * chain_bwd needs a caller-provided scratch workspace.  Some callers have
 * no way to provide one: a host program whose pool allocator reserved the
 * device's memory up front and exposes no C handle to it, a plugin that must
 * not grow the host process's device footprint after start-up, or a
 * latency-bound loop that cannot afford cudaMalloc/cudaFree, which may
 * synchronise the whole device.  This entry point takes the same arguments
 * as chain_bwd minus the workspace and uses instead a fixed scratch array
 * compiled into the library: CHAIN_NOALLOC_SCRATCH_BYTES (32 MiB) of device
 * memory that every GPU which loads the library holds until the process
 * exits.  It never calls cudaMalloc, cudaFree or any allocating routine.
 *
 * Limit: chain_bwd_workspace_size_f(A, C, f) must not exceed
 * CHAIN_NOALLOC_SCRATCH_BYTES, else the call returns CHAIN_ERR_SCRATCH_LIMIT
 * before enqueuing anything.  For the attention backward that is
 * BH * n <= 8,388,608 query rows (4 bytes each); for the MLP backward
 * M * N <= 8,388,608 elements of X W1 (H and dT, 2 bytes each), e.g. M = 2048
 * rows at N = 4096 hidden units.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture begins.  The address is kept for the life of the
 * process: after a device reset (cudaDeviceReset) the array is a new one and
 * the kept address is stale, so like the rest of this library (see
 * "Device resets" above) this entry point must not be called after a reset.
 * All calls on a device share the one array and leave their partial
 * results in it; each call re-initialises what it reads.  Calls whose
 * execution overlaps on the GPU (different streams, or host threads without
 * ordering) race on the array and give wrong gradients: order them.
 */
#define CHAIN_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int chain_bwd_noalloc(const chain_tensor_t *dO, const chain_tensor_t *A,
                      const chain_tensor_t *B, const chain_tensor_t *C,
                      const chain_tensor_t *O, const chain_tensor_t *LSE, int f,
                      int mask, float scale, chain_tensor_t *dA,
                      chain_tensor_t *dB, chain_tensor_t *dC, void *stream);

/*
 * chain_fwd_sp -- softmax attention read from, and written back to, the
 * Ulysses sequence-shard layout: the all-to-all relayout of Q, K and V, the
 * attention of one head group over the whole sequence, and the inverse
 * relayout of O, in one kernel ("Ulysses Sequence Parallelism", "Contexte
 * Technique" and "Analyse et Implications"; the unit is the O = f(A B) C of
 * "Memory-efficient tensor parallelism", FITEE 10.1631/FITEE.2400602).  The
 * head-major copies never exist in memory: the tensor-core loads read 128-row
 * boxes straight out of the shards.
 *   Q, K, V, O  [p][n_loc][H][d] bf16: shard s holds positions
 *               [s*n_loc, (s+1)*n_loc); d = 64 or 128, contiguous; other
 *               strides multiples of 16 bytes; 16-byte aligned.  O may have
 *               its own strides.
 *   head_group  g in [0, p): the call attends heads [g*H/p, (g+1)*H/p) over
 *               all n = p*n_loc positions and writes exactly those heads of
 *               O; the other heads of O are left untouched.
 *   mask, scale as for chain_fwd with f = CHAIN_F_SOFTMAX.
 *   LSE         [H/p][n] fp32, natural log, head-major (h relative to the
 *               group).
 * Same results, bit for bit, as sp_relayout of Q, K and V, then chain_fwd,
 * then sp_relayout_inverse of O.  Returns CHAIN_ERR_UNSUPPORTED unless n_loc
 * is a multiple of 128 (a tile must not straddle two shards), CHAIN_ERR_ARG
 * for a shape, stride or alignment violation, CHAIN_ERR_DTYPE unless bf16.
 * Asynchronous on `stream`.
 */
int chain_fwd_sp(const chain_tensor_t *Q, const chain_tensor_t *K,
                 const chain_tensor_t *V, int p, int head_group, int mask,
                 float scale, chain_tensor_t *O, chain_tensor_t *LSE,
                 void *stream);

/*
 * chain_fwd_sp_f16pv -- chain_fwd_sp with P V taken as one f16 product, as
 * chain_fwd_f16pv does: Q, K read from and O written to the Ulysses
 * sequence shards [p][n_loc][H][d] bf16 (same rules as chain_fwd_sp); the
 * f16 copy of the group's V heads, head-major, is written by a pre-pass that
 * reads the shards, so V's relayout is part of its re-encoding.
 *   workspace  at least chain_fwd_sp_f16pv_workspace_size(V, p) bytes,
 *              16-byte aligned.
 * Same results, bit for bit, as sp_relayout of Q, K and V, then
 * chain_fwd_f16pv, then sp_relayout_inverse of O.  Errors as chain_fwd_sp,
 * plus CHAIN_ERR_ARG for a missing or short workspace.
 */
size_t chain_fwd_sp_f16pv_workspace_size(const chain_tensor_t *V, int p);
int chain_fwd_sp_f16pv(const chain_tensor_t *Q, const chain_tensor_t *K,
                       const chain_tensor_t *V, int p, int head_group, int mask,
                       float scale, chain_tensor_t *O, chain_tensor_t *LSE,
                       void *workspace, size_t ws_bytes, void *stream);

/*
 * chain_fwd_varlen -- softmax attention over a batch of sequences of
 * different lengths packed end to end (the long-sequence regime of "Ulysses
 * Sequence Parallelism", "Contexte Technique", batches sequences of uneven
 * length; the unit is the O = f(A B) C of "Memory-efficient tensor
 * parallelism", FITEE 10.1631/FITEE.2400602).  Each sequence attends to
 * itself only.
 *   Q, O        [total][H][d] bf16;  K, V  [total][Hkv][d] bf16 (Hkv divides
 *               H: grouped-query attention as in chain_fwd); d = 64 or 128,
 *               contiguous; row and head strides multiples of 16 bytes.
 *   cu_seqlens  DEVICE int32 [batch + 1]: sequence b is rows
 *               [cu_seqlens[b], cu_seqlens[b+1]); nondecreasing, last =
 *               total.  Offsets are clamped to [0, total] on the device.
 *   max_seqlen  at least the longest sequence; a longer sequence is not
 *               computed and the next chain_check() returns CHAIN_ERR_ARG.
 *   mask, scale as for chain_fwd with f = CHAIN_F_SOFTMAX (causal positions
 *               count from each sequence's start).
 *   LSE         [H][total] fp32, natural log.
 * Rows of each sequence are computed exactly as chain_fwd computes that
 * sequence alone.  Returns CHAIN_ERR_UNSUPPORTED when H * batch *
 * ceil(max_seqlen / 256) exceeds 2^31 - 1 (one thread block per head,
 * sequence and pair of 128-row query tiles).  Asynchronous on `stream`.
 */
int chain_fwd_varlen(const chain_tensor_t *Q, const chain_tensor_t *K,
                     const chain_tensor_t *V, const int32_t *cu_seqlens, int batch,
                     int max_seqlen, int mask, float scale, chain_tensor_t *O,
                     chain_tensor_t *LSE, void *stream);

/*
 * chain_bwd_varlen -- gradients of chain_fwd_varlen (softmax attention over
 * sequences packed end to end), S and P recomputed from LSE as in chain_bwd.
 *   dO, Q, O, dQ  [total][H][d] bf16, one set of strides for the four;
 *   K, V, dK, dV  [total][Hkv][d] bf16, one set of strides for the four
 *                 (grouped-query attention: dK, dV sum over each group);
 *   LSE           [H][total] fp32 as written by chain_fwd_varlen (dense);
 *   cu_seqlens, batch, max_seqlen, mask, scale as for chain_fwd_varlen (a
 *                 sequence longer than max_seqlen is not computed and the
 *                 next chain_check() returns CHAIN_ERR_ARG).
 *   workspace     at least 4 * H * total bytes rounded up to 256, 16-byte
 *                 aligned (chain_bwd_workspace_size(Q, Q) returns it).
 * Each sequence's gradients are those chain_bwd gives for it alone.
 * Returns CHAIN_ERR_UNSUPPORTED when H * batch * ceil(max_seqlen / 128)
 * exceeds 2^31 - 1 (one thread block per head, sequence and 128-row tile).
 */
int chain_bwd_varlen(const chain_tensor_t *dO, const chain_tensor_t *Q,
                     const chain_tensor_t *K, const chain_tensor_t *V,
                     const chain_tensor_t *O, const chain_tensor_t *LSE,
                     const int32_t *cu_seqlens, int batch, int max_seqlen, int mask,
                     float scale, chain_tensor_t *dQ, chain_tensor_t *dK,
                     chain_tensor_t *dV, void *workspace, size_t ws_bytes, void *stream);

/*
 * chain_fwd_f16pv -- softmax attention forward, the same operation as
 * chain_fwd with f = CHAIN_F_SOFTMAX on bf16 inputs (the unit O = f(A B) C
 * of "Memory-efficient tensor parallelism", FITEE 10.1631/FITEE.2400602,
 * abstract, tiled as in "Ulysses Sequence Parallelism", "Contexte
 * Technique"), with the second product P V taken as ONE f16 tensor-core
 * product instead of chain_fwd's compensated bf16 pair: P enters as f16 (11
 * significant bits) and V as an f16 copy in the caller's workspace.
 *   Q [BH][n][d], K, V [BHkv][n][d] bf16 (BHkv dividing BH), O [BH][n][d]
 *   bf16, LSE [BH][n] fp32; d = 64 or 128; 3-D or 4-D (B*H folded); row and
 *   head pitches multiples of 16 bytes.  mask, scale as for chain_fwd.
 *   workspace  at least chain_fwd_f16pv_workspace_size(Q, V) bytes, 16-byte
 *              aligned: V in f16 (2 * BHkv * n * d bytes) and per-head
 *              scale factors.
 * The copy of V carries one power-of-two scale per K/V head that puts the
 * head's largest |v| in [2^14, 2^15); every value is then exact in f16 except
 * values below 2^-31 of that maximum, rounded with an error of at most 2^-39
 * of it.  The epilogue undoes the scale.  Error: one bf16 rounding of O plus
 * P's f16 rounding (~2^-12 relative, random over the keys).  Returns
 * CHAIN_ERR_DTYPE unless bf16, CHAIN_ERR_ARG for a shape, stride, alignment
 * or workspace violation, CHAIN_ERR_UNSUPPORTED for more than 65,535 K/V
 * heads.  Asynchronous on `stream`.
 */
size_t chain_fwd_f16pv_workspace_size(const chain_tensor_t *Q, const chain_tensor_t *V);
int chain_fwd_f16pv(const chain_tensor_t *Q, const chain_tensor_t *K,
                    const chain_tensor_t *V, int mask, float scale, chain_tensor_t *O,
                    chain_tensor_t *LSE, void *workspace, size_t ws_bytes, void *stream);

/*
 * chain_fwd_varlen_f16pv -- chain_fwd_varlen (sequences of different lengths
 * packed end to end, each attending to itself only) with P V taken as one
 * f16 product, as chain_fwd_f16pv does.
 *   Q, K, V, O, LSE, cu_seqlens, batch, max_seqlen, mask, scale  as for
 *               chain_fwd_varlen.
 *   workspace  at least chain_fwd_varlen_f16pv_workspace_size(V) bytes,
 *              16-byte aligned: V in f16, head-major [Hkv][total][d], and
 *              one power-of-two scale per K/V head (taken over all of the
 *              batch's rows of that head, as chain_fwd_f16pv takes it over
 *              all of a head's rows).
 * Error bound as for chain_fwd_f16pv.  LSE is bit for bit what
 * chain_fwd_f16pv writes for each sequence alone, and so is O whenever no
 * nonzero |v| of a head is below 2^-31 of that head's largest and the
 * largest is at least 2^-80 (the per-head scale, a power of two, then
 * changes no rounding).  Errors as chain_fwd_varlen,
 * plus CHAIN_ERR_ARG for a missing or short workspace and
 * CHAIN_ERR_UNSUPPORTED for more than 65,535 K/V heads;
 * chain_fwd_varlen_f16pv_workspace_size returns 0 for a V it cannot take.
 */
size_t chain_fwd_varlen_f16pv_workspace_size(const chain_tensor_t *V);
int chain_fwd_varlen_f16pv(const chain_tensor_t *Q, const chain_tensor_t *K,
                           const chain_tensor_t *V, const int32_t *cu_seqlens, int batch,
                           int max_seqlen, int mask, float scale, chain_tensor_t *O,
                           chain_tensor_t *LSE, void *workspace, size_t ws_bytes,
                           void *stream);

/*
 * chain_fwd_fp8 -- softmax attention, O = softmax(scale Q K^T) (v_scale V),
 * on 8-bit float inputs: the unit O = f(A B) C of "Memory-efficient tensor
 * parallelism" (FITEE 10.1631/FITEE.2400602, abstract) with f = row softmax,
 * read from e4m3 tensors.  The pages define no 8-bit variant: this entry
 * stores the three inputs in half the bytes of bf16 and runs the Q K^T
 * product at the 8-bit tensor-core rate.
 *   Q  [BH][n][128], K, V  [BHkv][n][128] CHAIN_E4M3 (3-D, or 4-D with B*H
 *      folded), BHkv dividing BH (grouped-query attention as in chain_fwd);
 *      rows contiguous, row and head strides multiples of 16 bytes.
 *   scale    multiplies Q K^T in fp32 (fold Q's and K's dequantisation
 *            factors into it); > 0 and finite.
 *   v_scale  V's dequantisation factor, applied to O in fp32; finite.
 *   O        [BH][n][128] bf16;  LSE [BH][n] fp32, natural log, scale included.
 *   mask     as for chain_fwd.
 *   workspace  at least chain_fwd_fp8_workspace_size(V) bytes (2 * BHkv * n *
 *            128, rounded up to 256), 16-byte aligned: V re-encoded as f16
 *            (exactly: every e4m3 value is an f16 value times 2^8).
 * Arithmetic: the Q K^T products of e4m3 values are exact, accumulated in
 * fp32; P enters the P V product as f16 (11 significant bits) with V's exact
 * f16 copy; fp32 accumulation; one bf16 rounding of O.  Inputs must be finite
 * (a NaN code is read as +-480).  Returns CHAIN_ERR_DTYPE unless Q, K, V are
 * e4m3 and O bf16, CHAIN_ERR_UNSUPPORTED for d != 128, CHAIN_ERR_ARG for a
 * shape, stride, alignment or workspace violation.  Asynchronous on `stream`.
 */
size_t chain_fwd_fp8_workspace_size(const chain_tensor_t *V);
int chain_fwd_fp8(const chain_tensor_t *Q, const chain_tensor_t *K,
                  const chain_tensor_t *V, int mask, float scale, float v_scale,
                  chain_tensor_t *O, chain_tensor_t *LSE, void *workspace,
                  size_t ws_bytes, void *stream);

/*
 * sp_relayout -- Ulysses sequence shards -> head-major for one head group
 * ("Ulysses Sequence Parallelism", "Contexte Technique": every position of
 * the sequence, a subset of the heads).
 *   shards [p][n_loc][H][d]: shard s holds positions [s*n_loc, (s+1)*n_loc).
 *   out    [H/p][p*n_loc][d]: out[h][s*n_loc+t][e] = shards[s][t][g*H/p+h][e]
 *   with g = head_group in [0, p).  Bit-exact copy of any 1-, 2- or 4-byte
 *   element type; d * element size must be a multiple of 16 bytes.
 *   Size limit: the shards may hold at most 2^32 - 2^22 - 1 16-byte vectors
 *   (p * n_loc * H * d * element size / 16; 64 GiB less 64 MiB), else
 *   CHAIN_ERR_ARG before anything is enqueued.
 */
int sp_relayout(const chain_tensor_t *shards, int p, int head_group,
                chain_tensor_t *out, void *stream);

/*
 * sp_relayout_inverse -- head-major -> sequence shards (the second
 * exchange of the Ulysses layer, "Analyse et Implications"):
 *   shards[s][t][g*H/p+h][e] = in[h][s*n_loc+t][e]; the other heads of
 *   `shards` are left untouched.  Same element, alignment and size rules.
 */
int sp_relayout_inverse(const chain_tensor_t *in, int p, int head_group,
                        chain_tensor_t *shards, void *stream);

/*
 * chain_check -- synchronise `stream`, then read and clear the device
 * status word.  Returns CHAIN_ERR_TIMEOUT if a bounded wait expired in any
 * kernel since the last check, CHAIN_ERR_ARG if a kernel met an argument only
 * it could check (chain_fwd_varlen: a sequence longer than max_seqlen),
 * CHAIN_ERR_CUDA on a CUDA error, else 0.
 * `detail` (may be NULL) receives the code of the wait site that expired.
 */
int chain_check(void *stream, int *detail);

/*
 * chain_set_wait_limit_ns -- limit of every device-side bounded wait
 * (default 2e9 ns).  Takes effect for launches issued afterwards.
 */
void chain_set_wait_limit_ns(uint64_t ns);

/*
 * chain_set_timing_events -- measurement hook.  While set (count > 0), every
 * chain_fwd / chain_bwd / sp_relayout call issued from the calling host
 * thread records events[k] (cudaEvent_t, k < count) on its stream at the
 * k-th boundary of its main kernels: events[0] just before the first main
 * kernel, events[1] just after it, events[2] after the second (the
 * backward has two main kernels: dK/dV, then dQ; its small preprocess runs
 * before events[0]).  The f16 forms count their pre-pass as the first
 * main kernel, except chain_fwd_f16h: its main kernel may start while the
 * pre-pass still runs, so it records events[0] before the pre-pass and
 * events[1] after the main kernel only.  Boundaries beyond count are not
 * recorded.  Pass NULL, 0 to clear.  At most 4 events; events are owned by
 * the caller.
 */
void chain_set_timing_events(void *const *events, int count);

/*
 * chain_selftest_wait_timeout -- launches one CTA that waits on a barrier
 * nothing will ever complete, with the bounded wait of every kernel here,
 * and returns after the wait expires.  chain_check() then reports
 * CHAIN_ERR_TIMEOUT.  Exercises the failure path without faulting the GPU.
 */
int chain_selftest_wait_timeout(uint64_t limit_ns, void *stream);

/*
 * chain_umma_selftest -- diagnostic of the tensor-core building block:
 * D[128][N] (f32) = A[128][K] . B, with A [128][K] bf16 row-major and B
 * either [N][K] (flags bit 0 clear, i.e. D = A B^T) or [K][N] (bit 0 set),
 * loaded by TMA into 128-byte-swizzled shared memory and multiplied by
 * tcgen05.mma into tensor memory.  With flags bit 1 set, A is instead
 * written into tensor memory by the threads (row i in lane i, two bf16 per
 * column) and read from there by the MMA.  K in {64, 128, 192, 256},
 * N in {64, 128}; all pointers are device addresses.
 */
int chain_umma_selftest(const void *A, const void *B, float *D, int N, int K,
                        int flags, void *stream);

/* Static description of a status code. */
const char *chain_status_string(int status);

/* CUDA error code of the most recent CHAIN_ERR_CUDA on this thread. */
int chain_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* CHAIN_GB300_H */
