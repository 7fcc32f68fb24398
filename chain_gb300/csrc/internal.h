// internal.h -- host-side declarations shared by the translation units of
// the library (launchers and tensor-map helpers).  Not part of the ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sm103.cuh"

namespace chain {

// Encodes a 2-D/3-D bf16 or f32 tiled tensor map with 128-byte swizzle.
// dims/strides are innermost first; strides (bytes) exclude the innermost.
// Returns cudaSuccess or cudaErrorInvalidValue on encode failure.
cudaError_t make_tmap(CUtensorMap *map, CUtensorMapDataType dt, int rank, const void *base,
                      const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box);

struct AttnFwdArgs {
  const void *Q, *K, *V;  // [BH][n][d]
  int64_t q_sbh, q_srow, k_sbh, k_srow, v_sbh, v_srow;
  void *O;
  int64_t o_sbh, o_srow;
  float *LSE;
  int64_t lse_sbh;
  int BH, n, d, causal;
  int BHkv;  // K/V heads; BH / BHkv query heads share each (grouped-query attention)
  float scale;
  // Sequence split into n / n_loc shards: position s*n_loc + t lives at
  // s*x_sshard + t*x_srow (elements).  n_loc = n for one contiguous run.
  int n_loc;
  int64_t q_sshard, k_sshard, v_sshard, o_sshard;
  // Variable-length batch: device int32 [nbatch + 1] row offsets into the
  // packed rows (n = total rows), or null.
  const int *cu_seqlens;
  int nbatch, max_seqlen;
  float v_scale = 1.0f;  // e4m3 inputs: the factor V's codes are multiplied by
};

cudaError_t launch_attn_fwd_bf16(const AttnFwdArgs &a, const WaitCfg &wc, cudaStream_t st);
// e4m3 Q, K, V (d = 128, dense); v16 = 2 x BHkv x n x 128 bytes of workspace
// (16-byte aligned) for the f16 copy of V.
cudaError_t launch_attn_fwd_fp8(const AttnFwdArgs &a, void *v16, const WaitCfg &wc,
                               cudaStream_t st);
// bf16 Q, K, V with P V as one f16 product (V re-encoded in f16 with a
// power-of-two scale per K/V head); ws = attn_fwd_pv16_workspace bytes,
// 16-byte aligned.  Head-major or sequence-shard layouts (n_loc < n), d = 64
// or 128.
size_t attn_fwd_pv16_workspace(int BHkv, int n, int d);
cudaError_t launch_attn_fwd_pv16(const AttnFwdArgs &a, void *ws, const WaitCfg &wc,
                                 cudaStream_t st);
cudaError_t launch_attn_fwd_f32(const AttnFwdArgs &a, const WaitCfg &wc, cudaStream_t st);

struct AttnBwdArgs {
  const void *Q, *K, *V, *O, *dO;  // bf16 [BH][n][d] (K, V: [BHkv][n][d]), row stride d
  const float *LSE;                // [BH][n]
  void *dQ, *dK, *dV;              // bf16, shaped as Q, K, V
  float *Dvec;                     // fp32 [BH][n] workspace
  int BH, n, d, causal;
  int BHkv;  // K/V heads (grouped-query attention: BH / BHkv query heads each)
  float scale;
  // element strides: Q, O, dO, dQ (row, head); K, V, dK, dV (row, head);
  // LSE and D head stride (rows contiguous)
  int64_t q_srow, q_shead, kv_srow, kv_shead, l_shead;
  // Variable-length batch: device int32 [nbatch + 1] row offsets into the
  // packed rows (n = total rows), or null.
  const int *cu_seqlens;
  int nbatch, max_seqlen;
};
cudaError_t launch_attn_bwd(const AttnBwdArgs &a, const WaitCfg &wc, cudaStream_t st);

struct MlpBwdArgs {
  const void *X, *W1, *W2, *dO;  // [M][K], [K][N], [N][P], [M][P] bf16 row-major
  void *dX, *dW1, *dW2;          // [M][K], [K][N], [N][P] bf16
  void *workspace;               // H and dT, [M][N] bf16 each
  int M, K, N, P, gelu;
};
cudaError_t launch_mlp_bwd(const MlpBwdArgs &a, const WaitCfg &wc, cudaStream_t st);

struct MlpArgs {
  const void *X, *W1, *W2;  // [M][K], [K][N], [N][P] bf16 row-major
  void *O;                  // [M][P] bf16
  int M, K, N, P;
  int gelu;                 // 1 = gelu_tanh, 0 = identity
};
cudaError_t launch_mlp_chain(const MlpArgs &a, const WaitCfg &wc, cudaStream_t st);
// The intermediate as one f16 tile against an f16 copy of W2 (in `ws`, at
// least mlp_f16h_workspace(N, P) bytes); cluster shapes only (P = 512, 768
// or 1024, N a multiple of 64), else cudaErrorNotSupported.
size_t mlp_f16h_workspace(int64_t N, int64_t P);
cudaError_t launch_mlp_chain_f16h(const MlpArgs &a, void *ws, const WaitCfg &wc,
                                  cudaStream_t st);

cudaError_t launch_relayout(const void *in, void *out, int64_t p, int64_t n_loc, int64_t H,
                            int64_t row_bytes, int64_t g, int inverse, cudaStream_t st);
// The relayout kernel indexes 16-byte vectors in 32 bits with a grid-stride
// loop of at most kRelayoutMaxGrid blocks x 256 threads x 4 vectors per step.
// Its counter may run one whole step past the last vector before the loop
// ends, so the sequence-major side's vector count plus one step must stay
// below 2^32 (checked before launch).
constexpr int64_t kRelayoutMaxGrid = 4096;
constexpr int64_t kRelayoutStepVectors = kRelayoutMaxGrid * 256 * 4;
inline bool relayout_fits_32bit(int64_t seq_vectors) {
  return seq_vectors > 0 && seq_vectors + kRelayoutStepVectors < (int64_t(1) << 32);
}

// Keeps `e` as the thread's last CUDA error and returns CHAIN_ERR_CUDA.
int record_cuda_error(cudaError_t e);

// Measurement hook (chain_set_timing_events): record the calling thread's
// event k, if set, at the k-th main-kernel boundary of a call.
void timing_mark(cudaStream_t st, int k);

cudaError_t launch_wait_selftest(const WaitCfg &wc, cudaStream_t st);
cudaError_t launch_umma_selftest(const void *A, const void *B, float *D, int N, int K,
                                 int flags, const WaitCfg &wc, cudaStream_t st);

}  // namespace chain
