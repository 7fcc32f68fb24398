// relayout.cu -- Ulysses sequence-shard <-> head-major permutation.
//
// "Ulysses Sequence Parallelism", "Contexte Technique": the sequence is
// split into chunks, and after the exchange every device holds all
// positions for a subset of heads.  The device-local half of that exchange
// for head group g (Hl = H/p heads, positions pos = s*n_loc + t):
//   forward:  out[h][pos][:] = in[pos][g*Hl + h][:]    (in = [p][n_loc][H][d])
//   inverse:  out[pos][g*Hl + h][:] = in[h][pos][:]
// Since shard s holds the contiguous positions [s*n_loc, (s+1)*n_loc), the
// shard index folds into pos and the map is a pure (pos, h) transpose of
// row-sized runs.  The kernel moves 16-byte vectors, iterating in the
// order of the side whose runs are longer (Hl rows of one position are
// contiguous there), so both loads and stores stay coalesced.  Bits are
// copied unchanged.
#include "internal.h"

namespace chain {
namespace {

constexpr int THREADS = 256;
constexpr int UNROLL = 4;

// Index i enumerates (pos, h, e) with e fastest: e in [0, vrow), h in
// [0, Hl).  `seq` is the sequence-major side [pos][H][vrow] (offset by the
// group), `hm` the head-major side [Hl][N][vrow].
__global__ void __launch_bounds__(THREADS)
    relayout_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, uint32_t N,
                    uint32_t H, uint32_t Hl, uint32_t vrow, uint32_t goff, uint32_t total,
                    int inverse) {
  const uint32_t stride = gridDim.x * THREADS;
  for (uint32_t base = blockIdx.x * THREADS + threadIdx.x; base < total;
       base += stride * UNROLL) {
    uint4 v[UNROLL];
    uint32_t didx[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const uint32_t i = base + u * stride;
      if (i < total) {
        const uint32_t e = i % vrow;
        const uint32_t r = i / vrow;
        const uint32_t h = r % Hl;
        const uint32_t pos = r / Hl;
        const uint32_t seq_i = (pos * H + goff + h) * vrow + e;
        const uint32_t hm_i = (h * N + pos) * vrow + e;
        const uint32_t s_i = inverse ? hm_i : seq_i;
        didx[u] = inverse ? seq_i : hm_i;
        v[u] = __ldcs(src + s_i);
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const uint32_t i = base + u * stride;
      if (i < total) __stcs(dst + didx[u], v[u]);
    }
  }
}

}  // namespace

cudaError_t launch_relayout(const void *in, void *out, int64_t p, int64_t n_loc, int64_t H,
                            int64_t row_bytes, int64_t g, int inverse, cudaStream_t st) {
  const int64_t Hl = H / p;
  const int64_t N = p * n_loc;
  const int64_t vrow = row_bytes / 16;
  const int64_t total = N * Hl * vrow;
  // 32-bit index arithmetic covers both sides (the sequence-major side has
  // N*H*vrow vectors), with room for the loop counter's last step.
  static_assert(THREADS * UNROLL * kRelayoutMaxGrid == kRelayoutStepVectors, "step size");
  if (!relayout_fits_32bit(N * H * vrow) || total == 0) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t want = (total + (int64_t)THREADS * UNROLL - 1) / ((int64_t)THREADS * UNROLL);
  int64_t cap = (int64_t)(sms > 0 ? sms : 152) * 8;
  if (cap > kRelayoutMaxGrid) cap = kRelayoutMaxGrid;
  const unsigned grid = (unsigned)(want < cap ? want : cap);
  timing_mark(st, 0);
  relayout_kernel<<<grid, THREADS, 0, st>>>(
      static_cast<const uint4 *>(in), static_cast<uint4 *>(out), (uint32_t)N, (uint32_t)H,
      (uint32_t)Hl, (uint32_t)vrow, (uint32_t)(g * Hl), (uint32_t)total, inverse);
  timing_mark(st, 1);
  return cudaGetLastError();
}

}  // namespace chain
