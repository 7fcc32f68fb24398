// chain_api.cu -- the C ABI declared in include/chain.h: argument checks on
// the host, dispatch to the kernels, tensor-map encoding, and the device
// status word that bounded waits report into.
#include <atomic>
#include <mutex>

#include "../../include/chain.h"
#include "internal.h"

namespace chain {

// One status word per device, read by chain_check().
__device__ DevStatus g_status;

namespace {

thread_local int t_last_cuda_error = 0;
constexpr int kMaxTimingEvents = 4;
thread_local cudaEvent_t t_events[kMaxTimingEvents] = {};
thread_local int t_nevents = 0;
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};

struct DevInfo {
  bool init = false;
  bool ok = false;
  int sms = 0;
  DevStatus *status = nullptr;
};
constexpr int MAX_DEV = 64;
DevInfo g_dev[MAX_DEV];
std::mutex g_mu;

// Signature of the driver's cuTensorMapEncodeTiled, resolved at run time
// so the library needs no link-time dependency on libcuda.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return CHAIN_ERR_CUDA;
}

// Checks the current device (compute capability 10.3) and resolves the
// status word's device address once per device.
int device_ready(DevInfo **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= MAX_DEV) return CHAIN_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo &di = g_dev[dev];
  if (!di.init) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e);
    cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    di.ok = (major == 10 && minor == 3);
    if (di.ok) {
      void *addr = nullptr;
      if ((e = cudaGetSymbolAddress(&addr, g_status)) != cudaSuccess) return cuda_fail(e);
      di.status = static_cast<DevStatus *>(addr);
      if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
          return cuda_fail(e != cudaSuccess ? e : cudaErrorNotSupported);
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
      }
    }
    di.init = true;
  }
  if (!di.ok) return CHAIN_ERR_DEVICE;
  *out = &di;
  return CHAIN_OK;
}

WaitCfg wait_cfg(const DevInfo *di) {
  WaitCfg w;
  w.status = di->status;
  w.limit_ns = g_wait_limit_ns.load();
  return w;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A [.., rows, cols] view: innermost stride 1, the others given.
struct View {
  void *ptr;
  int dtype;
  int64_t outer;   // product of leading dims (BH for attention)
  int64_t rows;    // n or M
  int64_t cols;    // d or K
  int64_t s_outer; // elements between consecutive outer indices
  int64_t s_row;   // elements between rows
};

int esize(int dtype) {
  return dtype == CHAIN_BF16 ? 2 : (dtype == CHAIN_F32 ? 4 : (dtype == CHAIN_E4M3 ? 1 : 0));
}

// Accepts 2-D [rows][cols], 3-D [BH][rows][cols] and 4-D [B][H][rows][cols]
// where the two leading dims fold into one stride.
int view_of(const chain_tensor_t *t, int min_nd, View *v) {
  if (!t || !t->ptr) return CHAIN_ERR_ARG;
  if (t->ndim < min_nd || t->ndim > 4) return CHAIN_ERR_ARG;
  if (esize(t->dtype) == 0) return CHAIN_ERR_DTYPE;
  const int nd = t->ndim;
  for (int i = 0; i < nd; ++i)
    if (t->shape[i] < 0 || t->stride[i] < 0) return CHAIN_ERR_ARG;
  if (t->stride[nd - 1] != 1) return CHAIN_ERR_ARG;
  v->ptr = t->ptr;
  v->dtype = t->dtype;
  v->cols = t->shape[nd - 1];
  v->rows = nd >= 2 ? t->shape[nd - 2] : 1;
  v->s_row = nd >= 2 ? t->stride[nd - 2] : v->cols;
  // the stride of a size-1 dimension is arbitrary (frameworks report any
  // value there): use the canonical one
  if (v->rows == 1) v->s_row = v->cols;
  if (nd <= 2) {
    v->outer = 1;
    v->s_outer = v->rows * v->s_row;
  } else if (nd == 3) {
    v->outer = t->shape[0];
    v->s_outer = t->stride[0];
  } else {
    if (t->shape[0] > 1 && t->shape[1] > 1 && t->stride[0] != t->shape[1] * t->stride[1])
      return CHAIN_ERR_ARG;
    v->outer = t->shape[0] * t->shape[1];
    v->s_outer = t->shape[1] > 1 ? t->stride[1] : t->stride[0];
  }
  if (v->outer == 1) v->s_outer = v->rows * v->s_row;
  if (v->rows > 1 && v->s_row < v->cols) return CHAIN_ERR_ARG;
  if (v->outer > 1 && v->s_outer < v->rows * v->s_row) return CHAIN_ERR_ARG;
  return CHAIN_OK;
}

bool pitch16(const View &v) {
  const int es = esize(v.dtype);
  return aligned16(v.ptr) && ((v.s_row * es) % 16 == 0) && ((v.s_outer * es) % 16 == 0) &&
         ((v.cols * es) % 16 == 0);
}

bool same_shape(const View &a, const View &b) {
  return a.outer == b.outer && a.rows == b.rows && a.cols == b.cols;
}

// K or V of grouped-query attention for queries q: the same [n][d] rows and
// a head count that divides q's (each K/V head serves q.outer / kv.outer
// consecutive query heads).
bool kv_shape(const View &q, const View &kv) {
  return kv.rows == q.rows && kv.cols == q.cols && kv.outer >= 1 && q.outer % kv.outer == 0;
}

// LSE [BH][n] (2-D), or [B][H][n] (3-D) folded, innermost contiguous.
int lse_view(const chain_tensor_t *t, int64_t BH, int64_t n, int64_t *s_bh) {
  if (!t || !t->ptr) return CHAIN_ERR_ARG;
  if (t->dtype != CHAIN_F32) return CHAIN_ERR_DTYPE;
  if (t->ndim < 1 || t->ndim > 3 || t->stride[t->ndim - 1] != 1) return CHAIN_ERR_ARG;
  int64_t outer = 1;
  for (int i = 0; i + 1 < t->ndim; ++i) outer *= t->shape[i];
  if (t->shape[t->ndim - 1] != n || outer != BH) return CHAIN_ERR_ARG;
  if (t->ndim == 1) {
    *s_bh = n;
  } else if (t->ndim == 2) {
    *s_bh = t->stride[0];
  } else {
    if (t->shape[1] > 1 && t->stride[0] != t->shape[1] * t->stride[1]) return CHAIN_ERR_ARG;
    *s_bh = t->stride[1];
  }
  if (BH > 1 && *s_bh < n) return CHAIN_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(t->ptr) & 3u) != 0) return CHAIN_ERR_ARG;
  return CHAIN_OK;
}

}  // namespace

int record_cuda_error(cudaError_t e) { return cuda_fail(e); }

void timing_mark(cudaStream_t st, int k) {
  if (k < t_nevents && t_events[k]) cudaEventRecord(t_events[k], st);
}

cudaError_t make_tmap(CUtensorMap *map, CUtensorMapDataType dt, int rank, const void *base,
                      const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box) {
  if (!g_encode) return cudaErrorInitializationError;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides_bytes[i];
  CUresult r = g_encode(map, dt, (cuuint32_t)rank, const_cast<void *>(base), gd, gs, bx, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace chain

using namespace chain;

extern "C" {

const char *chain_status_string(int status) {
  switch (status) {
    case CHAIN_OK: return "ok";
    case CHAIN_ERR_ARG: return "invalid argument (pointer, shape, stride or alignment)";
    case CHAIN_ERR_DTYPE: return "unsupported element type";
    case CHAIN_ERR_DEVICE: return "current device is not compute capability 10.3";
    case CHAIN_ERR_CUDA: return "CUDA call failed (see chain_last_cuda_error)";
    case CHAIN_ERR_TIMEOUT: return "a bounded device-side wait expired";
    case CHAIN_ERR_UNSUPPORTED: return "valid request this library does not implement";
    case CHAIN_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than the fixed array of chain_bwd_noalloc";
    default: return "unknown status";
  }
}

int chain_last_cuda_error(void) { return t_last_cuda_error; }

void chain_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns ? ns : 1); }

void chain_set_timing_events(void *const *events, int count) {
  if (!events || count <= 0) {
    t_nevents = 0;
    return;
  }
  t_nevents = count < kMaxTimingEvents ? count : kMaxTimingEvents;
  for (int k = 0; k < t_nevents; ++k) t_events[k] = static_cast<cudaEvent_t>(events[k]);
}

int chain_check(void *stream, int *detail) {
  DevInfo *di = nullptr;
  int rc = device_ready(&di);
  if (rc != CHAIN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e);
  DevStatus hs;
  e = cudaMemcpyFromSymbol(&hs, g_status, sizeof hs);
  if (e != cudaSuccess) return cuda_fail(e);
  if (detail) *detail = hs.site;
  if (hs.timeout || hs.reserved[0]) {
    DevStatus zero = {0, 0, {0, 0}};
    e = cudaMemcpyToSymbol(g_status, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e);
    // a bounded wait expired, or a kernel met an argument only it could check
    return hs.timeout ? CHAIN_ERR_TIMEOUT : CHAIN_ERR_ARG;
  }
  return CHAIN_OK;
}

int chain_selftest_wait_timeout(uint64_t limit_ns, void *stream) {
  DevInfo *di = nullptr;
  int rc = device_ready(&di);
  if (rc != CHAIN_OK) return rc;
  WaitCfg wc = wait_cfg(di);
  wc.limit_ns = limit_ns ? limit_ns : 1;
  cudaError_t e = launch_wait_selftest(wc, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CHAIN_OK : cuda_fail(e);
}

int chain_umma_selftest(const void *A, const void *B, float *D, int N, int K, int flags,
                        void *stream) {
  if (!A || !B || !D || (N != 64 && N != 128) || K <= 0 || K % 64 || K > 256)
    return CHAIN_ERR_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(D)) return CHAIN_ERR_ARG;
  DevInfo *di = nullptr;
  int rc = device_ready(&di);
  if (rc != CHAIN_OK) return rc;
  cudaError_t e = launch_umma_selftest(A, B, D, N, K, flags & 3, wait_cfg(di),
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CHAIN_OK : cuda_fail(e);
}

int chain_fwd(const chain_tensor_t *A, const chain_tensor_t *B, const chain_tensor_t *C, int f,
              int mask, float scale, chain_tensor_t *O, chain_tensor_t *LSE, void *stream) {
  if (f != CHAIN_F_IDENTITY && f != CHAIN_F_SOFTMAX && f != CHAIN_F_GELU_TANH)
    return CHAIN_ERR_ARG;
  if (mask != CHAIN_MASK_NONE && mask != CHAIN_MASK_CAUSAL) return CHAIN_ERR_ARG;
  View a, b, c, o;
  int rc;
  if ((rc = view_of(A, 2, &a)) || (rc = view_of(B, 2, &b)) || (rc = view_of(C, 2, &c)) ||
      (rc = view_of(O, 2, &o)))
    return rc;
  if (a.dtype != b.dtype || a.dtype != c.dtype || a.dtype != o.dtype) return CHAIN_ERR_DTYPE;
  if (a.dtype == CHAIN_E4M3) return CHAIN_ERR_DTYPE;  // 8-bit inputs: chain_fwd_fp8
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  if (f == CHAIN_F_SOFTMAX) {
    if (!kv_shape(a, b) || !same_shape(b, c) || !same_shape(a, o)) return CHAIN_ERR_ARG;
    if (a.cols != 64 && a.cols != 128) return CHAIN_ERR_ARG;
    if (a.rows < 1 || a.outer < 1) return CHAIN_ERR_ARG;
    if (a.rows > (1 << 30) || a.outer > 65535 * 16) return CHAIN_ERR_ARG;
    if (!(scale > 0.0f) || !(scale < 1e30f)) return CHAIN_ERR_ARG;
    if (!pitch16(a) || !pitch16(b) || !pitch16(c) || !pitch16(o)) return CHAIN_ERR_ARG;
    int64_t lse_sbh = 0;
    if ((rc = lse_view(LSE, a.outer, a.rows, &lse_sbh))) return rc;
    AttnFwdArgs args;
    args.Q = a.ptr; args.K = b.ptr; args.V = c.ptr;
    args.q_sbh = a.s_outer; args.q_srow = a.s_row;
    args.k_sbh = b.s_outer; args.k_srow = b.s_row;
    args.v_sbh = c.s_outer; args.v_srow = c.s_row;
    args.O = o.ptr; args.o_sbh = o.s_outer; args.o_srow = o.s_row;
    args.LSE = static_cast<float *>(LSE->ptr); args.lse_sbh = lse_sbh;
    args.BH = (int)a.outer; args.n = (int)a.rows; args.d = (int)a.cols;
    args.BHkv = (int)b.outer;
    args.causal = mask == CHAIN_MASK_CAUSAL; args.scale = scale;
    args.n_loc = args.n;
    args.q_sshard = args.k_sshard = args.v_sshard = args.o_sshard = 0;
    args.cu_seqlens = nullptr; args.nbatch = 0; args.max_seqlen = 0;
    DevInfo *di = nullptr;
    if ((rc = device_ready(&di))) return rc;
    cudaError_t e;
    if (a.dtype == CHAIN_BF16) {
      e = launch_attn_fwd_bf16(args, wait_cfg(di), st);
    } else {
      if (a.cols != 64 || b.outer != a.outer) return CHAIN_ERR_UNSUPPORTED;
      e = launch_attn_fwd_f32(args, wait_cfg(di), st);
    }
    if (e == cudaErrorNotSupported) return CHAIN_ERR_UNSUPPORTED;
    return e == cudaSuccess ? CHAIN_OK : cuda_fail(e);
  }

  // MLP / identity chain: A [M][K], B [K][N], C [N][P], O [M][P], 2-D bf16.
  if (mask != CHAIN_MASK_NONE) return CHAIN_ERR_ARG;
  if (LSE && LSE->ptr) return CHAIN_ERR_ARG;
  if (A->ndim != 2 || B->ndim != 2 || C->ndim != 2 || O->ndim != 2) return CHAIN_ERR_ARG;
  if (a.dtype != CHAIN_BF16) return CHAIN_ERR_DTYPE;
  if (a.cols != b.rows || b.cols != c.rows || o.rows != a.rows || o.cols != c.cols)
    return CHAIN_ERR_ARG;
  if (!pitch16(a) || !pitch16(b) || !pitch16(c) || !pitch16(o)) return CHAIN_ERR_ARG;
  if (a.s_row != a.cols || b.s_row != b.cols || c.s_row != c.cols || o.s_row != o.cols)
    return CHAIN_ERR_ARG;
  MlpArgs m;
  m.X = a.ptr; m.W1 = b.ptr; m.W2 = c.ptr; m.O = o.ptr;
  m.M = (int)a.rows; m.K = (int)a.cols; m.N = (int)b.cols; m.P = (int)c.cols;
  m.gelu = f == CHAIN_F_GELU_TANH;
  if (m.M <= 0 || m.K <= 0 || m.N <= 0 || m.P <= 0) return CHAIN_ERR_ARG;
  if (m.M % 128 || m.K % 64 || m.N % 128 || m.P % 256) return CHAIN_ERR_UNSUPPORTED;
  DevInfo *di = nullptr;
  if ((rc = device_ready(&di))) return rc;
  cudaError_t e = launch_mlp_chain(m, wait_cfg(di), st);
  if (e == cudaErrorNotSupported) return CHAIN_ERR_UNSUPPORTED;
  return e == cudaSuccess ? CHAIN_OK : cuda_fail(e);
}

size_t chain_fwd_f16h_workspace_size(const chain_tensor_t *C) {
  View c;
  if (view_of(C, 2, &c) || C->ndim != 2 || c.dtype != CHAIN_BF16) return 0;
  if (c.rows < 1 || c.cols < 1 || c.rows > (1 << 30) || c.cols > (1 << 30)) return 0;
  return mlp_f16h_workspace(c.rows, c.cols);
}

int chain_fwd_f16h(const chain_tensor_t *A, const chain_tensor_t *B, const chain_tensor_t *C,
                   int f, chain_tensor_t *O, void *workspace, size_t ws_bytes, void *stream) {
  if (f != CHAIN_F_IDENTITY && f != CHAIN_F_GELU_TANH) return CHAIN_ERR_ARG;
  View a, b, c, o;
  int rc;
  if ((rc = view_of(A, 2, &a)) || (rc = view_of(B, 2, &b)) || (rc = view_of(C, 2, &c)) ||
      (rc = view_of(O, 2, &o)))
    return rc;
  if (A->ndim != 2 || B->ndim != 2 || C->ndim != 2 || O->ndim != 2) return CHAIN_ERR_ARG;
  if (a.dtype != CHAIN_BF16 || b.dtype != CHAIN_BF16 || c.dtype != CHAIN_BF16 ||
      o.dtype != CHAIN_BF16)
    return CHAIN_ERR_DTYPE;
  if (a.cols != b.rows || b.cols != c.rows || o.rows != a.rows || o.cols != c.cols)
    return CHAIN_ERR_ARG;
  if (!pitch16(a) || !pitch16(b) || !pitch16(c) || !pitch16(o)) return CHAIN_ERR_ARG;
  if (a.s_row != a.cols || b.s_row != b.cols || c.s_row != c.cols || o.s_row != o.cols)
    return CHAIN_ERR_ARG;
  MlpArgs m;
  m.X = a.ptr; m.W1 = b.ptr; m.W2 = c.ptr; m.O = o.ptr;
  m.M = (int)a.rows; m.K = (int)a.cols; m.N = (int)b.cols; m.P = (int)c.cols;
  m.gelu = f == CHAIN_F_GELU_TANH;
  if (m.M <= 0 || m.K <= 0 || m.N <= 0 || m.P <= 0) return CHAIN_ERR_ARG;
  if (!workspace || !aligned16(workspace) || ws_bytes < mlp_f16h_workspace(m.N, m.P))
    return CHAIN_ERR_ARG;
  if (m.M % 128 || m.K % 64 || m.N % 64 || m.P % 256 || m.P < 512 || m.P > 1024)
    return CHAIN_ERR_UNSUPPORTED;
  DevInfo *di = nullptr;
  if ((rc = device_ready(&di))) return rc;
  cudaError_t e = launch_mlp_chain_f16h(m, workspace, wait_cfg(di), static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return CHAIN_ERR_UNSUPPORTED;
  return e == cudaSuccess ? CHAIN_OK : cuda_fail(e);
}

static size_t mlp_ws_bytes(const View &a, const View &c) {
  // H and dT, [M][N] bf16 each (M = rows of X, N = rows of W2)
  const size_t b = (size_t)a.rows * (size_t)c.rows * 2 * 2;
  return (b + 255) & ~size_t(255);
}

size_t chain_bwd_workspace_size(const chain_tensor_t *A, const chain_tensor_t *C) {
  View a, c;
  if (view_of(A, 2, &a) || view_of(C, 2, &c)) return 0;
  if (!kv_shape(a, c)) {
    // different shapes: the MLP chain (A = X [M][K], C = W2 [N][P])
    if (A->ndim != 2 || C->ndim != 2) return 0;
    return mlp_ws_bytes(a, c);
  }
  const size_t dvec = (size_t)a.outer * a.rows * sizeof(float);
  return (dvec + 255) & ~size_t(255);
}

size_t chain_bwd_workspace_size_f(const chain_tensor_t *A, const chain_tensor_t *C, int f) {
  if (f == CHAIN_F_SOFTMAX) {
    View a, c;
    if (view_of(A, 2, &a) || view_of(C, 2, &c) || !kv_shape(a, c)) return 0;
    return ((size_t)a.outer * a.rows * sizeof(float) + 255) & ~size_t(255);
  }
  if (f != CHAIN_F_IDENTITY && f != CHAIN_F_GELU_TANH) return 0;
  View a, c;
  if (!A || !C || A->ndim != 2 || C->ndim != 2 || view_of(A, 2, &a) || view_of(C, 2, &c)) return 0;
  return mlp_ws_bytes(a, c);
}

// Backward of the MLP chain O = f(X W1) W2: dense row-major 2-D bf16.
static int mlp_bwd(const chain_tensor_t *dO, const chain_tensor_t *A, const chain_tensor_t *B,
                   const chain_tensor_t *C, int f, int mask, chain_tensor_t *dA,
                   chain_tensor_t *dB, chain_tensor_t *dC, void *workspace, size_t ws_bytes,
                   void *stream) {
  if (mask != CHAIN_MASK_NONE) return CHAIN_ERR_ARG;
  const chain_tensor_t *ts[7] = {dO, A, B, C, dA, dB, dC};
  View v[7];
  for (int i = 0; i < 7; ++i) {
    if (!ts[i] || ts[i]->ndim != 2) return CHAIN_ERR_ARG;
    int rc = view_of(ts[i], 2, &v[i]);
    if (rc) return rc;
    if (v[i].dtype != CHAIN_BF16) return CHAIN_ERR_DTYPE;
    if (v[i].s_row != v[i].cols || !aligned16(v[i].ptr)) return CHAIN_ERR_ARG;
  }
  const View &g = v[0], &x = v[1], &w1 = v[2], &w2 = v[3], &dx = v[4], &dw1 = v[5], &dw2 = v[6];
  const int64_t M = x.rows, K = x.cols, N = w1.cols, P = w2.cols;
  if (w1.rows != K || w2.rows != N || g.rows != M || g.cols != P) return CHAIN_ERR_ARG;
  if (!same_shape(dx, x) || !same_shape(dw1, w1) || !same_shape(dw2, w2)) return CHAIN_ERR_ARG;
  if (M <= 0 || K <= 0 || N <= 0 || P <= 0 || M * N >= (int64_t(1) << 36)) return CHAIN_ERR_ARG;
  if (M % 128 || K % 256 || N % 256 || P % 256) return CHAIN_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < mlp_ws_bytes(x, w2) || !aligned16(workspace)) return CHAIN_ERR_ARG;
  MlpBwdArgs m;
  m.X = x.ptr; m.W1 = w1.ptr; m.W2 = w2.ptr; m.dO = g.ptr;
  m.dX = dx.ptr; m.dW1 = dw1.ptr; m.dW2 = dw2.ptr; m.workspace = workspace;
  m.M = (int)M; m.K = (int)K; m.N = (int)N; m.P = (int)P; m.gelu = f == CHAIN_F_GELU_TANH;
  DevInfo *di = nullptr;
  int rc = device_ready(&di);
  if (rc) return rc;
  cudaError_t e = launch_mlp_bwd(m, wait_cfg(di), static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return CHAIN_ERR_UNSUPPORTED;
  return e == cudaSuccess ? CHAIN_OK : cuda_fail(e);
}

int chain_bwd(const chain_tensor_t *dO, const chain_tensor_t *A, const chain_tensor_t *B,
              const chain_tensor_t *C, const chain_tensor_t *O, const chain_tensor_t *LSE, int f,
              int mask, float scale, chain_tensor_t *dA, chain_tensor_t *dB, chain_tensor_t *dC,
              void *workspace, size_t ws_bytes, void *stream) {
  if (f != CHAIN_F_SOFTMAX) {
    if (f == CHAIN_F_IDENTITY || f == CHAIN_F_GELU_TANH)
      return mlp_bwd(dO, A, B, C, f, mask, dA, dB, dC, workspace, ws_bytes, stream);
    return CHAIN_ERR_ARG;
  }
  if (mask != CHAIN_MASK_NONE && mask != CHAIN_MASK_CAUSAL) return CHAIN_ERR_ARG;
  View g, q, k, v, o, dq, dk, dv;
  int rc;
  if ((rc = view_of(dO, 2, &g)) || (rc = view_of(A, 2, &q)) || (rc = view_of(B, 2, &k)) ||
      (rc = view_of(C, 2, &v)) || (rc = view_of(O, 2, &o)) || (rc = view_of(dA, 2, &dq)) ||
      (rc = view_of(dB, 2, &dk)) || (rc = view_of(dC, 2, &dv)))
    return rc;
  const View *all[8] = {&g, &q, &k, &v, &o, &dq, &dk, &dv};
  for (const View *x : all) {
    if (x->dtype != CHAIN_BF16) return CHAIN_ERR_DTYPE;
    // Q, dO, O, dQ of one shape; K, V, dK, dV of one (grouped-query) shape
    const bool kv_side = x == &k || x == &v || x == &dk || x == &dv;
    if (kv_side ? !(kv_shape(q, *x) && same_shape(*x, k)) : !same_shape(*x, q)) return CHAIN_ERR_ARG;
    // the backward kernels take densely packed [BH][n][d]
    if (x->s_row != x->cols || (x->outer > 1 && x->s_outer != x->rows * x->cols))
      return CHAIN_ERR_ARG;
    if (!aligned16(x->ptr)) return CHAIN_ERR_ARG;
  }
  if (q.cols != 64 && q.cols != 128) return CHAIN_ERR_ARG;
  if (!(scale > 0.0f) || !(scale < 1e30f)) return CHAIN_ERR_ARG;
  if (q.rows * q.cols * q.outer >= (int64_t(1) << 40)) return CHAIN_ERR_ARG;
  int64_t lse_sbh = 0;
  if ((rc = lse_view(LSE, q.outer, q.rows, &lse_sbh))) return rc;
  if (lse_sbh != q.rows) return CHAIN_ERR_ARG;
  const size_t need = chain_bwd_workspace_size(A, C);
  if (!workspace || ws_bytes < need || !aligned16(workspace)) return CHAIN_ERR_ARG;
  AttnBwdArgs args;
  args.Q = q.ptr; args.K = k.ptr; args.V = v.ptr; args.O = o.ptr; args.dO = g.ptr;
  args.LSE = static_cast<const float *>(LSE->ptr);
  args.dQ = dq.ptr; args.dK = dk.ptr; args.dV = dv.ptr;
  args.Dvec = static_cast<float *>(workspace);
  args.BH = (int)q.outer; args.n = (int)q.rows; args.d = (int)q.cols;
  args.BHkv = (int)k.outer;
  args.causal = mask == CHAIN_MASK_CAUSAL; args.scale = scale;
  args.q_srow = args.kv_srow = q.cols;
  args.q_shead = args.kv_shead = q.rows * q.cols;
  args.l_shead = q.rows;
  args.cu_seqlens = nullptr; args.nbatch = 0; args.max_seqlen = 0;
  DevInfo *di = nullptr;
  if ((rc = device_ready(&di))) return rc;
  cudaError_t e = launch_attn_bwd(args, wait_cfg(di), static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return CHAIN_ERR_UNSUPPORTED;
  return e == cudaSuccess ? CHAIN_OK : cuda_fail(e);
}

static int relayout_common(const chain_tensor_t *seq, const chain_tensor_t *hm, int p, int g,
                           int inverse, void *stream) {
  if (!seq || !hm || !seq->ptr || !hm->ptr) return CHAIN_ERR_ARG;
  if (seq->ndim != 4 || hm->ndim != 3) return CHAIN_ERR_ARG;
  if (seq->dtype != hm->dtype || esize(seq->dtype) == 0) return CHAIN_ERR_DTYPE;
  if (p <= 0 || g < 0 || g >= p) return CHAIN_ERR_ARG;
  const int64_t P = seq->shape[0], n_loc = seq->shape[1], H = seq->shape[2], d = seq->shape[3];
  if (P != p || n_loc <= 0 || H <= 0 || d <= 0 || H % p) return CHAIN_ERR_ARG;
  const int64_t Hl = H / p;
  if (hm->shape[0] != Hl || hm->shape[1] != p * n_loc || hm->shape[2] != d) return CHAIN_ERR_ARG;
  // both sides densely packed
  if (seq->stride[3] != 1 || seq->stride[2] != d || seq->stride[1] != H * d ||
      seq->stride[0] != n_loc * H * d)
    return CHAIN_ERR_ARG;
  if (hm->stride[2] != 1 || hm->stride[1] != d || hm->stride[0] != p * n_loc * d)
    return CHAIN_ERR_ARG;
  const int64_t row_bytes = d * esize(seq->dtype);
  if (row_bytes % 16 || !aligned16(seq->ptr) || !aligned16(hm->ptr)) return CHAIN_ERR_ARG;
  if (!relayout_fits_32bit(p * n_loc * H * (row_bytes / 16))) return CHAIN_ERR_ARG;
  DevInfo *di = nullptr;
  int rc = device_ready(&di);
  if (rc) return rc;
  cudaError_t e = inverse ? launch_relayout(hm->ptr, seq->ptr, p, n_loc, H, row_bytes, g, 1,
                                            static_cast<cudaStream_t>(stream))
                          : launch_relayout(seq->ptr, hm->ptr, p, n_loc, H, row_bytes, g, 0,
                                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CHAIN_OK : cuda_fail(e);
}

// A [p][n_loc][H][d] sequence-shard tensor, d contiguous, strides in 16-byte
// multiples, 16-byte aligned.
static int shard_view(const chain_tensor_t *t, int64_t p, int64_t n_loc, int64_t H, int64_t d) {
  if (!t || !t->ptr || t->ndim != 4) return CHAIN_ERR_ARG;
  if (t->dtype != CHAIN_BF16) return CHAIN_ERR_DTYPE;
  if (t->shape[0] != p || t->shape[1] != n_loc || t->shape[2] != H || t->shape[3] != d)
    return CHAIN_ERR_ARG;
  if (t->stride[3] != 1 || !aligned16(t->ptr)) return CHAIN_ERR_ARG;
  for (int i = 0; i < 3; ++i)
    if (t->stride[i] <= 0 || (t->stride[i] * 2) % 16) return CHAIN_ERR_ARG;
  return CHAIN_OK;
}

int chain_fwd_sp(const chain_tensor_t *Q, const chain_tensor_t *K, const chain_tensor_t *V,
                 int p, int head_group, int mask, float scale, chain_tensor_t *O,
                 chain_tensor_t *LSE, void *stream) {
  if (!Q || Q->ndim != 4) return CHAIN_ERR_ARG;
  if (mask != CHAIN_MASK_NONE && mask != CHAIN_MASK_CAUSAL) return CHAIN_ERR_ARG;
  if (p <= 0 || head_group < 0 || head_group >= p) return CHAIN_ERR_ARG;
  const int64_t n_loc = Q->shape[1], H = Q->shape[2], d = Q->shape[3];
  int rc;
  if ((rc = shard_view(Q, p, n_loc, H, d)) || (rc = shard_view(K, p, n_loc, H, d)) ||
      (rc = shard_view(V, p, n_loc, H, d)) || (rc = shard_view(O, p, n_loc, H, d)))
    return rc;
  if (n_loc <= 0 || H <= 0 || H % p || (d != 64 && d != 128)) return CHAIN_ERR_ARG;
  if (!(scale > 0.0f) || !(scale < 1e30f)) return CHAIN_ERR_ARG;
  const int64_t Hl = H / p, n = p * n_loc;
  if (n > (1 << 30) || Hl > 65535 * 16) return CHAIN_ERR_ARG;
  if (n_loc % 128) return CHAIN_ERR_UNSUPPORTED;  // a 128-row tile must not cross shards
  int64_t lse_sbh = 0;
  if ((rc = lse_view(LSE, Hl, n, &lse_sbh))) return rc;
  const int64_t h0 = (int64_t)head_group * Hl;
  AttnFwdArgs args;
  args.Q = static_cast<const __nv_bfloat16 *>(Q->ptr) + h0 * Q->stride[2];
  args.K = static_cast<const __nv_bfloat16 *>(K->ptr) + h0 * K->stride[2];
  args.V = static_cast<const __nv_bfloat16 *>(V->ptr) + h0 * V->stride[2];
  args.O = static_cast<__nv_bfloat16 *>(O->ptr) + h0 * O->stride[2];
  args.q_sbh = Q->stride[2]; args.q_srow = Q->stride[1]; args.q_sshard = Q->stride[0];
  args.k_sbh = K->stride[2]; args.k_srow = K->stride[1]; args.k_sshard = K->stride[0];
  args.v_sbh = V->stride[2]; args.v_srow = V->stride[1]; args.v_sshard = V->stride[0];
  args.o_sbh = O->stride[2]; args.o_srow = O->stride[1]; args.o_sshard = O->stride[0];
  args.LSE = static_cast<float *>(LSE->ptr); args.lse_sbh = lse_sbh;
  args.BH = (int)Hl; args.BHkv = (int)Hl; args.n = (int)n; args.d = (int)d;
  args.n_loc = (int)n_loc;
  args.cu_seqlens = nullptr; args.nbatch = 0; args.max_seqlen = 0;
  args.causal = mask == CHAIN_MASK_CAUSAL; args.scale = scale;
  DevInfo *di = nullptr;
  if ((rc = device_ready(&di))) return rc;
  cudaError_t e = launch_attn_fwd_bf16(args, wait_cfg(di), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CHAIN_OK : cuda_fail(e);
}

size_t chain_fwd_sp_f16pv_workspace_size(const chain_tensor_t *V, int p) {
  if (!V || V->ndim != 4 || p <= 0 || V->shape[0] != p || V->shape[2] % p) return 0;
  const int64_t n = p * V->shape[1], Hl = V->shape[2] / p, d = V->shape[3];
  if (n <= 0 || n > (1 << 30) || Hl <= 0 || Hl > 65535 * 16 || (d != 64 && d != 128)) return 0;
  return attn_fwd_pv16_workspace((int)Hl, (int)n, (int)d);
}

int chain_fwd_sp_f16pv(const chain_tensor_t *Q, const chain_tensor_t *K, const chain_tensor_t *V,
                       int p, int head_group, int mask, float scale, chain_tensor_t *O,
                       chain_tensor_t *LSE, void *workspace, size_t ws_bytes, void *stream) {
  if (!Q || Q->ndim != 4) return CHAIN_ERR_ARG;
  if (mask != CHAIN_MASK_NONE && mask != CHAIN_MASK_CAUSAL) return CHAIN_ERR_ARG;
  if (p <= 0 || head_group < 0 || head_group >= p) return CHAIN_ERR_ARG;
  const int64_t n_loc = Q->shape[1], H = Q->shape[2], d = Q->shape[3];
  int rc;
  if ((rc = shard_view(Q, p, n_loc, H, d)) || (rc = shard_view(K, p, n_loc, H, d)) ||
      (rc = shard_view(V, p, n_loc, H, d)) || (rc = shard_view(O, p, n_loc, H, d)))
    return rc;
  if (n_loc <= 0 || H <= 0 || H % p || (d != 64 && d != 128)) return CHAIN_ERR_ARG;
  if (!(scale > 0.0f) || !(scale < 1e30f)) return CHAIN_ERR_ARG;
  const int64_t Hl = H / p, n = p * n_loc;
  if (n > (1 << 30) || Hl > 65535 * 16) return CHAIN_ERR_ARG;
  if (n_loc % 128) return CHAIN_ERR_UNSUPPORTED;  // a 128-row tile must not cross shards
  int64_t lse_sbh = 0;
  if ((rc = lse_view(LSE, Hl, n, &lse_sbh))) return rc;
  if (!workspace || !aligned16(workspace) ||
      ws_bytes < attn_fwd_pv16_workspace((int)Hl, (int)n, (int)d))
    return CHAIN_ERR_ARG;
  if (Hl > 65535) return CHAIN_ERR_UNSUPPORTED;  // the V pre-pass grid's y extent
  const int64_t h0 = (int64_t)head_group * Hl;
  AttnFwdArgs args;
  args.Q = static_cast<const __nv_bfloat16 *>(Q->ptr) + h0 * Q->stride[2];
  args.K = static_cast<const __nv_bfloat16 *>(K->ptr) + h0 * K->stride[2];
  args.V = static_cast<const __nv_bfloat16 *>(V->ptr) + h0 * V->stride[2];
  args.O = static_cast<__nv_bfloat16 *>(O->ptr) + h0 * O->stride[2];
  args.q_sbh = Q->stride[2]; args.q_srow = Q->stride[1]; args.q_sshard = Q->stride[0];
  args.k_sbh = K->stride[2]; args.k_srow = K->stride[1]; args.k_sshard = K->stride[0];
  args.v_sbh = V->stride[2]; args.v_srow = V->stride[1]; args.v_sshard = V->stride[0];
  args.o_sbh = O->stride[2]; args.o_srow = O->stride[1]; args.o_sshard = O->stride[0];
  args.LSE = static_cast<float *>(LSE->ptr); args.lse_sbh = lse_sbh;
  args.BH = (int)Hl; args.BHkv = (int)Hl; args.n = (int)n; args.d = (int)d;
  args.n_loc = (int)n_loc;
  args.cu_seqlens = nullptr; args.nbatch = 0; args.max_seqlen = 0;
  args.causal = mask == CHAIN_MASK_CAUSAL; args.scale = scale;
  DevInfo *di = nullptr;
  if ((rc = device_ready(&di))) return rc;
  cudaError_t e = launch_attn_fwd_pv16(args, workspace, wait_cfg(di),
                                       static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return CHAIN_ERR_UNSUPPORTED;
  return e == cudaSuccess ? CHAIN_OK : cuda_fail(e);
}

// Packed variable-length tensor [total][H][d] bf16: d contiguous, row and
// head strides in 16-byte multiples, 16-byte aligned.
static int packed_view(const chain_tensor_t *t, int64_t total, int64_t H, int64_t d) {
  if (!t || !t->ptr || t->ndim != 3) return CHAIN_ERR_ARG;
  if (t->dtype != CHAIN_BF16) return CHAIN_ERR_DTYPE;
  if (t->shape[0] != total || t->shape[1] != H || t->shape[2] != d) return CHAIN_ERR_ARG;
  if (t->stride[2] != 1 || !aligned16(t->ptr)) return CHAIN_ERR_ARG;
  if (t->stride[0] <= 0 || t->stride[1] <= 0 || (t->stride[0] * 2) % 16 || (t->stride[1] * 2) % 16)
    return CHAIN_ERR_ARG;
  return CHAIN_OK;
}

int chain_fwd_varlen(const chain_tensor_t *Q, const chain_tensor_t *K, const chain_tensor_t *V,
                     const int32_t *cu_seqlens, int batch, int max_seqlen, int mask, float scale,
                     chain_tensor_t *O, chain_tensor_t *LSE, void *stream) {
  if (!Q || Q->ndim != 3 || !K || K->ndim != 3) return CHAIN_ERR_ARG;
  if (mask != CHAIN_MASK_NONE && mask != CHAIN_MASK_CAUSAL) return CHAIN_ERR_ARG;
  const int64_t total = Q->shape[0], H = Q->shape[1], d = Q->shape[2], Hkv = K->shape[1];
  int rc;
  if ((rc = packed_view(Q, total, H, d)) || (rc = packed_view(K, total, Hkv, d)) ||
      (rc = packed_view(V, total, Hkv, d)) || (rc = packed_view(O, total, H, d)))
    return rc;
  if (total < 1 || total > (1 << 30) || (d != 64 && d != 128)) return CHAIN_ERR_ARG;
  if (Hkv < 1 || H % Hkv || H > 65535 * 16) return CHAIN_ERR_ARG;
  if (!cu_seqlens || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return CHAIN_ERR_ARG;
  if (batch < 1 || batch > (1 << 20) || max_seqlen < 1 || max_seqlen > total) return CHAIN_ERR_ARG;
  if (!(scale > 0.0f) || !(scale < 1e30f)) return CHAIN_ERR_ARG;
  int64_t lse_sbh = 0;
  if ((rc = lse_view(LSE, H, total, &lse_sbh))) return rc;
  AttnFwdArgs args;
  args.Q = Q->ptr; args.K = K->ptr; args.V = V->ptr; args.O = O->ptr;
  args.q_sbh = Q->stride[1]; args.q_srow = Q->stride[0];
  args.k_sbh = K->stride[1]; args.k_srow = K->stride[0];
  args.v_sbh = V->stride[1]; args.v_srow = V->stride[0];
  args.o_sbh = O->stride[1]; args.o_srow = O->stride[0];
  args.LSE = static_cast<float *>(LSE->ptr); args.lse_sbh = lse_sbh;
  args.BH = (int)H; args.BHkv = (int)Hkv; args.n = (int)total; args.d = (int)d;
  args.causal = mask == CHAIN_MASK_CAUSAL; args.scale = scale;
  args.n_loc = args.n;
  args.q_sshard = args.k_sshard = args.v_sshard = args.o_sshard = 0;
  args.cu_seqlens = cu_seqlens; args.nbatch = batch; args.max_seqlen = max_seqlen;
  DevInfo *di = nullptr;
  if ((rc = device_ready(&di))) return rc;
  cudaError_t e = launch_attn_fwd_bf16(args, wait_cfg(di), static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return CHAIN_ERR_UNSUPPORTED;
  return e == cudaSuccess ? CHAIN_OK : cuda_fail(e);
}

size_t chain_fwd_varlen_f16pv_workspace_size(const chain_tensor_t *V) {
  if (!V || V->ndim != 3) return 0;
  const int64_t total = V->shape[0], Hkv = V->shape[1], d = V->shape[2];
  if (total < 1 || total > (1 << 30) || Hkv < 1 || Hkv > 65535 || (d != 64 && d != 128))
    return 0;
  return attn_fwd_pv16_workspace((int)Hkv, (int)total, (int)d);
}

int chain_fwd_varlen_f16pv(const chain_tensor_t *Q, const chain_tensor_t *K,
                           const chain_tensor_t *V, const int32_t *cu_seqlens, int batch,
                           int max_seqlen, int mask, float scale, chain_tensor_t *O,
                           chain_tensor_t *LSE, void *workspace, size_t ws_bytes, void *stream) {
  if (!Q || Q->ndim != 3 || !K || K->ndim != 3) return CHAIN_ERR_ARG;
  if (mask != CHAIN_MASK_NONE && mask != CHAIN_MASK_CAUSAL) return CHAIN_ERR_ARG;
  const int64_t total = Q->shape[0], H = Q->shape[1], d = Q->shape[2], Hkv = K->shape[1];
  int rc;
  if ((rc = packed_view(Q, total, H, d)) || (rc = packed_view(K, total, Hkv, d)) ||
      (rc = packed_view(V, total, Hkv, d)) || (rc = packed_view(O, total, H, d)))
    return rc;
  if (total < 1 || total > (1 << 30) || (d != 64 && d != 128)) return CHAIN_ERR_ARG;
  if (Hkv < 1 || H % Hkv || H > 65535 * 16) return CHAIN_ERR_ARG;
  if (!cu_seqlens || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return CHAIN_ERR_ARG;
  if (batch < 1 || batch > (1 << 20) || max_seqlen < 1 || max_seqlen > total) return CHAIN_ERR_ARG;
  if (!(scale > 0.0f) || !(scale < 1e30f)) return CHAIN_ERR_ARG;
  int64_t lse_sbh = 0;
  if ((rc = lse_view(LSE, H, total, &lse_sbh))) return rc;
  if (Hkv > 65535) return CHAIN_ERR_UNSUPPORTED;  // the V pre-pass grid's y extent
  if (!workspace || !aligned16(workspace) ||
      ws_bytes < attn_fwd_pv16_workspace((int)Hkv, (int)total, (int)d))
    return CHAIN_ERR_ARG;
  AttnFwdArgs args;
  args.Q = Q->ptr; args.K = K->ptr; args.V = V->ptr; args.O = O->ptr;
  args.q_sbh = Q->stride[1]; args.q_srow = Q->stride[0];
  args.k_sbh = K->stride[1]; args.k_srow = K->stride[0];
  args.v_sbh = V->stride[1]; args.v_srow = V->stride[0];
  args.o_sbh = O->stride[1]; args.o_srow = O->stride[0];
  args.LSE = static_cast<float *>(LSE->ptr); args.lse_sbh = lse_sbh;
  args.BH = (int)H; args.BHkv = (int)Hkv; args.n = (int)total; args.d = (int)d;
  args.causal = mask == CHAIN_MASK_CAUSAL; args.scale = scale;
  args.n_loc = args.n;
  args.q_sshard = args.k_sshard = args.v_sshard = args.o_sshard = 0;
  args.cu_seqlens = cu_seqlens; args.nbatch = batch; args.max_seqlen = max_seqlen;
  DevInfo *di = nullptr;
  if ((rc = device_ready(&di))) return rc;
  cudaError_t e = launch_attn_fwd_pv16(args, workspace, wait_cfg(di),
                                       static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return CHAIN_ERR_UNSUPPORTED;
  return e == cudaSuccess ? CHAIN_OK : cuda_fail(e);
}

int chain_bwd_varlen(const chain_tensor_t *dO, const chain_tensor_t *Q, const chain_tensor_t *K,
                     const chain_tensor_t *V, const chain_tensor_t *O, const chain_tensor_t *LSE,
                     const int32_t *cu_seqlens, int batch, int max_seqlen, int mask, float scale,
                     chain_tensor_t *dQ, chain_tensor_t *dK, chain_tensor_t *dV, void *workspace,
                     size_t ws_bytes, void *stream) {
  if (!Q || Q->ndim != 3 || !K || K->ndim != 3) return CHAIN_ERR_ARG;
  if (mask != CHAIN_MASK_NONE && mask != CHAIN_MASK_CAUSAL) return CHAIN_ERR_ARG;
  const int64_t total = Q->shape[0], H = Q->shape[1], d = Q->shape[2], Hkv = K->shape[1];
  const chain_tensor_t *qs[4] = {Q, O, dO, dQ}, *ks[4] = {K, V, dK, dV};
  int rc;
  for (int i = 0; i < 4; ++i) {
    if ((rc = packed_view(qs[i], total, H, d)) || (rc = packed_view(ks[i], total, Hkv, d))) return rc;
    // one stride pair serves each side
    if (qs[i]->stride[0] != Q->stride[0] || qs[i]->stride[1] != Q->stride[1]) return CHAIN_ERR_ARG;
    if (ks[i]->stride[0] != K->stride[0] || ks[i]->stride[1] != K->stride[1]) return CHAIN_ERR_ARG;
  }
  if (total < 1 || total > (1 << 30) || (d != 64 && d != 128)) return CHAIN_ERR_ARG;
  if (Hkv < 1 || H % Hkv || H > 65535 * 16) return CHAIN_ERR_ARG;
  if (!cu_seqlens || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return CHAIN_ERR_ARG;
  if (batch < 1 || batch > (1 << 20) || max_seqlen < 1 || max_seqlen > total) return CHAIN_ERR_ARG;
  if (!(scale > 0.0f) || !(scale < 1e30f)) return CHAIN_ERR_ARG;
  int64_t lse_sbh = 0;
  if ((rc = lse_view(LSE, H, total, &lse_sbh))) return rc;
  if (lse_sbh != total) return CHAIN_ERR_ARG;
  const size_t need = ((size_t)H * (size_t)total * sizeof(float) + 255) & ~size_t(255);
  if (!workspace || ws_bytes < need || !aligned16(workspace)) return CHAIN_ERR_ARG;
  AttnBwdArgs args;
  args.Q = Q->ptr; args.K = K->ptr; args.V = V->ptr; args.O = O->ptr; args.dO = dO->ptr;
  args.LSE = static_cast<const float *>(LSE->ptr);
  args.dQ = dQ->ptr; args.dK = dK->ptr; args.dV = dV->ptr;
  args.Dvec = static_cast<float *>(workspace);
  args.BH = (int)H; args.BHkv = (int)Hkv; args.n = (int)total; args.d = (int)d;
  args.causal = mask == CHAIN_MASK_CAUSAL; args.scale = scale;
  args.q_srow = Q->stride[0]; args.q_shead = Q->stride[1];
  args.kv_srow = K->stride[0]; args.kv_shead = K->stride[1];
  args.l_shead = total;
  args.cu_seqlens = cu_seqlens; args.nbatch = batch; args.max_seqlen = max_seqlen;
  DevInfo *di = nullptr;
  if ((rc = device_ready(&di))) return rc;
  cudaError_t e = launch_attn_bwd(args, wait_cfg(di), static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return CHAIN_ERR_UNSUPPORTED;
  return e == cudaSuccess ? CHAIN_OK : cuda_fail(e);
}

size_t chain_fwd_f16pv_workspace_size(const chain_tensor_t *Q, const chain_tensor_t *V) {
  View q, v;
  if (view_of(Q, 2, &q) || view_of(V, 2, &v) || !kv_shape(q, v)) return 0;
  if (q.rows < 1 || q.rows > (1 << 30) || v.outer < 1 || v.outer > 65535 * 16) return 0;
  return attn_fwd_pv16_workspace((int)v.outer, (int)v.rows, (int)v.cols);
}

int chain_fwd_f16pv(const chain_tensor_t *Q, const chain_tensor_t *K, const chain_tensor_t *V,
                    int mask, float scale, chain_tensor_t *O, chain_tensor_t *LSE,
                    void *workspace, size_t ws_bytes, void *stream) {
  if (mask != CHAIN_MASK_NONE && mask != CHAIN_MASK_CAUSAL) return CHAIN_ERR_ARG;
  View q, k, v, o;
  int rc;
  if ((rc = view_of(Q, 2, &q)) || (rc = view_of(K, 2, &k)) || (rc = view_of(V, 2, &v)) ||
      (rc = view_of(O, 2, &o)))
    return rc;
  if (q.dtype != CHAIN_BF16 || k.dtype != CHAIN_BF16 || v.dtype != CHAIN_BF16 ||
      o.dtype != CHAIN_BF16)
    return CHAIN_ERR_DTYPE;
  if (!kv_shape(q, k) || !same_shape(k, v) || !same_shape(q, o)) return CHAIN_ERR_ARG;
  if (q.cols != 64 && q.cols != 128) return CHAIN_ERR_ARG;
  if (q.rows < 1 || q.outer < 1) return CHAIN_ERR_ARG;
  if (q.rows > (1 << 30) || q.outer > 65535 * 16) return CHAIN_ERR_ARG;
  if (!(scale > 0.0f) || !(scale < 1e30f)) return CHAIN_ERR_ARG;
  if (!pitch16(q) || !pitch16(k) || !pitch16(v) || !pitch16(o)) return CHAIN_ERR_ARG;
  int64_t lse_sbh = 0;
  if ((rc = lse_view(LSE, q.outer, q.rows, &lse_sbh))) return rc;
  if (!workspace || !aligned16(workspace) ||
      ws_bytes < attn_fwd_pv16_workspace((int)v.outer, (int)v.rows, (int)v.cols))
    return CHAIN_ERR_ARG;
  if (v.outer > 65535) return CHAIN_ERR_UNSUPPORTED;  // the V pre-pass grid's y extent
  AttnFwdArgs args;
  args.Q = q.ptr; args.K = k.ptr; args.V = v.ptr;
  args.q_sbh = q.s_outer; args.q_srow = q.s_row;
  args.k_sbh = k.s_outer; args.k_srow = k.s_row;
  args.v_sbh = v.s_outer; args.v_srow = v.s_row;
  args.O = o.ptr; args.o_sbh = o.s_outer; args.o_srow = o.s_row;
  args.LSE = static_cast<float *>(LSE->ptr); args.lse_sbh = lse_sbh;
  args.BH = (int)q.outer; args.n = (int)q.rows; args.d = (int)q.cols;
  args.BHkv = (int)k.outer;
  args.causal = mask == CHAIN_MASK_CAUSAL; args.scale = scale;
  args.n_loc = args.n;
  args.q_sshard = args.k_sshard = args.v_sshard = args.o_sshard = 0;
  args.cu_seqlens = nullptr; args.nbatch = 0; args.max_seqlen = 0;
  DevInfo *di = nullptr;
  if ((rc = device_ready(&di))) return rc;
  cudaError_t e = launch_attn_fwd_pv16(args, workspace, wait_cfg(di),
                                       static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return CHAIN_ERR_UNSUPPORTED;
  return e == cudaSuccess ? CHAIN_OK : cuda_fail(e);
}

static size_t fp8_ws_bytes(const View &v) {
  return ((size_t)(v.outer * v.rows * v.cols * 2) + 255) & ~(size_t)255;
}

size_t chain_fwd_fp8_workspace_size(const chain_tensor_t *V) {
  View v;
  if (view_of(V, 2, &v) || v.dtype != CHAIN_E4M3) return 0;
  return fp8_ws_bytes(v);
}

int chain_fwd_fp8(const chain_tensor_t *Q, const chain_tensor_t *K, const chain_tensor_t *V,
                  int mask, float scale, float v_scale, chain_tensor_t *O, chain_tensor_t *LSE,
                  void *workspace, size_t ws_bytes, void *stream) {
  if (mask != CHAIN_MASK_NONE && mask != CHAIN_MASK_CAUSAL) return CHAIN_ERR_ARG;
  View q, k, v, o;
  int rc;
  if ((rc = view_of(Q, 2, &q)) || (rc = view_of(K, 2, &k)) || (rc = view_of(V, 2, &v)) ||
      (rc = view_of(O, 2, &o)))
    return rc;
  if (q.dtype != CHAIN_E4M3 || k.dtype != CHAIN_E4M3 || v.dtype != CHAIN_E4M3 ||
      o.dtype != CHAIN_BF16)
    return CHAIN_ERR_DTYPE;
  if (!kv_shape(q, k) || !same_shape(k, v) || !same_shape(q, o)) return CHAIN_ERR_ARG;
  if (q.rows < 1 || q.outer < 1) return CHAIN_ERR_ARG;
  if (q.rows > (1 << 30) || q.outer > 65535 * 16) return CHAIN_ERR_ARG;
  if (q.cols != 128) return q.cols == 64 ? CHAIN_ERR_UNSUPPORTED : CHAIN_ERR_ARG;
  if (!(scale > 0.0f) || !(scale < 1e30f)) return CHAIN_ERR_ARG;
  if (!(v_scale == v_scale) || !(v_scale < 1e30f) || !(v_scale > -1e30f)) return CHAIN_ERR_ARG;
  if (!pitch16(q) || !pitch16(k) || !pitch16(v) || !pitch16(o)) return CHAIN_ERR_ARG;
  int64_t lse_sbh = 0;
  if ((rc = lse_view(LSE, q.outer, q.rows, &lse_sbh))) return rc;
  if (!workspace || !aligned16(workspace) || ws_bytes < fp8_ws_bytes(v)) return CHAIN_ERR_ARG;
  AttnFwdArgs args;
  args.Q = q.ptr; args.K = k.ptr; args.V = v.ptr;
  args.q_sbh = q.s_outer; args.q_srow = q.s_row;
  args.k_sbh = k.s_outer; args.k_srow = k.s_row;
  args.v_sbh = v.s_outer; args.v_srow = v.s_row;
  args.O = o.ptr; args.o_sbh = o.s_outer; args.o_srow = o.s_row;
  args.LSE = static_cast<float *>(LSE->ptr); args.lse_sbh = lse_sbh;
  args.BH = (int)q.outer; args.n = (int)q.rows; args.d = 128;
  args.BHkv = (int)k.outer;
  args.causal = mask == CHAIN_MASK_CAUSAL; args.scale = scale;
  args.v_scale = v_scale;
  args.n_loc = args.n;
  args.q_sshard = args.k_sshard = args.v_sshard = args.o_sshard = 0;
  args.cu_seqlens = nullptr; args.nbatch = 0; args.max_seqlen = 0;
  DevInfo *di = nullptr;
  if ((rc = device_ready(&di))) return rc;
  cudaError_t e = launch_attn_fwd_fp8(args, workspace, wait_cfg(di),
                                      static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return CHAIN_ERR_UNSUPPORTED;
  return e == cudaSuccess ? CHAIN_OK : cuda_fail(e);
}

int sp_relayout(const chain_tensor_t *shards, int p, int head_group, chain_tensor_t *out,
                void *stream) {
  return relayout_common(shards, out, p, head_group, 0, stream);
}

int sp_relayout_inverse(const chain_tensor_t *in, int p, int head_group,
                        chain_tensor_t *shards, void *stream) {
  return relayout_common(shards, in, p, head_group, 1, stream);
}

}  // extern "C"
