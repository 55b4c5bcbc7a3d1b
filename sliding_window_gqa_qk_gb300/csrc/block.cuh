// The attention block around the attention core: the block's pre-norm, the
// four bias-free projections c_q, c_k, c_v, c_proj and the residual
// (autoresearch Administrator & Developer Guide §8.2.1 model table, "Pre-norm
// + residual": x = x + attn(norm(x)); train.py walkthrough post, model
// paragraph: RMSNorm on the block inputs).
//
// The pre-norm and its backward are row-wise kernels here. The projections
// are plain GEMMs and go to cuBLASLt (bf16 operands with fp32 accumulation in
// the bf16 library, fp32 throughout in the fp32 debug library). cuBLASLt is
// opened at run time with dlopen, so the library neither links against it
// nor fails to load where it is missing; the block entry points then return
// SWA_ERR_UNSUPPORTED. cuBLASLt gets a slice of the caller's workspace as its
// only device scratch.
#pragma once

#include <cublasLt.h>
#include <dlfcn.h>

#include <mutex>

#include "rowwise.cuh"

namespace swa {
namespace blk {

// ---------------------------------------------------------------------------
// Pre-norm: xn = x / sqrt(mean(x^2) + eps) per row of C channels (no gain),
// rstd kept for the backward. One warp per row; each lane moves 16-byte
// vectors of the row. C is a multiple of 8.
// ---------------------------------------------------------------------------
constexpr int kPnEpl = 16 / static_cast<int>(sizeof(elem_t));  // elements per 16-byte vector
constexpr int kPnWarps = 8;
constexpr int kPnBlocksPerSm = 4;

__global__ void __launch_bounds__(kPnWarps * 32) prenorm_fwd_kernel(const elem_t* __restrict__ x,
                                                                    elem_t* __restrict__ xn,
                                                                    float* __restrict__ rstd,
                                                                    long long rows, int C, float eps) {
  const int lane = threadIdx.x & 31;
  for (long long r = grid_warp(); r < rows; r += grid_warps()) {
    const elem_t* xr = x + r * C;
    float ss = 0.f;
    for (int c = lane * kPnEpl; c < C; c += 32 * kPnEpl) {
      float f[kPnEpl];
      unpack16(ld16(xr + c), f);
#pragma unroll
      for (int i = 0; i < kPnEpl; ++i) ss = fmaf(f[i], f[i], ss);
    }
    ss = row_sum<32>(ss);
    const float rs = rsqrtf(ss / C + eps);
    elem_t* yr = xn + r * C;
    for (int c = lane * kPnEpl; c < C; c += 32 * kPnEpl) {
      float f[kPnEpl];
      unpack16(ld16(xr + c), f);
#pragma unroll
      for (int i = 0; i < kPnEpl; ++i) f[i] *= rs;
      st16(yr + c, pack16(f));
    }
    if (lane == 0) rstd[r] = rs;
  }
}

// Backward of the pre-norm plus the residual: with xh = x r and g the
// gradient of xn (dxn, plus dgx on the first gch channels: the learned
// gate's gradient of the channels it read),
//   dx = dout + r (g - xh mean(g xh)).
__global__ void __launch_bounds__(kPnWarps * 32) prenorm_bwd_kernel(
    const elem_t* __restrict__ x, const float* __restrict__ rstd, const float* __restrict__ dxn,
    const float* __restrict__ dgx, int gch, const elem_t* __restrict__ dout, elem_t* __restrict__ dx,
    long long rows, int C) {
  const int lane = threadIdx.x & 31;
  for (long long r = grid_warp(); r < rows; r += grid_warps()) {
    const float rs = rstd[r];
    const elem_t* xr = x + r * C;
    const float* gr = dxn + r * C;
    const float* hr = dgx != nullptr ? dgx + r * gch : nullptr;
    auto grad = [&](int c, float (&g)[kPnEpl]) {
      ldf<kPnEpl>(gr + c, g);
      if (hr != nullptr && c < gch) {
#pragma unroll
        for (int i = 0; i < kPnEpl; ++i)
          if (c + i < gch) g[i] += hr[c + i];
      }
    };
    float dot = 0.f;
    for (int c = lane * kPnEpl; c < C; c += 32 * kPnEpl) {
      float f[kPnEpl], g[kPnEpl];
      unpack16(ld16(xr + c), f);
      grad(c, g);
#pragma unroll
      for (int i = 0; i < kPnEpl; ++i) dot = fmaf(g[i], f[i] * rs, dot);
    }
    const float mean = row_sum<32>(dot) / C;
    const elem_t* dor = dout + r * C;
    elem_t* dxr = dx + r * C;
    for (int c = lane * kPnEpl; c < C; c += 32 * kPnEpl) {
      float f[kPnEpl], g[kPnEpl], o[kPnEpl];
      unpack16(ld16(xr + c), f);
      unpack16(ld16(dor + c), o);
      grad(c, g);
#pragma unroll
      for (int i = 0; i < kPnEpl; ++i) o[i] += rs * (g[i] - f[i] * rs * mean);
      st16(dxr + c, pack16(o));
    }
  }
}

inline int prenorm_grid(long long rows) {
  const long long per = (rows + kPnWarps - 1) / kPnWarps;
  const long long cap = static_cast<long long>(num_sms()) * kPnBlocksPerSm;
  return static_cast<int>(per < cap ? (per < 1 ? 1 : per) : cap);
}

// ---------------------------------------------------------------------------
// cuBLASLt, opened at run time.
// ---------------------------------------------------------------------------
struct LtApi {
  decltype(&cublasLtCreate) create = nullptr;
  decltype(&cublasLtMatmulDescCreate) desc_create = nullptr;
  decltype(&cublasLtMatmulDescDestroy) desc_destroy = nullptr;
  decltype(&cublasLtMatmulDescSetAttribute) desc_set = nullptr;
  decltype(&cublasLtMatrixLayoutCreate) layout_create = nullptr;
  decltype(&cublasLtMatrixLayoutDestroy) layout_destroy = nullptr;
  decltype(&cublasLtMatmulPreferenceCreate) pref_create = nullptr;
  decltype(&cublasLtMatmulPreferenceDestroy) pref_destroy = nullptr;
  decltype(&cublasLtMatmulPreferenceSetAttribute) pref_set = nullptr;
  decltype(&cublasLtMatmulAlgoGetHeuristic) heuristic = nullptr;
  decltype(&cublasLtMatmul) matmul = nullptr;
  bool ok = false;
};

inline const LtApi& lt_api() {
  static const LtApi api = [] {
    LtApi a;
    void* h = dlopen("libcublasLt.so.13", RTLD_NOW | RTLD_LOCAL);
    if (h == nullptr) h = dlopen("libcublasLt.so", RTLD_NOW | RTLD_LOCAL);
    if (h == nullptr) return a;
    bool all = true;
    auto get = [&](auto& fn, const char* name) {
      fn = reinterpret_cast<std::remove_reference_t<decltype(fn)>>(dlsym(h, name));
      all = all && fn != nullptr;
    };
    get(a.create, "cublasLtCreate");
    get(a.desc_create, "cublasLtMatmulDescCreate");
    get(a.desc_destroy, "cublasLtMatmulDescDestroy");
    get(a.desc_set, "cublasLtMatmulDescSetAttribute");
    get(a.layout_create, "cublasLtMatrixLayoutCreate");
    get(a.layout_destroy, "cublasLtMatrixLayoutDestroy");
    get(a.pref_create, "cublasLtMatmulPreferenceCreate");
    get(a.pref_destroy, "cublasLtMatmulPreferenceDestroy");
    get(a.pref_set, "cublasLtMatmulPreferenceSetAttribute");
    get(a.heuristic, "cublasLtMatmulAlgoGetHeuristic");
    get(a.matmul, "cublasLtMatmul");
    a.ok = all;
    return a;
  }();
  return api;
}

// One cuBLASLt handle per device, created on the first block call made with
// that device current (host-side state of cuBLASLt).
inline swa_status lt_handle(cublasLtHandle_t* out) {
  const LtApi& L = lt_api();
  if (!L.ok) return SWA_ERR_UNSUPPORTED;
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static cublasLtHandle_t handles[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return SWA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (handles[dev] == nullptr && L.create(&handles[dev]) != CUBLAS_STATUS_SUCCESS) {
    handles[dev] = nullptr;
    return SWA_ERR_CUDA;
  }
  *out = handles[dev];
  return SWA_OK;
}

#if defined(SWA_ELEM_FP32)
constexpr cudaDataType_t kElemType = CUDA_R_32F;
#else
constexpr cudaDataType_t kElemType = CUDA_R_16BF;
#endif

// Column-major GEMM D[m x n] = op(A) op(B) + beta C, with C = D unless given:
// A is stored k x m (lda) when ta, else m x k; B is stored n x k (ldb) when
// tb, else k x n; C and D are m x n (ldd). A and B are elem_t; C and D are
// dt (elem_t or fp32). Accumulation and alpha / beta in fp32.
struct Gemm {
  bool ta = false, tb = false;
  int m = 0, n = 0, k = 0;
  const void* A = nullptr;
  int lda = 0;
  const void* B = nullptr;
  int ldb = 0;
  float beta = 0.f;
  const void* C = nullptr;
  void* D = nullptr;
  cudaDataType_t dt = kElemType;
  int ldd = 0;
};

// Largest power of two (at most 256) that divides the address: cuBLASLt's
// algorithm choice assumes 256-byte aligned operands unless told otherwise,
// and callers' tensors need only be 16-byte aligned.
inline uint32_t ptr_alignment(const void* p) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  uint32_t al = 256;
  while (al > 1 && (a & (al - 1)) != 0) al >>= 1;
  return al;
}

inline swa_status gemm(const Gemm& g, void* lt_ws, size_t lt_ws_bytes, cudaStream_t st) {
  if (g.m == 0 || g.n == 0) return SWA_OK;
  cublasLtHandle_t h = nullptr;
  swa_status s = lt_handle(&h);
  if (s != SWA_OK) return s;
  const LtApi& L = lt_api();
  cublasLtMatmulDesc_t desc = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  s = SWA_ERR_CUDA;
  const cublasOperation_t opa = g.ta ? CUBLAS_OP_T : CUBLAS_OP_N;
  const cublasOperation_t opb = g.tb ? CUBLAS_OP_T : CUBLAS_OP_N;
  const uint64_t wsb = lt_ws_bytes;
  const void* cptr = g.C != nullptr ? g.C : g.D;
  const uint32_t al[4] = {ptr_alignment(g.A), ptr_alignment(g.B), ptr_alignment(cptr), ptr_alignment(g.D)};
  const cublasLtMatmulPreferenceAttributes_t al_attr[4] = {
      CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_A_BYTES, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_B_BYTES,
      CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_C_BYTES, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_D_BYTES};
  auto set_alignments = [&]() {
    for (int i = 0; i < 4; ++i)
      if (L.pref_set(pref, al_attr[i], &al[i], sizeof(al[i])) != CUBLAS_STATUS_SUCCESS) return false;
    return true;
  };
  cublasLtMatmulHeuristicResult_t res{};
  int found = 0;
  const float alpha = 1.f;
  if (L.desc_create(&desc, CUBLAS_COMPUTE_32F, CUDA_R_32F) == CUBLAS_STATUS_SUCCESS &&
      L.desc_set(desc, CUBLASLT_MATMUL_DESC_TRANSA, &opa, sizeof(opa)) == CUBLAS_STATUS_SUCCESS &&
      L.desc_set(desc, CUBLASLT_MATMUL_DESC_TRANSB, &opb, sizeof(opb)) == CUBLAS_STATUS_SUCCESS &&
      L.layout_create(&la, kElemType, g.ta ? g.k : g.m, g.ta ? g.m : g.k, g.lda) == CUBLAS_STATUS_SUCCESS &&
      L.layout_create(&lb, kElemType, g.tb ? g.n : g.k, g.tb ? g.k : g.n, g.ldb) == CUBLAS_STATUS_SUCCESS &&
      L.layout_create(&lc, g.dt, g.m, g.n, g.ldd) == CUBLAS_STATUS_SUCCESS &&
      L.pref_create(&pref) == CUBLAS_STATUS_SUCCESS &&
      L.pref_set(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &wsb, sizeof(wsb)) ==
          CUBLAS_STATUS_SUCCESS &&
      set_alignments()) {
    if (L.heuristic(h, desc, la, lb, lc, lc, pref, 1, &res, &found) != CUBLAS_STATUS_SUCCESS || found < 1) {
      s = SWA_ERR_UNSUPPORTED;
    } else if (L.matmul(h, desc, &alpha, g.A, la, g.B, lb, &g.beta, cptr, lc, g.D, lc, &res.algo, lt_ws,
                        lt_ws_bytes, st) == CUBLAS_STATUS_SUCCESS) {
      s = SWA_OK;
    }
  }
  if (pref) L.pref_destroy(pref);
  if (lc) L.layout_destroy(lc);
  if (lb) L.layout_destroy(lb);
  if (la) L.layout_destroy(la);
  if (desc) L.desc_destroy(desc);
  return s;
}

// ---------------------------------------------------------------------------
// Workspace of the block calls. The attention's own workspace (sized for its
// backward) comes first, so its status word is the block workspace's header.
// ---------------------------------------------------------------------------
constexpr size_t kLtWsBytes = 32ull << 20;   // cuBLASLt scratch
constexpr int kMaxBlockGateCh = 32;

struct BlockLayout {
  size_t attn_bytes;   // attention workspace [0, attn_bytes)
  size_t xn;           // elem [B*T, C]    normed block input
  size_t rstd;         // f32  [B*T]
  size_t q, k, v, o;   // elem [B*T, Hq*d], [B*T, Hkv*d] x 2, [B*T, Hq*d]
  size_t lse;          // f32  [B, Hq, T]
  size_t lt;           // cuBLASLt scratch
  size_t fwd_end;
  size_t dO;           // elem [B*T, Hq*d]  gradient of the attention output
  size_t dq, dk, dv;   // elem
  size_t dxn;          // f32  [B*T, C]     gradient of the normed input
  size_t dgx;          // f32  [B*T, 32]    learned gate: gradient of the channels it read
  size_t bwd_end;
};

inline BlockLayout block_layout(int B, int T, int Hq, int Hkv, int d, int C) {
  BlockLayout L;
  const size_t bt = static_cast<size_t>(B) * static_cast<size_t>(T);
  const size_t es = sizeof(elem_t);
  size_t o = align256(ws_layout(B, T, Hq, Hkv, d).bwd_end);
  L.attn_bytes = o;
  L.xn = o; o = align256(o + bt * C * es);
  L.rstd = o; o = align256(o + bt * sizeof(float));
  L.q = o; o = align256(o + bt * Hq * d * es);
  L.k = o; o = align256(o + bt * Hkv * d * es);
  L.v = o; o = align256(o + bt * Hkv * d * es);
  L.o = o; o = align256(o + bt * Hq * d * es);
  L.lse = o; o = align256(o + bt * Hq * sizeof(float));
  L.lt = o; o += kLtWsBytes;
  L.fwd_end = o;
  L.dO = o; o = align256(o + bt * Hq * d * es);
  L.dq = o; o = align256(o + bt * Hq * d * es);
  L.dk = o; o = align256(o + bt * Hkv * d * es);
  L.dv = o; o = align256(o + bt * Hkv * d * es);
  L.dxn = o; o = align256(o + bt * C * sizeof(float));
  L.dgx = o; o = align256(o + bt * kMaxBlockGateCh * sizeof(float));
  L.bwd_end = o;
  return L;
}

}  // namespace blk
}  // namespace swa
