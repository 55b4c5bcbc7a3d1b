// Shared definitions of the attention-block kernels: element type of the
// build, kernel argument blocks, workspace layout and the band schedule.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

#if defined(SWA_ELEM_FP32)
using elem_t = float;
#else
using elem_t = __nv_bfloat16;
#endif

namespace swa {

// SM count of the current device (looked up once per device).
inline int num_sms() {
  constexpr int kMaxDev = 64;
  static int n_sm[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 1;
  if (n_sm[dev] <= 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    n_sm[dev] = n;
  }
  return n_sm[dev];
}

// ---------------------------------------------------------------------------
// Element conversions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Loads / stores N (2 or 4) consecutive elements as one vector access.
template <int N>
__device__ __forceinline__ void load_vec(const float* p, float (&out)[N]) {
  static_assert(N == 2 || N == 4, "");
  if constexpr (N == 4) {
    float4 t = *reinterpret_cast<const float4*>(p);
    out[0] = t.x; out[1] = t.y; out[2] = t.z; out[3] = t.w;
  } else {
    float2 t = *reinterpret_cast<const float2*>(p);
    out[0] = t.x; out[1] = t.y;
  }
}
template <int N>
__device__ __forceinline__ void load_vec(const __nv_bfloat16* p, float (&out)[N]) {
  static_assert(N == 2 || N == 4, "");
  if constexpr (N == 4) {
    uint2 t = *reinterpret_cast<const uint2*>(p);
    out[0] = __uint_as_float(t.x << 16); out[1] = __uint_as_float(t.x & 0xFFFF0000u);
    out[2] = __uint_as_float(t.y << 16); out[3] = __uint_as_float(t.y & 0xFFFF0000u);
  } else {
    uint32_t t = *reinterpret_cast<const uint32_t*>(p);
    out[0] = __uint_as_float(t << 16); out[1] = __uint_as_float(t & 0xFFFF0000u);
  }
}
template <int N>
__device__ __forceinline__ void store_vec(float* p, const float (&in)[N]) {
  if constexpr (N == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(in[0], in[1], in[2], in[3]);
  } else {
    *reinterpret_cast<float2*>(p) = make_float2(in[0], in[1]);
  }
}
template <int N>
__device__ __forceinline__ void store_vec(__nv_bfloat16* p, const float (&in)[N]) {
  if constexpr (N == 4) {
    *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(in[0], in[1]), pack_bf16x2(in[2], in[3]));
  } else {
    *reinterpret_cast<uint32_t*>(p) = pack_bf16x2(in[0], in[1]);
  }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// ---------------------------------------------------------------------------
// Band schedule: which key tiles a query tile touches, and which of those are
// entirely inside the visible band (no per-element mask needed).
//
// Visibility of key j to query i (0 <= i, j < T):
//   causal:     j <= i and (window < 0 or i - j <= window)
//   non-causal: window < 0 or |i - j| <= window
// ---------------------------------------------------------------------------
struct Band {
  int T;
  int window;  // < 0: none
  int causal;
};

__host__ __device__ __forceinline__ bool visible(const Band& b, int i, int j) {
  if (j >= b.T || i >= b.T) return false;
  if (b.causal) return j <= i && (b.window < 0 || i - j <= b.window);
  const int dd = i > j ? i - j : j - i;
  return b.window < 0 || dd <= b.window;
}

// Key tiles [lo, hi] (tile size bn) that hold a key visible to some query of
// rows [q0, q0 + bm) (clipped to T). Returns false when there are none.
__host__ __device__ __forceinline__ bool kv_tile_range(const Band& b, int q0, int bm, int bn,
                                                       int& lo, int& hi) {
  const int q1 = (q0 + bm < b.T ? q0 + bm : b.T) - 1;
  if (q1 < q0) return false;
  int klo = 0, khi = b.T - 1;
  if (b.window >= 0) {
    klo = q0 - b.window;
    if (klo < 0) klo = 0;
    if (!b.causal && q1 + b.window < khi) khi = q1 + b.window;
  }
  if (b.causal) khi = q1;
  lo = klo / bn;
  hi = khi / bn;
  return true;
}

// Query tiles [lo, hi] (tile size bm) that hold a query seeing some key of
// rows [k0, k0 + bn) (clipped to T).
__host__ __device__ __forceinline__ bool q_tile_range(const Band& b, int k0, int bn, int bm,
                                                      int& lo, int& hi) {
  const int k1 = (k0 + bn < b.T ? k0 + bn : b.T) - 1;
  if (k1 < k0) return false;
  int qlo = 0, qhi = b.T - 1;
  if (b.causal) qlo = k0;
  if (b.window >= 0) {
    if (k1 + b.window < qhi) qhi = k1 + b.window;
    if (!b.causal) {
      qlo = k0 - b.window;
      if (qlo < 0) qlo = 0;
    }
  }
  lo = qlo / bm;
  hi = qhi / bm;
  return true;
}

// True when every (query, key) pair of the two tiles is visible and inside
// [0, T): the tile needs no mask.
__host__ __device__ __forceinline__ bool tile_full(const Band& b, int q0, int bm, int k0, int bn) {
  const int q1 = q0 + bm - 1, k1 = k0 + bn - 1;
  if (q1 >= b.T || k1 >= b.T) return false;
  if (b.causal) return k1 <= q0 && (b.window < 0 || q1 - k0 <= b.window);
  return b.window < 0 || (q1 - k0 <= b.window && k1 - q0 <= b.window);
}

// ---------------------------------------------------------------------------
// Workspace layout (byte offsets from the workspace base; each region 256-byte
// aligned). Shapes use BHTD order (head-major) for the per-head tensors the
// attention kernels stream, so that one head's rows are contiguous.
// ---------------------------------------------------------------------------
struct WsLayout {
  size_t status;    // uint32 status word (header, 256 bytes); bytes 8..23:
                    // record of a zeroed dQ accumulator (offset, length)
  size_t qn;        // elem [B, Hq, T, d]
  size_t kn;        // elem [B, Hkv, T, d]
  size_t veff;      // elem [B, Hkv, T, d]
  size_t rstd_q;    // f32  [B, Hq, T]
  size_t rstd_k;    // f32  [B, Hkv, T]
  size_t gate;      // f32  [B, T, Hkv]     learned value-embedding gate values
  size_t fwd_end;
  size_t lse2;      // f32  [B, Hq, Tpad]   LSE * log2(e)
  size_t dvec;      // f32  [B, Hq, Tpad]   D = rowsum(dO * O)
  size_t dq_acc;    // f32  [B, Hq, T, d]   gradient of qn
  size_t dk_acc;    // f32  [B, Hkv, T, d]  gradient of kn
  size_t dv_acc;    // f32  [B, Hkv, T, d]  gradient of v_eff
  size_t gpart;     // f32  [2, post_blocks, d] per-block partial gain gradients
  size_t gpart_k;   // f32  [B * Hkv * ceil(T / 128), d] per-key-tile partials of dgk
  size_t gpart_w;   // f32  [post_blocks, 32 * 32] per-block partials of the gate weight gradient
  size_t bwd_end;
};

// Blocks of one backward-post segment: runs of 256 positions x (batch, head)
// pairs of the larger head count.
__host__ __device__ __forceinline__ int post_blocks(int B, int T, int Hq) {
  return (T + 255) / 256 * B * Hq;
}

__host__ __device__ __forceinline__ size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Per-head row vectors of the backward are padded to a multiple of 128 rows so
// that every 64- or 128-row slice starts 256-byte aligned (bulk copies).
__host__ __device__ __forceinline__ int t_pad(int T) { return (T + 127) / 128 * 128; }

__host__ __device__ inline WsLayout ws_layout(int B, int T, int Hq, int Hkv, int d) {
  WsLayout L;
  const size_t bt = static_cast<size_t>(B) * static_cast<size_t>(T);
  const size_t es = sizeof(elem_t);
  size_t o = 0;
  L.status = o; o += 256;
  L.qn = o; o = align256(o + bt * Hq * d * es);
  L.kn = o; o = align256(o + bt * Hkv * d * es);
  L.veff = o; o = align256(o + bt * Hkv * d * es);
  L.rstd_q = o; o = align256(o + bt * Hq * 4);
  L.rstd_k = o; o = align256(o + bt * Hkv * 4);
  L.gate = o; o = align256(o + bt * Hkv * 4);
  L.fwd_end = o;
  const size_t btp = static_cast<size_t>(B) * static_cast<size_t>(t_pad(T));
  L.lse2 = o; o = align256(o + btp * Hq * 4);
  L.dvec = o; o = align256(o + btp * Hq * 4);
  L.dq_acc = o; o = align256(o + bt * Hq * d * 4);
  L.dk_acc = o; o = align256(o + bt * Hkv * d * 4);
  L.dv_acc = o; o = align256(o + bt * Hkv * d * 4);
  L.gpart = o; o = align256(o + size_t(2) * post_blocks(B, T, Hq) * d * 4);
  L.gpart_k = o; o = align256(o + static_cast<size_t>(B) * Hkv * ((T + 127) / 128) * d * 4);
  L.gpart_w = o; o = align256(o + static_cast<size_t>(post_blocks(B, T, Hq)) * 32 * 32 * 4);
  L.bwd_end = o;
  return L;
}

// ---------------------------------------------------------------------------
// Kernel argument blocks
// ---------------------------------------------------------------------------
struct ProArgs {  // QK-norm + VE-mix prologue
  int B, T, Hq, Hkv, d, vocab;
  int nseg;         // 2: q and k rows; 3: also v rows
  float eps, ve_scale;
  const elem_t* q; const elem_t* k; const elem_t* v;
  const float* gq; const float* gk;
  const elem_t* ve; const int32_t* tok; const float* gate;
  elem_t* qn; elem_t* kn; elem_t* veff;
  float* rstd_q; float* rstd_k;
  const float* rcos; const float* rsin;   // rotary tables [rows, d/2], NULL: none
  // learned value-embedding gate (gw NULL: none): input rows, weights
  // [Hkv][gch], and where the gate values go ([B, T, Hkv])
  const elem_t* gx; long long gx_stride; const float* gw; int gch;
  float* gate_out;
  uint32_t* status;
};

struct PreArgs {  // backward preprocess: D = rowsum(dO * O), LSE2, clear dQ accumulator
  int B, T, Tpad, Hq, Hkv, d;
  const elem_t* o; const elem_t* dO; const float* lse;
  float* dvec; float* lse2; float* dq_acc;
  int clear_acc;
  // Record (offset, length) of a zeroed dQ accumulator left by the forward;
  // the clear is skipped when it names exactly this call's accumulator.
  const unsigned long long* acc_flag;
  unsigned long long acc_off, acc_len;
  const uint32_t* status;   // device status word: the record does not count after a timeout
  // dvec = d_mul * D, lse2 = lse2_mul * LSE + lse2_add (the forms the
  // attention backward kernels consume)
  float d_mul, lse2_mul, lse2_add;
};

struct PostArgs {  // backward post: RMSNorm backward, dv, dVE, gain partials
  int B, T, Hq, Hkv, d, vocab;
  float ve_scale;
  const elem_t* q; const elem_t* k;
  const float* gq; const float* gk;
  const int32_t* tok; const float* gate;
  const float* rstd_q; const float* rstd_k;
  const float* dq_acc; const float* dk_acc; const float* dv_acc;
  elem_t* dq; elem_t* dk; elem_t* dv;
  float* dve;        // NULL: skip
  float* gpart;      // [2, nblk_max, d]
  int nblk_max;      // post_blocks(B, T, Hq)
  const float* rcos; const float* rsin;   // rotary tables [rows, d/2], NULL: none
  uint32_t* status;
};

struct GainArgs {
  int d;                          // partial row length (a multiple of 32)
  const float* part_q; int n_q;   // partials of dgq: [n_q][d]
  const float* part_k; int n_k;   // partials of dgk: [n_k][d]
  float* dgq; float* dgk;
  int n_out;                      // columns written (<= d)
};

struct GateBwdArgs {  // backward of the learned value-embedding gate
  int B, T, Hkv, vocab, gch;
  long long gx_stride;
  float ve_scale;
  const elem_t* dv;    // [B, T, Hkv, d] gradient of v_eff (final dv)
  const elem_t* ve; const int32_t* tok;
  const float* gate;   // [B, T, Hkv] gate values of the forward
  const elem_t* gx; const float* gw;
  float* d_gx;         // [B, T, gch] or NULL
  float* gpart_w;      // [gridDim.x][1024]: [h * gch + c] partials of the weight gradient
};

// ---------------------------------------------------------------------------
// Projection GEMMs of the block (tc_gemm.cuh in the bf16 library, a SIMT
// kernel in the fp32 debug library)
// ---------------------------------------------------------------------------
enum GemmOut : int {
  GEMM_OUT_ELEM = 0,      // elem stores (D = A B + beta C, C elem or none)
  GEMM_OUT_F32 = 1,       // fp32 stores
  GEMM_OUT_F32_ADD = 2    // fp32 additions into D (K split over CTAs; D zeroed first)
};

// One GEMM, in row-major terms:
//   D_j[M][N_j] = sum over K segments s of A_s B_s  (+ beta C_j)
// A_s: [M][K_s] (a_mn false, row stride lda) or [K_s][M] (a_mn true).
// B:   [N][K] (b_mn false) or [K][N] (b_mn true), one tensor per K segment
//      (n_kseg > 1) or per N segment (n_kseg == 1).
// N segments (outputs) other than the last are multiples of 128 long, all
// multiples of 8; K segments other than the last multiples of 64. A, B and
// C are elem; D is elem (GEMM_OUT_ELEM) or fp32.
struct GemmCall {
  int M = 0;
  bool a_mn = false, b_mn = false;
  int n_kseg = 1;
  struct { const void* A; long long lda; int K; } kseg[3] = {};
  struct { const void* B; long long ldb; } bseg[3] = {};
  int n_nseg = 1;
  struct { int N; void* D; long long ldd; const void* C; long long ldc; } nseg[3] = {};
  int out = GEMM_OUT_ELEM;
  float beta = 0.f;
  int split = 1;           // requested K splits (fp32 outputs)
  uint32_t* status = nullptr;
  uint64_t wait_limit_ns = 2000000000ull;
  // The q, k, v projection with the attention's prologue in its epilogue
  // (bf16 library, head dim 128, T a multiple of 32, three N segments q, k,
  // v): besides the projections (D of the segments), qn and kn = the
  // QK-norm of the (rotated) q and k rows and their inverse RMS, head-major,
  // and on value-embedding layers v_eff = v + ve_scale * gate * VE[tok],
  // head-major, exactly as the prologue kernel writes them.
  struct {
    bool on;
    int T, Hq, Hkv, vocab;
    float eps, ve_scale;
    const float* gq; const float* gk;        // [128] or NULL (unit)
    const float* rope_t;                     // [2][64][T]: cos, sin transposed (position fastest), or NULL
    void* qn; void* kn; void* veff;          // [B, H, T, 128]
    float* rstd_q; float* rstd_k;            // [B, H, T]
    const void* ve; const int32_t* tok;      // VE table [vocab][Hkv * 128] or NULL
    const float* gate;                       // [B, T, Hkv] or NULL (1)
  } qkv = {};
};

}  // namespace swa
