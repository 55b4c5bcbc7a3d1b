// The attention block around the attention core: the block's pre-norm, the
// four bias-free projections c_q, c_k, c_v, c_proj and the residual
// (autoresearch Administrator & Developer Guide §8.2.1 model table, "Pre-norm
// + residual": x = x + attn(norm(x)); train.py walkthrough post, model
// paragraph: RMSNorm on the block inputs).
//
// The pre-norm and its backward are row-wise kernels here. The projections
// are GEMMs of this library: the tcgen05 kernel of tc_gemm.cuh in the bf16
// library (bf16 operands, fp32 accumulation), a plain fp32 SIMT kernel in the
// fp32 debug library.
#pragma once

#include "rowwise.cuh"
#if !defined(SWA_ELEM_FP32)
#include "tc_gemm.cuh"
#endif

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

// With gate_w (the learned value-embedding gate, on the fused projection
// path) it also writes gate[r, h] = 2 sigmoid(<gate_w[h], xn[r, :gch]>) for
// the Hkv kv heads, from the stored (rounded) xn: the value the prologue
// kernel computes otherwise. gch <= 32.
__global__ void __launch_bounds__(kPnWarps * 32) prenorm_fwd_kernel(const elem_t* __restrict__ x,
                                                                    elem_t* __restrict__ xn,
                                                                    float* __restrict__ rstd,
                                                                    long long rows, int C, float eps,
                                                                    const float* __restrict__ gate_w, int gch,
                                                                    int Hkv, float* __restrict__ gate_out) {
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
    float g0[kPnEpl];   // this lane's first stored values (the gate reads channels < gch)
#pragma unroll
    for (int i = 0; i < kPnEpl; ++i) g0[i] = 0.f;
    for (int c = lane * kPnEpl; c < C; c += 32 * kPnEpl) {
      float f[kPnEpl];
      unpack16(ld16(xr + c), f);
#pragma unroll
      for (int i = 0; i < kPnEpl; ++i) f[i] *= rs;
      const uint4 u = pack16(f);
      st16(yr + c, u);
      if (c < 32) unpack16(u, g0);
    }
    if (lane == 0) rstd[r] = rs;
    if (gate_w != nullptr) {
      for (int h = 0; h < Hkv; ++h) {
        float z = 0.f;
#pragma unroll
        for (int i = 0; i < kPnEpl; ++i) {
          const int c = lane * kPnEpl + i;
          if (c < gch) z = fmaf(gate_w[h * gch + c], g0[i], z);
        }
        z = row_sum<32>(z);
        if (lane == 0) gate_out[r * Hkv + h] = 2.0f / (1.0f + expf(-z));
      }
    }
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

// The rotary tables transposed for the fused q / k epilogue: out[0][c][t] =
// cos[t][c], out[1][c][t] = sin[t][c] (t < T, c < 64, head dim 128), so that
// the 32 lanes of a warp (32 consecutive positions) read one column in one
// 128-byte line. Block (32 positions, table blockIdx.y), 256 threads.
constexpr int kRtT = 32, kRtHalf = 64;
__global__ void __launch_bounds__(256) rope_transpose_kernel(const float* __restrict__ rcos,
                                                             const float* __restrict__ rsin,
                                                             float* __restrict__ out, int T) {
  __shared__ float tile[kRtT][kRtHalf + 1];
  const int t0 = blockIdx.x * kRtT;
  const float* src = blockIdx.y ? rsin : rcos;
#pragma unroll
  for (int r = 0; r < kRtT * kRtHalf / 256; ++r) {
    const int i = threadIdx.x + 256 * r, tt = i / kRtHalf, c = i % kRtHalf;
    tile[tt][c] = t0 + tt < T ? src[static_cast<long long>(t0 + tt) * kRtHalf + c] : 0.f;
  }
  __syncthreads();
  float* dst = out + static_cast<long long>(blockIdx.y) * kRtHalf * T;
#pragma unroll
  for (int r = 0; r < kRtT * kRtHalf / 256; ++r) {
    const int i = threadIdx.x + 256 * r, c = i / kRtT, tt = i % kRtT;
    if (t0 + tt < T) dst[static_cast<long long>(c) * T + t0 + tt] = tile[tt][c];
  }
}

inline int prenorm_grid(long long rows) {
  const long long per = (rows + kPnWarps - 1) / kPnWarps;
  const long long cap = static_cast<long long>(num_sms()) * kPnBlocksPerSm;
  return static_cast<int>(per < cap ? (per < 1 ? 1 : per) : cap);
}

#if defined(SWA_ELEM_FP32)
// ---------------------------------------------------------------------------
// fp32 debug GEMM: one thread per output element, fp32 accumulation over the
// K segments in order (the same GemmCall as the tensor-core kernel).
// ---------------------------------------------------------------------------
struct SimtGemmArgs {
  int M, N, n_kseg;
  bool a_mn, b_mn;
  const float* A[3];
  long long lda[3];
  int K[3];
  const float* B[3];
  long long ldb[3];
  float* D;
  long long ldd;
  const float* C;
  long long ldc;
  float beta;
};

__global__ void __launch_bounds__(256) gemm_simt_kernel(const SimtGemmArgs a) {
  const int n = blockIdx.x * 32 + threadIdx.x;
  const int m = blockIdx.y * 8 + threadIdx.y;
  if (m >= a.M || n >= a.N) return;
  float acc = 0.f;
  for (int s = 0; s < a.n_kseg; ++s) {
    const float* A = a.A[s];
    const float* B = a.B[s];
    for (int k = 0; k < a.K[s]; ++k) {
      const float av = a.a_mn ? A[static_cast<long long>(k) * a.lda[s] + m] : A[static_cast<long long>(m) * a.lda[s] + k];
      const float bv = a.b_mn ? B[static_cast<long long>(k) * a.ldb[s] + n] : B[static_cast<long long>(n) * a.ldb[s] + k];
      acc = fmaf(av, bv, acc);
    }
  }
  if (a.C != nullptr && a.beta != 0.f) acc = fmaf(a.beta, a.C[static_cast<long long>(m) * a.ldc + n], acc);
  a.D[static_cast<long long>(m) * a.ldd + n] = acc;
}

inline swa_status run_gemm(const GemmCall& g, cudaStream_t st) {
  if (g.M == 0) return SWA_OK;
  for (int j = 0; j < g.n_nseg; ++j) {
    const auto& o = g.nseg[j];
    if (o.N == 0) continue;
    SimtGemmArgs a{};
    a.M = g.M; a.N = o.N; a.n_kseg = g.n_kseg; a.a_mn = g.a_mn; a.b_mn = g.b_mn;
    for (int s = 0; s < g.n_kseg; ++s) {
      a.A[s] = static_cast<const float*>(g.kseg[s].A); a.lda[s] = g.kseg[s].lda; a.K[s] = g.kseg[s].K;
      const auto& b = g.bseg[g.n_kseg > 1 ? s : j];
      a.B[s] = static_cast<const float*>(b.B); a.ldb[s] = b.ldb;
    }
    a.D = static_cast<float*>(o.D); a.ldd = o.ldd;
    a.C = static_cast<const float*>(o.C); a.ldc = o.ldc; a.beta = g.beta;
    dim3 grid((o.N + 31) / 32, (g.M + 7) / 8);
    gemm_simt_kernel<<<grid, dim3(32, 8), 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SWA_ERR_CUDA;
  }
  return SWA_OK;
}
#else
inline swa_status run_gemm(const GemmCall& g, cudaStream_t st) { return tc::launch_gemm(g, st); }
#endif

// ---------------------------------------------------------------------------
// Workspace of the block calls. The attention's own workspace (sized for its
// backward) comes first, so its status word is the block workspace's header.
// ---------------------------------------------------------------------------
constexpr int kMaxBlockGateCh = 32;

struct BlockLayout {
  size_t attn_bytes;   // attention workspace [0, attn_bytes)
  size_t xn;           // elem [B*T, C]    normed block input
  size_t rstd;         // f32  [B*T]
  size_t q, k, v, o;   // elem [B*T, Hq*d], [B*T, Hkv*d] x 2, [B*T, Hq*d]
  size_t lse;          // f32  [B, Hq, T]
  size_t rope_t;       // f32  [2][d/2][T]  rotary tables transposed (fused q / k epilogue)
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
  L.rope_t = o; o = align256(o + static_cast<size_t>(T) * d * sizeof(float));
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
