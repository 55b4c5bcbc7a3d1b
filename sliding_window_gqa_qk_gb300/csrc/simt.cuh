// fp32 SIMT attention kernels of the debug build (libswaattn_fp32.so).
//
// They walk the same band schedule as the tensor-core kernels (64-row query
// tiles against 64-row key tiles, tiles outside the band skipped, the mask
// applied only on partial tiles) and use the same tile-wise online softmax,
// but do all arithmetic in fp32 FFMA so that the method can be checked to
// 1e-5 against the float64 oracle. The backward is split into a key-side
// kernel (dK, dV) and a query-side kernel (dQ) so that nothing is accumulated
// with atomics.
#pragma once

#include "common.cuh"

namespace swa {

constexpr int kSimtTile = 64;     // query and key tile rows
constexpr int kSimtWarps = 8;     // warps per block; each owns 8 rows of a tile

struct SimtFwdArgs {
  int B, T, Hq, Hkv, window, causal;
  float scale;
  const float* qn; const float* kn; const float* veff;   // [B, H, T, D]
  float* o;        // [B, T, Hq, D]
  float* lse;      // [B, Hq, T]
};

struct SimtBwdArgs {
  int B, T, Tpad, Hq, Hkv, window, causal;
  float scale;
  const float* qn; const float* kn; const float* veff;   // [B, H, T, D]
  const float* dO;     // [B, T, Hq, D]
  const float* lse;    // [B, Hq, T]
  const float* dvec;   // [B, Hq, Tpad]
  float* dq_acc;       // [B, Hq, T, D]  gradient of qn
  float* dk_acc;       // [B, Hkv, T, D] gradient of kn
  float* dv_acc;       // [B, Hkv, T, D] gradient of v_eff
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// Loads rows [r0, r0 + 64) of a [T, D] matrix into shared memory with row
// pitch P floats; rows at or beyond T are zero.
template <int D, int P>
__device__ __forceinline__ void load_tile(float* dst, const float* src, int r0, int T) {
  for (int idx = threadIdx.x; idx < kSimtTile * D; idx += blockDim.x) {
    const int r = idx / D, c = idx % D;
    dst[r * P + c] = (r0 + r < T) ? src[static_cast<long long>(r0 + r) * D + c] : 0.f;
  }
}

// Forward. Grid (query tiles, Hq, B). Lane l of a warp owns the scores of keys
// l and l + 32 of the current tile and the output columns l, l + 32, ...
template <int D>
__global__ void __launch_bounds__(kSimtWarps * 32) fwd_simt_kernel(SimtFwdArgs a) {
  constexpr int P = D + 1;               // padded pitch: conflict-free row reads
  constexpr int NC = D / 32;
  constexpr int RW = kSimtTile / kSimtWarps;
  extern __shared__ float sm[];
  float* sK = sm;                        // [64][P]
  float* sV = sK + kSimtTile * P;        // [64][P]
  float* sQ = sV + kSimtTile * P;        // [64][D]
  float* sP = sQ + kSimtTile * D;        // [warps][64]

  const int qt = gridDim.x - 1 - blockIdx.x;   // heavy (late) tiles first
  const int h = blockIdx.y, b = blockIdx.z;
  const int hk = h / (a.Hq / a.Hkv);
  const int lane = threadIdx.x & 31, warp = threadIdx.x / 32;
  const int q0 = qt * kSimtTile;
  const Band band{a.T, a.window, a.causal};
  const float* qbase = a.qn + (static_cast<long long>(b) * a.Hq + h) * a.T * D;
  const float* kbase = a.kn + (static_cast<long long>(b) * a.Hkv + hk) * a.T * D;
  const float* vbase = a.veff + (static_cast<long long>(b) * a.Hkv + hk) * a.T * D;

  load_tile<D, D>(sQ, qbase, q0, a.T);
  float m[RW], l[RW], acc[RW][NC];
#pragma unroll
  for (int r = 0; r < RW; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) acc[r][c] = 0.f;
  }
  int lo, hi;
  if (kv_tile_range(band, q0, kSimtTile, kSimtTile, lo, hi)) {
    for (int kt = lo; kt <= hi; ++kt) {
      const int k0 = kt * kSimtTile;
      __syncthreads();
      load_tile<D, P>(sK, kbase, k0, a.T);
      load_tile<D, P>(sV, vbase, k0, a.T);
      __syncthreads();
      const bool full = tile_full(band, q0, kSimtTile, k0, kSimtTile);
#pragma unroll
      for (int r = 0; r < RW; ++r) {
        const int i = q0 + warp * RW + r;
        if (i >= a.T) break;
        const float* qrow = sQ + (warp * RW + r) * D;
        float s0 = 0.f, s1 = 0.f;
        for (int c = 0; c < D; ++c) {
          const float qc = qrow[c];
          s0 = fmaf(qc, sK[lane * P + c], s0);
          s1 = fmaf(qc, sK[(lane + 32) * P + c], s1);
        }
        s0 *= a.scale;
        s1 *= a.scale;
        if (!full) {
          if (!visible(band, i, k0 + lane)) s0 = -INFINITY;
          if (!visible(band, i, k0 + lane + 32)) s1 = -INFINITY;
        }
        const float mt = warp_max(fmaxf(s0, s1));
        const float mnew = fmaxf(m[r], mt);
        if (mnew == -INFINITY) continue;             // nothing visible yet
        const float corr = expf(m[r] - mnew);        // 0 when m was -inf
        const float p0 = expf(s0 - mnew), p1 = expf(s1 - mnew);
        l[r] = l[r] * corr + warp_sum(p0 + p1);
        m[r] = mnew;
        float* pw = sP + warp * kSimtTile;
        pw[lane] = p0;
        pw[lane + 32] = p1;
        __syncwarp();
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[r][c] *= corr;
        for (int j = 0; j < kSimtTile; ++j) {
          const float pj = pw[j];
#pragma unroll
          for (int c = 0; c < NC; ++c) acc[r][c] = fmaf(pj, sV[j * P + lane + 32 * c], acc[r][c]);
        }
        __syncwarp();
      }
    }
  }
#pragma unroll
  for (int r = 0; r < RW; ++r) {
    const int i = q0 + warp * RW + r;
    if (i >= a.T) break;
    const bool empty = (l[r] == 0.f);
    const float inv = empty ? 0.f : 1.0f / l[r];
    float* orow = a.o + ((static_cast<long long>(b) * a.T + i) * a.Hq + h) * D;
#pragma unroll
    for (int c = 0; c < NC; ++c) orow[lane + 32 * c] = acc[r][c] * inv;
    if (lane == 0)
      a.lse[(static_cast<long long>(b) * a.Hq + h) * a.T + i] = empty ? -INFINITY : m[r] + logf(l[r]);
  }
}

// Query side of the backward: dqn_i = scale * sum_j P_ij (dP_ij - D_i) kn_j,
// with P_ij = exp(S_ij - LSE_i) and dP_ij = <dO_i, v_eff_j>. Grid (query
// tiles, Hq, B).
template <int D>
__global__ void __launch_bounds__(kSimtWarps * 32) bwd_dq_simt_kernel(SimtBwdArgs a) {
  constexpr int P = D + 1;
  constexpr int NC = D / 32;
  constexpr int RW = kSimtTile / kSimtWarps;
  extern __shared__ float sm[];
  float* sK = sm;                        // [64][P]
  float* sV = sK + kSimtTile * P;        // [64][P]
  float* sQ = sV + kSimtTile * P;        // [64][D]
  float* sG = sQ + kSimtTile * D;        // [64][D]  dO rows
  float* sP = sG + kSimtTile * D;        // [warps][64]

  const int qt = gridDim.x - 1 - blockIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
  const int hk = h / (a.Hq / a.Hkv);
  const int lane = threadIdx.x & 31, warp = threadIdx.x / 32;
  const int q0 = qt * kSimtTile;
  const Band band{a.T, a.window, a.causal};
  const long long bh = static_cast<long long>(b) * a.Hq + h;
  const float* kbase = a.kn + (static_cast<long long>(b) * a.Hkv + hk) * a.T * D;
  const float* vbase = a.veff + (static_cast<long long>(b) * a.Hkv + hk) * a.T * D;

  load_tile<D, D>(sQ, a.qn + bh * a.T * D, q0, a.T);
  for (int idx = threadIdx.x; idx < kSimtTile * D; idx += blockDim.x) {
    const int r = idx / D, c = idx % D;
    sG[idx] = (q0 + r < a.T)
                  ? a.dO[((static_cast<long long>(b) * a.T + q0 + r) * a.Hq + h) * D + c]
                  : 0.f;
  }
  float lse[RW], dd[RW], acc[RW][NC];
#pragma unroll
  for (int r = 0; r < RW; ++r) {
    const int i = q0 + warp * RW + r;
    lse[r] = i < a.T ? a.lse[bh * a.T + i] : 0.f;
    dd[r] = i < a.T ? a.dvec[bh * a.Tpad + i] : 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) acc[r][c] = 0.f;
  }
  int lo, hi;
  if (kv_tile_range(band, q0, kSimtTile, kSimtTile, lo, hi)) {
    for (int kt = lo; kt <= hi; ++kt) {
      const int k0 = kt * kSimtTile;
      __syncthreads();
      load_tile<D, P>(sK, kbase, k0, a.T);
      load_tile<D, P>(sV, vbase, k0, a.T);
      __syncthreads();
      const bool full = tile_full(band, q0, kSimtTile, k0, kSimtTile);
#pragma unroll
      for (int r = 0; r < RW; ++r) {
        const int i = q0 + warp * RW + r;
        if (i >= a.T) break;
        const float* qrow = sQ + (warp * RW + r) * D;
        const float* grow = sG + (warp * RW + r) * D;
        float s0 = 0.f, s1 = 0.f, g0 = 0.f, g1 = 0.f;
        for (int c = 0; c < D; ++c) {
          const float qc = qrow[c], gc = grow[c];
          s0 = fmaf(qc, sK[lane * P + c], s0);
          s1 = fmaf(qc, sK[(lane + 32) * P + c], s1);
          g0 = fmaf(gc, sV[lane * P + c], g0);
          g1 = fmaf(gc, sV[(lane + 32) * P + c], g1);
        }
        float p0 = expf(s0 * a.scale - lse[r]);
        float p1 = expf(s1 * a.scale - lse[r]);
        if (!full) {
          if (!visible(band, i, k0 + lane)) p0 = 0.f;
          if (!visible(band, i, k0 + lane + 32)) p1 = 0.f;
        }
        float* pw = sP + warp * kSimtTile;
        pw[lane] = p0 * (g0 - dd[r]);
        pw[lane + 32] = p1 * (g1 - dd[r]);
        __syncwarp();
        for (int j = 0; j < kSimtTile; ++j) {
          const float dsj = pw[j];
#pragma unroll
          for (int c = 0; c < NC; ++c) acc[r][c] = fmaf(dsj, sK[j * P + lane + 32 * c], acc[r][c]);
        }
        __syncwarp();
      }
    }
  }
#pragma unroll
  for (int r = 0; r < RW; ++r) {
    const int i = q0 + warp * RW + r;
    if (i >= a.T) break;
    float* dst = a.dq_acc + (bh * a.T + i) * D;
#pragma unroll
    for (int c = 0; c < NC; ++c) dst[lane + 32 * c] = acc[r][c] * a.scale;
  }
}

// Key side of the backward, one block per (key tile, kv head, batch), looping
// over the G query heads of the group and the query tiles of the band:
//   dv_eff_j += sum_i P_ij dO_i,   dkn_j += scale * sum_i P_ij (dP_ij - D_i) qn_i.
template <int D>
__global__ void __launch_bounds__(kSimtWarps * 32) bwd_dkv_simt_kernel(SimtBwdArgs a) {
  constexpr int P = D + 1;
  constexpr int NC = D / 32;
  constexpr int RW = kSimtTile / kSimtWarps;
  extern __shared__ float sm[];
  float* sQ = sm;                        // [64][P] query rows
  float* sG = sQ + kSimtTile * P;        // [64][P] dO rows
  float* sK = sG + kSimtTile * P;        // [64][D]
  float* sV = sK + kSimtTile * D;        // [64][D]
  float* sL = sV + kSimtTile * D;        // [64] LSE
  float* sD = sL + kSimtTile;            // [64] D
  float* sP = sD + kSimtTile;            // [warps][64] P
  float* sS = sP + kSimtWarps * kSimtTile;  // [warps][64] dS

  const int kt = gridDim.x - 1 - blockIdx.x;
  const int hk = blockIdx.y, b = blockIdx.z;
  const int G = a.Hq / a.Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x / 32;
  const int k0 = kt * kSimtTile;
  const Band band{a.T, a.window, a.causal};
  const long long bhk = static_cast<long long>(b) * a.Hkv + hk;

  load_tile<D, D>(sK, a.kn + bhk * a.T * D, k0, a.T);
  load_tile<D, D>(sV, a.veff + bhk * a.T * D, k0, a.T);
  float dk[RW][NC], dv[RW][NC];
#pragma unroll
  for (int r = 0; r < RW; ++r)
#pragma unroll
    for (int c = 0; c < NC; ++c) dk[r][c] = dv[r][c] = 0.f;

  int lo, hi;
  const bool any = q_tile_range(band, k0, kSimtTile, kSimtTile, lo, hi);
  for (int g = 0; any && g < G; ++g) {
    const int h = hk * G + g;
    const long long bh = static_cast<long long>(b) * a.Hq + h;
    for (int qt = lo; qt <= hi; ++qt) {
      const int q0 = qt * kSimtTile;
      __syncthreads();
      load_tile<D, P>(sQ, a.qn + bh * a.T * D, q0, a.T);
      for (int idx = threadIdx.x; idx < kSimtTile * D; idx += blockDim.x) {
        const int r = idx / D, c = idx % D;
        sG[r * P + c] = (q0 + r < a.T)
                            ? a.dO[((static_cast<long long>(b) * a.T + q0 + r) * a.Hq + h) * D + c]
                            : 0.f;
      }
      for (int r = threadIdx.x; r < kSimtTile; r += blockDim.x) {
        sL[r] = q0 + r < a.T ? a.lse[bh * a.T + q0 + r] : 0.f;
        sD[r] = q0 + r < a.T ? a.dvec[bh * a.Tpad + q0 + r] : 0.f;
      }
      __syncthreads();
      const bool full = tile_full(band, q0, kSimtTile, k0, kSimtTile);
#pragma unroll
      for (int r = 0; r < RW; ++r) {
        const int j = k0 + warp * RW + r;
        if (j >= a.T) break;
        const float* krow = sK + (warp * RW + r) * D;
        const float* vrow = sV + (warp * RW + r) * D;
        float s0 = 0.f, s1 = 0.f, g0 = 0.f, g1 = 0.f;
        for (int c = 0; c < D; ++c) {
          const float kc = krow[c], vc = vrow[c];
          s0 = fmaf(kc, sQ[lane * P + c], s0);
          s1 = fmaf(kc, sQ[(lane + 32) * P + c], s1);
          g0 = fmaf(vc, sG[lane * P + c], g0);
          g1 = fmaf(vc, sG[(lane + 32) * P + c], g1);
        }
        const int i0 = q0 + lane, i1 = q0 + lane + 32;
        float p0 = expf(s0 * a.scale - sL[lane]);
        float p1 = expf(s1 * a.scale - sL[lane + 32]);
        if (!full) {
          if (!visible(band, i0, j)) p0 = 0.f;
          if (!visible(band, i1, j)) p1 = 0.f;
        }
        float* pw = sP + warp * kSimtTile;
        float* sw = sS + warp * kSimtTile;
        pw[lane] = p0;
        pw[lane + 32] = p1;
        sw[lane] = p0 * (g0 - sD[lane]);
        sw[lane + 32] = p1 * (g1 - sD[lane + 32]);
        __syncwarp();
        for (int i = 0; i < kSimtTile; ++i) {
          const float pi = pw[i], si = sw[i];
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            dv[r][c] = fmaf(pi, sG[i * P + lane + 32 * c], dv[r][c]);
            dk[r][c] = fmaf(si, sQ[i * P + lane + 32 * c], dk[r][c]);
          }
        }
        __syncwarp();
      }
    }
  }
#pragma unroll
  for (int r = 0; r < RW; ++r) {
    const int j = k0 + warp * RW + r;
    if (j >= a.T) break;
    float* dkd = a.dk_acc + (bhk * a.T + j) * D;
    float* dvd = a.dv_acc + (bhk * a.T + j) * D;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      dkd[lane + 32 * c] = dk[r][c] * a.scale;
      dvd[lane + 32 * c] = dv[r][c];
    }
  }
}

template <int D>
constexpr size_t simt_fwd_smem() {
  return sizeof(float) * (2 * kSimtTile * (D + 1) + kSimtTile * D + kSimtWarps * kSimtTile);
}
template <int D>
constexpr size_t simt_dq_smem() {
  return sizeof(float) * (2 * kSimtTile * (D + 1) + 2 * kSimtTile * D + kSimtWarps * kSimtTile);
}
template <int D>
constexpr size_t simt_dkv_smem() {
  return sizeof(float) *
         (2 * kSimtTile * (D + 1) + 2 * kSimtTile * D + 2 * kSimtTile + 2 * kSimtWarps * kSimtTile);
}

}  // namespace swa
