// Row-wise, HBM-bound kernels around the attention core:
//   prologue   QK-norm of q and k, value-embedding mix of v   (forward)
//   bwd_pre    D = rowsum(dO * O), clear the dQ accumulator    (backward)
//   bwd_post   RMSNorm backward of q and k, dv, VE-table gradient, gain
//              gradient partials                               (backward)
//   gain_sum   deterministic sum of the gain partials           (backward)
//
// One warp owns one row of d elements (each lane d/32 consecutive elements);
// a warp processes kRowsPerIter rows per loop trip with all their loads issued
// before any arithmetic, to keep enough bytes in flight.
#pragma once

#include "common.cuh"

namespace swa {

constexpr int kRowWarps = 8;       // warps per block
constexpr int kRowsPerIter = 4;    // rows in flight per warp

// QK-norm ("RMSNorm of queries and keys right before the attention dot
// product", autoresearch train.py walkthrough post, model paragraph; the
// Administrator & Developer Guide §8.2.1 names F.rms_norm) and the
// value-embedding mix v + ve_scale * gate * VE[tok] (Guide §8.2.1,
// value-embedding row). blockIdx.y selects the segment: 0 = q rows,
// 1 = k rows, 2 = v rows (launched only on value-embedding layers).
// Inputs are [B, T, H, d]; outputs are written head-major [B, H, T, d].
template <int D>
__global__ void __launch_bounds__(kRowWarps * 32) prologue_kernel(ProArgs a) {
  constexpr int NV = D / 32;
  const int seg = blockIdx.y;
  const int H = seg == 0 ? a.Hq : a.Hkv;
  const long long rows = static_cast<long long>(a.B) * a.T * H;
  const int lane = threadIdx.x & 31;
  const int c0 = lane * NV;
  const long long nwarps = static_cast<long long>(gridDim.x) * kRowWarps;
  const long long w0 = static_cast<long long>(blockIdx.x) * kRowWarps + threadIdx.x / 32;

  if (seg < 2) {
    const elem_t* x = seg == 0 ? a.q : a.k;
    const float* gain = seg == 0 ? a.gq : a.gk;
    elem_t* y = seg == 0 ? a.qn : a.kn;
    float* rs = seg == 0 ? a.rstd_q : a.rstd_k;
    float g[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) g[i] = gain ? gain[c0 + i] : 1.0f;
    for (long long base = w0; base < rows; base += nwarps * kRowsPerIter) {
      float xv[kRowsPerIter][NV];
#pragma unroll
      for (int u = 0; u < kRowsPerIter; ++u) {
        const long long r = base + u * nwarps;
        if (r < rows) load_vec<NV>(x + r * D + c0, xv[u]);
      }
#pragma unroll
      for (int u = 0; u < kRowsPerIter; ++u) {
        const long long r = base + u * nwarps;
        if (r >= rows) break;
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i) ss = fmaf(xv[u][i], xv[u][i], ss);
        ss = warp_sum(ss);
        const float rstd = rsqrtf(ss / D + a.eps);
        float o[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) o[i] = xv[u][i] * rstd * g[i];
        const int h = static_cast<int>(r % H);
        const long long bt = r / H;
        const int t = static_cast<int>(bt % a.T);
        const long long b = bt / a.T;
        const long long orow = (b * H + h) * a.T + t;
        store_vec<NV>(y + orow * D + c0, o);
        if (lane == 0) rs[orow] = rstd;
      }
    }
  } else {
    const int Hd = a.Hkv * D;
    for (long long base = w0; base < rows; base += nwarps * kRowsPerIter) {
      float vv[kRowsPerIter][NV], ev[kRowsPerIter][NV], sc[kRowsPerIter];
#pragma unroll
      for (int u = 0; u < kRowsPerIter; ++u) {
        const long long r = base + u * nwarps;
        if (r >= rows) break;
        const int h = static_cast<int>(r % a.Hkv);
        const long long bt = r / a.Hkv;
        load_vec<NV>(a.v + r * D + c0, vv[u]);
        const int tok = a.ve ? a.tok[bt] : 0;
        sc[u] = a.ve_scale * (a.gate ? a.gate[bt * a.Hkv + h] : 1.0f);
        if (a.ve == nullptr) {
          // Plain layer (fp32 build only): v_eff is a head-major copy of v.
#pragma unroll
          for (int i = 0; i < NV; ++i) ev[u][i] = 0.f;
        } else if (tok >= 0 && tok < a.vocab) {
          load_vec<NV>(a.ve + static_cast<long long>(tok) * Hd + h * D + c0, ev[u]);
        } else {
          // An id outside the table contributes nothing and is reported.
#pragma unroll
          for (int i = 0; i < NV; ++i) ev[u][i] = 0.f;
          if (lane == 0) atomicOr(a.status, DEV_ERR_TOKEN);
        }
      }
#pragma unroll
      for (int u = 0; u < kRowsPerIter; ++u) {
        const long long r = base + u * nwarps;
        if (r >= rows) break;
        const int h = static_cast<int>(r % a.Hkv);
        const long long bt = r / a.Hkv;
        const int t = static_cast<int>(bt % a.T);
        const long long b = bt / a.T;
        float o[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) o[i] = fmaf(sc[u], ev[u][i], vv[u][i]);
        store_vec<NV>(a.veff + ((b * a.Hkv + h) * a.T + t) * D + c0, o);
      }
    }
  }
}

// D[b, h, t] = sum_c dO[b, t, h, c] * O[b, t, h, c] (the softmax-backward row
// term), LSE2[b, h, t] = LSE[b, h, t] * log2(e) (both in rows padded to Tpad),
// and (clear_acc) zero the fp32 dQ accumulator row [b, h, t, :].
template <int D>
__global__ void __launch_bounds__(kRowWarps * 32) bwd_pre_kernel(PreArgs a) {
  constexpr int NV = D / 32;
  const long long rows = static_cast<long long>(a.B) * a.T * a.Hq;
  const int lane = threadIdx.x & 31;
  const int c0 = lane * NV;
  const long long nwarps = static_cast<long long>(gridDim.x) * kRowWarps;
  const long long w0 = static_cast<long long>(blockIdx.x) * kRowWarps + threadIdx.x / 32;
  for (long long base = w0; base < rows; base += nwarps * kRowsPerIter) {
    float ov[kRowsPerIter][NV], gv[kRowsPerIter][NV];
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u) {
      const long long r = base + u * nwarps;
      if (r < rows) {
        load_vec<NV>(a.o + r * D + c0, ov[u]);
        load_vec<NV>(a.dO + r * D + c0, gv[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u) {
      const long long r = base + u * nwarps;
      if (r >= rows) break;
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i) s = fmaf(ov[u][i], gv[u][i], s);
      s = warp_sum(s);
      const int h = static_cast<int>(r % a.Hq);
      const long long bt = r / a.Hq;
      const int t = static_cast<int>(bt % a.T);
      const long long b = bt / a.T;
      const long long orow = (b * a.Hq + h) * a.T + t;
      const long long prow = (b * a.Hq + h) * a.Tpad + t;
      if (lane == 0) {
        a.dvec[prow] = s;
        a.lse2[prow] = a.lse[orow] * 1.4426950408889634f;
      }
      if (a.clear_acc) {
        float z[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) z[i] = 0.f;
        store_vec<NV>(a.dq_acc + orow * D + c0, z);
      }
    }
  }
}

// Backward of the prologue. blockIdx.y: 0 = q rows (RMSNorm backward of q from
// the gradient of qn, dgq partials), 1 = k rows (same for k), 2 = v rows
// (dv = gradient of v_eff; scatter ve_scale * gate * dv_eff into dVE).
// RMSNorm backward, with r = rstd, xh = x r, y = g xh:
//   dxh = g dy;  dx = r (dxh - xh mean(dxh xh));  dg += dy xh.
template <int D>
__global__ void __launch_bounds__(kRowWarps * 32) bwd_post_kernel(PostArgs a) {
  constexpr int NV = D / 32;
  const int seg = blockIdx.y;
  const int H = seg == 0 ? a.Hq : a.Hkv;
  const long long rows = static_cast<long long>(a.B) * a.T * H;
  const int lane = threadIdx.x & 31, warp = threadIdx.x / 32;
  const int c0 = lane * NV;
  const long long nwarps = static_cast<long long>(gridDim.x) * kRowWarps;
  const long long w0 = static_cast<long long>(blockIdx.x) * kRowWarps + warp;

  if (seg < 2) {
    const elem_t* x = seg == 0 ? a.q : a.k;
    const float* gain = seg == 0 ? a.gq : a.gk;
    const float* rs = seg == 0 ? a.rstd_q : a.rstd_k;
    const float* acc = seg == 0 ? a.dq_acc : a.dk_acc;
    elem_t* dx = seg == 0 ? a.dq : a.dk;
    float g[NV], gacc[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      g[i] = gain ? gain[c0 + i] : 1.0f;
      gacc[i] = 0.f;
    }
    for (long long base = w0; base < rows; base += nwarps * kRowsPerIter) {
      float xv[kRowsPerIter][NV], dy[kRowsPerIter][NV], rr[kRowsPerIter];
#pragma unroll
      for (int u = 0; u < kRowsPerIter; ++u) {
        const long long r = base + u * nwarps;
        if (r >= rows) break;
        const int h = static_cast<int>(r % H);
        const long long bt = r / H;
        const int t = static_cast<int>(bt % a.T);
        const long long b = bt / a.T;
        const long long orow = (b * H + h) * a.T + t;
        load_vec<NV>(x + r * D + c0, xv[u]);
        load_vec<NV>(acc + orow * D + c0, dy[u]);
        rr[u] = rs[orow];
      }
#pragma unroll
      for (int u = 0; u < kRowsPerIter; ++u) {
        const long long r = base + u * nwarps;
        if (r >= rows) break;
        float xh[NV], dxh[NV], dot = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          xh[i] = xv[u][i] * rr[u];
          dxh[i] = g[i] * dy[u][i];
          dot = fmaf(dxh[i], xh[i], dot);
          gacc[i] = fmaf(dy[u][i], xh[i], gacc[i]);
        }
        dot = warp_sum(dot) / D;
        float o[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) o[i] = rr[u] * (dxh[i] - xh[i] * dot);
        store_vec<NV>(dx + r * D + c0, o);
      }
    }
    // Block reduction of the gain partials: fixed order, no atomics.
    __shared__ float red[kRowWarps][D];
#pragma unroll
    for (int i = 0; i < NV; ++i) red[warp][c0 + i] = gacc[i];
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kRowWarps; ++w) s += red[w][c];
      a.gpart[(static_cast<long long>(seg) * gridDim.x + blockIdx.x) * D + c] = s;
    }
  } else {
    const int Hd = a.Hkv * D;
    for (long long base = w0; base < rows; base += nwarps * kRowsPerIter) {
      float dv[kRowsPerIter][NV];
#pragma unroll
      for (int u = 0; u < kRowsPerIter; ++u) {
        const long long r = base + u * nwarps;
        if (r >= rows) break;
        const int h = static_cast<int>(r % a.Hkv);
        const long long bt = r / a.Hkv;
        const int t = static_cast<int>(bt % a.T);
        const long long b = bt / a.T;
        load_vec<NV>(a.dv_acc + ((b * a.Hkv + h) * a.T + t) * D + c0, dv[u]);
      }
#pragma unroll
      for (int u = 0; u < kRowsPerIter; ++u) {
        const long long r = base + u * nwarps;
        if (r >= rows) break;
        store_vec<NV>(a.dv + r * D + c0, dv[u]);
        if (a.dve) {
          const int h = static_cast<int>(r % a.Hkv);
          const long long bt = r / a.Hkv;
          const int tok = a.tok[bt];
          if (tok >= 0 && tok < a.vocab) {
            const float s = a.ve_scale * (a.gate ? a.gate[bt * a.Hkv + h] : 1.0f);
            float* dst = a.dve + static_cast<long long>(tok) * Hd + h * D + c0;
#pragma unroll
            for (int i = 0; i < NV; ++i) atomicAdd(dst + i, s * dv[u][i]);
          }
        }
      }
    }
  }
}

// dgq[c] = sum over blocks of the q partials; dgk likewise (block 0: q, 1: k).
__global__ void gain_sum_kernel(GainArgs a) {
  float* out = blockIdx.x == 0 ? a.dgq : a.dgk;
  if (out == nullptr) return;
  const float* part = a.gpart + static_cast<long long>(blockIdx.x) * kPostBlocks * a.d;
  for (int c = threadIdx.x; c < a.d; c += blockDim.x) {
    float s = 0.f;
    for (int blk = 0; blk < kPostBlocks; ++blk) s += part[static_cast<long long>(blk) * a.d + c];
    out[c] = s;
  }
}

}  // namespace swa
