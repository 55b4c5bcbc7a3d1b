// Row-wise, HBM-bound kernels around the attention core:
//   prologue   QK-norm of q and k, value-embedding mix of v   (forward)
//   bwd_pre    D = rowsum(dO * O), LSE * log2 e, clear the dQ accumulator
//   bwd_post   RMSNorm backward of q and k, dv, VE-table gradient, gain
//              gradient partials                               (backward)
//   gain_sum   deterministic sum of the gain partials           (backward)
//
// Grids are 2-D: blockIdx.y = b * H + h, blockIdx.x = a run of consecutive
// positions t, so no per-row integer division is needed. One warp owns one
// row of d elements (each lane d/32 consecutive elements) and keeps
// kRowsPerIter rows in flight, all loads issued before any arithmetic.
#pragma once

#include "common.cuh"

namespace swa {

constexpr int kRowWarps = 8;                              // warps per block
constexpr int kRowsPerIter = 4;                           // rows in flight per warp
constexpr int kRowsPerBlock = kRowWarps * kRowsPerIter;   // 32 positions per block
constexpr int kPostRowsPerBlock = 256;                    // positions per post block

// QK-norm ("RMSNorm of queries and keys right before the attention dot
// product", autoresearch train.py walkthrough post, model paragraph; the
// Administrator & Developer Guide §8.2.1 names F.rms_norm) and the
// value-embedding mix v + ve_scale * gate * VE[tok] (Guide §8.2.1,
// value-embedding row). blockIdx.z selects the segment: 0 = q rows,
// 1 = k rows, 2 = v rows (launched on value-embedding layers, and by the fp32
// build on every layer to make a head-major copy of v).
// Inputs are [B, T, H, d]; outputs are written head-major [B, H, T, d].
template <int D>
__global__ void __launch_bounds__(kRowWarps * 32) prologue_kernel(ProArgs a) {
  constexpr int NV = D / 32;
  const int seg = blockIdx.z;
  const int H = seg == 0 ? a.Hq : a.Hkv;
  const int bh = blockIdx.y;
  if (bh >= a.B * H) return;
  const int b = bh / H, h = bh - (bh / H) * H;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = lane * NV;
  const int t0 = blockIdx.x * kRowsPerBlock + warp;      // rows t0 + u * kRowWarps
  const long long in_stride = static_cast<long long>(H) * D;
  const long long in0 = (static_cast<long long>(b) * a.T * H + h) * D + c0;   // t = 0
  const long long out0 = static_cast<long long>(bh) * a.T * D + c0;

  if (seg < 2) {
    const elem_t* x = seg == 0 ? a.q : a.k;
    const float* gain = seg == 0 ? a.gq : a.gk;
    elem_t* y = seg == 0 ? a.qn : a.kn;
    float* rs = seg == 0 ? a.rstd_q : a.rstd_k;
    float xv[kRowsPerIter][NV];
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u) {
      const int t = t0 + u * kRowWarps;
      if (t < a.T) load_vec<NV>(x + in0 + t * in_stride, xv[u]);
    }
    float g[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) g[i] = gain ? gain[c0 + i] : 1.0f;
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u) {
      const int t = t0 + u * kRowWarps;
      if (t >= a.T) break;
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i) ss = fmaf(xv[u][i], xv[u][i], ss);
      ss = warp_sum(ss);
      const float rstd = rsqrtf(ss / D + a.eps);
      float o[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) o[i] = xv[u][i] * rstd * g[i];
      store_vec<NV>(y + out0 + static_cast<long long>(t) * D, o);
      if (lane == 0) rs[static_cast<long long>(bh) * a.T + t] = rstd;
    }
  } else {
    const int Hd = a.Hkv * D;
    float vv[kRowsPerIter][NV], ev[kRowsPerIter][NV], sc[kRowsPerIter];
#pragma unroll
    for (int u = 0; u < kRowsPerIter; ++u) {
      const int t = t0 + u * kRowWarps;
      if (t >= a.T) break;
      const long long bt = static_cast<long long>(b) * a.T + t;
      load_vec<NV>(a.v + in0 + t * in_stride, vv[u]);
      sc[u] = a.ve_scale * (a.gate ? a.gate[bt * a.Hkv + h] : 1.0f);
      const int tok = a.ve ? a.tok[bt] : 0;
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
      const int t = t0 + u * kRowWarps;
      if (t >= a.T) break;
      float o[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) o[i] = fmaf(sc[u], ev[u][i], vv[u][i]);
      store_vec<NV>(a.veff + out0 + static_cast<long long>(t) * D, o);
    }
  }
}

// D[b, h, t] = sum_c dO[b, t, h, c] * O[b, t, h, c] (the softmax-backward row
// term), LSE2[b, h, t] = LSE[b, h, t] * log2(e) (both in rows padded to Tpad),
// and (clear_acc) zero the fp32 dQ accumulator row [b, h, t, :].
// Grid (ceil(T / 32), B * Hq).
template <int D>
__global__ void __launch_bounds__(kRowWarps * 32) bwd_pre_kernel(PreArgs a) {
  constexpr int NV = D / 32;
  const int bh = blockIdx.y;
  const int b = bh / a.Hq, h = bh - (bh / a.Hq) * a.Hq;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = lane * NV;
  const int t0 = blockIdx.x * kRowsPerBlock + warp;
  const long long in_stride = static_cast<long long>(a.Hq) * D;
  const long long in0 = (static_cast<long long>(b) * a.T * a.Hq + h) * D + c0;
  float ov[kRowsPerIter][NV], gv[kRowsPerIter][NV];
#pragma unroll
  for (int u = 0; u < kRowsPerIter; ++u) {
    const int t = t0 + u * kRowWarps;
    if (t < a.T) {
      load_vec<NV>(a.o + in0 + t * in_stride, ov[u]);
      load_vec<NV>(a.dO + in0 + t * in_stride, gv[u]);
    }
  }
#pragma unroll
  for (int u = 0; u < kRowsPerIter; ++u) {
    const int t = t0 + u * kRowWarps;
    if (t >= a.T) break;
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) s = fmaf(ov[u][i], gv[u][i], s);
    s = warp_sum(s);
    const long long prow = static_cast<long long>(bh) * a.Tpad + t;
    if (lane == 0) {
      a.dvec[prow] = s * a.d_mul;
      a.lse2[prow] = fmaf(a.lse[static_cast<long long>(bh) * a.T + t], a.lse2_mul, a.lse2_add);
    }
    if (a.clear_acc) {
      float z[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) z[i] = 0.f;
      store_vec<NV>(a.dq_acc + (static_cast<long long>(bh) * a.T + t) * D + c0, z);
    }
  }
}

// Backward of the prologue. Grid (ceil(T / 256), B * max(Hq, Hkv), 3);
// blockIdx.z: 0 = q rows (RMSNorm backward of q from the gradient of qn, dgq
// partials), 1 = k rows (same for k), 2 = v rows (dv = gradient of v_eff;
// scatter ve_scale * gate * dv_eff into dVE). RMSNorm backward, with
// r = rstd, xh = x r, y = g xh:
//   dxh = g dy;  dx = r (dxh - xh mean(dxh xh));  dg += dy xh.
// The gain partial of block (x, y) of segment s goes to
// gpart[s][y * gridDim.x + x][:].
template <int D>
__global__ void __launch_bounds__(kRowWarps * 32) bwd_post_kernel(PostArgs a) {
  constexpr int NV = D / 32;
  const int seg = blockIdx.z;
  const int H = seg == 0 ? a.Hq : a.Hkv;
  const int bh = blockIdx.y;
  if (bh >= a.B * H) return;
  const int b = bh / H, h = bh - (bh / H) * H;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = lane * NV;
  const long long in_stride = static_cast<long long>(H) * D;
  const long long in0 = (static_cast<long long>(b) * a.T * H + h) * D + c0;
  const long long acc0 = static_cast<long long>(bh) * a.T * D + c0;
  const int tb = blockIdx.x * kPostRowsPerBlock;
  const int tend = min(a.T, tb + kPostRowsPerBlock);

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
    for (int base = tb + warp; base < tend; base += kRowWarps * kRowsPerIter) {
      float xv[kRowsPerIter][NV], dy[kRowsPerIter][NV], rr[kRowsPerIter];
#pragma unroll
      for (int u = 0; u < kRowsPerIter; ++u) {
        const int t = base + u * kRowWarps;
        if (t >= tend) break;
        load_vec<NV>(x + in0 + t * in_stride, xv[u]);
        load_vec<NV>(acc + acc0 + static_cast<long long>(t) * D, dy[u]);
        rr[u] = rs[static_cast<long long>(bh) * a.T + t];
      }
#pragma unroll
      for (int u = 0; u < kRowsPerIter; ++u) {
        const int t = base + u * kRowWarps;
        if (t >= tend) break;
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
        store_vec<NV>(dx + in0 + t * in_stride, o);
      }
    }
    // Block reduction of the gain partials: fixed order, no atomics.
    __shared__ float red[kRowWarps][D];
#pragma unroll
    for (int i = 0; i < NV; ++i) red[warp][c0 + i] = gacc[i];
    __syncthreads();
    const long long blk = static_cast<long long>(bh) * gridDim.x + blockIdx.x;
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kRowWarps; ++w) s += red[w][c];
      a.gpart[(static_cast<long long>(seg) * a.nblk_max + blk) * D + c] = s;
    }
  } else {
    const int Hd = a.Hkv * D;
    for (int base = tb + warp; base < tend; base += kRowWarps * kRowsPerIter) {
      float dv[kRowsPerIter][NV];
#pragma unroll
      for (int u = 0; u < kRowsPerIter; ++u) {
        const int t = base + u * kRowWarps;
        if (t >= tend) break;
        load_vec<NV>(a.dv_acc + acc0 + static_cast<long long>(t) * D, dv[u]);
      }
#pragma unroll
      for (int u = 0; u < kRowsPerIter; ++u) {
        const int t = base + u * kRowWarps;
        if (t >= tend) break;
        store_vec<NV>(a.dv + in0 + t * in_stride, dv[u]);
        if (a.dve) {
          const long long bt = static_cast<long long>(b) * a.T + t;
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

// dgq[c] = sum of the q partials, dgk[c] = sum of the k partials (written by
// the backward-post kernel, or by the attention backward's epilogue), in a
// fixed order. Grid (2, d / 32), 256 threads: column = 32 * blockIdx.y + lane,
// each warp sums every 8th partial, then the 8 sums are added in order.
__global__ void __launch_bounds__(256) gain_sum_kernel(GainArgs a) {
  float* out = blockIdx.x == 0 ? a.dgq : a.dgk;
  if (out == nullptr) return;
  const int nblk = blockIdx.x == 0 ? a.n_q : a.n_k;
  const float* part = blockIdx.x == 0 ? a.part_q : a.part_k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.y * 32 + lane;
  float s = 0.f;
  for (int blk = warp; blk < nblk; blk += 8) s += part[static_cast<long long>(blk) * a.d + c];
  __shared__ float red[8][32];
  red[warp][lane] = s;
  __syncthreads();
  if (warp == 0) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[w][lane];
    out[c] = tot;
  }
}

}  // namespace swa
