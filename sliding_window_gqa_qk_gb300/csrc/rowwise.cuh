// Row-wise, HBM-bound kernels around the attention core:
//   prologue   QK-norm of q and k, value-embedding mix of v   (forward)
//   bwd_pre    D = rowsum(dO * O), LSE * log2 e, clear the dQ accumulator
//              (unless the forward left it zeroed)
//   bwd_post   RMSNorm backward of q and k, dv, VE-table gradient, gain
//              gradient partials                               (backward)
//   gain_sum   deterministic sum of the gain partials           (backward)
//
// The first three are persistent: a grid of a few blocks per SM whose warps
// walk a flat list of row groups (kRowSlots x rows-per-instruction
// consecutive positions of one (batch, head) row), group w, w + W, w + 2W,
// ... for warp w of W, so every warp gets the same amount of work. Each lane
// moves one 16-byte vector of a row per access (8 bf16 or 4 fp32 elements),
// LPR lanes cover a row, and a warp keeps kRowSlots such accesses per tensor
// in flight before any arithmetic. Row reductions are shuffles over the LPR
// lanes of a row.
#pragma once

#include "common.cuh"

namespace swa {

constexpr int kRowWarps = 8;        // warps per block of the row-wise kernels
constexpr int kPreBlocksPerSm = 4;  // persistent blocks per SM (register budget 64)
constexpr int kProBlocksPerSm = 2;  // prologue: register budget 128
constexpr int kPostBlocksPerSm = 2; // post: register budget 128
constexpr int kRowSlots = 4;        // 16-byte accesses in flight per lane and tensor
constexpr int kProSlots = 8;        // the prologue's (one tensor per row group)

// Lane layout of a D-element row of elem_t.
template <int D, int SLOTS = kRowSlots>
struct RowMap {
  static constexpr int EPL = 16 / static_cast<int>(sizeof(elem_t));  // elements per lane
  static constexpr int LPR = D / EPL;                                // lanes per row
  static constexpr int RPI = 32 / LPR;                               // rows per warp access
  static constexpr int RG = SLOTS * RPI;                             // rows per group
  static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "row layout");
};

// 16 bytes of elem_t <-> EPL floats.
__device__ __forceinline__ void unpack16(const uint4& r, float (&f)[8]) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void unpack16(const uint4& r, float (&f)[4]) {
  f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
  f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
}
__device__ __forceinline__ uint4 pack16(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}
__device__ __forceinline__ uint4 pack16(const float (&f)[4]) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                    __float_as_uint(f[3]));
}
__device__ __forceinline__ uint4 ld16(const void* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ void st16(void* p, const uint4& v) { *reinterpret_cast<uint4*>(p) = v; }

// n consecutive fp32 values (n = 4 or 8) as 16-byte accesses.
template <int N>
__device__ __forceinline__ void ldf(const float* p, float (&f)[N]) {
#pragma unroll
  for (int i = 0; i < N; i += 4) {
    const float4 t = *reinterpret_cast<const float4*>(p + i);
    f[i] = t.x; f[i + 1] = t.y; f[i + 2] = t.z; f[i + 3] = t.w;
  }
}
template <int N>
__device__ __forceinline__ void stf(float* p, const float (&f)[N]) {
#pragma unroll
  for (int i = 0; i < N; i += 4) *reinterpret_cast<float4*>(p + i) = make_float4(f[i], f[i + 1], f[i + 2], f[i + 3]);
}

// Sum over the LPR lanes of a row.
template <int LPR>
__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Rotary position embedding of one row, as the lanes hold it: channel c is
// paired with c + D/2, which sits LPR/2 lanes away, and the pair at position
// t turns by the angle whose cosine and sine are cos[t, c], sin[t, c]
// (c < D/2):  y_c = x_c cos + x_{c+D/2} sin,  y_{c+D/2} = -x_c sin + x_{c+D/2} cos.
// sgn = +1 applies the rotation, -1 its transpose (the backward). Every lane
// of the warp calls this (shuffles); rows past the end pass valid = false.
template <int D>
__device__ __forceinline__ void rotate_row(float (&x)[RowMap<D>::EPL], const float* rcos, const float* rsin,
                                           int t, bool valid, float sgn) {
  using M = RowMap<D>;
  constexpr int EPL = M::EPL;
  const int cl = (threadIdx.x & 31) % M::LPR;
  const bool first = cl < M::LPR / 2;
  float p[EPL], cs[EPL], sn[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) p[i] = __shfl_xor_sync(0xffffffffu, x[i], M::LPR / 2);
  if (valid) {
    const long long base = static_cast<long long>(t) * (D / 2) + (cl % (M::LPR / 2)) * EPL;
    ldf<EPL>(rcos + base, cs);
    ldf<EPL>(rsin + base, sn);
  } else {
#pragma unroll
    for (int i = 0; i < EPL; ++i) cs[i] = sn[i] = 0.f;
  }
  const float s = first ? sgn : -sgn;
#pragma unroll
  for (int i = 0; i < EPL; ++i) x[i] = fmaf(x[i], cs[i], s * p[i] * sn[i]);
}

// Warp index over the grid and the number of warps of the grid.
__device__ __forceinline__ long long grid_warp() {
  return static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
}
__device__ __forceinline__ long long grid_warps() {
  return static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
}

// QK-norm ("RMSNorm of queries and keys right before the attention dot
// product", autoresearch train.py walkthrough post, model paragraph; the
// Administrator & Developer Guide §8.2.1 names F.rms_norm) and the
// value-embedding mix v + ve_scale * gate * VE[tok] (Guide §8.2.1,
// value-embedding row). The group list holds the q rows, then the k rows,
// then (nseg = 3: value-embedding layers, and every layer of the fp32 build,
// which makes a head-major copy of v) the v rows. Inputs are [B, T, H, d];
// outputs are written head-major [B, H, T, d]. ROPE: q and k rows are
// rotated (rotate_row) before the norm. GATE: the v rows' gate is the
// learned 2 sigmoid(<w_h, x[b, t, :C]>), also written to a.gate_out.
template <int D, bool ROPE, bool GATE>
__global__ void __launch_bounds__(kRowWarps * 32, kProBlocksPerSm)
    prologue_kernel(ProArgs a) {
  using M = RowMap<D, kProSlots>;
  constexpr int EPL = M::EPL;
  const int lane = threadIdx.x & 31;
  const int slot = lane / M::LPR, c0 = (lane % M::LPR) * EPL;
  const int ngt = (a.T + M::RG - 1) / M::RG;
  const long long n_q = static_cast<long long>(a.B) * a.Hq * ngt;
  const long long n_k = static_cast<long long>(a.B) * a.Hkv * ngt;
  const long long n_all = n_q + n_k * (a.nseg == 3 ? 2 : 1);
  float gq[EPL], gk[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    gq[i] = a.gq ? a.gq[c0 + i] : 1.0f;
    gk[i] = a.gk ? a.gk[c0 + i] : 1.0f;
  }
  const int Hd = a.Hkv * D;
  for (long long gi = grid_warp(); gi < n_all; gi += grid_warps()) {
    const int seg = gi < n_q ? 0 : (gi < n_q + n_k ? 1 : 2);
    const long long loc = gi - (seg == 0 ? 0 : (seg == 1 ? n_q : n_q + n_k));
    const int H = seg == 0 ? a.Hq : a.Hkv;
    const int bh = static_cast<int>(loc / ngt);
    const int tg = static_cast<int>(loc - static_cast<long long>(bh) * ngt) * M::RG + slot;
    const int b = bh / H, h = bh - b * H;
    const long long in0 = (static_cast<long long>(b) * a.T * H + h) * D + c0;   // t = 0
    const long long in_stride = static_cast<long long>(H) * D;
    const long long out0 = static_cast<long long>(bh) * a.T * D + c0;
    if (seg < 2) {
      const elem_t* x = seg == 0 ? a.q : a.k;
      elem_t* y = seg == 0 ? a.qn : a.kn;
      float* rs = seg == 0 ? a.rstd_q : a.rstd_k;
      uint4 xr[kProSlots];
#pragma unroll
      for (int u = 0; u < kProSlots; ++u) {
        const int t = tg + u * M::RPI;
        xr[u] = t < a.T ? ld16(x + in0 + t * in_stride) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kProSlots; ++u) {
        const int t = tg + u * M::RPI;
        float xv[EPL];
        unpack16(xr[u], xv);
        if (ROPE) rotate_row<D>(xv, a.rcos, a.rsin, t, t < a.T, 1.f);
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) ss = fmaf(xv[i], xv[i], ss);
        ss = row_sum<M::LPR>(ss);
        const float rstd = rsqrtf(ss / D + a.eps);
        float o[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) o[i] = xv[i] * rstd * (seg == 0 ? gq[i] : gk[i]);
        if (t < a.T) {
          st16(y + out0 + static_cast<long long>(t) * D, pack16(o));
          if (c0 == 0) rs[static_cast<long long>(bh) * a.T + t] = rstd;
        }
      }
    } else {
      uint4 vr[kProSlots], er[kProSlots];
      float sc[kProSlots], lg[kProSlots];
      // Learned gate 2 sigmoid(<w_h, x[b, t, :C]>) of each row (all lanes
      // of the row take part in the dot product).
      if (GATE) {
        const int cl = lane % M::LPR;
#pragma unroll
        for (int u = 0; u < kProSlots; ++u) {
          const int t = tg + u * M::RPI;
          float z = 0.f;
          if (t < a.T) {
            const elem_t* xrow = a.gx + (static_cast<long long>(b) * a.T + t) * a.gx_stride;
            for (int c = cl; c < a.gch; c += M::LPR) z = fmaf(a.gw[h * a.gch + c], to_f32(xrow[c]), z);
          }
          z = row_sum<M::LPR>(z);
          lg[u] = 2.0f / (1.0f + expf(-z));
          if (t < a.T && cl == 0) a.gate_out[(static_cast<long long>(b) * a.T + t) * a.Hkv + h] = lg[u];
        }
      }
#pragma unroll
      for (int u = 0; u < kProSlots; ++u) {
        const int t = tg + u * M::RPI;
        er[u] = make_uint4(0u, 0u, 0u, 0u);
        sc[u] = 0.f;
        if (t >= a.T) continue;
        const long long bt = static_cast<long long>(b) * a.T + t;
        vr[u] = ld16(a.v + in0 + t * in_stride);
        if (a.ve == nullptr) continue;   // plain layer (fp32 build only): v_eff is a copy of v
        const int tok = a.tok[bt];
        if (tok >= 0 && tok < a.vocab) {
          er[u] = ld16(a.ve + static_cast<long long>(tok) * Hd + h * D + c0);
          sc[u] = a.ve_scale * (GATE ? lg[u] : (a.gate ? a.gate[bt * a.Hkv + h] : 1.0f));
        } else if (c0 == 0) {
          // An id outside the table contributes nothing and is reported.
          atomicOr(a.status, DEV_ERR_TOKEN);
        }
      }
#pragma unroll
      for (int u = 0; u < kProSlots; ++u) {
        const int t = tg + u * M::RPI;
        if (t >= a.T) continue;
        float vv[EPL], ev[EPL], o[EPL];
        unpack16(vr[u], vv);
        unpack16(er[u], ev);
#pragma unroll
        for (int i = 0; i < EPL; ++i) o[i] = fmaf(sc[u], ev[i], vv[i]);
        st16(a.veff + out0 + static_cast<long long>(t) * D, pack16(o));
      }
    }
  }
}

// D[b, h, t] = sum_c dO[b, t, h, c] * O[b, t, h, c] (the softmax-backward row
// term), LSE2[b, h, t] = LSE[b, h, t] * log2(e) (both in rows padded to Tpad;
// the d_mul / lse2_mul / lse2_add forms), and (unless the forward left it
// zeroed) zero the fp32 dQ accumulator row [b, h, t, :].
template <int D>
__global__ void __launch_bounds__(kRowWarps * 32, kPreBlocksPerSm) bwd_pre_kernel(PreArgs a) {
  using M = RowMap<D>;
  constexpr int EPL = M::EPL;
  const int lane = threadIdx.x & 31;
  const int slot = lane / M::LPR, c0 = (lane % M::LPR) * EPL;
  // the forward may already have zeroed exactly this accumulator (a record
  // that counts only while no wait has run out: a forward CTA that gave up
  // may not have zeroed its rows)
  const bool timed_out = a.status != nullptr && (*a.status & DEV_ERR_TIMEOUT) != 0u;
  const bool clear = a.clear_acc &&
                     !(a.acc_flag != nullptr && !timed_out && a.acc_flag[0] == a.acc_off &&
                       a.acc_flag[1] == a.acc_len);
  const int ngt = (a.T + M::RG - 1) / M::RG;
  const long long n_all = static_cast<long long>(a.B) * a.Hq * ngt;
  const long long in_stride = static_cast<long long>(a.Hq) * D;
  for (long long gi = grid_warp(); gi < n_all; gi += grid_warps()) {
    const int bh = static_cast<int>(gi / ngt);
    const int tg = static_cast<int>(gi - static_cast<long long>(bh) * ngt) * M::RG + slot;
    const int b = bh / a.Hq, h = bh - b * a.Hq;
    const long long in0 = (static_cast<long long>(b) * a.T * a.Hq + h) * D + c0;
    uint4 orw[kRowSlots], grw[kRowSlots];
    float lv[kRowSlots];   // the rows' LSE (read by the lanes that write D), with the rows
#pragma unroll
    for (int u = 0; u < kRowSlots; ++u) {
      const int t = tg + u * M::RPI;
      orw[u] = grw[u] = make_uint4(0u, 0u, 0u, 0u);
      lv[u] = 0.f;
      if (t < a.T) {
        orw[u] = ld16(a.o + in0 + t * in_stride);
        grw[u] = ld16(a.dO + in0 + t * in_stride);
        if (c0 == 0) lv[u] = a.lse[static_cast<long long>(bh) * a.T + t];
      }
    }
#pragma unroll
    for (int u = 0; u < kRowSlots; ++u) {
      const int t = tg + u * M::RPI;
      float ov[EPL], gv[EPL];
      unpack16(orw[u], ov);
      unpack16(grw[u], gv);
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) s = fmaf(ov[i], gv[i], s);
      s = row_sum<M::LPR>(s);
      if (t >= a.T) continue;
      const long long prow = static_cast<long long>(bh) * a.Tpad + t;
      if (c0 == 0) {
        a.dvec[prow] = s * a.d_mul;
        a.lse2[prow] = fmaf(lv[u], a.lse2_mul, a.lse2_add);
      }
      if (clear) {
        float z[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) z[i] = 0.f;
        stf<EPL>(a.dq_acc + (static_cast<long long>(bh) * a.T + t) * D + c0, z);
      }
    }
  }
}

// Backward of the prologue. Grid (nblk, segments); blockIdx.y: 0 = q rows
// (RMSNorm backward of q from the gradient of qn, dgq partials), 1 = k rows
// (same for k), 2 = v rows (dv = gradient of v_eff; scatter
// ve_scale * gate * dv_eff into dVE). RMSNorm backward, with r = rstd,
// xh = x r, y = g xh:
//   dxh = g dy;  dx = r (dxh - xh mean(dxh xh));  dg += dy xh.
// The gain partial of block x of segment s goes to gpart[s][x][:].
template <int D>
__global__ void __launch_bounds__(kRowWarps * 32, kPostBlocksPerSm) bwd_post_kernel(PostArgs a) {
  using M = RowMap<D>;
  constexpr int EPL = M::EPL;
  const int seg = blockIdx.y;
  const int H = seg == 0 ? a.Hq : a.Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int slot = lane / M::LPR, c0 = (lane % M::LPR) * EPL;
  const int ngt = (a.T + M::RG - 1) / M::RG;
  const long long n_all = static_cast<long long>(a.B) * H * ngt;
  const long long in_stride = static_cast<long long>(H) * D;
  const int Hd = a.Hkv * D;
  if (seg < 2) {
    const elem_t* x = seg == 0 ? a.q : a.k;
    const float* gain = seg == 0 ? a.gq : a.gk;
    const float* rs = seg == 0 ? a.rstd_q : a.rstd_k;
    const float* acc = seg == 0 ? a.dq_acc : a.dk_acc;
    elem_t* dx = seg == 0 ? a.dq : a.dk;
    float g[EPL], gacc[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      g[i] = gain ? gain[c0 + i] : 1.0f;
      gacc[i] = 0.f;
    }
    for (long long gi = grid_warp(); gi < n_all; gi += grid_warps()) {
      const int bh = static_cast<int>(gi / ngt);
      const int tg = static_cast<int>(gi - static_cast<long long>(bh) * ngt) * M::RG + slot;
      const int b = bh / H, h = bh - b * H;
      const long long in0 = (static_cast<long long>(b) * a.T * H + h) * D + c0;
      const long long acc0 = static_cast<long long>(bh) * a.T * D + c0;
      uint4 xr[kRowSlots];
      float dy[kRowSlots][EPL], rr[kRowSlots];
#pragma unroll
      for (int u = 0; u < kRowSlots; ++u) {
        const int t = tg + u * M::RPI;
        rr[u] = 0.f;
        if (t < a.T) {
          xr[u] = ld16(x + in0 + t * in_stride);
          ldf<EPL>(acc + acc0 + static_cast<long long>(t) * D, dy[u]);
          rr[u] = rs[static_cast<long long>(bh) * a.T + t];
        } else {
          xr[u] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int i = 0; i < EPL; ++i) dy[u][i] = 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < kRowSlots; ++u) {
        const int t = tg + u * M::RPI;
        float xh[EPL], dxh[EPL], dot = 0.f;
        unpack16(xr[u], xh);
        if (a.rcos != nullptr) rotate_row<D>(xh, a.rcos, a.rsin, t, t < a.T, 1.f);
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          xh[i] *= rr[u];
          dxh[i] = g[i] * dy[u][i];
          dot = fmaf(dxh[i], xh[i], dot);
          gacc[i] = fmaf(dy[u][i], xh[i], gacc[i]);
        }
        dot = row_sum<M::LPR>(dot) / D;
        float o[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) o[i] = rr[u] * (dxh[i] - xh[i] * dot);
        // the gradient of the rotated row, turned back by the transpose
        if (a.rcos != nullptr) rotate_row<D>(o, a.rcos, a.rsin, t, t < a.T, -1.f);
        if (t >= a.T) continue;
        st16(dx + in0 + t * in_stride, pack16(o));
      }
    }
    // Block reduction of the gain partials, in a fixed order: the row slots
    // of a warp (lanes c, c + LPR, ...), then the warps.
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
#pragma unroll
      for (int o = M::LPR; o < 32; o <<= 1) gacc[i] += __shfl_xor_sync(0xffffffffu, gacc[i], o);
    }
    __shared__ float red[kRowWarps][D];
    if (slot == 0) {
#pragma unroll
      for (int i = 0; i < EPL; ++i) red[warp][c0 + i] = gacc[i];
    }
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kRowWarps; ++w) s += red[w][c];
      a.gpart[(static_cast<long long>(seg) * a.nblk_max + blockIdx.x) * D + c] = s;
    }
  } else {
    for (long long gi = grid_warp(); gi < n_all; gi += grid_warps()) {
      const int bh = static_cast<int>(gi / ngt);
      const int tg = static_cast<int>(gi - static_cast<long long>(bh) * ngt) * M::RG + slot;
      const int b = bh / H, h = bh - b * H;
      const long long in0 = (static_cast<long long>(b) * a.T * H + h) * D + c0;
      const long long acc0 = static_cast<long long>(bh) * a.T * D + c0;
#pragma unroll
      for (int u = 0; u < kRowSlots; ++u) {
        const int t = tg + u * M::RPI;
        if (t >= a.T) continue;
        float dv[EPL];
        ldf<EPL>(a.dv_acc + acc0 + static_cast<long long>(t) * D, dv);
        st16(a.dv + in0 + t * in_stride, pack16(dv));
        if (a.dve) {
          const long long bt = static_cast<long long>(b) * a.T + t;
          const int tok = a.tok[bt];
          if (tok >= 0 && tok < a.vocab) {
            const float s = a.ve_scale * (a.gate ? a.gate[bt * a.Hkv + h] : 1.0f);
            float* dst = a.dve + static_cast<long long>(tok) * Hd + h * D + c0;
#pragma unroll
            for (int i = 0; i < EPL; ++i) atomicAdd(dst + i, s * dv[i]);
          }
        }
      }
    }
  }
}

// Backward of the learned value-embedding gate (autoresearch Administrator
// & Developer Guide §8.2.1, gate snippet, differentiated), one warp per
// position (b, t), persistent: for each kv head h
//   dgate_h = ve_scale <dv[b, t, h], VE[tok, h]>      (0 for a token outside the table)
//   dz_h    = dgate_h * gate_h (1 - gate_h / 2)       (d(2 sigmoid)/dz = 2 s (1 - s))
// then d_gx[b, t, c] = sum_h dz_h w[h, c] (lane c) and the block's partial
// of dW[h, c] = sum over its positions of dz_h x[b, t, c], reduced over the
// warps in a fixed order into gpart_w[block][h * gch + c] (rows of 1024).
template <int D>
__global__ void __launch_bounds__(kRowWarps * 32) ve_gate_bwd_kernel(GateBwdArgs a) {
  constexpr int CPL = D / 32;   // channels of d per lane
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long n_tok = static_cast<long long>(a.B) * a.T;
  const int Hd = a.Hkv * D;
  float wacc[32];
#pragma unroll
  for (int h = 0; h < 32; ++h) wacc[h] = 0.f;
  for (long long bt = grid_warp(); bt < n_tok; bt += grid_warps()) {
    const int tk = a.tok[bt];
    const bool in_table = tk >= 0 && tk < a.vocab;
    const float xc = lane < a.gch ? to_f32(a.gx[bt * a.gx_stride + lane]) : 0.f;
    float dgx = 0.f;
#pragma unroll
    for (int h = 0; h < 32; ++h) {
      if (h >= a.Hkv) break;
      float dot = 0.f;
      if (in_table) {
        float dvv[CPL], vev[CPL];
        load_vec<CPL>(a.dv + (bt * a.Hkv + h) * D + lane * CPL, dvv);
        load_vec<CPL>(a.ve + static_cast<long long>(tk) * Hd + h * D + lane * CPL, vev);
#pragma unroll
        for (int e = 0; e < CPL; ++e) dot = fmaf(dvv[e], vev[e], dot);
      }
      dot = warp_sum(dot);
      const float g = a.gate[bt * a.Hkv + h];
      const float dz = a.ve_scale * dot * g * (1.f - 0.5f * g);
      wacc[h] = fmaf(dz, xc, wacc[h]);
      if (lane < a.gch) dgx = fmaf(dz, a.gw[h * a.gch + lane], dgx);
    }
    if (a.d_gx != nullptr && lane < a.gch) a.d_gx[bt * a.gch + lane] = dgx;
  }
  __shared__ float red[kRowWarps][32];
#pragma unroll
  for (int h = 0; h < 32; ++h) {
    if (h >= a.Hkv) break;   // uniform over the block
    red[warp][lane] = wacc[h];
    __syncthreads();
    if (warp == 0 && lane < a.gch) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kRowWarps; ++w) s += red[w][lane];
      a.gpart_w[static_cast<long long>(blockIdx.x) * 1024 + h * a.gch + lane] = s;
    }
    __syncthreads();
  }
}

// Blocks of a persistent row-wise launch: `per_sm` per SM, no more than
// there are row groups (nor than `cap`).
inline int row_grid(long long groups, int per_sm, int cap) {
  long long n = static_cast<long long>(num_sms()) * per_sm;
  const long long per = (groups + kRowWarps - 1) / kRowWarps;
  if (per < n) n = per;
  if (cap > 0 && cap < n) n = cap;
  return n < 1 ? 1 : static_cast<int>(n);
}

// dgq[c] = sum of the q partials, dgk[c] = sum of the k partials (written by
// the backward-post kernel, or by the attention backward's epilogue), in a
// fixed order. Grid (2, d / 32), 1024 threads: column = 32 * blockIdx.y +
// lane; warp w sums partials w, w + 32, w + 64, ... in that order (eight
// loads in flight), then warp 0 adds the 32 warp sums in order.
constexpr int kGainWarps = 32;
__global__ void __launch_bounds__(kGainWarps * 32) gain_sum_kernel(GainArgs a) {
  float* out = blockIdx.x == 0 ? a.dgq : a.dgk;
  if (out == nullptr) return;
  const int nblk = blockIdx.x == 0 ? a.n_q : a.n_k;
  const float* part = blockIdx.x == 0 ? a.part_q : a.part_k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.y * 32 + lane;
  float s = 0.f;
  int blk = warp;
  for (; blk + 7 * kGainWarps < nblk; blk += 8 * kGainWarps) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = part[static_cast<long long>(blk + u * kGainWarps) * a.d + c];
#pragma unroll
    for (int u = 0; u < 8; ++u) s += v[u];
  }
  for (; blk < nblk; blk += kGainWarps) s += part[static_cast<long long>(blk) * a.d + c];
  __shared__ float red[kGainWarps][32];
  red[warp][lane] = s;
  __syncthreads();
  if (warp == 0) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kGainWarps; ++w) tot += red[w][lane];
    if (c < a.n_out) out[c] = tot;
  }
}

}  // namespace swa
