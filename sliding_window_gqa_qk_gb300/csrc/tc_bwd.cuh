// Backward attention core on the 5th-generation tensor cores (sm_103a).
//
// One CTA owns one 128-key tile of one (batch, kv head). It keeps its K and
// V tiles in shared memory and its dK and dV accumulators in TMEM, and loops
// over the G query heads of its GQA group and, for each, over the query tiles
// of the band (tiles outside the band are never visited). So dK and dV are
// reduced over the head group inside the CTA, without atomics. Per step, for
// a query tile of BQ rows:
//   S^T  = K Q^T          (TMEM)   P^T  = exp2(S^T c - LSE log2 e), masked on
//   dP^T = V dO^T         (TMEM)          partial tiles           (smem, bf16)
//   dS^T = P^T (dP^T - D)   (smem, bf16), D = rowsum(dO * O)
//   dV  += P^T dO,  dK += dS^T Q                                   (TMEM)
//   dQ   = dS K  (computed as dQ^T = K^T dS^T when d = 128)         (TMEM)
// dQ * scale is staged in shared memory and added into the fp32 dQ
// accumulator in global memory by TMA bulk reductions (the only cross-CTA
// exchange).
//
// Roles: warp 8 TMA producer (K, V once; Q, dO, LSE, D per step, 2 stages),
// warp 9 MMA issuer (one thread) and TMEM owner, warps 0-7 two warpgroups
// that split each step's columns in halves: thread t of warpgroup w owns key
// row t (TMEM lane t) and query columns [w BQ/2, (w+1) BQ/2) of S^T and dP^T,
// and half of the dQ tile in the drain.
//
// Softmax backward written out from the forward of the attention block
// (autoresearch Administrator & Developer Guide §8.2.1; train.py
// walkthrough post, model paragraph): dS = P * (dP - rowsum(dP * P)) with
// rowsum(dP * P) = rowsum(dO * O).
#pragma once

#include <cudaTypedefs.h>

#include "../../include/swa_attn.h"
#include "common.cuh"
#include "tc_fwd.cuh"

namespace swa {
namespace tc {

constexpr int kBK = 128;          // keys per CTA
constexpr int kBwdWarps = 10;
constexpr int kBwdThreads = kBwdWarps * 32;
constexpr int kBwdProducerWarp = 8;
constexpr int kBwdMmaWarp = 9;

struct BwdLaunch {
  int B, T, Hq, Hkv, d, window, causal;
  float scale;
  const elem_t* qn;    // [B, Hq, T, d]
  const elem_t* kn;    // [B, Hkv, T, d]
  const elem_t* v;     // [B, Hkv, T, d] (v_head_major) or [B, T, Hkv, d]
  bool v_head_major;
  const elem_t* dO;    // [B, T, Hq, d]
  const float* lse2;   // [B, Hq, Tpad]  LSE * log2(e)
  const float* dvec;   // [B, Hq, Tpad]  D
  int Tpad;
  float* dq_acc;       // [B, Hq, T, d]
  // key-side outputs, written by the epilogue of the kernel
  const elem_t* k;     // raw k [B, T, Hkv, d]
  const float* rstd_k; // [B, Hkv, T]
  const float* gk;     // [d] or NULL
  const int32_t* tok;  // [B, T] (VE layers)
  const float* gate;   // [B, T, Hkv] or NULL
  float* dve;          // [vocab, Hkv * d] or NULL
  float ve_scale;
  int vocab;
  elem_t* dk;          // [B, T, Hkv, d]
  elem_t* dv;          // [B, T, Hkv, d]
  float* gpart_k;      // [B * Hkv * n_ktiles, d]
  uint32_t* status;
  uint64_t wait_limit_ns;
  unsigned long long* acc_flag;   // dQ-accumulator record in the workspace header
  float* dkn_out;      // rotary: fp32 dkn [B, Hkv, T, d] for the post kernel (NULL: none)
};

struct BwdParams {
  int T, Tpad, Hq, Hkv, window, causal, n_ktiles;
  float scale, scale_log2;
  float dk_mul, dv_mul;   // factors applied to the dK and dV accumulators
  float* dq_acc;          // fp32 [B, Hq, T, d] (kernels that add into it directly)
  const float* lse2;
  const float* dvec;
  const elem_t* k;
  const float* rstd_k;
  const float* gk;
  const int32_t* tok;
  const float* gate;
  float* dve;
  float ve_scale;
  int vocab;
  elem_t* dk;
  elem_t* dv;
  float* gpart_k;
  uint32_t* status;
  uint64_t wait_limit_ns;
  // Rotary (non-null): the epilogue writes dkn = dK (fp32, [B, Hkv, T, d])
  // here and leaves the RMSNorm and rotary backward of k, with its gain
  // partials, to the post kernel (they need whole rotated rows).
  float* dkn_out;
  int n_bhk;                  // B * Hkv
  int chunk;                  // (batch, kv head) pairs per scheduling chunk (1-D grids)
  // Record of a forward that zeroed the dQ accumulator (offset, length);
  // the kernels that add into the accumulator mark it used (length 0).
  unsigned long long* acc_flag;
};

// Sum over the 32 lanes of each of 32 values: afterwards lane L holds the
// sum of column L (a butterfly that halves the kept columns at each step).
__device__ __forceinline__ float transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

// Key-side epilogue of a backward CTA, fused so that dK and dV never leave
// the chip in fp32. Thread t of warpgroup wg owns key row j = k0 + t and the
// head-dim columns [wg D/2, (wg+1) D/2) of dK (scaled here) and dV in TMEM.
//   dk  = RMSNorm backward of k: r (g dkn - xh mean(g dkn xh)),  xh = k r
//   dgk partial of this key tile = sum over its rows of dkn xh
//   dv  = dV (the gradient of v_eff);  dVE[tok] += ve_scale gate dV
// (the RMSNorm and VE-mix backward of the autoresearch Administrator &
// Developer Guide §8.2.1 blocks, differentiated). `have` is false when the
// CTA visited no query tile (dK = dV = 0). The two warpgroups exchange their
// half-row dot products through `sdot` and named barrier 3; `sgain` holds the
// per-warp column sums. The raw k rows come from global memory, or (sk != 0)
// from the key tile in shared memory as the TMA loaded it (128-byte swizzled
// 64-column regions of kBK rows). dv goes out first (staged in sdv, TMA
// store), so that the store reads it while dk is computed, then dk (sdk).
// `have` says that dV is final (the caller may call this before the last
// products of dK have completed); dk_ready() is called once dv is out and
// returns whether dK is final too (waiting for it, and for the raw k rows).
// Every thread of both warpgroups must call this.
template <int D, class DkReady>
__device__ __forceinline__ void kv_epilogue(const BwdParams& prm, uint32_t tDK, uint32_t tDV,
                                            bool have, int wg, int t, int b, int hk, int kt,
                                            float* sdot, float* sgain, uint32_t sdk, uint32_t sdv,
                                            const CUtensorMap* tmDK, const CUtensorMap* tmDV,
                                            uint32_t sk, DkReady&& dk_ready) {
  constexpr int HD = D / 2, NCH = HD / 32;
  float* sg = sdot + 256;                    // gains of this warpgroup's columns
  sgain += HD * 2;                           // per-warp column sums follow the gains
  const int lane = t & 31, warp4 = t >> 5;
  const int j = kt * kBK + t;
  const bool valid = j < prm.T;
  const long long bt = static_cast<long long>(b) * prm.T + j;
  const long long rowoff = (bt * prm.Hkv + hk) * D + wg * HD;   // into k / dk / dv
  const float r = valid ? prm.rstd_k[(static_cast<long long>(b) * prm.Hkv + hk) * prm.T + j] : 0.f;
  const bool rope = prm.dkn_out != nullptr;
  // dv and the VE-table gradient
  const int tok = (prm.dve != nullptr && valid) ? prm.tok[bt] : -1;
  const bool ve_ok = tok >= 0 && tok < prm.vocab;
  const float vs =
      ve_ok ? prm.dv_mul * prm.ve_scale * (prm.gate ? prm.gate[bt * prm.Hkv + hk] : 1.f) : 0.f;
  const float dvm = prm.dv_mul;
  uint32_t dvr[NCH][32];
  if (have) {
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) tmem_ld32(tDV + ch * 32, dvr[ch]);
    tmem_wait_ld(dvr[0]);
#pragma unroll
    for (int ch = 1; ch < NCH; ++ch) reg_fence(dvr[ch]);
  } else {
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
      for (int e = 0; e < 32; ++e) dvr[ch][e] = 0u;
  }
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    const uint32_t* a = dvr[ch];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = make_uint4(pack_bf16x2(__uint_as_float(a[8 * q]) * dvm, __uint_as_float(a[8 * q + 1]) * dvm),
                                 pack_bf16x2(__uint_as_float(a[8 * q + 2]) * dvm, __uint_as_float(a[8 * q + 3]) * dvm),
                                 pack_bf16x2(__uint_as_float(a[8 * q + 4]) * dvm, __uint_as_float(a[8 * q + 5]) * dvm),
                                 pack_bf16x2(__uint_as_float(a[8 * q + 6]) * dvm, __uint_as_float(a[8 * q + 7]) * dvm));
      st_shared_v4(sw128_addr(sdv, kBK, t, (wg * HD + ch * 32) / 8 + q), w.x, w.y, w.z, w.w);
    }
    if (ve_ok) {
      float* dst = prm.dve + static_cast<long long>(tok) * prm.Hkv * D + hk * D + wg * HD + ch * 32;
#pragma unroll
      for (int e = 0; e < 32; e += 4)
        red_add_v4_f32(dst + e, vs * __uint_as_float(a[e]), vs * __uint_as_float(a[e + 1]),
                       vs * __uint_as_float(a[e + 2]), vs * __uint_as_float(a[e + 3]));
    }
  }
  // dv out while dk is computed
  fence_async_smem();
  named_bar_sync(3, 256);
  if (wg == 0 && t == 0) {
    // rows past T fall outside the tensor and are not written
    for (int c = 0; c < D / 64; ++c) tma_store_4d(tmDV, sdv + c * kBK * 128, 64 * c, kt * kBK, hk, b);
    bulk_commit_group();
  }
  const bool have_dk = dk_ready() && have;
  if (rope) {
    // dkn rows (fp32) for the post kernel, this warpgroup's half of the row
    uint32_t dkr[NCH][32];
    if (have_dk) {
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) tmem_ld32(tDK + ch * 32, dkr[ch]);
      tmem_wait_ld(dkr[0]);
#pragma unroll
      for (int ch = 1; ch < NCH; ++ch) reg_fence(dkr[ch]);
    } else {
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
        for (int e = 0; e < 32; ++e) dkr[ch][e] = 0u;
    }
    if (valid) {
      float4* dst = reinterpret_cast<float4*>(
          prm.dkn_out + ((static_cast<long long>(b) * prm.Hkv + hk) * prm.T + j) * D + wg * HD);
      const float m = prm.dk_mul;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          dst[(ch * 32 + e) / 4] =
              make_float4(__uint_as_float(dkr[ch][e]) * m, __uint_as_float(dkr[ch][e + 1]) * m,
                          __uint_as_float(dkr[ch][e + 2]) * m, __uint_as_float(dkr[ch][e + 3]) * m);
    }
  }
  if (!rope) {
    // (the scratch may share memory with operands of the products that
    // dk_ready() waited for)
    if (t < HD) sg[wg * HD + t] = prm.gk ? prm.gk[wg * HD + t] : 1.f;
    // All loads first: dK (TMEM) and the k row (global).
    uint32_t dkr[NCH][32];
    if (have_dk) {
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) tmem_ld32(tDK + ch * 32, dkr[ch]);
    }
    uint4 xr[NCH * 4];
    if (valid && sk != 0) {
#pragma unroll
      for (int q = 0; q < NCH * 4; ++q) xr[q] = ld_shared_v4u(sw128_addr(sk, kBK, t, wg * (HD / 8) + q));
    } else if (valid) {
      const uint4* src = reinterpret_cast<const uint4*>(prm.k + rowoff);
#pragma unroll
      for (int q = 0; q < NCH * 4; ++q) xr[q] = src[q];
    } else {
#pragma unroll
      for (int q = 0; q < NCH * 4; ++q) xr[q] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (have_dk) {
      tmem_wait_ld(dkr[0]);
#pragma unroll
      for (int ch = 1; ch < NCH; ++ch) reg_fence(dkr[ch]);
    } else {
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
        for (int e = 0; e < 32; ++e) dkr[ch][e] = 0u;
    }
    named_bar_sync(3, 256);                    // gains staged
    auto xval = [&](int c) {                   // c in [0, HD)
      const uint4 u = xr[c >> 3];
      const uint32_t w = ((c & 7) >> 1) == 0 ? u.x : ((c & 7) >> 1) == 1 ? u.y : ((c & 7) >> 1) == 2 ? u.z : u.w;
      return (c & 1) ? __uint_as_float(w & 0xFFFF0000u) : __uint_as_float(w << 16);
    };
    float pdot = 0.f;
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int c = ch * 32 + e;
        pdot = fmaf(sg[wg * HD + c] * __uint_as_float(dkr[ch][e]), xval(c), pdot);
      }
    pdot *= prm.dk_mul * r;
    sdot[wg * 128 + t] = pdot;
    named_bar_sync(3, 256);
    const float mean = (pdot + sdot[(1 - wg) * 128 + t]) / D;
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
      uint32_t pk[16];
      float gt[32];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        const int c = ch * 32 + e;
        const float dk0 = __uint_as_float(dkr[ch][e]) * prm.dk_mul;
        const float dk1 = __uint_as_float(dkr[ch][e + 1]) * prm.dk_mul;
        const float xh0 = xval(c) * r, xh1 = xval(c + 1) * r;
        pk[e / 2] = pack_bf16x2(r * (sg[wg * HD + c] * dk0 - xh0 * mean),
                                r * (sg[wg * HD + c + 1] * dk1 - xh1 * mean));
        gt[e] = dk0 * xh0;                     // gain term, 0 on rows past T (r = 0)
        gt[e + 1] = dk1 * xh1;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st_shared_v4(sw128_addr(sdk, kBK, t, (wg * HD + ch * 32) / 8 + q), pk[4 * q], pk[4 * q + 1],
                     pk[4 * q + 2], pk[4 * q + 3]);
      sgain[(wg * 4 + warp4) * HD + ch * 32 + lane] = transpose_sum32(gt, lane);
    }
  }
  fence_async_smem();
  named_bar_sync(3, 256);   // (also orders the column sums in sgain before their reads)
  if (wg == 0 && t == 0) {
    if (!rope) {
      for (int c = 0; c < D / 64; ++c) tma_store_4d(tmDK, sdk + c * kBK * 128, 64 * c, kt * kBK, hk, b);
      bulk_commit_group();
    }
    bulk_wait_group_read<0>();   // the tiles are read out of shared memory
  }
  if (!rope && t < HD) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) sum += sgain[(wg * 4 + w) * HD + t];
    prm.gpart_k[(static_cast<long long>(b * prm.Hkv + hk) * prm.n_ktiles + kt) * D + wg * HD + t] = sum;
  }
}

template <int D>
struct BwdCfg {
  static constexpr int BQ = D == 128 ? 64 : 128;   // query rows per step
  static constexpr int HC = BQ / 2;                // S^T columns per warpgroup
  static constexpr int kKV = kBK * D * 2;          // K or V tile bytes
  static constexpr int kQ = BQ * D * 2;            // Q or dO tile bytes
  static constexpr int kP = kBK * BQ * 2;          // P^T or dS^T bytes
  static constexpr int kStage = 16384;             // dQ staging per warpgroup and buffer
  static constexpr int kStageBufs = D == 128 ? 2 : 1;  // buffers (shared memory budget)
  static constexpr int oK = 0;
  static constexpr int oV = oK + kKV;
  static constexpr int oQ = oV + kKV;              // 2 stages
  static constexpr int oG = oQ + 2 * kQ;           // dO, 2 stages
  static constexpr int oP = oG + 2 * kQ;
  static constexpr int oS = oP + kP;
  static constexpr int oR = oS + kP;               // dQ staging [buffers][2 warpgroups]
  static constexpr int oL = oR + 2 * kStageBufs * kStage;  // LSE2, 2 stages of BQ floats
  static constexpr int oD = oL + 2 * BQ * 4;       // D, 2 stages
  static constexpr int kBytes = oD + 2 * BQ * 4;
  static constexpr int kAlloc = kBytes + 1024;
  // TMEM columns
  static constexpr uint32_t cS = 0, cDP = BQ, cDV = 2 * BQ, cDK = 2 * BQ + D, cDQ = 2 * BQ + 2 * D;
  static_assert(kAlloc + 256 <= 232448, "shared memory budget (dynamic + static)");
  static_assert(2 * BQ + 2 * D + 64 <= 512, "TMEM budget");
};

enum {
  BB_KV = 0,
  BB_QFULL = 1,    // +stage
  BB_QEMPTY = 3,   // +stage
  BB_SFULL = 5,
  BB_DPFULL = 6,
  BB_PREADY = 7,
  BB_DSREADY = 8,
  BB_DQFULL = 9,
  BB_DQFREE = 10,
  BB_FINAL = 11,
  BB_COUNT = 12
};

// Writes one 16-byte chunk of row r of a [rows][cols] bf16 K-major tile in
// the 128-byte swizzle layout (cols / 64 regions of rows * 128 bytes).
__device__ __forceinline__ void st_sw128_chunk(uint32_t tile, int rows, int r, int chunk,
                                               uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  const uint32_t region = static_cast<uint32_t>(chunk >> 3) * rows * 128;
  const uint32_t addr = tile + region + (r >> 3) * 1024 + (r & 7) * 128 +
                        static_cast<uint32_t>((chunk & 7) ^ (r & 7)) * 16;
  st_shared_v4(addr, a, b, c, d);
}

template <int D, bool kPolled>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                  const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmDK,
                  const __grid_constant__ CUtensorMap tmDV, const BwdParams prm) {
  using C = BwdCfg<D>;
  constexpr int BQ = C::BQ;
  constexpr int HC = C::HC;
  constexpr int KCH = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t bars[BB_COUNT];
  __shared__ uint32_t tmem_base_sh;
  __shared__ uint32_t abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bhk = blockIdx.x;                 // b * Hkv + hk
  const int b = bhk / prm.Hkv, hk = bhk % prm.Hkv;
  const int kt = blockIdx.y;                  // early key tiles (heaviest) first
  const int k0 = kt * kBK;
  const int G = prm.Hq / prm.Hkv;
  const Band band{prm.T, prm.window, prm.causal};
  int qlo = 0, qhi = -1;
  q_tile_range(band, k0, kBK, BQ, qlo, qhi);
  const int nq = qhi - qlo + 1;
  const int n_it = nq > 0 ? nq * G : 0;
  const WaitCtl<kPolled> ctl{&abort_flag, prm.status, prm.wait_limit_ns};
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (threadIdx.x == 0) {
    // the accumulator is about to receive this launch's additions
    if (blockIdx.x == 0 && blockIdx.y == 0 && prm.acc_flag != nullptr) prm.acc_flag[1] = 0ull;
    abort_flag = 0;
    mbar_init(bar(BB_KV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(BB_QFULL + s), 1);
      mbar_init(bar(BB_QEMPTY + s), 1);
    }
    mbar_init(bar(BB_SFULL), 1);
    mbar_init(bar(BB_DPFULL), 1);
    mbar_init(bar(BB_PREADY), 8);
    mbar_init(bar(BB_DSREADY), 8);
    mbar_init(bar(BB_DQFULL), 1);
    mbar_init(bar(BB_DQFREE), 8);
    mbar_init(bar(BB_FINAL), 1);
    fence_mbar_init();
  }
  if (warp == kBwdMmaWarp) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == kBwdProducerWarp) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && n_it > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmG);
      mbar_arrive_expect_tx(bar(BB_KV), 2 * C::kKV);
      for (int c = 0; c < KCH; ++c) {
        tma_load_4d(sbase + C::oK + c * kBK * 128, &tmK, bar(BB_KV), 64 * c, k0, hk, b);
        tma_load_4d(sbase + C::oV + c * kBK * 128, &tmV, bar(BB_KV), 64 * c, k0, hk, b);
      }
      int last[2] = {-1, -1};
      for (int it = 0; it < n_it; ++it) {
        const int st = it & 1;
        const int h = hk * G + it / nq;
        const int q0 = (qlo + it % nq) * BQ;
        if (it >= 2 && !mbar_wait(bar(BB_QEMPTY + st), ((it - 2) >> 1) & 1, ctl)) break;
        last[st] = it;
        mbar_arrive_expect_tx(bar(BB_QFULL + st), 2 * C::kQ + 2 * BQ * 4);
        for (int c = 0; c < KCH; ++c) {
          tma_load_4d(sbase + C::oQ + st * C::kQ + c * BQ * 128, &tmQ, bar(BB_QFULL + st), 64 * c,
                      q0, h, b);
          tma_load_4d(sbase + C::oG + st * C::kQ + c * BQ * 128, &tmG, bar(BB_QFULL + st), 64 * c,
                      q0, h, b);
        }
        const long long row = (static_cast<long long>(b) * prm.Hq + h) * prm.Tpad + q0;
        bulk_load(sbase + C::oL + st * BQ * 4, prm.lse2 + row, BQ * 4, bar(BB_QFULL + st));
        bulk_load(sbase + C::oD + st * BQ * 4, prm.dvec + row, BQ * 4, bar(BB_QFULL + st));
      }
      // Let every copy this thread started land before the CTA can exit.
      mbar_wait_drain(bar(BB_KV), 0, kDrainLimitNs);
      for (int s = 0; s < 2; ++s)
        if (last[s] >= 0) mbar_wait_drain(bar(BB_QFULL + s), (last[s] >> 1) & 1, kDrainLimitNs);
    }
  } else if (warp == kBwdMmaWarp) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && n_it > 0) {
      constexpr uint32_t idST = idesc_bf16_f32(kBK, BQ, 0, 0);   // S^T, dP^T
      constexpr uint32_t idKV = idesc_bf16_f32(kBK, D, 0, 1);    // dV, dK
      constexpr uint32_t idQ = idesc_bf16_f32(128, 64, 1, 1);    // dQ^T (D=128) or dQ (D=64)
      const uint32_t sK = sbase + C::oK, sV = sbase + C::oV;
      const uint32_t sP = sbase + C::oP, sS = sbase + C::oS;
      bool ok = mbar_wait(bar(BB_KV), 0, ctl);
      for (int it = 0; it < n_it && ok; ++it) {
        const int st = it & 1, ph = it & 1;
        const uint32_t sQ = sbase + C::oQ + st * C::kQ, sG = sbase + C::oG + st * C::kQ;
        if (!(ok = mbar_wait(bar(BB_QFULL + st), (it >> 1) & 1, ctl))) break;
        tc_fence_after();
        // S^T = K Q^T and dP^T = V dO^T (K = D)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offA = (kk >> 2) * (kBK * 128) + (kk & 3) * 32;
          const uint32_t offB = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
          umma_bf16_ss(tmem + C::cS, sdesc_sw128(sK + offA, 16, 1024),
                       sdesc_sw128(sQ + offB, 16, 1024), idST, kk > 0);
        }
        umma_commit(bar(BB_SFULL));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offA = (kk >> 2) * (kBK * 128) + (kk & 3) * 32;
          const uint32_t offB = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
          umma_bf16_ss(tmem + C::cDP, sdesc_sw128(sV + offA, 16, 1024),
                       sdesc_sw128(sG + offB, 16, 1024), idST, kk > 0);
        }
        umma_commit(bar(BB_DPFULL));
        // dV += P^T dO (K = BQ queries)
        if (!(ok = mbar_wait(bar(BB_PREADY), ph, ctl))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          umma_bf16_ss(tmem + C::cDV, sdesc_sw128(sP + (kk >> 2) * (kBK * 128) + (kk & 3) * 32, 16, 1024),
                       sdesc_sw128(sG + kk * 2048, BQ * 128, 1024), idKV, (it > 0 || kk > 0));
        }
        // dK += dS^T Q
        if (!(ok = mbar_wait(bar(BB_DSREADY), ph, ctl))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          umma_bf16_ss(tmem + C::cDK, sdesc_sw128(sS + (kk >> 2) * (kBK * 128) + (kk & 3) * 32, 16, 1024),
                       sdesc_sw128(sQ + kk * 2048, BQ * 128, 1024), idKV, (it > 0 || kk > 0));
        }
        // dQ (K = 128 keys); its TMEM columns must have been drained.
        if (it >= 1 && !(ok = mbar_wait(bar(BB_DQFREE), (it - 1) & 1, ctl))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint32_t aa = (D == 128 ? sK : sS) + kk * 2048;
          const uint32_t bb = (D == 128 ? sS : sK) + kk * 2048;
          umma_bf16_ss(tmem + C::cDQ, sdesc_sw128(aa, kBK * 128, 1024),
                       sdesc_sw128(bb, kBK * 128, 1024), idQ, kk > 0);
        }
        umma_commit(bar(BB_DQFULL));
        umma_commit(bar(BB_QEMPTY + st));
      }
      umma_commit(bar(BB_FINAL));
      mbar_wait_drain(bar(BB_FINAL), 0, kDrainLimitNs);
    }
  } else {
    // ------------- softmax-backward warpgroups (warps 0-3 and 4-7) -------------
    const int wg = warp >> 2;                        // 0 or 1: column half
    const int t = threadIdx.x & 127;                 // key row / TMEM lane
    const int j = k0 + t;                            // key position
    const int c0 = wg * HC;                          // first S^T column of this half
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c = prm.scale_log2;
    const uint32_t sP = sbase + C::oP, sS = sbase + C::oS;
    const bool leader = (t == 0);
    // Wait outcomes are made warp-uniform (mbar_wait_warp) and warpgroup-
    // uniform at the drain's named barrier, so that after a timeout every
    // thread of the warpgroup leaves the loop at the same point.
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int st = it & 1, ph = it & 1;
      const int h = hk * G + it / nq;
      const int q0 = (qlo + it % nq) * BQ;
      const bool full = tile_full(band, q0, BQ, k0, kBK);
      // visible query columns of this key row (partial tiles): [clo, chi]
      int clo = 0, chi = BQ - 1;
      if (!full) {
        if (j >= prm.T) {
          clo = 1; chi = 0;
        } else {
          if (prm.T - 1 - q0 < chi) chi = prm.T - 1 - q0;
          if (prm.causal) {
            if (j - q0 > clo) clo = j - q0;
            if (prm.window >= 0 && j + prm.window - q0 < chi) chi = j + prm.window - q0;
          } else if (prm.window >= 0) {
            if (j - prm.window - q0 > clo) clo = j - prm.window - q0;
            if (j + prm.window - q0 < chi) chi = j + prm.window - q0;
          }
        }
      }
      uint32_t sr[HC / 32][32];
      // LSE2 and D of 32 of this half's columns, from shared memory
      const uint32_t sL = sbase + C::oL + st * BQ * 4 + c0 * 4;
      const uint32_t sDv = sbase + C::oD + st * BQ * 4 + c0 * 4;
      auto load32 = [&](uint32_t base, int cc, float (&v)[32]) {
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 a = ld_shared_v4f(base + (cc * 32 + e) * 4);
          v[e] = a.x; v[e + 1] = a.y; v[e + 2] = a.z; v[e + 3] = a.w;
        }
      };
      ok = ok && mbar_wait_warp(bar(BB_QFULL + st), (it >> 1) & 1, ctl);
      ok = ok && mbar_wait_warp(bar(BB_SFULL), ph, ctl);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < HC / 32; ++cc)
          tmem_ld32(tmem + C::cS + lane_off + c0 + cc * 32, sr[cc]);
        tmem_wait_ld(sr[0]);
#pragma unroll
        for (int cc = 1; cc < HC / 32; ++cc) reg_fence(sr[cc]);
        // P^T = exp2(S^T c - LSE2), masked on partial tiles
#pragma unroll
        for (int cc = 0; cc < HC / 32; ++cc) {
          float lse2[32];
          load32(sL, cc, lse2);
          if (full) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              sr[cc][e] = __float_as_uint(ex2_approx(fmaf(__uint_as_float(sr[cc][e]), c, -lse2[e])));
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int col = c0 + cc * 32 + e;
              const float p = ex2_approx(fmaf(__uint_as_float(sr[cc][e]), c, -lse2[e]));
              sr[cc][e] = __float_as_uint((col >= clo && col <= chi) ? p : 0.f);
            }
          }
        }
#pragma unroll
        for (int ch = 0; ch < HC / 8; ++ch) {
          const int cc = ch >> 2, e0 = (ch & 3) * 8;
          st_sw128_chunk(sP, kBK, t, c0 / 8 + ch,
                         pack_bf16x2(__uint_as_float(sr[cc][e0 + 0]), __uint_as_float(sr[cc][e0 + 1])),
                         pack_bf16x2(__uint_as_float(sr[cc][e0 + 2]), __uint_as_float(sr[cc][e0 + 3])),
                         pack_bf16x2(__uint_as_float(sr[cc][e0 + 4]), __uint_as_float(sr[cc][e0 + 5])),
                         pack_bf16x2(__uint_as_float(sr[cc][e0 + 6]), __uint_as_float(sr[cc][e0 + 7])));
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BB_PREADY));
      }
      // dS^T = P^T (dP^T - D)
      ok = ok && mbar_wait_warp(bar(BB_DPFULL), ph, ctl);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < HC / 32; ++cc) {
          uint32_t dp[32];
          float dd[32];
          tmem_ld32(tmem + C::cDP + lane_off + c0 + cc * 32, dp);
          load32(sDv, cc, dd);
          tmem_wait_ld(dp);
          if (full) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              sr[cc][e] = __float_as_uint(__uint_as_float(sr[cc][e]) *
                                          (__uint_as_float(dp[e]) - dd[e]));
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int col = c0 + cc * 32 + e;
              const float ds = __uint_as_float(sr[cc][e]) * (__uint_as_float(dp[e]) - dd[e]);
              sr[cc][e] = __float_as_uint((col >= clo && col <= chi) ? ds : 0.f);
            }
          }
        }
#pragma unroll
        for (int ch = 0; ch < HC / 8; ++ch) {
          const int cc = ch >> 2, e0 = (ch & 3) * 8;
          st_sw128_chunk(sS, kBK, t, c0 / 8 + ch,
                         pack_bf16x2(__uint_as_float(sr[cc][e0 + 0]), __uint_as_float(sr[cc][e0 + 1])),
                         pack_bf16x2(__uint_as_float(sr[cc][e0 + 2]), __uint_as_float(sr[cc][e0 + 3])),
                         pack_bf16x2(__uint_as_float(sr[cc][e0 + 4]), __uint_as_float(sr[cc][e0 + 5])),
                         pack_bf16x2(__uint_as_float(sr[cc][e0 + 6]), __uint_as_float(sr[cc][e0 + 7])));
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BB_DSREADY));
      }
      // dQ drain: TMEM -> registers -> (scaled) shared staging -> TMA add.
      // D=128: dQ^T, lane = head-dim index t, this half's 32 query columns.
      // D=64:  dQ,   lane = query row t,     this half's 32 head-dim columns.
      uint32_t dq[32];
      ok = ok && mbar_wait_warp(bar(BB_DQFULL), ph, ctl);
      if (ok) {
        tc_fence_after();
        tmem_ld32(tmem + C::cDQ + lane_off + wg * 32, dq);
        tmem_wait_ld(dq);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BB_DQFREE));
      }
      const uint32_t stage = sbase + C::oR + ((it % C::kStageBufs) * 2 + wg) * C::kStage;
      // the add issued from this buffer kStageBufs steps ago must have read it
      if (leader) bulk_wait_group_read<C::kStageBufs - 1>();
      ok = named_bar_and(1 + wg, 128, ok);
      if (!ok) break;
      if constexpr (D == 128) {
        // staging [32 queries][128 d] fp32, row-major
#pragma unroll
        for (int e = 0; e < 32; ++e)
          st_shared_f32(stage + e * 512 + t * 4, __uint_as_float(dq[e]) * prm.scale);
      } else {
        // staging [128 queries][32 d] fp32, 128-byte swizzle
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint32_t addr = stage + (t >> 3) * 1024 + (t & 7) * 128 +
                                static_cast<uint32_t>(ch ^ (t & 7)) * 16;
          asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                       "f"(__uint_as_float(dq[4 * ch]) * prm.scale),
                       "f"(__uint_as_float(dq[4 * ch + 1]) * prm.scale),
                       "f"(__uint_as_float(dq[4 * ch + 2]) * prm.scale),
                       "f"(__uint_as_float(dq[4 * ch + 3]) * prm.scale)
                       : "memory");
        }
      }
      fence_async_smem();
      named_bar_sync(1 + wg, 128);
      if (leader) {
        const int bh = b * prm.Hq + h;
        if constexpr (D == 128) tma_reduce_add_3d(&tmDQ, stage, 0, q0 + wg * 32, bh);
        else tma_reduce_add_3d(&tmDQ, stage, wg * 32, q0, bh);
        bulk_commit_group();
      }
    }
    if (leader) bulk_wait_group_all();
    // ---- epilogue: key-side gradients (scratch in the free Q stage buffer) ----
    tc_fence_after();
    float* scratch = reinterpret_cast<float*>(smem + C::oQ);
    const uint32_t sdk = sbase + C::oQ + 4096, sdv = sdk + kBK * D * 2;
    kv_epilogue<D>(prm, tmem + C::cDK + lane_off + wg * (D / 2), tmem + C::cDV + lane_off + wg * (D / 2),
                   ok && n_it > 0, wg, t, b, hk, kt, scratch, scratch + 256, sdk, sdv, &tmDK, &tmDV, 0u,
                   [] { return true; });
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kBwdMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// fp32 tensor map of the dQ accumulator [B*Hq][T][D] for the bulk adds:
// D = 128: boxes of 32 query rows x 128 columns, no swizzle;
// D = 64:  boxes of 128 query rows x 32 columns, 128-byte swizzle.
inline bool map_dq_acc(CUtensorMap* m, float* base, int BH, int T, int D) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4, static_cast<cuuint64_t>(T) * D * 4};
  cuuint32_t box[3] = {D == 128 ? 128u : 32u, D == 128 ? 32u : 128u, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            D == 128 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
inline swa_status launch_bwd_d(const BwdLaunch& f, cudaStream_t st) {
  using C = BwdCfg<D>;
  CUtensorMap mq, mk, mv, mg, mdq, mdk, mdv;
  if (!map_token_major(&mdk, f.dk, f.B, f.Hkv, f.T, D) || !map_token_major(&mdv, f.dv, f.B, f.Hkv, f.T, D))
    return SWA_ERR_CUDA;
  if (!make_map_4d(&mq, f.qn, D, f.T, f.Hq, f.B, D, static_cast<long long>(f.T) * D,
                   static_cast<long long>(f.Hq) * f.T * D, C::BQ) ||
      !make_map_4d(&mg, f.dO, D, f.T, f.Hq, f.B, static_cast<long long>(f.Hq) * D, D,
                   static_cast<long long>(f.T) * f.Hq * D, C::BQ) ||
      !map_head_major(&mk, f.kn, f.B, f.Hkv, f.T, D) ||
      !map_dq_acc(&mdq, f.dq_acc, f.B * f.Hq, f.T, D))
    return SWA_ERR_CUDA;
  const bool okv = f.v_head_major ? map_head_major(&mv, f.v, f.B, f.Hkv, f.T, D)
                                  : map_token_major(&mv, f.v, f.B, f.Hkv, f.T, D);
  if (!okv) return SWA_ERR_CUDA;
  BwdParams p{};
  p.T = f.T; p.Tpad = f.Tpad; p.Hq = f.Hq; p.Hkv = f.Hkv; p.window = f.window; p.causal = f.causal;
  p.n_ktiles = (f.T + kBK - 1) / kBK;
  p.scale = f.scale;
  p.scale_log2 = f.scale * 1.4426950408889634f;
  p.lse2 = f.lse2; p.dvec = f.dvec;
  p.dk_mul = f.scale; p.dv_mul = 1.f;
  p.k = f.k; p.rstd_k = f.rstd_k; p.gk = f.gk; p.tok = f.tok; p.gate = f.gate; p.dve = f.dve;
  p.ve_scale = f.ve_scale; p.vocab = f.vocab; p.dk = f.dk; p.dv = f.dv; p.gpart_k = f.gpart_k;
  p.status = f.status; p.wait_limit_ns = f.wait_limit_ns;
  p.acc_flag = f.acc_flag;
  p.dkn_out = f.dkn_out;
  dim3 grid(f.B * f.Hkv, p.n_ktiles);
  auto launch = [&](auto kern) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kAlloc) != cudaSuccess)
      return SWA_ERR_CUDA;
    kern<<<grid, kBwdThreads, C::kAlloc, st>>>(mq, mk, mv, mg, mdq, mdk, mdv, p);
    return cudaGetLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
  };
  return p.wait_limit_ns < kPollBelowNs ? launch(bwd_tc_kernel<D, true>) : launch(bwd_tc_kernel<D, false>);
}

// d = 64 (d = 128 has its own kernel, tc_bwd128.cuh).
inline swa_status launch_bwd(const BwdLaunch& f, cudaStream_t st) {
  return f.d == 64 ? launch_bwd_d<64>(f, st) : SWA_ERR_UNSUPPORTED;
}

}  // namespace tc
}  // namespace swa
