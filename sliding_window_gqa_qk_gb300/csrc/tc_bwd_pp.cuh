// Backward attention core for d = 128 with two ping-pong pipelines (sm_103a).
//
// Same work split as tc_bwd.cuh (one CTA per 128-key tile of a (batch, kv
// head), dK and dV accumulated in TMEM over the GQA group and the in-band
// 64-row query tiles), but consecutive query tiles alternate between two
// pipelines so that the tensor core computes one pipeline's matmuls while
// the other pipeline's warpgroup does its element-wise work:
//   pipeline X (warpgroup X, warps 4X..4X+3) owns steps i = X, X+2, ...:
//     S^T_X  = K Q_i^T,  dP^T_X = V dO_i^T                      (TMEM, 64 cols each)
//     P^T = exp2(S^T c - LSE2), dS^T = P^T (dP^T - D)          (smem, bf16)
//     dV += P^T dO_i,  dK += dS^T Q_i                           (TMEM, shared)
//     dQ_i^T = K^T dS^T into S^T_X's columns; drained to smem (the
//     pipeline's P/dS buffer, free by then) and added into the fp32 dQ
//     accumulator by one TMA bulk reduction.
//   warp 8 TMA producer (K, V once; Q, dO, LSE2, D per step, 3 stages),
//   warp 9 MMA issuer: A(0) A(1) | B(0) C(0) B(1) C(1) A(2) A(3) | ...
//     with A = S^T, dP^T; B = dV; C = dK, dQ.
// TMEM: S^T_0/dQ^T_0 [0,64), dP^T_0 [64,128), S^T_1/dQ^T_1 [128,192),
// dP^T_1 [192,256), dV [256,384), dK [384,512).
// Registers: the softmax warpgroups run with 216 per thread, warpgroup 2
// (producer, MMA, two idle warps) with 72 (setmaxnreg; 384 x 168 at launch).
//
// Softmax backward written out from the forward of the attention block
// (autoresearch Administrator & Developer Guide §8.2.1; train.py
// walkthrough post, model paragraph).
#pragma once

#include "tc_bwd.cuh"

namespace swa {
namespace tc {

constexpr int kPPThreads = 384;
constexpr int kPPRegsSoftmax = 216;
constexpr int kPPRegsOther = 72;
static_assert(2 * 128 * kPPRegsSoftmax + 128 * kPPRegsOther <= kPPThreads * 168,
              "register split exceeds the launch's registers");

struct PPCfg {
  static constexpr int D = 128;
  static constexpr int BQ = 64;
  static constexpr int NST = 3;                    // Q / dO / LSE2 / D stages
  static constexpr int kKV = kBK * D * 2;          // 32 KB
  static constexpr int kQ = BQ * D * 2;            // 16 KB
  static constexpr int kPS = 2 * kBK * BQ * 2;     // P^T + dS^T = 32 KB = dQ staging [64][128] fp32
  static constexpr int oK = 0;
  static constexpr int oV = oK + kKV;
  static constexpr int oQ = oV + kKV;              // NST stages
  static constexpr int oG = oQ + NST * kQ;         // NST stages
  static constexpr int oPS = oG + NST * kQ;        // 2 pipelines
  static constexpr int oL = oPS + 2 * kPS;         // NST stages of BQ floats
  static constexpr int oD = oL + NST * BQ * 4;
  static constexpr int kBytes = oD + NST * BQ * 4;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc + 256 <= 232448, "shared memory budget (dynamic + static)");
};

enum {
  QB_KV = 0,
  QB_QFULL = 1,     // +stage (3)
  QB_QEMPTY = 4,    // +stage (3)
  QB_SFULL = 7,     // +pipeline
  QB_DPFULL = 9,    // +pipeline
  QB_PREADY = 11,   // +pipeline
  QB_DSREADY = 13,  // +pipeline
  QB_DQFULL = 15,   // +pipeline
  QB_DQFREE = 17,   // +pipeline
  QB_FINAL = 19,
  QB_COUNT = 20
};

__global__ void __launch_bounds__(kPPThreads, 1)
    bwd_tc_pp_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                     const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmDK,
                     const __grid_constant__ CUtensorMap tmDV, const BwdParams prm) {
  using C = PPCfg;
  constexpr int D = C::D, BQ = C::BQ, NST = C::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t bars[QB_COUNT];
  __shared__ uint32_t tmem_base_sh;
  __shared__ uint32_t abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bhk = blockIdx.x;
  const int b = bhk / prm.Hkv, hk = bhk % prm.Hkv;
  const int k0 = static_cast<int>(blockIdx.y) * kBK;
  const int G = prm.Hq / prm.Hkv;
  const Band band{prm.T, prm.window, prm.causal};
  int qlo = 0, qhi = -1;
  q_tile_range(band, k0, kBK, BQ, qlo, qhi);
  const int nq = qhi - qlo + 1;
  const int n_it = nq > 0 ? nq * G : 0;
  const WaitCtl ctl{&abort_flag, prm.status, prm.wait_limit_ns};
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar(QB_KV), 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar(QB_QFULL + s), 1);
      mbar_init(bar(QB_QEMPTY + s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(QB_SFULL + x), 1);
      mbar_init(bar(QB_DPFULL + x), 1);
      mbar_init(bar(QB_PREADY + x), 4);
      mbar_init(bar(QB_DSREADY + x), 4);
      mbar_init(bar(QB_DQFULL + x), 1);
      mbar_init(bar(QB_DQFREE + x), 4);
    }
    mbar_init(bar(QB_FINAL), 1);
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  constexpr uint32_t cDV = 256, cDK = 384;
  bool final_ok = false;

  if (warp >= 8) {
    setmaxnreg_dec<kPPRegsOther>();
    if (warp == 8 && lane == 0 && n_it > 0) {
      // ---------------- TMA producer ----------------
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmG);
      mbar_arrive_expect_tx(bar(QB_KV), 2 * C::kKV);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_4d(sbase + C::oK + c * kBK * 128, &tmK, bar(QB_KV), 64 * c, k0, hk, b);
        tma_load_4d(sbase + C::oV + c * kBK * 128, &tmV, bar(QB_KV), 64 * c, k0, hk, b);
      }
      int last[NST] = {-1, -1, -1};
      for (int it = 0; it < n_it; ++it) {
        const int st = it % NST;
        const int h = hk * G + it / nq;
        const int q0 = (qlo + it % nq) * BQ;
        if (it >= NST && !mbar_wait(bar(QB_QEMPTY + st), ((it / NST) - 1) & 1, ctl)) break;
        last[st] = it;
        mbar_arrive_expect_tx(bar(QB_QFULL + st), 2 * C::kQ + 2 * BQ * 4);
        for (int c = 0; c < D / 64; ++c) {
          tma_load_4d(sbase + C::oQ + st * C::kQ + c * BQ * 128, &tmQ, bar(QB_QFULL + st), 64 * c,
                      q0, h, b);
          tma_load_4d(sbase + C::oG + st * C::kQ + c * BQ * 128, &tmG, bar(QB_QFULL + st), 64 * c,
                      q0, h, b);
        }
        const long long row = (static_cast<long long>(b) * prm.Hq + h) * prm.Tpad + q0;
        bulk_load(sbase + C::oL + st * BQ * 4, prm.lse2 + row, BQ * 4, bar(QB_QFULL + st));
        bulk_load(sbase + C::oD + st * BQ * 4, prm.dvec + row, BQ * 4, bar(QB_QFULL + st));
      }
      mbar_wait_drain(bar(QB_KV), 0, prm.wait_limit_ns);
      for (int s = 0; s < NST; ++s)
        if (last[s] >= 0) mbar_wait_drain(bar(QB_QFULL + s), (last[s] / NST) & 1, prm.wait_limit_ns);
    } else if (warp == 9 && lane == 0 && n_it > 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t idST = idesc_bf16_f32(kBK, BQ, 0, 0);   // S^T, dP^T: M=128 keys, N=64
      constexpr uint32_t idKV = idesc_bf16_f32(kBK, D, 0, 1);    // dV, dK: M=128 keys, N=128
      constexpr uint32_t idQ = idesc_bf16_f32(128, BQ, 1, 1);    // dQ^T: M=128 (d), N=64
      const uint32_t sK = sbase + C::oK, sV = sbase + C::oV;
      bool ok = mbar_wait(bar(QB_KV), 0, ctl);
      // Descriptor bases, computed once; every MMA adds an offset.
      const uint64_t dKk = sdesc_sw128(sK, 16, 1024), dVk = sdesc_sw128(sV, 16, 1024);
      const uint64_t dKmn = sdesc_sw128(sK, kBK * 128, 1024);
      const uint64_t dQk0 = sdesc_sw128(sbase + C::oQ, 16, 1024);
      const uint64_t dGk0 = sdesc_sw128(sbase + C::oG, 16, 1024);
      const uint64_t dQmn0 = sdesc_sw128(sbase + C::oQ, BQ * 128, 1024);
      const uint64_t dGmn0 = sdesc_sw128(sbase + C::oG, BQ * 128, 1024);
      const uint64_t dPk0 = sdesc_sw128(sbase + C::oPS, 16, 1024);
      const uint64_t dSmn0 = sdesc_sw128(sbase + C::oPS + kBK * BQ * 2, kBK * 128, 1024);
      auto opA = [&](int i) -> bool {   // S^T, dP^T of step i
        const int X = i & 1, st = i % NST;
        if (!mbar_wait(bar(QB_QFULL + st), (i / NST) & 1, ctl)) return false;
        if (i >= 2 && !mbar_wait(bar(QB_DQFREE + X), ((i - 2) >> 1) & 1, ctl)) return false;
        tc_fence_after();
        const uint64_t qd = sdesc_add(dQk0, st * C::kQ), gd = sdesc_add(dGk0, st * C::kQ);
        const uint32_t tS = tmem + X * 128;
        static_for<0, D / 16>([&](auto kc) {
          constexpr int kk = decltype(kc)::value;
          constexpr uint32_t offA = ((kk >> 2) * (kBK * 128) + (kk & 3) * 32) >> 4;
          constexpr uint32_t offB = ((kk >> 2) * (BQ * 128) + (kk & 3) * 32) >> 4;
          umma_ss_imm<idST, offA, offB>(tS, dKk, qd, kk > 0, 1u);
        });
        umma_commit(bar(QB_SFULL + X));
        static_for<0, D / 16>([&](auto kc) {
          constexpr int kk = decltype(kc)::value;
          constexpr uint32_t offA = ((kk >> 2) * (kBK * 128) + (kk & 3) * 32) >> 4;
          constexpr uint32_t offB = ((kk >> 2) * (BQ * 128) + (kk & 3) * 32) >> 4;
          umma_ss_imm<idST, offA, offB>(tS + 64, dVk, gd, kk > 0, 1u);
        });
        umma_commit(bar(QB_DPFULL + X));
        return true;
      };
      auto opB = [&](int i) -> bool {   // dV += P^T dO
        const int X = i & 1, st = i % NST;
        if (!mbar_wait(bar(QB_PREADY + X), (i >> 1) & 1, ctl)) return false;
        tc_fence_after();
        const uint64_t pd = sdesc_add(dPk0, X * C::kPS), gd = sdesc_add(dGmn0, st * C::kQ);
        static_for<0, BQ / 16>([&](auto kc) {
          constexpr int kk = decltype(kc)::value;
          umma_ss_imm<idKV, kk * 2, kk * 128>(tmem + cDV, pd, gd, (i > 0 || kk > 0), 1u);
        });
        return true;
      };
      auto opC = [&](int i) -> bool {   // dK += dS^T Q; dQ^T = K^T dS^T
        const int X = i & 1, st = i % NST;
        if (!mbar_wait(bar(QB_DSREADY + X), (i >> 1) & 1, ctl)) return false;
        tc_fence_after();
        const uint64_t sd = sdesc_add(dPk0, X * C::kPS + kBK * BQ * 2);
        const uint64_t qd = sdesc_add(dQmn0, st * C::kQ), smn = sdesc_add(dSmn0, X * C::kPS);
        static_for<0, BQ / 16>([&](auto kc) {
          constexpr int kk = decltype(kc)::value;
          umma_ss_imm<idKV, kk * 2, kk * 128>(tmem + cDK, sd, qd, (i > 0 || kk > 0), 1u);
        });
        static_for<0, kBK / 16>([&](auto kc) {
          constexpr int kk = decltype(kc)::value;
          umma_ss_imm<idQ, kk * 128, kk * 128>(tmem + X * 128, dKmn, smn, kk > 0, 1u);
        });
        umma_commit(bar(QB_DQFULL + X));
        umma_commit(bar(QB_QEMPTY + st));
        return true;
      };
      if (ok) ok = opA(0);
      if (ok && n_it > 1) ok = opA(1);
      for (int i = 0; i < n_it && ok; i += 2) {
        ok = opB(i) && opC(i);
        if (ok && i + 1 < n_it) ok = opB(i + 1) && opC(i + 1);
        if (ok && i + 2 < n_it) ok = opA(i + 2);
        if (ok && i + 3 < n_it) ok = opA(i + 3);
      }
      umma_commit(bar(QB_FINAL));
      mbar_wait_drain(bar(QB_FINAL), 0, prm.wait_limit_ns);
    }
  } else {
    // ------------- softmax-backward warpgroups: pipeline X = warp / 4 -------------
    setmaxnreg_inc<kPPRegsSoftmax>();
    const int X = warp >> 2;
    const int t = threadIdx.x & 127;                 // key row / TMEM lane (d index in the drain)
    const int j = k0 + t;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c = prm.scale_log2;
    const uint32_t sPS = sbase + C::oPS + X * C::kPS;     // P^T, then dS^T, then dQ staging
    const uint32_t sP = sPS, sS = sPS + kBK * BQ * 2;
    const uint32_t tS = tmem + X * 128 + lane_off, tDP = tS + 64;
    const bool leader = (t == 0);
    bool ok = true;
    for (int i = X; i < n_it; i += 2) {
      const int st = i % NST, ph = (i >> 1) & 1;
      const int h = hk * G + i / nq;
      const int q0 = (qlo + i % nq) * BQ;
      const bool full = tile_full(band, q0, BQ, k0, kBK);
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
      const uint32_t sL = sbase + C::oL + st * BQ * 4;
      const uint32_t sDv = sbase + C::oD + st * BQ * 4;
      uint32_t sr[2][32];
      ok = ok && mbar_wait_warp(bar(QB_QFULL + st), (i / NST) & 1, ctl);
      ok = ok && mbar_wait_warp(bar(QB_SFULL + X), ph, ctl);
      if (ok) {
        tc_fence_after();
        tmem_ld32(tS, sr[0]);
        tmem_ld32(tS + 32, sr[1]);
        tmem_wait_ld(sr[0]);
        reg_fence(sr[1]);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 lv = ld_shared_v4f(sL + (cc * 32 + e) * 4);
            const float l4[4] = {lv.x, lv.y, lv.z, lv.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float p = ex2_approx(fmaf(__uint_as_float(sr[cc][e + u]), c, -l4[u]));
              const int col = cc * 32 + e + u;
              sr[cc][e + u] = __float_as_uint((full || (col >= clo && col <= chi)) ? p : 0.f);
            }
          }
        }
      }
      // The previous step's dQ bulk add must have finished reading this buffer.
      if (leader) bulk_wait_group_read<0>();
      ok = named_bar_and(1 + X, 128, ok);
      if (!ok) break;
#pragma unroll
      for (int ch = 0; ch < BQ / 8; ++ch) {
        const int cc = ch >> 2, e0 = (ch & 3) * 8;
        st_sw128_chunk(sP, kBK, t, ch,
                       pack_bf16x2(__uint_as_float(sr[cc][e0 + 0]), __uint_as_float(sr[cc][e0 + 1])),
                       pack_bf16x2(__uint_as_float(sr[cc][e0 + 2]), __uint_as_float(sr[cc][e0 + 3])),
                       pack_bf16x2(__uint_as_float(sr[cc][e0 + 4]), __uint_as_float(sr[cc][e0 + 5])),
                       pack_bf16x2(__uint_as_float(sr[cc][e0 + 6]), __uint_as_float(sr[cc][e0 + 7])));
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(QB_PREADY + X));
      // dS^T = P^T (dP^T - D)
      ok = ok && mbar_wait_warp(bar(QB_DPFULL + X), ph, ctl);
      if (ok) {
        tc_fence_after();
        uint32_t dp[2][32];
        tmem_ld32(tDP, dp[0]);
        tmem_ld32(tDP + 32, dp[1]);
        tmem_wait_ld(dp[0]);
        reg_fence(dp[1]);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 dv = ld_shared_v4f(sDv + (cc * 32 + e) * 4);
            const float d4[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int col = cc * 32 + e + u;
              const float ds = __uint_as_float(sr[cc][e + u]) * (__uint_as_float(dp[cc][e + u]) - d4[u]);
              sr[cc][e + u] = __float_as_uint((full || (col >= clo && col <= chi)) ? ds : 0.f);
            }
          }
        }
#pragma unroll
        for (int ch = 0; ch < BQ / 8; ++ch) {
          const int cc = ch >> 2, e0 = (ch & 3) * 8;
          st_sw128_chunk(sS, kBK, t, ch,
                         pack_bf16x2(__uint_as_float(sr[cc][e0 + 0]), __uint_as_float(sr[cc][e0 + 1])),
                         pack_bf16x2(__uint_as_float(sr[cc][e0 + 2]), __uint_as_float(sr[cc][e0 + 3])),
                         pack_bf16x2(__uint_as_float(sr[cc][e0 + 4]), __uint_as_float(sr[cc][e0 + 5])),
                         pack_bf16x2(__uint_as_float(sr[cc][e0 + 6]), __uint_as_float(sr[cc][e0 + 7])));
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(QB_DSREADY + X));
      }
      // dQ drain: dQ^T (lane = head-dim index t, 64 query columns) -> staging
      // [64 queries][128 d] fp32 in this pipeline's P/dS buffer -> TMA add.
      ok = ok && mbar_wait_warp(bar(QB_DQFULL + X), ph, ctl);
      uint32_t dq[2][32];
      if (ok) {
        tc_fence_after();
        tmem_ld32(tS, dq[0]);
        tmem_ld32(tS + 32, dq[1]);
        tmem_wait_ld(dq[0]);
        reg_fence(dq[1]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(QB_DQFREE + X));
      }
      ok = named_bar_and(1 + X, 128, ok);
      if (!ok) break;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
#pragma unroll
        for (int e = 0; e < 32; ++e)
          st_shared_f32(sPS + (cc * 32 + e) * 512 + t * 4, __uint_as_float(dq[cc][e]) * prm.scale);
      fence_async_smem();
      named_bar_sync(1 + X, 128);
      if (leader) {
        tma_reduce_add_3d(&tmDQ, sPS, 0, q0, b * prm.Hq + h);
        bulk_commit_group();
      }
    }
    if (leader) bulk_wait_group_all();
    // ---- epilogue: key-side gradients (scratch in the free Q stage buffers) ----
    final_ok = ok && n_it > 0 && mbar_wait_warp(bar(QB_FINAL), 0, ctl);
    tc_fence_after();
    float* scratch = reinterpret_cast<float*>(smem + C::oQ);
    const uint32_t sdk = sbase + C::oQ + 4096, sdv = sdk + kBK * D * 2;
    kv_epilogue<D>(prm, tmem + cDK + lane_off + X * 64, tmem + cDV + lane_off + X * 64, final_ok, X,
                   t, b, hk, static_cast<int>(blockIdx.y), scratch, scratch + 256, sdk, sdv, &tmDK,
                   &tmDV);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// fp32 tensor map of the dQ accumulator [B*Hq][T][128] with boxes of 64 query
// rows x 128 columns (no swizzle) for the bulk adds of the ping-pong kernel.
inline bool map_dq_acc_64(CUtensorMap* m, float* base, int BH, int T) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {128 * 4, static_cast<cuuint64_t>(T) * 128 * 4};
  cuuint32_t box[3] = {128, 64, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline swa_status launch_bwd_pp(const BwdLaunch& f, cudaStream_t st) {
  using C = PPCfg;
  CUtensorMap mq, mk, mv, mg, mdq, mdk, mdv;
  if (!map_token_major(&mdk, f.dk, f.B, f.Hkv, f.T, 128) ||
      !map_token_major(&mdv, f.dv, f.B, f.Hkv, f.T, 128))
    return SWA_ERR_CUDA;
  if (!make_map_4d(&mq, f.qn, 128, f.T, f.Hq, f.B, 128, static_cast<long long>(f.T) * 128,
                   static_cast<long long>(f.Hq) * f.T * 128, C::BQ) ||
      !make_map_4d(&mg, f.dO, 128, f.T, f.Hq, f.B, static_cast<long long>(f.Hq) * 128, 128,
                   static_cast<long long>(f.T) * f.Hq * 128, C::BQ) ||
      !map_head_major(&mk, f.kn, f.B, f.Hkv, f.T, 128) ||
      !map_dq_acc_64(&mdq, f.dq_acc, f.B * f.Hq, f.T))
    return SWA_ERR_CUDA;
  const bool okv = f.v_head_major ? map_head_major(&mv, f.v, f.B, f.Hkv, f.T, 128)
                                  : map_token_major(&mv, f.v, f.B, f.Hkv, f.T, 128);
  if (!okv) return SWA_ERR_CUDA;
  BwdParams p{};
  p.T = f.T; p.Tpad = f.Tpad; p.Hq = f.Hq; p.Hkv = f.Hkv; p.window = f.window; p.causal = f.causal;
  p.n_ktiles = (f.T + kBK - 1) / kBK;
  p.scale = f.scale;
  p.scale_log2 = f.scale * 1.4426950408889634f;
  p.lse2 = f.lse2; p.dvec = f.dvec;
  p.k = f.k; p.rstd_k = f.rstd_k; p.gk = f.gk; p.tok = f.tok; p.gate = f.gate; p.dve = f.dve;
  p.ve_scale = f.ve_scale; p.vocab = f.vocab; p.dk = f.dk; p.dv = f.dv; p.gpart_k = f.gpart_k;
  p.status = f.status; p.wait_limit_ns = f.wait_limit_ns;
  if (cudaFuncSetAttribute(bwd_tc_pp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kAlloc) != cudaSuccess)
    return SWA_ERR_CUDA;
  dim3 grid(f.B * f.Hkv, p.n_ktiles);
  bwd_tc_pp_kernel<<<grid, kPPThreads, C::kAlloc, st>>>(mq, mk, mv, mg, mdq, mdk, mdv, p);
  return cudaGetLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

// Backward dispatch: the ping-pong kernel for d = 128, the split-column one
// for d = 64.
inline swa_status launch_bwd_any(const BwdLaunch& f, cudaStream_t st) {
  return f.d == 128 ? launch_bwd_pp(f, st) : launch_bwd(f, st);
}

}  // namespace tc
}  // namespace swa
