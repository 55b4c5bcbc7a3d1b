// Forward attention core, two query heads per CTA (sm_103a tcgen05).
//
// When a GQA group holds an even number of query heads, heads 2p and 2p + 1
// read the same kv head and have the same band, so one CTA computes the same
// 128-row query tile of both (tiles A and B) against one stream of K/V tiles:
//   warp 8      TMA producer: Q_A, Q_B once; K_j, V_j double-buffered;
//   warp 9      MMA issuer (one thread) and TMEM owner, issuing
//               ... PV_A(j-1), S_A(j), PV_B(j-1), S_B(j), PV_A(j), ...
//               so that while one softmax warpgroup works on its S, the
//               tensor core computes the other tile's PV and next S;
//   warps 0-3   softmax of tile A, warps 4-7 softmax of tile B: thread t
//               owns query row t (TMEM lane t), keeps the running max m and
//               sum l, rescales its O row only when m grows by more than 2^8,
//               and writes P = exp2(S c - m) as bf16 pairs back into the S
//               columns of TMEM, where the PV MMA reads it as its A operand.
// TMEM: S_A [0,128), S_B [128,256), O_A [256, 256+d), O_B [256+d, 256+2d).
// In-order execution of one CTA's MMAs makes S_X(j) overwrite P_X(j-1) only
// after PV_X(j-1) has read it; the commit that signals S_X(j) also covers
// PV_X(j-1), so O_X may be rescaled as soon as S_X(j) is visible.
//
// The method (QK-norm'd q and k from the prologue, grouped-query attention
// with kv head h / G, causal sliding-window or full causal band) follows the
// autoresearch train.py walkthrough post (model paragraph) and the
// autoresearch Administrator & Developer Guide §8.2.1 and §6.3.
#pragma once

#include "tc_fwd.cuh"

namespace swa {
namespace tc {

// 12 warps: softmax warpgroups 0 and 1, warpgroup 2 = producer (warp 8),
// MMA issuer (warp 9) and two idle warps. The launch gives every thread 168
// registers (384 x 168 = 64512); warpgroup 2 drops to 72 and the softmax
// warpgroups rise to 216 (2 x 128 x 216 + 128 x 72 = 64512).
constexpr int kPairThreads = 384;
constexpr int kPairRegsSoftmax = 216;
constexpr int kPairRegsOther = 72;
static_assert(2 * 128 * kPairRegsSoftmax + 128 * kPairRegsOther <= kPairThreads * 168,
              "register split exceeds the launch's registers");

template <int D>
struct FwdPairSmem {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kQA = 0;
  static constexpr int kQB = kTile;
  static constexpr int kK0 = 2 * kTile;             // 2 stages
  static constexpr int kV0 = kK0 + 2 * kTile;       // 2 stages
  static constexpr int kBytes = kV0 + 2 * kTile;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc + 256 <= 232448, "shared memory budget (dynamic + static)");
};

enum {
  PB_Q = 0,
  PB_KFULL = 1,    // +stage
  PB_KEMPTY = 3,   // +stage
  PB_VFULL = 5,    // +stage
  PB_VEMPTY = 7,   // +stage
  PB_SFULL = 9,    // +tile
  PB_PFULL = 11,   // +tile
  PB_PV = 13,      // +tile: PV_X(j) completed
  PB_FINAL = 15,
  PB_COUNT = 16
};

template <int D>
__global__ void __launch_bounds__(kPairThreads, 1)
    fwd_tc_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                       const FwdParams prm) {
  using L = FwdPairSmem<D>;
  constexpr int KCH = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t bars[PB_COUNT];
  __shared__ uint32_t tmem_base_sh;
  __shared__ uint32_t abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int npair = prm.Hq / 2;
  const int pair = static_cast<int>(blockIdx.x) % npair, b = static_cast<int>(blockIdx.x) / npair;
  const int hA = 2 * pair;
  const int hk = hA / (prm.Hq / prm.Hkv);
  const int qt = prm.n_qtiles - 1 - static_cast<int>(blockIdx.y);   // heavy tiles first
  const int q0 = qt * kBM;
  const Band band{prm.T, prm.window, prm.causal};
  int kt_lo = 0, kt_hi = -1;
  kv_tile_range(band, q0, kBM, kBN, kt_lo, kt_hi);
  const int n_tiles = kt_hi - kt_lo + 1;
  const WaitCtl ctl{&abort_flag, prm.status, prm.wait_limit_ns};
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar(PB_Q), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(PB_KFULL + s), 1);
      mbar_init(bar(PB_KEMPTY + s), 1);
      mbar_init(bar(PB_VFULL + s), 1);
      mbar_init(bar(PB_VEMPTY + s), 1);
      mbar_init(bar(PB_SFULL + s), 1);
      mbar_init(bar(PB_PFULL + s), 4);
      mbar_init(bar(PB_PV + s), 1);
    }
    mbar_init(bar(PB_FINAL), 1);
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
  if (warp >= 8) {
  setmaxnreg_dec<kPairRegsOther>();
  const uint32_t one = (lane == 0);   // the lane that issues in warp-wide loops
  if (warp == 8) {
    // ---------------- TMA producer (whole warp, lane 0 issues) ----------------
    if (n_tiles > 0) {
      if (one) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
      }
      mbar_arrive_expect_tx_w(bar(PB_Q), 2 * L::kTile, one);
      for (int c = 0; c < KCH; ++c) {
        tma_load_4d_w(sbase + L::kQA + c * 16384, &tmQ, bar(PB_Q), 64 * c, q0, hA, b, one);
        tma_load_4d_w(sbase + L::kQB + c * 16384, &tmQ, bar(PB_Q), 64 * c, q0, hA + 1, b, one);
      }
      bool ok = true;
      int last_k[2] = {-1, -1}, last_v[2] = {-1, -1};
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int s = j & 1;
        const int k0 = (kt_lo + j) * kBN;
        if (j >= 2) ok = mbar_wait_warp(bar(PB_KEMPTY + s), ((j - 2) >> 1) & 1, ctl);
        if (!ok) break;
        mbar_arrive_expect_tx_w(bar(PB_KFULL + s), L::kTile, one);
        for (int c = 0; c < KCH; ++c)
          tma_load_4d_w(sbase + L::kK0 + s * L::kTile + c * 16384, &tmK, bar(PB_KFULL + s), 64 * c,
                        k0, hk, b, one);
        last_k[s] = j;
        if (j >= 2) ok = mbar_wait_warp(bar(PB_VEMPTY + s), ((j - 2) >> 1) & 1, ctl);
        if (!ok) break;
        mbar_arrive_expect_tx_w(bar(PB_VFULL + s), L::kTile, one);
        for (int c = 0; c < KCH; ++c)
          tma_load_4d_w(sbase + L::kV0 + s * L::kTile + c * 16384, &tmV, bar(PB_VFULL + s), 64 * c,
                        k0, hk, b, one);
        last_v[s] = j;
      }
      mbar_wait_drain(bar(PB_Q), 0, prm.wait_limit_ns);
      for (int s = 0; s < 2; ++s) {
        if (last_k[s] >= 0) mbar_wait_drain(bar(PB_KFULL + s), (last_k[s] >> 1) & 1, prm.wait_limit_ns);
        if (last_v[s] >= 0) mbar_wait_drain(bar(PB_VFULL + s), (last_v[s] >> 1) & 1, prm.wait_limit_ns);
      }
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer (whole warp, lane 0 issues) ----------------
    if (n_tiles > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, 0, 0);
      constexpr uint32_t idO = idesc_bf16_f32(kBM, D, 0, 1);
      // Descriptor bases, computed once; every MMA adds a constant offset.
      const uint64_t dQ0 = sdesc_sw128(sbase + L::kQA, 16, 1024);
      const uint64_t dK0 = sdesc_sw128(sbase + L::kK0, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(sbase + L::kV0, 16384, 1024);
      auto issue_s = [&](int X, int j) {
        const uint64_t qd = sdesc_add(dQ0, X * L::kTile), kd = sdesc_add(dK0, (j & 1) * L::kTile);
        const uint32_t dst = tmem + X * 128;
        static_for<0, D / 16>([&](auto kc) {
          constexpr int kk = decltype(kc)::value;
          constexpr uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          umma_ss_imm<idS, off, off>(dst, qd, kd, kk > 0 ? 1u : 0u, one);
        });
        umma_commit_w(bar(PB_SFULL + X), one);
      };
      auto issue_pv = [&](int X, int j) {
        const uint64_t vd = sdesc_add(dV0, (j & 1) * L::kTile);
        const uint32_t dst = tmem + 256 + X * D, pa = tmem + X * 128;
        umma_ts_imm<idO, 0, 0>(dst, pa, vd, j > 0 ? 1u : 0u, one);
        static_for<1, kBN / 16>([&](auto kc) {
          constexpr int kk = decltype(kc)::value;
          umma_ts_imm<idO, kk * 8, kk * 2048 / 16>(dst, pa, vd, 1u, one);
        });
        umma_commit_w(bar(PB_PV + X), one);
      };
      bool ok = mbar_wait_warp(bar(PB_Q), 0, ctl) && mbar_wait_warp(bar(PB_KFULL), 0, ctl);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        issue_s(1, 0);
        umma_commit_w(bar(PB_KEMPTY), one);
      }
      for (int j = 1; j < n_tiles && ok; ++j) {
        const int s = j & 1, sp = (j - 1) & 1;
        ok = mbar_wait_warp(bar(PB_KFULL + s), (j >> 1) & 1, ctl) &&
             mbar_wait_warp(bar(PB_PFULL + 0), (j - 1) & 1, ctl) &&
             mbar_wait_warp(bar(PB_VFULL + sp), ((j - 1) >> 1) & 1, ctl);
        if (!ok) break;
        tc_fence_after();
        issue_pv(0, j - 1);
        issue_s(0, j);
        if (!(ok = mbar_wait_warp(bar(PB_PFULL + 1), (j - 1) & 1, ctl))) break;
        tc_fence_after();
        issue_pv(1, j - 1);
        umma_commit_w(bar(PB_VEMPTY + sp), one);
        issue_s(1, j);
        umma_commit_w(bar(PB_KEMPTY + s), one);
      }
      if (ok) {
        const int j = n_tiles - 1;
        ok = mbar_wait_warp(bar(PB_PFULL + 0), j & 1, ctl) &&
             mbar_wait_warp(bar(PB_VFULL + (j & 1)), (j >> 1) & 1, ctl);
        if (ok) {
          tc_fence_after();
          issue_pv(0, j);
          if ((ok = mbar_wait_warp(bar(PB_PFULL + 1), j & 1, ctl))) {
            tc_fence_after();
            issue_pv(1, j);
            umma_commit_w(bar(PB_VEMPTY + (j & 1)), one);
          }
        }
      }
      umma_commit_w(bar(PB_FINAL), one);
      mbar_wait_drain(bar(PB_FINAL), 0, prm.wait_limit_ns);
    }
  }
  } else {
    // ---------------- softmax warpgroups (A: warps 0-3, B: warps 4-7) ----------------
    setmaxnreg_inc<kPairRegsSoftmax>();
    const int X = warp >> 2;
    const int h = hA + X;
    const int row = threadIdx.x & 127;        // TMEM lane
    const int i = q0 + row;                   // query position
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + X * 128 + lane_off;
    const uint32_t tO = tmem + 256 + X * D + lane_off;
    const float c = prm.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = n_tiles > 0;
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int k0 = (kt_lo + j) * kBN;
      ok = mbar_wait_warp(bar(PB_SFULL + X), j & 1, ctl);
      if (!ok) break;
      tc_fence_after();
      // Visible key columns of this row on a partial tile: [clo, chi].
      const bool full = tile_full(band, q0, kBM, k0, kBN);
      int clo = 0, chi = kBN - 1;
      if (!full) {
        if (i >= prm.T) {
          clo = 1; chi = 0;
        } else {
          if (prm.T - 1 - k0 < chi) chi = prm.T - 1 - k0;
          if (prm.causal) {
            if (i - k0 < chi) chi = i - k0;
            if (prm.window >= 0 && i - prm.window - k0 > clo) clo = i - prm.window - k0;
          } else if (prm.window >= 0) {
            if (i + prm.window - k0 < chi) chi = i + prm.window - k0;
            if (i - prm.window - k0 > clo) clo = i - prm.window - k0;
          }
        }
      }
      auto mask = [&](uint32_t (&r)[32], int cc) {
        if (!full) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int col = cc * 32 + e;
            if (col < clo || col > chi) r[e] = __float_as_uint(-INFINITY);
          }
        }
      };
      uint32_t sr[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + cc * 32, sr[cc]);
      tmem_wait_ld(sr[0]);
      reg_fence(sr[1]);
      reg_fence(sr[2]);
      reg_fence(sr[3]);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) mask(sr[cc], cc);
      // Row maximum: eight independent three-input chains, then a short tree.
      float mq[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int cc = q >> 1, e0 = (q & 1) * 16;
        float a = fmax3(__uint_as_float(sr[cc][e0]), __uint_as_float(sr[cc][e0 + 1]),
                        __uint_as_float(sr[cc][e0 + 2]));
#pragma unroll
        for (int e = 3; e < 15; e += 2)
          a = fmax3(a, __uint_as_float(sr[cc][e0 + e]), __uint_as_float(sr[cc][e0 + e + 1]));
        mq[q] = fmaxf(a, __uint_as_float(sr[cc][e0 + 15]));
      }
      const float mx = fmaxf(fmax3(mq[0], mq[1], mq[2]),
                             fmax3(fmax3(mq[3], mq[4], mq[5]), mq[6], mq[7]));
      const float mt = mx * c;
      float alpha = 1.f;
      bool rescale_o = false;
      if (mt > m + kRescaleLog2) {     // also the first finite maximum (m = -inf)
        if (m != -INFINITY) {
          alpha = ex2_approx(m - mt);
          rescale_o = true;
        }
        l *= alpha;
        m = mt;
      }
      // PV_X(j-1) has completed: the commit that signalled S_X(j) covers it.
      if (__any_sync(0xffffffffu, rescale_o)) {
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t orr[32];
          tmem_ld32(tO + cc * 32, orr);
          tmem_wait_ld(orr);
#pragma unroll
          for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
          tmem_st32(tO + cc * 32, orr);
        }
      }
      // P = exp2(S c - m) as bf16 pairs into S's first 64 columns; the
      // scale-and-shift and the row sum run two lanes per instruction.
      const float nm = (m == -INFINITY) ? 0.f : -m;
      float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int w = 0; w < 32; ++w) {
          const int cc = half * 2 + (w >> 4), e = (w & 15) * 2;
          float x0, x1;
          ffma2(x0, x1, __uint_as_float(sr[cc][e]), __uint_as_float(sr[cc][e + 1]), c, c, nm, nm);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          fadd2_acc(ls[2 * (w & 3)], ls[2 * (w & 3) + 1], p0, p1);
          pk[w] = pack_bf16x2(p0, p1);
        }
        tmem_st32(tS + half * 32, pk);
      }
      const float lsum = ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      l += lsum;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(PB_PFULL + X));
    }
    // ---- epilogue: O / l, LSE ----
    if (ok) ok = mbar_wait_warp(bar(PB_PV + X), (n_tiles - 1) & 1, ctl);
    // O / l goes through this warpgroup's Q tile (no longer read by any MMA)
    // in the 128-byte swizzle layout, then out with bulk tensor stores.
    const uint32_t sOut = sbase + (X == 0 ? L::kQA : L::kQB);
    if (ok) {
      tc_fence_after();
      const bool empty = !(l > 0.f);
      const float inv = empty ? 0.f : 1.0f / l;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t orr[32];
        tmem_ld32(tO + cc * 32, orr);
        tmem_wait_ld(orr);
#pragma unroll
        for (int e = 0; e < 32; e += 8)
          st_shared_v4(sw128_addr(sOut, kBM, row, (cc * 32 + e) / 8),
                       pack_bf16x2(__uint_as_float(orr[e + 0]) * inv, __uint_as_float(orr[e + 1]) * inv),
                       pack_bf16x2(__uint_as_float(orr[e + 2]) * inv, __uint_as_float(orr[e + 3]) * inv),
                       pack_bf16x2(__uint_as_float(orr[e + 4]) * inv, __uint_as_float(orr[e + 5]) * inv),
                       pack_bf16x2(__uint_as_float(orr[e + 6]) * inv, __uint_as_float(orr[e + 7]) * inv));
      }
      if (i < prm.T) {
        prm.lse[(static_cast<long long>(b) * prm.Hq + h) * prm.T + i] =
            empty ? -INFINITY : (m + log2f(l)) * 0.69314718055994531f;
      }
      fence_async_smem();
    }
    ok = named_bar_and(1 + X, 128, ok);
    if (ok && row == 0) {
      for (int c = 0; c < KCH; ++c) tma_store_4d(&tmO, sOut + c * 16384, 64 * c, q0, h, b);
      bulk_commit_group();
      bulk_wait_group_all();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
inline swa_status launch_fwd_pair_d(const FwdLaunch& f, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mo;
  if (!map_head_major(&mq, f.qn, f.B, f.Hq, f.T, D) || !map_head_major(&mk, f.kn, f.B, f.Hkv, f.T, D) ||
      !map_token_major(&mo, f.o, f.B, f.Hq, f.T, D))
    return SWA_ERR_CUDA;
  const bool okv = f.v_head_major ? map_head_major(&mv, f.v, f.B, f.Hkv, f.T, D)
                                  : map_token_major(&mv, f.v, f.B, f.Hkv, f.T, D);
  if (!okv) return SWA_ERR_CUDA;
  FwdParams p{};
  p.T = f.T; p.Hq = f.Hq; p.Hkv = f.Hkv; p.window = f.window; p.causal = f.causal;
  p.n_qtiles = (f.T + kBM - 1) / kBM;
  p.scale_log2 = f.scale * 1.4426950408889634f;
  p.o = f.o; p.lse = f.lse; p.status = f.status; p.wait_limit_ns = f.wait_limit_ns;
  if (cudaFuncSetAttribute(fwd_tc_pair_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           FwdPairSmem<D>::kAlloc) != cudaSuccess)
    return SWA_ERR_CUDA;
  dim3 grid(f.B * (f.Hq / 2), p.n_qtiles);
  fwd_tc_pair_kernel<D><<<grid, kPairThreads, FwdPairSmem<D>::kAlloc, st>>>(mq, mk, mv, mo, p);
  return cudaGetLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

// Forward dispatch: two heads per CTA when the GQA group size is even, one
// head per CTA otherwise.
inline swa_status launch_fwd_any(const FwdLaunch& f, cudaStream_t st) {
  if ((f.Hq / f.Hkv) % 2 == 0)
    return f.d == 64 ? launch_fwd_pair_d<64>(f, st) : launch_fwd_pair_d<128>(f, st);
  return launch_fwd(f, st);
}

}  // namespace tc
}  // namespace swa
