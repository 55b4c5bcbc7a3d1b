// Backward attention core for d = 128 with 128-query steps (sm_103a).
//
// One CTA per 128-key tile of a (batch, kv head): K and V stay in shared
// memory, dK and dV accumulate in TMEM over the GQA group and the in-band
// 128-row query tiles, so the GQA reduction of dK and dV happens inside the
// CTA. Every product of a step is a full M = 128, N = 128 tcgen05 MMA:
//   S^T  = K Q_i^T            (TMEM [0,128): lanes = keys, columns = queries)
//   dP^T = V dO_i^T           (TMEM [128,256))
//   P^T  = scale exp2(S^T c - LSE log2 e)     -> bf16 into S^T's columns
//   dS^T = P^T (dP^T - D)                     -> bf16 to shared memory
//   dV  += P^T dO_i           (A operand from TMEM)
//   dQ_i^T = K^T dS^T         (into dP^T's columns; B operand dS^T from shared memory)
//   dK  += dS^T Q_i           (A operand dS^T from TMEM, beside P^T)
// P^T and dS^T carry the softmax scale, so dK and dQ come out final and dV
// is divided by it in the epilogue.
//
// Roles (16 warps): warpgroups 0 and 1 do the element-wise work, each on 64
// of the step's 128 query columns (thread = key row = TMEM lane): per step
// P(i), then dS(i). Warpgroup 2 drains dQ^T(i) from TMEM into the staging
// boxes, off the element-wise warps' path. Warp 12 is the TMA producer of K,
// V (once) and of Q with LSE and D (two stages); warp 15 of dO (one stage,
// reloaded as soon as dV of the step completed); warp 14 adds the staged dQ
// boxes into the fp32 accumulator; warp 13 issues the MMAs from one thread,
// in the order
//   S(0) dP(0) | dV(i) [dQ(i) dK(i)] S(i+1) dP(i+1) | ...
// dQ^T(i) comes before dK(i) so that its drain starts one product earlier;
// dP^T(i+1) waits for that drain (it reuses the columns).
// dQ^T(i) goes from TMEM to shared memory in four [32 queries][128] fp32
// boxes, two in the dedicated staging buffer (free once the previous step's
// boxes there were read) and two in the dS^T buffer (free once dQ^T(i), its
// only reader, completed; dS^T(i+1) waits for the reducer), and from there into the fp32 dQ
// accumulator by TMA bulk reductions. Those run at the rate the L2 accepts fp32 adds (about 6.6 TB/s
// over the whole GPU, about 21 bytes per clock per SM), 64 KB per step.
// Registers (setmaxnreg; 512 x 128 at launch): element-wise warpgroups 176
// per thread, drain warpgroup 96, the four single-role warps 56.
//
// Softmax backward written out from the forward of the attention block
// (autoresearch Administrator & Developer Guide §8.2.1; train.py
// walkthrough post, model paragraph).
#pragma once

#include "tc_bwd.cuh"

namespace swa {
namespace tc {

constexpr int kB2Threads = 512;
constexpr int kB2RegsSoftmax = 176;   // element-wise warpgroups 0, 1
constexpr int kB2RegsDrain = 96;      // drain warpgroup (warps 8-11)
constexpr int kB2RegsOther = 56;      // producers, MMA issuer, reducer (warps 12-15)
constexpr int kB2ProdWarp = 12, kB2MmaWarp = 13, kB2RedWarp = 14, kB2GWarp = 15;
static_assert(2 * 128 * kB2RegsSoftmax + 128 * kB2RegsDrain + 128 * kB2RegsOther <= kB2Threads * 128,
              "register split exceeds the launch's registers");

struct B2Cfg {
  static constexpr int D = 128;
  static constexpr int BQ = 128;                 // queries per step
  static constexpr int kTile = 128 * 128 * 2;    // 32 KB: K, V, a Q or dO stage, dS^T
  static constexpr int kHalf = kTile / 2;        // a 64-column half (one SW128 region)
  static constexpr int oK = 0;
  static constexpr int oV = oK + kTile;
  static constexpr int oQ = oV + kTile;          // 2 stages
  static constexpr int oG = oQ + 2 * kTile;      // dO, one stage
  static constexpr int oS = oG + kTile;          // dS^T [128 keys][128 queries]
  static constexpr int oX = oS + kTile;          // dQ staging: the second box of each warpgroup
  static constexpr int oL = oX + kTile;          // 2 stages x BQ floats: log2(scale) - LSE log2(e)
  static constexpr int oD = oL + 2 * BQ * 4;     // 2 stages x BQ floats: -D
  static constexpr int oBar = oD + 2 * BQ * 4;   // mbarriers, TMEM base, abort flag
  static constexpr int kBytes = oBar + 256;
  // The whole budget is dynamic shared memory (no static shared variables),
  // so the dynamic base is the start of the CTA's window (1024-aligned).
  static_assert(kBytes <= 232448, "shared memory budget");
};

enum {
  B2_KV = 0,
  B2_QFULL = 1,      // +stage: Q, LSE, D of a step landed
  B2_QEMPTY = 3,     // +stage: the dK product of the step completed (Q stage reusable)
  B2_GFULL = 5,      // dO landed
  B2_GFREE = 7,      // the dV product of the step completed (dO stage reusable)
  B2_SFULL = 9,      // S^T in TMEM
  B2_DPFULL = 10,    // dP^T in TMEM
  B2_PREADY = 11,    // P^T in TMEM (8 warps)
  B2_DSREADY = 12,   // dS^T in TMEM and shared memory (8 warps)
  B2_DQFULL = 13,    // dQ^T in TMEM
  B2_DQFREE = 14,    // dQ^T read out of TMEM (8 warps)
  B2_STAGED = 15,    // the step's four dQ boxes are in shared memory (8 warps)
  B2_XFREE = 16,     // the dQ boxes in the staging buffer were read
  B2_DSFREE = 17,    // the dQ boxes staged in the dS^T buffer were read
  B2_FINAL = 18,
  B2_KRAW = 19,      // the raw k rows of the key tile landed (for the epilogue)
  B2_COUNT = 20
};

// Visible query columns [clo, chi] of key row j among the 64 queries
// starting at qb, on a tile that is not entirely inside the band.
__device__ __forceinline__ void key_row_span(const Band& band, int j, int qb, int& clo, int& chi) {
  clo = 0;
  chi = 63;
  if (j >= band.T) {
    clo = 1;
    chi = 0;
    return;
  }
  if (band.T - 1 - qb < chi) chi = band.T - 1 - qb;
  if (band.causal) {
    if (j - qb > clo) clo = j - qb;
    if (band.window >= 0 && j + band.window - qb < chi) chi = j + band.window - qb;
  } else if (band.window >= 0) {
    if (j - band.window - qb > clo) clo = j - band.window - qb;
    if (j + band.window - qb < chi) chi = j + band.window - qb;
  }
}

// 64 fp32 values (two 32-column TMEM loads) -> 32 bf16 pairs of consecutive
// columns.
__device__ __forceinline__ void pack64(const uint32_t (&v)[2][32], uint32_t (&pk)[32]) {
#pragma unroll
  for (int w = 0; w < 32; ++w)
    pk[w] = pack_bf16x2(__uint_as_float(v[w >> 4][(w & 15) * 2]),
                        __uint_as_float(v[w >> 4][(w & 15) * 2 + 1]));
}

template <bool kPolled>
__global__ void __launch_bounds__(kB2Threads, 1)
    bwd_tc128_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                     const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmDK,
                     const __grid_constant__ CUtensorMap tmDV, const __grid_constant__ CUtensorMap tmKr,
                     const BwdParams prm) {
  using C = B2Cfg;
  constexpr int D = C::D, BQ = C::BQ;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {   // swizzle atoms need 1024-byte aligned tiles (uniform over the CTA)
    if (threadIdx.x == 0) atomicOr(prm.status, DEV_ERR_BOUNDS);
    return;
  }
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(smem + C::oBar + B2_COUNT * 8);
  uint32_t* abort_flag = tmem_base_sh + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA -> (key tile, batch x kv head). The (batch, kv head) pairs are cut
  // into chunks of prm.chunk; within a chunk the CTAs go key tile by key tile
  // (all pairs of key tile 0, then of key tile 1, ...). On a causal band the
  // early key tiles see the most query tiles, so the heavy CTAs of a chunk
  // start first and the grid ends on light ones, while the Q, dO and dQ rows
  // that the running CTAs share (one chunk's worth) stay in L2.
  int kt, bhk;
  {
    const int id = static_cast<int>(blockIdx.x);
    const int per = prm.chunk * prm.n_ktiles;
    const int ch = id / per;
    const int r = id - ch * per;
    const int rest = prm.n_bhk - ch * prm.chunk;
    const int cn = rest < prm.chunk ? rest : prm.chunk;
    kt = r / cn;
    bhk = ch * prm.chunk + (r - kt * cn);
  }
  const int b = bhk / prm.Hkv, hk = bhk % prm.Hkv;
  const int k0 = kt * kBK;
  const int G = prm.Hq / prm.Hkv;
  const Band band{prm.T, prm.window, prm.causal};
  int qlo = 0, qhi = -1;
  q_tile_range(band, k0, kBK, BQ, qlo, qhi);
  const int nq = qhi - qlo + 1;
  const int n_it = nq > 0 ? nq * G : 0;
  const WaitCtl<kPolled> ctl{abort_flag, prm.status, prm.wait_limit_ns};
  auto bar = [&](int i) { return sbase + C::oBar + 8u * static_cast<uint32_t>(i); };

  if (threadIdx.x == 0) {
    // the accumulator is about to receive this launch's additions
    if (blockIdx.x == 0 && prm.acc_flag != nullptr) prm.acc_flag[1] = 0ull;
    *abort_flag = 0;
    mbar_init(bar(B2_KV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B2_QFULL + s), 1);
      mbar_init(bar(B2_QEMPTY + s), 1);
    }
    mbar_init(bar(B2_GFULL), 1);
    mbar_init(bar(B2_GFREE), 1);
    mbar_init(bar(B2_SFULL), 1);
    mbar_init(bar(B2_DPFULL), 1);
    mbar_init(bar(B2_PREADY), 8);
    mbar_init(bar(B2_DSREADY), 8);
    mbar_init(bar(B2_DQFULL), 1);
    mbar_init(bar(B2_DQFREE), 4);
    mbar_init(bar(B2_STAGED), 4);
    mbar_init(bar(B2_XFREE), 1);
    mbar_init(bar(B2_DSFREE), 1);
    mbar_init(bar(B2_FINAL), 1);
    mbar_init(bar(B2_KRAW), 1);
    fence_mbar_init();
  }
  if (warp == kB2MmaWarp) {
    tmem_alloc(smem_u32(tmem_base_sh), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_sh;
  constexpr uint32_t cS = 0, cDP = 128, cDV = 256, cDK = 384;

  if (warp >= kB2ProdWarp) {
    setmaxnreg_dec<kB2RegsOther>();
    if (warp == kB2ProdWarp && lane == 0 && n_it > 0) {
      // ---------------- TMA producer of K, V, and per step Q, LSE, D ----------------
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(bar(B2_KV), 2 * C::kTile);
      for (int c = 0; c < 2; ++c) {
        tma_load_4d(sbase + C::oK + c * C::kHalf, &tmK, bar(B2_KV), 64 * c, k0, hk, b);
        tma_load_4d(sbase + C::oV + c * C::kHalf, &tmV, bar(B2_KV), 64 * c, k0, hk, b);
      }
      int last[2] = {-1, -1};
      for (int it = 0; it < n_it; ++it) {
        const int s = it & 1;
        const int h = hk * G + it / nq;
        const int q0 = (qlo + it % nq) * BQ;
        // the stage is free once the dK product two steps back completed (and,
        // with dQ boxes staged in it, once those were read)
        if (it >= 2 && !mbar_wait(bar(B2_QEMPTY + s), ((it >> 1) - 1) & 1, ctl)) break;
        last[s] = it;
        mbar_arrive_expect_tx(bar(B2_QFULL + s), C::kTile + 2 * BQ * 4);
        for (int c = 0; c < 2; ++c)
          tma_load_4d(sbase + C::oQ + s * C::kTile + c * C::kHalf, &tmQ, bar(B2_QFULL + s), 64 * c,
                      q0, h, b);
        const long long row = (static_cast<long long>(b) * prm.Hq + h) * prm.Tpad + q0;
        bulk_load(sbase + C::oL + s * BQ * 4, prm.lse2 + row, BQ * 4, bar(B2_QFULL + s));
        bulk_load(sbase + C::oD + s * BQ * 4, prm.dvec + row, BQ * 4, bar(B2_QFULL + s));
        if (it == n_it - 1 && prm.dkn_out == nullptr) {
          // the epilogue's inverse RMS of the k rows into L2, a step ahead
          const float* rs = prm.rstd_k + (static_cast<long long>(b) * prm.Hkv + hk) * prm.T + k0;
          const uint32_t nrs = static_cast<uint32_t>(prm.T - k0 < kBK ? prm.T - k0 : kBK) * 4;
          // whole 16-byte units inside the row only (a bulk prefetch needs
          // a 16-byte aligned start and size)
          const uintptr_t a0 = (reinterpret_cast<uintptr_t>(rs) + 15) & ~uintptr_t(15);
          const uintptr_t a1 = (reinterpret_cast<uintptr_t>(rs) + nrs) & ~uintptr_t(15);
          if (a1 > a0) bulk_prefetch_l2(reinterpret_cast<const void*>(a0), static_cast<uint32_t>(a1 - a0));
        }
      }
      // The epilogue's raw k rows into the Q stage that the last step does
      // not use, once the dK product of the step before it has completed.
      bool kraw = false;
      if (prm.dkn_out == nullptr && !*reinterpret_cast<volatile uint32_t*>(abort_flag)) {
        const int s = n_it & 1;
        if (n_it < 2 || mbar_wait(bar(B2_QEMPTY + s), ((n_it >> 1) - 1) & 1, ctl)) {
          mbar_arrive_expect_tx(bar(B2_KRAW), C::kTile);
          for (int c = 0; c < 2; ++c)
            tma_load_4d(sbase + C::oQ + s * C::kTile + c * C::kHalf, &tmKr, bar(B2_KRAW), 64 * c, k0, hk, b);
          kraw = true;
        }
      }
      mbar_wait_drain(bar(B2_KV), 0, kDrainLimitNs);
      for (int s = 0; s < 2; ++s)
        if (last[s] >= 0) mbar_wait_drain(bar(B2_QFULL + s), (last[s] >> 1) & 1, kDrainLimitNs);
      if (kraw) mbar_wait_drain(bar(B2_KRAW), 0, kDrainLimitNs);
    } else if (warp == kB2GWarp && lane == 0 && n_it > 0) {
      // ---------------- TMA producer of dO (one stage) ----------------
      tma_prefetch_desc(&tmG);
      int last = -1;
      for (int it = 0; it < n_it; ++it) {
        const int h = hk * G + it / nq;
        const int q0 = (qlo + it % nq) * BQ;
        // the stage is free once dV of the previous step completed
        if (it >= 1 && !mbar_wait(bar(B2_GFREE), (it - 1) & 1, ctl)) break;
        last = it;
        mbar_arrive_expect_tx(bar(B2_GFULL), C::kTile);
        for (int c = 0; c < 2; ++c)
          tma_load_4d(sbase + C::oG + c * C::kHalf, &tmG, bar(B2_GFULL), 64 * c, q0, h, b);
      }
      if (last >= 0) mbar_wait_drain(bar(B2_GFULL), last & 1, kDrainLimitNs);
    } else if (warp == kB2RedWarp && lane == 0 && n_it > 0) {
      // ---------------- dQ reducer ----------------
      // Step m's dQ boxes, for each warpgroup X: queries qb.. in half X of the
      // step's Q stage, qb+32.. in half X of the staging buffer, added into
      // the fp32 accumulator by bulk reductions. These run at the rate the L2
      // accepts fp32 adds (about 6.6 TB/s over the whole GPU, about 21 bytes
      // per clock per SM, so about 3000 clocks per step); each buffer is
      // handed back as soon as its boxes have been read, the Q stage first.
      tma_prefetch_desc(&tmDQ);
      for (int m = 0; m < n_it; ++m) {
        if (!mbar_wait(bar(B2_STAGED), m & 1, ctl)) break;
        const int h = hk * G + m / nq;
        const int q0 = (qlo + m % nq) * BQ;
        for (int X = 0; X < 2; ++X)
          tma_reduce_add_3d(&tmDQ, sbase + C::oS + X * C::kHalf, 0, q0 + 64 * X,
                            b * prm.Hq + h);
        bulk_commit_group();
        for (int X = 0; X < 2; ++X)
          tma_reduce_add_3d(&tmDQ, sbase + C::oX + X * C::kHalf, 0, q0 + 64 * X + 32, b * prm.Hq + h);
        bulk_commit_group();
        bulk_wait_group_read<1>();
        mbar_arrive(bar(B2_DSFREE));
        bulk_wait_group_read<0>();
        mbar_arrive(bar(B2_XFREE));
      }
      bulk_wait_group_read<0>();   // shared memory stays valid until read
    } else if (warp == kB2MmaWarp && lane == 0 && n_it > 0) {
      // ---------------- MMA issuer (one thread) ----------------
      constexpr uint32_t idN = idesc_bf16_f32(128, 128, 0, 0);    // S^T, dP^T
      constexpr uint32_t idKV = idesc_bf16_f32(128, 128, 0, 1);   // dV, dK (A from TMEM)
      constexpr uint32_t idQ = idesc_bf16_f32(128, 128, 1, 1);    // dQ^T = K^T dS^T
      const uint64_t dKk = sdesc_sw128(sbase + C::oK, 16, 1024);
      const uint64_t dVk = sdesc_sw128(sbase + C::oV, 16, 1024);
      const uint64_t dKmn = sdesc_sw128(sbase + C::oK, C::kHalf, 1024);
      const uint64_t dQk0 = sdesc_sw128(sbase + C::oQ, 16, 1024);
      const uint64_t dGk = sdesc_sw128(sbase + C::oG, 16, 1024);
      const uint64_t dQmn0 = sdesc_sw128(sbase + C::oQ, C::kHalf, 1024);
      const uint64_t dGmn = sdesc_sw128(sbase + C::oG, C::kHalf, 1024);
      const uint64_t dSmn = sdesc_sw128(sbase + C::oS, C::kHalf, 1024);
      // K-major operands: K step kk is 32 bytes into a row of its 64-column region.
      auto issue_S = [&](int i) {    // S^T = K Q_i^T
        const uint64_t qd = sdesc_add(dQk0, (i & 1) * C::kTile);
        static_for<0, 8>([&](auto kc) {
          constexpr int kk = decltype(kc)::value;
          constexpr uint32_t off = ((kk >> 2) * C::kHalf + (kk & 3) * 32) >> 4;
          umma_ss_imm<idN, off, off>(tmem + cS, dKk, qd, kk > 0, 1u);
        });
        umma_commit(bar(B2_SFULL));
      };
      auto issue_dP = [&](int i) {   // dP^T = V dO_i^T
        static_for<0, 8>([&](auto kc) {
          constexpr int kk = decltype(kc)::value;
          constexpr uint32_t off = ((kk >> 2) * C::kHalf + (kk & 3) * 32) >> 4;
          umma_ss_imm<idN, off, off>(tmem + cDP, dVk, dGk, kk > 0, 1u);
        });
        umma_commit(bar(B2_DPFULL));
      };
      // A operands from TMEM: K step kk (16 queries) is 8 columns; queries
      // 0-63 sit in the first 32 columns of warpgroup 0's 64, queries 64-127
      // in warpgroup 1's. MN-major B: K step kk is 16 rows (2048 bytes) on.
      auto issue_dV = [&](int i) {   // dV += P^T dO_i; then the dO stage is free
        static_for<0, 8>([&](auto kc) {
          constexpr int kk = decltype(kc)::value;
          umma_ts_imm<idKV, (kk >> 2) * 64 + (kk & 3) * 8, kk * 128>(tmem + cDV, tmem + cS, dGmn,
                                                                      (i > 0 || kk > 0), 1u);
        });
        umma_commit(bar(B2_GFREE));
      };
      auto issue_dQdK = [&](int i) {   // dQ_i^T = K^T dS^T, then dK += dS^T Q_i (A from shared memory)
        static_for<0, 8>([&](auto kc) {
          constexpr int kk = decltype(kc)::value;
          umma_ss_imm<idQ, kk * 128, kk * 128>(tmem + cDP, dKmn, dSmn, kk > 0, 1u);
        });
        umma_commit(bar(B2_DQFULL));
        const uint64_t qd = sdesc_add(dQmn0, (i & 1) * C::kTile);
        // A = dS^T from TMEM (columns 32-63 of each warpgroup's 64 in S^T's region)
        static_for<0, 8>([&](auto kc) {
          constexpr int kk = decltype(kc)::value;
          umma_ts_imm<idKV, 32 + (kk >> 2) * 64 + (kk & 3) * 8, kk * 128>(tmem + cDK, tmem + cS, qd,
                                                                            (i > 0 || kk > 0), 1u);
        });
        umma_commit(bar(B2_QEMPTY + (i & 1)));   // the last reader of the Q stage
      };
      bool ok = mbar_wait(bar(B2_KV), 0, ctl) && mbar_wait(bar(B2_QFULL), 0, ctl);
      if (ok) {
        tc_fence_after();
        issue_S(0);
      }
      ok = ok && mbar_wait(bar(B2_GFULL), 0, ctl);
      if (ok) {
        tc_fence_after();
        issue_dP(0);
      }
      for (int i = 0; i < n_it && ok; ++i) {
        const int ph = i & 1;
        const bool more = i + 1 < n_it;
        const int s1 = (i + 1) & 1, ph1 = ((i + 1) >> 1) & 1;
        if (!(ok = mbar_wait(bar(B2_PREADY), ph, ctl))) break;
        tc_fence_after();
        issue_dV(i);
        if (!(ok = mbar_wait(bar(B2_DSREADY), ph, ctl))) break;
        tc_fence_after();
        issue_dQdK(i);
        if (more) {
          if (!(ok = mbar_wait(bar(B2_QFULL + s1), ph1, ctl))) break;
          tc_fence_after();
          issue_S(i + 1);
        }
        if (more) {
          // dP^T(i+1) overwrites dQ^T(i): wait until it was read out.
          if (!(ok = mbar_wait(bar(B2_DQFREE), ph, ctl) && mbar_wait(bar(B2_GFULL), (i + 1) & 1, ctl)))
            break;
          tc_fence_after();
          issue_dP(i + 1);
        }
      }
      umma_commit(bar(B2_FINAL));
      mbar_wait_drain(bar(B2_FINAL), 0, kDrainLimitNs);
    }
  } else if (warp >= 8) {
    // --------- drain warpgroup: dQ^T(i) (lane = head-dim index) -> staged boxes ---------
    // Boxes [32 queries][128] fp32: queries 64X .. 64X + 31 in half X of the
    // dS^T buffer (free once dQ^T(i), its only reader, completed: DQFULL; the
    // next dS^T waits until the reducer has read them), 64X + 32 .. 64X + 63 in half X
    // of the staging buffer (free once the reducer read the previous step's
    // boxes there). TMEM is handed back (DQFREE) as soon as every column has
    // been read. The Q stages hold no dQ, so a Q stage is reloaded as soon as
    // dK of its step completed.
    setmaxnreg_dec<kB2RegsDrain>();
    const int t = threadIdx.x & 127;
    const uint32_t tDQ = tmem + cDP + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    for (int i = 0; i < n_it; ++i) {
      if (!mbar_wait_warp(bar(B2_DQFULL), i & 1, ctl)) break;
      tc_fence_after();
      uint32_t a[2][32];
      tmem_ld32(tDQ + 32, a[0]);
      tmem_ld32(tDQ + 96, a[1]);
      tmem_wait_ld(a[0]);
      reg_fence(a[1]);
      if (i > 0 && !mbar_wait_warp(bar(B2_XFREE), (i - 1) & 1, ctl)) break;
#pragma unroll
      for (int X = 0; X < 2; ++X)
#pragma unroll
        for (int e = 0; e < 32; ++e)
          st_shared_f32(sbase + C::oX + X * C::kHalf + e * 512 + t * 4, __uint_as_float(a[X][e]));
      tmem_ld32(tDQ, a[0]);
      tmem_ld32(tDQ + 64, a[1]);
      tmem_wait_ld(a[0]);
      reg_fence(a[1]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B2_DQFREE));
#pragma unroll
      for (int X = 0; X < 2; ++X)
#pragma unroll
        for (int e = 0; e < 32; ++e)
          st_shared_f32(sbase + C::oS + X * C::kHalf + e * 512 + t * 4,
                        __uint_as_float(a[X][e]));
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B2_STAGED));   // the reducer adds them
    }
  } else {
    // --------- element-wise warpgroups: X = warp / 4 owns query columns [64X, 64X + 64) ---------
    setmaxnreg_inc<kB2RegsSoftmax>();
    const int X = warp >> 2;
    const int t = threadIdx.x & 127;                // key row / TMEM lane (head-dim row of dQ^T)
    const int j = k0 + t;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c = prm.scale_log2;
    const uint32_t tS = tmem + cS + 64 * X + lane_off;     // S^T, then P^T in its first 32 columns
    const uint32_t tDP = tmem + cDP + 64 * X + lane_off;   // dP^T, then dS^T, then dQ^T
    const uint32_t sSx = sbase + C::oS + X * C::kHalf;     // dS^T region X
    // Per step the order is P(i), dS(i), drain(i).
    uint32_t sr[2][32];   // P^T of the step whose dS^T comes next (fp32)
    // ---- P^T(i) = scale exp2(S^T c - LSE log2 e), zero off the band ----
    auto p_phase = [&](int i) -> bool {
      const int s = i & 1;
      const int q0 = (qlo + i % nq) * BQ;
      const int qb = q0 + 64 * X;
      const float4* L4 = reinterpret_cast<const float4*>(smem + C::oL + s * BQ * 4 + X * 256);
      if (!(mbar_wait_warp(bar(B2_QFULL + s), (i >> 1) & 1, ctl) &&
            mbar_wait_warp(bar(B2_SFULL), i & 1, ctl)))
        return false;
      tc_fence_after();
      tmem_ld32(tS, sr[0]);
      tmem_ld32(tS + 32, sr[1]);
      tmem_wait_ld(sr[0]);
      reg_fence(sr[1]);
#pragma unroll
      for (int k4 = 0; k4 < 16; ++k4) {
        const float4 lv = L4[k4];
        const int cc = k4 >> 3, e = (k4 & 7) * 4;
        float x0, x1, x2, x3;
        ffma2(x0, x1, __uint_as_float(sr[cc][e]), __uint_as_float(sr[cc][e + 1]), c, c, lv.x, lv.y);
        ffma2(x2, x3, __uint_as_float(sr[cc][e + 2]), __uint_as_float(sr[cc][e + 3]), c, c, lv.z, lv.w);
        sr[cc][e] = __float_as_uint(ex2_approx(x0));
        sr[cc][e + 1] = __float_as_uint(ex2_approx(x1));
        sr[cc][e + 2] = __float_as_uint(ex2_approx(x2));
        sr[cc][e + 3] = __float_as_uint(ex2_approx(x3));
      }
      if (!tile_full(band, q0, BQ, k0, kBK)) {
        int clo, chi;
        key_row_span(band, j, qb, clo, chi);
        // visible iff clo <= col <= chi: one unsigned compare per column
        // (an empty span masks every column)
        const unsigned lo = chi < clo ? 64u : static_cast<unsigned>(clo);
        const unsigned span = chi < clo ? 0u : static_cast<unsigned>(chi - clo);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const unsigned col = static_cast<unsigned>(cc * 32 + e);
            if (col - lo > span) sr[cc][e] = 0u;
          }
      }
      uint32_t pk[32];
      pack64(sr, pk);
      tmem_st32(tS, pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B2_PREADY));
      return true;
    };
    // ---- dS^T(i) = P^T (dP^T - D) with the scaled P^T ----
    auto ds_phase = [&](int i) -> bool {
      const float4* D4 = reinterpret_cast<const float4*>(smem + C::oD + (i & 1) * BQ * 4 + X * 256);
      if (!mbar_wait_warp(bar(B2_DPFULL), i & 1, ctl)) return false;
      tc_fence_after();
      uint32_t dp[2][32];
      tmem_ld32(tDP, dp[0]);
      tmem_ld32(tDP + 32, dp[1]);
      tmem_wait_ld(dp[0]);
      reg_fence(dp[1]);
#pragma unroll
      for (int k4 = 0; k4 < 16; ++k4) {
        const float4 dv = D4[k4];
        const int cc = k4 >> 3, e = (k4 & 7) * 4;
        float x0, x1, x2, x3;
        fadd2(x0, x1, __uint_as_float(dp[cc][e]), __uint_as_float(dp[cc][e + 1]), dv.x, dv.y);
        fadd2(x2, x3, __uint_as_float(dp[cc][e + 2]), __uint_as_float(dp[cc][e + 3]), dv.z, dv.w);
        fmul2(x0, x1, x0, x1, __uint_as_float(sr[cc][e]), __uint_as_float(sr[cc][e + 1]));
        fmul2(x2, x3, x2, x3, __uint_as_float(sr[cc][e + 2]), __uint_as_float(sr[cc][e + 3]));
        dp[cc][e] = __float_as_uint(x0);
        dp[cc][e + 1] = __float_as_uint(x1);
        dp[cc][e + 2] = __float_as_uint(x2);
        dp[cc][e + 3] = __float_as_uint(x3);
      }
      uint32_t pk[32];
      pack64(dp, pk);
      // MN-major B operand of dQ^T, in this warpgroup's half of the dS^T
      // buffer, once the dQ box of step i - 1 staged there has been read
      if (i > 0 && !mbar_wait_warp(bar(B2_DSFREE), (i - 1) & 1, ctl)) return false;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        st_sw128_chunk(sSx, kBK, t, ch, pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      // and into TMEM beside P^T: the A operand of dK
      tmem_st32(tS + 32, pk);
      tmem_wait_st();
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B2_DSREADY));
      return true;
    };
    bool ok = n_it > 0;
    // After each step, wait for its dV product: after the last, dV is final
    // and V (read by the last dP^T before it) is free.
    for (int i = 0; i < n_it && ok; ++i)
      ok = p_phase(i) && ds_phase(i) && mbar_wait_warp(bar(B2_GFREE), i & 1, ctl);
    tc_fence_after();
    // The epilogue stages dv in V while the last dQ^T and dK products still
    // run; once every product has completed (K free; dK final) it stages dk
    // in K and keeps its scratch in a Q stage, while the reducer may still be
    // reading the last dQ boxes out of the dS^T buffer and the staging buffer.
    const bool raw_k = prm.dkn_out == nullptr;
    bool final_ok = false;
    auto dk_ready = [&] {
      final_ok = ok && n_it > 0 && mbar_wait_warp(bar(B2_FINAL), 0, ctl) &&
                 (!raw_k || mbar_wait_warp(bar(B2_KRAW), 0, ctl));
      tc_fence_after();
      return final_ok;
    };
    // the raw k rows in the Q stage the last step did not use, the scratch
    // in the other
    const uint32_t sk = raw_k && n_it > 0 ? sbase + C::oQ + (n_it & 1) * C::kTile : 0u;
    float* scratch = reinterpret_cast<float*>(smem + C::oQ + ((n_it - 1) & 1) * C::kTile);
    const uint32_t sdk = sbase + C::oK, sdv = sbase + C::oV;
    kv_epilogue<D>(prm, tmem + cDK + lane_off + X * 64, tmem + cDV + lane_off + X * 64, ok && n_it > 0, X,
                   t, b, hk, kt, scratch, scratch + 256, sdk, sdv, &tmDK, &tmDV, sk, dk_ready);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kB2MmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// fp32 tensor map of the dQ accumulator [B*Hq][T][128] with boxes of `rows`
// query rows x 128 columns (no swizzle) for bulk reductions.
inline bool map_dq_acc_rows(CUtensorMap* m, float* base, int BH, int T, int rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {128 * 4, static_cast<cuuint64_t>(T) * 128 * 4};
  cuuint32_t box[3] = {128, static_cast<cuuint32_t>(rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline swa_status launch_bwd128(const BwdLaunch& f, cudaStream_t st) {
  using C = B2Cfg;
  CUtensorMap mq, mk, mv, mg, mdq, mdk, mdv, mkr;
  if (!map_token_major(&mdk, f.dk, f.B, f.Hkv, f.T, 128) ||
      !map_token_major(&mdv, f.dv, f.B, f.Hkv, f.T, 128) ||
      !map_head_major(&mq, f.qn, f.B, f.Hq, f.T, 128) ||
      !map_token_major(&mg, f.dO, f.B, f.Hq, f.T, 128) ||
      !map_head_major(&mk, f.kn, f.B, f.Hkv, f.T, 128) ||
      !map_dq_acc_rows(&mdq, f.dq_acc, f.B * f.Hq, f.T, 32) ||
      !map_token_major(&mkr, f.k, f.B, f.Hkv, f.T, 128))
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
  // P^T and dS^T carry the softmax scale: dK and dQ come out final, dV is
  // divided by it in the epilogue.
  p.dk_mul = 1.f; p.dv_mul = 1.f / f.scale;
  p.dq_acc = f.dq_acc;
  p.k = f.k; p.rstd_k = f.rstd_k; p.gk = f.gk; p.tok = f.tok; p.gate = f.gate; p.dve = f.dve;
  p.ve_scale = f.ve_scale; p.vocab = f.vocab; p.dk = f.dk; p.dv = f.dv; p.gpart_k = f.gpart_k;
  p.status = f.status; p.wait_limit_ns = f.wait_limit_ns;

  // chunks of about 2.5 waves of CTAs
  p.n_bhk = f.B * f.Hkv;
  const int want = (5 * num_sms() + 2 * p.n_ktiles - 1) / (2 * p.n_ktiles);
  p.chunk = want < 1 ? 1 : (want > p.n_bhk ? p.n_bhk : want);
  p.acc_flag = f.acc_flag;
  p.dkn_out = f.dkn_out;
  const long long n_cta = static_cast<long long>(p.n_ktiles) * p.n_bhk;
  if (n_cta > 0x7fffffffLL) return SWA_ERR_UNSUPPORTED;
  auto launch = [&](auto kern) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kBytes) != cudaSuccess)
      return SWA_ERR_CUDA;
    kern<<<static_cast<unsigned>(n_cta), kB2Threads, C::kBytes, st>>>(mq, mk, mv, mg, mdq, mdk, mdv, mkr, p);
    return cudaGetLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
  };
  return p.wait_limit_ns < kPollBelowNs ? launch(bwd_tc128_kernel<true>) : launch(bwd_tc128_kernel<false>);
}

}  // namespace tc
}  // namespace swa
