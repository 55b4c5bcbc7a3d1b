// Forward attention core, persistent: one CTA per SM loops over work items,
// each item two 128-row query tiles A and B that read the same kv head,
// against one stream of K/V tiles (sm_103a tcgen05): with an even GQA group
// the same query tile of the query heads 2p, 2p + 1 (same band); with an odd
// group (plain multi-head attention included) the query tiles 2m + 1 and 2m
// of one head, against the union of their bands.
//   warp 8      TMA producer: per item Q_A, Q_B, then the item's K_j, V_j
//               (two stages each, shared with the next item's tiles);
//   warp 9      MMA issuer (lane 0 of the converged warp issues):
//               ... PV_A(j-1), S_A(j), PV_B(j-1), S_B(j), PV_A(j), ...
//   warps 0-3   softmax of tile A, warps 4-7 of tile B: thread t owns query
//               row t (TMEM lane t), keeps the running max m and sum l,
//               rescales its O row only when m grows by more than 2^8, and
//               writes P = exp2(S c - m) as bf16 pairs back into S's columns
//               of TMEM, where the PV MMA reads it as its A operand.
// Across items: the Q tiles of the next item load as soon as the last S MMA
// of the current one completed, so the next item's first S products run
// while the softmax warpgroups finish the current item's epilogue (O / l
// from TMEM, bf16 through a 64-column staging half per warpgroup, TMA store;
// LSE); a warpgroup's first PV of an item waits until its O has been read
// out of TMEM. Items go heaviest first (query tiles from the end of the
// sequence) and are dealt to the CTAs in a back-and-forth order, so the
// per-CTA totals stay within a few percent.
// TMEM: S_A [0,128), S_B [128,256), O_A [256, 256+d), O_B [256+d, 256+2d).
//
// The method (QK-norm'd q and k from the prologue, grouped-query attention
// with kv head h / G, causal sliding-window or full causal band) follows the
// autoresearch train.py walkthrough post (model paragraph) and the
// autoresearch Administrator & Developer Guide §8.2.1 and §6.3.
#pragma once

#include <algorithm>
#include <vector>

#include "tc_fwd.cuh"

namespace swa {
namespace tc {

constexpr int kPerThreads = 384;
constexpr int kPerRegsSoftmax = 216;
constexpr int kPerRegsOther = 72;
static_assert(2 * 128 * kPerRegsSoftmax + 128 * kPerRegsOther <= kPerThreads * 168,
              "register split exceeds the launch's registers");

template <int D>
struct FwdPerSmem {
  static constexpr int kTile = 128 * D * 2;   // a 128-row Q, K or V tile
  static constexpr int kHalf = 128 * 64 * 2;  // one 64-column SW128 region (16 KB)
  static constexpr int kQA = 0;
  static constexpr int kQB = kTile;
  static constexpr int kK0 = 2 * kTile;       // 2 stages
  static constexpr int kV0 = kK0 + 2 * kTile; // 2 stages
  static constexpr int kO0 = kV0 + 2 * kTile; // O staging: one 64-column half per warpgroup
  static constexpr int kBar = kO0 + 2 * kHalf;
  static constexpr int kZero = kBar + 256;     // zeros, the source of the dQ-accumulator clears
  static constexpr int kZeroBytes = 2048;
  static constexpr int kBytes = kZero + kZeroBytes;
  // Dynamic shared memory only (no static shared variables), so its base is
  // the start of the CTA's window and 1024-byte aligned.
  static_assert(kBytes <= 232448, "shared memory budget");
};

enum {
  QP_QFULL = 0,
  QP_QEMPTY = 1,   // every S product of the item completed
  QP_KFULL = 2,    // +stage
  QP_KEMPTY = 4,   // +stage
  QP_VFULL = 6,    // +stage
  QP_VEMPTY = 8,   // +stage
  QP_SFULL = 10,   // +tile
  QP_PFULL = 12,   // +tile
  QP_PV = 14,      // +tile: PV_X of the tile completed
  QP_OFREE = 16,   // +tile: O_X of the item read out of TMEM (4 warps)
  QP_FINAL = 18,
  QP_COUNT = 19
};

struct FwdPerParams {
  int B, T, Hq, Hkv, window, causal, n_qtiles, n_items;
  int pair_heads;    // 1: items pair two query heads (even GQA group); 0: two query tiles of one head
  float scale_log2;  // softmax scale * log2(e)
  float* lse;
  uint32_t* status;
  uint64_t wait_limit_ns;
  // With a workspace sized for the backward: zero the fp32 dQ accumulator
  // [B, Hq, T, D] of the rows each item covers (null: leave it), and record
  // the zeroed byte range (acc_off, acc_len) in acc_flag[0..1].
  float* dq_acc;
  unsigned long long* acc_flag;
  unsigned long long acc_off, acc_len;
};

// Items of each CTA, chosen on the host (the items in index order, heaviest
// first, each onto the CTA with the least work so far): CTA c takes
// item[off[c]] .. item[off[c + 1] - 1] in that order. n = 0: no table (more
// items or CTAs than it holds); then rounds of G items, even rounds dealt in
// CTA order, odd rounds in reverse, so that the heavy rounds even out.
constexpr int kPerMaxCtas = 256, kPerMaxItems = 8192;
struct FwdSched {
  int n;
  uint16_t off[kPerMaxCtas + 1];
  uint16_t item[kPerMaxItems];
};

// The k-th item of CTA c of G; -1 past its last item.
__device__ __forceinline__ int per_item(const FwdSched& sc, int k, int c, int G, int n_items) {
  if (sc.n > 0) {
    const int beg = sc.off[c];
    return k < sc.off[c + 1] - beg ? static_cast<int>(sc.item[beg + k]) : -1;
  }
  const int idx = k * G + ((k & 1) ? (G - 1 - c) : c);
  return idx < n_items ? idx : -1;
}

// One work item: the query tiles A and B (128 rows each, heads hA / hB,
// first rows q0A / q0B) that run against one stream of K/V tiles
// [kt_lo, kt_lo + n_tiles) of kv head hA / (Hq / Hkv).
struct PerItem {
  int b, hA, hB, q0A, q0B, kt_lo, n_tiles;
};

// Item index -> item, the heaviest first (query tiles from the end of the
// sequence, where the band holds the most key tiles).
//   Even GQA group: A and B are the same query tile of the two query heads
//   2p, 2p + 1 of a group (same kv head, same band).
//   Odd group (e.g. plain multi-head attention): A and B are the adjacent
//   query tiles 2m + 1 and 2m of one head; they share the kv head, and the K/V
//   stream is the union of their bands (a tile outside one of them is fully
//   masked for that tile's rows; A may lie past the end of the sequence).
__host__ __device__ __forceinline__ PerItem per_decode(int w, const FwdPerParams& p, const Band& band) {
  PerItem it;
  int lo = 0, hi = -1;
  if (p.pair_heads) {
    const int npair = p.Hq / 2;
    const int per_q = p.B * npair;
    const int qt = p.n_qtiles - 1 - w / per_q;
    const int rest = w % per_q;
    it.b = rest / npair;
    it.hA = 2 * (rest % npair);
    it.hB = it.hA + 1;
    it.q0A = it.q0B = qt * kBM;
    kv_tile_range(band, it.q0A, kBM, kBN, lo, hi);
  } else {
    const int per_q = p.B * p.Hq;
    const int m = (p.n_qtiles + 1) / 2 - 1 - w / per_q;
    const int rest = w % per_q;
    it.b = rest / p.Hq;
    it.hA = it.hB = rest % p.Hq;
    it.q0B = 2 * m * kBM;
    it.q0A = it.q0B + kBM;
    int lo2 = 0, hi2 = -1;
    kv_tile_range(band, it.q0B, kBM, kBN, lo, hi);
    if (it.q0A < p.T && kv_tile_range(band, it.q0A, kBM, kBN, lo2, hi2)) {
      if (lo2 < lo) lo = lo2;
      if (hi2 > hi) hi = hi2;
    }
  }
  it.kt_lo = lo;
  it.n_tiles = hi - lo + 1;
  return it;
}

template <int D, bool kPolled>
__global__ void __launch_bounds__(kPerThreads, 1)
    fwd_tc_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                          const FwdPerParams prm, const __grid_constant__ FwdSched sched) {
  using L = FwdPerSmem<D>;
  constexpr int KCH = D / 64;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {   // swizzle atoms need 1024-byte aligned tiles (uniform over the CTA)
    if (threadIdx.x == 0) atomicOr(prm.status, DEV_ERR_BOUNDS);
    return;
  }
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(smem + L::kBar + QP_COUNT * 8);
  uint32_t* abort_flag = tmem_base_sh + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
  const int Gq = prm.Hq / prm.Hkv;
  const Band band{prm.T, prm.window, prm.causal};
  const WaitCtl<kPolled> ctl{abort_flag, prm.status, prm.wait_limit_ns};
  auto bar = [&](int i) { return sbase + L::kBar + 8u * static_cast<uint32_t>(i); };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(QP_QFULL), 1);
    mbar_init(bar(QP_QEMPTY), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(QP_KFULL + s), 1);
      mbar_init(bar(QP_KEMPTY + s), 1);
      mbar_init(bar(QP_VFULL + s), 1);
      mbar_init(bar(QP_VEMPTY + s), 1);
      mbar_init(bar(QP_SFULL + s), 1);
      mbar_init(bar(QP_PFULL + s), 4);
      mbar_init(bar(QP_PV + s), 1);
      mbar_init(bar(QP_OFREE + s), 4);
    }
    mbar_init(bar(QP_FINAL), 1);
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_base_sh), 512);
    tmem_relinquish();
  }
  if (prm.dq_acc != nullptr && threadIdx.x < L::kZeroBytes / 16) {
    reinterpret_cast<uint4*>(smem + L::kZero)[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
    fence_async_smem();   // visible to the bulk copies that read it
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_sh;

  if (warp >= 8) {
    setmaxnreg_dec<kPerRegsOther>();
    const uint32_t one = (lane == 0);   // the lane that issues in warp-wide loops
    if (warp == 8) {
      // ---------------- TMA producer (whole warp, lane 0 issues) ----------------
      if (one) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
      }
      bool ok = true;
      int g = 0, it = 0;
      int last_k[2] = {-1, -1}, last_v[2] = {-1, -1};
      for (int k = 0; ok; ++k) {
        const int w = per_item(sched, k, cta, G, prm.n_items);
        if (w < 0) break;
        const PerItem I = per_decode(w, prm, band);
        if (I.n_tiles <= 0) continue;
        const int hk = I.hA / Gq;
        // Q of this item: the previous item's S products have completed
        if (it > 0 && !(ok = mbar_wait_warp(bar(QP_QEMPTY), (it - 1) & 1, ctl))) break;
        mbar_arrive_expect_tx_w(bar(QP_QFULL), 2 * L::kTile, one);
        for (int c = 0; c < KCH; ++c) {
          tma_load_4d_w(sbase + L::kQA + c * L::kHalf, &tmQ, bar(QP_QFULL), 64 * c, I.q0A, I.hA, I.b, one);
          tma_load_4d_w(sbase + L::kQB + c * L::kHalf, &tmQ, bar(QP_QFULL), 64 * c, I.q0B, I.hB, I.b, one);
        }
        for (int j = 0; j < I.n_tiles && ok; ++j, ++g) {
          const int s = g & 1;
          const int k0 = (I.kt_lo + j) * kBN;
          if (g >= 2) ok = mbar_wait_warp(bar(QP_KEMPTY + s), ((g >> 1) - 1) & 1, ctl);
          if (!ok) break;
          mbar_arrive_expect_tx_w(bar(QP_KFULL + s), L::kTile, one);
          for (int c = 0; c < KCH; ++c)
            tma_load_4d_w(sbase + L::kK0 + s * L::kTile + c * L::kHalf, &tmK, bar(QP_KFULL + s), 64 * c,
                          k0, hk, I.b, one);
          last_k[s] = g;
          if (g >= 2) ok = mbar_wait_warp(bar(QP_VEMPTY + s), ((g >> 1) - 1) & 1, ctl);
          if (!ok) break;
          mbar_arrive_expect_tx_w(bar(QP_VFULL + s), L::kTile, one);
          for (int c = 0; c < KCH; ++c)
            tma_load_4d_w(sbase + L::kV0 + s * L::kTile + c * L::kHalf, &tmV, bar(QP_VFULL + s), 64 * c,
                          k0, hk, I.b, one);
          last_v[s] = g;
          if (prm.dq_acc != nullptr && one) {
            // A share of the item's rows of the backward's dQ accumulator
            // (per head one contiguous run of up to 128 rows of D floats),
            // spread over its key tiles, as bulk copies of the zero block.
            int nr[2];
            uint32_t run[2];
            int per[2];
            for (int x = 0; x < 2; ++x) {
              const int q0x = x ? I.q0B : I.q0A;
              nr[x] = prm.T - q0x < kBM ? prm.T - q0x : kBM;
              if (nr[x] < 0) nr[x] = 0;
              run[x] = static_cast<uint32_t>(nr[x]) * D * 4;
              per[x] = static_cast<int>((run[x] + L::kZeroBytes - 1) / L::kZeroBytes);
            }
            const int total = per[0] + per[1];
            const int c1 = (j + 1) * total / I.n_tiles;
            for (int cpy = j * total / I.n_tiles; cpy < c1; ++cpy) {
              const int x = cpy < per[0] ? 0 : 1;
              const uint32_t off = static_cast<uint32_t>(cpy - (x ? per[0] : 0)) * L::kZeroBytes;
              const uint32_t bytes = run[x] - off < static_cast<uint32_t>(L::kZeroBytes) ? run[x] - off
                                                                                         : L::kZeroBytes;
              const int hx = x ? I.hB : I.hA, q0x = x ? I.q0B : I.q0A;
              float* dst = prm.dq_acc + ((static_cast<long long>(I.b) * prm.Hq + hx) * prm.T + q0x) * D;
              bulk_store(reinterpret_cast<uint8_t*>(dst) + off, sbase + L::kZero, bytes);
            }
            bulk_commit_group();
          }
        }
        ++it;
      }
      if (it > 0) mbar_wait_drain(bar(QP_QFULL), (it - 1) & 1, kDrainLimitNs);
      for (int s = 0; s < 2; ++s) {
        if (last_k[s] >= 0) mbar_wait_drain(bar(QP_KFULL + s), (last_k[s] >> 1) & 1, kDrainLimitNs);
        if (last_v[s] >= 0) mbar_wait_drain(bar(QP_VFULL + s), (last_v[s] >> 1) & 1, kDrainLimitNs);
      }
      if (one) bulk_wait_group_all();   // the zero-block copies have finished
    } else if (warp == 9) {
      // ---------------- MMA issuer (whole warp, lane 0 issues) ----------------
      constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, 0, 0);
      constexpr uint32_t idO = idesc_bf16_f32(kBM, D, 0, 1);
      const uint64_t dQ0 = sdesc_sw128(sbase + L::kQA, 16, 1024);
      const uint64_t dK0 = sdesc_sw128(sbase + L::kK0, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(sbase + L::kV0, L::kHalf, 1024);
      auto issue_s = [&](int X, int g) {
        const uint64_t qd = sdesc_add(dQ0, X * L::kTile), kd = sdesc_add(dK0, (g & 1) * L::kTile);
        const uint32_t dst = tmem + X * 128;
        static_for<0, D / 16>([&](auto kc) {
          constexpr int kk = decltype(kc)::value;
          constexpr uint32_t off = ((kk >> 2) * L::kHalf + (kk & 3) * 32) >> 4;
          umma_ss_imm<idS, off, off>(dst, qd, kd, kk > 0 ? 1u : 0u, one);
        });
        umma_commit_w(bar(QP_SFULL + X), one);
      };
      auto issue_pv = [&](int X, int g, bool first) {
        const uint64_t vd = sdesc_add(dV0, (g & 1) * L::kTile);
        const uint32_t dst = tmem + 256 + X * D, pa = tmem + X * 128;
        umma_ts_imm<idO, 0, 0>(dst, pa, vd, first ? 0u : 1u, one);
        static_for<1, kBN / 16>([&](auto kc) {
          constexpr int kk = decltype(kc)::value;
          umma_ts_imm<idO, kk * 8, kk * 2048 / 16>(dst, pa, vd, 1u, one);
        });
        umma_commit_w(bar(QP_PV + X), one);
      };
      bool ok = true;
      int g = 0, it = 0;
      for (int k = 0; ok; ++k) {
        const int w = per_item(sched, k, cta, G, prm.n_items);
        if (w < 0) break;
        const PerItem I = per_decode(w, prm, band);
        const int n = I.n_tiles;
        if (n <= 0) continue;
        const int g0 = g;
        // a warpgroup's first PV of the item overwrites its O: wait until the
        // previous item's O was read out
        auto wait_ofree = [&](int X) {
          return it == 0 || mbar_wait_warp(bar(QP_OFREE + X), (it - 1) & 1, ctl);
        };
        ok = mbar_wait_warp(bar(QP_QFULL), it & 1, ctl) &&
             mbar_wait_warp(bar(QP_KFULL + (g0 & 1)), (g0 >> 1) & 1, ctl);
        if (!ok) break;
        tc_fence_after();
        issue_s(0, g0);
        issue_s(1, g0);
        umma_commit_w(bar(QP_KEMPTY + (g0 & 1)), one);
        for (int j = 1; j < n && ok; ++j) {
          const int gj = g0 + j, gp = gj - 1;
          const bool ready = __all_sync(0xffffffffu, mbar_test3(bar(QP_KFULL + (gj & 1)), (gj >> 1) & 1,
                                                                  bar(QP_PFULL + 0), gp & 1,
                                                                  bar(QP_VFULL + (gp & 1)), (gp >> 1) & 1) != 0);
          ok = (ready || (mbar_wait_warp(bar(QP_KFULL + (gj & 1)), (gj >> 1) & 1, ctl) &&
                          mbar_wait_warp(bar(QP_PFULL + 0), gp & 1, ctl) &&
                          mbar_wait_warp(bar(QP_VFULL + (gp & 1)), (gp >> 1) & 1, ctl))) &&
               (j > 1 || wait_ofree(0));
          if (!ok) break;
          tc_fence_after();
          issue_pv(0, gp, j == 1);
          issue_s(0, gj);
          if (!(ok = mbar_wait_warp(bar(QP_PFULL + 1), gp & 1, ctl) && (j > 1 || wait_ofree(1)))) break;
          tc_fence_after();
          issue_pv(1, gp, j == 1);
          umma_commit_w(bar(QP_VEMPTY + (gp & 1)), one);
          issue_s(1, gj);
          umma_commit_w(bar(QP_KEMPTY + (gj & 1)), one);
        }
        if (!ok) break;
        // every S product of the item is issued: Q is free once they complete
        umma_commit_w(bar(QP_QEMPTY), one);
        const int gl = g0 + n - 1;
        ok = mbar_wait_warp(bar(QP_PFULL + 0), gl & 1, ctl) &&
             mbar_wait_warp(bar(QP_VFULL + (gl & 1)), (gl >> 1) & 1, ctl) && (n > 1 || wait_ofree(0));
        if (!ok) break;
        tc_fence_after();
        issue_pv(0, gl, n == 1);
        if (!(ok = mbar_wait_warp(bar(QP_PFULL + 1), gl & 1, ctl) && (n > 1 || wait_ofree(1)))) break;
        tc_fence_after();
        issue_pv(1, gl, n == 1);
        umma_commit_w(bar(QP_VEMPTY + (gl & 1)), one);
        g += n;
        ++it;
      }
      umma_commit_w(bar(QP_FINAL), one);
      mbar_wait_drain(bar(QP_FINAL), 0, kDrainLimitNs);
    }
  } else {
    // ---------------- softmax warpgroups (A: warps 0-3, B: warps 4-7) ----------------
    setmaxnreg_inc<kPerRegsSoftmax>();
    const int X = warp >> 2;
    const int row = threadIdx.x & 127;        // TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + X * 128 + lane_off;
    const uint32_t tO = tmem + 256 + X * D + lane_off;
    const uint32_t sOut = sbase + L::kO0 + X * L::kHalf;   // this warpgroup's staging half
    const bool leader = (row == 0);
    const float c = prm.scale_log2;
    bool ok = true;
    int g = 0, it = 0;
    for (int k = 0; ok; ++k) {
      const int w = per_item(sched, k, cta, G, prm.n_items);
      if (w < 0) break;
      const PerItem I = per_decode(w, prm, band);
      const int n = I.n_tiles;
      if (n <= 0) continue;
      const int h = X ? I.hB : I.hA;
      const int q0 = X ? I.q0B : I.q0A;
      const int i = q0 + row;                 // query position
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n && ok; ++j) {
        const int gj = g + j;
        const int k0 = (I.kt_lo + j) * kBN;
        ok = mbar_wait_warp(bar(QP_SFULL + X), gj & 1, ctl);
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
        uint32_t sr[4][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + cc * 32, sr[cc]);
        tmem_wait_ld(sr[0]);
        reg_fence(sr[1]);
        reg_fence(sr[2]);
        reg_fence(sr[3]);
        if (!full) {
          // visible iff clo <= col <= chi: one unsigned compare per column
          // (an empty span masks every column)
          const unsigned lo = chi < clo ? static_cast<unsigned>(kBN) : static_cast<unsigned>(clo);
          const unsigned span = chi < clo ? 0u : static_cast<unsigned>(chi - clo);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const unsigned col = static_cast<unsigned>(cc * 32 + e);
              if (col - lo > span) sr[cc][e] = __float_as_uint(-INFINITY);
            }
        }
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
        // PV_X of the previous tile has completed: the commit that signalled
        // this S covers it (only within the item: O is not rescaled at j = 0).
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
          for (int w2 = 0; w2 < 32; ++w2) {
            const int cc = half * 2 + (w2 >> 4), e = (w2 & 15) * 2;
            float x0, x1;
            ffma2(x0, x1, __uint_as_float(sr[cc][e]), __uint_as_float(sr[cc][e + 1]), c, c, nm, nm);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            fadd2_acc(ls[2 * (w2 & 3)], ls[2 * (w2 & 3) + 1], p0, p1);
            pk[w2] = pack_bf16x2(p0, p1);
          }
          tmem_st32(tS + half * 32, pk);
        }
        l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(QP_PFULL + X));
      }
      // The four warps leave together (a wait that gave up raised the CTA's
      // abort flag, so every other wait gives up too) before the named
      // barriers of the epilogue.
      ok = named_bar_and(1 + X, 128, ok);
      if (!ok) break;
      // ---- epilogue: O / l (from TMEM, then O may be overwritten), LSE ----
      const int gl = g + n - 1;
      ok = named_bar_and(1 + X, 128, mbar_wait_warp(bar(QP_PV + X), gl & 1, ctl));
      if (!ok) break;
      tc_fence_after();
      const bool empty = !(l > 0.f);
      const float inv = empty ? 0.f : 1.0f / l;
      uint32_t orr[D / 32][32];
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) tmem_ld32(tO + cc * 32, orr[cc]);
      tmem_wait_ld(orr[0]);
#pragma unroll
      for (int cc = 1; cc < D / 32; ++cc) reg_fence(orr[cc]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(QP_OFREE + X));
      if (i < prm.T) {
        prm.lse[(static_cast<long long>(I.b) * prm.Hq + h) * prm.T + i] =
            empty ? -INFINITY : (m + log2f(l)) * 0.69314718055994531f;
      }
      // bf16 O through this warpgroup's 64-column staging half, one TMA store
      // of 128 rows x 64 columns per round (none for a tile past the end).
#pragma unroll
      for (int r = 0; r < KCH && q0 < prm.T; ++r) {
        if (leader) bulk_wait_group_read<0>();   // the previous store has read the half
        named_bar_sync(1 + X, 128);
#pragma unroll
        for (int cc = 2 * r; cc < 2 * r + 2; ++cc)
#pragma unroll
          for (int e = 0; e < 32; e += 8)
            st_shared_v4(sw128_addr(sOut, kBM, row, (cc * 32 + e - 64 * r) / 8),
                         pack_bf16x2(__uint_as_float(orr[cc][e + 0]) * inv, __uint_as_float(orr[cc][e + 1]) * inv),
                         pack_bf16x2(__uint_as_float(orr[cc][e + 2]) * inv, __uint_as_float(orr[cc][e + 3]) * inv),
                         pack_bf16x2(__uint_as_float(orr[cc][e + 4]) * inv, __uint_as_float(orr[cc][e + 5]) * inv),
                         pack_bf16x2(__uint_as_float(orr[cc][e + 6]) * inv, __uint_as_float(orr[cc][e + 7]) * inv));
        fence_async_smem();
        named_bar_sync(1 + X, 128);
        if (leader) {
          tma_store_4d(&tmO, sOut, 64 * r, q0, h, I.b);
          bulk_commit_group();
        }
      }
      g += n;
      ++it;
    }
    if (leader) bulk_wait_group_all();
    if (cta == 0 && threadIdx.x == 0 && prm.acc_flag != nullptr) {
      // a forward that did not zero the accumulator may have overwritten it
      prm.acc_flag[0] = prm.acc_off;
      prm.acc_flag[1] = (ok && prm.dq_acc != nullptr) ? prm.acc_len : 0ull;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// The item table of a launch: each item (in index order, heaviest first)
// onto the CTA with the least work so far; work = key tiles x 5 + 7 (a key
// tile pair against the fixed cost of an item: its first S, epilogue and
// hand-over, measured at about 1.4 tile pairs). Kept for the next call with
// the same shape (one per host thread).
inline const FwdSched& fwd_schedule(const FwdPerParams& p, int grid) {
  thread_local FwdSched s;
  thread_local long long key[9] = {-1};
  const long long k[9] = {p.B, p.T, p.Hq, p.Hkv, p.window, p.causal, p.pair_heads, p.n_items, grid};
  bool same = true;
  for (int i = 0; i < 9; ++i) same = same && key[i] == k[i];
  if (same) return s;
  for (int i = 0; i < 9; ++i) key[i] = k[i];
  s.n = 0;
  if (p.n_items > kPerMaxItems || grid > kPerMaxCtas) return s;
  const Band band{p.T, p.window, p.causal};
  std::vector<int> owner(p.n_items), count(grid, 0);
  std::vector<std::pair<long long, int>> heap;   // min-heap of (work, cta)
  for (int c = 0; c < grid; ++c) heap.push_back({0, c});
  auto cmp = [](const std::pair<long long, int>& a, const std::pair<long long, int>& b) { return a > b; };
  std::make_heap(heap.begin(), heap.end(), cmp);
  for (int w = 0; w < p.n_items; ++w) {
    const PerItem I = per_decode(w, p, band);
    std::pop_heap(heap.begin(), heap.end(), cmp);
    owner[w] = heap.back().second;
    heap.back().first += I.n_tiles > 0 ? 5LL * I.n_tiles + 7 : 0;
    ++count[owner[w]];
    std::push_heap(heap.begin(), heap.end(), cmp);
  }
  s.off[0] = 0;
  for (int c = 0; c < grid; ++c) s.off[c + 1] = static_cast<uint16_t>(s.off[c] + count[c]);
  std::vector<int> fill(s.off, s.off + grid);
  for (int w = 0; w < p.n_items; ++w) s.item[fill[owner[w]]++] = static_cast<uint16_t>(w);
  s.n = p.n_items;
  return s;
}

template <int D>
inline swa_status launch_fwd_persist_d(const FwdLaunch& f, cudaStream_t st) {
  using L = FwdPerSmem<D>;
  CUtensorMap mq, mk, mv, mo;
  if (!map_head_major(&mq, f.qn, f.B, f.Hq, f.T, D) || !map_head_major(&mk, f.kn, f.B, f.Hkv, f.T, D) ||
      !map_token_major(&mo, f.o, f.B, f.Hq, f.T, D))
    return SWA_ERR_CUDA;
  const bool okv = f.v_head_major ? map_head_major(&mv, f.v, f.B, f.Hkv, f.T, D)
                                  : map_token_major(&mv, f.v, f.B, f.Hkv, f.T, D);
  if (!okv) return SWA_ERR_CUDA;
  FwdPerParams p{};
  p.B = f.B; p.T = f.T; p.Hq = f.Hq; p.Hkv = f.Hkv; p.window = f.window; p.causal = f.causal;
  p.n_qtiles = (f.T + kBM - 1) / kBM;
  p.pair_heads = (f.Hq / f.Hkv) % 2 == 0;
  p.n_items = p.pair_heads ? f.B * (f.Hq / 2) * p.n_qtiles : f.B * f.Hq * ((p.n_qtiles + 1) / 2);
  p.scale_log2 = f.scale * 1.4426950408889634f;
  p.lse = f.lse; p.status = f.status; p.wait_limit_ns = f.wait_limit_ns;
  p.dq_acc = f.dq_acc; p.acc_flag = f.acc_flag;
  p.acc_off = f.acc_off; p.acc_len = f.acc_len;
  const int grid = p.n_items < num_sms() ? p.n_items : num_sms();
  const FwdSched& sched = fwd_schedule(p, grid);
  auto launch = [&](auto kern) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes) != cudaSuccess)
      return SWA_ERR_CUDA;
    kern<<<grid, kPerThreads, L::kBytes, st>>>(mq, mk, mv, mo, p, sched);
    return cudaGetLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
  };
  return p.wait_limit_ns < kPollBelowNs ? launch(fwd_tc_persist_kernel<D, true>)
                                        : launch(fwd_tc_persist_kernel<D, false>);
}

// Forward dispatch: the persistent kernel for every group size (even groups
// pair two query heads per item, odd groups two query tiles of one head).
inline swa_status launch_fwd_any2(const FwdLaunch& f, cudaStream_t st) {
  return f.d == 64 ? launch_fwd_persist_d<64>(f, st) : launch_fwd_persist_d<128>(f, st);
}

}  // namespace tc
}  // namespace swa
