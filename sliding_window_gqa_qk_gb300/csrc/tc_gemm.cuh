// Projection GEMMs of the attention block on the 5th-generation tensor cores
// (sm_103a): D = A B (+ C), bf16 operands, fp32 accumulation in TMEM.
//
// The block (autoresearch Administrator & Developer Guide §8.2.1 model table,
// "Pre-norm + residual"; train.py walkthrough post, model paragraph) runs
// its four bias-free projections c_q, c_k, c_v, c_proj and their gradients
// as GEMMs of three operand layouts:
//   A K-major [M][K] or M-major [K][M];  B K-major [N][K] or N-major [K][N]
// (row-major storage with a row stride). One launch may join
//   - up to three segments along N, each with its own B and its own output
//     (the q, k and v projections of one normed input in one launch), or
//   - up to three segments along K, each with its own A and B (the gradient
//     of the normed input, dq wq + dk wk + dv wv, in one launch),
// and may split K over several CTAs whose fp32 results are added into the
// output (weight gradients, K = B*T).
//
// Persistent kernel, one CTA per SM, 128 x 256 output tiles, K in steps of
// 64 (one 128-byte swizzle atom per operand row):
//   warp 0      TMA producer: per K step an A box of 128 rows and a B box of
//               256 rows (in halves of 128, each from its N segment), four
//               stages of 48 KB;
//   warp 1      MMA issuer (one thread): four M=128 N=256 K=16 products per
//               K step into one of two TMEM accumulators (2 x 256 columns),
//               so the epilogue of a tile overlaps the main loop of the next;
//   warps 4-7   epilogue: thread = output row (TMEM lane); per 128 bytes of
//               output row (64 bf16 or 32 fp32 columns) the warp's 32 rows go
//               from TMEM to registers (the residual C, loaded by TMA into
//               the same buffer, added), into a 128-byte-swizzled staging
//               buffer of 4 KB, and out by one TMA store (or, for split K,
//               one TMA fp32 reduce-add); two buffers per warp.
// The q, k, v projection with the attention's prologue in its epilogue runs
// three stages and two epilogue warpgroups (warps 4-11, one head of the
// tile each): per head row the projection rounded to bf16 (the raw q, k, v
// the backward reads), then for q and k the rotary turn and the QK-norm in
// two passes over the row (sum of squares; scaled rows), the rotary tables
// read transposed (position fastest, one 128-byte line per warp and column)
// and the gains from shared memory; for v the value-embedding mix.
// Ragged M, N and K: TMA reads zeros past the ends and clips its stores at
// them.
#pragma once

#include "rowwise.cuh"
#include "tc_fwd.cuh"

namespace swa {
namespace tc {

constexpr int kGmM = 128, kGmN = 256, kGmK = 64;
constexpr int kGmProdWarp = 0, kGmMmaWarp = 1, kGmEpiWarp0 = 4;

// Shape of a launch: the plain GEMM runs four K stages and one epilogue
// warpgroup; the q, k, v projection with the fused prologue three stages and
// two epilogue warpgroups (one head of the tile each: its epilogue does the
// prologue's work), their staging buffers in the stage it gives up.
template <bool QKV>
struct GmShape {
  static constexpr int kStages = QKV ? 3 : 4;
  static constexpr int kEpiWarps = QKV ? 8 : 4;
  static constexpr int kThreads = 128 + 32 * kEpiWarps;
  static constexpr int kA = kGmM * kGmK * 2;        // 16 KB
  static constexpr int kB = kGmN * kGmK * 2;        // 32 KB
  static constexpr int kStage = kA + kB;
  static constexpr int kStg = 32 * 128;             // epilogue staging: 32 rows x 128 bytes
  static constexpr int oStg = kStages * kStage;     // [epilogue warps][2 buffers]
  static constexpr int oBar = oStg + 2 * kEpiWarps * kStg;   // barriers, TMEM base, abort flag
  static constexpr int oGain = oBar + 256;                    // QK-norm gains gq, gk: fp32 [2][128]
  static constexpr int kBytes = oGain + (QKV ? 1024 : 0);
  static_assert(kBytes <= 232448, "shared memory budget");
};

enum {
  GM_FULL = 0,        // +stage: the stage's boxes landed
  GM_EMPTY = 4,       // +stage: the products that read the stage completed
  GM_ACCFULL = 8,     // +buffer: a tile's accumulator is complete
  GM_ACCEMPTY = 10,   // +buffer: the epilogue read the accumulator (every epilogue warp)
  GM_FINAL = 12,      // every product the MMA thread issued completed
  GM_CLOAD = 13,      // +2 warp + buffer: the residual's box landed in a staging buffer
  GM_COUNT = 21
};

// An output segment along N: columns [n0, n0 + n) of the product go to the
// output tensor map of the segment.
struct GmNSeg {
  int n0, n;
};

// The q, k, v projection's fused prologue (GemmCall::qkv).
struct GmQkv {
  int T, Hq, Hkv, vocab;
  float eps, ve_scale;
  const float* gq; const float* gk;
  const float* rope_t;      // [2][64][T] cos, sin with the position fastest
  float* rstd_q; float* rstd_k;
  const elem_t* ve; const int32_t* tok; const float* gate;
};

struct GmParams {
  int M, N;
  int n_kseg;               // 1..3; segment s has kt_end[s] - kt_begin[s] K steps (A map s, B map s)
  int kt0[4];               // first K step of each K segment (kt0[n_kseg] = total K steps)
  int n_nseg;               // 1..3 (B map of N segment j is j when n_kseg == 1)
  GmNSeg nseg[3];
  int out;
  float beta;               // with a residual (one N segment, bf16 output): D = A B + beta C
  int has_c;
  int n_mt, n_nt, n_split, kt_per_split;
  uint32_t* status;
  uint64_t wait_limit_ns;
  GmQkv qkv;
};

// N segment holding product column n (-1: none; segments are 128-aligned
// except for the end of the last).
__device__ __forceinline__ int gm_nseg_of(const GmParams& p, int n) {
  if (n >= p.N) return -1;
  int s = 0;
  while (s + 1 < p.n_nseg && n >= p.nseg[s + 1].n0) ++s;
  return s;
}

template <bool AMN, bool BMN, bool QKV>
__global__ void __launch_bounds__(GmShape<QKV>::kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                   const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2,
                   const __grid_constant__ CUtensorMap tmD0, const __grid_constant__ CUtensorMap tmD1,
                   const __grid_constant__ CUtensorMap tmD2, const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmE0, const __grid_constant__ CUtensorMap tmE1,
                   const __grid_constant__ CUtensorMap tmE2, const GmParams prm) {
  using S = GmShape<QKV>;
  constexpr int kGmStages = S::kStages;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {   // swizzle atoms need 1024-byte aligned tiles (uniform over the CTA)
    if (threadIdx.x == 0) atomicOr(prm.status, DEV_ERR_BOUNDS);
    return;
  }
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(smem + S::oBar + GM_COUNT * 8);
  uint32_t* abort_flag = tmem_base_sh + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitCtl<false> ctl{abort_flag, prm.status, prm.wait_limit_ns};
  auto bar = [&](int i) { return sbase + S::oBar + 8u * static_cast<uint32_t>(i); };
  const int n_items = prm.n_mt * prm.n_nt * prm.n_split;
  const int kt_total = prm.kt0[prm.n_kseg];

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kGmStages; ++s) {
      mbar_init(bar(GM_FULL + s), 1);
      mbar_init(bar(GM_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(GM_ACCFULL + b), 1);
      mbar_init(bar(GM_ACCEMPTY + b), S::kEpiWarps);
    }
    mbar_init(bar(GM_FINAL), 1);
    for (int i = 0; i < 8; ++i) mbar_init(bar(GM_CLOAD + i), 1);
    fence_mbar_init();
  }
  if constexpr (QKV) {   // the gains (1 where absent), read by every row of every q / k head
    float* gs = reinterpret_cast<float*>(smem + S::oGain);
    for (int i = threadIdx.x; i < 256; i += blockDim.x) {
      const float* g = i < 128 ? prm.qkv.gq : prm.qkv.gk;
      gs[i] = g ? g[i & 127] : 1.f;
    }
  }
  if (warp == kGmMmaWarp) {
    tmem_alloc(smem_u32(tmem_base_sh), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_sh;

  // item -> (split, m tile, n tile), n fastest: consecutive items share A rows
  auto decode = [&](int w, int& mt, int& nt, int& kb, int& ke) {
    nt = w % prm.n_nt;
    mt = (w / prm.n_nt) % prm.n_mt;
    const int sp = w / (prm.n_nt * prm.n_mt);
    kb = sp * prm.kt_per_split;
    ke = kb + prm.kt_per_split < kt_total ? kb + prm.kt_per_split : kt_total;
  };

  if (warp == kGmProdWarp) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      const CUtensorMap* mA[3] = {&tmA0, &tmA1, &tmA2};
      const CUtensorMap* mB[3] = {&tmB0, &tmB1, &tmB2};
      for (int i = 0; i < 3; ++i) {
        tma_prefetch_desc(mA[i]);
        tma_prefetch_desc(mB[i]);
      }
      uint32_t it = 0;
      int last[kGmStages];
      for (int s2 = 0; s2 < kGmStages; ++s2) last[s2] = -1;
      bool ok = true;
      for (int w = static_cast<int>(blockIdx.x); w < n_items && ok; w += static_cast<int>(gridDim.x)) {
        int mt, nt, kb, ke;
        decode(w, mt, nt, kb, ke);
        const int m0 = mt * kGmM, n0 = nt * kGmN;
        // the N segment of each 128-column half, its first column within the segment
        int hs[2], hn[2];
        for (int h = 0; h < 2; ++h) {
          hs[h] = gm_nseg_of(prm, n0 + 128 * h);
          hn[h] = hs[h] >= 0 ? n0 + 128 * h - prm.nseg[hs[h]].n0 : 0;
        }
        const uint32_t bytes = S::kA + (hs[0] >= 0 ? S::kB / 2 : 0) + (hs[1] >= 0 ? S::kB / 2 : 0);
        int ks = 0;
        for (int kt = kb; kt < ke; ++kt, ++it) {
          while (ks + 1 < prm.n_kseg && kt >= prm.kt0[ks + 1]) ++ks;
          const int kl = (kt - prm.kt0[ks]) * kGmK;   // K offset within the segment
          const uint32_t s = it % kGmStages;
          if (it >= kGmStages && !(ok = mbar_wait(bar(GM_EMPTY + s), ((it / kGmStages) - 1) & 1, ctl))) break;
          last[s] = static_cast<int>(it);
          const uint32_t sA = sbase + s * S::kStage, sB = sA + S::kA;
          mbar_arrive_expect_tx(bar(GM_FULL + s), bytes);
          const CUtensorMap* ma = mA[ks];
          if constexpr (!AMN) {
            tma_load_2d(sA, ma, bar(GM_FULL + s), kl, m0);
          } else {
            tma_load_2d(sA, ma, bar(GM_FULL + s), m0, kl);
            tma_load_2d(sA + S::kA / 2, ma, bar(GM_FULL + s), m0 + 64, kl);
          }
          for (int h = 0; h < 2; ++h) {
            if (hs[h] < 0) continue;
            const CUtensorMap* mb = mB[prm.n_kseg > 1 ? ks : hs[h]];
            const uint32_t dst = sB + h * (S::kB / 2);
            if constexpr (!BMN) {
              tma_load_2d(dst, mb, bar(GM_FULL + s), kl, hn[h]);
            } else {
              tma_load_2d(dst, mb, bar(GM_FULL + s), hn[h], kl);
              tma_load_2d(dst + S::kB / 4, mb, bar(GM_FULL + s), hn[h] + 64, kl);
            }
          }
        }
      }
      // every copy this thread issued lands before the CTA can exit
      for (int s = 0; s < kGmStages; ++s)
        if (last[s] >= 0) mbar_wait_drain(bar(GM_FULL + s), (last[s] / kGmStages) & 1, kDrainLimitNs);
    }
  } else if (warp == kGmMmaWarp) {
    if (lane == 0) {
      // ---------------- MMA issuer (one thread) ----------------
      constexpr uint32_t idesc = idesc_bf16_f32(kGmM, kGmN, AMN ? 1 : 0, BMN ? 1 : 0);
      // K-major: K step kk (16 elements) is 32 bytes into each 128-byte row;
      // MN-major: 16 K rows (2048 bytes) on. MN-major boxes of 64 columns sit
      // 8 KB apart (A: 2, B: 4 per stage).
      const uint64_t dA0 = AMN ? sdesc_sw128(sbase, S::kA / 2, 1024) : sdesc_sw128(sbase, 16, 1024);
      const uint64_t dB0 = BMN ? sdesc_sw128(sbase + S::kA, S::kB / 4, 1024) : sdesc_sw128(sbase + S::kA, 16, 1024);
      uint32_t it = 0;
      int tcount = 0;
      bool ok = true;
      for (int w = static_cast<int>(blockIdx.x); w < n_items && ok; w += static_cast<int>(gridDim.x), ++tcount) {
        int mt, nt, kb, ke;
        decode(w, mt, nt, kb, ke);
        const int buf = tcount & 1;
        if (tcount >= 2 && !(ok = mbar_wait(bar(GM_ACCEMPTY + buf), ((tcount >> 1) - 1) & 1, ctl))) break;
        tc_fence_after();
        const uint32_t acc = tmem + static_cast<uint32_t>(buf * kGmN);
        for (int kt = kb; kt < ke; ++kt, ++it) {
          const uint32_t s = it % kGmStages;
          if (!(ok = mbar_wait(bar(GM_FULL + s), (it / kGmStages) & 1, ctl))) break;
          tc_fence_after();
          const uint64_t da = sdesc_add(dA0, s * S::kStage), db = sdesc_add(dB0, s * S::kStage);
          const uint32_t first = (kt == kb);
          static_for<0, kGmK / 16>([&](auto kc) {
            constexpr int kk = decltype(kc)::value;
            constexpr uint32_t aoff = (AMN ? kk * 2048 : kk * 32) >> 4;
            constexpr uint32_t boff = (BMN ? kk * 2048 : kk * 32) >> 4;
            umma_ss_imm<idesc, aoff, boff>(acc, da, db, (kk > 0 || !first) ? 1u : 0u, 1u);
          });
          umma_commit(bar(GM_EMPTY + s));
        }
        if (!ok) break;
        umma_commit(bar(GM_ACCFULL + buf));
      }
      // every product issued completes before TMEM and shared memory are
      // released (after a timeout too)
      umma_commit(bar(GM_FINAL));
      mbar_wait_drain(bar(GM_FINAL), 0, kDrainLimitNs);
    }
  } else if (QKV && warp >= kGmEpiWarp0) {
    // -------- q, k, v epilogue: thread = row; one 128-column half = one head --------
    // Per head row: the projection rounded to bf16 (stored as the raw q, k
    // or v the backward reads); for q and k the rotary turn (pairs c, c + 64)
    // and the QK-norm of the rounded values, for v on value-embedding layers
    // v + ve_scale * gate * VE[tok]: the prologue kernel's arithmetic.
    const GmQkv& e = prm.qkv;
    const int q = warp & 3;
    const int ew = warp - kGmEpiWarp0;          // epilogue warp 0..7
    const int hsel = ew >> 2;                   // the half (head) of the tile this warpgroup takes
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const CUtensorMap* mD[3] = {&tmD0, &tmD1, &tmD2};
    const CUtensorMap* mE[3] = {&tmE0, &tmE1, &tmE2};
    if (lane == 0)
      for (int i = 0; i < 3; ++i) {
        tma_prefetch_desc(mD[i]);
        tma_prefetch_desc(mE[i]);
      }
    int cnt = 0;
    // 32 rows x 128 bytes (32 words per row) through a staging buffer and
    // one TMA store
    // (stage_open: the next buffer, once its previous store has read it;
    // stage_put: 16 bytes of the lane's row; stage_close: the store)
    auto stage_open = [&]() {
      const int b = cnt & 1;
      if (lane == 0 && cnt >= 2) bulk_wait_group_read<1>();
      __syncwarp();
      return sbase + S::oStg + static_cast<uint32_t>((ew * 2 + b) * S::kStg);
    };
    auto stage_put = [&](uint32_t stg, int j, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
      st_shared_v4(stg + lane * 128 + ((j ^ (lane & 7)) << 4), a, b, c, d);
    };
    auto stage_close = [&](uint32_t stg, const CUtensorMap* map, int x, int y) {
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(map, stg, x, y);
        bulk_commit_group();
      }
      ++cnt;
    };
    auto stage_store = [&](const uint32_t* w32, const CUtensorMap* map, int x, int y) {
      const uint32_t stg = stage_open();
#pragma unroll
      for (int j = 0; j < 8; ++j) stage_put(stg, j, w32[4 * j], w32[4 * j + 1], w32[4 * j + 2], w32[4 * j + 3]);
      stage_close(stg, map, x, y);
    };
    auto lo = [](uint32_t w) { return __uint_as_float(w << 16); };
    auto hi = [](uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); };
    const bool rope = e.rope_t != nullptr;
    int tcount = 0;
    for (int w = static_cast<int>(blockIdx.x); w < n_items; w += static_cast<int>(gridDim.x), ++tcount) {
      int mt, nt, kb, ke;
      decode(w, mt, nt, kb, ke);
      const int buf = tcount & 1;
      const int row0 = mt * kGmM + q * 32;     // the warp's 32 rows: one batch element (T % 32 == 0)
      const int m = row0 + lane;
      const bool valid = m < prm.M;
      const int bb = row0 / e.T, t0 = row0 - bb * e.T, t = t0 + lane;
      const int n0 = nt * kGmN;
      if (!mbar_wait_warp(bar(GM_ACCFULL + buf), (tcount >> 1) & 1, ctl)) break;
      tc_fence_after();
      {
        const int h = hsel;
        const int n = n0 + 128 * h;
        const int sg = gm_nseg_of(prm, n);
        if (sg < 0) {   // uniform: this half is past N; the accumulator's share is free
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(GM_ACCEMPTY + buf));
          continue;
        }
        const int nl = n - prm.nseg[sg].n0;
        const int head = nl >> 7;
        // the VE-table row of a v head: into L2 before the accumulator is
        // read, into registers (a half at a time) once the raw row is stored
        int tok = -1;
        bool tok_ok = false;
        const elem_t* vrow = e.ve;
        if (sg == 2 && e.ve != nullptr) {
          tok = valid ? e.tok[m] : -1;
          tok_ok = tok >= 0 && tok < e.vocab;
          vrow = e.ve + (static_cast<long long>(tok_ok ? tok : 0) * e.Hkv + head) * 128;
          if (tok_ok) bulk_prefetch_l2(vrow, 256);
        }
        uint32_t pk[64];     // the row's 128 values rounded to bf16, in pairs
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t v[32];
          tmem_ld32(tmem + static_cast<uint32_t>(buf * kGmN + 128 * h + 32 * j) + lane_off, v);
          tmem_wait_ld(v);
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[16 * j + i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        }
        // this warp's columns are in registers: its share of the accumulator is free
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(GM_ACCEMPTY + buf));
        stage_store(pk, mD[sg], nl, row0);
        stage_store(pk + 32, mD[sg], nl + 64, row0);
        if (sg < 2) {
          const float* gsm = reinterpret_cast<const float*>(smem + S::oGain) + (sg == 0 ? 0 : 128);
          const int H = sg == 0 ? e.Hq : e.Hkv;
          // column c of the tables for the lane's position: one 128-byte
          // line per warp
          const float* cs = rope ? e.rope_t + (valid ? t : 0) : nullptr;
          const float* sn = rope ? cs + 64LL * e.T : nullptr;
          // the rotated pairs (c, c + 64), c = 8 k .. 8 k + 7, in fp32 from
          // the rounded values; recomputed in the second pass rather than
          // kept (a row of 128 fp32 values does not fit beside the rest)
          auto rotated = [&](int k, float (&xr)[8], float (&yr)[8]) {
            float co[8], si[8];
            if (rope) {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                co[j] = cs[static_cast<long long>(8 * k + j) * e.T];
                si[j] = sn[static_cast<long long>(8 * k + j) * e.T];
              }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int c = 8 * k + j;
              const float x = (c & 1) ? hi(pk[c / 2]) : lo(pk[c / 2]);
              const float y = (c & 1) ? hi(pk[32 + c / 2]) : lo(pk[32 + c / 2]);
              xr[j] = rope ? fmaf(x, co[j], y * si[j]) : x;
              yr[j] = rope ? fmaf(y, co[j], -x * si[j]) : y;
            }
          };
          float ssp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float xr[8], yr[8];
            rotated(k, xr, yr);
#pragma unroll
            for (int j = 0; j < 8; ++j) ssp[j & 3] = fmaf(yr[j], yr[j], fmaf(xr[j], xr[j], ssp[j & 3]));
          }
          const float rstd = rsqrtf(((ssp[0] + ssp[1]) + (ssp[2] + ssp[3])) / 128.f + e.eps);
          if (valid) (sg == 0 ? e.rstd_q : e.rstd_k)[(static_cast<long long>(bb) * H + head) * e.T + t] = rstd;
          const int yrow = (bb * H + head) * e.T + t0;
          // both halves of the normed row (channels 0..63, 64..127) at once,
          // 8 channels of each at a time, into the warp's two buffers
          if (lane == 0) bulk_wait_group_read<0>();
          __syncwarp();
          const uint32_t stg0 = sbase + S::oStg + static_cast<uint32_t>((ew * 2 + (cnt & 1)) * S::kStg);
          const uint32_t stg1 = sbase + S::oStg + static_cast<uint32_t>((ew * 2 + ((cnt + 1) & 1)) * S::kStg);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float xr[8], yr[8];
            rotated(k, xr, yr);
            uint32_t o0[4], o1[4];
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
              const float2 g0 = *reinterpret_cast<const float2*>(gsm + 8 * k + j);
              const float2 g1 = *reinterpret_cast<const float2*>(gsm + 64 + 8 * k + j);
              o0[j / 2] = pack_bf16x2(xr[j] * rstd * g0.x, xr[j + 1] * rstd * g0.y);
              o1[j / 2] = pack_bf16x2(yr[j] * rstd * g1.x, yr[j + 1] * rstd * g1.y);
            }
            stage_put(stg0, k, o0[0], o0[1], o0[2], o0[3]);
            stage_put(stg1, k, o1[0], o1[1], o1[2], o1[3]);
          }
          stage_close(stg0, mE[sg], 0, yrow);
          stage_close(stg1, mE[sg], 64, yrow);
        } else if (e.ve != nullptr) {
          uint4 er[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) er[j] = tok_ok ? ld16(vrow + 8 * j) : make_uint4(0u, 0u, 0u, 0u);
          if (valid && !tok_ok) atomicOr(prm.status, DEV_ERR_TOKEN);   // contributes nothing, reported
          const float sc = tok_ok ? e.ve_scale * (e.gate ? e.gate[static_cast<long long>(m) * e.Hkv + head] : 1.f) : 0.f;
          const int yrow = (bb * e.Hkv + head) * e.T + t0;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint32_t stg = stage_open();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float ev[8];
              unpack16(er[j], ev);
              // the register takes the second half's piece once read
              if (half == 0) er[j] = tok_ok ? ld16(vrow + 64 + 8 * j) : make_uint4(0u, 0u, 0u, 0u);
              uint32_t o[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint32_t w = pk[32 * half + 4 * j + i];
                o[i] = pack_bf16x2(fmaf(sc, ev[2 * i], lo(w)), fmaf(sc, ev[2 * i + 1], hi(w)));
              }
              stage_put(stg, j, o[0], o[1], o[2], o[3]);
            }
            stage_close(stg, mE[2], 64 * half, yrow);
          }
        }
      }
    }
    if (lane == 0) bulk_wait_group_all();   // every store has completed
  } else if (!QKV && warp >= kGmEpiWarp0) {
    // ---------------- epilogue: thread = row (TMEM lane) ----------------
    const int q = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const CUtensorMap* mD[3] = {&tmD0, &tmD1, &tmD2};
    if (lane == 0) {
      for (int i = 0; i < 3; ++i) tma_prefetch_desc(mD[i]);
      if (prm.has_c) tma_prefetch_desc(&tmC);
    }
    const bool bf = prm.out == GEMM_OUT_ELEM;
    const int W = bf ? 64 : 32;               // columns per 128-byte row chunk
    const float beta = prm.beta;
    int cnt = 0;                              // chunks staged by this warp
    int tcount = 0;
    for (int w = static_cast<int>(blockIdx.x); w < n_items; w += static_cast<int>(gridDim.x), ++tcount) {
      int mt, nt, kb, ke;
      decode(w, mt, nt, kb, ke);
      const int buf = tcount & 1;
      if (!mbar_wait_warp(bar(GM_ACCFULL + buf), (tcount >> 1) & 1, ctl)) break;
      tc_fence_after();
      const int row0 = mt * kGmM + q * 32;
      const int n0 = nt * kGmN;
      bool ok = true;
#pragma unroll 1
      for (int cc = 0; cc < kGmN / W; ++cc, ++cnt) {
        const int n = n0 + cc * W;
        const int sg = gm_nseg_of(prm, n);
        if (sg < 0) break;   // uniform: the rest of the tile is past N
        const int nl = n - prm.nseg[sg].n0;
        const int b = cnt & 1;
        const uint32_t stg = sbase + S::oStg + static_cast<uint32_t>((q * 2 + b) * S::kStg);
        // the store issued from this buffer two chunks ago has read it
        if (lane == 0 && cnt >= 2) bulk_wait_group_read<1>();
        __syncwarp();
        if (prm.has_c && lane == 0) {
          mbar_arrive_expect_tx(bar(GM_CLOAD + q * 2 + b), S::kStg);
          tma_load_2d(stg, &tmC, bar(GM_CLOAD + q * 2 + b), nl, row0);
        }
        uint32_t v[2][32];
        const uint32_t tcol = tmem + static_cast<uint32_t>(buf * kGmN + cc * W) + lane_off;
        tmem_ld32(tcol, v[0]);
        if (bf) tmem_ld32(tcol + 32, v[1]);
        tmem_wait_ld(v[0]);
        reg_fence(v[1]);
        uint32_t pk[32];   // this row's 128 bytes as 32 words
        if (bf) {
          float c[64];
          if (prm.has_c) {
            if (!(ok = mbar_wait_warp(bar(GM_CLOAD + q * 2 + b), (cnt >> 1) & 1, ctl))) break;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 raw = ld_shared_v4f(stg + lane * 128 + ((j ^ (lane & 7)) << 4));
              const uint4 u = make_uint4(__float_as_uint(raw.x), __float_as_uint(raw.y), __float_as_uint(raw.z),
                                         __float_as_uint(raw.w));
              float f8[8];
              unpack16(u, f8);
#pragma unroll
              for (int e = 0; e < 8; ++e) c[8 * j + e] = f8[e];
            }
          }
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            float x0 = __uint_as_float(v[e >> 4][(e & 15) * 2]);
            float x1 = __uint_as_float(v[e >> 4][(e & 15) * 2 + 1]);
            if (prm.has_c) {
              x0 = fmaf(beta, c[2 * e], x0);
              x1 = fmaf(beta, c[2 * e + 1], x1);
            }
            pk[e] = pack_bf16x2(x0, x1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) pk[e] = v[0][e];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          st_shared_v4(stg + lane * 128 + ((j ^ (lane & 7)) << 4), pk[4 * j], pk[4 * j + 1], pk[4 * j + 2],
                       pk[4 * j + 3]);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (prm.out == GEMM_OUT_F32_ADD) tma_reduce_add_2d(mD[sg], stg, nl, row0);
          else tma_store_2d(mD[sg], stg, nl, row0);
          bulk_commit_group();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(GM_ACCEMPTY + buf));
      if (!ok) break;
    }
    if (lane == 0) bulk_wait_group_all();   // every store has completed
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kGmMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

// 2-D tensor map of a row-major [outer][inner] matrix (bf16, or fp32 when
// f32) with a row stride of `ld` elements; boxes of 128 bytes of a row (64
// bf16 or 32 fp32) x box_outer rows, 128-byte swizzle; loads read zeros past
// the ends, stores are clipped there.
inline bool map_2d(CUtensorMap* m, const void* base, long long inner, long long outer, long long ld,
                   int box_outer, bool f32 = false) {
  auto fn = encode_fn();
  if (fn == nullptr || inner < 1 || outer < 1) return false;
  const int es_bytes = f32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * es_bytes};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / es_bytes), static_cast<cuuint32_t>(box_outer)};
  cuuint32_t es[2] = {1, 1};
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline swa_status launch_gemm(const GemmCall& g, cudaStream_t st) {
  if (g.M == 0) return SWA_OK;
  if (g.n_kseg < 1 || g.n_kseg > 3 || g.n_nseg < 1 || g.n_nseg > 3 || (g.n_kseg > 1 && g.n_nseg > 1))
    return SWA_ERR_INVALID_ARG;
  GmParams p{};
  p.M = g.M;
  p.n_kseg = g.n_kseg;
  int kt = 0;
  for (int s = 0; s < g.n_kseg; ++s) {
    if (s + 1 < g.n_kseg && g.kseg[s].K % kGmK != 0) return SWA_ERR_INVALID_ARG;
    p.kt0[s] = kt;
    kt += (g.kseg[s].K + kGmK - 1) / kGmK;
  }
  p.kt0[g.n_kseg] = kt;
  int n = 0;
  p.n_nseg = g.n_nseg;
  for (int j = 0; j < g.n_nseg; ++j) {
    if ((j + 1 < g.n_nseg && g.nseg[j].N % 128 != 0) || g.nseg[j].N % 8 != 0) return SWA_ERR_INVALID_ARG;
    p.nseg[j] = GmNSeg{n, g.nseg[j].N};
    n += g.nseg[j].N;
  }
  p.N = n;
  if (n == 0 || kt == 0) return SWA_OK;
  p.n_mt = (g.M + kGmM - 1) / kGmM;
  p.n_nt = (n + kGmN - 1) / kGmN;
  int split = g.out == GEMM_OUT_ELEM ? 1 : (g.split < 1 ? 1 : g.split);
  if (split > kt) split = kt;
  p.kt_per_split = (kt + split - 1) / split;
  p.n_split = (kt + p.kt_per_split - 1) / p.kt_per_split;   // no empty split
  p.out = g.out;
  if (p.out == GEMM_OUT_F32 && p.n_split > 1) p.out = GEMM_OUT_F32_ADD;
  if (p.out == GEMM_OUT_F32_ADD) {
    for (int j = 0; j < g.n_nseg; ++j) {
      const auto& o = g.nseg[j];
      if (cudaMemset2DAsync(o.D, static_cast<size_t>(o.ldd) * 4, 0, static_cast<size_t>(o.N) * 4, g.M, st) !=
          cudaSuccess)
        return SWA_ERR_CUDA;
    }
  }
  p.beta = g.beta;
  p.has_c = (g.out == GEMM_OUT_ELEM && g.beta != 0.f && g.nseg[0].C != nullptr) ? 1 : 0;
  if (p.has_c && g.n_nseg != 1) return SWA_ERR_INVALID_ARG;
  p.status = g.status;
  p.wait_limit_ns = g.wait_limit_ns;
  // tensor maps: A per K segment; B per K segment or per N segment
  CUtensorMap ma[3], mb[3];
  for (int s = 0; s < 3; ++s) {
    const int ss = s < g.n_kseg ? s : 0;
    const auto& a = g.kseg[ss];
    const bool ok = g.a_mn ? map_2d(&ma[s], a.A, g.M, a.K, a.lda, 64) : map_2d(&ma[s], a.A, a.K, g.M, a.lda, 128);
    if (!ok) return SWA_ERR_CUDA;
  }
  for (int s = 0; s < 3; ++s) {
    const bool by_k = g.n_kseg > 1;
    const int ss = s < (by_k ? g.n_kseg : g.n_nseg) ? s : 0;
    const auto& b = g.bseg[ss];
    const int bn = by_k ? n : g.nseg[ss].N;
    const int bk = by_k ? g.kseg[ss].K : g.kseg[0].K;
    const bool ok = g.b_mn ? map_2d(&mb[s], b.B, bn, bk, b.ldb, 64) : map_2d(&mb[s], b.B, bk, bn, b.ldb, 128);
    if (!ok) return SWA_ERR_CUDA;
  }
  // outputs: one map per N segment (32-row boxes of 128 bytes), and the residual
  CUtensorMap md[3], mc;
  const bool f32 = p.out != GEMM_OUT_ELEM;
  for (int j = 0; j < 3; ++j) {
    const auto& o = g.nseg[j < g.n_nseg ? j : 0];
    if (!map_2d(&md[j], o.D, o.N, g.M, o.ldd, 32, f32)) return SWA_ERR_CUDA;
  }
  if (p.has_c) {
    if (!map_2d(&mc, g.nseg[0].C, g.nseg[0].N, g.M, g.nseg[0].ldc, 32)) return SWA_ERR_CUDA;
  } else {
    mc = md[0];
  }
  // the fused prologue's head-major outputs: [B * H * T][128] row views
  CUtensorMap me[3] = {md[0], md[0], md[0]};
  const auto& e = g.qkv;
  if (e.on) {
    if (g.n_nseg != 3 || g.n_kseg != 1 || g.a_mn || g.b_mn || p.out != GEMM_OUT_ELEM || p.has_c || e.T % 32 != 0 ||
        g.M % e.T != 0 || g.nseg[0].N != e.Hq * 128 || g.nseg[1].N != e.Hkv * 128 || g.nseg[2].N != e.Hkv * 128)
      return SWA_ERR_INVALID_ARG;
    const long long rq = static_cast<long long>(g.M) * e.Hq, rk = static_cast<long long>(g.M) * e.Hkv;
    if (!map_2d(&me[0], e.qn, 128, rq, 128, 32) || !map_2d(&me[1], e.kn, 128, rk, 128, 32)) return SWA_ERR_CUDA;
    if (e.ve != nullptr && !map_2d(&me[2], e.veff, 128, rk, 128, 32)) return SWA_ERR_CUDA;
    p.qkv = GmQkv{e.T, e.Hq, e.Hkv, e.vocab, e.eps, e.ve_scale, e.gq, e.gk, e.rope_t, e.rstd_q, e.rstd_k,
                  static_cast<const elem_t*>(e.ve), e.tok, e.gate};
  }
  const int items = p.n_mt * p.n_nt * p.n_split;
  const int grid = items < num_sms() ? items : num_sms();
  auto launch = [&](auto kern, auto shape) {
    using S = decltype(shape);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes) != cudaSuccess)
      return SWA_ERR_CUDA;
    kern<<<grid, S::kThreads, S::kBytes, st>>>(ma[0], ma[1], ma[2], mb[0], mb[1], mb[2], md[0], md[1], md[2],
                                               mc, me[0], me[1], me[2], p);
    return cudaGetLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
  };
  if (e.on) return launch(gemm_tc_kernel<false, false, true>, GmShape<true>{});
  if (!g.a_mn && !g.b_mn) return launch(gemm_tc_kernel<false, false, false>, GmShape<false>{});
  if (!g.a_mn && g.b_mn) return launch(gemm_tc_kernel<false, true, false>, GmShape<false>{});
  if (g.a_mn && g.b_mn) return launch(gemm_tc_kernel<true, true, false>, GmShape<false>{});
  return launch(gemm_tc_kernel<true, false, false>, GmShape<false>{});
}

}  // namespace tc
}  // namespace swa
