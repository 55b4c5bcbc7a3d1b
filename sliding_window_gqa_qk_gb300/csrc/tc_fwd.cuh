// Forward attention core on the 5th-generation tensor cores (sm_103a).
//
// One CTA computes one 128-row query tile of one (batch, query head):
//   warp 4      TMA producer: the Q tile once, then K and V tiles of the band
//               (two stages each), 128-byte-swizzled boxes of 64 columns;
//   warp 5      MMA issuer (one thread) and TMEM owner:
//               S_j = Q K_j^T into one of two S accumulators in TMEM,
//               O  += P_j V_j into the O accumulator in TMEM;
//   warps 0-3   softmax: thread t owns query row t (TMEM lane t). It reads its
//               row of S_j, masks it when the tile is partial, keeps the
//               running row maximum m and sum l, writes P_j = exp2(S_j c - m)
//               as bf16 into shared memory, rescales its O row only when the
//               maximum grew by more than 2^8 (the result is exact either way:
//               the final division uses the same m), and at the end writes
//               O / l and LSE = (m + log2 l) ln 2.
// Key tiles entirely outside the causal / sliding band are never loaded;
// tiles entirely inside it are not masked (the band schedule of common.cuh).
//
// The method: QK-norm'd queries and keys (prologue), grouped-query attention
// with kv head h / G, causal sliding-window or full causal mask per layer
// (autoresearch train.py walkthrough post, model paragraph; autoresearch
// Administrator & Developer Guide §8.2.1 and §6.3).
#pragma once

#include <cudaTypedefs.h>

#include "../../include/swa_attn.h"
#include "common.cuh"

namespace swa {
namespace tc {

constexpr int kBM = 128;          // query rows per CTA
constexpr int kBN = 128;          // keys per tile
constexpr int kFwdThreads = 192;  // 6 warps
constexpr float kRescaleLog2 = 8.0f;

struct FwdLaunch {
  int B, T, Hq, Hkv, d, window, causal;
  float scale;
  const elem_t* qn;  // [B, Hq, T, d]
  const elem_t* kn;  // [B, Hkv, T, d]
  const elem_t* v;   // [B, Hkv, T, d] (v_head_major) or [B, T, Hkv, d]
  bool v_head_major;
  elem_t* o;         // [B, T, Hq, d]
  float* lse;        // [B, Hq, T]
  uint32_t* status;
  uint64_t wait_limit_ns;
  // Optional (persistent kernel only): fp32 dQ accumulator of the backward
  // [B, Hq, T, d] to zero, and where to record the zeroed byte range.
  float* dq_acc;
  unsigned long long* acc_flag;
  unsigned long long acc_off, acc_len;
};

struct FwdParams {
  int T, Hq, Hkv, window, causal, n_qtiles;
  float scale_log2;  // softmax scale * log2(e)
  elem_t* o;
  float* lse;
  uint32_t* status;
  uint64_t wait_limit_ns;
};

template <int D>
struct FwdSmem {
  static constexpr int kTileBytes = 128 * D * 2;        // 128 rows x D bf16
  static constexpr int kPBytes = kBM * kBN * 2;         // 128 x 128 bf16
  static constexpr int kQ = 0;
  static constexpr int kK0 = kQ + kTileBytes;
  static constexpr int kV0 = kK0 + 2 * kTileBytes;
  static constexpr int kP0 = kV0 + 2 * kTileBytes;
  static constexpr int kBytes = kP0 + 2 * kPBytes;
  static constexpr int kAlloc = kBytes + 1024;          // slack for 1024-byte alignment
  static_assert(kAlloc + 256 <= 232448, "shared memory budget (dynamic + static)");
};

// Barrier indices
enum {
  FB_Q = 0,
  FB_KFULL = 1,   // +stage
  FB_KEMPTY = 3,  // +stage
  FB_VFULL = 5,
  FB_VEMPTY = 7,
  FB_SFULL = 9,   // +buffer
  FB_SFREE = 11,
  FB_PFULL = 13,
  FB_PV = 15,     // +buffer: PV_j completed (j % 2)
  FB_FINAL = 17,
  FB_COUNT = 18
};

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams prm) {
  using L = FwdSmem<D>;
  constexpr int KCH = D / 64;      // 64-column swizzle regions per row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t bars[FB_COUNT];
  __shared__ uint32_t tmem_base_sh;
  __shared__ uint32_t abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // blockIdx.x = b * Hq + h; blockIdx.y walks the query tiles heaviest (most
  // key tiles) first, so that the last CTAs to start are the short ones.
  const int qt = prm.n_qtiles - 1 - static_cast<int>(blockIdx.y);
  const int h = static_cast<int>(blockIdx.x) % prm.Hq, b = static_cast<int>(blockIdx.x) / prm.Hq;
  const int hk = h / (prm.Hq / prm.Hkv);
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
    mbar_init(bar(FB_Q), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(FB_KFULL + s), 1);
      mbar_init(bar(FB_KEMPTY + s), 1);
      mbar_init(bar(FB_VFULL + s), 1);
      mbar_init(bar(FB_VEMPTY + s), 1);
      mbar_init(bar(FB_SFULL + s), 1);
      mbar_init(bar(FB_SFREE + s), 4);
      mbar_init(bar(FB_PFULL + s), 4);
      mbar_init(bar(FB_PV + s), 1);
    }
    mbar_init(bar(FB_FINAL), 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t tS = tmem;          // S buffers: columns [0,128) and [128,256)
  const uint32_t tO = tmem + 256;    // O: columns [256, 256 + D)

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(bar(FB_Q), L::kTileBytes);
      for (int c = 0; c < KCH; ++c)
        tma_load_4d(sbase + L::kQ + c * 16384, &tmQ, bar(FB_Q), 64 * c, q0, h, b);
      bool ok = true;
      int last_k[2] = {-1, -1}, last_v[2] = {-1, -1};
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int s = j & 1;
        const int k0 = (kt_lo + j) * kBN;
        if (j >= 2) ok = mbar_wait(bar(FB_KEMPTY + s), ((j - 2) >> 1) & 1, ctl);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(FB_KFULL + s), L::kTileBytes);
        for (int c = 0; c < KCH; ++c)
          tma_load_4d(sbase + L::kK0 + s * L::kTileBytes + c * 16384, &tmK, bar(FB_KFULL + s),
                      64 * c, k0, hk, b);
        last_k[s] = j;
        if (j >= 2) ok = mbar_wait(bar(FB_VEMPTY + s), ((j - 2) >> 1) & 1, ctl);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(FB_VFULL + s), L::kTileBytes);
        for (int c = 0; c < KCH; ++c)
          tma_load_4d(sbase + L::kV0 + s * L::kTileBytes + c * 16384, &tmV, bar(FB_VFULL + s),
                      64 * c, k0, hk, b);
        last_v[s] = j;
      }
      // Let every copy this thread started land before the CTA can exit.
      mbar_wait_drain(bar(FB_Q), 0, prm.wait_limit_ns);
      for (int s = 0; s < 2; ++s) {
        if (last_k[s] >= 0) mbar_wait_drain(bar(FB_KFULL + s), (last_k[s] >> 1) & 1, prm.wait_limit_ns);
        if (last_v[s] >= 0) mbar_wait_drain(bar(FB_VFULL + s), (last_v[s] >> 1) & 1, prm.wait_limit_ns);
      }
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, 0, 0);
      constexpr uint32_t idO = idesc_bf16_f32(kBM, D, 0, 1);
      bool ok = mbar_wait(bar(FB_Q), 0, ctl);
      auto issue_pv = [&](int j) -> bool {
        const int s = j & 1;
        if (!mbar_wait(bar(FB_PFULL + s), (j >> 1) & 1, ctl)) return false;
        if (!mbar_wait(bar(FB_VFULL + s), (j >> 1) & 1, ctl)) return false;
        tc_fence_after();
        const uint32_t pa = sbase + L::kP0 + s * L::kPBytes;
        const uint32_t va = sbase + L::kV0 + s * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(pa + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(va + kk * 2048, 16384, 1024);
          umma_bf16_ss(tO, ad, bd, idO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(FB_PV + s));
        umma_commit(bar(FB_VEMPTY + s));
        return true;
      };
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int s = j & 1;
        ok = mbar_wait(bar(FB_KFULL + s), (j >> 1) & 1, ctl);
        if (ok && j >= 2) ok = mbar_wait(bar(FB_SFREE + s), ((j - 2) >> 1) & 1, ctl);
        if (!ok) break;
        tc_fence_after();
        const uint32_t qa = sbase + L::kQ;
        const uint32_t ka = sbase + L::kK0 + s * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_bf16_ss(tS + s * 128, sdesc_sw128(qa + off, 16, 1024),
                       sdesc_sw128(ka + off, 16, 1024), idS, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(FB_SFULL + s));
        umma_commit(bar(FB_KEMPTY + s));
        if (j >= 1) ok = issue_pv(j - 1);
      }
      if (ok) issue_pv(n_tiles - 1);
      // Every MMA of this CTA has completed once FB_FINAL fires.
      umma_commit(bar(FB_FINAL));
      mbar_wait_drain(bar(FB_FINAL), 0, prm.wait_limit_ns);
    }
  } else {
    // ---------------- softmax warpgroup (warps 0-3) ----------------
    const int row = threadIdx.x;              // 0..127 = TMEM lane
    const int i = q0 + row;                   // query position
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float c = prm.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = n_tiles > 0;
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int s = j & 1;
      const int k0 = (kt_lo + j) * kBN;
      ok = mbar_wait(bar(FB_SFULL + s), (j >> 1) & 1, ctl);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + s * 128 + lane_off + cc * 32, sr[cc]);
      tmem_wait_ld(sr[0]);
      reg_fence(sr[1]);
      reg_fence(sr[2]);
      reg_fence(sr[3]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(FB_SFREE + s));

      // mask partial tiles: keep columns [clo, chi] of this row
      if (!tile_full(band, q0, kBM, k0, kBN)) {
        int clo = 0, chi = kBN - 1;
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
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int col = cc * 32 + e;
            if (col < clo || col > chi) sr[cc][e] = __float_as_uint(-INFINITY);
          }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
#pragma unroll
        for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(sr[cc][e]));
      const float mt = mx * c;   // row max of this tile, log2 units
      // Rescale decision (exact either way, see the header comment).
      float alpha = 1.f;
      bool rescale_o = false;
      if (mt > m + kRescaleLog2 || (m == -INFINITY && mt > -INFINITY)) {
        if (m != -INFINITY) {
          alpha = ex2_approx(m - mt);
          rescale_o = true;
        }
        l *= alpha;
        m = mt;
      }
      if (j >= 1 && __any_sync(0xffffffffu, rescale_o)) {
        // O must hold PV_{j-1} before it is rescaled.
        ok = mbar_wait(bar(FB_PV + ((j - 1) & 1)), ((j - 1) >> 1) & 1, ctl);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t orr[32];
          tmem_ld32(tO + lane_off + cc * 32, orr);
          tmem_wait_ld(orr);
#pragma unroll
          for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
          tmem_st32(tO + lane_off + cc * 32, orr);
        }
        tmem_wait_st();
      }
      // P_j buffer s is free once PV_{j-2} has completed.
      if (j >= 2) {
        ok = mbar_wait(bar(FB_PV + s), ((j - 2) >> 1) & 1, ctl);
        if (!ok) break;
      }
      const float mref = (m == -INFINITY) ? 0.f : m;
      const uint32_t prow = sbase + L::kP0 + s * L::kPBytes + (row >> 3) * 1024 + (row & 7) * 128;
      float lsum = 0.f;
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {   // 16 chunks of 8 keys
        const int cc = ch >> 2, e0 = (ch & 3) * 8;
        float p[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          p[e] = ex2_approx(fmaf(__uint_as_float(sr[cc][e0 + e]), c, -mref));
          lsum += p[e];
        }
        const uint32_t region = (ch >> 3) * 16384;
        const uint32_t chunk = static_cast<uint32_t>((ch & 7) ^ (row & 7)) * 16;
        st_shared_v4(prow + region + chunk, pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]),
                     pack_bf16x2(p[4], p[5]), pack_bf16x2(p[6], p[7]));
      }
      l += lsum;
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(FB_PFULL + s));
    }
    // ---- epilogue: O / l, LSE ----
    if (ok) ok = mbar_wait(bar(FB_PV + ((n_tiles - 1) & 1)), ((n_tiles - 1) >> 1) & 1, ctl);
    if (ok) {
      tc_fence_after();
      const bool empty = !(l > 0.f);
      const float inv = empty ? 0.f : 1.0f / l;
      elem_t* orow = prm.o + ((static_cast<long long>(b) * prm.T + i) * prm.Hq + h) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t orr[32];
        tmem_ld32(tO + lane_off + cc * 32, orr);
        tmem_wait_ld(orr);
        if (i < prm.T) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 pk;
            pk.x = pack_bf16x2(__uint_as_float(orr[e + 0]) * inv, __uint_as_float(orr[e + 1]) * inv);
            pk.y = pack_bf16x2(__uint_as_float(orr[e + 2]) * inv, __uint_as_float(orr[e + 3]) * inv);
            pk.z = pack_bf16x2(__uint_as_float(orr[e + 4]) * inv, __uint_as_float(orr[e + 5]) * inv);
            pk.w = pack_bf16x2(__uint_as_float(orr[e + 6]) * inv, __uint_as_float(orr[e + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + cc * 32 + e) = pk;
          }
        }
      }
      if (i < prm.T) {
        prm.lse[(static_cast<long long>(b) * prm.Hq + h) * prm.T + i] =
            empty ? -INFINITY : (m + log2f(l)) * 0.69314718055994531f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 4-D bf16 tensor map over [B][H][T][d]-indexed data with the given element
// strides of the T, H and B dimensions; boxes of 64 columns x 128 rows with
// the 128-byte swizzle. Rows past T read as zero.
inline bool make_map_4d(CUtensorMap* m, const void* base, int d, int T, int H, int B,
                        long long sT, long long sH, long long sB, int box_rows = 128) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(sT) * 2, static_cast<cuuint64_t>(sH) * 2,
                           static_cast<cuuint64_t>(sB) * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Head-major [B, H, T, d] tensor.
inline bool map_head_major(CUtensorMap* m, const void* base, int B, int H, int T, int d) {
  return make_map_4d(m, base, d, T, H, B, d, static_cast<long long>(T) * d,
                     static_cast<long long>(H) * T * d);
}
// Token-major [B, T, H, d] tensor.
inline bool map_token_major(CUtensorMap* m, const void* base, int B, int H, int T, int d) {
  return make_map_4d(m, base, d, T, H, B, static_cast<long long>(H) * d, d,
                     static_cast<long long>(T) * H * d);
}

template <int D>
inline swa_status launch_fwd_d(const FwdLaunch& f, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!map_head_major(&mq, f.qn, f.B, f.Hq, f.T, D) || !map_head_major(&mk, f.kn, f.B, f.Hkv, f.T, D))
    return SWA_ERR_CUDA;
  const bool okv = f.v_head_major ? map_head_major(&mv, f.v, f.B, f.Hkv, f.T, D)
                                  : map_token_major(&mv, f.v, f.B, f.Hkv, f.T, D);
  if (!okv) return SWA_ERR_CUDA;
  FwdParams p{};
  p.T = f.T; p.Hq = f.Hq; p.Hkv = f.Hkv; p.window = f.window; p.causal = f.causal;
  p.n_qtiles = (f.T + kBM - 1) / kBM;
  p.scale_log2 = f.scale * 1.4426950408889634f;
  p.o = f.o; p.lse = f.lse; p.status = f.status; p.wait_limit_ns = f.wait_limit_ns;
  if (cudaFuncSetAttribute(fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           FwdSmem<D>::kAlloc) != cudaSuccess)
    return SWA_ERR_CUDA;
  dim3 grid(f.B * f.Hq, p.n_qtiles);
  fwd_tc_kernel<D><<<grid, kFwdThreads, FwdSmem<D>::kAlloc, st>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

inline swa_status launch_fwd(const FwdLaunch& f, cudaStream_t st) {
  return f.d == 64 ? launch_fwd_d<64>(f, st) : launch_fwd_d<128>(f, st);
}

}  // namespace tc
}  // namespace swa
