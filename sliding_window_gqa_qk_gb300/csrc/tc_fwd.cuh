// Definitions shared by the tcgen05 attention kernels (sm_103a): tile sizes,
// the forward's launch arguments, and the host-side TMA tensor maps of the
// [B][H][T][d]-indexed tensors (128-byte swizzled boxes of 64 columns).
#pragma once

#include <cudaTypedefs.h>

#include "../../include/swa_attn.h"
#include "common.cuh"

namespace swa {
namespace tc {

constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per tile
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

}  // namespace tc
}  // namespace swa
