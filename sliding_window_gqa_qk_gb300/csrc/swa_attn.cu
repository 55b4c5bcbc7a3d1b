// Host side of the C ABI declared in include/swa_attn.h: argument checks,
// workspace layout, TMA descriptor set-up and the kernel launch sequence.
//
// Built twice from this file: with SWA_ELEM_FP32 (fp32 SIMT debug library)
// and without (bf16 tcgen05 library).
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/swa_attn.h"
#include "common.cuh"
#include "rowwise.cuh"
#include "block.cuh"

#if defined(SWA_ELEM_FP32)
#include "simt.cuh"
#else
#include "tc_fwd.cuh"
#include "tc_fwd_persist.cuh"
#include "tc_bwd.cuh"
#include "tc_bwd128.cuh"
#endif

using namespace swa;

namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per pipeline wait (default)

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// Validated view of one call.
struct Call {
  swa_params p;
  bool empty;
  float scale;
  WsLayout L;
  uint8_t* ws;
  cudaStream_t stream;
  const float* rcos = nullptr;   // rotary tables [rows, d/2], NULL: none
  const float* rsin = nullptr;
  const elem_t* gx = nullptr;    // learned VE gate: input rows, weights [Hkv][gch]
  long long gx_stride = 0;
  const float* gw = nullptr;
  int gch = 0;
  float* d_gw = nullptr;         // its gradients (backward outputs, NULL: skip)
  float* d_gx = nullptr;
  uint64_t wait_ns = kWaitLimitNs;   // time limit of one pipeline wait
};

// Extras of a call. Rotary: none (both tables NULL), or both tables, 16-byte
// aligned, with at least T rows. Learned gate: gate_w NULL (none), or
// gate_x and gate_w set, 1 <= gate_ch <= 32, gate_x_stride >= gate_ch,
// Hkv <= 32, and no ve_gate argument.
constexpr int kMaxGateCh = 32, kMaxGateHeads = 32;
swa_status set_extras(Call& c, const swa_extras* e, const float* ve_gate) {
  if (e == nullptr) return SWA_OK;
  if (e->wait_limit_ns != 0) c.wait_ns = e->wait_limit_ns;
  if (e->rope_cos != nullptr || e->rope_sin != nullptr) {
    if (e->rope_cos == nullptr || e->rope_sin == nullptr || !aligned(e->rope_cos, 16) ||
        !aligned(e->rope_sin, 16) || e->rope_rows < c.p.T)
      return SWA_ERR_INVALID_ARG;
    c.rcos = e->rope_cos;
    c.rsin = e->rope_sin;
  }
  if (e->gate_w != nullptr) {
    if (e->gate_x == nullptr || e->gate_ch < 1 || e->gate_ch > kMaxGateCh ||
        e->gate_x_stride < e->gate_ch || c.p.Hkv > kMaxGateHeads || ve_gate != nullptr)
      return SWA_ERR_INVALID_ARG;
    c.gx = static_cast<const elem_t*>(e->gate_x);
    c.gx_stride = e->gate_x_stride;
    c.gw = e->gate_w;
    c.gch = e->gate_ch;
    c.d_gw = e->d_gate_w;
    c.d_gx = e->d_gate_x;
  }
  return SWA_OK;
}

swa_status check_params(const swa_params* p) {
  if (p == nullptr) return SWA_ERR_INVALID_ARG;
  if (p->B < 0 || p->T < 0 || p->Hq < 1 || p->Hkv < 1 || p->d < 1) return SWA_ERR_INVALID_ARG;
  if (p->Hq % p->Hkv != 0) return SWA_ERR_INVALID_ARG;
  if (p->window < -1) return SWA_ERR_INVALID_ARG;
  if (p->causal != 0 && p->causal != 1) return SWA_ERR_INVALID_ARG;
  if (!std::isfinite(p->softmax_scale) || p->softmax_scale < 0.f) return SWA_ERR_INVALID_ARG;
  if (!std::isfinite(p->eps) || p->eps < 0.f) return SWA_ERR_INVALID_ARG;
  if (!std::isfinite(p->ve_scale)) return SWA_ERR_INVALID_ARG;
  if (p->d != 64 && p->d != 128) return SWA_ERR_UNSUPPORTED;
  // Grid and index limits: (batch, head) pairs index a grid dimension of at
  // most 65535 blocks in the row-wise kernels, tiles of 128 positions index
  // grid y of the attention kernels (< 65536), positions are 32-bit TMA
  // coordinates.
  if (p->T > (1 << 22) || static_cast<long long>(p->B) * p->Hq > 65535) return SWA_ERR_UNSUPPORTED;
  return SWA_OK;
}

swa_status check_device() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SWA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return SWA_ERR_CUDA;
  if (major != 10 || minor != 3) return SWA_ERR_UNSUPPORTED;  // built for sm_103a only
  return SWA_OK;
}

swa_status begin(Call& c, const swa_params* p, void* workspace, size_t ws_bytes, bool bwd,
                 void* stream) {
  swa_status s = check_params(p);
  if (s != SWA_OK) return s;
  c.p = *p;
  c.empty = (p->B == 0 || p->T == 0);
  c.scale = p->softmax_scale > 0.f ? p->softmax_scale : 1.0f / std::sqrt(static_cast<float>(p->d));
  c.L = ws_layout(p->B, p->T, p->Hq, p->Hkv, p->d);
  c.ws = static_cast<uint8_t*>(workspace);
  c.stream = static_cast<cudaStream_t>(stream);
  if (workspace == nullptr || !aligned(workspace, 256)) return SWA_ERR_INVALID_ARG;
  if (ws_bytes < (bwd ? c.L.bwd_end : c.L.fwd_end)) return SWA_ERR_WORKSPACE;
  return SWA_OK;
}

bool tensor_ok(const void* ptr) { return ptr != nullptr && aligned(ptr, 16); }

// Device status word in a workspace header.
uint32_t* at_status(uint8_t* ws) { return reinterpret_cast<uint32_t*>(ws); }

swa_status launched() {
  return cudaGetLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

template <typename T>
T* at(const Call& c, size_t off) {
  return reinterpret_cast<T*>(c.ws + off);
}


swa_status run_prologue(const Call& c, const elem_t* q, const elem_t* k, const elem_t* v,
                        const float* gq, const float* gk, const elem_t* ve, const int32_t* tok,
                        const float* gate, bool copy_v) {
  const swa_params& p = c.p;
  ProArgs a{};
  a.B = p.B; a.T = p.T; a.Hq = p.Hq; a.Hkv = p.Hkv; a.d = p.d; a.vocab = p.vocab;
  a.eps = p.eps; a.ve_scale = p.ve_scale;
  a.q = q; a.k = k; a.v = v; a.gq = gq; a.gk = gk; a.ve = ve; a.tok = tok; a.gate = gate;
  a.qn = at<elem_t>(c, c.L.qn); a.kn = at<elem_t>(c, c.L.kn); a.veff = at<elem_t>(c, c.L.veff);
  a.rstd_q = at<float>(c, c.L.rstd_q); a.rstd_k = at<float>(c, c.L.rstd_k);
  a.rcos = c.rcos; a.rsin = c.rsin;
  if (ve != nullptr && c.gw != nullptr) {
    a.gx = c.gx; a.gx_stride = c.gx_stride; a.gw = c.gw; a.gch = c.gch;
    a.gate_out = at<float>(c, c.L.gate);
  }
  a.status = at<uint32_t>(c, c.L.status);
  a.nseg = (ve != nullptr || copy_v) ? 3 : 2;
  const int rg = p.d == 64 ? RowMap<64, kProSlots>::RG : RowMap<128, kProSlots>::RG;
  const long long ngt = (p.T + rg - 1) / rg;
  const long long groups = ngt * p.B * (p.Hq + p.Hkv * (a.nseg - 1));
  const bool rope = a.rcos != nullptr, learned = a.gw != nullptr;
  const int grid = row_grid(groups, kProBlocksPerSm, 0);
  auto launch = [&](auto kern) { kern<<<grid, kRowWarps * 32, 0, c.stream>>>(a); };
  if (p.d == 64) {
    if (rope) learned ? launch(prologue_kernel<64, true, true>) : launch(prologue_kernel<64, true, false>);
    else learned ? launch(prologue_kernel<64, false, true>) : launch(prologue_kernel<64, false, false>);
  } else {
    if (rope) learned ? launch(prologue_kernel<128, true, true>) : launch(prologue_kernel<128, true, false>);
    else learned ? launch(prologue_kernel<128, false, true>) : launch(prologue_kernel<128, false, false>);
  }
  return launched();
}

}  // namespace

// Scratch of swa_attn_fwd_noalloc: a fixed device array, so that the call
// allocates nothing. Host code may not use this name as a device address (on
// the host it names a stand-in); noalloc_scratch() looks the address up.
static __device__ __align__(256) unsigned char swa_noalloc_scratch[SWA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 256;
std::mutex g_noalloc_mu;
struct NoallocAddr {
  CUcontext ctx;   // context current when the address was looked up
  void* addr;
};
NoallocAddr g_noalloc[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent from the driver (through the runtime's entry-point query,
// so the library does not link against the driver library).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  }
  return fn;
}

// Device address of swa_noalloc_scratch on the current device. Looked up once
// per device (with that device current), and again when the calling thread's
// current context is not the one of that lookup: after cudaDeviceReset, or
// under a context the caller made current, the module can sit elsewhere.
swa_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SWA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SWA_ERR_UNSUPPORTED;
  CtxGetCurrentFn get = ctx_get_current();
  if (get == nullptr) return SWA_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return SWA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocAddr& e = g_noalloc[dev];
  if (ctx == nullptr || e.addr == nullptr || e.ctx != ctx) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, swa_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return SWA_ERR_CUDA;
    // the lookup makes the device's primary context current if none was
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return SWA_ERR_CUDA;
    e.ctx = ctx;
    e.addr = ptr;
  }
  *out = e.addr;
  return SWA_OK;
}

}  // namespace

namespace {

// The forward of swa_attn_fwd. prepare_bwd: a workspace sized for the
// backward also gets its dQ accumulator zeroed by the forward kernel (the
// no-allocation entry point passes false).
swa_status fwd_impl(const swa_params* p, const swa_extras* ex, const void* q, const void* k,
                    const void* v, const float* gq, const float* gk, const void* ve,
                    const int32_t* tok, const float* ve_gate, void* o, float* lse, void* workspace,
                    size_t ws_bytes, unsigned flags, void* stream, bool prepare_bwd) {
  Call c;
  swa_status s = begin(c, p, workspace, ws_bytes, false, stream);
  if (s != SWA_OK) return s;
  if ((s = set_extras(c, ex, ve_gate)) != SWA_OK) return s;
  if ((flags & ~SWA_REUSE_PROLOGUE) != 0) return SWA_ERR_INVALID_ARG;
  if (!tensor_ok(q) || !tensor_ok(k) || !tensor_ok(v) || !tensor_ok(o) || lse == nullptr)
    return SWA_ERR_INVALID_ARG;
  if (ve != nullptr && (!aligned(ve, 16) || tok == nullptr || p->vocab < 1))
    return SWA_ERR_INVALID_ARG;
  if (c.empty) return SWA_OK;
  if ((s = check_device()) != SWA_OK) return s;
  const elem_t* qe = static_cast<const elem_t*>(q);
  const elem_t* ke = static_cast<const elem_t*>(k);
  const elem_t* vin = static_cast<const elem_t*>(v);
  const elem_t* vee = static_cast<const elem_t*>(ve);
#if defined(SWA_ELEM_FP32)
  const bool copy_v = true;
#else
  const bool copy_v = false;
#endif
  if (!(flags & SWA_REUSE_PROLOGUE)) {
    if ((s = run_prologue(c, qe, ke, vin, gq, gk, vee, tok, ve_gate, copy_v)) != SWA_OK) return s;
  }
#if defined(SWA_ELEM_FP32)
  SimtFwdArgs a{};
  a.B = p->B; a.T = p->T; a.Hq = p->Hq; a.Hkv = p->Hkv; a.window = p->window;
  a.causal = p->causal; a.scale = c.scale;
  a.qn = at<float>(c, c.L.qn); a.kn = at<float>(c, c.L.kn); a.veff = at<float>(c, c.L.veff);
  a.o = static_cast<float*>(o); a.lse = lse;
  dim3 grid((p->T + kSimtTile - 1) / kSimtTile, p->Hq, p->B);
  if (p->d == 64) {
    cudaFuncSetAttribute(fwd_simt_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(simt_fwd_smem<64>()));
    fwd_simt_kernel<64><<<grid, kSimtWarps * 32, simt_fwd_smem<64>(), c.stream>>>(a);
  } else {
    cudaFuncSetAttribute(fwd_simt_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(simt_fwd_smem<128>()));
    fwd_simt_kernel<128><<<grid, kSimtWarps * 32, simt_fwd_smem<128>(), c.stream>>>(a);
  }
  return launched();
#else
  tc::FwdLaunch f{};
  f.B = p->B; f.T = p->T; f.Hq = p->Hq; f.Hkv = p->Hkv; f.d = p->d;
  f.window = p->window; f.causal = p->causal; f.scale = c.scale;
  f.qn = at<elem_t>(c, c.L.qn); f.kn = at<elem_t>(c, c.L.kn);
  f.v = (ve != nullptr) ? at<elem_t>(c, c.L.veff) : vin;
  f.v_head_major = (ve != nullptr);
  f.o = static_cast<elem_t*>(o); f.lse = lse;
  f.status = at<uint32_t>(c, c.L.status);
  f.wait_limit_ns = c.wait_ns;
  // The forward is compute-bound, so it can zero the backward's dQ
  // accumulator at little cost; the backward's preprocess then skips it.
  f.acc_flag = at<unsigned long long>(c, c.L.status + 8);
  if (prepare_bwd && ws_bytes >= c.L.bwd_end) {
    f.dq_acc = at<float>(c, c.L.dq_acc);
    f.acc_off = c.L.dq_acc;
    f.acc_len = static_cast<unsigned long long>(p->B) * p->T * p->Hq * p->d * sizeof(float);
  }
  return tc::launch_fwd_any2(f, c.stream);
#endif
}

swa_status bwd_impl(const swa_params* p, const swa_extras* ex, const void* q, const void* k,
                    const void* v, const float* gq, const float* gk, const void* ve,
                    const int32_t* tok, const float* ve_gate, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv, float* dgq, float* dgk, float* dve,
                    void* workspace, size_t ws_bytes, unsigned flags, void* stream) {
  Call c;
  swa_status s = begin(c, p, workspace, ws_bytes, true, stream);
  if (s != SWA_OK) return s;
  if ((s = set_extras(c, ex, ve_gate)) != SWA_OK) return s;
  // with the learned gate, the gate values are the ones the forward (or the
  // prologue below) left in the workspace
  const float* gate_vals = (ve != nullptr && c.gw != nullptr) ? at<float>(c, c.L.gate) : ve_gate;
  const unsigned known = SWA_REUSE_PROLOGUE | SWA_BWD_STAGE_PRE | SWA_BWD_STAGE_MAIN | SWA_BWD_STAGE_POST;
  if ((flags & ~known) != 0) return SWA_ERR_INVALID_ARG;
  if (!tensor_ok(q) || !tensor_ok(k) || !tensor_ok(v) || !tensor_ok(o) || !tensor_ok(dO) ||
      !tensor_ok(dq) || !tensor_ok(dk) || !tensor_ok(dv) || lse == nullptr)
    return SWA_ERR_INVALID_ARG;
  if (ve != nullptr && (!aligned(ve, 16) || tok == nullptr || p->vocab < 1))
    return SWA_ERR_INVALID_ARG;
  unsigned stages = flags & (SWA_BWD_STAGE_PRE | SWA_BWD_STAGE_MAIN | SWA_BWD_STAGE_POST);
  if (stages == 0) stages = SWA_BWD_STAGE_PRE | SWA_BWD_STAGE_MAIN | SWA_BWD_STAGE_POST;
  const swa_params& P = c.p;
  cudaStream_t st = c.stream;
  if (c.empty) {
    // Nothing to differentiate: the shared-parameter gradients are zero.
    if (stages & SWA_BWD_STAGE_POST) {
      if (dgq && cudaMemsetAsync(dgq, 0, sizeof(float) * P.d, st) != cudaSuccess) return SWA_ERR_CUDA;
      if (dgk && cudaMemsetAsync(dgk, 0, sizeof(float) * P.d, st) != cudaSuccess) return SWA_ERR_CUDA;
      if (dve && ve && cudaMemsetAsync(dve, 0, sizeof(float) * P.vocab * P.Hkv * P.d, st) != cudaSuccess)
        return SWA_ERR_CUDA;
      if (c.gw && c.d_gw &&
          cudaMemsetAsync(c.d_gw, 0, sizeof(float) * P.Hkv * c.gch, st) != cudaSuccess)
        return SWA_ERR_CUDA;
    }
    return SWA_OK;
  }
  if ((s = check_device()) != SWA_OK) return s;
  const elem_t* qe = static_cast<const elem_t*>(q);
  const elem_t* ke = static_cast<const elem_t*>(k);
  const elem_t* vin = static_cast<const elem_t*>(v);
  const elem_t* vee = static_cast<const elem_t*>(ve);
#if defined(SWA_ELEM_FP32)
  const bool copy_v = true;
  const int clear_acc = 0;
  constexpr bool kFp32Build = true;
#else
  const bool copy_v = false;
  const int clear_acc = 1;
  constexpr bool kFp32Build = false;
#endif
  if ((stages & SWA_BWD_STAGE_PRE) && !(flags & SWA_REUSE_PROLOGUE)) {
    if ((s = run_prologue(c, qe, ke, vin, gq, gk, vee, tok, gate_vals, copy_v)) != SWA_OK) return s;
  }
  if (stages & SWA_BWD_STAGE_PRE) {
    PreArgs a{};
    a.B = P.B; a.T = P.T; a.Tpad = t_pad(P.T); a.Hq = P.Hq; a.Hkv = P.Hkv; a.d = P.d;
    a.o = static_cast<const elem_t*>(o); a.dO = static_cast<const elem_t*>(dO); a.lse = lse;
    a.dvec = at<float>(c, c.L.dvec); a.lse2 = at<float>(c, c.L.lse2);
    a.dq_acc = at<float>(c, c.L.dq_acc);
    a.clear_acc = clear_acc;
    a.acc_flag = at<unsigned long long>(c, c.L.status + 8);
    a.acc_off = c.L.dq_acc;
    a.acc_len = static_cast<unsigned long long>(P.B) * P.T * P.Hq * P.d * sizeof(float);
    a.status = at<uint32_t>(c, c.L.status);
    // The d = 128 tensor-core backward takes -D and log2(scale) - LSE log2(e)
    // (its P carries the softmax scale); the others take D and LSE log2(e).
    const bool scaled_p = !kFp32Build && P.d == 128;
    a.d_mul = scaled_p ? -1.f : 1.f;
    a.lse2_mul = scaled_p ? -1.4426950408889634f : 1.4426950408889634f;
    a.lse2_add = scaled_p ? log2f(c.scale) : 0.f;
    const int rg = P.d == 64 ? RowMap<64>::RG : RowMap<128>::RG;
    const int grid = row_grid(static_cast<long long>((P.T + rg - 1) / rg) * P.B * P.Hq, kPreBlocksPerSm, 0);
    if (P.d == 64) bwd_pre_kernel<64><<<grid, kRowWarps * 32, 0, st>>>(a);
    else bwd_pre_kernel<128><<<grid, kRowWarps * 32, 0, st>>>(a);
    if ((s = launched()) != SWA_OK) return s;
#if !defined(SWA_ELEM_FP32)
    // the attention backward adds the VE-table gradient into dve
    if (dve && ve) {
      if (cudaMemsetAsync(dve, 0, sizeof(float) * P.vocab * P.Hkv * P.d, st) != cudaSuccess)
        return SWA_ERR_CUDA;
    }
#endif
  }
  if (stages & SWA_BWD_STAGE_MAIN) {
#if defined(SWA_ELEM_FP32)
    SimtBwdArgs a{};
    a.B = P.B; a.T = P.T; a.Tpad = t_pad(P.T); a.Hq = P.Hq; a.Hkv = P.Hkv; a.window = P.window;
    a.causal = P.causal; a.scale = c.scale;
    a.qn = at<float>(c, c.L.qn); a.kn = at<float>(c, c.L.kn); a.veff = at<float>(c, c.L.veff);
    a.dO = static_cast<const float*>(dO); a.lse = lse; a.dvec = at<float>(c, c.L.dvec);
    a.dq_acc = at<float>(c, c.L.dq_acc); a.dk_acc = at<float>(c, c.L.dk_acc);
    a.dv_acc = at<float>(c, c.L.dv_acc);
    const int nt = (P.T + kSimtTile - 1) / kSimtTile;
    if (P.d == 64) {
      cudaFuncSetAttribute(bwd_dq_simt_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(simt_dq_smem<64>()));
      cudaFuncSetAttribute(bwd_dkv_simt_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(simt_dkv_smem<64>()));
      bwd_dq_simt_kernel<64><<<dim3(nt, P.Hq, P.B), kSimtWarps * 32, simt_dq_smem<64>(), st>>>(a);
      bwd_dkv_simt_kernel<64><<<dim3(nt, P.Hkv, P.B), kSimtWarps * 32, simt_dkv_smem<64>(), st>>>(a);
    } else {
      cudaFuncSetAttribute(bwd_dq_simt_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(simt_dq_smem<128>()));
      cudaFuncSetAttribute(bwd_dkv_simt_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(simt_dkv_smem<128>()));
      bwd_dq_simt_kernel<128><<<dim3(nt, P.Hq, P.B), kSimtWarps * 32, simt_dq_smem<128>(), st>>>(a);
      bwd_dkv_simt_kernel<128><<<dim3(nt, P.Hkv, P.B), kSimtWarps * 32, simt_dkv_smem<128>(), st>>>(a);
    }
    if ((s = launched()) != SWA_OK) return s;
#else
    tc::BwdLaunch b{};
    b.B = P.B; b.T = P.T; b.Hq = P.Hq; b.Hkv = P.Hkv; b.d = P.d;
    b.window = P.window; b.causal = P.causal; b.scale = c.scale;
    b.qn = at<elem_t>(c, c.L.qn); b.kn = at<elem_t>(c, c.L.kn);
    b.v = (ve != nullptr) ? at<elem_t>(c, c.L.veff) : vin;
    b.v_head_major = (ve != nullptr);
    b.dO = static_cast<const elem_t*>(dO);
    b.lse2 = at<float>(c, c.L.lse2); b.dvec = at<float>(c, c.L.dvec); b.Tpad = t_pad(P.T);
    b.dq_acc = at<float>(c, c.L.dq_acc);
    // key-side gradients come out of the kernel's epilogue
    b.k = ke; b.rstd_k = at<float>(c, c.L.rstd_k); b.gk = gk; b.tok = tok; b.gate = gate_vals;
    b.dve = (ve != nullptr) ? dve : nullptr; b.ve_scale = P.ve_scale; b.vocab = P.vocab;
    b.dk = static_cast<elem_t*>(dk); b.dv = static_cast<elem_t*>(dv);
    b.gpart_k = at<float>(c, c.L.gpart_k);
    b.status = at<uint32_t>(c, c.L.status);
    b.wait_limit_ns = c.wait_ns;
    b.acc_flag = at<unsigned long long>(c, c.L.status + 8);
    // with rotary the k-side norm backward moves to the post kernel
    b.dkn_out = c.rcos != nullptr ? at<float>(c, c.L.dk_acc) : nullptr;
    if ((s = (P.d == 128 ? tc::launch_bwd128(b, st) : tc::launch_bwd(b, st))) != SWA_OK) return s;
#endif
  }
  if (stages & SWA_BWD_STAGE_POST) {
#if defined(SWA_ELEM_FP32)
    if (dve && ve) {
      if (cudaMemsetAsync(dve, 0, sizeof(float) * P.vocab * P.Hkv * P.d, st) != cudaSuccess)
        return SWA_ERR_CUDA;
    }
    const int post_segments = 3;   // q, k and v rows
#else
    // q rows; k and v were done by the attention backward, except the k-side
    // norm and rotary backward when there are rotary tables
    const int post_segments = c.rcos != nullptr ? 2 : 1;
#endif
    PostArgs a{};
    a.B = P.B; a.T = P.T; a.Hq = P.Hq; a.Hkv = P.Hkv; a.d = P.d; a.vocab = P.vocab;
    a.ve_scale = P.ve_scale;
    a.q = qe; a.k = ke; a.gq = gq; a.gk = gk; a.tok = tok; a.gate = gate_vals;
    a.rstd_q = at<float>(c, c.L.rstd_q); a.rstd_k = at<float>(c, c.L.rstd_k);
    a.dq_acc = at<float>(c, c.L.dq_acc); a.dk_acc = at<float>(c, c.L.dk_acc);
    a.dv_acc = at<float>(c, c.L.dv_acc);
    a.dq = static_cast<elem_t*>(dq); a.dk = static_cast<elem_t*>(dk); a.dv = static_cast<elem_t*>(dv);
    a.dve = (ve != nullptr) ? dve : nullptr;
    a.gpart = at<float>(c, c.L.gpart);
    a.rcos = c.rcos; a.rsin = c.rsin;
    a.nblk_max = post_blocks(P.B, P.T, P.Hq);
    a.status = at<uint32_t>(c, c.L.status);
    // one gain partial per block: no more blocks than the workspace holds
    const int rg = P.d == 64 ? RowMap<64>::RG : RowMap<128>::RG;
    const int nblk = row_grid(static_cast<long long>((P.T + rg - 1) / rg) * P.B * P.Hq, kPostBlocksPerSm,
                               a.nblk_max);
    dim3 grid(nblk, post_segments);
    if (P.d == 64) bwd_post_kernel<64><<<grid, kRowWarps * 32, 0, st>>>(a);
    else bwd_post_kernel<128><<<grid, kRowWarps * 32, 0, st>>>(a);
    if ((s = launched()) != SWA_OK) return s;
    if (dgq || dgk) {
#if defined(SWA_ELEM_FP32)
      const float* part_k = at<float>(c, c.L.gpart) + static_cast<size_t>(post_blocks(P.B, P.T, P.Hq)) * P.d;
      const int n_k = nblk;
#else
      const bool post_k = c.rcos != nullptr;
      const float* part_k = post_k ? at<float>(c, c.L.gpart) + static_cast<size_t>(post_blocks(P.B, P.T, P.Hq)) * P.d
                                   : at<float>(c, c.L.gpart_k);
      const int n_k = post_k ? nblk : P.B * P.Hkv * ((P.T + 127) / 128);
#endif
      GainArgs g{P.d, at<float>(c, c.L.gpart), nblk, part_k, n_k, dgq, dgk, P.d};
      gain_sum_kernel<<<dim3(2, P.d / 32), kGainWarps * 32, 0, st>>>(g);
      if ((s = launched()) != SWA_OK) return s;
    }
    if (ve != nullptr && c.gw != nullptr && (c.d_gw != nullptr || c.d_gx != nullptr)) {
      // learned gate: dgate from the final dv, then the gate's own backward
      GateBwdArgs ga{};
      ga.B = P.B; ga.T = P.T; ga.Hkv = P.Hkv; ga.vocab = P.vocab; ga.gch = c.gch;
      ga.gx_stride = c.gx_stride; ga.ve_scale = P.ve_scale;
      ga.dv = static_cast<const elem_t*>(dv); ga.ve = vee; ga.tok = tok;
      ga.gate = at<float>(c, c.L.gate); ga.gx = c.gx; ga.gw = c.gw; ga.d_gx = c.d_gx;
      ga.gpart_w = at<float>(c, c.L.gpart_w);
      const int gblk = row_grid(static_cast<long long>(P.B) * P.T, kPreBlocksPerSm,
                                post_blocks(P.B, P.T, P.Hq));
      if (P.d == 64) ve_gate_bwd_kernel<64><<<gblk, kRowWarps * 32, 0, st>>>(ga);
      else ve_gate_bwd_kernel<128><<<gblk, kRowWarps * 32, 0, st>>>(ga);
      if ((s = launched()) != SWA_OK) return s;
      if (c.d_gw != nullptr) {
        const int width = P.Hkv * c.gch;
        GainArgs gw{(width + 31) / 32 * 32, at<float>(c, c.L.gpart_w), gblk, nullptr, 0, c.d_gw,
                    nullptr, width};
        // partial rows are 1024 floats apart
        gw.d = 1024;
        gain_sum_kernel<<<dim3(1, (width + 31) / 32), kGainWarps * 32, 0, st>>>(gw);
        if ((s = launched()) != SWA_OK) return s;
      }
    }
  }
  return SWA_OK;
}

// ---------------------------------------------------------------------------
// The block around the attention core: pre-norm, c_q / c_k / c_v, attention,
// c_proj and the residual (block.cuh).
// ---------------------------------------------------------------------------
struct BlockCall {
  int B, T, Hq, Hkv, d, C;
  long long rows;                // B * T
  blk::BlockLayout L;
  uint8_t* ws;
  cudaStream_t st;
  swa_extras ex{};               // the caller's extras with the gate's input set to the normed x
  const swa_extras* exp = nullptr;
};

swa_status block_begin(BlockCall& b, const swa_params* p, const swa_extras* ex, const swa_block_weights* w,
                       const void* x, const void* ve, const int32_t* tok, void* workspace, size_t ws_bytes,
                       bool bwd, void* stream) {
  swa_status s = check_params(p);
  if (s != SWA_OK) return s;
  if (w == nullptr || x == nullptr || !aligned(x, 16)) return SWA_ERR_INVALID_ARG;
  if (w->C < 8 || w->C % 8 != 0 || w->C > (1 << 16)) return SWA_ERR_INVALID_ARG;
  for (const void* m : {w->wq, w->wk, w->wv, w->wo})
    if (!tensor_ok(m)) return SWA_ERR_INVALID_ARG;
  b.B = p->B; b.T = p->T; b.Hq = p->Hq; b.Hkv = p->Hkv; b.d = p->d; b.C = w->C;
  b.rows = static_cast<long long>(p->B) * p->T;
  if (b.rows > 0x7fffffffLL) return SWA_ERR_UNSUPPORTED;   // GEMM dimensions are 32-bit
  b.L = blk::block_layout(p->B, p->T, p->Hq, p->Hkv, p->d, w->C);
  if (workspace == nullptr || !aligned(workspace, 256)) return SWA_ERR_INVALID_ARG;
  if (ws_bytes < (bwd ? b.L.bwd_end : b.L.fwd_end)) return SWA_ERR_WORKSPACE;
  b.ws = static_cast<uint8_t*>(workspace);
  b.st = static_cast<cudaStream_t>(stream);
  if (ex != nullptr) {
    // the block gives the learned gate its input (the normed x) and takes
    // the gradient of the channels it read
    if (ex->gate_x != nullptr || ex->d_gate_x != nullptr) return SWA_ERR_INVALID_ARG;
    b.ex = *ex;
    if (ex->gate_w != nullptr) {
      if (ex->gate_ch < 1 || ex->gate_ch > blk::kMaxBlockGateCh || ex->gate_ch > w->C)
        return SWA_ERR_INVALID_ARG;
      b.ex.gate_x = b.ws + b.L.xn;
      b.ex.gate_x_stride = w->C;
      if (bwd) b.ex.d_gate_x = reinterpret_cast<float*>(b.ws + b.L.dgx);
    }
    b.exp = &b.ex;
  }
  // Everything the attention calls check, checked here before the first
  // launch, so that a non-OK return launched nothing.
  Call c;
  c.p = *p;
  if ((s = set_extras(c, b.exp, nullptr)) != SWA_OK) return s;
  if (ve != nullptr && (!aligned(ve, 16) || tok == nullptr || p->vocab < 1)) return SWA_ERR_INVALID_ARG;
  return SWA_OK;
}

swa_status block_fwd_impl(const swa_params* p, const swa_extras* ex, const swa_block_weights* w,
                          const void* x, const float* gq, const float* gk, const void* ve,
                          const int32_t* tok, void* out, void* workspace, size_t ws_bytes, void* stream) {
  BlockCall b;
  swa_status s = block_begin(b, p, ex, w, x, ve, tok, workspace, ws_bytes, false, stream);
  if (s != SWA_OK) return s;
  if (!tensor_ok(out)) return SWA_ERR_INVALID_ARG;
  if (b.rows == 0) return SWA_OK;
  if ((s = check_device()) != SWA_OK) return s;
  uint8_t* ws = b.ws;
  const int C = b.C, nq = b.Hq * b.d, nkv = b.Hkv * b.d, rows = static_cast<int>(b.rows);
  elem_t* xn = reinterpret_cast<elem_t*>(ws + b.L.xn);
  uint32_t* status = at_status(ws);
  const WsLayout A = ws_layout(b.B, b.T, b.Hq, b.Hkv, b.d);   // the attention's workspace, first in the block's
  // The q, k, v projection with the attention's prologue (QK-norm, rotary,
  // value-embedding mix) in its epilogue: bf16 library, head dim 128, T a
  // multiple of 32. Elsewhere the projection, then the prologue kernel.
#if defined(SWA_ELEM_FP32)
  const bool fold = false;
#else
  const bool fold = b.d == 128 && b.T % 32 == 0;
#endif
  const bool learned = b.exp != nullptr && b.ex.gate_w != nullptr && ve != nullptr;
  float* gate_vals = reinterpret_cast<float*>(ws + A.gate);
  blk::prenorm_fwd_kernel<<<blk::prenorm_grid(b.rows), blk::kPnWarps * 32, 0, b.st>>>(
      static_cast<const elem_t*>(x), xn, reinterpret_cast<float*>(ws + b.L.rstd), b.rows, C, p->eps,
      fold && learned ? b.ex.gate_w : nullptr, b.ex.gate_ch, b.Hkv, gate_vals);
  if ((s = launched()) != SWA_OK) return s;
  // q, k, v = xn w^T: A = xn [rows][C], B = the weights [out][C] (K-major),
  // one launch with an output per projection where every head block of the
  // kv projections is a multiple of 128 columns long, else one per projection
  const float* rcos = b.exp != nullptr ? b.ex.rope_cos : nullptr;
  float* rope_t = reinterpret_cast<float*>(ws + b.L.rope_t);
  if (fold && rcos != nullptr) {
    const dim3 grid(static_cast<unsigned>((b.T + blk::kRtT - 1) / blk::kRtT), 2);
    blk::rope_transpose_kernel<<<grid, 256, 0, b.st>>>(rcos, b.ex.rope_sin, rope_t, b.T);
    if ((s = launched()) != SWA_OK) return s;
  }
  const void* wmat[3] = {w->wq, w->wk, w->wv};
  const size_t dst[3] = {b.L.q, b.L.k, b.L.v};
  const int nout[3] = {nq, nkv, nkv};
  const bool fused = nq % 128 == 0 && nkv % 128 == 0;
  for (int i = 0; i < (fused ? 1 : 3); ++i) {
    GemmCall g;
    g.M = rows; g.status = status;
    g.kseg[0] = {xn, C, C};
    g.n_nseg = fused ? 3 : 1;
    for (int j = 0; j < g.n_nseg; ++j) {
      const int t = fused ? j : i;
      g.bseg[j] = {wmat[t], C};
      g.nseg[j] = {nout[t], ws + dst[t], nout[t], nullptr, 0};
    }
    if (fold) {
      auto& e = g.qkv;
      e.on = true;
      e.T = b.T; e.Hq = b.Hq; e.Hkv = b.Hkv; e.vocab = p->vocab; e.eps = p->eps; e.ve_scale = p->ve_scale;
      e.gq = gq; e.gk = gk;
      e.rope_t = rcos != nullptr ? rope_t : nullptr;
      e.qn = ws + A.qn; e.kn = ws + A.kn; e.veff = ws + A.veff;
      e.rstd_q = reinterpret_cast<float*>(ws + A.rstd_q); e.rstd_k = reinterpret_cast<float*>(ws + A.rstd_k);
      e.ve = ve; e.tok = tok; e.gate = learned ? gate_vals : nullptr;
    }
    if ((s = blk::run_gemm(g, b.st)) != SWA_OK) return s;
  }
  s = fwd_impl(p, b.exp, ws + b.L.q, ws + b.L.k, ws + b.L.v, gq, gk, ve, tok, nullptr, ws + b.L.o,
               reinterpret_cast<float*>(ws + b.L.lse), ws, b.L.attn_bytes, fold ? SWA_REUSE_PROLOGUE : 0, stream,
               true);
  if (s != SWA_OK) return s;
  // out = x + o wo^T: A = o [rows][nq], B = wo [C][nq] (K-major), C = x
  GemmCall g;
  g.M = rows; g.status = status;
  g.kseg[0] = {ws + b.L.o, nq, nq};
  g.bseg[0] = {w->wo, nq};
  g.nseg[0] = {C, out, C, x, C};
  g.beta = 1.f;
  return blk::run_gemm(g, b.st);
}

swa_status block_bwd_impl(const swa_params* p, const swa_extras* ex, const swa_block_weights* w,
                          const void* x, const float* gq, const float* gk, const void* ve,
                          const int32_t* tok, const void* dout, void* dx, float* dwq, float* dwk,
                          float* dwv, float* dwo, float* dgq, float* dgk, float* dve, void* workspace,
                          size_t ws_bytes, void* stream) {
  BlockCall b;
  swa_status s = block_begin(b, p, ex, w, x, ve, tok, workspace, ws_bytes, true, stream);
  if (s != SWA_OK) return s;
  if (!tensor_ok(dout) || !tensor_ok(dx)) return SWA_ERR_INVALID_ARG;
  uint8_t* ws = b.ws;
  const int C = b.C, nq = b.Hq * b.d, nkv = b.Hkv * b.d, rows = static_cast<int>(b.rows);
  if (b.rows == 0) {
    // nothing to differentiate: every weight gradient is zero
    const size_t n[4] = {static_cast<size_t>(nq) * C, static_cast<size_t>(nkv) * C,
                         static_cast<size_t>(nkv) * C, static_cast<size_t>(C) * nq};
    float* dw[4] = {dwq, dwk, dwv, dwo};
    for (int i = 0; i < 4; ++i)
      if (dw[i] && cudaMemsetAsync(dw[i], 0, n[i] * sizeof(float), b.st) != cudaSuccess) return SWA_ERR_CUDA;
    return bwd_impl(p, b.exp, ws + b.L.q, ws + b.L.k, ws + b.L.v, gq, gk, ve, tok, nullptr, ws + b.L.o,
                    reinterpret_cast<const float*>(ws + b.L.lse), ws + b.L.dO, ws + b.L.dq, ws + b.L.dk,
                    ws + b.L.dv, dgq, dgk, dve, ws, b.L.attn_bytes, 0, stream);
  }
  if ((s = check_device()) != SWA_OK) return s;
  uint32_t* status = at_status(ws);
  const elem_t* xn = reinterpret_cast<const elem_t*>(ws + b.L.xn);
  // K = B*T GEMMs (the weight gradients) split K over about one wave of CTAs
  auto splits = [&](int m, int n) {
    const int tiles = ((m + 127) / 128) * ((n + 255) / 256);
    const int k = num_sms() / tiles;
    return k < 1 ? 1 : k;
  };
  // dwo [C][nq] = dout^T o: A = dout as [rows][C] (M-major), B = o [rows][nq] (N-major)
  if (dwo != nullptr) {
    GemmCall g;
    g.M = C; g.a_mn = true; g.b_mn = true; g.status = status;
    g.kseg[0] = {dout, C, rows};
    g.bseg[0] = {ws + b.L.o, nq};
    g.nseg[0] = {nq, dwo, nq, nullptr, 0};
    g.out = GEMM_OUT_F32; g.split = splits(C, nq);
    if ((s = blk::run_gemm(g, b.st)) != SWA_OK) return s;
  }
  // gradient of the attention output: dO = dout wo, B = wo [C][nq] (N-major)
  {
    GemmCall g;
    g.M = rows; g.b_mn = true; g.status = status;
    g.kseg[0] = {dout, C, C};
    g.bseg[0] = {w->wo, nq};
    g.nseg[0] = {nq, ws + b.L.dO, nq, nullptr, 0};
    if ((s = blk::run_gemm(g, b.st)) != SWA_OK) return s;
  }
  s = bwd_impl(p, b.exp, ws + b.L.q, ws + b.L.k, ws + b.L.v, gq, gk, ve, tok, nullptr, ws + b.L.o,
               reinterpret_cast<const float*>(ws + b.L.lse), ws + b.L.dO, ws + b.L.dq, ws + b.L.dk,
               ws + b.L.dv, dgq, dgk, dve, ws, b.L.attn_bytes, SWA_REUSE_PROLOGUE, stream);
  if (s != SWA_OK) return s;
  const void* wmat[3] = {w->wq, w->wk, w->wv};
  const size_t grad[3] = {b.L.dq, b.L.dk, b.L.dv};
  const int nout[3] = {nq, nkv, nkv};
  float* dw[3] = {dwq, dwk, dwv};
  for (int i = 0; i < 3; ++i) {
    // dw [n_out][C] = grad^T xn: A = grad as [rows][n_out] (M-major), B = xn [rows][C] (N-major)
    if (dw[i] == nullptr) continue;
    GemmCall g;
    g.M = nout[i]; g.a_mn = true; g.b_mn = true; g.status = status;
    g.kseg[0] = {ws + grad[i], nout[i], rows};
    g.bseg[0] = {xn, C};
    g.nseg[0] = {C, dw[i], C, nullptr, 0};
    g.out = GEMM_OUT_F32; g.split = splits(nout[i], C);
    if ((s = blk::run_gemm(g, b.st)) != SWA_OK) return s;
  }
  // dxn = dq wq + dk wk + dv wv: three K segments, B = the weights [n_out][C] (N-major)
  float* dxn = reinterpret_cast<float*>(ws + b.L.dxn);
  {
    GemmCall g;
    g.M = rows; g.b_mn = true; g.status = status;
    g.n_kseg = 3;
    for (int i = 0; i < 3; ++i) {
      g.kseg[i] = {ws + grad[i], nout[i], nout[i]};
      g.bseg[i] = {wmat[i], C};
    }
    g.nseg[0] = {C, dxn, C, nullptr, 0};
    g.out = GEMM_OUT_F32;
    if ((s = blk::run_gemm(g, b.st)) != SWA_OK) return s;
  }
  // the gate applies on value-embedding calls only (as in the attention calls)
  const bool gate = b.exp != nullptr && b.ex.gate_w != nullptr && ve != nullptr;
  blk::prenorm_bwd_kernel<<<blk::prenorm_grid(b.rows), blk::kPnWarps * 32, 0, b.st>>>(
      static_cast<const elem_t*>(x), reinterpret_cast<const float*>(ws + b.L.rstd), dxn,
      gate ? reinterpret_cast<const float*>(ws + b.L.dgx) : nullptr, gate ? b.ex.gate_ch : 0,
      static_cast<const elem_t*>(dout), static_cast<elem_t*>(dx), b.rows, C);
  return launched();
}

}  // namespace

namespace {

// Device buffer of swa_attn_step_host: the attention's backward workspace,
// then device copies of the inputs and outputs (256-byte aligned each).
struct StepHostLayout {
  size_t ws_bytes;
  size_t q, k, v, gq, gk, ve, tok, gate, dO, o, lse, dq, dk, dv, dgq, dgk, dve, end;
  size_t q_bytes, kv_bytes, gain_bytes, ve_bytes, tok_bytes, gate_bytes, lse_bytes, dve_bytes;
};

StepHostLayout step_host_layout(const swa_params& p) {
  StepHostLayout L;
  const size_t bt = static_cast<size_t>(p.B) * static_cast<size_t>(p.T);
  const size_t es = sizeof(elem_t);
  const size_t vocab = p.vocab > 0 ? static_cast<size_t>(p.vocab) : 0;
  L.q_bytes = bt * p.Hq * p.d * es;
  L.kv_bytes = bt * p.Hkv * p.d * es;
  L.gain_bytes = static_cast<size_t>(p.d) * sizeof(float);
  L.ve_bytes = vocab * p.Hkv * p.d * es;
  L.tok_bytes = bt * sizeof(int32_t);
  L.gate_bytes = bt * p.Hkv * sizeof(float);
  L.lse_bytes = bt * p.Hq * sizeof(float);
  L.dve_bytes = vocab * p.Hkv * p.d * sizeof(float);
  L.ws_bytes = align256(ws_layout(p.B, p.T, p.Hq, p.Hkv, p.d).bwd_end);
  size_t o = L.ws_bytes;
  auto take = [&](size_t bytes) { const size_t at = o; o = align256(o + bytes); return at; };
  L.q = take(L.q_bytes); L.k = take(L.kv_bytes); L.v = take(L.kv_bytes);
  L.gq = take(L.gain_bytes); L.gk = take(L.gain_bytes); L.ve = take(L.ve_bytes);
  L.tok = take(L.tok_bytes); L.gate = take(L.gate_bytes); L.dO = take(L.q_bytes);
  L.o = take(L.q_bytes); L.lse = take(L.lse_bytes); L.dq = take(L.q_bytes);
  L.dk = take(L.kv_bytes); L.dv = take(L.kv_bytes); L.dgq = take(L.gain_bytes);
  L.dgk = take(L.gain_bytes); L.dve = take(L.dve_bytes);
  L.end = o;
  return L;
}

}  // namespace

// ---------------------------------------------------------------------------
// Exported C ABI
// ---------------------------------------------------------------------------
extern "C" {

size_t swa_attn_workspace_size(const swa_params* p, int for_backward) {
  if (check_params(p) != SWA_OK) return 0;
  const WsLayout L = ws_layout(p->B, p->T, p->Hq, p->Hkv, p->d);
  return for_backward ? L.bwd_end : L.fwd_end;
}

swa_status swa_attn_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
  if (workspace == nullptr || !aligned(workspace, 256) || ws_bytes < 256) return SWA_ERR_INVALID_ARG;
  if (cudaMemsetAsync(workspace, 0, 256, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SWA_ERR_CUDA;
  return SWA_OK;
}

swa_status swa_attn_fwd(const swa_params* p, const void* q, const void* k, const void* v,
                        const float* gq, const float* gk, const void* ve, const int32_t* tok,
                        const float* ve_gate, void* o, float* lse, void* workspace,
                        size_t ws_bytes, unsigned flags, void* stream) {
  return fwd_impl(p, nullptr, q, k, v, gq, gk, ve, tok, ve_gate, o, lse, workspace, ws_bytes, flags,
                  stream, true);
}

swa_status swa_attn_fwd_ex(const swa_params* p, const swa_extras* ex, const void* q, const void* k,
                             const void* v, const float* gq, const float* gk, const void* ve,
                             const int32_t* tok, const float* ve_gate, void* o, float* lse,
                             void* workspace, size_t ws_bytes, unsigned flags, void* stream) {
  return fwd_impl(p, ex, q, k, v, gq, gk, ve, tok, ve_gate, o, lse, workspace, ws_bytes, flags,
                  stream, true);
}

swa_status swa_attn_bwd(const swa_params* p, const void* q, const void* k, const void* v,
                        const float* gq, const float* gk, const void* ve, const int32_t* tok,
                        const float* ve_gate, const void* o, const float* lse, const void* dO,
                        void* dq, void* dk, void* dv, float* dgq, float* dgk, float* dve,
                        void* workspace, size_t ws_bytes, unsigned flags, void* stream) {
  return bwd_impl(p, nullptr, q, k, v, gq, gk, ve, tok, ve_gate, o, lse, dO, dq, dk, dv, dgq, dgk, dve,
                  workspace, ws_bytes, flags, stream);
}

swa_status swa_attn_bwd_ex(const swa_params* p, const swa_extras* ex, const void* q, const void* k,
                             const void* v, const float* gq, const float* gk, const void* ve,
                             const int32_t* tok, const float* ve_gate, const void* o,
                             const float* lse, const void* dO, void* dq, void* dk, void* dv,
                             float* dgq, float* dgk, float* dve, void* workspace, size_t ws_bytes,
                             unsigned flags, void* stream) {
  return bwd_impl(p, ex, q, k, v, gq, gk, ve, tok, ve_gate, o, lse, dO, dq, dk, dv, dgq, dgk, dve,
                  workspace, ws_bytes, flags, stream);
}

swa_status swa_attn_check_status(void* workspace, void* stream) {
  if (workspace == nullptr || !aligned(workspace, 256)) return SWA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SWA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SWA_ERR_CUDA;
  if (word != 0) {
    if (cudaMemsetAsync(workspace, 0, sizeof(word), st) != cudaSuccess) return SWA_ERR_CUDA;
    // After a wait ran out, a forward may not have zeroed all of the dQ
    // accumulator it recorded as zeroed: drop the record (its length word).
    if ((word & DEV_ERR_TIMEOUT) &&
        cudaMemsetAsync(static_cast<uint8_t*>(workspace) + 16, 0, 8, st) != cudaSuccess)
      return SWA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SWA_ERR_CUDA;
  }
  if (word & DEV_ERR_TIMEOUT) return SWA_ERR_TIMEOUT;
  if (word & (DEV_ERR_TOKEN | DEV_ERR_BOUNDS)) return SWA_ERR_DEVICE_CHECK;
  return SWA_OK;
}

swa_status swa_attn_fwd_noalloc(const swa_params* p, const void* q, const void* k,
                                const void* v, const float* gq, const float* gk, const void* ve,
                                const int32_t* tok, const float* ve_gate, void* o, float* lse,
                                void* stream) {
  const swa_status s = check_params(p);
  if (s != SWA_OK) return s;
  if (ws_layout(p->B, p->T, p->Hq, p->Hkv, p->d).fwd_end > SWA_NOALLOC_SCRATCH_BYTES)
    return SWA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const swa_status ss = noalloc_scratch(&scratch);
  if (ss != SWA_OK) return ss;
  return fwd_impl(p, nullptr, q, k, v, gq, gk, ve, tok, ve_gate, o, lse, scratch,
                  SWA_NOALLOC_SCRATCH_BYTES, 0, stream, false);
}

size_t swa_attn_step_host_size(const swa_params* p) {
  if (check_params(p) != SWA_OK) return 0;
  return step_host_layout(*p).end;
}

swa_status swa_attn_step_host(const swa_params* p, const swa_extras* ex, const void* q,
                              const void* k, const void* v, const float* gq, const float* gk,
                              const void* ve, const int32_t* tok, const float* ve_gate,
                              const void* dO, void* o, float* lse, void* dq, void* dk, void* dv,
                              float* dgq, float* dgk, float* dve, void* device_buffer,
                              size_t device_bytes, void* stream) {
  swa_status s = check_params(p);
  if (s != SWA_OK) return s;
  if (q == nullptr || k == nullptr || v == nullptr || dO == nullptr || o == nullptr || lse == nullptr ||
      dq == nullptr || dk == nullptr || dv == nullptr || device_buffer == nullptr ||
      !aligned(device_buffer, 256))
    return SWA_ERR_INVALID_ARG;
  if ((ve == nullptr) != (tok == nullptr) || (ve != nullptr && p->vocab <= 0)) return SWA_ERR_INVALID_ARG;
  const StepHostLayout L = step_host_layout(*p);
  if (device_bytes < L.end) return SWA_ERR_WORKSPACE;
  if (p->B == 0 || p->T == 0) return SWA_OK;
  uint8_t* base = static_cast<uint8_t*>(device_buffer);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto dev = [&](size_t off, const void* host) -> void* { return host ? base + off : nullptr; };
  auto up = [&](size_t off, const void* host, size_t bytes) {
    return host == nullptr || bytes == 0 ||
           cudaMemcpyAsync(base + off, host, bytes, cudaMemcpyHostToDevice, st) == cudaSuccess;
  };
  auto down = [&](void* host, size_t off, size_t bytes) {
    return host == nullptr || bytes == 0 ||
           cudaMemcpyAsync(host, base + off, bytes, cudaMemcpyDeviceToHost, st) == cudaSuccess;
  };
  if (!(up(L.q, q, L.q_bytes) && up(L.k, k, L.kv_bytes) && up(L.v, v, L.kv_bytes) &&
        up(L.gq, gq, L.gain_bytes) && up(L.gk, gk, L.gain_bytes) && up(L.ve, ve, L.ve_bytes) &&
        up(L.tok, tok, L.tok_bytes) && up(L.gate, ve_gate, L.gate_bytes) && up(L.dO, dO, L.q_bytes)))
    return SWA_ERR_CUDA;
  const float* gq_d = static_cast<const float*>(dev(L.gq, gq));
  const float* gk_d = static_cast<const float*>(dev(L.gk, gk));
  const void* ve_d = dev(L.ve, ve);
  const int32_t* tok_d = static_cast<const int32_t*>(dev(L.tok, tok));
  const float* gate_d = static_cast<const float*>(dev(L.gate, ve_gate));
  float* lse_d = reinterpret_cast<float*>(base + L.lse);
  s = fwd_impl(p, ex, base + L.q, base + L.k, base + L.v, gq_d, gk_d, ve_d, tok_d, gate_d, base + L.o, lse_d,
               base, L.ws_bytes, 0, stream, true);
  if (s != SWA_OK) return s;
  s = bwd_impl(p, ex, base + L.q, base + L.k, base + L.v, gq_d, gk_d, ve_d, tok_d, gate_d, base + L.o, lse_d,
               base + L.dO, base + L.dq, base + L.dk, base + L.dv, static_cast<float*>(dev(L.dgq, dgq)),
               static_cast<float*>(dev(L.dgk, dgk)), static_cast<float*>(dev(L.dve, ve ? dve : nullptr)),
               base, L.ws_bytes, SWA_REUSE_PROLOGUE, stream);
  if (s != SWA_OK) return s;
  if (!(down(o, L.o, L.q_bytes) && down(lse, L.lse, L.lse_bytes) && down(dq, L.dq, L.q_bytes) &&
        down(dk, L.dk, L.kv_bytes) && down(dv, L.dv, L.kv_bytes) && down(dgq, L.dgq, L.gain_bytes) &&
        down(dgk, L.dgk, L.gain_bytes) && down(ve ? dve : nullptr, L.dve, L.dve_bytes)))
    return SWA_ERR_CUDA;
  return SWA_OK;
}

size_t swa_block_workspace_size(const swa_params* p, int C, int for_backward) {
  if (check_params(p) != SWA_OK || C < 8 || C % 8 != 0 || C > (1 << 16)) return 0;
  const blk::BlockLayout L = blk::block_layout(p->B, p->T, p->Hq, p->Hkv, p->d, C);
  return for_backward ? L.bwd_end : L.fwd_end;
}

swa_status swa_block_fwd(const swa_params* p, const swa_extras* ex, const swa_block_weights* w,
                         const void* x, const float* gq, const float* gk, const void* ve,
                         const int32_t* tok, void* out, void* workspace, size_t ws_bytes, void* stream) {
  return block_fwd_impl(p, ex, w, x, gq, gk, ve, tok, out, workspace, ws_bytes, stream);
}

swa_status swa_block_bwd(const swa_params* p, const swa_extras* ex, const swa_block_weights* w,
                         const void* x, const float* gq, const float* gk, const void* ve,
                         const int32_t* tok, const void* dout, void* dx, float* dwq, float* dwk,
                         float* dwv, float* dwo, float* dgq, float* dgk, float* dve, void* workspace,
                         size_t ws_bytes, void* stream) {
  return block_bwd_impl(p, ex, w, x, gq, gk, ve, tok, dout, dx, dwq, dwk, dwv, dwo, dgq, dgk, dve,
                        workspace, ws_bytes, stream);
}

int swa_sssl_window(int layer, int n_layer, const char* pattern, int T) {
  if (pattern == nullptr || pattern[0] == '\0' || n_layer < 1 || layer < 0 || layer >= n_layer ||
      T < 0)
    return -2;
  const size_t n = std::strlen(pattern);
  for (size_t i = 0; i < n; ++i)
    if (pattern[i] != 'S' && pattern[i] != 'L') return -2;
  if (layer == n_layer - 1) return -1;  // the last layer is always global
  return pattern[static_cast<size_t>(layer) % n] == 'S' ? T / 2 : -1;
}

int swa_has_ve(int layer, int n_layer) {
  if (n_layer < 1 || layer < 0 || layer >= n_layer) return -1;
  return (layer % 2) == ((n_layer - 1) % 2) ? 1 : 0;
}

const char* swa_strerror(swa_status s) {
  switch (s) {
    case SWA_OK: return "ok";
    case SWA_ERR_INVALID_ARG: return "invalid argument";
    case SWA_ERR_UNSUPPORTED: return "unsupported configuration (head dim, sizes or GPU)";
    case SWA_ERR_CUDA: return "CUDA call failed";
    case SWA_ERR_TIMEOUT: return "a device pipeline wait ran out of time";
    case SWA_ERR_WORKSPACE: return "workspace too small";
    case SWA_ERR_DEVICE_CHECK: return "device check failed (token id outside the table)";
  }
  return "unknown status";
}

const char* swa_build_info(void) {
#if defined(SWA_ELEM_FP32)
  return "swa_attn fp32 SIMT debug build, sm_103a";
#else
  return "swa_attn bf16 tcgen05 build, sm_103a";
#endif
}

}  // extern "C"
