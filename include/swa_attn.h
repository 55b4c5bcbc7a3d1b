/*
 * swa_attn.h - C ABI of the GB300 (sm_103a) attention-block library.
 *
 * The block computed here is the attention of the autoresearch GPT training
 * script as its pages describe it:
 *   - QK-norm: RMSNorm of queries and keys right before the attention dot
 *     product (autoresearch train.py walkthrough post, model paragraph;
 *     "autoresearch Administrator & Developer Guide" §8.2.1, F.rms_norm row),
 *     here with optional learned per-channel gains gq, gk of shape [d];
 *   - grouped-query attention, n_kv_head <= n_head (Guide §8.2.1, GQA row;
 *     §6.3 techniques table): query head h reads kv head h / (Hq / Hkv);
 *   - a causal sliding window or full causal mask per layer, chosen by the
 *     "SSSL" window pattern (post, model paragraph; Guide §3.4 WINDOW_PATTERN);
 *   - on value-embedding layers, v_eff = v + ve_scale * gate * VE[token]
 *     (Guide §8.2.1, value-embedding row and its gate snippet).
 *
 * Two shared libraries export these symbols:
 *   libswaattn.so       bf16 tensors, tcgen05 tensor-core kernels (the product path);
 *   libswaattn_fp32.so  fp32 tensors, SIMT FFMA kernels (a debug build with
 *                       the same band schedule, used to check the method at
 *                       fp32 precision).
 * "elem" below is bf16 (raw 16-bit bit patterns) in the first, float in the
 * second. Gains, LSE, gate and all gradients of shared parameters are fp32 in
 * both.
 *
 * Conventions common to every call:
 *   - All tensor pointers are DEVICE pointers of the current CUDA device; the
 *     caller owns every buffer, including the workspace. The library never
 *     allocates or frees device memory.
 *   - Layouts are dense row-major:
 *       q, o, dO, dq       [B, T, Hq,  d]   elem
 *       k, v, dk, dv       [B, T, Hkv, d]   elem
 *       lse                [B, Hq, T]       fp32, natural-log sum of exp of the
 *                                           scaled, masked logits of each row
 *       gq, gk, dgq, dgk   [d]              fp32
 *       ve, dve            [vocab, Hkv*d]   elem (ve) / fp32 (dve)
 *       tok                [B, T]           int32
 *       ve_gate            [B, T, Hkv]      fp32
 *   - Tensor pointers must be 16-byte aligned; the workspace 256-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream). SWA_ERR_INVALID_ARG, SWA_ERR_WORKSPACE and the unsupported-
 *     size checks come before the first launch: nothing was launched. A
 *     failing CUDA call inside a call (SWA_ERR_CUDA) can come after earlier
 *     launches of that call; its outputs are then undefined. Errors found on the device (a bounded wait that ran
 *     out, a token id outside [0, vocab)) are OR-ed into a status word in the
 *     workspace header and read back by swa_attn_check_status().
 *   - B == 0 or T == 0 is a valid empty problem: nothing is computed; the
 *     backward still zero-fills dgq, dgk and dve.
 */
#ifndef SWA_ATTN_H
#define SWA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum swa_status {
  SWA_OK = 0,
  SWA_ERR_INVALID_ARG = 1,  /* bad shape, NULL pointer, misalignment, bad flag   */
  SWA_ERR_UNSUPPORTED = 2,  /* valid but not built: d not in {64,128}, wrong GPU  */
  SWA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed                  */
  SWA_ERR_TIMEOUT = 4,      /* device: a bounded pipeline wait ran out            */
  SWA_ERR_WORKSPACE = 5,    /* workspace too small for this problem               */
  SWA_ERR_DEVICE_CHECK = 6  /* device: a token id outside [0, vocab) was skipped  */
} swa_status;

/* Problem description shared by every call. */
typedef struct swa_params {
  int B, T;         /* batch, sequence length (>= 0)                              */
  int Hq, Hkv;      /* query heads, kv heads; Hq % Hkv == 0                       */
  int d;            /* head dim: 64 or 128                                         */
  int window;       /* -1: no window. Else, causal: key j visible to query i iff
                       i - window <= j <= i; non-causal: iff |i - j| <= window.
                       window >= T - 1 is the same as -1.                          */
  int causal;       /* 1: causal (every layer of the SSSL stack); 0: bidirectional */
  float softmax_scale; /* 0: 1/sqrt(d)                                             */
  float eps;        /* RMSNorm epsilon, >= 0 (the script's F.rms_norm default is
                       used by callers that pass 1e-6)                             */
  float ve_scale;   /* multiplies gate * VE[tok]; ignored when ve == NULL          */
  int vocab;        /* rows of the VE table; ignored when ve == NULL               */
} swa_params;

/* flags */
#define SWA_REUSE_PROLOGUE 1u  /* the workspace still holds this problem's QK-norm /
                                  VE-mix outputs from an earlier call with the same
                                  inputs: skip recomputing them                       */
#define SWA_BWD_STAGE_PRE 2u   /* backward stages to run; none of the three bits set */
#define SWA_BWD_STAGE_MAIN 4u  /* means all of them. PRE: D = rowsum(dO * O), clear   */
#define SWA_BWD_STAGE_POST 8u  /* the accumulators unless the forward left them
                                  zeroed (and dve); MAIN: the attention
                                  backward with the key-side RMSNorm backward (dk,
                                  dv, dve); POST: query-side RMSNorm backward and
                                  the gain gradients.
                                  Running them one call at a time, in this order,
                                  gives the same result as one call with all three.  */

/*
 * Bytes of workspace a problem needs (forward only, or forward + backward).
 * Returns 0 when the parameters are invalid. The workspace holds a 256-byte
 * header (device status word, record of a zeroed dQ accumulator), the
 * QK-norm outputs qn, kn and their inverse
 * RMS, v_eff on VE layers, and for the backward the fp32 accumulators.
 * A fresh workspace must be initialised once with swa_attn_workspace_init().
 */
size_t swa_attn_workspace_size(const swa_params* p, int for_backward);

/* Zeroes the workspace header (status word) on `stream`. */
swa_status swa_attn_workspace_init(void* workspace, size_t ws_bytes, void* stream);

/*
 * Forward: o = softmax(scale * qn kn^T + mask) v_eff and lse, where
 * qn = gq * q / sqrt(mean(q^2) + eps) (likewise kn) and v_eff = v on plain
 * layers, v + ve_scale * gate * VE[tok] on value-embedding layers.
 *   gq, gk   may be NULL (unit gains).
 *   ve       NULL: no value embedding (tok, ve_gate ignored). Else tok is
 *            required and ve_gate may be NULL (gate = 1, the pages' gate at
 *            initialisation: 2 * sigmoid(0)).
 *   flags    0 or SWA_REUSE_PROLOGUE.
 * Writes o and lse, and the prologue outputs into the workspace (kept for the
 * backward's SWA_REUSE_PROLOGUE). When ws_bytes is at least the backward
 * size (swa_attn_workspace_size(p, 1)) and Hq / Hkv is even, the forward
 * kernel also zeroes the backward's fp32 dQ accumulator and records that in
 * the workspace header; the next backward of the same problem on this
 * workspace then skips that clear. Any later call that may overwrite the
 * accumulator drops the record (a forward that does not zero it, the
 * backward's main stage).
 */
swa_status swa_attn_fwd(const swa_params* p, const void* q, const void* k, const void* v,
                        const float* gq, const float* gk, const void* ve, const int32_t* tok,
                        const float* ve_gate, void* o, float* lse, void* workspace,
                        size_t ws_bytes, unsigned flags, void* stream);

/*
 * Backward of the forward for the loss <o, dO>: gradients of q, k, v, the
 * gains and the VE table. Inputs as in swa_attn_fwd plus the forward's o and
 * lse and the upstream gradient dO. Outputs (overwritten, not accumulated):
 *   dq, dk, dv       required.
 *   dgq, dgk         may be NULL (not computed); when non-NULL they receive
 *                    the full gain gradient (summed over batch, time, heads).
 *                    With gq (gk) NULL the gain is 1 and dgq (dgk) is still the
 *                    gradient with respect to it.
 *   dve              may be NULL; when non-NULL (and ve != NULL) it receives
 *                    the gradient of the VE table, zero in rows no token used.
 * The gradient of a given ve_gate is not produced (it is an input); the
 * learned gate of swa_attn_bwd_ex produces its own gradients.
 * flags: SWA_REUSE_PROLOGUE and the SWA_BWD_STAGE_* bits.
 */
swa_status swa_attn_bwd(const swa_params* p, const void* q, const void* k, const void* v,
                        const float* gq, const float* gk, const void* ve, const int32_t* tok,
                        const float* ve_gate, const void* o, const float* lse, const void* dO,
                        void* dq, void* dk, void* dv, float* dgq, float* dgk, float* dve,
                        void* workspace, size_t ws_bytes, unsigned flags, void* stream);

/*
 * Extras of the _ex entry points (each part optional; all-NULL extras, or a
 * NULL pointer, make them identical to swa_attn_fwd / swa_attn_bwd).
 *
 * Rotary position embedding, fused into the QK-norm prologue (rotation
 * first, then the norm, so the norm comes right before the dot product, as
 * in the autoresearch train.py walkthrough post, model paragraph; the
 * Administrator & Developer Guide §8.2.1 model table, "Rotary embeddings"
 * row, has the cos / sin tables precomputed once by the caller). The pages
 * print neither the channel pairing nor the sign; this library pairs channel
 * c with c + d/2 and turns the pair of position t by the angle of row t,
 * column c:
 *   y_c       =  x_c cos[t][c] + x_{c+d/2} sin[t][c]
 *   y_{c+d/2} = -x_c sin[t][c] + x_{c+d/2} cos[t][c]        (c < d/2)
 *   rope_cos, rope_sin  fp32 [rope_rows][d/2] row-major, 16-byte aligned,
 *                       rope_rows >= T (row t is position t); both NULL: none.
 *
 * Learned value-embedding gate (Guide §8.2.1, the gate snippet): on VE
 * calls, gate[b,t,h] = 2 * sigmoid(sum_c gate_w[h][c] * gate_x[b,t,c]), used
 * in place of the ve_gate argument (which must then be NULL):
 *   gate_x         elem (bf16 / fp32 per library) rows of the block input;
 *                  channel c of position (b, t) at gate_x[(b*T + t)*gate_x_stride + c]
 *   gate_x_stride  elements between consecutive (b, t) rows (>= gate_ch)
 *   gate_w         fp32 [Hkv][gate_ch]; NULL: no learned gate
 *   gate_ch        1 .. 32 channels (32 in the pages); Hkv <= 32
 *   d_gate_w       backward output, fp32 [Hkv][gate_ch] (overwritten), or NULL
 *   d_gate_x       backward output, fp32 [B, T, gate_ch] (overwritten): the
 *                  gradient of the channels read (the caller adds it into
 *                  its gradient of the block input), or NULL
 * The forward keeps the gate values in the workspace for the backward.
 *
 * Time limit of the kernels' pipeline waits (not from the pages: a property
 * of this library's kernels, whose warps hand work to each other through
 * shared-memory barriers):
 *   wait_limit_ns  0: the default, 2 s per wait. Else the limit of every
 *                  pipeline wait of this call's tensor-core kernels. A wait
 *                  that runs out makes its CTA give up: it records
 *                  SWA_ERR_TIMEOUT in the workspace status word, lets the
 *                  copies and MMAs it issued land (those waits keep their
 *                  own 2 s limit), and returns; the call's outputs are then
 *                  undefined. A short limit is how a caller (or a test) can
 *                  make this path run. Limits below 1 ms are kept by polling
 *                  the barrier without suspending; longer ones by the
 *                  barrier's suspending wait, with the clock read every 64
 *                  polls. The fp32 debug build has no such waits and ignores
 *                  the field.
 */
typedef struct {
  const float* rope_cos;
  const float* rope_sin;
  int rope_rows;
  const void* gate_x;
  long long gate_x_stride;
  const float* gate_w;
  int gate_ch;
  float* d_gate_w;
  float* d_gate_x;
  unsigned long long wait_limit_ns;
} swa_extras;

/* swa_attn_fwd with extras (arguments otherwise identical). */
swa_status swa_attn_fwd_ex(const swa_params* p, const swa_extras* ex, const void* q, const void* k,
                           const void* v, const float* gq, const float* gk, const void* ve,
                           const int32_t* tok, const float* ve_gate, void* o, float* lse,
                           void* workspace, size_t ws_bytes, unsigned flags, void* stream);

/* swa_attn_bwd with extras: with rotary, dq and dk are the gradients of the
 * unrotated q and k (the transposed rotation of the norm backward's result);
 * with the learned gate, d_gate_w and d_gate_x as above (written by the POST
 * stage). A backward with SWA_REUSE_PROLOGUE needs the same extras as its
 * forward. */
swa_status swa_attn_bwd_ex(const swa_params* p, const swa_extras* ex, const void* q, const void* k,
                           const void* v, const float* gq, const float* gk, const void* ve,
                           const int32_t* tok, const float* ve_gate, const void* o,
                           const float* lse, const void* dO, void* dq, void* dk, void* dv,
                           float* dgq, float* dgk, float* dve, void* workspace, size_t ws_bytes,
                           unsigned flags, void* stream);

/*
 * Forward without a caller-provided workspace: the same computation and
 * outputs as swa_attn_fwd (flags 0), but its scratch (QK-norm / VE-mix
 * outputs and the status word) lives in one fixed array of
 * SWA_NOALLOC_SCRATCH_BYTES of device memory inside the library. The pages
 * have no counterpart of this call; it exists for callers that cannot
 * allocate device memory at the point where they run the attention: a
 * plug-in whose host framework owns every allocation, a service that must not
 * grow its memory after start-up, or a latency-critical path that cannot
 * afford cudaMalloc's implicit device synchronisation.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 *     routine. The array is part of the library's device code, so every GPU
 *     that loads the library holds it until the process exits.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current), and a call looks it up again
 *     when the calling thread's current CUDA context is not the one of that
 *     lookup (after cudaDeviceReset, or under a context the caller made
 *     current); make the first call on a device, and the first after such a
 *     change, before any stream capture begins.
 *   - Problems whose forward workspace (swa_attn_workspace_size(p, 0)) is
 *     larger than the array are rejected with SWA_ERR_WORKSPACE, launching
 *     nothing.
 *   - Every call, from any stream or thread, shares the one array and it
 *     keeps the last call's contents: calls that overlap on the GPU race and
 *     corrupt each other's results; order them (same stream or events).
 *     Nothing in it has to start at zero (the prologue writes every value the
 *     forward reads).
 *   - Device-side checks are not reported: when one fires (a token id outside
 *     [0, vocab), a pipeline wait that ran out) this call still returns
 *     SWA_OK, and o and lse are undefined. Callers that need to see those
 *     checks use swa_attn_fwd with a workspace and swa_attn_check_status.
 */
#define SWA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
swa_status swa_attn_fwd_noalloc(const swa_params* p, const void* q, const void* k,
                                const void* v, const float* gq, const float* gk, const void* ve,
                                const int32_t* tok, const float* ve_gate, void* o, float* lse,
                                void* stream);

/*
 * One training step of one attention call with every tensor in HOST memory:
 * the inputs are copied host -> device, the forward and the backward run
 * (the backward reusing the forward's QK-norm / VE-mix outputs), and o, lse
 * and the gradients are copied device -> host, all enqueued on `stream` in
 * that order; the call returns without waiting (synchronize the stream, or
 * record an event after it, before reading the outputs). The pages have no
 * counterpart of this call: it is the library's end-to-end path for callers
 * whose data lives on the host.
 *   q, k, v, dO, gq, gk, ve, tok, ve_gate   host inputs, the layouts and
 *                  meanings of swa_attn_fwd / swa_attn_bwd (gq, gk, ve, tok,
 *                  ve_gate may be NULL as there)
 *   o, lse, dq, dk, dv, dgq, dgk, dve        host outputs, as there
 *                  (dgq, dgk, dve may be NULL: not computed, not copied)
 *   ex             as for the _ex calls; its rotary tables and gate weights
 *                  are DEVICE pointers (not copied)
 *   device_buffer  device memory of at least swa_attn_step_host_size(p)
 *                  bytes, 256-byte aligned, passed to swa_attn_workspace_init
 *                  once before its first use; it holds the attention's
 *                  workspace (so swa_attn_check_status reads it) and the
 *                  device copies of every input and output. Reusing it on the
 *                  same stream is safe (stream order); on several streams at
 *                  once, give each its own buffer.
 * Copies from and to pageable host memory make the CUDA runtime stage them
 * and block the calling thread; page-locked (pinned) host buffers let them
 * run asynchronously and overlap work on other streams. Each copy is one
 * cudaMemcpyAsync. Errors: SWA_ERR_INVALID_ARG for a NULL required pointer
 * or a misaligned device buffer, SWA_ERR_WORKSPACE for a buffer too small,
 * both before anything is enqueued; then those of swa_attn_fwd and
 * swa_attn_bwd, and SWA_ERR_CUDA when a copy cannot be enqueued (the outputs
 * are then undefined).
 */
size_t swa_attn_step_host_size(const swa_params* p);
swa_status swa_attn_step_host(const swa_params* p, const swa_extras* ex, const void* q,
                              const void* k, const void* v, const float* gq, const float* gk,
                              const void* ve, const int32_t* tok, const float* ve_gate,
                              const void* dO, void* o, float* lse, void* dq, void* dk, void* dv,
                              float* dgq, float* dgk, float* dve, void* device_buffer,
                              size_t device_bytes, void* stream);

/*
 * The whole attention block around the core: the block's pre-norm, the four
 * bias-free projections c_q, c_k, c_v, c_proj and the residual
 * (autoresearch Administrator & Developer Guide §8.2.1 model table,
 * "Pre-norm + residual": x = x + attn(norm(x)); train.py walkthrough post,
 * model paragraph: RMSNorm on the block inputs):
 *   xn  = x / sqrt(mean_c(x^2) + eps)               (no gain; eps of swa_params)
 *   q   = xn wq^T, k = xn wk^T, v = xn wv^T         (viewed as [B, T, H, d])
 *   o   = the attention of swa_attn_fwd_ex on (q, k, v), with the learned
 *         gate (if any) reading the first gate_ch channels of xn
 *   out = x + o wo^T                                (o viewed as [B, T, Hq*d])
 * Weights use the torch.nn.Linear layout [out_features][in_features], elem:
 *   wq [Hq*d][C], wk and wv [Hkv*d][C], wo [C][Hq*d];  x, out, dout, dx
 *   [B, T, C] elem;  weight gradients dwq, dwk, dwv, dwo fp32, same shapes
 *   as the weights (overwritten; NULL skips one).
 * C (the model width) is a multiple of 8, at most 65536; B*T < 2^31.
 * Extras: rotary tables and gate_w / gate_ch / d_gate_w as for the _ex
 * calls; gate_x and d_gate_x must be NULL (the block supplies the gate's
 * input and adds the gradient of the channels it read into dx); gate_ch <= C.
 * As in the attention calls, the gate applies on value-embedding calls only
 * (ve != NULL); without a VE table it is ignored and d_gate_w is not written.
 * The projections run on this library's own GEMM kernels (tcgen05 tensor
 * cores with bf16 operands and fp32 accumulation in the bf16 library, fp32
 * SIMT in the fp32 debug library); the weight gradients split B*T over
 * several CTAs and add their fp32 partial sums into dwq, dwk, dwv and dwo,
 * so their last bits can differ from run to run. The workspace
 * (swa_block_workspace_size) holds the attention's workspace first (so
 * swa_attn_check_status reads the block workspace too),
 * then the forward's saved tensors (xn, q, k, v, o, lse) and a transposed
 * copy of the rotary tables; swa_block_bwd needs the workspace that
 * swa_block_fwd filled for the same inputs.
 */
typedef struct {
  int C;              /* model width: channels of x                         */
  const void* wq;     /* [Hq*d][C]  elem                                     */
  const void* wk;     /* [Hkv*d][C] elem                                     */
  const void* wv;     /* [Hkv*d][C] elem                                     */
  const void* wo;     /* [C][Hq*d]  elem                                     */
} swa_block_weights;

/* Bytes of workspace for swa_block_fwd (for_backward = 0) or for the pair
 * swa_block_fwd + swa_block_bwd (for_backward = 1); 0 for invalid arguments. */
size_t swa_block_workspace_size(const swa_params* p, int C, int for_backward);

/* out = x + c_proj(attention(c_q, c_k, c_v of the normed x)). */
swa_status swa_block_fwd(const swa_params* p, const swa_extras* ex, const swa_block_weights* w,
                         const void* x, const float* gq, const float* gk, const void* ve,
                         const int32_t* tok, void* out, void* workspace, size_t ws_bytes, void* stream);

/* Gradients of <out, dout>: dx (elem, including the residual's dout), the
 * weight gradients, and the attention's dgq, dgk, dve, d_gate_w as in
 * swa_attn_bwd_ex. */
swa_status swa_block_bwd(const swa_params* p, const swa_extras* ex, const swa_block_weights* w,
                         const void* x, const float* gq, const float* gk, const void* ve,
                         const int32_t* tok, const void* dout, void* dx, float* dwq, float* dwk,
                         float* dwv, float* dwo, float* dgq, float* dgk, float* dve, void* workspace,
                         size_t ws_bytes, void* stream);

/*
 * Synchronises `stream`, reads the workspace status word, clears it, and
 * returns SWA_OK, SWA_ERR_TIMEOUT or SWA_ERR_DEVICE_CHECK (timeout wins).
 * After a timeout it also drops the record of a zeroed dQ accumulator (a
 * forward that gave up may not have zeroed it), so the next backward clears
 * the accumulator itself.
 */
swa_status swa_attn_check_status(void* workspace, void* stream);

/*
 * Window of layer `layer` of an `n_layer` stack under a window pattern of
 * 'S' (sliding, window T/2) and 'L' (full) characters, e.g. "SSSL": the
 * layer's character is pattern[layer % strlen(pattern)] and the last layer is
 * always full (post, model paragraph; Guide §3.4). Returns T/2 or -1; -2 on
 * invalid arguments (NULL/empty pattern, a character other than S/L, layer
 * out of [0, n_layer)).
 */
int swa_sssl_window(int layer, int n_layer, const char* pattern, int T);

/*
 * 1 if layer `layer` of an `n_layer` stack mixes value embeddings into v:
 * alternating layers, the last always included (Guide §8.2.1, has_ve); 0 if
 * not; -1 on invalid arguments.
 */
int swa_has_ve(int layer, int n_layer);

/* Static, human-readable text of a status code. */
const char* swa_strerror(swa_status s);

/* Static text naming the build: element type and kernel family. */
const char* swa_build_info(void);

#ifdef __cplusplus
}
#endif

#endif /* SWA_ATTN_H */
