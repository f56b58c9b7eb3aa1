/*
 * hla.h — C ABI of the GB300 Lightning Attention RNN mixer library (libhla.so).
 *
 * The mixer is the RNN layer of HypeNet, arXiv 2601.22156 ("Hybrid Linear
 * Attention Done Right"), Appendix A, Eq. 18, with the fixed per-head forget
 * rate of Eq. 19.  Per sequence b and head h, with row vectors and a state
 * S in R^{d x d} (d_k rows, d_v columns):
 *
 *   q_t  = Norm(q_raw_t),  k_t = Norm(k_raw_t)          QK-RMSNorm (Eq. 12)
 *   q~_t = RoPE_p(q_t),    k~_t = RoPE_p(k_t) / sqrt(d)  HyPE RoPE in RNN layers
 *   S_t  = gamma_h S_{t-1} + k~_t^T v_t
 *   o_t  = q~_t S_t
 *   y_t  = Norm(o_t) * sigmoid(gate_t)                   output norm + gate (Eq. 14)
 *
 * Norm is RMSNorm x / sqrt(mean(x^2) + norm_eps) with unit weight.  RoPE uses
 * the rotate-half pairing (x_i, x_{i+d/2}), i < d/2, rotated by the angle
 * p * rope_base^(-2i/d), at position p = pos_offset + t (0-based).  The
 * mixer entry points take q, k, v as the projected per-head rows and gate as
 * the pre-sigmoid logit x W_z; the projections themselves (x W_{q,k,v,z} with
 * the feature map fused, and the output projection W_o) are separate entry
 * points at the end of this header.  Every RNN head owns its own k and v (the
 * paper's GQA-to-MHA decoupling, Eq. 13), so q, k, v and gate all carry H heads.
 *
 * Conventions shared by every entry point
 *   - Activations q, k, v, gate, y, dy, dq, dk, dv, dgate: device memory,
 *     [B, T, H, d] contiguous (d fastest), element type shape->dtype
 *     (fp32 or bf16).  o (optional): fp32 [B, T, H, d].
 *   - States: device memory, fp32 [B, H, d, d], d_v index fastest.
 *   - gamma: HOST memory, fp32 [H], every value in (0, 1].  It is read during
 *     the call and copied into the launch parameters (so a captured CUDA graph
 *     keeps the values it saw at capture time).
 *   - Every device pointer must be 16-byte aligned.  The caller owns and
 *     allocates every buffer, including the workspace; the library never
 *     allocates, frees or synchronizes.  All work is enqueued on `stream`
 *     (NULL = the legacy default stream) of the current device.
 *   - Arguments are validated before anything is launched: a bad argument
 *     returns HLA_ERR_INVALID_ARG / HLA_ERR_UNSUPPORTED / HLA_ERR_WORKSPACE and
 *     enqueues nothing.  HLA_ERR_CUDA means a launch was rejected by the CUDA
 *     runtime; faults during execution surface at the caller's next sync.
 *   - No C++ exception crosses the ABI.  There is no mutable global state
 *     (the one exception is hla_prefill_noalloc's shared scratch array, see
 *     there): calls on different streams may run concurrently from several
 *     threads.
 *   - Supported: d_k == d_v in {64, 128}; chunk in {64, 128}; B >= 0;
 *     T >= 0 (T == 1 for hla_decode_step); 1 <= H <= 256; 0 <= pos_offset
 *     and pos_offset + T < 2^62.
 *   - An empty batch or sequence (B == 0 or T == 0) computes nothing: the
 *     pointers of tensors with no elements may be NULL, hla_prefill leaves
 *     state_out = state_in (zeros when state_in is NULL) and
 *     hla_prefill_backward leaves dstate_in = dstate_out (zeros when
 *     dstate_out is NULL); the workspace status word is still cleared.
 */
#ifndef HLA_H_
#define HLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HLA_ABI_VERSION 7

typedef enum {
  HLA_OK = 0,
  HLA_ERR_INVALID_ARG = 1, /* NULL/misaligned pointer, non-positive size, bad gamma/eps/base */
  HLA_ERR_UNSUPPORTED = 2, /* valid but not implemented here (d, chunk, dtype, H range)      */
  HLA_ERR_WORKSPACE = 3,   /* workspace pointer NULL or ws_bytes below the required size     */
  HLA_ERR_CUDA = 4,        /* the CUDA runtime rejected a launch or an attribute call        */
  HLA_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up (read from the status word) */
} hla_status;

typedef enum { HLA_F32 = 0, HLA_BF16 = 1 } hla_dtype;

/* Problem description shared by all entry points. */
typedef struct {
  int32_t B;          /* sequences                                              */
  int32_t T;          /* tokens per sequence in this call (1 for a decode step)  */
  int32_t H;          /* heads                                                  */
  int32_t dk;         /* key/query head dim d_k                                 */
  int32_t dv;         /* value head dim d_v (must equal dk)                     */
  int32_t chunk;      /* token tile of the chunked prefill: 64 or 128           */
  int32_t dtype;      /* hla_dtype of q, k, v, gate, y and the gradients        */
  int32_t decode_split; /* hla_decode_step: CTAs per (sequence, head), see there;  */
                       /* 0 for every other entry point                         */
  int64_t pos_offset; /* RoPE position of token 0 (prefill and backward)        */
  double rope_base;   /* RoPE base theta (1e6 for HypeNet-2B/5B/9B, Table 6)    */
  float norm_eps;     /* RMSNorm epsilon of the QK norms and the output norm    */
  int32_t passes;     /* hla_prefill / hla_prefill_features, tensor-core path:  */
                      /* 0 = the library's choice, 1 = one launch, 3 = three     */
                      /* (see hla_prefill); 0 for every other entry point       */
} hla_shape;

typedef void *hla_stream; /* a cudaStream_t */

/*
 * Optional per-pass tracing (the last argument of hla_prefill and
 * hla_prefill_backward; NULL = none).  events[i] are caller-created
 * cudaEvent_t handles; the library records events[i] on `stream` right before
 * its i-th kernel launch and events[n_passes] after the last one, for every
 * i < count.  Elapsed times between consecutive events are the device times
 * of the individual passes.  The library creates, destroys and synchronizes
 * nothing.
 *
 * test_wait_cycles exercises the bounded waits (testing only; 0 in normal
 * use): when > 0, the first wait of every output-pass CTA of a tensor-core
 * hla_prefill (the issuing thread waiting for the workers' feature map of
 * the first tile) gives up after that many SM clock cycles.  The CTA then
 * issues nothing more, lets every copy and MMA it issued complete, runs its
 * remaining waits out on their normal budget and leaves; the call's status
 * word reads non-zero (HLA_ERR_TIMEOUT) and its outputs are not valid.  The
 * device and the stream stay usable.
 */
#define HLA_TRACE_MAX 16
typedef struct {
  void *events[HLA_TRACE_MAX];
  int32_t count;
  int64_t test_wait_cycles;
} hla_trace;

/* ABI version of the loaded library (HLA_ABI_VERSION). */
int hla_abi_version(void);

/* Static, human-readable name of a status code. */
const char *hla_status_string(hla_status status);

/*
 * Eq. 19 forget rates: gamma_out[h] = exp(-2^(-8(h+1)/H)) for the 0-based
 * head h (the paper's head h+1), evaluated in fp64 and rounded to fp32.
 * Host memory; returns HLA_ERR_INVALID_ARG for H < 1 or a NULL pointer.
 */
hla_status hla_gamma_schedule(int32_t H, float *gamma_out);

/* Device workspace bytes hla_prefill needs for this shape (0 on a bad shape). */
size_t hla_prefill_workspace_size(const hla_shape *shape);

/*
 * Kernels one hla_prefill (or hla_prefill_features) call with this shape and
 * gamma (HOST fp32 [H]) launches, and one hla_prefill_backward call (with a
 * forward workspace, with_fwd_ws != 0, or without); -1 on a bad argument.
 * For profiling and graph planning; the memsets of the status word are not
 * kernels and are not counted.
 */
int32_t hla_prefill_launches(const hla_shape *shape, const float *gamma);
int32_t hla_backward_launches(const hla_shape *shape, const float *gamma, int32_t with_fwd_ws);

/*
 * Bytes of the features hla_prefill can save for hla_prefill_backward (its
 * `saved` argument).  Non-zero only for bf16 at d = 128 (the tensor-core
 * path); 0 on a bad shape or where saving is not supported.  Layout, all
 * device memory, B, T, H of the shape, d = 128:
 *   q~   fp16 [B, T, H, d]   RoPE(Norm(q))            at byte 0
 *   k~   fp16 [B, T, H, d]   RoPE(Norm(k)) / sqrt(d)  at byte 2 B T H d
 *   fp32 [4, B, H, T]                                  at byte 4 B T H d:
 *        [0] 1 / RMS(q_t), [1] 1 / RMS(k_t)   (RMS(x) = sqrt(mean(x^2) + eps))
 *        [2] q~_t . k~_t, accumulated in fp32 before the fp16 rounding
 *        [3] 1 / RMS(o_t), the output norm's scale (written by the output pass
 *            of hla_prefill or hla_prefill_features; hla_project_in leaves it)
 * Total B T H (4 d + 16) bytes.
 */
size_t hla_saved_bytes(const hla_shape *shape);

/*
 * Forward over T tokens (prefill), Eq. 18 for every (b, h, t).
 *   q, k, v, gate  in:  [B, T, H, d], shape->dtype, raw (pre-norm, pre-RoPE,
 *                       pre-sigmoid)
 *   gamma          in:  HOST fp32 [H]
 *   state_in       in:  fp32 [B, H, d, d] state before token 0; NULL = zeros
 *   state_out      out: fp32 [B, H, d, d] state after token T-1; NULL = skip;
 *                       may be the same pointer as state_in
 *   y              out: [B, T, H, d], shape->dtype
 *   o              out: fp32 [B, T, H, d] mixer output before the output
 *                       norm; NULL = skip
 *   ws, ws_bytes   device scratch of at least hla_prefill_workspace_size()
 *                  bytes; its contents on entry are ignored.  Its last 256
 *                  bytes hold a uint32 device status word, cleared by the
 *                  call: non-zero after the call completes means a bounded
 *                  device-side wait gave up (HLA_ERR_TIMEOUT) and the outputs
 *                  of the affected segments are not valid
 *   trace          optional pass events (see hla_trace); NULL = none
 *   saved          out: optional, hla_saved_bytes() bytes of device memory;
 *                  the call also writes the features the backward needs
 *                  there (layout at hla_saved_bytes), so that
 *                  hla_prefill_backward can read them instead of recomputing
 *                  the q/k feature map.  NULL = skip.  Only bf16 at d = 128
 *                  can save: elsewhere a non-NULL pointer returns
 *                  HLA_ERR_UNSUPPORTED.  With no rows (B == 0 or T == 0)
 *                  nothing is written.  o and the state are the same with
 *                  and without it; y too up to its last bf16 bit: saving,
 *                  the gate's sigmoid is taken as 1 / (1 + 2^(-z log2 e)),
 *                  which stays positive down to z ~ -87 so that the backward
 *                  can divide y by it again (hla_prefill_backward's y),
 *                  where without saving it is 0.5 + 0.5 tanh(z / 2).
 * The output of token t depends on all tokens <= t of its sequence and on
 * state_in; sequences and heads are independent.
 *
 * Launches.  The T axis of each (sequence, head) is cut into segments that
 * run as separate CTAs; each needs the state entering it.  With
 * shape->passes == 3 a local-state pass sums each segment's own tokens, a
 * scan over the segments chains those sums into the entering states, and the
 * output pass runs from them (plus a partial-sum kernel where a head's sums
 * are split in pieces).  With shape->passes == 1 everything is one launch:
 * each output CTA first sums the tokens before its segment that are still
 * within the decay horizon (weights gamma^m whose tail beyond it sums to at
 * most 2^-40; every token before it when gamma = 1) on top of gamma^t0
 * state_in, then runs its segment; no CTA waits for another.  Both write the
 * state entering every segment to the workspace.  0 lets the library choose:
 * three passes (measured faster at every workload of this library; one launch
 * saves the 0.1 ms of the local-state pass and the scan at 512K tokens but
 * costs the output kernel more).  The fp32 CUDA-core path (fp32 or d = 64)
 * always runs three passes.
 */
hla_status hla_prefill(const hla_shape *shape, const void *q, const void *k, const void *v,
                       const void *gate, const float *gamma, const float *state_in,
                       float *state_out, void *y, float *o, void *ws, size_t ws_bytes,
                       hla_stream stream, const hla_trace *trace, void *saved);

/*
 * hla_prefill from features instead of raw q and k: the layer whose input
 * projection ran through hla_project_in (Appendix A, Eq. 18; the feature map
 * RMSNorm + RoPE is already applied there).
 *   features  in/out: hla_saved_bytes(shape) bytes in the layout documented
 *                 there (fp16 q~ and k~, fp32 1/RMS(q), 1/RMS(k), q~ . k~), as
 *                 written by hla_project_in or by an hla_prefill `saved`; the
 *                 call writes its fourth scalar plane (1/RMS(o)) and reads the
 *                 rest
 *   v, gate, gamma, state_in, state_out, y, o, ws, ws_bytes, trace:
 *                 as for hla_prefill (the same workspace size)
 * Tensor-core path only: bf16 at d = 128, else HLA_ERR_UNSUPPORTED.  The
 * result equals hla_prefill on the raw q and k that produced the features, up
 * to the rounding of q~ and k~ to fp16, which hla_prefill applies as well.
 * The same `features` buffer can then be passed to hla_prefill_backward as its
 * `saved` argument (with q = k = NULL).
 */
hla_status hla_prefill_features(const hla_shape *shape, void *features, const void *v,
                                const void *gate, const float *gamma, const float *state_in,
                                float *state_out, void *y, float *o, void *ws, size_t ws_bytes,
                                hla_stream stream, const hla_trace *trace);

/*
 * hla_prefill for callers that cannot allocate device memory.  The paper has
 * no counterpart to this entry point; it exists for deployments where the
 * caller may not call cudaMalloc: a plugin inside an engine that owns all
 * device memory through its own pool, a serving loop that must not allocate
 * (or risk an allocation failure or an implicit synchronization) once it is
 * running, or a certified build that forbids allocation after start-up.
 *
 * Same arguments and results as hla_prefill, minus the workspace: the
 * per-segment states live in a fixed scratch array of
 * HLA_NOALLOC_SCRATCH_BYTES inside the library's own device memory, which
 * every GPU that loads the library holds until the process exits.  It runs
 * the fp32 CUDA-core kernels (every dtype and d).
 *   - Limit: B * H * d * d * 4 bytes (one fp32 state per sequence and head)
 *     must fit in HLA_NOALLOC_SCRATCH_BYTES, i.e. B * H <= 512 at d = 128;
 *     larger problems return HLA_ERR_WORKSPACE before anything is launched.
 *     Within the limit the T axis is cut into fewer, longer segments when
 *     needed, so results match hla_prefill up to fp32 rounding; near the
 *     limit (B * H close to 512 at d = 128) that is a single segment per
 *     (sequence, head), which leaves the T axis without parallelism.
 *   - Set-up: the first call on a device looks up that device's address of
 *     the scratch array (cudaGetSymbolAddress, with the device current) and
 *     caches it.  Under CUDA's lazy module loading (the default) that first
 *     call is also when the runtime commits the array's device memory and
 *     loads the kernels it runs, so it is the one call that makes the runtime
 *     reserve device memory.  An empty call (B == 0 or T == 0, which may pass
 *     NULL tensors) performs that set-up and launches nothing: make it once
 *     per device at start-up, before a memory pool claims the device, and
 *     before any stream capture.  Every later call allocates nothing.  (With
 *     CUDA_MODULE_LOADING=EAGER the runtime commits it all when the library
 *     loads.)  The cached address belongs to the device's context: after
 *     cudaDeviceReset the entry point must not be called again in that process.
 *   - Sharing: every call on a device uses the same scratch array, which keeps
 *     the last call's contents (the first pass overwrites all of it, so
 *     nothing needs clearing).  Calls that overlap on the GPU race on it:
 *     the caller must not run two of them at the same time on one device
 *     (different streams or threads included).
 */
#define HLA_NOALLOC_SCRATCH_BYTES (32u << 20)
hla_status hla_prefill_noalloc(const hla_shape *shape, const void *q, const void *k,
                               const void *v, const void *gate, const float *gamma,
                               const float *state_in, float *state_out, void *y, float *o,
                               hla_stream stream);

/*
 * One decode step: Eq. 18 for a single new token per sequence (shape->T must
 * be 1).  The state is read once and written once.
 *   shape->decode_split  how many CTAs share one (sequence, head): 1 = one CTA
 *                       owns the whole d x d state; 2, 4 or 8 = a thread-block
 *                       cluster of that many CTAs, each owning d / split of
 *                       the state's columns (the output RMSNorm's sum of
 *                       squares is reduced across the cluster), which spreads
 *                       a small batch over more SMs; 0 = chosen by the library
 *                       (one CTA: a batch-1 step is bound by latency, and the
 *                       split gains only while the state sits in L2).  The new
 *                       state is bit-identical for every split; o and y differ
 *                       only by the order of the q~ S sum.  Any other value
 *                       returns HLA_ERR_INVALID_ARG.
 *   q, k, v, gate  in:  [B, 1, H, d], shape->dtype
 *   gamma          in:  HOST fp32 [H]
 *   pos            in:  device int64 [B], RoPE position of each sequence's
 *                       token; NULL = every sequence at shape->pos_offset
 *   state_in       in:  fp32 [B, H, d, d] (required)
 *   state_out      out: fp32 [B, H, d, d]; may equal state_in (in-place)
 *   y              out: [B, 1, H, d], shape->dtype
 *   o              out: fp32 [B, 1, H, d] before the output norm; NULL = skip
 */
hla_status hla_decode_step(const hla_shape *shape, const void *q, const void *k, const void *v,
                           const void *gate, const float *gamma, const int64_t *pos,
                           const float *state_in, float *state_out, void *y, float *o,
                           hla_stream stream);

/* Device workspace bytes hla_prefill_backward needs (0 on a bad shape). */
size_t hla_backward_workspace_size(const hla_shape *shape);

/*
 * Backward of hla_prefill: gradients of L = <dy, y> + <dstate_out, state_out>
 * with respect to the raw inputs (the chain rule through Eq. 18; gamma is a
 * fixed constant of the method, Eq. 19, and gets no gradient).
 *   q, k, v, gate, gamma, state_in   the forward call's inputs (state_in NULL = zeros)
 *   dy          in:  [B, T, H, d], shape->dtype, gradient of y
 *   dstate_out  in:  fp32 [B, H, d, d] gradient of state_out; NULL = zeros
 *   dq, dk, dv, dgate  out: [B, T, H, d], shape->dtype
 *   dstate_in   out: fp32 [B, H, d, d] gradient of state_in; NULL = skip
 *   ws, ws_bytes     device scratch of hla_backward_workspace_size() bytes;
 *                    as for hla_prefill, its last 256 bytes hold the device
 *                    status word (non-zero after completion: a bounded wait
 *                    gave up and the gradients are not valid)
 *   trace            optional pass events (see hla_trace); NULL = none
 *   fwd_ws           optional: the workspace of an hla_prefill call with the
 *                    same shape, q, k, v, gamma and state_in, already enqueued
 *                    before this call (same stream, or ordered by the caller)
 *                    and not reused since.  That call left the state entering
 *                    every segment in it, and the backward reads them instead
 *                    of recomputing them (it skips two of its passes).  Read
 *                    only.  NULL = recompute.  Passing a workspace that does
 *                    not hold those states gives wrong gradients; nothing can
 *                    check it.
 *   saved            optional: the `saved` buffer of an hla_prefill call with
 *                    the same shape, q and k, or the `features` of
 *                    hla_project_in / hla_prefill_features, enqueued before
 *                    this call and not reused since.  The backward passes read
 *                    q~, k~ and the norms from it instead of recomputing them,
 *                    and raw q and k are not read: they may be NULL.  Read
 *                    only.  NULL = recompute.  HLA_ERR_UNSUPPORTED unless bf16
 *                    at d = 128.  Gradients agree with the
 *                    recomputing path up to the fp16 rounding of q~ and k~
 *                    (the RMSNorm backward then starts from the rounded
 *                    features).
 *   y                optional, with `saved` only (HLA_ERR_INVALID_ARG without):
 *                    the forward's output y ([B, T, H, d], shape->dtype) of the
 *                    hla_prefill / hla_prefill_features call that wrote `saved`
 *                    (and the fourth scalar plane of it, 1/RMS(o)).  The dq pass
 *                    then takes the normalized output n = y / sigmoid(gate)
 *                    (the forward's own sigmoid, so the division undoes its
 *                    gating up to the rounding of y) and 1/RMS(o) from there
 *                    instead of recomputing o: three of its seven tile
 *                    products and the causal mask drop out.  Where the
 *                    forward's sigmoid was 0 (gate below about -87) n is taken
 *                    as 0, which the recomputing path does not need.  A y
 *                    that is not that call's output gives wrong gradients;
 *                    nothing can check it.  NULL = recompute o.
 * Without y, o and the per-chunk states inside a segment are recomputed;
 * hla_prefill stores neither.
 */
hla_status hla_prefill_backward(const hla_shape *shape, const void *q, const void *k,
                                const void *v, const void *gate, const float *gamma,
                                const float *state_in, const void *dy, const float *dstate_out,
                                void *dq, void *dk, void *dv, void *dgate, float *dstate_in,
                                void *ws, size_t ws_bytes, hla_stream stream,
                                const hla_trace *trace, const void *fwd_ws, const void *saved,
                                const void *y);

/*
 * The hybrid's other mixer: causal softmax attention without positional
 * encoding, with the position-dependent logit scale of arXiv 2601.22156,
 * Section 5.1 "Attention Logits Scaling" (Eq. 11) and Appendix A "Attention
 * Layers" (Eq. 17), followed by the same output norm and gate:
 *
 *   s_t  = log_a(t + a)   (t the paper's 1-based position: here p + 1, p = pos_offset + t)
 *   q~_t = s_t q_t / sqrt(d)
 *   o_t  = sum_{i <= t} softmax_i(q~_t . k_i) v_i     (keys: this call's tokens 0..t)
 *   y_t  = Norm(o_t) * sigmoid(gate_t)
 *
 * Query head h reads key/value head h / (Hq / Hkv) (grouped-query attention).
 * No QK-norm is applied (a base model's QK-norm is the caller's).
 */
typedef struct {
  int32_t B;          /* sequences                                               */
  int32_t T;          /* tokens per sequence                                     */
  int32_t Hq;         /* query heads                                             */
  int32_t Hkv;        /* key/value heads; must divide Hq                         */
  int32_t d;          /* head dim (128)                                          */
  int32_t dtype;      /* hla_dtype of q, k, v, gate and y (HLA_BF16)             */
  int64_t pos_offset; /* position of token 0                                     */
  double a;           /* the logit-scale base a > 1 (500 / 600 / 900, Table 6)   */
  float norm_eps;     /* RMSNorm epsilon of the output norm                      */
} hla_attn_shape;

/* Device workspace bytes hla_attention_prefill needs (its status word); 0 on a
 * bad shape. */
size_t hla_attention_workspace_size(const hla_attn_shape *shape);

/*
 * Causal attention over T tokens.  Tensor cores only: bf16 at d = 128 (other
 * shapes return HLA_ERR_UNSUPPORTED); 1 <= Hkv, Hkv divides Hq, Hq <= 256.
 *   q, gate   in:  [B, T, Hq, d] bf16
 *   k, v      in:  [B, T, Hkv, d] bf16
 *   y         out: [B, T, Hq, d] bf16
 *   o         out: fp32 [B, T, Hq, d] attention output before the norm; NULL = skip
 *   ws, ws_bytes   device scratch of hla_attention_workspace_size() bytes: a
 *                  uint32 status word, cleared by the call, non-zero after it
 *                  completes when a bounded device-side wait gave up
 * Pointer, stream and error conventions as above.
 */
hla_status hla_attention_prefill(const hla_attn_shape *shape, const void *q, const void *k,
                                 const void *v, const void *gate, void *y, float *o, void *ws,
                                 size_t ws_bytes, hla_stream stream);

/*
 * The projections around the RNN mixer (Appendix A, Eq. 18, "RNN Layers"):
 * q_t = Norm(x_t W_q), k_t = Norm(x_t W_k), v_t = x_t W_v,
 * z_t = sigmoid(x_t W_z) and y_t = (Norm(o_t) . z_t) W_o^T, with W_q, W_k, W_v,
 * W_z, W_o in R^{D x d} per head (D the model width).  Tensor-core GEMMs with
 * bf16 operands and fp32 accumulation.  Each call's workspace holds only its
 * device status word (hla_project_workspace_size() bytes): cleared by the
 * call, non-zero after it completes when a bounded device-side wait gave up.
 */
size_t hla_project_workspace_size(void);

/*
 * Input projection of every head at once, the mixer's feature map fused into
 * the epilogue: from the fp32 products x W_q,h and x W_k,h it writes the
 * features hla_prefill_features and hla_prefill_backward read (q~, k~ as
 * fp16, 1/RMS(q), 1/RMS(k) and the fp32 q~ . k~); raw q and k never reach
 * memory.  v = x W_v,h and the gate logit x W_z,h are written as bf16.
 *   shape     B, T, H, dk = dv = 128, dtype HLA_BF16, pos_offset, rope_base and
 *             norm_eps as for hla_prefill (chunk 64 or 128, decode_split 0)
 *   d_model   D, a positive multiple of 64
 *   x         in:  bf16 [B, T, D]
 *   w_qkvz    in:  bf16 [H, 4, d, D]: for head h, the transposes of the paper's
 *                  W_q, W_k, W_v, W_z in that order (row c of w_qkvz[h][j] is
 *                  column c of W_j,h: a linear layer's output-major weight)
 *   features  out: hla_saved_bytes(shape) bytes (layout there; the fourth
 *             scalar plane, 1/RMS(o), is left for hla_prefill_features)
 *   v, gate   out: bf16 [B, T, H, d]
 * HLA_ERR_UNSUPPORTED unless bf16 at d = 128 with D % 64 == 0 and B T < 2^31.
 */
hla_status hla_project_in(const hla_shape *shape, int32_t d_model, const void *x,
                          const void *w_qkvz, void *features, void *v, void *gate, void *ws,
                          size_t ws_bytes, hla_stream stream);

/*
 * Output projection: out[m] = u[m] W_o^T for M rows, u the gated, normalized
 * mixer rows of all heads side by side (hla_prefill's y viewed as [M, H d]).
 *   u     in:  bf16 [M, n_in], n_in = H d a positive multiple of 64
 *   w_o   in:  bf16 [d_model, n_in]: the paper's W_o of every head side by
 *              side (column h d + c belongs to head h)
 *   out   out: bf16 [M, d_model], d_model a positive multiple of 128
 */
hla_status hla_project_out(int64_t M, int32_t n_in, int32_t d_model, const void *u,
                           const void *w_o, void *out, void *ws, size_t ws_bytes,
                           hla_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* HLA_H_ */
