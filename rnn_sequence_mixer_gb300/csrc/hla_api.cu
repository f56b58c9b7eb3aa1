// hla_api.cu — the extern "C" entry points of libhla.so: argument validation,
// the segment plan, workspace carving and kernel dispatch.  Nothing here
// allocates, frees or synchronizes.
#include <math.h>
#include <algorithm>
#include <string.h>

#include <new>

#include "hla_internal.cuh"

namespace hla {

// decode_split.cu: the decode step with the state's columns split over a
// cluster of `split` (2, 4 or 8) CTAs per (sequence, head).
cudaError_t launch_decode_split(const MixerParams &P, int dtype, int split, cudaStream_t st);

namespace {

// The segment plan sizes its grid for a GB300: 152 SMs, one resident CTA per
// SM in the tensor-core passes (each holds ~200 KB of shared memory and all
// 512 TMEM columns).
constexpr int kSMs = 152;
// Fixed cost of one segment, in tiles: the CTA's set-up, its entering state
// read from the workspace, the pipeline filling and draining, and its step in
// the fp32 scan.
constexpr int kSegOverhead = 2;

// CTAs per (sequence, head) of a decode step when the caller leaves it to the
// library: one.  Measured on a GB300, the column split did not pay with the
// state coming from HBM (B = 1, H = 16: 4.5 us per step at split 8 against
// 4.0 us) and gained at most 7% with the state already in L2 (split 4 at
// B * H <= 32; slower from B * H = 64 on): a batch-1 step is bound by latency,
// not by one SM's bandwidth.  Callers that keep the state in L2 can ask for it.
constexpr int kAutoDecodeSplit = 1;

}  // namespace

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

hla_status check_shape(const hla_shape *s, bool decode) {
  if (!s) return HLA_ERR_INVALID_ARG;
  // B = 0 or T = 0 (an empty batch or sequence) is valid: the call has nothing to compute.
  if (s->B < 0 || s->T < 0 || s->H < 1 || s->dk < 1 || s->dv < 1) return HLA_ERR_INVALID_ARG;
  if (decode ? (s->decode_split < 0 || s->decode_split > 8 || (s->decode_split & (s->decode_split - 1)))
             : s->decode_split != 0)
    return HLA_ERR_INVALID_ARG;
  if (!(s->rope_base > 0.0) || !isfinite(s->rope_base)) return HLA_ERR_INVALID_ARG;
  if (!(s->norm_eps >= 0.0f) || !isfinite(s->norm_eps)) return HLA_ERR_INVALID_ARG;
  if (s->pos_offset < 0 || s->pos_offset > (1LL << 62) - (long long)s->T) return HLA_ERR_INVALID_ARG;
  if (s->passes != 0 && (decode || (s->passes != 1 && s->passes != 3))) return HLA_ERR_INVALID_ARG;
  if (s->dtype != HLA_F32 && s->dtype != HLA_BF16) return HLA_ERR_UNSUPPORTED;
  if (s->dk != s->dv || (s->dk != 64 && s->dk != 128)) return HLA_ERR_UNSUPPORTED;
  if (s->H > kMaxHeads) return HLA_ERR_UNSUPPORTED;
  if (decode) {
    if (s->T != 1) return HLA_ERR_INVALID_ARG;
  } else if (s->chunk != 64 && s->chunk != 128) {
    return HLA_ERR_UNSUPPORTED;
  }
  // Element counts must stay well inside 64-bit and grid limits.
  long long rows = (long long)s->B * s->T * s->H;
  if (rows > (1LL << 40)) return HLA_ERR_UNSUPPORTED;
  if (s->B > 65535 || s->H > 65535) return HLA_ERR_UNSUPPORTED;
  return HLA_OK;
}

hla_status check_gamma(const float *gamma, int H) {
  if (!gamma) return HLA_ERR_INVALID_ARG;
  for (int h = 0; h < H; ++h)
    if (!(gamma[h] > 0.0f && gamma[h] <= 1.0f)) return HLA_ERR_INVALID_ARG;
  return HLA_OK;
}

hla_status need(const void *p) { return (p && aligned16(p)) ? HLA_OK : HLA_ERR_INVALID_ARG; }
hla_status maybe(const void *p) { return (!p || aligned16(p)) ? HLA_OK : HLA_ERR_INVALID_ARG; }
// A tensor with no elements may be NULL.
hla_status need_unless(bool empty, const void *p) { return empty ? maybe(p) : need(p); }

// The state a call with nothing to compute leaves behind: out = in (copied on
// the stream unless they alias), or zeros without an input; B * H states.
cudaError_t pass_state(const hla_shape &s, const float *in, float *out, cudaStream_t st) {
  if (!out || s.B == 0) return cudaSuccess;
  const size_t bytes = (size_t)s.B * s.H * s.dk * s.dv * sizeof(float);
  if (!in) return cudaMemsetAsync(out, 0, bytes, st);
  if (in == out) return cudaSuccess;
  return cudaMemcpyAsync(out, in, bytes, cudaMemcpyDeviceToDevice, st);
}

namespace {

#define HLA_TRY(x)                          \
  do {                                      \
    hla_status _s = (x);                    \
    if (_s != HLA_OK) return _s;            \
  } while (0)

#define HLA_LAUNCH(x)                                   \
  do {                                                  \
    cudaError_t _e = (x);                               \
    if (_e != cudaSuccess) return HLA_ERR_CUDA;         \
  } while (0)

// Records trace->events[i] before pass i (and after the last pass).
struct Tracer {
  const hla_trace *t;
  cudaStream_t st;
  int next = 0;
  cudaError_t mark() {
    cudaError_t e = cudaSuccess;
    if (t && next < t->count && next < HLA_TRACE_MAX && t->events[next])
      e = cudaEventRecord((cudaEvent_t)t->events[next], st);
    ++next;
    return e;
  }
};

hla_status check_trace(const hla_trace *t) {
  if (t && (t->count < 0 || t->count > HLA_TRACE_MAX || t->test_wait_cycles < 0))
    return HLA_ERR_INVALID_ARG;
  return HLA_OK;
}

}  // namespace

void fill_common(MixerParams &P, const hla_shape &s, const float *gamma) {
  memset(&P, 0, sizeof(P));
  P.B = s.B;
  P.T = s.T;
  P.H = s.H;
  P.D = s.dk;
  P.chunk = s.chunk;
  P.pos_offset = s.pos_offset;
  P.eps = s.norm_eps;
  P.kscale = (float)(1.0 / sqrt((double)s.dk));
  for (int h = 0; h < s.H; ++h) P.gamma[h] = gamma[h];
  fill_rope(P, s.dk, s.rope_base);
}

Plan make_plan(const hla_shape &s) {
  Plan p;
  p.nchunk = ceil_div(s.T, s.chunk);
  long long units = (long long)s.B * s.H;
  if (units == 0 || p.nchunk == 0) {  // empty batch or sequence: no segments
    p.nseg = 0;
    p.seg_len = s.chunk;
    return p;
  }
  // Every segment of every (b, h) is one CTA, and CTAs run in waves of kSMs.
  // Pick the segment count that minimises the time of the slowest SM,
  // waves x (tiles per segment + kSegOverhead); ties go to fewer segments.
  // Segment counts past 16 waves of CTAs only add overhead.
  const long long max_seg = std::min<long long>(p.nchunk, std::max<long long>(1, (16LL * kSMs + units - 1) / units));
  long long best_cost = -1;
  int best_cps = p.nchunk;
  for (long long nseg = 1; nseg <= max_seg; ++nseg) {
    const int cps = ceil_div(p.nchunk, nseg);
    if (ceil_div(p.nchunk, cps) != nseg) continue;  // same split as a smaller count
    const long long waves = (units * nseg + kSMs - 1) / kSMs;
    const long long cost = waves * (cps + kSegOverhead);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_cps = cps;
    }
  }
  p.nseg = ceil_div(p.nchunk, best_cps);
  p.seg_len = best_cps * s.chunk;
  return p;
}

size_t seg_bytes(const hla_shape &s, const Plan &p) {
  return (size_t)s.B * s.H * p.nseg * (size_t)s.dk * s.dv * sizeof(float);
}

// Pieces per segment the tensor-core local-state passes can write: every tile
// of a full segment (gamma = 1), an upper bound for any gamma.  0 on the
// CUDA-core path, whose local-state pass writes the segment states directly.
int part_count(const hla_shape &s, const Plan &p) {
  if (!(s.dtype == HLA_BF16 && s.dk == 128) || p.nseg == 0) return 0;
  return ceil_div(ceil_div(p.seg_len, s.chunk), kPieceTiles);
}

// The partial-sum buffer (only when a segment can have more than one piece).
size_t part_bytes(const hla_shape &s, const Plan &p) {
  const int n = part_count(s, p);
  return n > 1 ? (size_t)s.B * s.H * p.nseg * (size_t)n * s.dk * s.dv * sizeof(float) : 0;
}

// Whether a tensor-core prefill runs in one launch: only when the caller asks
// (shape->passes == 1).  Measured on a GB300 at the 512K workload, one launch
// took 2.35 ms against 2.18 ms for the three passes: the window phase in the
// output kernel costs its tile loop ~5% (the kernel runs at the 96-register
// limit of its 640 threads) and the slowest heads' windows (67 tiles) lengthen
// their CTAs, while the local-state pass and the scan it saves take 0.1 ms.
bool one_launch(const hla_shape &s, const Plan &p, const float *gamma) {
  (void)p;
  (void)gamma;
  return s.passes == 1;
}

// Whether a shape can save its features: the tensor-core path (bf16, d = 128).
bool can_save(const hla_shape &s) { return s.dtype == HLA_BF16 && s.dk == 128; }

// Bytes of the saved features of a shape: fp16 q~ and k~, and four fp32
// scalars per row.  0 where the shape cannot save them (or has no rows).
size_t saved_bytes(const hla_shape &s) {
  if (!can_save(s)) return 0;
  return saved_scalar_offset(s.B, s.T, s.H, s.dk) +
         (size_t)kSavedPlanes * s.B * s.T * s.H * sizeof(float);
}

void fill_rope_u(unsigned long long *u, int D, double base) {
  // One-entry per-thread cache: the table depends only on (base, D).
  thread_local double cached_base = -1.0;
  thread_local int cached_D = 0;
  thread_local unsigned long long cached[kMaxPairs];
  if (cached_base != base || cached_D != D) {
    const double two_pi = 6.283185307179586476925286766559;
    for (int i = 0; i < D / 2; ++i) {
      double v = pow(base, -2.0 * (double)i / (double)D) / two_pi;
      v -= floor(v);
      double scaled = ldexp(v, 64);
      cached[i] = scaled >= 18446744073709551615.0 ? 0ull : (unsigned long long)scaled;
    }
    cached_base = base;
    cached_D = D;
  }
  for (int i = 0; i < D / 2; ++i) u[i] = cached[i];
}

void fill_rope(MixerParams &P, int D, double base) { fill_rope_u(P.rope_u, D, base); }

}  // namespace hla

using namespace hla;

extern "C" {

int hla_abi_version(void) { return HLA_ABI_VERSION; }

const char *hla_status_string(hla_status s) {
  switch (s) {
    case HLA_OK: return "HLA_OK";
    case HLA_ERR_INVALID_ARG: return "HLA_ERR_INVALID_ARG: invalid argument";
    case HLA_ERR_UNSUPPORTED: return "HLA_ERR_UNSUPPORTED: unsupported shape or dtype";
    case HLA_ERR_WORKSPACE: return "HLA_ERR_WORKSPACE: workspace missing or too small";
    case HLA_ERR_CUDA: return "HLA_ERR_CUDA: CUDA launch failed";
    case HLA_ERR_TIMEOUT: return "HLA_ERR_TIMEOUT: device wait timed out";
  }
  return "HLA_ERR_UNKNOWN";
}

hla_status hla_gamma_schedule(int32_t H, float *gamma_out) {
  if (H < 1 || !gamma_out) return HLA_ERR_INVALID_ARG;
  for (int h = 0; h < H; ++h)
    gamma_out[h] = (float)exp(-pow(2.0, -8.0 * (double)(h + 1) / (double)H));
  return HLA_OK;
}

size_t hla_prefill_workspace_size(const hla_shape *s) {
  if (check_shape(s, false) != HLA_OK) return 0;
  Plan p = make_plan(*s);
  return seg_bytes(*s, p) + part_bytes(*s, p) + kStatusBytes;
}

int32_t hla_prefill_launches(const hla_shape *s, const float *gamma) {
  if (check_shape(s, false) != HLA_OK || check_gamma(gamma, s->H) != HLA_OK) return -1;
  const Plan p = make_plan(*s);
  if (p.nseg == 0) return 0;
  const bool tc = s->dtype == HLA_BF16 && s->dk == 128;
  if (!tc) return 3;
  if (one_launch(*s, p, gamma)) return 1;
  // local-state pass (every segment but the last) and its piece sums, scan, outputs
  const int state = p.nseg > 1 ? 1 + (part_count(*s, p) > 1 ? 1 : 0) : 0;
  return state + 2;
}

int32_t hla_backward_launches(const hla_shape *s, const float *gamma, int32_t with_fwd_ws) {
  if (check_shape(s, false) != HLA_OK || check_gamma(gamma, s->H) != HLA_OK) return -1;
  const Plan p = make_plan(*s);
  if (p.nseg == 0) return 0;
  const bool tc = s->dtype == HLA_BF16 && s->dk == 128;
  // forward states (local-state pass and scan) unless read from the forward's workspace
  const int sums = tc ? (p.nseg > 1 ? 1 + (part_count(*s, p) > 1 ? 1 : 0) : 0) : 1;
  const int fwd = with_fwd_ws ? 0 : sums + 1;
  // dq pass, state-gradient sums, their scan, dk/dv pass
  return fwd + 1 + sums + 1 + 1;
}

size_t hla_saved_bytes(const hla_shape *s) {
  if (check_shape(s, false) != HLA_OK) return 0;
  return saved_bytes(*s);
}

size_t hla_backward_workspace_size(const hla_shape *s) {
  if (check_shape(s, false) != HLA_OK) return 0;
  Plan p = make_plan(*s);
  size_t rows = (size_t)s->B * s->T * s->H;
  return 2 * seg_bytes(*s, p) + part_bytes(*s, p) + rows * (size_t)s->dv * sizeof(float) +
         kStatusBytes;
}

}  // extern "C"

namespace {

// hla_prefill, and hla_prefill_features (features = the saved-layout q~, k~
// and scalars given in place of raw q and k; tensor-core path only).
hla_status prefill_impl(const hla_shape *s, const void *q, const void *k, const void *features,
                        const void *v, const void *gate, const float *gamma, const float *state_in,
                        float *state_out, void *y, float *o, void *ws, size_t ws_bytes,
                        hla_stream stream, const hla_trace *trace, void *saved) {
  HLA_TRY(check_shape(s, false));
  HLA_TRY(check_gamma(gamma, s->H));
  const bool empty = s->B == 0 || s->T == 0;
  if (features) {
    HLA_TRY(need_unless(empty, features));
  } else {
    HLA_TRY(need_unless(empty, q));
    HLA_TRY(need_unless(empty, k));
  }
  HLA_TRY(need_unless(empty, v));
  HLA_TRY(need_unless(empty, gate));
  HLA_TRY(need_unless(empty, y));
  HLA_TRY(maybe(state_in));
  HLA_TRY(maybe(state_out));
  HLA_TRY(maybe(o));
  HLA_TRY(check_trace(trace));
  HLA_TRY(maybe(saved));
  if ((saved || features) && !can_save(*s)) return HLA_ERR_UNSUPPORTED;
  Plan plan = make_plan(*s);
  size_t need_ws = seg_bytes(*s, plan) + part_bytes(*s, plan) + kStatusBytes;
  if (!ws || !aligned16(ws) || ws_bytes < need_ws) return HLA_ERR_WORKSPACE;
  if (empty) {
    cudaStream_t st = (cudaStream_t)stream;
    Tracer tr{trace, st};
    HLA_LAUNCH(cudaMemsetAsync((char *)ws + need_ws - kStatusBytes, 0, sizeof(unsigned int), st));
    HLA_LAUNCH(pass_state(*s, state_in, state_out, st));
    for (int i = 0; i < 4; ++i) HLA_LAUNCH(tr.mark());
    return HLA_OK;
  }

  MixerParams P;
  fill_common(P, *s, gamma);
  P.nseg = plan.nseg;
  P.seg_len = plan.seg_len;
  P.q = q; P.k = k; P.v = v; P.g = gate;
  P.state_in = state_in;
  P.state_out = state_out;
  P.y = y;
  P.o = o;
  P.seg = (float *)ws;
  P.npart = part_count(*s, plan);
  P.part = P.npart > 1 ? (float *)((char *)ws + seg_bytes(*s, plan)) : nullptr;
  P.err = (unsigned int *)((char *)ws + need_ws - kStatusBytes);
  if (features) {  // read by both passes
    P.features_in = 1;
    P.saved = (unsigned char *)const_cast<void *>(features);
  }
  if (trace && trace->test_wait_cycles > 0) P.test_wait_cycles = trace->test_wait_cycles;
  cudaStream_t st = (cudaStream_t)stream;
  const bool tc = tc_supported(P, s->dtype);
  Tracer tr{trace, st};
  HLA_LAUNCH(cudaMemsetAsync(P.err, 0, sizeof(unsigned int), st));
  if (tc && one_launch(*s, plan, gamma)) {
    // one launch: each output CTA forms its entering state from the decay window
    P.fused = 1;
    if (!features) P.saved = (unsigned char *)saved;
    for (int i = 0; i < 3; ++i) HLA_LAUNCH(tr.mark());  // no local-state pass, no scan
    HLA_LAUNCH(launch_tc_seg_output(P, st));
    HLA_LAUNCH(tr.mark());
    return HLA_OK;
  }
  HLA_LAUNCH(tr.mark());
  // tensor cores: the last segment's local state is not summed; its output
  // pass writes state_out from the state it carries
  P.state_seg0 = 0;
  P.state_nseg = P.nseg - 1;
  HLA_LAUNCH(tc ? launch_tc_seg_state(P, st) : launch_simt_seg_state(P, s->dtype, st));
  if (!features) P.saved = (unsigned char *)saved;  // written by the output pass only
  HLA_LAUNCH(tr.mark());
  HLA_LAUNCH(launch_state_scan(P, !tc && state_out != nullptr, st));
  HLA_LAUNCH(tr.mark());
  HLA_LAUNCH(tc ? launch_tc_seg_output(P, st) : launch_simt_seg_output(P, s->dtype, st));
  HLA_LAUNCH(tr.mark());
  return HLA_OK;
}

}  // namespace

extern "C" {

hla_status hla_prefill(const hla_shape *s, const void *q, const void *k, const void *v,
                       const void *gate, const float *gamma, const float *state_in,
                       float *state_out, void *y, float *o, void *ws, size_t ws_bytes,
                       hla_stream stream, const hla_trace *trace, void *saved) {
  return prefill_impl(s, q, k, nullptr, v, gate, gamma, state_in, state_out, y, o, ws, ws_bytes,
                      stream, trace, saved);
}

hla_status hla_prefill_features(const hla_shape *s, void *features, const void *v,
                                const void *gate, const float *gamma, const float *state_in,
                                float *state_out, void *y, float *o, void *ws, size_t ws_bytes,
                                hla_stream stream, const hla_trace *trace) {
  if (!features) return HLA_ERR_INVALID_ARG;
  return prefill_impl(s, nullptr, nullptr, features, v, gate, gamma, state_in, state_out, y, o, ws,
                      ws_bytes, stream, trace, nullptr);
}

hla_status hla_decode_step(const hla_shape *s, const void *q, const void *k, const void *v,
                           const void *gate, const float *gamma, const int64_t *pos,
                           const float *state_in, float *state_out, void *y, float *o,
                           hla_stream stream) {
  HLA_TRY(check_shape(s, true));
  HLA_TRY(check_gamma(gamma, s->H));
  const bool empty = s->B == 0;
  HLA_TRY(need_unless(empty, q));
  HLA_TRY(need_unless(empty, k));
  HLA_TRY(need_unless(empty, v));
  HLA_TRY(need_unless(empty, gate));
  HLA_TRY(need_unless(empty, y));
  HLA_TRY(need_unless(empty, state_in));
  HLA_TRY(need_unless(empty, state_out));
  HLA_TRY(maybe(o));
  if (empty) return HLA_OK;
  if (pos && ((uintptr_t)pos & 7u)) return HLA_ERR_INVALID_ARG;
  // In-place is allowed; any other overlap of the two state buffers is not.
  size_t sb = (size_t)s->B * s->H * s->dk * s->dv * sizeof(float);
  const char *a = (const char *)state_in, *b = (const char *)state_out;
  if (a != b && a < b + sb && b < a + sb) return HLA_ERR_INVALID_ARG;
  MixerParams P;
  fill_common(P, *s, gamma);
  P.q = q; P.k = k; P.v = v; P.g = gate;
  P.pos = (const long long *)pos;
  P.state_in = state_in;
  P.state_out = state_out;
  P.y = y;
  P.o = o;
  const int split = s->decode_split ? s->decode_split : kAutoDecodeSplit;
  if (split == 1) HLA_LAUNCH(launch_decode(P, s->dtype, (cudaStream_t)stream));
  else HLA_LAUNCH(launch_decode_split(P, s->dtype, split, (cudaStream_t)stream));
  return HLA_OK;
}

hla_status hla_prefill_backward(const hla_shape *s, const void *q, const void *k, const void *v,
                                const void *gate, const float *gamma, const float *state_in,
                                const void *dy, const float *dstate_out, void *dq, void *dk,
                                void *dv, void *dgate, float *dstate_in, void *ws,
                                size_t ws_bytes, hla_stream stream, const hla_trace *trace,
                                const void *fwd_ws, const void *saved, const void *y) {
  HLA_TRY(check_shape(s, false));
  HLA_TRY(check_gamma(gamma, s->H));
  const bool empty = s->B == 0 || s->T == 0;
  // with saved features the raw q and k are not read: they may be NULL
  const void *acts[] = {v, gate, dy, dq, dk, dv, dgate};
  for (const void *a : acts) HLA_TRY(need_unless(empty, a));
  HLA_TRY(saved ? maybe(q) : need_unless(empty, q));
  HLA_TRY(saved ? maybe(k) : need_unless(empty, k));
  HLA_TRY(maybe(state_in));
  HLA_TRY(maybe(dstate_out));
  HLA_TRY(maybe(dstate_in));
  HLA_TRY(check_trace(trace));
  HLA_TRY(maybe(fwd_ws));
  HLA_TRY(maybe(saved));
  HLA_TRY(maybe(y));
  if (saved && !can_save(*s)) return HLA_ERR_UNSUPPORTED;
  if (y && !saved) return HLA_ERR_INVALID_ARG;  // y stands in for o only with the saved 1/RMS(o)
  Plan plan = make_plan(*s);
  size_t sbytes = seg_bytes(*s, plan);
  size_t need_ws = hla_backward_workspace_size(s);
  if (!ws || !aligned16(ws) || ws_bytes < need_ws) return HLA_ERR_WORKSPACE;
  if (empty) {  // no tokens: the state gradient passes through unchanged
    cudaStream_t st = (cudaStream_t)stream;
    Tracer tr{trace, st};
    HLA_LAUNCH(cudaMemsetAsync((char *)ws + need_ws - kStatusBytes, 0, sizeof(unsigned int), st));
    HLA_LAUNCH(pass_state(*s, dstate_out, dstate_in, st));
    for (int i = 0; i < 7; ++i) HLA_LAUNCH(tr.mark());
    return HLA_OK;
  }

  MixerParams P;
  fill_common(P, *s, gamma);
  P.nseg = plan.nseg;
  P.seg_len = plan.seg_len;
  P.q = q; P.k = k; P.v = v; P.g = gate;
  P.state_in = state_in;
  P.dy = dy;
  P.y_in = y;
  P.dstate_out = dstate_out;
  P.dq = dq; P.dk = dk; P.dv = dv; P.dg = dgate;
  P.dstate_in = dstate_in;
  // the state entering each segment: from the forward's workspace (written
  // by its scan, read only here) or recomputed into this workspace
  P.seg = fwd_ws ? (float *)const_cast<void *>(fwd_ws) : (float *)ws;
  P.seg2 = (float *)((char *)ws + sbytes);
  P.npart = part_count(*s, plan);
  P.part = P.npart > 1 ? (float *)((char *)ws + 2 * sbytes) : nullptr;
  P.dO = (float *)((char *)ws + 2 * sbytes + part_bytes(*s, plan));
  // the tensor-core path keeps do in bf16: the second half of its region holds
  // the per-token diagonal v_t . do_t
  P.ddiag = (float *)((char *)P.dO + (size_t)s->B * s->T * s->H * s->dv * 2);
  P.err = (unsigned int *)((char *)ws + need_ws - kStatusBytes);
  cudaStream_t st = (cudaStream_t)stream;
  const bool tc = tc_supported(P, s->dtype);
  Tracer tr{trace, st};
  HLA_LAUNCH(cudaMemsetAsync(P.err, 0, sizeof(unsigned int), st));
  HLA_LAUNCH(tr.mark());
  P.state_seg0 = 0;  // entering states only: the last segment's sum is not needed
  P.state_nseg = P.nseg - 1;
  // recomputed from raw k (the forward's own arithmetic, so the states are
  // bit-identical to those a forward workspace holds), or, when the caller
  // gave saved features without raw k, from the k~ saved there
  P.saved = (unsigned char *)const_cast<void *>(saved);
  P.features_in = (saved && !k) ? 1 : 0;
  if (!fwd_ws) HLA_LAUNCH(tc ? launch_tc_seg_state(P, st) : launch_simt_seg_state(P, s->dtype, st));
  P.features_in = 0;
  HLA_LAUNCH(tr.mark());
  if (!fwd_ws) HLA_LAUNCH(launch_state_scan(P, false, st));
  HLA_LAUNCH(tr.mark());
  P.saved = (unsigned char *)const_cast<void *>(saved);  // read by the three passes below
  HLA_LAUNCH(tc ? launch_tc_bwd_dq(P, st) : launch_simt_bwd_dq(P, s->dtype, st));
  HLA_LAUNCH(tr.mark());
  // tensor cores: the first segment's state-gradient sum is not formed; its
  // dk/dv pass writes dstate_in from the gradient it carries
  P.state_seg0 = 1;
  P.state_nseg = P.nseg - 1;
  HLA_LAUNCH(tc ? launch_tc_seg_gstate(P, st) : launch_simt_seg_gstate(P, s->dtype, st));
  HLA_LAUNCH(tr.mark());
  HLA_LAUNCH(launch_grad_scan(P, !tc && dstate_in != nullptr, st));
  HLA_LAUNCH(tr.mark());
  HLA_LAUNCH(tc ? launch_tc_bwd_dkdv(P, st) : launch_simt_bwd_dkdv(P, s->dtype, st));
  HLA_LAUNCH(tr.mark());
  return HLA_OK;
}

size_t hla_project_workspace_size(void) { return kStatusBytes; }

hla_status hla_project_in(const hla_shape *s, int32_t d_model, const void *x, const void *w_qkvz,
                          void *features, void *v, void *gate, void *ws, size_t ws_bytes,
                          hla_stream stream) {
  HLA_TRY(check_shape(s, false));
  if (d_model < 1) return HLA_ERR_INVALID_ARG;
  if (!can_save(*s) || d_model % 64) return HLA_ERR_UNSUPPORTED;
  const long long M = (long long)s->B * s->T;
  if (M > 0x7fffffffLL) return HLA_ERR_UNSUPPORTED;
  const bool empty = M == 0;
  HLA_TRY(need_unless(empty, x));
  HLA_TRY(need_unless(empty, w_qkvz));
  HLA_TRY(need_unless(empty, features));
  HLA_TRY(need_unless(empty, v));
  HLA_TRY(need_unless(empty, gate));
  if (!ws || !aligned16(ws) || ws_bytes < kStatusBytes) return HLA_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned int *err = (unsigned int *)ws;
  HLA_LAUNCH(cudaMemsetAsync(err, 0, sizeof(unsigned int), st));
  if (empty) return HLA_OK;
  ProjParams P;
  memset(&P, 0, sizeof(P));
  P.M = (int)M;
  P.N = 4 * s->H * s->dk;
  P.K = d_model;
  P.T = s->T;
  P.H = s->H;
  P.pos_offset = s->pos_offset;
  P.eps = s->norm_eps;
  P.kscale = (float)(1.0 / sqrt((double)s->dk));
  unsigned char *f = (unsigned char *)features;
  P.qt = f;
  P.kt = f + saved_k_offset(s->B, s->T, s->H, s->dk);
  P.scal = (float *)(f + saved_scalar_offset(s->B, s->T, s->H, s->dk));
  P.v = v;
  P.g = gate;
  P.err = err;
  fill_rope_u(P.rope_u, s->dk, s->rope_base);
  HLA_LAUNCH(launch_proj_in(P, x, w_qkvz, st));
  return HLA_OK;
}

hla_status hla_project_out(int64_t M, int32_t n_in, int32_t d_model, const void *u, const void *w_o,
                           void *out, void *ws, size_t ws_bytes, hla_stream stream) {
  if (M < 0 || n_in < 1 || d_model < 1) return HLA_ERR_INVALID_ARG;
  if (M > 0x7fffffffLL || n_in % 64 || d_model % 128) return HLA_ERR_UNSUPPORTED;
  const bool empty = M == 0;
  HLA_TRY(need_unless(empty, u));
  HLA_TRY(need_unless(empty, w_o));
  HLA_TRY(need_unless(empty, out));
  if (!ws || !aligned16(ws) || ws_bytes < kStatusBytes) return HLA_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned int *err = (unsigned int *)ws;
  HLA_LAUNCH(cudaMemsetAsync(err, 0, sizeof(unsigned int), st));
  if (empty) return HLA_OK;
  ProjParams P;
  memset(&P, 0, sizeof(P));
  P.M = (int)M;
  P.N = d_model;
  P.K = n_in;
  P.out = out;
  P.err = err;
  HLA_LAUNCH(launch_proj_out(P, u, w_o, st));
  return HLA_OK;
}

}  // extern "C"
