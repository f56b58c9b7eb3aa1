// hla_internal.cuh — launch parameters, work plan and device helpers shared by
// the CUDA kernels of libhla.so.  Nothing here is visible through the C ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "hla.h"

namespace hla {

constexpr int kMaxHeads = 256;
constexpr int kMaxPairs = 64;  // d/2 for d <= 128

// Everything a kernel needs, passed by value (about 1.7 KB of launch
// parameters).  gamma and the RoPE phase increments travel here, so no device
// table has to be allocated or uploaded.
struct MixerParams {
  int B, T, H, D;
  int chunk;    // token tile of the chunked prefill (64 or 128)
  int nseg;     // segments per (b, h)
  int seg_len;  // tokens per segment (a multiple of chunk; the last may be short)
  int features_in;  // tensor-core forward: q~, k~ and the q~ . k~ diagonal are read from
                    // `saved` (hla_prefill_features) instead of computed from raw q, k
  long long pos_offset;
  int fused;        // tensor-core forward in one launch: every output CTA forms the state
                    // entering its segment from the decay window before it (window_tiles)
  int pad1;
  long long test_wait_cycles;  // > 0: testing the expiry path (hla_trace); the budget of the
                               // output pass's first wait for a tile's feature map
  float eps;
  float kscale;  // 1 / sqrt(D), applied to k~ after RoPE
  const void *q, *k, *v, *g;
  const float *state_in;
  float *state_out;
  void *y;
  float *o;
  float *seg;              // [B, H, nseg, D, D] per-segment states
  float *seg2;             // backward: [B, H, nseg, D, D] per-segment state gradients
  // Tensor-core local-state passes: each CTA covers one piece of a segment (see
  // piece_tiles; npart pieces per segment at most, 0 on the CUDA-core path).
  // With npart > 1, part holds [B, H, nseg, npart, D, D] partial sums that
  // part_sum adds into seg / seg2; with npart = 1 the pass writes seg / seg2
  // directly and part is nullptr.
  float *part;
  int npart;
  // Segments [state_seg0, state_seg0 + state_nseg) that a tensor-core local-state
  // pass covers: the forward's sums of the last segment feed only the final
  // state, and the state gradient's of the first only dstate_in, which the
  // output and dk/dv passes write from the state they carry instead.
  int state_seg0, state_nseg;
  float *dO;               // backward: [B, T, H, D] gradient of o (fp32; bf16 on the tensor-core path)
  float *ddiag;            // backward, tensor-core path: [B, H, T] fp32 v_t . do_t (token-contiguous)
  const long long *pos;    // decode: [B] positions or nullptr
  const void *dy;
  const void *y_in;        // backward, tensor-core path with saved features: the forward's
                           // y, from which the dq pass takes the normalized output
                           // (nullptr = recompute o)
  const float *dstate_out;
  void *dq, *dk, *dv, *dg;
  float *dstate_in;
  unsigned int *err;       // device status word: bits set when a bounded wait gave up
  // Features saved by the forward for the backward (tensor-core path only;
  // nullptr = none): q~ and k~ as fp16 [B, T, H, D] (k~ includes 1/sqrt(d)),
  // then fp32 [4][B, H, T]: 1/RMS(q), 1/RMS(k), the fp32 q~_t . k~_t and
  // 1/RMS(o) (the output norm's scale).  Written by the output pass when the
  // forward is given one (the first three by the projection when it made the
  // features, the fourth by the output pass that uses them), read by the
  // backward passes instead of recomputing the feature map (and, given y, o).
  unsigned char *saved;
  float gamma[kMaxHeads];
  // RoPE phase increment of pair i, in units of 2^-64 turns:
  // round(frac(rope_base^(-2i/D) / (2 pi)) * 2^64).  The angle of position p is
  // (p * rope_u[i] mod 2^64) * 2^-64 turns, exact modular arithmetic, so the
  // phase stays accurate at any position.
  unsigned long long rope_u[kMaxPairs];
};

// Launch parameters of the projection GEMMs (tc_proj.cu): out[M, N] =
// A[M, K] W[N, K]^T with bf16 A and W.
struct ProjParams {
  int M, N, K;            // problem size
  int n_mt, n_nt;         // output tiles (set by the launcher)
  int T, H;               // projection in: row m = b T + t, N = 4 H d
  long long pos_offset;   // projection in: RoPE position of t = 0
  float eps, kscale;      // projection in: RMSNorm epsilon, 1 / sqrt(d)
  void *qt, *kt;          // projection in: fp16 [M, H, d] q~ and k~
  float *scal;            // projection in: fp32 [3, B, H, T] 1/RMS(q), 1/RMS(k), q~ . k~
  void *v, *g;            // projection in: bf16 [M, H, d] v and the gate logit
  void *out;              // projection out: bf16 [M, N]
  unsigned int *err;      // device status word
  unsigned long long rope_u[kMaxPairs];  // RoPE phase increments (as in MixerParams)
};

// Segment decomposition of the T axis.  Each (b, h, segment) is one unit of
// inter-CTA parallelism; the per-segment states are combined by a scan.
struct Plan {
  int nchunk;
  int nseg;
  int seg_len;
};

__host__ __device__ inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// ------------------------------------------------------------------ device helpers

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// cos / sin of the RoPE angle of pair i at position p.
__device__ __forceinline__ void rope_cs(long long p, unsigned long long u, float &c, float &s) {
  unsigned long long ph = (unsigned long long)p * u;    // turns, mod 1, in 2^-64 units
  float x = (float)(long long)ph * 1.0842021724855044e-19f;  // 2^-63: half-turns in [-1, 1)
  sincospif(x, &s, &c);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + __expf(-z)); }

// gamma^m in fp32 for small non-negative m (exp2 of m log2 gamma).
__device__ __forceinline__ float gpow(float log2g, float m) { return exp2f(m * log2g); }

// ------------------------------------------------------------------ pieces of the local-state passes
// The local state of a segment weights token s by gamma^m, m = L - 1 - s from
// the segment's end (forward) or m = s + 1 from its start (state gradient).
// Tokens with m >= W = decay_rows(log2 gamma) are left out: their weights sum
// to at most sum_{m >= W} gamma^m = gamma^W / (1 - gamma) <= 2^-40, so
// together they change each state element by at most 2^-40 max_s |k~_s^T v_s|
// (elementwise), far below the 2^-9 rounding of the bf16 operands the sums
// are taken on.  The pass skips their tiles; the tiles that remain are cut
// into pieces of kPieceTiles, each one CTA writing its own partial sum, which
// the scan adds in a fixed order.  gamma = 1 keeps every token.
constexpr int kPieceTiles = 48;
constexpr float kDecayTailLog2 = 40.f;  // -log2 of the bound on the weights left out

// fp32 throughout, device code only (the host never needs W): the smallest W
// with W |log2 gamma| >= 40 + log2(1 / (1 - gamma)).
__host__ __device__ inline long long decay_rows(float log2g) {
  if (!(log2g < 0.f)) return 1LL << 40;  // gamma = 1: nothing decays
  const float one_minus = -expm1f(log2g * 0.69314718f);  // 1 - gamma, accurate near gamma = 1
  const float w = (kDecayTailLog2 - log2f(one_minus)) / -log2g;
  return w >= 1.0995116e12f ? (1LL << 40) : (long long)w + 1;
}

// Tiles of CV tokens right before token t0 that the state entering a segment
// at t0 needs: those holding a token with weight gamma^m, m = t0 - 1 - s, inside
// the decay horizon (decay_rows), and none before token 0.  State_in enters
// with gamma^t0 on top.
__host__ __device__ inline int window_tiles(float log2g, long long t0, int CV) {
  if (t0 <= 0) return 0;
  const long long W = decay_rows(log2g);
  const long long nt = (W + CV - 1) / CV;
  return (int)(nt < t0 / CV ? nt : t0 / CV);
}

// Tiles [lo, hi) of a segment of L tokens (ntile tiles of CV) that piece p
// covers; lo >= hi when the piece is empty.  grad: weights from the start.
__host__ __device__ inline void piece_tiles(long long W, int L, int CV, int p, bool grad, int &lo,
                                            int &hi) {
  const int ntile = (L + CV - 1) / CV;
  if (!grad) {  // rows s >= L - W carry weight
    const int first = (long long)L > W ? (int)(((long long)L - W) / CV) : 0;
    hi = ntile - p * kPieceTiles;
    lo = hi - kPieceTiles > first ? hi - kPieceTiles : first;
  } else {      // rows s <= W - 2 carry weight
    const int last = W >= 2 ? (int)((W - 2) / CV + 1 < ntile ? (W - 2) / CV + 1 : ntile) : 0;
    lo = p * kPieceTiles;
    hi = lo + kPieceTiles < last ? lo + kPieceTiles : last;
  }
}

// Number of non-empty pieces of that segment (pieces 0 .. n-1).
__host__ __device__ inline int piece_count(long long W, int L, int CV, bool grad) {
  const int ntile = (L + CV - 1) / CV;
  int nt;
  if (!grad) {
    const int first = (long long)L > W ? (int)(((long long)L - W) / CV) : 0;
    nt = ntile - first;
  } else {
    nt = W >= 2 ? (int)((W - 2) / CV + 1 < ntile ? (W - 2) / CV + 1 : ntile) : 0;
  }
  return (nt + kPieceTiles - 1) / kPieceTiles;
}

// ------------------------------------------------------------------ saved features
// Byte offset of k~ in the saved buffer, and of the fp32 per-row scalars.
__host__ __device__ inline size_t saved_k_offset(int B, int T, int H, int D) {
  return (size_t)B * T * H * D * 2;
}
__host__ __device__ inline size_t saved_scalar_offset(int B, int T, int H, int D) {
  return 2 * saved_k_offset(B, T, H, D);
}
enum { kSavedRq = 0, kSavedRk = 1, kSavedDiag = 2, kSavedRo = 3, kSavedPlanes = 4 };
// Scalar f of row (b, h, t).
__device__ __forceinline__ float *saved_scalar(const MixerParams &P, int f, int b, int h, int t) {
  float *base = reinterpret_cast<float *>(P.saved + saved_scalar_offset(P.B, P.T, P.H, P.D));
  return base + (((size_t)f * P.B + b) * P.H + h) * (size_t)P.T + t;
}

// ------------------------------------------------------------------ host side

Plan make_plan(const hla_shape &s);
bool aligned16(const void *p);
hla_status check_shape(const hla_shape *s, bool decode);
hla_status check_gamma(const float *gamma, int H);
hla_status need(const void *p);
hla_status maybe(const void *p);
hla_status need_unless(bool empty, const void *p);
cudaError_t pass_state(const hla_shape &s, const float *in, float *out, cudaStream_t st);
void fill_common(MixerParams &P, const hla_shape &s, const float *gamma);
size_t seg_bytes(const hla_shape &s, const Plan &p);
size_t part_bytes(const hla_shape &s, const Plan &p);
size_t saved_bytes(const hla_shape &s);
int part_count(const hla_shape &s, const Plan &p);
void fill_rope(MixerParams &P, int D, double base);
void fill_rope_u(unsigned long long *u, int D, double base);

// Kernel launchers (return the cudaError_t of the launch).
cudaError_t launch_decode(const MixerParams &P, int dtype, cudaStream_t st);
cudaError_t launch_state_scan(const MixerParams &P, bool write_state_out, cudaStream_t st);
cudaError_t launch_grad_scan(const MixerParams &P, bool write_dstate_in, cudaStream_t st);
cudaError_t launch_part_sum(const MixerParams &P, bool grad, cudaStream_t st);
cudaError_t launch_simt_seg_state(const MixerParams &P, int dtype, cudaStream_t st);
// Load the kernels of the fp32 CUDA-core forward (for dtype and D) and of the
// forward scan without launching them.
cudaError_t prepare_simt_forward(int dtype, int D);
cudaError_t prepare_state_scan();
cudaError_t launch_simt_seg_output(const MixerParams &P, int dtype, cudaStream_t st);
cudaError_t launch_simt_bwd_dq(const MixerParams &P, int dtype, cudaStream_t st);
cudaError_t launch_simt_seg_gstate(const MixerParams &P, int dtype, cudaStream_t st);
cudaError_t launch_simt_bwd_dkdv(const MixerParams &P, int dtype, cudaStream_t st);
bool tc_supported(const MixerParams &P, int dtype);
cudaError_t launch_tc_seg_state(const MixerParams &P, cudaStream_t st);
cudaError_t launch_tc_seg_output(const MixerParams &P, cudaStream_t st);
cudaError_t launch_tc_seg_gstate(const MixerParams &P, cudaStream_t st);
cudaError_t launch_tc_bwd_dq(const MixerParams &P, cudaStream_t st);
cudaError_t launch_tc_bwd_dkdv(const MixerParams &P, cudaStream_t st);
cudaError_t launch_proj_in(ProjParams &P, const void *x, const void *w, cudaStream_t st);
cudaError_t launch_proj_out(ProjParams &P, const void *u, const void *w, cudaStream_t st);

// Bytes reserved at the end of a workspace for the device status word.
constexpr size_t kStatusBytes = 256;

}  // namespace hla
