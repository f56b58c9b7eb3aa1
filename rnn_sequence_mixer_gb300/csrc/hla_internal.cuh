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
  int pad0;
  long long pos_offset;
  float eps;
  float kscale;  // 1 / sqrt(D), applied to k~ after RoPE
  const void *q, *k, *v, *g;
  const float *state_in;
  float *state_out;
  void *y;
  float *o;
  float *seg;              // [B, H, nseg, D, D] per-segment states
  float *seg2;             // backward: [B, H, nseg, D, D] per-segment state gradients
  float *dO;               // backward: [B, T, H, D] gradient of o (fp32; bf16 on the tensor-core path)
  float *ddiag;            // backward, tensor-core path: [B, T, H] fp32 v_t . do_t
  const long long *pos;    // decode: [B] positions or nullptr
  const void *dy;
  const float *dstate_out;
  void *dq, *dk, *dv, *dg;
  float *dstate_in;
  unsigned int *err;       // device status word: bits set when a bounded wait gave up
  float gamma[kMaxHeads];
  // RoPE phase increment of pair i, in units of 2^-64 turns:
  // round(frac(rope_base^(-2i/D) / (2 pi)) * 2^64).  The angle of position p is
  // (p * rope_u[i] mod 2^64) * 2^-64 turns, exact modular arithmetic, so the
  // phase stays accurate at any position.
  unsigned long long rope_u[kMaxPairs];
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
void fill_rope(MixerParams &P, int D, double base);

// Kernel launchers (return the cudaError_t of the launch).
cudaError_t launch_decode(const MixerParams &P, int dtype, cudaStream_t st);
cudaError_t launch_state_scan(const MixerParams &P, bool write_state_out, cudaStream_t st);
cudaError_t launch_grad_scan(const MixerParams &P, bool write_dstate_in, cudaStream_t st);
cudaError_t launch_simt_seg_state(const MixerParams &P, int dtype, cudaStream_t st);
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

// Bytes reserved at the end of a workspace for the device status word.
constexpr size_t kStatusBytes = 256;

}  // namespace hla
