// scan.cu — fp32 scans over the segments of each (b, h) sequence.
//
// Forward (state_scan): segment g holds on entry its local state
//   Delta_g = sum_{s in g} gamma^{end_g - s} k~_s^T v_s        (zero initial state)
// and on exit the state entering it, S_g; the recurrence is the segment-level
// form of Eq. 18 (arXiv 2601.22156, Appendix A):
//   S_0 = state_in (or 0),   S_{g+1} = gamma^{L_g} S_g + Delta_g,
// and S_nseg is the final state.  Every element of the d x d state is an
// independent linear recurrence, so one thread walks four consecutive elements
// through the segments; consecutive threads own consecutive elements (coalesced).
//
// Backward (grad_scan) runs the mirror recurrence from the end: segment g
// holds on entry
//   DeltaG_g = sum_{s in g} gamma^{s - start_g + 1} q~_s^T do_s
// and on exit E_g, the gradient reaching the state at g's last token from
// later tokens (dstate_out for the last segment):
//   E_{nseg-1} = dstate_out,   E_{g-1} = gamma^{L_g} E_g + DeltaG_g,
// and dstate_in = E_{-1}.
//
// The tensor-core local-state passes write one partial sum per piece of a
// segment (piece_tiles in hla_internal.cuh); part_sum adds a segment's pieces
// in order into its seg / seg2 slot before the scan.
#include "hla_internal.cuh"

namespace hla {

namespace {

constexpr int kScanThreads = 256;
constexpr int kBatch = 8;
constexpr int kVec = 4;  // state elements per thread (one 16-byte access)

typedef float4 V4;
__device__ __forceinline__ V4 v4_fma(float a, V4 x, V4 y) {
  return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}
__device__ __forceinline__ V4 v4_add(V4 x, V4 y) {
  return make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w);
}

// Each thread walks kVec consecutive elements of one (b, h) state through the
// segments: the d x d elements are independent recurrences, and 16-byte
// accesses give each thread four of them in flight at once.
__global__ void __launch_bounds__(kScanThreads) state_scan_kernel(const MixerParams P,
                                                                  int write_out) {
  const size_t DD = (size_t)P.D * P.D;
  const size_t e = ((size_t)blockIdx.y * kScanThreads + threadIdx.x) * kVec;
  if (e >= DD) return;
  const int bh = blockIdx.x;
  const int h = bh % P.H;
  const float l2g = log2f(P.gamma[h]);
  const int last_len = P.T - (P.nseg - 1) * P.seg_len;
  const float carry_full = exp2f((float)P.seg_len * l2g);
  const float carry_last = exp2f((float)last_len * l2g);
  V4 S = P.state_in ? *reinterpret_cast<const V4 *>(P.state_in + (size_t)bh * DD + e)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
  float *seg = P.seg + (size_t)bh * P.nseg * DD + e;
  // Batches of independent loads ahead of the dependent chain (the slots are
  // overwritten in place, so each batch is loaded before any of it is stored).
  for (int g0 = 0; g0 < P.nseg; g0 += kBatch) {
    V4 delta[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      delta[j] = g0 + j < P.nseg ? *reinterpret_cast<const V4 *>(seg + (size_t)(g0 + j) * DD)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int g = g0 + j;
      if (g < P.nseg) {
        *reinterpret_cast<V4 *>(seg + (size_t)g * DD) = S;
        S = v4_fma(g == P.nseg - 1 ? carry_last : carry_full, S, delta[j]);
      }
    }
  }
  if (write_out) *reinterpret_cast<V4 *>(P.state_out + (size_t)bh * DD + e) = S;
}

__global__ void __launch_bounds__(kScanThreads) grad_scan_kernel(const MixerParams P,
                                                                 int write_out) {
  const size_t DD = (size_t)P.D * P.D;
  const size_t e = ((size_t)blockIdx.y * kScanThreads + threadIdx.x) * kVec;
  if (e >= DD) return;
  const int bh = blockIdx.x;
  const int h = bh % P.H;
  const float l2g = log2f(P.gamma[h]);
  const int last_len = P.T - (P.nseg - 1) * P.seg_len;
  const float carry_full = exp2f((float)P.seg_len * l2g);
  const float carry_last = exp2f((float)last_len * l2g);
  V4 E = P.dstate_out ? *reinterpret_cast<const V4 *>(P.dstate_out + (size_t)bh * DD + e)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
  float *seg = P.seg2 + (size_t)bh * P.nseg * DD + e;
  for (int g1 = P.nseg - 1; g1 >= 0; g1 -= kBatch) {
    V4 delta[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      delta[j] = g1 - j >= 0 ? *reinterpret_cast<const V4 *>(seg + (size_t)(g1 - j) * DD)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int g = g1 - j;
      if (g >= 0) {
        *reinterpret_cast<V4 *>(seg + (size_t)g * DD) = E;
        E = v4_fma(g == P.nseg - 1 ? carry_last : carry_full, E, delta[j]);
      }
    }
  }
  if (write_out) *reinterpret_cast<V4 *>(P.dstate_in + (size_t)bh * DD + e) = E;
}

// Delta_g (or DeltaG_g) = sum of the segment's non-empty pieces, p = 0, 1, ...
// One thread per kVec state elements of one (b, h, segment).
__global__ void __launch_bounds__(kScanThreads) part_sum_kernel(const MixerParams P, int grad) {
  const size_t DD = (size_t)P.D * P.D;
  const size_t e = ((size_t)blockIdx.x * kScanThreads + threadIdx.x) * kVec;
  if (e >= DD) return;
  const int g = P.state_seg0 + blockIdx.y, bh = blockIdx.z;
  const int h = bh % P.H;
  const int L = g == P.nseg - 1 ? P.T - (P.nseg - 1) * P.seg_len : P.seg_len;
  const int np = piece_count(decay_rows(log2f(P.gamma[h])), L, P.chunk, grad != 0);
  const float *part = P.part + ((size_t)bh * P.nseg + g) * P.npart * DD + e;
  const V4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  V4 acc[4] = {z, z, z, z};
  for (int p0 = 0; p0 < np; p0 += 4) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (p0 + j < np) acc[j] = v4_add(acc[j], *reinterpret_cast<const V4 *>(part + (size_t)(p0 + j) * DD));
  }
  float *dst = (grad ? P.seg2 : P.seg) + ((size_t)bh * P.nseg + g) * DD + e;
  *reinterpret_cast<V4 *>(dst) = v4_add(v4_add(acc[0], acc[1]), v4_add(acc[2], acc[3]));
}

}  // namespace

cudaError_t launch_part_sum(const MixerParams &P, bool grad, cudaStream_t st) {
  dim3 grid(ceil_div((long long)P.D * P.D, kScanThreads * kVec), P.state_nseg, P.B * P.H);
  part_sum_kernel<<<grid, kScanThreads, 0, st>>>(P, grad ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t prepare_state_scan() {
  cudaFuncAttributes a;
  return cudaFuncGetAttributes(&a, state_scan_kernel);
}

cudaError_t launch_state_scan(const MixerParams &P, bool write_state_out, cudaStream_t st) {
  dim3 grid(P.B * P.H, ceil_div((long long)P.D * P.D, kScanThreads * kVec));
  state_scan_kernel<<<grid, kScanThreads, 0, st>>>(P, write_state_out ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_grad_scan(const MixerParams &P, bool write_dstate_in, cudaStream_t st) {
  dim3 grid(P.B * P.H, ceil_div((long long)P.D * P.D, kScanThreads * kVec));
  grad_scan_kernel<<<grid, kScanThreads, 0, st>>>(P, write_dstate_in ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace hla
