// simt_forward.cu — fp32 CUDA-core kernels of the chunked prefill.
//
//   seg_state_kernel   (b, h, segment) -> local state Delta_g of the segment
//                      (zero initial state), chunk by chunk:
//                      S <- gamma^c S + (diag(gamma^{c-1-j}) K~)^T V
//   seg_output_kernel  (b, h, segment) -> y (and o) of every token, starting
//                      from the segment's entering state written by the scan:
//                      O = diag(gamma^{i+1}) Q~ S + (Q~ K~^T (.) D) V
//                      y = Norm(O) * sigmoid(gate)
// Both follow Eq. 18 of arXiv 2601.22156 (Appendix A) in its chunked form.
#include "simt_common.cuh"

namespace hla {
namespace simt {

namespace {

template <typename DT, int D>
__global__ void __launch_bounds__(NT) seg_state_kernel(const __grid_constant__ MixerParams P) {
  using Dm = Dims<D>;
  constexpr int LD = Dm::LD;
  extern __shared__ float sm[];
  float *S = sm;
  float *Kt = S + Dm::STATE;
  float *Vs = Kt + Dm::TILE;
  float *pw = Vs + Dm::TILE;

  const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = g * P.seg_len;
  const int t1 = min(P.T, t0 + P.seg_len);
  fill_pow<D>(pw, log2f(P.gamma[h]));
  for (int e = threadIdx.x; e < D * D; e += NT) S[(e / D) * LD + (e % D)] = 0.f;

  for (int c0 = t0; c0 < t1; c0 += CS) {
    const int c = min(CS, t1 - c0);
    __syncthreads();
    load_tile<DT, D>(Kt, (const DT *)P.k, P, b, h, c0, c);
    load_tile<DT, D>(Vs, (const DT *)P.v, P, b, h, c0, c);
    __syncthreads();
    for (int t = warp; t < c; t += NT / 32)
      feature_one<D>(Kt + t * LD, P.pos_offset + c0 + t, P, lane, P.kscale);
    __syncthreads();
    const float carry = pw[c];
    block_mm<4, 4>(
        D, D, c, [&](int m, int kk) { return Kt[kk * LD + m] * pw[c - 1 - kk]; },
        [&](int kk, int n) { return Vs[kk * LD + n]; },
        [&](int m, int n, float acc) { S[m * LD + n] = fmaf(carry, S[m * LD + n], acc); });
  }
  __syncthreads();
  float *out = P.seg + (((size_t)b * P.H + h) * P.nseg + g) * (size_t)D * D;
  for (int e = threadIdx.x; e < D * D; e += NT) out[e] = S[(e / D) * LD + (e % D)];
}

template <typename DT, int D>
__global__ void __launch_bounds__(NT) seg_output_kernel(const __grid_constant__ MixerParams P) {
  using Dm = Dims<D>;
  constexpr int LD = Dm::LD, LDA = Dm::LDA;
  extern __shared__ float sm[];
  float *S = sm;
  float *Qt = S + Dm::STATE;
  float *Kt = Qt + Dm::TILE;
  float *Vs = Kt + Dm::TILE;
  float *Os = Vs + Dm::TILE;
  float *A = Os + Dm::TILE;
  float *pw = A + Dm::SQ;

  const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = g * P.seg_len;
  const int t1 = min(P.T, t0 + P.seg_len);
  fill_pow<D>(pw, log2f(P.gamma[h]));
  const float *sin_ = P.seg + (((size_t)b * P.H + h) * P.nseg + g) * (size_t)D * D;
  for (int e = threadIdx.x; e < D * D; e += NT) S[(e / D) * LD + (e % D)] = sin_[e];
  const DT *gate = (const DT *)P.g;
  DT *y = (DT *)P.y;

  for (int c0 = t0; c0 < t1; c0 += CS) {
    const int c = min(CS, t1 - c0);
    __syncthreads();
    load_tile<DT, D>(Qt, (const DT *)P.q, P, b, h, c0, c);
    load_tile<DT, D>(Kt, (const DT *)P.k, P, b, h, c0, c);
    load_tile<DT, D>(Vs, (const DT *)P.v, P, b, h, c0, c);
    __syncthreads();
    for (int t = warp; t < c; t += NT / 32) {
      float rq, rk;
      feature_qk<D>(Qt + t * LD, Kt + t * LD, P.pos_offset + c0 + t, P, lane, rq, rk);
    }
    __syncthreads();
    // A = (Q~ K~^T) (.) D
    block_mm<4, 4>(
        CS, CS, D, [&](int m, int kk) { return Qt[m * LD + kk]; },
        [&](int kk, int n) { return Kt[n * LD + kk]; },
        [&](int m, int n, float acc) { A[m * LDA + n] = (n <= m) ? acc * pw[m - n] : 0.f; });
    __syncthreads();
    // O = diag(gamma^{i+1}) Q~ S + A V
    block_mm2<4, 4>(
        CS, D, D, [&](int m, int kk) { return Qt[m * LD + kk]; },
        [&](int kk, int n) { return S[kk * LD + n]; }, c,
        [&](int m, int kk) { return A[m * LDA + kk]; },
        [&](int kk, int n) { return Vs[kk * LD + n]; },
        [&](int m, int n, float inter, float intra) {
          Os[m * LD + n] = fmaf(pw[min(m + 1, CS)], inter, intra);
        });
    __syncthreads();
    // y = Norm(o) * sigmoid(gate), one warp per token.
    for (int t = warp; t < c; t += NT / 32) {
      const float *orow = Os + t * LD;
      float a = 0.f;
      for (int j = lane; j < D; j += 32) a += orow[j] * orow[j];
      const float ro = rsqrtf(warp_sum(a) / (float)D + P.eps);
      const size_t base = (((size_t)b * P.T + c0 + t) * P.H + h) * D;
      for (int j = lane; j < D; j += 32) {
        const float oj = orow[j];
        y[base + j] = from_f<DT>(oj * ro * sigmoidf_(to_f(gate[base + j])));
        if (P.o) P.o[base + j] = oj;
      }
    }
    // S <- gamma^c S + (diag(gamma^{c-1-j}) K~)^T V  (independent of the loop above)
    const float carry = pw[c];
    block_mm<4, 4>(
        D, D, c, [&](int m, int kk) { return Kt[kk * LD + m] * pw[c - 1 - kk]; },
        [&](int kk, int n) { return Vs[kk * LD + n]; },
        [&](int m, int n, float acc) { S[m * LD + n] = fmaf(carry, S[m * LD + n], acc); });
  }
}

template <typename DT, int D>
size_t state_smem() {
  using Dm = Dims<D>;
  return sizeof(float) * (Dm::STATE + 2 * Dm::TILE + CS + 1);
}
template <typename DT, int D>
size_t output_smem() {
  using Dm = Dims<D>;
  return sizeof(float) * (Dm::STATE + 4 * Dm::TILE + Dm::SQ + CS + 1);
}

template <typename DT, int D>
cudaError_t run_state(const MixerParams &P, cudaStream_t st) {
  const size_t smem = state_smem<DT, D>();
  cudaError_t e = cudaFuncSetAttribute(seg_state_kernel<DT, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  seg_state_kernel<DT, D><<<dim3(P.nseg, P.H, P.B), NT, smem, st>>>(P);
  return cudaGetLastError();
}

template <typename DT, int D>
cudaError_t run_output(const MixerParams &P, cudaStream_t st) {
  const size_t smem = output_smem<DT, D>();
  cudaError_t e = cudaFuncSetAttribute(seg_output_kernel<DT, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  seg_output_kernel<DT, D><<<dim3(P.nseg, P.H, P.B), NT, smem, st>>>(P);
  return cudaGetLastError();
}

// Loads both kernels of one instantiation (under lazy module loading a
// kernel's module is loaded, and its device memory committed, the first time
// the runtime touches the kernel) without launching anything.
template <typename DT, int D>
cudaError_t prepare() {
  cudaError_t e = cudaFuncSetAttribute(seg_state_kernel<DT, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)state_smem<DT, D>());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(seg_output_kernel<DT, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)output_smem<DT, D>());
}

}  // namespace
}  // namespace simt

cudaError_t prepare_simt_forward(int dtype, int D) {
  if (dtype == HLA_BF16)
    return D == 128 ? simt::prepare<__nv_bfloat16, 128>() : simt::prepare<__nv_bfloat16, 64>();
  return D == 128 ? simt::prepare<float, 128>() : simt::prepare<float, 64>();
}

cudaError_t launch_simt_seg_state(const MixerParams &P, int dtype, cudaStream_t st) {
  if (dtype == HLA_BF16)
    return P.D == 128 ? simt::run_state<__nv_bfloat16, 128>(P, st)
                      : simt::run_state<__nv_bfloat16, 64>(P, st);
  return P.D == 128 ? simt::run_state<float, 128>(P, st) : simt::run_state<float, 64>(P, st);
}

cudaError_t launch_simt_seg_output(const MixerParams &P, int dtype, cudaStream_t st) {
  if (dtype == HLA_BF16)
    return P.D == 128 ? simt::run_output<__nv_bfloat16, 128>(P, st)
                      : simt::run_output<__nv_bfloat16, 64>(P, st);
  return P.D == 128 ? simt::run_output<float, 128>(P, st) : simt::run_output<float, 64>(P, st);
}

}  // namespace hla
