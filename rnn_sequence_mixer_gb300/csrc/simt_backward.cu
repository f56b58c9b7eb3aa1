// simt_backward.cu — fp32 CUDA-core kernels of the prefill backward.
//
// Gradients of L = <dy, y> + <dstate_out, S_T> through Eq. 18 of
// arXiv 2601.22156 (Appendix A), evaluated chunk by chunk.  With the states S
// entering each chunk recomputed by the forward segment pass + scan:
//
//   bwd_dq_kernel     (forward over the chunks of a segment)
//       O    = diag(gamma^{i+1}) Q~ S + (Q~ K~^T (.) D) V           (recomputed)
//       dgate = dy n sigma(g)(1 - sigma(g)),  dn = dy sigma(g)
//       dO   = r (dn - n mean(dn n)),  n = O r                      (output RMSNorm)
//       dQ~  = diag(gamma^{i+1}) dO S^T + (dO V^T (.) D) K~
//       dq   = RMSNorm^T RoPE^T dQ~
//   seg_gstate_kernel (backward over the chunks of a segment)
//       G   <- gamma^c G + (diag(gamma^{i+1}) Q~)^T dO   -> DeltaG of the segment
//   bwd_dkdv_kernel   (backward over the chunks, E = gradient reaching the
//                      state at the chunk's last token from later tokens)
//       dK~ = (V dO^T (.) D^T) Q~ + diag(gamma^{c-1-i}) V E^T
//       dV  = (K~ Q~^T (.) D^T) dO + diag(gamma^{c-1-i}) K~ E
//       E   <- gamma^c E + (diag(gamma^{i+1}) Q~)^T dO
//       dk  = RMSNorm^T RoPE^T dK~ / sqrt(d)
// where D^T_ij = gamma^{j-i} for j >= i.
#include "simt_common.cuh"

namespace hla {
namespace simt {

namespace {

template <typename DT, int D>
__global__ void __launch_bounds__(NT) bwd_dq_kernel(const __grid_constant__ MixerParams P) {
  using Dm = Dims<D>;
  constexpr int LD = Dm::LD, LDA = Dm::LDA;
  extern __shared__ float sm[];
  float *S = sm;
  float *Qt = S + Dm::STATE;   // q~, later dQ~
  float *Kt = Qt + Dm::TILE;
  float *Vs = Kt + Dm::TILE;
  float *Os = Vs + Dm::TILE;   // o, later dO
  float *A = Os + Dm::TILE;    // masked scores, later masked dO V^T
  float *pw = A + Dm::SQ;
  float *rq = pw + CS + 1;

  const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = g * P.seg_len;
  const int t1 = min(P.T, t0 + P.seg_len);
  fill_pow<D>(pw, log2f(P.gamma[h]));
  const float *sin_ = P.seg + (((size_t)b * P.H + h) * P.nseg + g) * (size_t)D * D;
  for (int e = threadIdx.x; e < D * D; e += NT) S[(e / D) * LD + (e % D)] = sin_[e];
  const DT *gate = (const DT *)P.g, *dy = (const DT *)P.dy, *q = (const DT *)P.q;
  DT *dg = (DT *)P.dg, *dq = (DT *)P.dq;

  for (int c0 = t0; c0 < t1; c0 += CS) {
    const int c = min(CS, t1 - c0);
    __syncthreads();
    load_tile<DT, D>(Qt, q, P, b, h, c0, c);
    load_tile<DT, D>(Kt, (const DT *)P.k, P, b, h, c0, c);
    load_tile<DT, D>(Vs, (const DT *)P.v, P, b, h, c0, c);
    __syncthreads();
    for (int t = warp; t < c; t += NT / 32) {
      float r_q, r_k;
      feature_qk<D>(Qt + t * LD, Kt + t * LD, P.pos_offset + c0 + t, P, lane, r_q, r_k);
      if (lane == 0) rq[t] = r_q;
    }
    __syncthreads();
    block_mm<4, 4>(
        CS, CS, D, [&](int m, int kk) { return Qt[m * LD + kk]; },
        [&](int kk, int n) { return Kt[n * LD + kk]; },
        [&](int m, int n, float acc) { A[m * LDA + n] = (n <= m) ? acc * pw[m - n] : 0.f; });
    __syncthreads();
    block_mm2<4, 4>(
        CS, D, D, [&](int m, int kk) { return Qt[m * LD + kk]; },
        [&](int kk, int n) { return S[kk * LD + n]; }, c,
        [&](int m, int kk) { return A[m * LDA + kk]; },
        [&](int kk, int n) { return Vs[kk * LD + n]; },
        [&](int m, int n, float inter, float intra) {
          Os[m * LD + n] = fmaf(pw[min(m + 1, CS)], inter, intra);
        });
    __syncthreads();
    // Output-gate and output-norm backward, one warp per token: Os <- dO.
    for (int t = warp; t < c; t += NT / 32) {
      float *orow = Os + t * LD;
      float a = 0.f;
      for (int j = lane; j < D; j += 32) a += orow[j] * orow[j];
      const float ro = rsqrtf(warp_sum(a) / (float)D + P.eps);
      const size_t base = (((size_t)b * P.T + c0 + t) * P.H + h) * D;
      float m = 0.f;
      for (int j = lane; j < D; j += 32) {
        const float n = orow[j] * ro;
        const float z = sigmoidf_(to_f(gate[base + j]));
        const float dyv = to_f(dy[base + j]);
        dg[base + j] = from_f<DT>(dyv * n * z * (1.f - z));
        m += dyv * z * n;
      }
      m = warp_sum(m) / (float)D;
      for (int j = lane; j < D; j += 32) {
        const float n = orow[j] * ro;
        const float z = sigmoidf_(to_f(gate[base + j]));
        const float dn = to_f(dy[base + j]) * z;
        const float dov = ro * (dn - n * m);
        orow[j] = dov;
        P.dO[base + j] = dov;
      }
    }
    __syncthreads();
    // A <- (dO V^T) (.) D
    block_mm<4, 4>(
        CS, CS, D, [&](int m, int kk) { return Os[m * LD + kk]; },
        [&](int kk, int n) { return Vs[n * LD + kk]; },
        [&](int m, int n, float acc) { A[m * LDA + n] = (n <= m) ? acc * pw[m - n] : 0.f; });
    __syncthreads();
    // dQ~ = diag(gamma^{i+1}) dO S^T + A K~   (into Qt; q~ is no longer needed)
    block_mm2<4, 4>(
        CS, D, D, [&](int m, int kk) { return Os[m * LD + kk]; },
        [&](int kk, int n) { return S[n * LD + kk]; }, c,
        [&](int m, int kk) { return A[m * LDA + kk]; },
        [&](int kk, int n) { return Kt[kk * LD + n]; },
        [&](int m, int n, float inter, float intra) {
          Qt[m * LD + n] = fmaf(pw[min(m + 1, CS)], inter, intra);
        });
    __syncthreads();
    for (int t = warp; t < c; t += NT / 32) {
      const size_t base = (((size_t)b * P.T + c0 + t) * P.H + h) * D;
      feature_backward<DT, D>(Qt + t * LD, q + base, rq[t], 1.f, P.pos_offset + c0 + t, P, lane,
                              dq + base);
    }
    const float carry = pw[c];
    block_mm<4, 4>(
        D, D, c, [&](int m, int kk) { return Kt[kk * LD + m] * pw[c - 1 - kk]; },
        [&](int kk, int n) { return Vs[kk * LD + n]; },
        [&](int m, int n, float acc) { S[m * LD + n] = fmaf(carry, S[m * LD + n], acc); });
  }
}

template <typename DT, int D>
__global__ void __launch_bounds__(NT) seg_gstate_kernel(const __grid_constant__ MixerParams P) {
  using Dm = Dims<D>;
  constexpr int LD = Dm::LD;
  extern __shared__ float sm[];
  float *G = sm;
  float *Qt = G + Dm::STATE;
  float *dOs = Qt + Dm::TILE;
  float *pw = dOs + Dm::TILE;

  const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = g * P.seg_len;
  const int t1 = min(P.T, t0 + P.seg_len);
  fill_pow<D>(pw, log2f(P.gamma[h]));
  for (int e = threadIdx.x; e < D * D; e += NT) G[(e / D) * LD + (e % D)] = 0.f;
  const int nch = ceil_div(t1 - t0, CS);
  for (int n = nch - 1; n >= 0; --n) {
    const int c0 = t0 + n * CS;
    const int c = min(CS, t1 - c0);
    __syncthreads();
    load_tile<DT, D>(Qt, (const DT *)P.q, P, b, h, c0, c);
    load_tile<float, D>(dOs, P.dO, P, b, h, c0, c);
    __syncthreads();
    for (int t = warp; t < c; t += NT / 32) feature_one<D>(Qt + t * LD, P.pos_offset + c0 + t, P, lane, 1.f);
    __syncthreads();
    const float carry = pw[c];
    block_mm<4, 4>(
        D, D, c, [&](int m, int kk) { return Qt[kk * LD + m] * pw[kk + 1]; },
        [&](int kk, int nn) { return dOs[kk * LD + nn]; },
        [&](int m, int nn, float acc) { G[m * LD + nn] = fmaf(carry, G[m * LD + nn], acc); });
  }
  __syncthreads();
  float *out = P.seg2 + (((size_t)b * P.H + h) * P.nseg + g) * (size_t)D * D;
  for (int e = threadIdx.x; e < D * D; e += NT) out[e] = G[(e / D) * LD + (e % D)];
}

template <typename DT, int D>
__global__ void __launch_bounds__(NT) bwd_dkdv_kernel(const __grid_constant__ MixerParams P) {
  using Dm = Dims<D>;
  constexpr int LD = Dm::LD, LDA = Dm::LDA;
  extern __shared__ float sm[];
  float *E = sm;
  float *Qt = E + Dm::STATE;
  float *Kt = Qt + Dm::TILE;
  float *Vs = Kt + Dm::TILE;
  float *dOs = Vs + Dm::TILE;
  float *dKs = dOs + Dm::TILE;
  float *M1 = dKs + Dm::TILE;
  float *M2 = M1 + Dm::SQ;
  float *pw = M2 + Dm::SQ;
  float *rk = pw + CS + 1;

  const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = g * P.seg_len;
  const int t1 = min(P.T, t0 + P.seg_len);
  fill_pow<D>(pw, log2f(P.gamma[h]));
  const float *ein = P.seg2 + (((size_t)b * P.H + h) * P.nseg + g) * (size_t)D * D;
  for (int e = threadIdx.x; e < D * D; e += NT) E[(e / D) * LD + (e % D)] = ein[e];
  const DT *k = (const DT *)P.k;
  DT *dk = (DT *)P.dk, *dv = (DT *)P.dv;
  const int nch = ceil_div(t1 - t0, CS);
  for (int n = nch - 1; n >= 0; --n) {
    const int c0 = t0 + n * CS;
    const int c = min(CS, t1 - c0);
    __syncthreads();
    load_tile<DT, D>(Qt, (const DT *)P.q, P, b, h, c0, c);
    load_tile<DT, D>(Kt, k, P, b, h, c0, c);
    load_tile<DT, D>(Vs, (const DT *)P.v, P, b, h, c0, c);
    load_tile<float, D>(dOs, P.dO, P, b, h, c0, c);
    __syncthreads();
    for (int t = warp; t < c; t += NT / 32) {
      float r_q, r_k;
      feature_qk<D>(Qt + t * LD, Kt + t * LD, P.pos_offset + c0 + t, P, lane, r_q, r_k);
      if (lane == 0) rk[t] = r_k;
    }
    __syncthreads();
    // M1 = (K~ Q~^T) (.) D^T,  M2 = (V dO^T) (.) D^T
    block_mm<4, 4>(
        CS, CS, D, [&](int m, int kk) { return Kt[m * LD + kk]; },
        [&](int kk, int nn) { return Qt[nn * LD + kk]; },
        [&](int m, int nn, float acc) { M1[m * LDA + nn] = (nn >= m) ? acc * pw[nn - m] : 0.f; });
    block_mm<4, 4>(
        CS, CS, D, [&](int m, int kk) { return Vs[m * LD + kk]; },
        [&](int kk, int nn) { return dOs[nn * LD + kk]; },
        [&](int m, int nn, float acc) { M2[m * LDA + nn] = (nn >= m) ? acc * pw[nn - m] : 0.f; });
    __syncthreads();
    // dV = M1 dO + diag(gamma^{c-1-i}) K~ E   -> global
    block_mm2<4, 4>(
        CS, D, c, [&](int m, int kk) { return M1[m * LDA + kk]; },
        [&](int kk, int nn) { return dOs[kk * LD + nn]; }, D,
        [&](int m, int kk) { return Kt[m * LD + kk]; },
        [&](int kk, int nn) { return E[kk * LD + nn]; },
        [&](int m, int nn, float intra, float inter) {
          if (m < c) {
            const size_t base = (((size_t)b * P.T + c0 + m) * P.H + h) * D;
            dv[base + nn] = from_f<DT>(fmaf(pw[c - 1 - m], inter, intra));
          }
        });
    // dK~ = M2 Q~ + diag(gamma^{c-1-i}) V E^T   -> shared
    block_mm2<4, 4>(
        CS, D, c, [&](int m, int kk) { return M2[m * LDA + kk]; },
        [&](int kk, int nn) { return Qt[kk * LD + nn]; }, D,
        [&](int m, int kk) { return Vs[m * LD + kk]; },
        [&](int kk, int nn) { return E[nn * LD + kk]; },
        [&](int m, int nn, float intra, float inter) {
          dKs[m * LD + nn] = m < c ? fmaf(pw[c - 1 - m], inter, intra) : 0.f;
        });
    __syncthreads();
    for (int t = warp; t < c; t += NT / 32) {
      const size_t base = (((size_t)b * P.T + c0 + t) * P.H + h) * D;
      feature_backward<DT, D>(dKs + t * LD, k + base, rk[t], P.kscale, P.pos_offset + c0 + t, P,
                              lane, dk + base);
    }
    const float carry = pw[c];
    block_mm<4, 4>(
        D, D, c, [&](int m, int kk) { return Qt[kk * LD + m] * pw[kk + 1]; },
        [&](int kk, int nn) { return dOs[kk * LD + nn]; },
        [&](int m, int nn, float acc) { E[m * LD + nn] = fmaf(carry, E[m * LD + nn], acc); });
  }
}

template <int D>
size_t dq_smem() {
  using Dm = Dims<D>;
  return sizeof(float) * (Dm::STATE + 4 * Dm::TILE + Dm::SQ + 2 * CS + 1);
}
template <int D>
size_t gstate_smem() {
  using Dm = Dims<D>;
  return sizeof(float) * (Dm::STATE + 2 * Dm::TILE + CS + 1);
}
template <int D>
size_t dkdv_smem() {
  using Dm = Dims<D>;
  return sizeof(float) * (Dm::STATE + 5 * Dm::TILE + 2 * Dm::SQ + 2 * CS + 1);
}

template <typename K>
cudaError_t launch_seg(K kernel, size_t smem, const MixerParams &P, cudaStream_t st) {
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kernel<<<dim3(P.nseg, P.H, P.B), NT, smem, st>>>(P);
  return cudaGetLastError();
}

}  // namespace
}  // namespace simt

cudaError_t launch_simt_bwd_dq(const MixerParams &P, int dtype, cudaStream_t st) {
  using namespace simt;
  if (dtype == HLA_BF16)
    return P.D == 128 ? launch_seg(bwd_dq_kernel<__nv_bfloat16, 128>, dq_smem<128>(), P, st)
                      : launch_seg(bwd_dq_kernel<__nv_bfloat16, 64>, dq_smem<64>(), P, st);
  return P.D == 128 ? launch_seg(bwd_dq_kernel<float, 128>, dq_smem<128>(), P, st)
                    : launch_seg(bwd_dq_kernel<float, 64>, dq_smem<64>(), P, st);
}

cudaError_t launch_simt_seg_gstate(const MixerParams &P, int dtype, cudaStream_t st) {
  using namespace simt;
  if (dtype == HLA_BF16)
    return P.D == 128 ? launch_seg(seg_gstate_kernel<__nv_bfloat16, 128>, gstate_smem<128>(), P, st)
                      : launch_seg(seg_gstate_kernel<__nv_bfloat16, 64>, gstate_smem<64>(), P, st);
  return P.D == 128 ? launch_seg(seg_gstate_kernel<float, 128>, gstate_smem<128>(), P, st)
                    : launch_seg(seg_gstate_kernel<float, 64>, gstate_smem<64>(), P, st);
}

cudaError_t launch_simt_bwd_dkdv(const MixerParams &P, int dtype, cudaStream_t st) {
  using namespace simt;
  if (dtype == HLA_BF16)
    return P.D == 128 ? launch_seg(bwd_dkdv_kernel<__nv_bfloat16, 128>, dkdv_smem<128>(), P, st)
                      : launch_seg(bwd_dkdv_kernel<__nv_bfloat16, 64>, dkdv_smem<64>(), P, st);
  return P.D == 128 ? launch_seg(bwd_dkdv_kernel<float, 128>, dkdv_smem<128>(), P, st)
                    : launch_seg(bwd_dkdv_kernel<float, 64>, dkdv_smem<64>(), P, st);
}

}  // namespace hla
