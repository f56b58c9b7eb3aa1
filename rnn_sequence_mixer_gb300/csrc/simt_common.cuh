// simt_common.cuh — building blocks of the fp32 CUDA-core (SIMT) chunked
// kernels: shared-memory tiles, a register-tiled shared-memory matrix product
// and the row-wise QK-norm + RoPE feature map.
//
// The SIMT kernels evaluate the mixer in the chunked (block) form of the
// recurrence of Eq. 18 (arXiv 2601.22156, Appendix A): for a chunk of c
// tokens starting with state S,
//   O     = diag(gamma^{i+1}) Q~ S + (Q~ K~^T (.) D) V,   D_ij = gamma^{i-j} (i >= j)
//   S'    = gamma^c S + (diag(gamma^{c-1-j}) K~)^T V
// with every product accumulated in fp32.  They serve fp32 inputs (which need
// fp32 accuracy end to end) and every shape the tensor-core path does not.
#pragma once

#include "hla_internal.cuh"

namespace hla {
namespace simt {

constexpr int NT = 256;  // threads per CTA (8 warps)
constexpr int CS = 32;   // tokens per sub-chunk

template <int D>
struct Dims {
  static constexpr int LD = D + 1;    // padded row stride of [rows][D] tiles (bank-conflict free
                                      // for both row- and column-wise walks)
  static constexpr int LDA = CS + 1;  // padded row stride of CS x CS tiles
  static constexpr int TILE = CS * LD;
  static constexpr int STATE = D * LD;
  static constexpr int SQ = CS * LDA;
};

// For every (m, n) in [0, M) x [0, N): epi(m, n, sum_{k<K} A(m, k) B(k, n)).
// Each thread owns a TM x TN micro-tile whose rows are M/TM apart and whose
// columns are N/TN apart, so consecutive threads touch consecutive columns.
template <int TM, int TN, typename FA, typename FB, typename FE>
__device__ __forceinline__ void block_mm(int M, int N, int K, FA A, FB B, FE epi) {
  const int gm = M / TM, gn = N / TN;
  for (int t = threadIdx.x; t < gm * gn; t += NT) {
    const int tm = t / gn, tn = t - (t / gn) * gn;
    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
    for (int kk = 0; kk < K; ++kk) {
      float a[TM], b[TN];
#pragma unroll
      for (int i = 0; i < TM; ++i) a[i] = A(tm + i * gm, kk);
#pragma unroll
      for (int j = 0; j < TN; ++j) b[j] = B(kk, tn + j * gn);
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) epi(tm + i * gm, tn + j * gn, acc[i][j]);
  }
}

// Two products sharing the output grid: epi(m, n, sum_k A1 B1, sum_k A2 B2).
template <int TM, int TN, typename FA1, typename FB1, typename FA2, typename FB2, typename FE>
__device__ __forceinline__ void block_mm2(int M, int N, int K1, FA1 A1, FB1 B1, int K2, FA2 A2,
                                          FB2 B2, FE epi) {
  const int gm = M / TM, gn = N / TN;
  for (int t = threadIdx.x; t < gm * gn; t += NT) {
    const int tm = t / gn, tn = t - (t / gn) * gn;
    float acc1[TM][TN], acc2[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) acc1[i][j] = acc2[i][j] = 0.f;
    for (int kk = 0; kk < K1; ++kk) {
      float a[TM], b[TN];
#pragma unroll
      for (int i = 0; i < TM; ++i) a[i] = A1(tm + i * gm, kk);
#pragma unroll
      for (int j = 0; j < TN; ++j) b[j] = B1(kk, tn + j * gn);
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc1[i][j] = fmaf(a[i], b[j], acc1[i][j]);
    }
    for (int kk = 0; kk < K2; ++kk) {
      float a[TM], b[TN];
#pragma unroll
      for (int i = 0; i < TM; ++i) a[i] = A2(tm + i * gm, kk);
#pragma unroll
      for (int j = 0; j < TN; ++j) b[j] = B2(kk, tn + j * gn);
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc2[i][j] = fmaf(a[i], b[j], acc2[i][j]);
    }
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) epi(tm + i * gm, tn + j * gn, acc1[i][j], acc2[i][j]);
  }
}

// Rows [c0, c0 + c) of a [B, T, H, D] tensor for (b, h) into a CS x LD fp32
// tile; rows >= c are zero.
template <typename DT, int D>
__device__ __forceinline__ void load_tile(float *tile, const DT *X, const MixerParams &P, int b,
                                          int h, int c0, int c) {
  constexpr int LD = Dims<D>::LD;
  const size_t tstride = (size_t)P.H * D;
  const size_t base = (((size_t)b * P.T + c0) * P.H + h) * D;
  for (int idx = threadIdx.x; idx < CS * D; idx += NT) {
    const int t = idx / D, j = idx - (idx / D) * D;
    tile[t * LD + j] = t < c ? to_f(X[base + (size_t)t * tstride + j]) : 0.f;
  }
}

// In-place feature map of one token: x <- RoPE_p(x * r_x) * scale for the q
// row (scale 1) and the k row (scale kscale), sharing the rotation angles.
// Executed by one warp; returns the RMS scales through rq / rk.
template <int D>
__device__ __forceinline__ void feature_qk(float *xq, float *xk, long long p,
                                           const MixerParams &P, int lane, float &rq, float &rk) {
  float aq = 0.f, ak = 0.f;
  for (int i = lane; i < D; i += 32) {
    aq += xq[i] * xq[i];
    ak += xk[i] * xk[i];
  }
  aq = warp_sum(aq);
  ak = warp_sum(ak);
  rq = rsqrtf(aq / (float)D + P.eps);
  rk = rsqrtf(ak / (float)D + P.eps);
  const float sk = rk * P.kscale;
  for (int i = lane; i < D / 2; i += 32) {
    float c, s;
    rope_cs(p, P.rope_u[i], c, s);
    float u = xq[i] * rq, w = xq[i + D / 2] * rq;
    xq[i] = u * c - w * s;
    xq[i + D / 2] = u * s + w * c;
    u = xk[i] * sk;
    w = xk[i + D / 2] * sk;
    xk[i] = u * c - w * s;
    xk[i + D / 2] = u * s + w * c;
  }
}

// The same map for a single row: x <- RoPE_p(x * r_x) * scale; returns r_x.
template <int D>
__device__ __forceinline__ float feature_one(float *x, long long p, const MixerParams &P, int lane,
                                             float scale) {
  float a = 0.f;
  for (int i = lane; i < D; i += 32) a += x[i] * x[i];
  a = warp_sum(a);
  const float r = rsqrtf(a / (float)D + P.eps);
  const float rs = r * scale;
  for (int i = lane; i < D / 2; i += 32) {
    float c, s;
    rope_cs(p, P.rope_u[i], c, s);
    const float u = x[i] * rs, w = x[i + D / 2] * rs;
    x[i] = u * c - w * s;
    x[i + D / 2] = u * s + w * c;
  }
  return r;
}

// Gradient of a raw row x through x -> RoPE_p(Norm(x)) * scale, given the
// gradient gf of the feature (a D-vector in shared memory) and the RMS scale
// r of x.  Executed by one warp; writes D elements of out.
//   dn  = RoPE_p^T gf * scale
//   dx  = r (dn - n mean(dn * n)),  n = x r
template <typename DT, int D>
__device__ __forceinline__ void feature_backward(const float *gf, const DT *x, float r, float scale,
                                                 long long p, const MixerParams &P, int lane,
                                                 DT *out) {
  constexpr int NP = (D / 2 + 31) / 32;
  float dn0[NP], dn1[NP], n0[NP], n1[NP];
  float m = 0.f;
#pragma unroll
  for (int u = 0; u < NP; ++u) {
    const int i = lane + 32 * u;
    dn0[u] = dn1[u] = n0[u] = n1[u] = 0.f;
    if (i < D / 2) {
      float c, s;
      rope_cs(p, P.rope_u[i], c, s);
      const float a = gf[i] * scale, b = gf[i + D / 2] * scale;
      dn0[u] = a * c + b * s;
      dn1[u] = -a * s + b * c;
      n0[u] = to_f(x[i]) * r;
      n1[u] = to_f(x[i + D / 2]) * r;
      m += dn0[u] * n0[u] + dn1[u] * n1[u];
    }
  }
  m = warp_sum(m) / (float)D;
#pragma unroll
  for (int u = 0; u < NP; ++u) {
    const int i = lane + 32 * u;
    if (i < D / 2) {
      out[i] = from_f<DT>(r * (dn0[u] - n0[u] * m));
      out[i + D / 2] = from_f<DT>(r * (dn1[u] - n1[u] * m));
    }
  }
}

template <int D>
__device__ __forceinline__ void fill_pow(float *pw, float l2g) {
  for (int i = threadIdx.x; i <= CS; i += NT) pw[i] = gpow(l2g, (float)i);
}

}  // namespace simt
}  // namespace hla
