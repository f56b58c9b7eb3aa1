// decode.cu — one decode step of the Lightning Attention mixer (Eq. 18 of
// arXiv 2601.22156, Appendix A, for a single new token per sequence).
//
// The step is bound by HBM: per (b, h) it reads and writes the d x d fp32
// state once (2 * 4 d^2 bytes) and touches only 5 d-vectors besides.  One CTA
// owns one (b, h).  Every thread first issues all of its state loads (16-byte
// vectors, a warp covers one 512-byte state row at d = 128), then the CTA
// normalises and rotates q and k while those loads are in flight, updates its
// slice S <- gamma S + k~^T v, streams it back, and accumulates its share of
// o = q~ S.  A shared-memory reduction finishes o, the output RMSNorm and the
// sigmoid gate.
#include "hla_internal.cuh"

namespace hla {

namespace {

constexpr int kDecodeThreads = 256;

template <typename DT, int D>
__global__ void __launch_bounds__(kDecodeThreads) decode_kernel(const MixerParams P) {
  constexpr int TPR = D / 4;                // threads per state row (float4 each)
  constexpr int RPP = kDecodeThreads / TPR; // rows covered per pass
  constexpr int NR = D / RPP;               // rows per thread
  __shared__ float sq[D], sk[D], sv[D], sg[D];
  __shared__ float4 red[RPP][TPR];
  __shared__ float ssum[kDecodeThreads / 32];
  __shared__ float sscale[2];

  const int tid = threadIdx.x;
  const int bh = blockIdx.x;
  const int b = bh / P.H, h = bh - b * P.H;
  const size_t row = (size_t)bh * D;  // [B, 1, H, D]
  const size_t soff = (size_t)bh * D * D;
  const int c4 = tid % TPR, r0 = tid / TPR;

  // 1. issue the state loads first: they are the long pole.
  const float4 *Sin = reinterpret_cast<const float4 *>(P.state_in + soff);
  float4 s[NR];
#pragma unroll
  for (int n = 0; n < NR; ++n) s[n] = __ldcs(&Sin[(size_t)(r0 + n * RPP) * TPR + c4]);

  // 2. token rows
  const DT *q = (const DT *)P.q, *k = (const DT *)P.k, *v = (const DT *)P.v, *g = (const DT *)P.g;
  for (int i = tid; i < D; i += kDecodeThreads) {
    sq[i] = to_f(q[row + i]);
    sk[i] = to_f(k[row + i]);
    sv[i] = to_f(v[row + i]);
    sg[i] = to_f(g[row + i]);
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  if (warp < 2) {  // warp 0: RMS of q, warp 1: RMS of k
    const float *x = warp == 0 ? sq : sk;
    float a = 0.f;
    for (int i = lane; i < D; i += 32) a += x[i] * x[i];
    a = warp_sum(a);
    if (lane == 0) sscale[warp] = rsqrtf(a / (float)D + P.eps);
  }
  __syncthreads();
  const long long p = P.pos ? P.pos[b] : P.pos_offset;
  float qr[2] = {0.f, 0.f}, kr[2] = {0.f, 0.f};
  int pi = tid;  // pair index handled by this thread (tid < D/2)
  if (pi < D / 2) {
    float c, sn;
    rope_cs(p, P.rope_u[pi], c, sn);
    float rq = sscale[0], rk = sscale[1] * P.kscale;
    float a = sq[pi] * rq, bb = sq[pi + D / 2] * rq;
    qr[0] = a * c - bb * sn;
    qr[1] = a * sn + bb * c;
    a = sk[pi] * rk;
    bb = sk[pi + D / 2] * rk;
    kr[0] = a * c - bb * sn;
    kr[1] = a * sn + bb * c;
  }
  __syncthreads();
  if (pi < D / 2) {
    sq[pi] = qr[0];
    sq[pi + D / 2] = qr[1];
    sk[pi] = kr[0];
    sk[pi + D / 2] = kr[1];
  }
  __syncthreads();

  // 3. S <- gamma S + k~^T v, written back; o partials = q~ S.
  const float gm = P.gamma[h];
  const float4 vv = reinterpret_cast<const float4 *>(sv)[c4];
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 *Sout = reinterpret_cast<float4 *>(P.state_out + soff);
#pragma unroll
  for (int n = 0; n < NR; ++n) {
    const int r = r0 + n * RPP;
    const float kk = sk[r], qq = sq[r];
    float4 t = s[n];
    t.x = fmaf(gm, t.x, kk * vv.x);
    t.y = fmaf(gm, t.y, kk * vv.y);
    t.z = fmaf(gm, t.z, kk * vv.z);
    t.w = fmaf(gm, t.w, kk * vv.w);
    __stcs(&Sout[(size_t)r * TPR + c4], t);
    acc.x = fmaf(qq, t.x, acc.x);
    acc.y = fmaf(qq, t.y, acc.y);
    acc.z = fmaf(qq, t.z, acc.z);
    acc.w = fmaf(qq, t.w, acc.w);
  }
  red[r0][c4] = acc;
  __syncthreads();

  // 4. o_j = sum over row groups; RMSNorm(o) * sigmoid(gate).
  float oj = 0.f;
  if (tid < D) {
    const float *rf = reinterpret_cast<const float *>(&red[0][0]);
#pragma unroll
    for (int pp = 0; pp < RPP; ++pp) oj += rf[pp * D + tid];
  }
  float sq_part = warp_sum(tid < D ? oj * oj : 0.f);
  if (lane == 0) ssum[warp] = sq_part;
  __syncthreads();
  if (tid < D) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeThreads / 32; ++w) tot += ssum[w];
    const float ro = rsqrtf(tot / (float)D + P.eps);
    const float yj = oj * ro * sigmoidf_(sg[tid]);
    ((DT *)P.y)[row + tid] = from_f<DT>(yj);
    if (P.o) P.o[row + tid] = oj;
  }
}

}  // namespace

cudaError_t launch_decode(const MixerParams &P, int dtype, cudaStream_t st) {
  dim3 grid(P.B * P.H);
  if (dtype == HLA_BF16) {
    if (P.D == 128) decode_kernel<__nv_bfloat16, 128><<<grid, kDecodeThreads, 0, st>>>(P);
    else decode_kernel<__nv_bfloat16, 64><<<grid, kDecodeThreads, 0, st>>>(P);
  } else {
    if (P.D == 128) decode_kernel<float, 128><<<grid, kDecodeThreads, 0, st>>>(P);
    else decode_kernel<float, 64><<<grid, kDecodeThreads, 0, st>>>(P);
  }
  return cudaGetLastError();
}

}  // namespace hla
