// decode_split.cu — one decode step of the Lightning Attention mixer (Eq. 18
// of arXiv 2601.22156, Appendix A, one new token per sequence) for small
// batches: the d_v columns of each (b, h) state are split over a thread-block
// cluster of C CTAs.
//
// At B * H of a few dozen, one CTA per (b, h) leaves most of the 152 SMs idle
// and each busy SM streams a whole 64 KiB state in and out.  Here CTA c of a
// cluster owns state columns [c d/C, (c + 1) d/C): it reads and writes only
// those (in place stays safe), normalises and rotates q and k itself (a few
// hundred bytes, recomputed by every CTA of the cluster), and forms o for its
// columns.  The output RMSNorm needs sum_j o_j^2 over all d columns: every CTA
// leaves its part in shared memory, and after a cluster barrier each reads the
// C parts over distributed shared memory in rank order (so every CTA adds
// them in the same order and gets the same norm).  A second cluster barrier
// keeps each CTA's shared memory alive until the others have read it.
#include "hla_internal.cuh"

namespace hla {

namespace {

constexpr int kSplitThreads = 128;

__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// A float in the shared memory of CTA `rank` of this cluster, at the offset
// that `p` has in this CTA's.
__device__ __forceinline__ float ld_cluster(const float *p, unsigned rank) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(r) : "memory");
  return v;
}

template <typename DT, int D, int C>
__global__ void __launch_bounds__(kSplitThreads) decode_split_kernel(const MixerParams P) {
  constexpr int W = D / C;                  // state columns of this CTA
  constexpr int TPR = W / 4;                // threads per state row (float4 each)
  constexpr int RPP = kSplitThreads / TPR;  // rows covered per pass
  constexpr int NR = D / RPP;               // rows per thread
  constexpr int NWARP = kSplitThreads / 32;
  static_assert(W % 4 == 0 && kSplitThreads % TPR == 0 && D % RPP == 0 && D <= kSplitThreads,
                "column split layout");
  __shared__ float sq[D], sk[D];
  __shared__ float4 red[RPP][TPR];
  __shared__ float wsum[NWARP];
  __shared__ float sscale[2];
  __shared__ float ssq;  // this CTA's part of sum o^2; read by the whole cluster

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned cr = cluster_rank();
  const int bh = blockIdx.x / C;
  const int b = bh / P.H, h = bh - b * P.H;
  const size_t row = (size_t)bh * D;                      // [B, 1, H, D]
  const size_t soff = (size_t)bh * D * D + (size_t)cr * W;  // column block of the state
  const int c4 = tid % TPR, r0 = tid / TPR;
  const int col = (int)cr * W + 4 * c4;  // first of this thread's four columns

  // 1. the state loads first: they are the long pole.
  float4 s[NR];
#pragma unroll
  for (int n = 0; n < NR; ++n)
    s[n] = __ldcs(reinterpret_cast<const float4 *>(P.state_in + soff + (size_t)(r0 + n * RPP) * D) + c4);

  // 2. token rows: all of q and k (the norms need them), this thread's v columns
  const DT *q = (const DT *)P.q, *k = (const DT *)P.k, *v = (const DT *)P.v, *g = (const DT *)P.g;
  if (tid < D) {
    sq[tid] = to_f(q[row + tid]);
    sk[tid] = to_f(k[row + tid]);
  }
  const float4 vv = make_float4(to_f(v[row + col]), to_f(v[row + col + 1]), to_f(v[row + col + 2]),
                                to_f(v[row + col + 3]));
  __syncthreads();
  if (warp < 2) {  // warp 0: RMS of q, warp 1: RMS of k
    const float *x = warp == 0 ? sq : sk;
    float a = 0.f;
    for (int i = lane; i < D; i += 32) a += x[i] * x[i];
    a = warp_sum(a);
    if (lane == 0) sscale[warp] = rsqrtf(a / (float)D + P.eps);
  }
  __syncthreads();
  const long long p = P.pos ? P.pos[b] : P.pos_offset;
  const int pi = tid;  // rotation pair (pi, pi + D/2) of this thread, for tid < D/2
  float qr[2] = {0.f, 0.f}, kr[2] = {0.f, 0.f};
  if (pi < D / 2) {
    float c, sn;
    rope_cs(p, P.rope_u[pi], c, sn);
    const float rq = sscale[0], rk = sscale[1] * P.kscale;
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

  // 3. S <- gamma S + k~^T v on this CTA's columns, written back; o partials.
  const float gm = P.gamma[h];
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int n = 0; n < NR; ++n) {
    const int r = r0 + n * RPP;
    const float kk = sk[r], qq = sq[r];
    float4 t = s[n];
    t.x = fmaf(gm, t.x, kk * vv.x);
    t.y = fmaf(gm, t.y, kk * vv.y);
    t.z = fmaf(gm, t.z, kk * vv.z);
    t.w = fmaf(gm, t.w, kk * vv.w);
    __stcs(reinterpret_cast<float4 *>(P.state_out + soff + (size_t)r * D) + c4, t);
    acc.x = fmaf(qq, t.x, acc.x);
    acc.y = fmaf(qq, t.y, acc.y);
    acc.z = fmaf(qq, t.z, acc.z);
    acc.w = fmaf(qq, t.w, acc.w);
  }
  red[r0][c4] = acc;
  __syncthreads();

  // 4. o_j over the row groups (thread j < W owns column cr W + j), the sum of
  // o^2 across the cluster, then RMSNorm(o) * sigmoid(gate).
  float oj = 0.f;
  if (tid < W) {
    const float *rf = reinterpret_cast<const float *>(&red[0][0]);
#pragma unroll
    for (int pp = 0; pp < RPP; ++pp) oj += rf[pp * W + tid];
  }
  const float part = warp_sum(tid < W ? oj * oj : 0.f);
  if (lane == 0) wsum[warp] = part;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < NWARP; ++w) t += wsum[w];
    ssq = t;
  }
  cluster_sync_all();  // every CTA's ssq is written
  float tot = 0.f;
  if (tid < W) {
#pragma unroll
    for (int c = 0; c < C; ++c) tot += ld_cluster(&ssq, (unsigned)c);
  }
  cluster_arrive();  // this CTA has read the others' ssq
  if (tid < W) {
    const int j = (int)cr * W + tid;
    const float ro = rsqrtf(tot / (float)D + P.eps);
    ((DT *)P.y)[row + j] = from_f<DT>(oj * ro * sigmoidf_(to_f(g[row + j])));
    if (P.o) P.o[row + j] = oj;
  }
  cluster_wait();  // nobody reads this CTA's ssq any more
}

template <typename DT, int D, int C>
cudaError_t launch_split_t(const MixerParams &P, cudaStream_t st) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)(P.B * P.H * C));
  cfg.blockDim = dim3(kSplitThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_split_kernel<DT, D, C>, P);
}

template <typename DT, int D>
cudaError_t launch_split_d(const MixerParams &P, int split, cudaStream_t st) {
  switch (split) {
    case 2: return launch_split_t<DT, D, 2>(P, st);
    case 4: return launch_split_t<DT, D, 4>(P, st);
    case 8: return launch_split_t<DT, D, 8>(P, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode_split(const MixerParams &P, int dtype, int split, cudaStream_t st) {
  if (dtype == HLA_BF16)
    return P.D == 128 ? launch_split_d<__nv_bfloat16, 128>(P, split, st)
                      : launch_split_d<__nv_bfloat16, 64>(P, split, st);
  return P.D == 128 ? launch_split_d<float, 128>(P, split, st) : launch_split_d<float, 64>(P, split, st);
}

}  // namespace hla
