// tc_prefill.cu — tensor-core (tcgen05) prefill for bf16 inputs at d = 128.
//
// The chunked form of Eq. 18 (arXiv 2601.22156, Appendix A): for a tile of
// c <= 128 tokens entering with state S,
//   P     = Q~ K~^T                                  MMA1  (M=128, N=128, K=d)
//   O_int = Q~ S                                     MMA2  (K = d_k)
//   S'    = gamma^c S + (diag(gamma^{c-1-j}) K~)^T V MMA4  (accumulated onto S in TMEM)
//   O_in  = (P (.) D) V,  D_ij = gamma^{i-j}, i >= j MMA3
//   o_i   = gamma^{i+1} O_int[i] + O_in[i],  y = Norm(o) * sigmoid(gate)
// The accumulators (P, O_int, O_in and the fp32 state S) live in the 512
// columns of tensor memory; operands are 16-bit tiles in shared memory in the
// 128-byte-swizzled layout of umma.cuh.  Q~, K~ and S enter MMA1/MMA2 as fp16
// (11-bit significand): with bf16 there, the rounding of q~ . k~ dominates the
// error of y wherever o nearly cancels (fast-decaying heads), which fp16 cuts
// fourfold.  S is scaled by a power of two into fp16 range each tile and the
// scale is undone in the epilogue.  P (.) D, K~dec and V stay bf16 (V is a
// bf16 input; MMA3/MMA4 run bf16 x bf16).  One CTA of 512 threads owns one
// (b, h, segment); every CUDA-core phase maps thread (warp w, lane l) to tile
// row i = 32 (w % 4) + l and column quarter (w / 4), which is also the TMEM
// lane / column block that warp may access.  Thread 0 issues the MMAs.
//
//   tc_state_kernel:  the segment's local state, S_seg = sum over its tokens
//                     of gamma^{end-s} k~_s^T v_s, one MMA per tile
//                     accumulated in TMEM (no rescaling between tiles: the
//                     decay weight of every key row is folded into K~).
//   tc_output_kernel: the outputs of the segment from the entering state
//                     written by the fp32 scan (scan.cu).
#include <cuda_fp16.h>

#include "hla_internal.cuh"
#include "umma.cuh"

namespace hla {
namespace tc {

namespace {

constexpr int D = 128;
constexpr int ROWS = 128;       // rows of every operand tile
constexpr int NT = 512;         // threads per CTA
constexpr int TILE = ROWS * D * 2;  // bytes of one bf16 tile (32 KiB)

// ------------------------------------------------------------------ small helpers

__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint4 pack8(const float *f) {
  return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}

__device__ __forceinline__ uint32_t pack2h(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint4 pack8h(const float *f) {
  return make_uint4(pack2h(f[0], f[1]), pack2h(f[2], f[3]), pack2h(f[4], f[5]),
                    pack2h(f[6], f[7]));
}

__device__ __forceinline__ void st_tile(unsigned char *tile, int row, int chunk, const uint4 &v) {
  *reinterpret_cast<uint4 *>(tile + umma::sw128_off(row, chunk, ROWS)) = v;
}

__device__ __forceinline__ uint4 ldg16(const void *p) {
  return __ldg(reinterpret_cast<const uint4 *>(p));
}

// Row `i` of token tile starting at c0 of a [B, T, H, D] bf16 tensor, uint4 index u (0..15).
__device__ __forceinline__ const __nv_bfloat16 *row_ptr(const void *X, const MixerParams &P, int b,
                                                        int h, long long t) {
  return (const __nv_bfloat16 *)X + (((size_t)b * P.T + t) * P.H + h) * D;
}

struct Shared {
  float red_q[4][ROWS];
  float red_k[4][ROWS];
  float red_o[4][ROWS];
  float2 rb[D / 2];
  float pw[ROWS + 1];
  float smax[NT / 32];
  uint64_t bar[2];
  uint32_t tmem_base;
};

// Loads of this thread's part of a q or k row: elements [16 qd, 16 qd + 16)
// and [64 + 16 qd, 64 + 16 qd + 16) (the two halves of its 16 RoPE pairs).
__device__ __forceinline__ void load_pairs(uint4 (&r)[4], const __nv_bfloat16 *row, int qd,
                                           bool valid) {
  if (valid) {
    r[0] = ldg16(row + 16 * qd);
    r[1] = ldg16(row + 16 * qd + 8);
    r[2] = ldg16(row + 64 + 16 * qd);
    r[3] = ldg16(row + 64 + 16 * qd + 8);
  } else {
    r[0] = r[1] = r[2] = r[3] = make_uint4(0, 0, 0, 0);
  }
}

// Loads of elements [32 qd, 32 qd + 32) of a row.
__device__ __forceinline__ void load_quarter(uint4 (&r)[4], const __nv_bfloat16 *row, int qd,
                                             bool valid) {
#pragma unroll
  for (int u = 0; u < 4; ++u) r[u] = valid ? ldg16(row + 32 * qd + 8 * u) : make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ float sumsq_pairs(const uint4 (&r)[4]) {
  float s = 0.f;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    float f[8];
    unpack8(r[u], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) s = fmaf(f[e], f[e], s);
  }
  return s;
}

// Rotate this thread's 16 pairs of a raw row (scaled by `scale`) with the
// per-pair cos/sin in (c, s); writes the 32 rotated values into lo/hi halves.
__device__ __forceinline__ void rotate(const uint4 (&r)[4], float scale, const float (&c)[16],
                                       const float (&s)[16], float (&lo)[16], float (&hi)[16]) {
  float a[16], b[16];
  unpack8(r[0], *reinterpret_cast<float(*)[8]>(&a[0]));
  unpack8(r[1], *reinterpret_cast<float(*)[8]>(&a[8]));
  unpack8(r[2], *reinterpret_cast<float(*)[8]>(&b[0]));
  unpack8(r[3], *reinterpret_cast<float(*)[8]>(&b[8]));
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const float x0 = a[u] * scale, x1 = b[u] * scale;
    lo[u] = x0 * c[u] - x1 * s[u];
    hi[u] = x0 * s[u] + x1 * c[u];
  }
}

// Store 32 values (pairs lo/hi of this thread) into a K-major feature tile
// row, as bf16 or (half = true) fp16.
__device__ __forceinline__ void store_pairs(unsigned char *tile, int row, int qd,
                                            const float (&lo)[16], const float (&hi)[16],
                                            float mul, bool half = false) {
  float t[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) t[u] = lo[u] * mul;
  st_tile(tile, row, 2 * qd, half ? pack8h(&t[0]) : pack8(&t[0]));
  st_tile(tile, row, 2 * qd + 1, half ? pack8h(&t[8]) : pack8(&t[8]));
#pragma unroll
  for (int u = 0; u < 16; ++u) t[u] = hi[u] * mul;
  st_tile(tile, row, 8 + 2 * qd, half ? pack8h(&t[0]) : pack8(&t[0]));
  st_tile(tile, row, 9 + 2 * qd, half ? pack8h(&t[8]) : pack8(&t[8]));
}

__device__ __forceinline__ void sync_tc() {
  umma::fence_before();
  __syncthreads();
  umma::fence_after();
}

// ------------------------------------------------------------------ local state pass

__global__ void __launch_bounds__(NT, 1) tc_state_kernel(const __grid_constant__ MixerParams P) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char *Kd[2] = {base, base + 2 * TILE};
  unsigned char *Vs[2] = {base + TILE, base + 3 * TILE};
  Shared &sh = *reinterpret_cast<Shared *>(base + 4 * TILE);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sub = warp & 3, qd = warp >> 2, i = 32 * sub + lane;
  const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int t0 = g * P.seg_len, t1 = min(P.T, t0 + P.seg_len);
  const int CV = P.chunk;
  const int L = t1 - t0;
  const float l2g = log2f(P.gamma[h]);

  if (tid == 0) {
    umma::mbar_init(&sh.bar[0], 1);
    umma::mbar_init(&sh.bar[1], 1);
    umma::mbar_fence_init();
  }
  if (warp == 0) umma::tmem_alloc(&sh.tmem_base, 128);
  // Per-thread rotation of its 16 pairs at offset i within a tile.
  float rc[16], rs[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) rope_cs(i, P.rope_u[16 * qd + u], rc[u], rs[u]);
  sync_tc();
  const uint32_t tm = sh.tmem_base;
  const uint32_t idesc = umma::idesc_bf16(128, 128, true, true);

  const int ntile = ceil_div(L, CV);
  bool failed = false;
  uint4 kr[4], vr[4];
  {
    const bool ok = i < min(CV, L);
    load_pairs(kr, row_ptr(P.k, P, b, h, t0 + (ok ? i : 0)), qd, ok);
    load_quarter(vr, row_ptr(P.v, P, b, h, t0 + (ok ? i : 0)), qd, ok);
  }
  for (int n = 0; n < ntile; ++n) {
    const int c0 = t0 + n * CV, c = min(CV, t1 - c0);
    const int buf = n & 1;
    // base rotation of this tile
    if (tid < D / 2) {
      float cc, ss;
      rope_cs(P.pos_offset + c0, P.rope_u[tid], cc, ss);
      sh.rb[tid] = make_float2(cc, ss);
    }
    sh.red_k[qd][i] = sumsq_pairs(kr);
    // buffer `buf` was read by the MMA of tile n - 2
    const bool late = n >= 2 && !umma::mbar_wait(&sh.bar[buf], ((n >> 1) - 1) & 1);
    umma::fence_after();
    if (__syncthreads_or(late)) {
      failed = true;
      break;
    }
    const float rk = rsqrtf((sh.red_k[0][i] + sh.red_k[1][i] + sh.red_k[2][i] + sh.red_k[3][i]) /
                                (float)D + P.eps);
    float cs[16], sn[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const float2 bb = sh.rb[16 * qd + u];
      cs[u] = bb.x * rc[u] - bb.y * rs[u];
      sn[u] = bb.y * rc[u] + bb.x * rs[u];
    }
    float lo[16], hi[16];
    rotate(kr, rk * P.kscale, cs, sn, lo, hi);
    // decay weight of this key row towards the end of the segment
    const float wgt = i < c ? exp2f((float)(L - 1 - (c0 - t0 + i)) * l2g) : 0.f;
    store_pairs(Kd[buf], i, qd, lo, hi, wgt);
#pragma unroll
    for (int u = 0; u < 4; ++u) st_tile(Vs[buf], i, 4 * qd + u, vr[u]);
    // prefetch the next tile
    if (n + 1 < ntile) {
      const int n0 = c0 + CV;
      const bool ok = i < min(CV, t1 - n0);
      load_pairs(kr, row_ptr(P.k, P, b, h, ok ? n0 + i : n0), qd, ok);
      load_quarter(vr, row_ptr(P.v, P, b, h, ok ? n0 + i : n0), qd, ok);
    }
    umma::fence_async_smem();
    sync_tc();
    if (tid == 0) {
      const uint32_t a = umma::smem_u32(Kd[buf]), bv = umma::smem_u32(Vs[buf]);
#pragma unroll
      for (int kk = 0; kk < ROWS / 16; ++kk)
        umma::mma_ss(tm, umma::desc_mnmajor(a, kk, ROWS), umma::desc_mnmajor(bv, kk, ROWS), idesc,
                     (n > 0 || kk > 0) ? 1u : 0u);
      umma::commit(&sh.bar[buf]);
    }
  }
  // wait for the last MMA (its completion covers all earlier ones)
  if (!failed) {
    const int last = ntile - 1;
    const bool late = !umma::mbar_wait(&sh.bar[last & 1], (last >> 1) & 1);
    umma::fence_after();
    failed = __syncthreads_or(late);
  }
  float *out = P.seg + (((size_t)b * P.H + h) * P.nseg + g) * (size_t)D * D;
  if (!failed) {
    float v[32];
    umma::tmem_ld32(tm + ((uint32_t)(32 * sub) << 16) + 32 * qd, v);
    float4 *o4 = reinterpret_cast<float4 *>(out + (size_t)i * D + 32 * qd);
#pragma unroll
    for (int u = 0; u < 8; ++u) o4[u] = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
  } else {
    const float nan = __int_as_float(0x7fc00000);
    for (int e = tid; e < D * D; e += NT) out[e] = nan;
    if (P.err) atomicOr(P.err, 1u);
  }
  sync_tc();
  if (warp == 0) umma::tmem_dealloc(tm, 128);
}

// ------------------------------------------------------------------ output pass

__global__ void __launch_bounds__(NT, 1) tc_output_kernel(const __grid_constant__ MixerParams P) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char *Qt = base, *Kt = base + TILE, *Kd = base + 2 * TILE, *Vs = base + 3 * TILE,
                *Pm = base + 4 * TILE, *Sb = base + 5 * TILE;
  Shared &sh = *reinterpret_cast<Shared *>(base + 6 * TILE);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sub = warp & 3, qd = warp >> 2, i = 32 * sub + lane;
  const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int t0 = g * P.seg_len, t1 = min(P.T, t0 + P.seg_len);
  const int CV = P.chunk;
  const float l2g = log2f(P.gamma[h]);

  if (tid == 0) {
    umma::mbar_init(&sh.bar[0], 1);
    umma::mbar_init(&sh.bar[1], 1);
    umma::mbar_fence_init();
  }
  if (tid <= ROWS) sh.pw[tid] = exp2f((float)tid * l2g);
  if (warp == 0) umma::tmem_alloc(&sh.tmem_base, 512);
  float rc[16], rs[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) rope_cs(i, P.rope_u[16 * qd + u], rc[u], rs[u]);
  sync_tc();
  const uint32_t tm = sh.tmem_base;
  const uint32_t lane_base = (uint32_t)(32 * sub) << 16;
  const uint32_t tP = tm, tOi = tm + 128, tOa = tm + 256, tS = tm + 384;

  // entering state of the segment -> TMEM (fp32)
  {
    const float *sin_ = P.seg + (((size_t)b * P.H + h) * P.nseg + g) * (size_t)D * D;
    const float4 *s4 = reinterpret_cast<const float4 *>(sin_ + (size_t)i * D + 32 * qd);
    float v[32];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float4 x = s4[u];
      v[4 * u] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
    }
    umma::tmem_st32(tS + lane_base + 32 * qd, v);
    umma::tmem_wait_st();
  }

  const uint32_t id_qk = umma::idesc_bf16(128, 128, false, false, true);  // fp16 Q~ K~^T
  const uint32_t id_qs = umma::idesc_bf16(128, 128, false, true, true);   // fp16 Q~ S
  const uint32_t id_pv = umma::idesc_bf16(128, 128, false, true);         // bf16 Pm V
  const uint32_t id_mn = umma::idesc_bf16(128, 128, true, true);          // bf16 K~dec^T V
  const int ntile = ceil_div(t1 - t0, CV);
  uint4 qr[4], kr[4];
  {
    const bool ok = i < min(CV, t1 - t0);
    load_pairs(qr, row_ptr(P.q, P, b, h, ok ? t0 + i : t0), qd, ok);
    load_pairs(kr, row_ptr(P.k, P, b, h, ok ? t0 + i : t0), qd, ok);
  }
  __nv_bfloat16 *y = (__nv_bfloat16 *)P.y;

  bool failed = false;
  for (int n = 0; n < ntile; ++n) {
    const int c0 = t0 + n * CV, c = min(CV, t1 - c0);
    const bool valid = i < c;
    if (tid < D / 2) {
      float cc, ss;
      rope_cs(P.pos_offset + c0, P.rope_u[tid], cc, ss);
      sh.rb[tid] = make_float2(cc, ss);
    }
    uint4 vr[4];
    load_quarter(vr, row_ptr(P.v, P, b, h, valid ? c0 + i : c0), qd, valid);
    // State phase, part 1: max |S| over the tile (S is fp32 in TMEM).
    {
      float v[32];
      umma::tmem_ld32(tS + lane_base + 32 * qd, v);
      float m = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) m = fmaxf(m, fabsf(v[e]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) sh.smax[warp] = m;
    }
    sh.red_q[qd][i] = sumsq_pairs(qr);
    sh.red_k[qd][i] = sumsq_pairs(kr);
    __syncthreads();
    // State phase, part 2: Sb = fp16(S * 2^-e) with 2^e >= max |S|; then S <- gamma^c S.
    float s_inv;  // 2^e: multiplies Q~ Sb back to the scale of S
    {
      float m = 0.f;
#pragma unroll
      for (int w = 0; w < NT / 32; ++w) m = fmaxf(m, sh.smax[w]);
      int e = 0;
      if (m > 0.f) frexpf(m, &e);
      const float s_fwd = ldexpf(1.f, -e);
      s_inv = ldexpf(1.f, e);
      float v[32];
      umma::tmem_ld32(tS + lane_base + 32 * qd, v);
      float t[8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
#pragma unroll
        for (int e2 = 0; e2 < 8; ++e2) t[e2] = v[8 * u + e2] * s_fwd;
        st_tile(Sb, i, 4 * qd + u, pack8h(t));
      }
      const float carry = sh.pw[c];
#pragma unroll
      for (int e2 = 0; e2 < 32; ++e2) v[e2] *= carry;
      umma::tmem_st32(tS + lane_base + 32 * qd, v);
    }
    // Feature map: q~ = RoPE(Norm(q)), k~ = RoPE(Norm(k)) / sqrt(d), k~dec = gamma^{c-1-i} k~.
    {
      const float rq = rsqrtf((sh.red_q[0][i] + sh.red_q[1][i] + sh.red_q[2][i] + sh.red_q[3][i]) /
                                  (float)D + P.eps);
      const float rk = rsqrtf((sh.red_k[0][i] + sh.red_k[1][i] + sh.red_k[2][i] + sh.red_k[3][i]) /
                                  (float)D + P.eps);
      float cs[16], sn[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float2 bb = sh.rb[16 * qd + u];
        cs[u] = bb.x * rc[u] - bb.y * rs[u];
        sn[u] = bb.y * rc[u] + bb.x * rs[u];
      }
      float lo[16], hi[16];
      rotate(qr, rq, cs, sn, lo, hi);
      store_pairs(Qt, i, qd, lo, hi, 1.f, true);
      rotate(kr, rk * P.kscale, cs, sn, lo, hi);
      store_pairs(Kt, i, qd, lo, hi, 1.f, true);
      store_pairs(Kd, i, qd, lo, hi, valid ? sh.pw[c - 1 - i] : 0.f);
#pragma unroll
      for (int u = 0; u < 4; ++u) st_tile(Vs, i, 4 * qd + u, vr[u]);
    }
    // prefetch the next tile's q and k rows
    if (n + 1 < ntile) {
      const int n0 = c0 + CV;
      const bool ok = i < min(CV, t1 - n0);
      load_pairs(qr, row_ptr(P.q, P, b, h, ok ? n0 + i : n0), qd, ok);
      load_pairs(kr, row_ptr(P.k, P, b, h, ok ? n0 + i : n0), qd, ok);
    }
    umma::tmem_wait_st();
    umma::fence_async_smem();
    sync_tc();
    if (tid == 0) {
      const uint32_t aq = umma::smem_u32(Qt), ak = umma::smem_u32(Kt), ad = umma::smem_u32(Kd),
                     av = umma::smem_u32(Vs), as = umma::smem_u32(Sb);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma::mma_ss(tP, umma::desc_kmajor(aq, kk, ROWS), umma::desc_kmajor(ak, kk, ROWS), id_qk,
                     kk > 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma::mma_ss(tOi, umma::desc_kmajor(aq, kk, ROWS), umma::desc_mnmajor(as, kk, ROWS), id_qs,
                     kk > 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma::mma_ss(tS, umma::desc_mnmajor(ad, kk, ROWS), umma::desc_mnmajor(av, kk, ROWS), id_mn,
                     1u);
      umma::commit(&sh.bar[0]);
    }
    uint4 gr[4];
    load_quarter(gr, row_ptr(P.g, P, b, h, valid ? c0 + i : c0), qd, valid);
    {
      const bool late = !umma::mbar_wait(&sh.bar[0], n & 1);
      umma::fence_after();
      if (__syncthreads_or(late)) {
        failed = true;
        break;
      }
    }
    // Mask: Pm = bf16((Q~ K~^T) (.) D), causal with gamma^{i-j}.
    {
      float v[32];
      umma::tmem_ld32(tP + lane_base + 32 * qd, v);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int j = 32 * qd + e;
        v[e] = (j <= i && valid) ? v[e] * sh.pw[i - j] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) st_tile(Pm, i, 4 * qd + u, pack8(&v[8 * u]));
    }
    umma::fence_async_smem();
    sync_tc();
    if (tid == 0) {
      const uint32_t ap = umma::smem_u32(Pm), av = umma::smem_u32(Vs);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma::mma_ss(tOa, umma::desc_kmajor(ap, kk, ROWS), umma::desc_mnmajor(av, kk, ROWS), id_pv,
                     kk > 0);
      umma::commit(&sh.bar[1]);
    }
    {
      const bool late = !umma::mbar_wait(&sh.bar[1], n & 1);
      umma::fence_after();
      if (__syncthreads_or(late)) {
        failed = true;
        break;
      }
    }
    // Epilogue: o = gamma^{i+1} O_int + O_in; y = Norm(o) * sigmoid(gate).
    float o[32];
    {
      float a[32];
      umma::tmem_ld32(tOi + lane_base + 32 * qd, a);
      umma::tmem_ld32(tOa + lane_base + 32 * qd, o);
      const float inter = sh.pw[i + 1] * s_inv;
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        o[e] = fmaf(inter, a[e], o[e]);
        ss = fmaf(o[e], o[e], ss);
      }
      sh.red_o[qd][i] = ss;
    }
    __syncthreads();
    if (valid) {
      const float ro = rsqrtf((sh.red_o[0][i] + sh.red_o[1][i] + sh.red_o[2][i] + sh.red_o[3][i]) /
                                  (float)D + P.eps);
      const size_t row = (((size_t)b * P.T + c0 + i) * P.H + h) * D + 32 * qd;
      uint4 *y4 = reinterpret_cast<uint4 *>(y + row);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float gf[8], t[8];
        unpack8(gr[u], gf);
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = o[8 * u + e] * ro * sigmoidf_(gf[e]);
        y4[u] = pack8(t);
      }
      if (P.o) {
        float4 *o4 = reinterpret_cast<float4 *>(P.o + row);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          o4[u] = make_float4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
      }
    }
  }
  if (failed && tid == 0 && P.err) atomicOr(P.err, 2u);
  sync_tc();
  if (warp == 0) umma::tmem_dealloc(tm, 512);
}

constexpr size_t kStateSmem = 4 * TILE + sizeof(Shared) + 1024;
constexpr size_t kOutputSmem = 6 * TILE + sizeof(Shared) + 1024;

}  // namespace
}  // namespace tc

bool tc_supported(const MixerParams &P, int dtype) { return dtype == HLA_BF16 && P.D == 128; }

cudaError_t launch_tc_seg_state(const MixerParams &P, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(tc::tc_state_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)tc::kStateSmem);
  if (e != cudaSuccess) return e;
  tc::tc_state_kernel<<<dim3(P.nseg, P.H, P.B), tc::NT, tc::kStateSmem, st>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_tc_seg_output(const MixerParams &P, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(tc::tc_output_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)tc::kOutputSmem);
  if (e != cudaSuccess) return e;
  tc::tc_output_kernel<<<dim3(P.nseg, P.H, P.B), tc::NT, tc::kOutputSmem, st>>>(P);
  return cudaGetLastError();
}

}  // namespace hla
