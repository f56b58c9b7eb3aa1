// tc_common.cuh — pieces shared by the tensor-core (tcgen05) kernels of the
// prefill and of its backward: operand-tile geometry, 16-bit packing, the
// q/k feature map (RMSNorm, RoPE) applied in place on swizzled tiles,
// barriers with bounded waits, and the TMA descriptors of [B, T, H, 128]
// 16-bit tensors.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "hla_internal.cuh"
#include "umma.cuh"

namespace hla {
namespace tc {

namespace {

constexpr int D = 128;
constexpr int ROWS = 128;           // rows of every operand tile
constexpr int NWORK = 16;              // worker warps (CUDA-core work), 4 warpgroups
constexpr int NTO = (NWORK + 4) * 32;  // + one warpgroup: its first warp issues MMAs / TMA copies
                                       // (registers are granted per warpgroup, so a lone 17th
                                       // warp would cost as much as four)
constexpr int DM_STRIDE = 264;      // row pitch (floats) of the causal-mask decay table
constexpr int TILE = ROWS * D * 2;  // bytes of one 16-bit tile (32 KiB)
constexpr int HALF_TILE = TILE / 2; // one 64-column block

// ------------------------------------------------------------------ small helpers

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t pack2h(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

// ------------------------------------------------------------------ packed fp32
// sm_100-class SMs run fp32 multiplies and FMAs on register pairs
// (mul.rn.f32x2, fma.rn.f32x2): one instruction does two lanes of work with the
// rounding of the scalar forms.  The element-wise phases use them to halve
// their share of the issue slots.
typedef unsigned long long f2;  // {lo, hi}

__device__ __forceinline__ f2 mk2(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ f2 dup2(float x) { return mk2(x, x); }
__device__ __forceinline__ void split2(f2 r, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ float hsum2(f2 r) {
  float lo, hi;
  split2(r, lo, hi);
  return lo + hi;
}
// bf16x2 / fp16x2 word <-> two fp32 lanes
__device__ __forceinline__ f2 f2_of_bf(uint32_t w) {
  return mk2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ f2 f2_of_h(uint32_t w) {
  const float2 t = __half22float2(*reinterpret_cast<const __half2 *>(&w));
  return mk2(t.x, t.y);
}
__device__ __forceinline__ uint32_t bf_of_f2(f2 r) {
  float lo, hi;
  split2(r, lo, hi);
  return pack2(lo, hi);
}
__device__ __forceinline__ uint32_t h_of_f2(f2 r) {
  float lo, hi;
  split2(r, lo, hi);
  return pack2h(lo, hi);
}
// the eight bf16 (fp16) of a 16-byte chunk as four fp32 pairs, and back
__device__ __forceinline__ void unpack4x2(const uint4 &u, f2 (&x)[4]) {
  x[0] = f2_of_bf(u.x); x[1] = f2_of_bf(u.y); x[2] = f2_of_bf(u.z); x[3] = f2_of_bf(u.w);
}
__device__ __forceinline__ void unpack4x2h(const uint4 &u, f2 (&x)[4]) {
  x[0] = f2_of_h(u.x); x[1] = f2_of_h(u.y); x[2] = f2_of_h(u.z); x[3] = f2_of_h(u.w);
}
__device__ __forceinline__ uint4 pack4x2(const f2 *x) {
  return make_uint4(bf_of_f2(x[0]), bf_of_f2(x[1]), bf_of_f2(x[2]), bf_of_f2(x[3]));
}
__device__ __forceinline__ uint4 pack4x2h(const f2 *x) {
  return make_uint4(h_of_f2(x[0]), h_of_f2(x[1]), h_of_f2(x[2]), h_of_f2(x[3]));
}
// 32 fp32 values (a TMEM row slice) as 16 pairs, and back
__device__ __forceinline__ void pairs_of(const float (&v)[32], f2 (&x)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) x[e] = mk2(v[2 * e], v[2 * e + 1]);
}
__device__ __forceinline__ void floats_of(const f2 (&x)[16], float (&v)[32]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) split2(x[e], v[2 * e], v[2 * e + 1]);
}

__device__ __forceinline__ uint4 *tile_at(unsigned char *tile, int row, int chunk) {
  return reinterpret_cast<uint4 *>(tile + umma::sw128_off(row, chunk, ROWS));
}

// This thread's 16 RoPE pairs of a row sit in chunks {2qd, 2qd+1} (elements
// 16qd..16qd+15) and {8+2qd, 9+2qd} (elements 64+16qd..): read them from an
// operand tile.
__device__ __forceinline__ void ld_pairs(unsigned char *tile, int row, int qd, uint4 (&r)[4]) {
  r[0] = *tile_at(tile, row, 2 * qd);
  r[1] = *tile_at(tile, row, 2 * qd + 1);
  r[2] = *tile_at(tile, row, 8 + 2 * qd);
  r[3] = *tile_at(tile, row, 9 + 2 * qd);
}

__device__ __forceinline__ float sumsq_pairs(const uint4 (&r)[4]) {
  f2 s = 0ull;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    f2 x[4];
    unpack4x2(r[u], x);
#pragma unroll
    for (int e = 0; e < 4; ++e) s = fma2(x[e], x[e], s);
  }
  return hsum2(s);
}

// one pass over this lane's pairs of a row: sums of a_e^2, b_e^2 and a_e b_e
// (fp32; the raw q . k gives the fp32 diagonal q~_i . k~_i)
__device__ __forceinline__ void norms_and_dot(const uint4 (&a)[4], const uint4 (&b)[4],
                                              float &saa, float &sbb, float &sab) {
  f2 aa = 0ull, bb = 0ull, ab = 0ull;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    f2 x[4], y[4];
    unpack4x2(a[u], x);
    unpack4x2(b[u], y);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      aa = fma2(x[e], x[e], aa);
      bb = fma2(y[e], y[e], bb);
      ab = fma2(x[e], y[e], ab);
    }
  }
  saa = hsum2(aa);
  sbb = hsum2(bb);
  sab = hsum2(ab);
}

// cos / sin of the RoPE angle of pair u at position p on the special-function
// unit.  The exact fixed-point phase t (turns, mod 1) becomes a float without a
// conversion instruction: its top 23 bits under the exponent of 1.0 give
// f = 1 + t, and x = 2 pi (1.5 - f) = pi - 2 pi t lies in (-pi, pi], where
// sin x = sin(2 pi t) and cos x = -cos(2 pi t).  Absolute error ~1e-6, far below
// the 16-bit rounding of the operands.
__device__ __forceinline__ void rope_fast(long long p, unsigned long long u, float &c, float &s) {
  const unsigned long long ph = (unsigned long long)p * u;
  const float f = __uint_as_float(0x3f800000u | ((uint32_t)(ph >> 32) >> 9));
  const float x = fmaf(f, -6.2831853071795865f, 9.4247779607693797f);
  float cx;
  __sincosf(x, &s, &cx);
  c = -cx;
}

// Shared-memory copy of MixerParams::rope_u, transposed so that the four lanes
// that own pair groups 0..3 of a row read consecutive words:
// ru[4 m + g] = rope_u[16 g + m] for pair m of group g.
__device__ __forceinline__ void load_rope_table(unsigned long long *ru, const MixerParams &P,
                                                int tid) {
  if (tid < kMaxPairs) ru[4 * (tid & 15) + (tid >> 4)] = P.rope_u[tid];
}

// the hardware tanh (sigmoid through it: 1 / (1 + e^-z) = 0.5 + 0.5 tanh(z / 2)).
__device__ __forceinline__ float tanh_fast(float x) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(x));
  return t;
}

// the special-function unit's reciprocal (one instruction; the forward's gate
// and the backward's division by it both use it, so they agree bit for bit)
__device__ __forceinline__ float rcp_fast(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// sigmoid of two lanes as 1 / (1 + 2^(-z log2 e)): unlike 0.5 + 0.5 tanh(z / 2)
// it stays above 0 (and keeps its relative precision) down to z ~ -87, so a
// gated output y = n sigmoid(z) can be divided by it again (the backward's
// dq pass from y).  The forward's gate and that division use this one form.
__device__ __forceinline__ f2 sigmoid_e2(f2 z) {
  const f2 t2 = mul2(z, dup2(-1.4426950408889634f));
  float a, b;
  split2(t2, a, b);
  float ea, eb;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(ea) : "f"(a));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(eb) : "f"(b));
  return mk2(rcp_fast(1.f + ea), rcp_fast(1.f + eb));
}
// The same sigmoid and its reciprocal 1 + 2^(-z log2 e) (exact in the first
// rounding: what the forward divided by), for dividing y again.
__device__ __forceinline__ void sigmoid_e2_inv(f2 z, f2 &sg, f2 &inv) {
  const f2 t2 = mul2(z, dup2(-1.4426950408889634f));
  float a, b;
  split2(t2, a, b);
  float ea, eb;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(ea) : "f"(a));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(eb) : "f"(b));
  const float ia = 1.f + ea, ib = 1.f + eb;
  sg = mk2(rcp_fast(ia), rcp_fast(ib));
  inv = mk2(ia, ib);
}

// Decay table of the causal mask, read backwards, in four copies shifted by
// one element so that every lane's 32 weights start 16-byte aligned:
// dm[cp][x] = gamma^(127 - x - cp) for x + cp <= 127, else 0.  Rows are padded
// to DM_STRIDE floats so that the eight lanes of a quarter-warp hit distinct
// banks.  Filled by all `nthreads` threads of the CTA.
__device__ __forceinline__ void fill_mask_table(float (*dm)[DM_STRIDE], float log2g, int tid,
                                                int nthreads) {
  for (int e = tid; e < 4 * DM_STRIDE; e += nthreads) {
    const int cp = e / DM_STRIDE, x = e % DM_STRIDE;
    dm[cp][x] = x + cp <= ROWS - 1 ? exp2f((float)(ROWS - 1 - x - cp) * log2g) : 0.f;
  }
}

// Causal decay of columns [col, col + 32) of score row i, in place on 16
// pairs: x_j *= gamma^(i - j) for j <= i, 0 for j > i.  The weight of column
// col + e is dm[cp][s0 - cp + e] with s0 = 127 - i + col, cp = s0 & 3.
__device__ __forceinline__ void mask_lower_table(f2 (&x)[16], const float (*dm)[DM_STRIDE], int i,
                                                 int col) {
  const int s0 = ROWS - 1 - i + col, cp = s0 & 3;
  const float4 *wt = reinterpret_cast<const float4 *>(&dm[cp][s0 - cp]);
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const float4 w = wt[u];
    x[2 * u] = mul2(x[2 * u], mk2(w.x, w.y));
    x[2 * u + 1] = mul2(x[2 * u + 1], mk2(w.z, w.w));
  }
}

// The transposed mask's table: du[cp][y] = gamma^(y + cp - 127) for
// y + cp >= 127, else 0 (same layout and padding as fill_mask_table).
__device__ __forceinline__ void fill_mask_table_upper(float (*du)[DM_STRIDE], float log2g, int tid,
                                                      int nthreads) {
  for (int e = tid; e < 4 * DM_STRIDE; e += nthreads) {
    const int cp = e / DM_STRIDE, x = e % DM_STRIDE + cp;
    du[cp][e % DM_STRIDE] = x >= ROWS - 1 ? exp2f((float)(x - (ROWS - 1)) * log2g) : 0.f;
  }
}

// Transposed causal decay of columns [col, col + 32) of row i, in place:
// x_j *= gamma^(j - i) for j >= i, 0 for j < i.  The weight of column col + e
// is du[cp][s - cp + e] with s = 127 + col - i, cp = s & 3.
__device__ __forceinline__ void mask_upper_table(f2 (&x)[16], const float (*du)[DM_STRIDE], int i,
                                                 int col) {
  const int s = ROWS - 1 + col - i, cp = s & 3;
  const float4 *wt = reinterpret_cast<const float4 *>(&du[cp][s - cp]);
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const float4 w = wt[u];
    x[2 * u] = mul2(x[2 * u], mk2(w.x, w.y));
    x[2 * u + 1] = mul2(x[2 * u + 1], mk2(w.z, w.w));
  }
}

// RoPE of one 8-element chunk pair, two fp32 lanes at a time: lo = x0 c - x1 s,
// hi = x0 s + x1 c for x0 = a r, x1 = b r (a: first-half elements, b: their
// partners d/2 further on).  cs / sn / nsn hold cos, sin and -sin of the 8 angles.
__device__ __forceinline__ void rotate8(const uint4 &a, const uint4 &b, f2 r, const f2 (&cs)[4],
                                       const f2 (&sn)[4], const f2 (&nsn)[4], f2 (&lo)[4],
                                       f2 (&hi)[4]) {
  f2 xa[4], xb[4];
  unpack4x2(a, xa);
  unpack4x2(b, xb);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const f2 x0 = mul2(xa[e], r), x1 = mul2(xb[e], r);
    lo[e] = fma2(x0, cs[e], mul2(x1, nsn[e]));
    hi[e] = fma2(x0, sn[e], mul2(x1, cs[e]));
  }
}

// cos, sin, -sin of this thread's 8 angles of half `hf` at position p, paired.
__device__ __forceinline__ void rope8(long long p, const unsigned long long *ru, int hf, int qd,
                                      f2 (&cs)[4], f2 (&sn)[4], f2 (&nsn)[4]) {
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float c0, s0, c1, s1;
    rope_fast(p, ru[4 * (8 * hf + 2 * e) + qd], c0, s0);
    rope_fast(p, ru[4 * (8 * hf + 2 * e + 1) + qd], c1, s1);
    cs[e] = mk2(c0, c1);
    sn[e] = mk2(s0, s1);
    nsn[e] = mk2(-s0, -s1);
  }
}

// ------------------------------------------------------------------ RoPE angles by angle addition
// The angle of pair m at position p0 + b is the sum of its angles at p0 and at
// b, so cos / sin at p0 + b follow from those at p0 (computed once per group
// of 8 rows) and at b = 0..7 (a per-CTA table) with one complex product:
// four packed FMAs for two angles instead of the fixed-point phase and the
// special-function unit for each.  A RopeTab holds one position's 64 angles
// as float4 {cos m, cos m+1, sin m, sin m+1} for m = 16 qd + 2 jj at [qd][jj];
// the padding entry staggers the four quarters across the banks.
struct RopeTab {
  float4 v[4][9];
};

// Entry (qd, jj) of the table of position p, from the exact phase (rope_fast);
// `ru` is the kernel's load_rope_table copy.
__device__ __forceinline__ float4 rope_entry(long long p, const unsigned long long *ru, int qd, int jj) {
  float c0, s0, c1, s1;
  rope_fast(p, ru[4 * (2 * jj) + qd], c0, s0);
  rope_fast(p, ru[4 * (2 * jj + 1) + qd], c1, s1);
  return make_float4(c0, c1, s0, s1);
}

// The eight small-offset tables, b = 0..7 (the whole CTA, before its first barrier).
__device__ __forceinline__ void fill_rope_small(RopeTab *small, const unsigned long long *ru_global,
                                                int tid, int nthreads) {
  for (int e = tid; e < 8 * 32; e += nthreads) {
    const int b = e >> 5, qd = (e >> 3) & 3, jj = e & 7;
    float c0, s0, c1, s1;
    rope_fast(b, ru_global[16 * qd + 2 * jj], c0, s0);
    rope_fast(b, ru_global[16 * qd + 2 * jj + 1], c1, s1);
    small[b].v[qd][jj] = make_float4(c0, c1, s0, s1);
  }
}

// cos, sin, -sin of a thread's 8 angles of half `hf` (pairs 16 qd + 8 hf ..),
// from the rows' base table `bt` and offset table `st` (both at [qd][0]).
__device__ __forceinline__ void rope8_tab(const float4 *bt, const float4 *st, int hf, f2 (&cs)[4],
                                          f2 (&sn)[4], f2 (&nsn)[4]) {
  const f2 m1 = dup2(-1.f);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float4 B = bt[4 * hf + e], S = st[4 * hf + e];
    const f2 cb = mk2(B.x, B.y), sb = mk2(B.z, B.w), co = mk2(S.x, S.y), so = mk2(S.z, S.w);
    cs[e] = fma2(cb, co, mul2(sb, mul2(so, m1)));  // cos(a + b) = ca cb - sa sb
    sn[e] = fma2(sb, co, mul2(cb, so));            // sin(a + b) = sa cb + ca sb
    nsn[e] = mul2(sn[e], m1);
  }
}

// Rotate this thread's 16 pairs of raw row `r` (times `scale`) at position p
// and store them, as fp16 (half) or bf16, into the same chunks of `tile`.
// `ru` is the kernel's table from load_rope_table.
__device__ __forceinline__ void feature_store(const uint4 (&r)[4], float scale, long long p, int qd,
                                              const unsigned long long *ru, unsigned char *tile,
                                              int row, bool half) {
  const f2 sc = dup2(scale);
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    f2 cs[4], sn[4], nsn[4], lo[4], hi[4];
    rope8(p, ru, hf, qd, cs, sn, nsn);
    rotate8(r[hf], r[2 + hf], sc, cs, sn, nsn, lo, hi);
    *tile_at(tile, row, 2 * qd + hf) = half ? pack4x2h(lo) : pack4x2(lo);
    *tile_at(tile, row, 8 + 2 * qd + hf) = half ? pack4x2h(hi) : pack4x2(hi);
  }
}

// q~ and k~ of one row at once (shared angles), both fp16, in place.  Returns
// this thread's part of the fp32 dot product q~ . k~ (before the rounding to
// fp16), for callers that need the diagonal of Q~ K~^T exactly.
__device__ __forceinline__ float feature_qk_store(const uint4 (&qr)[4], const uint4 (&kr)[4],
                                                 float rq, float rk, long long p, int qd,
                                                 const unsigned long long *ru, unsigned char *Qt,
                                                 unsigned char *Kt, int row) {
  f2 dot = 0ull;
  const f2 sq = dup2(rq), sk = dup2(rk);
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    f2 cs[4], sn[4], nsn[4], qlo[4], qhi[4], klo[4], khi[4];
    rope8(p, ru, hf, qd, cs, sn, nsn);
    rotate8(qr[hf], qr[2 + hf], sq, cs, sn, nsn, qlo, qhi);
    *tile_at(Qt, row, 2 * qd + hf) = pack4x2h(qlo);
    *tile_at(Qt, row, 8 + 2 * qd + hf) = pack4x2h(qhi);
    rotate8(kr[hf], kr[2 + hf], sk, cs, sn, nsn, klo, khi);
    *tile_at(Kt, row, 2 * qd + hf) = pack4x2h(klo);
    *tile_at(Kt, row, 8 + 2 * qd + hf) = pack4x2h(khi);
#pragma unroll
    for (int e = 0; e < 4; ++e) dot = fma2(qlo[e], klo[e], fma2(qhi[e], khi[e], dot));
  }
  return hsum2(dot);
}

// feature_qk_store with the angles from a base and an offset RopeTab row
// (rope8_tab) instead of the phase of each angle.
__device__ __forceinline__ float feature_qk_store_tab(const uint4 (&qr)[4], const uint4 (&kr)[4],
                                                     float rq, float rk, const float4 *bt,
                                                     const float4 *st, int qd, unsigned char *Qt,
                                                     unsigned char *Kt, int row) {
  f2 dot = 0ull;
  const f2 sq = dup2(rq), sk = dup2(rk);
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    f2 cs[4], sn[4], nsn[4], qlo[4], qhi[4], klo[4], khi[4];
    rope8_tab(bt, st, hf, cs, sn, nsn);
    rotate8(qr[hf], qr[2 + hf], sq, cs, sn, nsn, qlo, qhi);
    *tile_at(Qt, row, 2 * qd + hf) = pack4x2h(qlo);
    *tile_at(Qt, row, 8 + 2 * qd + hf) = pack4x2h(qhi);
    rotate8(kr[hf], kr[2 + hf], sk, cs, sn, nsn, klo, khi);
    *tile_at(Kt, row, 2 * qd + hf) = pack4x2h(klo);
    *tile_at(Kt, row, 8 + 2 * qd + hf) = pack4x2h(khi);
#pragma unroll
    for (int e = 0; e < 4; ++e) dot = fma2(qlo[e], klo[e], fma2(qhi[e], khi[e], dot));
  }
  return hsum2(dot);
}

__device__ __forceinline__ void sync_tc() {
  umma::fence_before();
  __syncthreads();
  umma::fence_after();
}

// TMA of one raw [rows, 128] bf16 tile (rows = chunk) of token rows
// [c0, c0 + rows) for (b, h): two boxes of 64 columns.
__device__ __forceinline__ void tma_tile(unsigned char *dst, const CUtensorMap *map, int b, int h,
                                         int c0, uint64_t *bar) {
  umma::tma_load_4d(dst, map, 0, h, c0, b, bar);
  umma::tma_load_4d(dst + HALF_TILE, map, 64, h, c0, b, bar);
}

// L2 prefetch of the same tile (no shared-memory destination, no barrier).
__device__ __forceinline__ void tma_prefetch_tile(const CUtensorMap *map, int b, int h, int c0) {
  umma::tma_prefetch_4d(map, 0, h, c0, b);
  umma::tma_prefetch_4d(map, 64, h, c0, b);
}

// TMA store of a [rows, 128] bf16 operand-layout tile to token rows
// [c0, c0 + rows) of (b, h): two boxes of 64 columns.  Rows past T are not
// written.
__device__ __forceinline__ void tma_store_tile(const CUtensorMap *map, const unsigned char *src,
                                               int b, int h, int c0) {
  umma::tma_store_4d(map, src, 0, h, c0, b);
  umma::tma_store_4d(map, src + HALF_TILE, 64, h, c0, b);
}

// Named barrier among `nthreads` threads (ids 1..15; id 0 is __syncthreads).
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Bounded wait that becomes a no-op once this thread has seen a timeout, so a
// failure never strands other warps at a barrier: the loop runs to its end
// with invalid data and the status word reports it.
__device__ __forceinline__ void wait_or_fail(uint64_t *bar, uint32_t parity, bool &failed) {
  if (!failed && !umma::mbar_wait(bar, parity)) failed = true;
  umma::fence_after();
}
// The same without the tcgen05 fence (which costs the waiting thread tens of
// cycles each time): for waits whose consumer is no tcgen05 operation (a TMA
// copy's data read by this thread, a copy issued into a freed buffer), or
// where one fence_after before a group of MMAs covers every wait before it.
__device__ __forceinline__ void wait_plain(uint64_t *bar, uint32_t parity, bool &failed) {
  if (!failed && !umma::mbar_wait(bar, parity)) failed = true;
}

// A 4-byte global -> shared copy that holds no register while it is in flight
// (cp.async); its data is there for this thread after cp_async_wait().
__device__ __forceinline__ void cp_async4(void *dst_smem, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(umma::smem_u32(dst_smem)),
               "l"(__cvta_generic_to_global(src))
               : "memory");
}
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// One elected arrive per warp on a worker-count barrier, after the warp's
// shared-memory writes (generic proxy) and TMEM stores are complete.
__device__ __forceinline__ void warp_arrive(uint64_t *bar, int lane) {
  umma::fence_async_smem();
  umma::fence_before();
  __syncwarp();
  if (lane == 0) umma::mbar_arrive(bar);
}

// ------------------------------------------------------------------ host side

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeFn>(p);
  }();
  return fn;
}

// 4-D map over a [B, T, H, 128] 16-bit tensor (bf16 unless `dt` says fp16)
// with a box of 64 columns x 1 head x `rows` tokens x 1 sequence, 128-byte
// swizzled (the operand tile layout).
cudaError_t make_map(CUtensorMap *map, const void *ptr, const MixerParams &P, int rows,
                     CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  EncodeFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  if (!ptr) return cudaErrorInvalidValue;  // a map over no tensor would read address 0
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)P.H, (cuuint64_t)P.T, (cuuint64_t)P.B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)P.H * D * 2,
                                 (cuuint64_t)P.T * P.H * D * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, dt, 4, const_cast<void *>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace
}  // namespace tc
}  // namespace hla
