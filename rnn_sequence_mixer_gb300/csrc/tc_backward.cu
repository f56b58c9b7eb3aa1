// tc_backward.cu — tensor-core (tcgen05) kernels of the prefill backward for
// bf16 inputs at d = 128.
//
// The loss is L = <dy, y> + <dstate_out, S_T> with y from Eq. 18 of
// arXiv 2601.22156 (Appendix A).  Per tile of c <= 128 tokens entering with
// state S (read from the forward's workspace when the caller passes it, else
// recomputed by the forward local-state pass and scan), D_ij = gamma^{i-j} for
// i >= j:
//
//   tc_bwd_dq_kernel (tiles in order, S carried in TMEM as in the forward)
//     O     = diag(gamma^{i+1}) Q~ S + (Q~ K~^T (.) D) V          (recompute;
//             given the forward's y and saved 1/RMS(o) instead:
//             n = y (1 + 2^(-g log2 e)), no O)
//     dgate = dy n sigma(g) (1 - sigma(g)),  n = O r,  r = 1/RMS(O)
//     dO    = r (dn - n mean(dn n)),  dn = dy sigma(g)              (to the workspace, bf16)
//     dQ~   = diag(gamma^{i+1}) dO S^T + ((dO V^T) (.) D) K~
//     dq    = Norm^T RoPE^T dQ~
//     S    <- gamma^c S + K~^T diag(gamma^{c-1-j}) V
//   tc_state_kernel<true> (tc_prefill.cu) then sums q~^T do per segment and
//   the fp32 scan (scan.cu) turns those sums into E, the gradient reaching the
//   state at each segment's last token from later tokens.
//   tc_bwd_dkdv_kernel (tiles in reverse, E carried in TMEM)
//     dV  = ((K~ Q~^T) (.) D^T) dO + diag(gamma^{c-1-i}) K~ E
//     dK~ = ((V dO^T) (.) D^T) Q~ + diag(gamma^{c-1-i}) V E^T
//     E  <- gamma^c E + Q~^T diag(gamma^{i+1}) dO
//     dk  = Norm^T RoPE^T dK~ / sqrt(d)
//
// Precision: K~ Q~^T runs on fp16 operands (its rounding would dominate dv
// on fast-decaying heads with bf16), the recomputed O uses the forward's fp16
// Q~ K~^T / Q~ S products, and every other product has bf16 operands with fp32
// accumulation.  Two diagonal entries are taken in fp32 on the CUDA cores
// instead: q~_i . k~_i (where it nearly cancels, o_i is small and dO_i ~ 1/|o_i|
// magnifies its error) and v_i . do_i (do_i is orthogonal to o_i, so this
// cancels wherever o_i is close to a multiple of v_i, e.g. at t = 0).  Decay
// weights that multiply a whole operand row are folded into that operand
// (K~dec, Vdec, dOw); gamma^{i+1} on the rows of dO S^T is applied to that
// product in TMEM before the intra-chunk term accumulates onto it.
//
// Threads: both kernels are warp-specialized like the forward output pass:
// 16 worker warps own the CUDA-core phases (thread (warp w, lane l) owns tile
// row i = 32 (w % 4) + l, its TMEM lane, and column quarter qd = w / 4; the
// feature map uses row 8 w + l / 4 and pair quarter l % 4) and one issuer
// thread issues the MMAs and TMA copies; they hand off through mbarriers.
#include <type_traits>

#include "tc_common.cuh"

namespace hla {
namespace tc {

namespace {

// 32 fp32 values of a row (16 pairs) as packed bf16 into 16 TMEM columns at
// taddr (an MMA A operand in tensor memory).  Element e (0..31, none when e < 0)
// is replaced by dval first.  Selects in registers: no dynamic indexing.
__device__ __forceinline__ void store_tmem_bf16(uint32_t taddr, const f2 (&x)[16], int e, float dval) {
  uint32_t w[16];
#pragma unroll
  for (int e2 = 0; e2 < 16; ++e2) {
    float lo, hi;
    split2(x[e2], lo, hi);
    lo = e == 2 * e2 ? dval : lo;
    hi = e == 2 * e2 + 1 ? dval : hi;
    w[e2] = pack2(lo, hi);
  }
  umma::tmem_st16u(taddr, w);
}

// Gradient with respect to a raw q or k row, through RoPE and RMSNorm, for this
// thread's 16 RoPE pairs of row i (elements 16 qd .. 16 qd + 15 and their
// partners 64 further on).  g~ = gscale * (the gradient of the rotated,
// normalized row) is read from TMEM at tmem_row (the lane's base address,
// column 0); raw holds the raw row's pairs (ld_pairs layout).
// With g = RoPE^T g~, x the raw row and r = 1 / RMS(x):
//   dL/dx = r g - r^3 x (g . x) / d.
// Writes it as bf16 into the same chunks of `out`.  The two row sums need the
// other three threads of the row (warps sub, sub + 4, sub + 8, sub + 12): red
// is a [2][4][ROWS] scratch and the call holds named barrier 5 + sub.
__device__ __forceinline__ void feature_grad_pairs(uint32_t tmem_row, const uint4 (&raw)[4],
                                                   float gscale, long long pos, int i, int qd,
                                                   int sub, float eps, const unsigned long long *ru,
                                                   float (*red)[4][ROWS], unsigned char *out) {
  float alo[16], ahi[16];
  {
    uint32_t ra[16], rb[16];
    umma::tmem_ld16_nowait(tmem_row + 16 * qd, ra);
    umma::tmem_ld16_nowait(tmem_row + 64 + 16 * qd, rb);
    umma::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      alo[e] = __uint_as_float(ra[e]) * gscale;
      ahi[e] = __uint_as_float(rb[e]) * gscale;
    }
  }
  f2 g0[8], g1[8];
  f2 sx = 0ull, sgx = 0ull;
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    f2 cs[4], sn[4], nsn[4], x0[4], x1[4];
    rope8(pos, ru, hf, qd, cs, sn, nsn);
    unpack4x2(raw[hf], x0);
    unpack4x2(raw[2 + hf], x1);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const f2 a = mk2(alo[8 * hf + 2 * e], alo[8 * hf + 2 * e + 1]);
      const f2 bq = mk2(ahi[8 * hf + 2 * e], ahi[8 * hf + 2 * e + 1]);
      // transpose of (x0, x1) -> (x0 c - x1 s, x0 s + x1 c)
      g0[4 * hf + e] = fma2(a, cs[e], mul2(bq, sn[e]));
      g1[4 * hf + e] = fma2(bq, cs[e], mul2(a, nsn[e]));
      sx = fma2(x0[e], x0[e], fma2(x1[e], x1[e], sx));
      sgx = fma2(g0[4 * hf + e], x0[e], fma2(g1[4 * hf + e], x1[e], sgx));
    }
  }
  red[0][qd][i] = hsum2(sx);
  red[1][qd][i] = hsum2(sgx);
  named_sync(5 + sub, 128);
  const float r = rsqrtf((red[0][0][i] + red[0][1][i] + red[0][2][i] + red[0][3][i]) / (float)D + eps);
  const float m = r * (red[1][0][i] + red[1][1][i] + red[1][2][i] + red[1][3][i]) / (float)D;
  const f2 r2 = dup2(r), cx = dup2(-r * r * m);  // dL/dx = r g - r^2 m x
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    f2 x0[4], x1[4], lo[4], hi[4];
    unpack4x2(raw[hf], x0);
    unpack4x2(raw[2 + hf], x1);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      lo[e] = fma2(x0[e], cx, mul2(g0[4 * hf + e], r2));
      hi[e] = fma2(x1[e], cx, mul2(g1[4 * hf + e], r2));
    }
    *tile_at(out, i, 2 * qd + hf) = pack4x2(lo);
    *tile_at(out, i, 8 + 2 * qd + hf) = pack4x2(hi);
  }
}

// The same gradient from the saved features instead of the raw row.  With
// x^ = Norm(x) rotated (x^ = xscale * xt, xt the saved fp16 row in ld_pairs
// layout), r = 1 / RMS(x) saved by the forward and g~ = gscale * (the TMEM
// row): RoPE is orthogonal, so g . Norm(x) = g~ . x^ and
//   dL/dx = r RoPE^T (g~ - x^ (g~ . x^) / d),
// one row sum instead of two and no raw row (gscale rides on r: the bracket
// is linear in g~).  red is [4][ROWS]; the call holds named barrier 5 + sub.
__device__ __forceinline__ void feature_grad_saved(uint32_t tmem_row, const uint4 (&xt)[4],
                                                   float gscale, float xscale, float r,
                                                   long long pos, int i, int qd, int sub,
                                                   const unsigned long long *ru,
                                                   float (*red)[ROWS], unsigned char *out) {
  f2 a[8], bq[8];
  {
    uint32_t ra[16], rb[16];
    umma::tmem_ld16_nowait(tmem_row + 16 * qd, ra);
    umma::tmem_ld16_nowait(tmem_row + 64 + 16 * qd, rb);
    umma::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      a[e] = mk2(__uint_as_float(ra[2 * e]), __uint_as_float(ra[2 * e + 1]));
      bq[e] = mk2(__uint_as_float(rb[2 * e]), __uint_as_float(rb[2 * e + 1]));
    }
  }
  f2 sgx = 0ull;
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {  // the fp16 row stays packed until it is used
    f2 x0[4], x1[4];
    unpack4x2h(xt[hf], x0);
    unpack4x2h(xt[2 + hf], x1);
#pragma unroll
    for (int e = 0; e < 4; ++e) sgx = fma2(a[4 * hf + e], x0[e], fma2(bq[4 * hf + e], x1[e], sgx));
  }
  red[qd][i] = hsum2(sgx);
  named_sync(5 + sub, 128);
  // g~ - x^ (g~ . x^) / d = gscale (a + cx * xt), a the TMEM row
  const f2 cx = dup2(-xscale * xscale * (red[0][i] + red[1][i] + red[2][i] + red[3][i]) / (float)D);
  const f2 r2 = dup2(r * gscale);
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    f2 cs[4], sn[4], nsn[4], lo[4], hi[4], x0[4], x1[4];
    rope8(pos, ru, hf, qd, cs, sn, nsn);
    unpack4x2h(xt[hf], x0);
    unpack4x2h(xt[2 + hf], x1);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const f2 u0 = fma2(x0[e], cx, a[4 * hf + e]);
      const f2 u1 = fma2(x1[e], cx, bq[4 * hf + e]);
      // transpose of (x0, x1) -> (x0 c - x1 s, x0 s + x1 c), then times r
      lo[e] = mul2(fma2(u0, cs[e], mul2(u1, sn[e])), r2);
      hi[e] = mul2(fma2(u1, cs[e], mul2(u0, nsn[e])), r2);
    }
    *tile_at(out, i, 2 * qd + hf) = pack4x2(lo);
    *tile_at(out, i, 8 + 2 * qd + hf) = pack4x2(hi);
  }
}

// ------------------------------------------------------------------ dq pass

struct DqShared {
  unsigned long long ru[kMaxPairs];  // RoPE phase increments (load_rope_table)
  float red_do[2][4][ROWS];  // [W4] quarter parts of sum o^2 and sum dn.o of each row
  float red_dq[2][4][ROWS];  // [W6] quarter parts of sum q^2 and sum g.q of each row
  float vd_part[4][ROWS];    // [W4] -> [W5] quarter parts of the fp32 v_i . do_i
  float qk_diag[2][ROWS];    // [W1] -> [W3] fp32 q~_i . k~_i of tile n (n & 1)
  float r_saved[2][4][ROWS]; // saved features: 1 / RMS(q) of row i of tile n (n & 1), for
                             // [W6] of thread (qd, i)
  float r_o[2][4][ROWS];     // given y: the saved 1 / RMS(o) of row i of tile n, for [W4]
  float pw[ROWS + 1];
  alignas(16) float dm[4][DM_STRIDE];  // causal-mask decay table (fill_mask_table)
  float smax[NWORK];
  uint64_t bar_q;       // TMA: raw q of tile n into Q
  uint64_t bar_k[2];    // TMA: raw k into K buffer 0 / 1
  uint64_t bar_v;       // TMA: v into V
  uint64_t bar_g;       // TMA: gate of tile n into Q
  uint64_t bar_qr;      // TMA: raw q of tile n into its (freed) K buffer, for [W6]
  uint64_t bar_dy;      // TMA: dy of tile n into PM (once the dgate store of tile n - 1 has read it)
  uint64_t bar_y;       // given y: TMA of y of tile n into SB
  uint64_t bar_p;       // MMA1 done (P)
  uint64_t bar_o;       // MMA2 done (O = Q~ Sb)
  uint64_t bar_m3;      // MMA3 done (O complete)
  uint64_t bar_m56;     // MMA5 + MMA6 done (dP, I)
  uint64_t bar_m74;     // MMA7 + MMA4 done (dQ~ complete, S carried)
  uint64_t bar_feat, bar_sb, bar_pm, bar_do, bar_w5, bar_w6;  // workers, one arrive per warp
  uint32_t tmem_base;
  uint32_t failed;
};

// sigmoid of two lanes: 1 / (1 + e^-z) = 0.5 + 0.5 tanh(z / 2)
__device__ __forceinline__ f2 sigmoid2(f2 z) {
  const f2 half = dup2(0.5f);
  float a, b;
  split2(mul2(z, half), a, b);
  return fma2(mk2(tanh_fast(a), tanh_fast(b)), half, half);
}

// dq pass, warp-specialized: per tile n the forward is recomputed (O), the
// output norm and gate are differentiated (dgate, dO) and dQ~ is formed, while
// the state S is carried through TMEM as in the forward output pass.
//   MMA1  P  = Q~ K~^T               (fp16)      into tP
//   MMA2  O  = Q~ Sb                 (fp16)      into tA[n & 1]
//   MMA3  O += Pm V                  (bf16)
//   MMA5  dP = dO V^T                (bf16)      into tP
//   MMA6  I  = dO S^T                (bf16)      into tA[n & 1] (O is dead)
//   MMA7  dQ~ = gamma^{i+1} I + dPm K~           (I scaled in TMEM first)
//   MMA4  S  += K~^T Vdec,  Vdec_j = gamma^{c-1-j} v_j  (the decay rides on V,
//         so K~ serves MMA7 and MMA4 unchanged)
// Worker warps (0..15) run, per loop step n:
//   [W1] q~, k~ of tile n (fp16, in place)       [W2] Sb = fp16(S 2^-e), S <- gamma^c S
//   [W3] Pm (into the P columns of TMEM), O <- gamma^{i+1} 2^e O, K~ -> bf16,
//        Sb -> bf16 S
//   [W4] dgate -> PM (over dy), dO -> Q (over the gate), fp32 v_i . do_i
//   [W6] dq of tile n - 1 (RoPE^T, RMSNorm backward) in its K buffer, over its raw q
//   [W5] dPm (fp32 v_i . do_i on the diagonal) into the dP columns of TMEM,
//        I <- gamma^{i+1} I, V -> Vdec
// so the dq epilogue of tile n - 1 runs while MMA5 / MMA6 of tile n are in
// flight.  The issuer warp (16) waits for each hand-off, issues the MMAs and
// moves every tile by TMA: q, k (double-buffered), v, the gate (into Q once
// MMA2 has read it), dy (into PM once the dgate store of the tile before has
// read it: a tile ahead), raw q again for [W6] (into the K buffer that MMA7 /
// MMA4 freed), and the stores of dgate, dO and dq.  MMA3 and MMA7 take their A
// operands (Pm, dPm) from tensor memory.  No operand is read by plain loads:
// 16-byte loads of dy from 32 rows per warp instruction crowded the load
// pipeline and stalled every later shared-memory access of the warps (~20 % of
// a tile).
// kSaved: tmq / tmk map the forward's saved fp16 q~, k~.  [W1] is skipped
// (MMA1 waits for the copies instead), the q~ . k~ diagonal and 1/RMS(q) come
// from the saved scalars, and [W6] works on q~ (feature_grad_saved).
// kY (with kSaved): tmyi maps the forward's y, and o is not recomputed: no
// MMA1, MMA2, MMA3, no [W3].  Q starts a tile with the gate and SB with y; the
// step runs [W1] (the 1/RMS(q), 1/RMS(o) slots; k~ -> bf16), [W4] from y
// (n = y (1 + 2^(-gate log2 e)), the reciprocal of the forward's sigmoid
// form, and the saved 1/RMS(o)), then [W2] (S as bf16 into SB, over y, and
// S <- gamma^c S), [W6] of tile n - 1, [W5].  MMA5 follows [W4] and MMA6
// follows [W2]; the next gate and y land once MMA6 has read SB.
template <bool kSaved, bool kY = false>
__global__ void __launch_bounds__(NTO, 1)
    tc_bwd_dq_kernel(const __grid_constant__ MixerParams P, const __grid_constant__ CUtensorMap tmq,
                     const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ CUtensorMap tmg, const __grid_constant__ CUtensorMap tmo,
                     const __grid_constant__ CUtensorMap tmdg, const __grid_constant__ CUtensorMap tmdq,
                     const __grid_constant__ CUtensorMap tmdy, const __grid_constant__ CUtensorMap tmyi) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  // Q:  raw q -> q~ (fp16) -> gate -> dO (bf16)                 -> next raw q
  // K j: raw k -> k~ (fp16) -> k~ (bf16) -> raw q -> dq (bf16)  -> k two tiles on
  // V:  v -> Vdec;  SB: Sb (fp16, scaled) -> S (bf16);  PM: dy -> dgate
  unsigned char *Qs = base, *Vs = base + 3 * TILE, *SB = base + 4 * TILE, *PM = base + 5 * TILE;
  DqShared &sh = *reinterpret_cast<DqShared *>(base + 6 * TILE);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int t0 = g * P.seg_len, t1 = min(P.T, t0 + P.seg_len);
  const int CV = P.chunk;
  const int ntile = ceil_div(t1 - t0, CV);
  const float l2g = log2f(P.gamma[h]);
  const uint32_t tile_bytes = (uint32_t)CV * D * 2;

  if (tid == 0) {
    uint64_t *bars[] = {&sh.bar_q, &sh.bar_k[0], &sh.bar_k[1], &sh.bar_v, &sh.bar_g, &sh.bar_qr, &sh.bar_dy,
                        &sh.bar_y, &sh.bar_p, &sh.bar_o, &sh.bar_m3, &sh.bar_m56, &sh.bar_m74};
    for (uint64_t *bar : bars) umma::mbar_init(bar, 1);
    uint64_t *wbars[] = {&sh.bar_feat, &sh.bar_sb, &sh.bar_pm, &sh.bar_do, &sh.bar_w5, &sh.bar_w6};
    for (uint64_t *bar : wbars) umma::mbar_init(bar, NWORK);
    umma::mbar_fence_init();
    sh.failed = 0;
  }
  if (tid <= ROWS) sh.pw[tid] = exp2f((float)tid * l2g);
  fill_mask_table(sh.dm, l2g, tid, NTO);
  load_rope_table(sh.ru, P, tid);
  if (warp == 0) umma::tmem_alloc(&sh.tmem_base, 512);
  if (CV < ROWS)  // rows [CV, 128) of V (and, with saved features, of Q and both
                  // K buffers, which [W1] would have zeroed) are never written by TMA
    for (int e = tid; e < (kSaved ? 4 : 1) * (ROWS - CV) * 16; e += NTO) {
      const int t = e / ((ROWS - CV) * 16), r = e % ((ROWS - CV) * 16);
      *tile_at(t == 0 ? Vs : base + (t - 1) * TILE, CV + r / 16, r % 16) = make_uint4(0, 0, 0, 0);
    }
  sync_tc();
  const uint32_t tm = sh.tmem_base;
  const uint32_t tP = tm, tS = tm + 384;
  bool failed = false;

  if (warp >= NWORK) {
    // ---------------------------------------------------------------- issuer warpgroup
    if (warp == NWORK && lane == 0) {
      const uint32_t id_qk = umma::idesc_bf16(128, 128, false, false, true);  // fp16 Q~ K~^T
      const uint32_t id_qs = umma::idesc_bf16(128, 128, false, true, true);   // fp16 Q~ Sb
      const uint32_t id_kmn = umma::idesc_bf16(128, 128, false, true);        // Pm V, dPm K~
      const uint32_t id_kk = umma::idesc_bf16(128, 128, false, false);        // dO V^T, dO S^T
      const uint32_t id_mnmn = umma::idesc_bf16(128, 128, true, true);        // K~^T Vdec
      const uint32_t aq = umma::smem_u32(Qs), av = umma::smem_u32(Vs), asb = umma::smem_u32(SB);
      if (kY) {  // given y: Q starts with the gate and SB with y
        umma::mbar_expect_tx(&sh.bar_g, tile_bytes);
        tma_tile(Qs, &tmg, b, h, t0, &sh.bar_g);
        umma::mbar_expect_tx(&sh.bar_y, tile_bytes);
        tma_tile(SB, &tmyi, b, h, t0, &sh.bar_y);
      } else {
        umma::mbar_expect_tx(&sh.bar_q, tile_bytes);
        tma_tile(Qs, &tmq, b, h, t0, &sh.bar_q);
      }
      for (int n = 0; n < 2 && n < ntile; ++n) {
        umma::mbar_expect_tx(&sh.bar_k[n], tile_bytes);
        tma_tile(base + (1 + n) * TILE, &tmk, b, h, t0 + n * CV, &sh.bar_k[n]);
      }
      umma::mbar_expect_tx(&sh.bar_v, tile_bytes);
      tma_tile(Vs, &tmv, b, h, t0, &sh.bar_v);
      umma::mbar_expect_tx(&sh.bar_dy, tile_bytes);
      tma_tile(PM, &tmdy, b, h, t0, &sh.bar_dy);
      tma_prefetch_tile(&tmg, b, h, t0);
      // tile n with its k in buffer BUF = n & 1, a compile-time constant (tiles
      // go in pairs), so that every MMA descriptor is loop-invariant
      auto tile_step = [&](int n, auto nbuf) {
        constexpr int buf = decltype(nbuf)::value;
        const uint32_t ph = n & 1;
        const int c0 = t0 + n * CV;
        unsigned char *Kt = base + (1 + buf) * TILE;
        const uint32_t ak = umma::smem_u32(Kt);
        const uint32_t ta = tm + 128 + 128 * buf;
        if (kY && n + 1 < ntile) {  // next tile's operands into L2 ahead of their copies
          tma_prefetch_tile(&tmg, b, h, c0 + CV);
          tma_prefetch_tile(&tmyi, b, h, c0 + CV);
          tma_prefetch_tile(&tmdy, b, h, c0 + CV);
          tma_prefetch_tile(&tmv, b, h, c0 + CV);
          tma_prefetch_tile(&tmk, b, h, c0 + CV);
          tma_prefetch_tile(&tmq, b, h, c0);
        }
        if (!kY) {  // o recomputed: MMA1, MMA2, MMA3 (given y, none of them)
        // MMA1 once q~, k~ are written (copied, when saved); MMA2 once Sb is
        if (kSaved) {
          wait_plain(&sh.bar_q, ph, failed);
          wait_plain(&sh.bar_k[buf], (n >> 1) & 1, failed);
        } else {
          wait_plain(&sh.bar_feat, ph, failed);
        }
        if (!failed) {
          umma::fence_after();  // covers the waits before this group of MMAs
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma::mma_ss(tP, umma::desc_kmajor(aq, kk, ROWS), umma::desc_kmajor(ak, kk, ROWS), id_qk, kk > 0);
          umma::commit(&sh.bar_p);
        }
        wait_plain(&sh.bar_sb, ph, failed);
        if (!failed) {
          umma::fence_after();  // covers the waits before this group of MMAs
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma::mma_ss(ta, umma::desc_kmajor(aq, kk, ROWS), umma::desc_mnmajor(asb, kk, ROWS), id_qs, kk > 0);
          umma::commit(&sh.bar_o);
        }
        // MMA2 done: Q takes this tile's gate
        wait_plain(&sh.bar_o, ph, failed);
        if (!failed) {
          umma::mbar_expect_tx(&sh.bar_g, tile_bytes);
          tma_tile(Qs, &tmg, b, h, c0, &sh.bar_g);
          if (n + 1 < ntile) {  // next tile's operands into L2 ahead of their copies
            tma_prefetch_tile(&tmq, b, h, c0 + CV);
            tma_prefetch_tile(&tmk, b, h, c0 + CV);
            tma_prefetch_tile(&tmv, b, h, c0 + CV);
            tma_prefetch_tile(&tmg, b, h, c0 + CV);
            tma_prefetch_tile(&tmdy, b, h, c0 + CV);
          }
        }
        // MMA3 once Pm, the scaled O and V are in place
        wait_plain(&sh.bar_pm, ph, failed);
        wait_plain(&sh.bar_v, ph, failed);
        if (!failed) {
          umma::fence_after();  // covers the waits before this group of MMAs
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // A = Pm from the P columns of TMEM
            umma::mma_ts(ta, tP + 32 * (kk >> 1) + 8 * (kk & 1), umma::desc_mnmajor(av, kk, ROWS),
                         id_kmn, 1u);
          umma::commit(&sh.bar_m3);
        }
        }  // !kY
        // dgate (PM) and dO (Q) out; MMA5, MMA6 from dO (given y, MMA5 also waits
        // for v, and MMA6 for S, which [W2] turns into bf16 after [W4])
        wait_plain(&sh.bar_do, ph, failed);
        if (kY) wait_plain(&sh.bar_v, ph, failed);
        if (!failed) {
          tma_store_tile(&tmdg, PM, b, h, c0);
          tma_store_tile(&tmo, Qs, b, h, c0);
          umma::bulk_commit();
          umma::fence_after();  // covers the waits before this group of MMAs
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma::mma_ss(tP, umma::desc_kmajor(aq, kk, ROWS), umma::desc_kmajor(av, kk, ROWS), id_kk, kk > 0);
        }
        if (kY) wait_plain(&sh.bar_sb, ph, failed);
        if (!failed) {
          if (kY) umma::fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma::mma_ss(ta, umma::desc_kmajor(aq, kk, ROWS), umma::desc_kmajor(asb, kk, ROWS), id_kk, kk > 0);
          umma::commit(&sh.bar_m56);
          umma::bulk_wait_read();
          if (n + 1 < ntile) {  // the dgate store has read PM: it takes dy of the next tile
            umma::mbar_expect_tx(&sh.bar_dy, tile_bytes);
            tma_tile(PM, &tmdy, b, h, c0 + CV, &sh.bar_dy);
          }
        }
        // MMA5 / MMA6 done and dO stored: Q takes the next q (given y: the next
        // gate, and SB, which MMA6 has read, the next y)
        wait_plain(&sh.bar_m56, ph, failed);
        if (!failed && n + 1 < ntile) {
          if (kY) {
            umma::mbar_expect_tx(&sh.bar_g, tile_bytes);
            tma_tile(Qs, &tmg, b, h, c0 + CV, &sh.bar_g);
            umma::mbar_expect_tx(&sh.bar_y, tile_bytes);
            tma_tile(SB, &tmyi, b, h, c0 + CV, &sh.bar_y);
          } else {
            umma::mbar_expect_tx(&sh.bar_q, tile_bytes);
            tma_tile(Qs, &tmq, b, h, c0 + CV, &sh.bar_q);
          }
        }
        // dq of tile n - 1 is in its K buffer: store it, then that buffer takes k of tile n + 1
        if (n >= 1) {
          wait_plain(&sh.bar_w6, (n - 1) & 1, failed);
          unsigned char *Kp = base + (2 - buf) * TILE;
          if (!failed) {
            tma_store_tile(&tmdq, Kp, b, h, c0 - CV);
            umma::bulk_commit();
            if (n + 1 < ntile) {
              umma::bulk_wait_read();
              umma::mbar_expect_tx(&sh.bar_k[buf ^ 1], tile_bytes);
              tma_tile(Kp, &tmk, b, h, c0 + CV, &sh.bar_k[buf ^ 1]);
            }
          }
        }
        // MMA7 and MMA4 once dPm, the scaled I and Vdec are in place
        wait_plain(&sh.bar_w5, ph, failed);
        if (!failed) {
          umma::fence_after();  // covers the waits before this group of MMAs
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // A = dPm from the dP columns of TMEM
            umma::mma_ts(ta, tP + 32 * (kk >> 1) + 8 * (kk & 1), umma::desc_mnmajor(ak, kk, ROWS),
                         id_kmn, 1u);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma::mma_ss(tS, umma::desc_mnmajor(ak, kk, ROWS), umma::desc_mnmajor(av, kk, ROWS), id_mnmn, 1u);
          umma::commit(&sh.bar_m74);
        }
        // both done: V takes the next v, this K buffer takes raw q of tile n for [W6]
        wait_plain(&sh.bar_m74, ph, failed);
        if (!failed) {
          if (n + 1 < ntile) {
            umma::mbar_expect_tx(&sh.bar_v, tile_bytes);
            tma_tile(Vs, &tmv, b, h, c0 + CV, &sh.bar_v);
          }
          umma::mbar_expect_tx(&sh.bar_qr, tile_bytes);
          tma_tile(Kt, &tmq, b, h, c0, &sh.bar_qr);

        }
            };
      for (int n = 0; n < ntile; n += 2) {
        tile_step(n, std::integral_constant<int, 0>{});
        if (n + 1 < ntile) tile_step(n + 1, std::integral_constant<int, 1>{});
      }
      // dq of the last tile
      wait_plain(&sh.bar_w6, (ntile - 1) & 1, failed);
      if (!failed) {
        tma_store_tile(&tmdq, base + (1 + ((ntile - 1) & 1)) * TILE, b, h, t0 + (ntile - 1) * CV);
        umma::bulk_commit();
      }
      umma::bulk_wait_all();
    }
  } else {
    // ---------------------------------------------------------------- worker warps
    const int sub = warp & 3, qd = warp >> 2, i = 32 * sub + lane;  // TMEM phases
    const int fr = 8 * warp + (lane >> 2), fu = lane & 3;           // feature map: row, quarter
    const uint32_t lane_base = (uint32_t)(32 * sub) << 16;
    const uint32_t col = 32 * qd;
    const uint32_t myS = tS + lane_base + col, myP = tP + lane_base + col;
    {  // entering state of the segment -> TMEM (fp32)
      const float *sin_ = P.seg + (((size_t)b * P.H + h) * P.nseg + g) * (size_t)D * D;
      const float4 *s4 = reinterpret_cast<const float4 *>(sin_ + (size_t)i * D + col);
      float v[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 x = s4[u];
        v[4 * u] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
      }
      umma::tmem_st32(myS, v);
      umma::tmem_wait_st();
    }
    int prev_c0 = 0;
    for (int n = 0; n <= ntile; ++n) {
      const bool have = n < ntile, drain = n >= 1;
      const int buf = n & 1;
      const uint32_t ph = n & 1;
      const int c0 = t0 + n * CV, c = have ? min(CV, t1 - c0) : 0;
      const bool valid = i < c;
      const uint32_t ta = tm + 128 + 128 * buf + lane_base;        // tA of tile n (this lane)
      const uint32_t tap = tm + 128 + 128 * (buf ^ 1) + lane_base; // tA of tile n - 1
      unsigned char *Kt = base + (1 + buf) * TILE, *Kp = base + (2 - buf) * TILE;
      if (have) {
        // [W1] raw q, k of tile n: row fr, pairs [16 fu, 16 fu + 16); norms by shuffles
        if (!kY) wait_plain(&sh.bar_q, ph, failed);
        wait_plain(&sh.bar_k[buf], (n >> 1) & 1, failed);
        if (!kSaved) {
          uint4 qr[4], kr[4];
          ld_pairs(Qs, fr, fu, qr);
          ld_pairs(Kt, fr, fu, kr);
          if (!(fr < c))  // rows past the tile hold stale bytes: use zeros
            qr[0] = qr[1] = qr[2] = qr[3] = kr[0] = kr[1] = kr[2] = kr[3] = make_uint4(0, 0, 0, 0);
          float sq, sk, qk;
          norms_and_dot(qr, kr, sq, sk, qk);
          sq += __shfl_xor_sync(0xffffffffu, sq, 1);
          sk += __shfl_xor_sync(0xffffffffu, sk, 1);
          qk += __shfl_xor_sync(0xffffffffu, qk, 1);
          sq += __shfl_xor_sync(0xffffffffu, sq, 2);
          sk += __shfl_xor_sync(0xffffffffu, sk, 2);
          qk += __shfl_xor_sync(0xffffffffu, qk, 2);
          const float rq = rsqrtf(sq / (float)D + P.eps);
          const float rk = rsqrtf(sk / (float)D + P.eps) * P.kscale;
          if (fu == 0) sh.qk_diag[buf][fr] = qk * rq * rk;  // q~_i . k~_i in fp32
          feature_qk_store(qr, kr, rq, rk, P.pos_offset + c0 + fr, fu, sh.ru, Qs, Kt, fr);
          warp_arrive(&sh.bar_feat, lane);
        } else if (!kY) {  // saved scalars of row i into slots only this thread reads: 1 / RMS(q_i)
                  // for [W6] one step later and, on the diagonal warps, q~_i . k~_i for [W3]
          if (valid) {
            cp_async4(&sh.r_saved[buf][qd][i], saved_scalar(P, kSavedRq, b, h, c0 + i));
            if (qd == sub) cp_async4(&sh.qk_diag[buf][i], saved_scalar(P, kSavedDiag, b, h, c0 + i));
          } else {
            sh.r_saved[buf][qd][i] = 0.f;
            if (qd == sub) sh.qk_diag[buf][i] = 0.f;
          }
        } else {  // given y: 1 / RMS(q_i) for [W6] and 1 / RMS(o_i) for [W4]; k~ -> bf16
                  // for MMA7 / MMA4 right away (no MMA reads the fp16 k~ here)
          if (valid) {
            cp_async4(&sh.r_saved[buf][qd][i], saved_scalar(P, kSavedRq, b, h, c0 + i));
            cp_async4(&sh.r_o[buf][qd][i], saved_scalar(P, kSavedRo, b, h, c0 + i));
          } else {
            sh.r_saved[buf][qd][i] = 0.f;
            sh.r_o[buf][qd][i] = 0.f;
          }
          uint4 kraw[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) kraw[u] = *tile_at(Kt, i, 4 * qd + u);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            f2 f[4];
            unpack4x2h(kraw[u], f);
            *tile_at(Kt, i, 4 * qd + u) = pack4x2(f);
          }
        }

        if (!kY) {
        // [W2] after MMA7 / MMA4 of tile n - 1: Sb = fp16(S 2^-e) per column quarter, S <- gamma^c S
        if (n >= 1) wait_or_fail(&sh.bar_m74, (n - 1) & 1, failed);
        float s_inv;
        {
          float sv[32];
          umma::tmem_ld2x16(myS, sv);
          float m = 0.f;
#pragma unroll
          for (int e = 0; e < 32; ++e) m = fmaxf(m, fabsf(sv[e]));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (lane == 0) sh.smax[warp] = m;
          named_sync(1 + qd, 128);
          m = fmaxf(fmaxf(sh.smax[4 * qd], sh.smax[4 * qd + 1]),
                    fmaxf(sh.smax[4 * qd + 2], sh.smax[4 * qd + 3]));
          int e = 0;
          if (m > 0.f) frexpf(m, &e);
          const f2 s_fwd = dup2(ldexpf(1.f, -e));
          s_inv = ldexpf(1.f, e);
          f2 x[16];
          pairs_of(sv, x);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            f2 t[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) t[e2] = mul2(x[4 * u + e2], s_fwd);
            *tile_at(SB, i, 4 * qd + u) = pack4x2h(t);
          }
          const f2 carry = dup2(sh.pw[c]);
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) x[e2] = mul2(x[e2], carry);
          floats_of(x, sv);
          umma::tmem_st32(myS, sv);
          umma::tmem_wait_st();
        }
        warp_arrive(&sh.bar_sb, lane);

        // [W3] after MMA1: Pm (with the fp32 diagonal), k~ -> bf16; after MMA2:
        // O <- gamma^{i+1} 2^e O, Sb -> bf16 S
        // k~ fp16 -> bf16 for MMA7 / MMA4: with saved features k~ came by TMA,
        // so its row is converted while MMA1 (which reads it) may still run, and
        // written once MMA1 is done
        uint4 kbf[4];
        if (kSaved) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            f2 f[4];
            unpack4x2h(*tile_at(Kt, i, 4 * qd + u), f);
            kbf[u] = pack4x2(f);
          }
        }
        wait_or_fail(&sh.bar_p, ph, failed);
        {
          float pv[32];
          umma::tmem_ld2x16(myP, pv);
          f2 x[16];
          pairs_of(pv, x);
          mask_lower_table(x, sh.dm, i, (int)col);
          if (kSaved) {
#pragma unroll
            for (int u = 0; u < 4; ++u) *tile_at(Kt, i, 4 * qd + u) = kbf[u];
          } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) {  // k~ written by other threads in [W1]: after MMA1
              uint4 *p = tile_at(Kt, i, 4 * qd + u);
              f2 f[4];
              unpack4x2h(*p, f);
              *p = pack4x2(f);
            }
          }
          // Pm as packed bf16 over the first 16 of the 32 P columns this thread has
          // read: MMA3 takes its A operand from there (K-step kk at column
          // 32 (kk / 2) + 8 (kk % 2)), which leaves PM free for dy.  The diagonal
          // entry (element i - 32 qd on the warps with qd == sub) comes from fp32
          // features (written in [W1], met at [W2]'s barrier).
          if (kSaved) cp_async_wait();
          store_tmem_bf16(myP, x, qd == sub ? i - (int)col : -1, qd == sub ? sh.qk_diag[buf][i] : 0.f);
          // Sb -> S (bf16, unscaled) for MMA6: read and converted now (MMA2 only
          // reads Sb), written once MMA2 is done
          const f2 si = dup2(s_inv);
          uint4 snew[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            f2 f[4];
            unpack4x2h(*tile_at(SB, i, 4 * qd + u), f);
#pragma unroll
            for (int e = 0; e < 4; ++e) f[e] = mul2(f[e], si);
            snew[u] = pack4x2(f);
          }
          wait_or_fail(&sh.bar_o, ph, failed);  // MMA2 done: SB is free to rewrite
#pragma unroll
          for (int u = 0; u < 4; ++u) *tile_at(SB, i, 4 * qd + u) = snew[u];
          float ov[32];
          umma::tmem_ld2x16(ta + col, ov);
          const f2 f = dup2(sh.pw[i + 1] * s_inv);
          f2 y2[16];
          pairs_of(ov, y2);
#pragma unroll
          for (int e = 0; e < 16; ++e) y2[e] = mul2(y2[e], f);
          floats_of(y2, ov);
          umma::tmem_st32(ta + col, ov);
          umma::tmem_wait_st();
        }
        warp_arrive(&sh.bar_pm, lane);
        }  // !kY
      }

      if (have && !kY) {
        // [W4] after MMA3: output norm and gate backward.  n = o r, z = sigmoid(gate),
        // dn = dy z, dgate = dn n (1 - z), dO = r (dn - n mean(dn n)); rows past the tile get 0
        wait_plain(&sh.bar_g, ph, failed);
        wait_plain(&sh.bar_v, ph, failed);
        wait_plain(&sh.bar_dy, ph, failed);
        {
          // every gate and dy chunk of the row first, while MMA3 may still run
          // (the TMEM accesses below are ordered against shared-memory accesses,
          // so loads after them would wait)
          uint4 graw[4], draw[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            graw[u] = *tile_at(Qs, i, 4 * qd + u);
            draw[u] = *tile_at(PM, i, 4 * qd + u);
          }
          wait_or_fail(&sh.bar_m3, ph, failed);
          float o[32];
          umma::tmem_ld2x16(ta + col, o);
          f2 ox[16];
          pairs_of(o, ox);
          // z = sigmoid(gate) once per element, kept in fp32 in this thread's P
          // columns of TMEM until the second loop (MMA3 has read Pm from them
          // and MMA5 writes dP there only after this phase)
          f2 so2 = 0ull, sdo = 0ull;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            float zs[16];
#pragma unroll
            for (int uu = 0; uu < 2; ++uu) {
              const int u = 2 * hf + uu;
              f2 gz[4], dv[4];
              unpack4x2(graw[u], gz);
              unpack4x2(draw[u], dv);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const f2 z = sigmoid2(gz[e]);
                const f2 dn = mul2(dv[e], z);
                so2 = fma2(ox[4 * u + e], ox[4 * u + e], so2);
                sdo = fma2(dn, ox[4 * u + e], sdo);
                split2(z, zs[8 * uu + 2 * e], zs[8 * uu + 2 * e + 1]);
              }
            }
            umma::tmem_st16(myP + 16 * hf, zs);
          }
          umma::tmem_wait_st();
          sh.red_do[0][qd][i] = hsum2(so2);
          sh.red_do[1][qd][i] = hsum2(sdo);
          named_sync(5 + sub, 128);
          const float ro = rsqrtf((sh.red_do[0][0][i] + sh.red_do[0][1][i] + sh.red_do[0][2][i] +
                                   sh.red_do[0][3][i]) / (float)D + P.eps);
          const float mean = ro * (sh.red_do[1][0][i] + sh.red_do[1][1][i] + sh.red_do[1][2][i] +
                                   sh.red_do[1][3][i]) / (float)D;
          const f2 ro2 = dup2(ro), nmean = dup2(-mean), one = dup2(1.f), keep = dup2(valid ? 1.f : 0.f);
          f2 vd = 0ull;
          uint32_t zr[2][16];  // z back from TMEM under one wait
          umma::tmem_ld16_nowait(myP, zr[0]);
          umma::tmem_ld16_nowait(myP + 16, zr[1]);
          umma::tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float zs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) zs[e] = __uint_as_float(zr[u >> 1][8 * (u & 1) + e]);
            uint4 *gp = tile_at(Qs, i, 4 * qd + u);
            f2 dv[4], vv[4], dg[4], dd[4];
            unpack4x2(*tile_at(PM, i, 4 * qd + u), dv);
            unpack4x2(*tile_at(Vs, i, 4 * qd + u), vv);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const f2 z = mk2(zs[2 * e], zs[2 * e + 1]);
              const f2 dn = mul2(dv[e], z);
              const f2 nv = mul2(ox[4 * u + e], ro2);
              dg[e] = mul2(mul2(dn, nv), fma2(z, dup2(-1.f), one));
              dd[e] = mul2(mul2(ro2, fma2(nv, nmean, dn)), keep);
              vd = fma2(vv[e], dd[e], vd);
            }
            *tile_at(PM, i, 4 * qd + u) = pack4x2(dg);
            *gp = pack4x2(dd);
          }
          sh.vd_part[qd][i] = hsum2(vd);
        }
        warp_arrive(&sh.bar_do, lane);
      }

      if (have && kY) {
        // [W4] given y: the output norm and gate backward from the forward's y,
        // with no o recomputed.  z = sigmoid(gate) in the forward's own form, so
        // n = y / z = y (1 + 2^(-gate log2 e)) undoes its gating (to the bf16
        // rounding of y; 0 where the forward's z was 0, gate < about -87);
        // r = 1/RMS(o) from the forward.  dn = dy z, dgate = dn n (1 - z),
        // dO = r (dn - n mean(dn n)); rows past the tile get 0.  v (refilled only
        // once MMA4 of the tile before has read Vdec) is waited for after the
        // first loop, which does not read it.
        wait_plain(&sh.bar_g, ph, failed);
        wait_plain(&sh.bar_y, ph, failed);
        wait_plain(&sh.bar_dy, ph, failed);
        {
          uint4 graw[4], yraw[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            graw[u] = *tile_at(Qs, i, 4 * qd + u);
            yraw[u] = *tile_at(SB, i, 4 * qd + u);
          }
          // z and n kept in fp32 in this thread's P and tA columns of TMEM until
          // the second loop (MMA5 writes dP, and MMA6 I, only after this phase)
          f2 sdn = 0ull;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            float zs[16], ns[16];
#pragma unroll
            for (int uu = 0; uu < 2; ++uu) {
              const int u = 2 * hf + uu;
              f2 gz[4], yv[4], dv[4];
              unpack4x2(graw[u], gz);
              unpack4x2(yraw[u], yv);
              unpack4x2(*tile_at(PM, i, 4 * qd + u), dv);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                f2 z, iz;
                sigmoid_e2_inv(gz[e], z, iz);
                float n0, n1;
                split2(mul2(yv[e], iz), n0, n1);
                if (!(fabsf(n0) <= 3.0e38f)) n0 = 0.f;  // z was 0 (or y not finite)
                if (!(fabsf(n1) <= 3.0e38f)) n1 = 0.f;
                const f2 nv = mk2(n0, n1);
                sdn = fma2(mul2(dv[e], z), nv, sdn);
                split2(z, zs[8 * uu + 2 * e], zs[8 * uu + 2 * e + 1]);
                ns[8 * uu + 2 * e] = n0;
                ns[8 * uu + 2 * e + 1] = n1;
              }
            }
            umma::tmem_st16(myP + 16 * hf, zs);
            umma::tmem_st16(ta + col + 16 * hf, ns);
          }
          umma::tmem_wait_st();
          sh.red_do[1][qd][i] = hsum2(sdn);
          named_sync(5 + sub, 128);
          cp_async_wait();  // this thread's 1/RMS(o) and 1/RMS(q) slots
          wait_plain(&sh.bar_v, ph, failed);
          const float ro = sh.r_o[buf][qd][i];
          const float mean = (sh.red_do[1][0][i] + sh.red_do[1][1][i] + sh.red_do[1][2][i] +
                              sh.red_do[1][3][i]) / (float)D;
          const f2 ro2 = dup2(ro), nmean = dup2(-mean), one = dup2(1.f), keep = dup2(valid ? 1.f : 0.f);
          f2 vd = 0ull;
          uint32_t zr[2][16], nr[2][16];  // z and n back from TMEM under one wait
          umma::tmem_ld16_nowait(myP, zr[0]);
          umma::tmem_ld16_nowait(myP + 16, zr[1]);
          umma::tmem_ld16_nowait(ta + col, nr[0]);
          umma::tmem_ld16_nowait(ta + col + 16, nr[1]);
          umma::tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 *gp = tile_at(Qs, i, 4 * qd + u);
            f2 dv[4], vv[4], dg[4], dd[4];
            unpack4x2(*tile_at(PM, i, 4 * qd + u), dv);
            unpack4x2(*tile_at(Vs, i, 4 * qd + u), vv);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int w = 8 * (u & 1) + 2 * e;
              const f2 z = mk2(__uint_as_float(zr[u >> 1][w]), __uint_as_float(zr[u >> 1][w + 1]));
              const f2 nv = mk2(__uint_as_float(nr[u >> 1][w]), __uint_as_float(nr[u >> 1][w + 1]));
              const f2 dn = mul2(dv[e], z);
              dg[e] = mul2(mul2(dn, nv), fma2(z, dup2(-1.f), one));
              dd[e] = mul2(mul2(ro2, fma2(nv, nmean, dn)), keep);
              vd = fma2(vv[e], dd[e], vd);
            }
            *tile_at(PM, i, 4 * qd + u) = pack4x2(dg);
            *gp = pack4x2(dd);
          }
          sh.vd_part[qd][i] = hsum2(vd);
        }
        warp_arrive(&sh.bar_do, lane);

        // [W2] given y, after [W4] (y is in SB until then): S (bf16, for MMA6)
        // over y, S <- gamma^c S, once MMA7 / MMA4 of tile n - 1 are done
        if (n >= 1) wait_or_fail(&sh.bar_m74, (n - 1) & 1, failed);
        {
          float sv[32];
          umma::tmem_ld2x16(myS, sv);
          f2 x[16];
          pairs_of(sv, x);
#pragma unroll
          for (int u = 0; u < 4; ++u) *tile_at(SB, i, 4 * qd + u) = pack4x2(&x[4 * u]);
          const f2 carry = dup2(sh.pw[c]);
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) x[e2] = mul2(x[e2], carry);
          floats_of(x, sv);
          umma::tmem_st32(myS, sv);
          umma::tmem_wait_st();
        }
        warp_arrive(&sh.bar_sb, lane);
      }

      if (drain) {
        // [W6] dq of tile n - 1: dQ~ from TMEM, RoPE^T, RMSNorm backward against raw q
        // (the K buffer of tile n - 1), in place; pairs m = 16 qd .. 16 qd + 15.  Runs
        // while MMA5 / MMA6 of tile n are in flight.
        // (in the last step no [W2] has waited for MMA7 of tile n - 1: wait here)
        if (!have) wait_or_fail(&sh.bar_m74, (n - 1) & 1, failed);
        wait_plain(&sh.bar_qr, (n - 1) & 1, failed);
        {
          uint4 qr[4];
          ld_pairs(Kp, i, qd, qr);
          if (kSaved)
            feature_grad_saved(tap, qr, 1.f, 1.f, sh.r_saved[buf ^ 1][qd][i], P.pos_offset + prev_c0 + i,
                               i, qd, sub, sh.ru, sh.red_dq[0], Kp);
          else
            feature_grad_pairs(tap, qr, 1.f, P.pos_offset + prev_c0 + i, i, qd, sub, P.eps, sh.ru,
                               sh.red_dq, Kp);
        }
        warp_arrive(&sh.bar_w6, lane);
      }

      else if (have) {
        named_sync(5 + sub, 128);  // orders [W4]'s vd_part before [W5] reads it
      }

      if (have) {
        // [W5] after MMA5 / MMA6: dPm (diagonal: fp32 v_i . do_i) over the dP
        // columns of TMEM (MMA7's A operand, laid out as Pm in [W3]),
        // I <- gamma^{i+1} I, V -> Vdec (in place)
        wait_or_fail(&sh.bar_m56, ph, failed);
        {
          float pv[32];
          umma::tmem_ld2x16(myP, pv);
          f2 x[16];
          pairs_of(pv, x);
          mask_lower_table(x, sh.dm, i, (int)col);
          const float vd = qd == sub ? sh.vd_part[0][i] + sh.vd_part[1][i] + sh.vd_part[2][i] +
                                           sh.vd_part[3][i]
                                     : 0.f;
          store_tmem_bf16(myP, x, qd == sub ? i - (int)col : -1, vd);
          if (qd == sub && valid) P.ddiag[((size_t)b * P.H + h) * P.T + c0 + i] = vd;
          float iv[32];
          umma::tmem_ld2x16(ta + col, iv);
          const f2 wi = dup2(sh.pw[i + 1]);
          pairs_of(iv, x);
#pragma unroll
          for (int e = 0; e < 16; ++e) x[e] = mul2(x[e], wi);
          floats_of(x, iv);
          umma::tmem_st32(ta + col, iv);
          const f2 wv = dup2(valid ? sh.pw[c - 1 - i] : 0.f);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 *p = tile_at(Vs, i, 4 * qd + u);
            f2 f[4];
            unpack4x2(*p, f);
#pragma unroll
            for (int e = 0; e < 4; ++e) f[e] = mul2(f[e], wv);
            *p = pack4x2(f);
          }
          umma::tmem_wait_st();
        }
        warp_arrive(&sh.bar_w5, lane);
        prev_c0 = c0;
      }
    }
  }
  if (failed) atomicOr(&sh.failed, 1u);
  sync_tc();
  if (sh.failed && tid == 0 && P.err) atomicOr(P.err, 4u);
  if (warp == 0) umma::tmem_dealloc(tm, 512);
}

// ------------------------------------------------------------------ dk / dv pass

struct DkdvShared {
  unsigned long long ru[kMaxPairs];  // RoPE phase increments (load_rope_table)
  float red_dk[2][4][ROWS];  // [V6b] quarter parts of sum k^2 and sum g.k of each row
  float qk_diag[ROWS];       // [V1] -> [V3] fp32 k~_i . q~_i of the tile
  float r_saved[4][ROWS];    // saved features: 1 / RMS(k) of row i for [V6] of thread (qd, i)
  float pw[ROWS + 1];
  alignas(16) float du[4][DM_STRIDE];  // transposed causal-mask table (fill_mask_table_upper)
  uint64_t bar_q, bar_k, bar_v, bar_dot;                    // TMA loads of q, k, v, dO
  uint64_t bar_kr;                                          // TMA: raw k again, into X, for [V6]
  uint64_t bar_m1, bar_m2, bar_dv, bar_dk, bar_eupd;        // MMA commits
  uint64_t bar_feat, bar_eb, bar_x, bar_xp, bar_dvout, bar_dkout;  // workers
  uint32_t tmem_base;
  uint32_t failed;
};

// dk / dv pass, warp-specialized, over the tiles of a segment in reverse, with
// E (the gradient reaching the state from later tokens) carried in TMEM:
//   M1   = K~ Q~^T (fp16)                       into tA
//   M2   = V dO^T                               into tB
//   dV   = X dO + K~dec Eb,    X  = M1 (.) D^T  (fp32 k~_i . q~_i on the diagonal)
//   dK~  = X' Q~ + Vdec Eb^T,  X' = M2 (.) D^T  (fp32 v_i . do_i on the diagonal)
//   E   <- gamma^c E + Q~^T dOw,  dOw = diag(gamma^{i+1}) dO
// with D^T_ij = gamma^{j-i} for j >= i, K~dec / Vdec rows scaled by gamma^{c-1-i}
// and Eb = bf16(E) at the tile's end.  X and X' are MMA A operands in tensor
// memory (packed bf16, 64 columns each next to E).  Worker warps, per tile:
//   [V1] q~, k~ (fp16, in place)             [V2] Eb, E <- gamma^c E
//   [V3] X -> TMEM, k~ -> K~dec               [V4] Vdec, q~ -> bf16, X' -> TMEM
//   [V5] dv -> K (over K~dec), dO -> dOw      [V6] dk (RoPE^T, RMSNorm backward
//                                                  against raw k) -> X (over raw k)
// The issuer warp issues the MMAs as their operands are ready (the E update
// right behind dK~: both only read Q~), stores dv and dk by TMA and refills Q,
// K, V and dO for the tile before as each is freed: V once dK~ has read Vdec
// (a whole tile before its next reader, M2), since dk leaves through X.  Raw
// k for the RMSNorm backward arrives by TMA in the X buffer, once the dk store
// of the tile after has read it; the v . do diagonal (one word per row) is the
// only plain load.
// kSaved: tmq / tmk map the forward's saved fp16 q~, k~.  [V1] is skipped (M1
// waits for the copies instead), the k~ . q~ diagonal and 1/RMS(k) are read
// from the saved scalars, X receives k~ and [V6] uses feature_grad_saved.
template <bool kSaved>
__global__ void __launch_bounds__(NTO, 1)
    tc_bwd_dkdv_kernel(const __grid_constant__ MixerParams P, const __grid_constant__ CUtensorMap tmq,
                       const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                       const __grid_constant__ CUtensorMap tmo, const __grid_constant__ CUtensorMap tmdk,
                       const __grid_constant__ CUtensorMap tmdv) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  // Q: raw q -> q~ (fp16) -> q~ (bf16).  K: raw k -> k~ (fp16) -> K~dec -> dv.
  // V: v -> Vdec.  DO: dO -> dOw.  EB: Eb.  X: raw k (saved k~) of the tile, for [V6] -> dk.
  unsigned char *Qt = base, *Kt = base + TILE, *Vt = base + 2 * TILE, *DOt = base + 3 * TILE;
  unsigned char *EB = base + 4 * TILE, *X = base + 5 * TILE;
  DkdvShared &sh = *reinterpret_cast<DkdvShared *>(base + 6 * TILE);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int t0 = g * P.seg_len, t1 = min(P.T, t0 + P.seg_len);
  const int CV = P.chunk;
  const int ntile = ceil_div(t1 - t0, CV);
  const float l2g = log2f(P.gamma[h]);
  const uint32_t tile_bytes = (uint32_t)CV * D * 2;

  if (tid == 0) {
    uint64_t *bars[] = {&sh.bar_q, &sh.bar_k, &sh.bar_v, &sh.bar_dot, &sh.bar_kr, &sh.bar_m1,
                        &sh.bar_m2, &sh.bar_dv, &sh.bar_dk, &sh.bar_eupd};
    for (uint64_t *bar : bars) umma::mbar_init(bar, 1);
    uint64_t *wbars[] = {&sh.bar_feat, &sh.bar_eb, &sh.bar_x, &sh.bar_xp, &sh.bar_dvout,
                         &sh.bar_dkout};
    for (uint64_t *bar : wbars) umma::mbar_init(bar, NWORK);
    umma::mbar_fence_init();
    sh.failed = 0;
  }
  if (tid <= ROWS) sh.pw[tid] = exp2f((float)tid * l2g);
  fill_mask_table_upper(sh.du, l2g, tid, NTO);
  load_rope_table(sh.ru, P, tid);
  if (warp == 0) umma::tmem_alloc(&sh.tmem_base, 512);
  if (CV < ROWS) {  // rows [CV, 128) of V and DO are never written by TMA: clear them once
    for (int e = tid; e < 2 * (ROWS - CV) * 16; e += NTO) {
      const int r = e % ((ROWS - CV) * 16);
      *tile_at(e < (ROWS - CV) * 16 ? Vt : DOt, CV + r / 16, r % 16) = make_uint4(0, 0, 0, 0);
    }
    if (kSaved)  // nor those of Q and K, which [V1] would have zeroed
      for (int e = tid; e < 2 * (ROWS - CV) * 16; e += NTO) {
        const int r = e % ((ROWS - CV) * 16);
        *tile_at(e < (ROWS - CV) * 16 ? Qt : Kt, CV + r / 16, r % 16) = make_uint4(0, 0, 0, 0);
      }
  }
  sync_tc();
  const uint32_t tm = sh.tmem_base;
  const uint32_t tA = tm, tB = tm + 128, tE = tm + 256, tX = tm + 384;  // tX: X, then X' at + 64
  bool failed = false;

  if (warp >= NWORK) {
    // ---------------------------------------------------------------- issuer warpgroup
    if (warp == NWORK && lane == 0) {
      const uint32_t id_kq16 = umma::idesc_bf16(128, 128, false, false, true);  // fp16 K~ Q~^T
      const uint32_t id_kmn = umma::idesc_bf16(128, 128, false, true);
      const uint32_t id_kk = umma::idesc_bf16(128, 128, false, false);
      const uint32_t id_mnmn = umma::idesc_bf16(128, 128, true, true);
      const uint32_t aQ = umma::smem_u32(Qt), aK = umma::smem_u32(Kt), aV = umma::smem_u32(Vt),
                     aDO = umma::smem_u32(DOt), aE = umma::smem_u32(EB);
      {
        const int cl = t0 + (ntile - 1) * CV;
        umma::mbar_expect_tx(&sh.bar_q, tile_bytes);
        tma_tile(Qt, &tmq, b, h, cl, &sh.bar_q);
        umma::mbar_expect_tx(&sh.bar_k, tile_bytes);
        tma_tile(Kt, &tmk, b, h, cl, &sh.bar_k);
        umma::mbar_expect_tx(&sh.bar_v, tile_bytes);
        tma_tile(Vt, &tmv, b, h, cl, &sh.bar_v);
        umma::mbar_expect_tx(&sh.bar_dot, tile_bytes);
        tma_tile(DOt, &tmo, b, h, cl, &sh.bar_dot);
        umma::mbar_expect_tx(&sh.bar_kr, tile_bytes);
        tma_tile(X, &tmk, b, h, cl, &sh.bar_kr);
      }
      bool x_pending = false;  // raw k of this tile waits for the dk store to leave X
      for (int it = 0; it < ntile; ++it) {
        const int n = ntile - 1 - it;
        const uint32_t ph = it & 1;
        const int c0 = t0 + n * CV;
        if (kSaved) {
          wait_or_fail(&sh.bar_q, ph, failed);
          wait_or_fail(&sh.bar_k, ph, failed);
        } else {
          wait_or_fail(&sh.bar_feat, ph, failed);
        }
        if (!failed) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // M1 = K~ Q~^T
            umma::mma_ss(tA, umma::desc_kmajor(aK, kk, ROWS), umma::desc_kmajor(aQ, kk, ROWS), id_kq16, kk > 0);
          umma::commit(&sh.bar_m1);
        }
        // X takes this tile's raw k once the dk store of the tile after has read
        // it (after M1, which needs neither; [V6] is the first reader)
        if (x_pending && !failed) {
          umma::bulk_wait_read();
          umma::mbar_expect_tx(&sh.bar_kr, tile_bytes);
          tma_tile(X, &tmk, b, h, c0, &sh.bar_kr);
        }
        x_pending = false;
        wait_or_fail(&sh.bar_v, ph, failed);
        wait_or_fail(&sh.bar_dot, ph, failed);
        if (!failed) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // M2 = V dO^T
            umma::mma_ss(tB, umma::desc_kmajor(aV, kk, ROWS), umma::desc_kmajor(aDO, kk, ROWS), id_kk, kk > 0);
          umma::commit(&sh.bar_m2);
          if (n > 0) {  // the tile before into L2 ahead of its copies
            tma_prefetch_tile(&tmq, b, h, c0 - CV);
            tma_prefetch_tile(&tmk, b, h, c0 - CV);
            tma_prefetch_tile(&tmv, b, h, c0 - CV);
            tma_prefetch_tile(&tmo, b, h, c0 - CV);
          }
        }
        wait_or_fail(&sh.bar_x, ph, failed);
        wait_or_fail(&sh.bar_eb, ph, failed);
        if (!failed) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dV = X dO (X in TMEM)
            umma::mma_ts(tA, tX + 8 * kk, umma::desc_mnmajor(aDO, kk, ROWS), id_kmn, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dV += K~dec Eb
            umma::mma_ss(tA, umma::desc_kmajor(aK, kk, ROWS), umma::desc_mnmajor(aE, kk, ROWS), id_kmn, 1u);
          umma::commit(&sh.bar_dv);
        }
        wait_or_fail(&sh.bar_xp, ph, failed);
        if (!failed) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dK~ = X' Q~ (X' in TMEM)
            umma::mma_ts(tB, tX + 64 + 8 * kk, umma::desc_mnmajor(aQ, kk, ROWS), id_kmn, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dK~ += Vdec Eb^T
            umma::mma_ss(tB, umma::desc_kmajor(aV, kk, ROWS), umma::desc_kmajor(aE, kk, ROWS), id_kk, 1u);
          umma::commit(&sh.bar_dk);
        }
        wait_or_fail(&sh.bar_dvout, ph, failed);
        if (!failed) {
          tma_store_tile(&tmdv, Kt, b, h, c0);
          umma::bulk_commit();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // E += Q~^T dOw
            umma::mma_ss(tE, umma::desc_mnmajor(aQ, kk, ROWS), umma::desc_mnmajor(aDO, kk, ROWS), id_mnmn, 1u);
          umma::commit(&sh.bar_eupd);
        }
        // E update done (on the last tile too: TMEM is freed at the end), and so
        // dK~ before it: Q, DO and V take the tile before; once the dv store has
        // left K, so does K
        wait_or_fail(&sh.bar_eupd, ph, failed);
        if (n > 0) {
          if (!failed) {
            umma::mbar_expect_tx(&sh.bar_q, tile_bytes);
            tma_tile(Qt, &tmq, b, h, c0 - CV, &sh.bar_q);
            umma::mbar_expect_tx(&sh.bar_dot, tile_bytes);
            tma_tile(DOt, &tmo, b, h, c0 - CV, &sh.bar_dot);
            umma::mbar_expect_tx(&sh.bar_v, tile_bytes);
            tma_tile(Vt, &tmv, b, h, c0 - CV, &sh.bar_v);
            umma::bulk_wait_read();
            umma::mbar_expect_tx(&sh.bar_k, tile_bytes);
            tma_tile(Kt, &tmk, b, h, c0 - CV, &sh.bar_k);
          }
        }
        // dk out of X (X takes raw k of the tile before after that tile's M1)
        wait_or_fail(&sh.bar_dkout, ph, failed);
        if (!failed) {
          tma_store_tile(&tmdk, X, b, h, c0);
          umma::bulk_commit();
          x_pending = n > 0;
        }
      }
      umma::bulk_wait_all();
    }
  } else {
    // ---------------------------------------------------------------- worker warps
    const int sub = warp & 3, qd = warp >> 2, i = 32 * sub + lane;  // TMEM phases
    const int fr = 8 * warp + (lane >> 2), fu = lane & 3;           // feature map: row, quarter
    const uint32_t lane_base = (uint32_t)(32 * sub) << 16;
    const uint32_t col = 32 * qd;
    {  // gradient reaching the segment's last state from later tokens -> TMEM
      const float *ein = P.seg2 + (((size_t)b * P.H + h) * P.nseg + g) * (size_t)D * D;
      const float4 *s4 = reinterpret_cast<const float4 *>(ein + (size_t)i * D + col);
      float v[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 x = s4[u];
        v[4 * u] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
      }
      umma::tmem_st32(tE + lane_base + col, v);
      umma::tmem_wait_st();
    }
    for (int it = 0; it < ntile; ++it) {
      const int n = ntile - 1 - it;
      const uint32_t ph = it & 1;
      const int c0 = t0 + n * CV, c = min(CV, t1 - c0);
      const bool valid = i < c;
      const long long pos = P.pos_offset + c0 + i;
      const float wdec = valid ? sh.pw[c - 1 - i] : 0.f;

      // [V1] q~, k~ (fp16, in place): row fr, pairs [16 fu, 16 fu + 16)
      wait_or_fail(&sh.bar_q, ph, failed);
      wait_or_fail(&sh.bar_k, ph, failed);
      if (!kSaved) {
        uint4 qr[4], kr[4];
        ld_pairs(Qt, fr, fu, qr);
        ld_pairs(Kt, fr, fu, kr);
        if (!(fr < c))
          qr[0] = qr[1] = qr[2] = qr[3] = kr[0] = kr[1] = kr[2] = kr[3] = make_uint4(0, 0, 0, 0);
        float sq, sk, qk;
        norms_and_dot(qr, kr, sq, sk, qk);
        sq += __shfl_xor_sync(0xffffffffu, sq, 1);
        sk += __shfl_xor_sync(0xffffffffu, sk, 1);
        qk += __shfl_xor_sync(0xffffffffu, qk, 1);
        sq += __shfl_xor_sync(0xffffffffu, sq, 2);
        sk += __shfl_xor_sync(0xffffffffu, sk, 2);
        qk += __shfl_xor_sync(0xffffffffu, qk, 2);
        const float rq = rsqrtf(sq / (float)D + P.eps);
        const float rk = rsqrtf(sk / (float)D + P.eps) * P.kscale;
        if (fu == 0) sh.qk_diag[fr] = qk * rq * rk;
        feature_qk_store(qr, kr, rq, rk, P.pos_offset + c0 + fr, fu, sh.ru, Qt, Kt, fr);
        warp_arrive(&sh.bar_feat, lane);
      } else {  // saved scalars of row i into slots only this thread reads (no
                // register held across the phases): 1 / RMS(k_i) for [V6] and, on
                // the diagonal warps, k~_i . q~_i for [V3]
        if (valid) {
          cp_async4(&sh.r_saved[qd][i], saved_scalar(P, kSavedRk, b, h, c0 + i));
          if (qd == sub) cp_async4(&sh.qk_diag[i], saved_scalar(P, kSavedDiag, b, h, c0 + i));
        } else {
          sh.r_saved[qd][i] = 0.f;
          if (qd == sub) sh.qk_diag[i] = 0.f;
        }
      }
      // [V2] after the E update of the tile after: Eb = bf16(E), E <- gamma^c E
      if (it > 0) wait_or_fail(&sh.bar_eupd, (it - 1) & 1, failed);
      {
        float ev[32];
        umma::tmem_ld2x16(tE + lane_base + col, ev);
        f2 x[16];
        pairs_of(ev, x);
#pragma unroll
        for (int u = 0; u < 4; ++u) *tile_at(EB, i, 4 * qd + u) = pack4x2(&x[4 * u]);
        const f2 carry = dup2(sh.pw[c]);
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] = mul2(x[e], carry);
        floats_of(x, ev);
        umma::tmem_st32(tE + lane_base + col, ev);
        umma::tmem_wait_st();
      }
      warp_arrive(&sh.bar_eb, lane);

      // [V3] after M1: X = bf16(M1 (.) D^T) with the fp32 diagonal; k~ -> K~dec
      // (with saved features k~ came by TMA, so its row is read and weighted
      // before M1 is done, and only the rewrite waits)
      uint4 kdnew[4];
      if (kSaved) {
        const f2 w = dup2(wdec);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          f2 f[4];
          unpack4x2h(*tile_at(Kt, i, 4 * qd + u), f);
#pragma unroll
          for (int e = 0; e < 4; ++e) f[e] = mul2(f[e], w);
          kdnew[u] = pack4x2(f);
        }
      }
      wait_or_fail(&sh.bar_m1, ph, failed);
      {
        float v[32];
        umma::tmem_ld2x16(tA + lane_base + col, v);
        f2 x[16];
        pairs_of(v, x);
        mask_upper_table(x, sh.du, i, (int)col);
        // X as packed bf16 into TMEM (row i, K = 32 qd .. 32 qd + 31 at columns
        // 16 qd ..); the diagonal entry (element i - 32 qd on the warps with
        // qd == sub) is k~_i . q~_i in fp32, written in [V1] by warps
        // 4 sub .. 4 sub + 3 and ordered by bar_feat -> M1
        if (kSaved) cp_async_wait();
        store_tmem_bf16(tX + lane_base + 16 * qd, x, qd == sub ? i - (int)col : -1,
                        qd == sub ? sh.qk_diag[i] : 0.f);
        if (kSaved) {
#pragma unroll
          for (int u = 0; u < 4; ++u) *tile_at(Kt, i, 4 * qd + u) = kdnew[u];
        } else {  // k~ written by other threads in [V1]: read after M1 (which orders them)
          const f2 w = dup2(wdec);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 *p = tile_at(Kt, i, 4 * qd + u);
            f2 f[4];
            unpack4x2h(*p, f);
#pragma unroll
            for (int e = 0; e < 4; ++e) f[e] = mul2(f[e], w);
            *p = pack4x2(f);
          }
        }
        umma::tmem_wait_st();
      }
      warp_arrive(&sh.bar_x, lane);

      // [V4] after M2: Vdec, q~ -> bf16; X' = M2 (.) D^T (fp32 v_i . do_i on the
      // diagonal, from the dq pass) into X once dV has read X
      {
        const float vdiag = (qd == sub && valid) ? P.ddiag[((size_t)b * P.H + h) * P.T + c0 + i] : 0.f;
        // v (once its copy is in) and q~ of the row are read and converted
        // before M2 is done (M2 only reads them); the rewrites wait for it
        wait_plain(&sh.bar_v, ph, failed);
        const f2 w = dup2(wdec);
        uint4 vnew[4], qnew[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          f2 f[4];
          unpack4x2(*tile_at(Vt, i, 4 * qd + u), f);
#pragma unroll
          for (int e = 0; e < 4; ++e) f[e] = mul2(f[e], w);
          vnew[u] = pack4x2(f);
          unpack4x2h(*tile_at(Qt, i, 4 * qd + u), f);
          qnew[u] = pack4x2(f);
        }
        wait_or_fail(&sh.bar_m2, ph, failed);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          *tile_at(Vt, i, 4 * qd + u) = vnew[u];
          *tile_at(Qt, i, 4 * qd + u) = qnew[u];
        }
        float v[32];
        umma::tmem_ld2x16(tB + lane_base + col, v);
        f2 x[16];
        pairs_of(v, x);
        mask_upper_table(x, sh.du, i, (int)col);
        store_tmem_bf16(tX + 64 + lane_base + 16 * qd, x, qd == sub ? i - (int)col : -1, vdiag);
        umma::tmem_wait_st();
      }
      warp_arrive(&sh.bar_xp, lane);

      // [V5] after dV: dv -> K over K~dec, for a TMA store; dO has been read by
      // M2 and dV: dO -> dOw = gamma^{i+1} dO in place, for the E update
      // (dO's row, in since its copy landed, is read and weighted first; the
      // rewrite waits for dV, the last MMA that reads dO unweighted)
      wait_plain(&sh.bar_dot, ph, failed);
      uint4 donew[4];
      {
        const f2 w = dup2(sh.pw[i + 1]);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          f2 f[4];
          unpack4x2(*tile_at(DOt, i, 4 * qd + u), f);
#pragma unroll
          for (int e = 0; e < 4; ++e) f[e] = mul2(f[e], w);
          donew[u] = pack4x2(f);
        }
      }
      wait_or_fail(&sh.bar_dv, ph, failed);
      {
        float v[32];
        umma::tmem_ld2x16(tA + lane_base + col, v);
        f2 x[16];
        pairs_of(v, x);
#pragma unroll
        for (int u = 0; u < 4; ++u) *tile_at(Kt, i, 4 * qd + u) = pack4x2(&x[4 * u]);
#pragma unroll
        for (int u = 0; u < 4; ++u) *tile_at(DOt, i, 4 * qd + u) = donew[u];
      }
      warp_arrive(&sh.bar_dvout, lane);

      // [V6] after dK~: dk, over the chunks of raw k it reads (this thread's own)
      wait_or_fail(&sh.bar_kr, ph, failed);
      {
        uint4 kraw[4];  // raw k (saved k~) pairs of row i, read before dK~ is done
        ld_pairs(X, i, qd, kraw);
        wait_or_fail(&sh.bar_dk, ph, failed);
        if (kSaved)
          feature_grad_saved(tB + lane_base, kraw, P.kscale, 1.f / P.kscale, sh.r_saved[qd][i], pos,
                             i, qd, sub, sh.ru, sh.red_dk[0], X);
        else
          feature_grad_pairs(tB + lane_base, kraw, P.kscale, pos, i, qd, sub, P.eps, sh.ru, sh.red_dk, X);
      }
      warp_arrive(&sh.bar_dkout, lane);
    }
    // the first segment's E after its first tile's update is the gradient of
    // the state entering the sequence
    if (P.dstate_in && g == 0) {
      wait_or_fail(&sh.bar_eupd, (ntile - 1) & 1, failed);
      float ev[32];
      umma::tmem_ld2x16(tE + lane_base + col, ev);
      float4 *o4 = reinterpret_cast<float4 *>(P.dstate_in + (((size_t)b * P.H + h) * D + i) * D + col);
#pragma unroll
      for (int u = 0; u < 8; ++u) o4[u] = make_float4(ev[4 * u], ev[4 * u + 1], ev[4 * u + 2], ev[4 * u + 3]);
    }
  }
  if (failed) atomicOr(&sh.failed, 1u);
  sync_tc();
  if (sh.failed && tid == 0 && P.err) atomicOr(P.err, 8u);
  if (warp == 0) umma::tmem_dealloc(tm, 512);
}

constexpr size_t kBwdSmem = 6 * TILE + sizeof(DkdvShared) + 1024;
static_assert(kBwdSmem <= 232448, "dk/dv pass exceeds 227 KiB of shared memory per CTA");
constexpr size_t kDqSmem = 6 * TILE + sizeof(DqShared) + 1024;
static_assert(kDqSmem <= 232448, "dq pass exceeds 227 KiB of shared memory per CTA");

}  // namespace
}  // namespace tc

namespace {
cudaError_t qk_maps(const MixerParams &P, CUtensorMap *mq, CUtensorMap *mk);

template <bool kSaved, bool kY>
cudaError_t launch_dq_variant(const MixerParams &P, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mg, mo, mdg, mdq, mdy, myi;
  cudaError_t e;
  if ((e = qk_maps(P, &mq, &mk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mv, P.v, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mg, P.g, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mo, P.dO, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mdg, P.dg, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mdq, P.dq, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mdy, P.dy, P, P.chunk)) != cudaSuccess) return e;
  // the forward's y (given y), else an unused copy of the dy map
  if ((e = tc::make_map(&myi, kY ? P.y_in : P.dy, P, P.chunk)) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc::tc_bwd_dq_kernel<kSaved, kY>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc::kDqSmem);
  if (e != cudaSuccess) return e;
  tc::tc_bwd_dq_kernel<kSaved, kY><<<dim3(P.nseg, P.H, P.B), tc::NTO, tc::kDqSmem, st>>>(
      P, mq, mk, mv, mg, mo, mdg, mdq, mdy, myi);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_tc_bwd_dq(const MixerParams &P, cudaStream_t st) {
  if (P.saved && P.y_in) return launch_dq_variant<true, true>(P, st);
  return P.saved ? launch_dq_variant<true, false>(P, st) : launch_dq_variant<false, false>(P, st);
}

namespace {
// q and k operand maps: the raw inputs, or the forward's saved fp16 q~, k~.
cudaError_t qk_maps(const MixerParams &P, CUtensorMap *mq, CUtensorMap *mk) {
  cudaError_t e;
  if (P.saved) {
    if ((e = tc::make_map(mq, P.saved, P, P.chunk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != cudaSuccess)
      return e;
    return tc::make_map(mk, P.saved + saved_k_offset(P.B, P.T, P.H, P.D), P, P.chunk,
                        CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  }
  if ((e = tc::make_map(mq, P.q, P, P.chunk)) != cudaSuccess) return e;
  return tc::make_map(mk, P.k, P, P.chunk);
}

template <bool kSaved>
cudaError_t launch_dkdv_variant(const MixerParams &P, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mo, mdk, mdv;
  cudaError_t e;
  if ((e = qk_maps(P, &mq, &mk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mv, P.v, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mo, P.dO, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mdk, P.dk, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mdv, P.dv, P, P.chunk)) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc::tc_bwd_dkdv_kernel<kSaved>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)tc::kBwdSmem);
  if (e != cudaSuccess) return e;
  tc::tc_bwd_dkdv_kernel<kSaved><<<dim3(P.nseg, P.H, P.B), tc::NTO, tc::kBwdSmem, st>>>(
      P, mq, mk, mv, mo, mdk, mdv);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_tc_bwd_dkdv(const MixerParams &P, cudaStream_t st) {
  return P.saved ? launch_dkdv_variant<true>(P, st) : launch_dkdv_variant<false>(P, st);
}

}  // namespace hla
