// tc_backward.cu — tensor-core (tcgen05) kernels of the prefill backward for
// bf16 inputs at d = 128.
//
// The loss is L = <dy, y> + <dstate_out, S_T> with y from Eq. 18 of
// arXiv 2601.22156 (Appendix A).  Per tile of c <= 128 tokens entering with
// state S (recomputed by the forward local-state pass and scan), D_ij =
// gamma^{i-j} for i >= j:
//
//   tc_bwd_dq_kernel (tiles in order, S carried in TMEM as in the forward)
//     O     = diag(gamma^{i+1}) Q~ S + (Q~ K~^T (.) D) V          MMA1-3 (recompute)
//     dgate = dy n sigma(g) (1 - sigma(g)),  n = O r,  r = 1/RMS(O)
//     dO    = r (dn - n mean(dn n)),  dn = dy sigma(g)              (to the workspace, bf16)
//     dQ~   = diag(gamma^{i+1}) dO S^T + ((dO V^T) (.) D) K~       MMA5-7
//     dq    = Norm^T RoPE^T dQ~
//     S    <- gamma^c S + (diag(gamma^{c-1-j}) K~)^T V              MMA4
//   tc_state_kernel<true> (tc_prefill.cu) then sums q~^T do per segment and
//   the fp32 scan (scan.cu) turns those sums into E, the gradient reaching the
//   state at each segment's last token from later tokens.
//   tc_bwd_dkdv_kernel (tiles in reverse, E carried in TMEM)
//     dV  = ((K~ Q~^T) (.) D^T) dO + diag(gamma^{c-1-i}) K~ E
//     dK~ = ((V dO^T) (.) D^T) Q~ + diag(gamma^{c-1-i}) V E^T
//     E  <- gamma^c E + (diag(gamma^{i+1}) Q~)^T dO
//     dk  = Norm^T RoPE^T dK~ / sqrt(d)
//
// Precision: K~ Q~^T runs on fp16 operands (its rounding would dominate dv
// on fast-decaying heads with bf16), the recomputed O uses the forward's fp16
// Q~ K~^T / Q~ S products, and every other product has bf16 operands with fp32
// accumulation.  Two diagonal entries are taken in fp32 on the CUDA cores
// instead: q~_i . k~_i (where it nearly cancels, o_i is small and dO_i ~ 1/|o_i|
// magnifies its error) and v_i . do_i (do_i is orthogonal to o_i, so this
// cancels wherever o_i is close to a multiple of v_i, e.g. at t = 0).  Decay weights that multiply a whole operand row are folded
// into that operand (K~dec, Vdec, Q~w); the one that multiplies a product row
// after the fact (gamma^{i+1} on dO S^T) gets its own TMEM accumulator.
//
// Threads: 512 per (b, h, segment), all in lockstep.  Thread (warp w, lane l)
// owns tile row i = 32 (w % 4) + l (its TMEM lane) and column quarter
// qd = w / 4; thread 0 issues the TMA copies and MMAs between CTA barriers.
#include "tc_common.cuh"

namespace hla {
namespace tc {

namespace {

struct BwdShared {
  unsigned long long ru[kMaxPairs];  // RoPE phase increments (load_rope_table)
  float red[4][ROWS];
  float red2[4][ROWS];
  float qk_diag[4][ROWS];  // parts of the fp32 q~_i . k~_i
  float vd_diag[4][ROWS];  // parts of the fp32 v_i . do_i
  float pw[ROWS + 1];
  float smax[NT / 32];
  uint64_t bar_tma[5];
  uint64_t bar_mma[6];
  uint32_t tmem_base;
};

// Sum of the four quarter parts of row i's diagonal entry.
__device__ __forceinline__ float diag_sum(const float (*part)[ROWS], int i) {
  return part[0][i] + part[1][i] + part[2][i] + part[3][i];
}

// Store 32 values of row i, columns [32 qd, 32 qd + 32), as bf16 into a tile.
__device__ __forceinline__ void store_quarter(unsigned char *tile, int i, int qd, const float (&v)[32]) {
#pragma unroll
  for (int u = 0; u < 4; ++u) *tile_at(tile, i, 4 * qd + u) = pack8(&v[8 * u]);
}

// Scale row i, columns [32 qd, 32 qd + 32) of a tile by w, converting fp16 ->
// bf16 (from_half) or bf16 -> bf16.
__device__ __forceinline__ void rescale_quarter(unsigned char *tile, int i, int qd, float w,
                                                bool from_half) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint4 *p = tile_at(tile, i, 4 * qd + u);
    float f[8];
    if (from_half)
      unpack8h(*p, f);
    else
      unpack8(*p, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] *= w;
    *p = pack8(f);
  }
}

// TMEM columns {16 qd .. 16 qd + 15} and {64 + 16 qd .. 64 + 16 qd + 15} of this
// thread's lane: the 16 RoPE pairs this thread owns.
__device__ __forceinline__ void tmem_ld_pairs(uint32_t taddr, int qd, float (&lo)[16],
                                              float (&hi)[16]) {
  umma::tmem_ld16(taddr + 16 * qd, lo);
  umma::tmem_ld16(taddr + 64 + 16 * qd, hi);
}

// This thread's 16 RoPE pairs of a raw input row (elements 16 qd .. 16 qd + 15
// and 64 + 16 qd ..), zeros when !valid.
__device__ __forceinline__ void load_pairs(uint4 (&ra)[4], const __nv_bfloat16 *raw, int qd,
                                           bool valid) {
  if (valid) {
    ra[0] = ldg16(raw + 16 * qd);
    ra[1] = ldg16(raw + 16 * qd + 8);
    ra[2] = ldg16(raw + 64 + 16 * qd);
    ra[3] = ldg16(raw + 64 + 16 * qd + 8);
  } else {
    ra[0] = ra[1] = ra[2] = ra[3] = make_uint4(0, 0, 0, 0);
  }
}

// Gradient of one feature row through RoPE and RMSNorm: g holds dL/d(rotated
// normalized row) for this thread's 16 pairs (lo = element m, hi = m + 64,
// m = 16 qd + e); ra = those pairs of the raw input row (load_pairs);
// r = 1 / RMS(raw).  Writes dL/draw for the pairs (bf16, zeros when !valid)
// into row i of the operand-layout tile `out`, for a TMA store.  The mean over
// the row needs the other three threads of the row: red is the [4][ROWS]
// scratch and the call holds one CTA barrier.
__device__ __forceinline__ void feature_grad_row(const float (&glo)[16], const float (&ghi)[16],
                                                 const uint4 (&ra)[4], float r, long long p,
                                                 int i, int qd, bool valid,
                                                 const unsigned long long *ru, float (*red)[ROWS],
                                                 unsigned char *out) {
  float n0[16], n1[16], g0[16], g1[16];
  {
    float f[8];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      unpack8(ra[hf], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) n0[8 * hf + e] = f[e] * r;
      unpack8(ra[2 + hf], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) n1[8 * hf + e] = f[e] * r;
    }
  }
  float dot = 0.f;
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    float c, s;
    rope_fast(p, ru[4 * e + qd], c, s);
    // transpose of (x0, x1) -> (x0 c - x1 s, x0 s + x1 c)
    g0[e] = glo[e] * c + ghi[e] * s;
    g1[e] = ghi[e] * c - glo[e] * s;
    dot = fmaf(g0[e], n0[e], fmaf(g1[e], n1[e], dot));
  }
  red[qd][i] = dot;
  __syncthreads();
  const float mean = (red[0][i] + red[1][i] + red[2][i] + red[3][i]) / (float)D;
  float a[16], bq[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    a[e] = valid ? r * (g0[e] - n0[e] * mean) : 0.f;
    bq[e] = valid ? r * (g1[e] - n1[e] * mean) : 0.f;
  }
  *tile_at(out, i, 2 * qd) = pack8(a);
  *tile_at(out, i, 2 * qd + 1) = pack8(a + 8);
  *tile_at(out, i, 8 + 2 * qd) = pack8(bq);
  *tile_at(out, i, 8 + 2 * qd + 1) = pack8(bq + 8);
}

// Bounded wait with a CTA-wide vote (every thread calls it); on a timeout
// every thread leaves the tile loop together.  A statement, not an expression:
// its `break` must reach the tile loop.
#define BWD_WAIT(bar, parity)          \
  if (wait_all((bar), (parity))) {     \
    failed = true;                     \
    break;                             \
  }

// ------------------------------------------------------------------ dq pass

__global__ void __launch_bounds__(NT, 1)
    tc_bwd_dq_kernel(const __grid_constant__ MixerParams P, const __grid_constant__ CUtensorMap tmq,
                     const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ CUtensorMap tmg, const __grid_constant__ CUtensorMap tmo,
                     const __grid_constant__ CUtensorMap tmdg, const __grid_constant__ CUtensorMap tmdq) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  // Q: raw q -> q~ (fp16); then gate (TMA) -> dO (bf16, in place; TMA-stored).
  // K pair j: raw k -> k~ (fp16) -> k~ (bf16) -> k~dec.
  // SB: Sb (fp16, scaled) -> S (bf16); then dq (TMA-stored).
  // PM: P (.) D; then dgate (TMA-stored); then dP (.) D.
  unsigned char *Qt = base, *Vt = base + 3 * TILE, *SB = base + 4 * TILE, *PM = base + 5 * TILE;
  BwdShared &sh = *reinterpret_cast<BwdShared *>(base + 6 * TILE);
  uint64_t *bar_q = &sh.bar_tma[0], *bar_k = &sh.bar_tma[1], *bar_v = &sh.bar_tma[3],
           *bar_g = &sh.bar_tma[4];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sub = warp & 3, qd = warp >> 2, i = 32 * sub + lane;
  const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int t0 = g * P.seg_len, t1 = min(P.T, t0 + P.seg_len);
  const int CV = P.chunk;
  const int ntile = ceil_div(t1 - t0, CV);
  const float gm = P.gamma[h];
  const float l2g = log2f(gm);
  const uint32_t tile_bytes = (uint32_t)CV * D * 2;

  if (tid == 0) {
    for (int j = 0; j < 5; ++j) umma::mbar_init(&sh.bar_tma[j], 1);
    for (int j = 0; j < 6; ++j) umma::mbar_init(&sh.bar_mma[j], 1);
    umma::mbar_fence_init();
  }
  if (tid <= ROWS) sh.pw[tid] = exp2f((float)tid * l2g);
  load_rope_table(sh.ru, P, tid);
  if (warp == 0) umma::tmem_alloc(&sh.tmem_base, 512);
  if (CV < ROWS)  // rows [CV, 128) of V are never written by TMA: clear them once
    for (int e = tid; e < (ROWS - CV) * 16; e += NT)
      *tile_at(Vt, CV + e / 16, e % 16) = make_uint4(0, 0, 0, 0);
  sync_tc();
  const uint32_t tm = sh.tmem_base;
  const uint32_t lb = (uint32_t)(32 * sub) << 16, col = 32 * qd;
  const uint32_t tP = tm + lb, tO = tm + 128 + lb, tI = tm + 256 + lb, tS = tm + 384 + lb;
  {  // entering state of the segment -> TMEM
    const float *sin_ = P.seg + (((size_t)b * P.H + h) * P.nseg + g) * (size_t)D * D;
    const float4 *s4 = reinterpret_cast<const float4 *>(sin_ + (size_t)i * D + col);
    float v[32];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float4 x = s4[u];
      v[4 * u] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
    }
    umma::tmem_st32(tS + col, v);
    umma::tmem_wait_st();
  }
  if (tid == 0) {
    umma::mbar_expect_tx(bar_q, tile_bytes);
    tma_tile(Qt, &tmq, b, h, t0, bar_q);
    for (int n = 0; n < 2 && n < ntile; ++n) {
      umma::mbar_expect_tx(&bar_k[n], tile_bytes);
      tma_tile(base + (1 + n) * TILE, &tmk, b, h, t0 + n * CV, &bar_k[n]);
    }
    umma::mbar_expect_tx(bar_v, tile_bytes);
    tma_tile(Vt, &tmv, b, h, t0, bar_v);
  }
  const uint32_t id_qk16 = umma::idesc_bf16(128, 128, false, false, true);
  const uint32_t id_qs16 = umma::idesc_bf16(128, 128, false, true, true);
  const uint32_t id_kmn = umma::idesc_bf16(128, 128, false, true);
  const uint32_t id_kk = umma::idesc_bf16(128, 128, false, false);
  const uint32_t id_mnmn = umma::idesc_bf16(128, 128, true, true);
  const uint32_t aQ = umma::smem_u32(Qt), aV = umma::smem_u32(Vt), aSB = umma::smem_u32(SB),
                 aPM = umma::smem_u32(PM);

  bool failed = false;
  for (int n = 0; n < ntile; ++n) {
    const int buf = n & 1;
    const uint32_t ph = n & 1;
    unsigned char *Kt = base + (1 + buf) * TILE;
    const uint32_t aK = aQ + (1 + buf) * TILE;
    const int c0 = t0 + n * CV, c = min(CV, t1 - c0);
    const bool valid = i < c;
    const long long pos = P.pos_offset + c0 + i;
    if (tid == 0) umma::bulk_wait_read();  // the previous dq store has left SB

    // [1] q~, k~ (fp16, in place); Sb = fp16(S 2^-e) per column quarter; S <- gamma^c S
    BWD_WAIT(bar_q, ph);
    BWD_WAIT(&bar_k[buf], (n >> 1) & 1);
    float rq, s_inv;
    {
      uint4 qr[4], kr[4];
      ld_pairs(Qt, i, qd, qr);
      ld_pairs(Kt, i, qd, kr);
      if (!valid) qr[0] = qr[1] = qr[2] = qr[3] = kr[0] = kr[1] = kr[2] = kr[3] = make_uint4(0, 0, 0, 0);
      sh.red[qd][i] = sumsq_pairs(qr);
      sh.red2[qd][i] = sumsq_pairs(kr);
      float sv[32];
      umma::tmem_ld2x16(tS + col, sv);
      float m = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) m = fmaxf(m, fabsf(sv[e]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) sh.smax[warp] = m;
      __syncthreads();
      rq = rsqrtf((sh.red[0][i] + sh.red[1][i] + sh.red[2][i] + sh.red[3][i]) / (float)D + P.eps);
      const float rk = rsqrtf((sh.red2[0][i] + sh.red2[1][i] + sh.red2[2][i] + sh.red2[3][i]) /
                                  (float)D + P.eps) * P.kscale;
      sh.qk_diag[qd][i] = feature_qk_store(qr, kr, rq, rk, pos, qd, sh.ru, Qt, Kt, i);
      m = fmaxf(fmaxf(sh.smax[4 * qd], sh.smax[4 * qd + 1]), fmaxf(sh.smax[4 * qd + 2], sh.smax[4 * qd + 3]));
      int e2 = 0;
      if (m > 0.f) frexpf(m, &e2);
      const float s_fwd = ldexpf(1.f, -e2);
      s_inv = ldexpf(1.f, e2);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float t[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = sv[8 * u + e] * s_fwd;
        *tile_at(SB, i, 4 * qd + u) = pack8h(t);
      }
      const float carry = sh.pw[c];
#pragma unroll
      for (int e = 0; e < 32; ++e) sv[e] *= carry;
      umma::tmem_st32(tS + col, sv);
      umma::tmem_wait_st();
    }
    umma::fence_async_smem();
    sync_tc();
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // MMA1: P = Q~ K~^T
        umma::mma_ss(tm, umma::desc_kmajor(aQ, kk, ROWS), umma::desc_kmajor(aK, kk, ROWS), id_qk16, kk > 0);
      umma::commit(&sh.bar_mma[0]);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // MMA2: O = Q~ Sb
        umma::mma_ss(tm + 128, umma::desc_kmajor(aQ, kk, ROWS), umma::desc_mnmajor(aSB, kk, ROWS), id_qs16,
                     kk > 0);
      umma::commit(&sh.bar_mma[1]);
    }

    // [2] Pm = bf16(P (.) D); k~ -> bf16; O <- gamma^{i+1} 2^e O; Sb -> S (bf16)
    BWD_WAIT(&sh.bar_mma[0], ph);
    {
      float pv[32];
      // the diagonal q~_i . k~_i from fp32 features: where it nearly cancels,
      // o_i and so 1 / RMS(o_i) hinge on it (fp16 operands lose it)
      mask_lower_block(tP + col, pv, i, sub, qd, valid, gm, sh.pw, true, diag_sum(sh.qk_diag, i));
      store_quarter(PM, i, qd, pv);
      rescale_quarter(Kt, i, qd, 1.f, true);
    }
    uint4 dyr[4];  // dy of row i for [3], loaded a phase early
    load_quarter(dyr, row_ptr(P.dy, P, b, h, valid ? c0 + i : c0), qd, valid);
    BWD_WAIT(&sh.bar_mma[1], ph);
    if (tid == 0) {  // MMA2 done: Q is free for this tile's gate
      umma::mbar_expect_tx(bar_g, tile_bytes);
      tma_tile(Qt, &tmg, b, h, c0, bar_g);
    }
    {
      float ov[32];
      umma::tmem_ld2x16(tO + col, ov);
      const float f = sh.pw[i + 1] * s_inv;
#pragma unroll
      for (int e = 0; e < 32; ++e) ov[e] *= f;
      umma::tmem_st32(tO + col, ov);
      rescale_quarter(SB, i, qd, s_inv, true);
      umma::tmem_wait_st();
    }
    umma::fence_async_smem();
    umma::fence_before();
    BWD_WAIT(bar_v, ph);
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // MMA3: O += Pm V
        umma::mma_ss(tm + 128, umma::desc_kmajor(aPM, kk, ROWS), umma::desc_mnmajor(aV, kk, ROWS), id_kmn, 1u);
      umma::commit(&sh.bar_mma[2]);
    }

    // [3] dgate and dO from O (output norm and gate backward): dgate -> PM,
    // dO -> Q over the gate (each thread rewrites only the chunks it read)
    BWD_WAIT(&sh.bar_mma[2], ph);
    BWD_WAIT(bar_g, ph);
    {
      float ov[32];
      umma::tmem_ld2x16(tO + col, ov);
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) ss = fmaf(ov[e], ov[e], ss);
      sh.red[qd][i] = ss;
      __syncthreads();
      const float ro = rsqrtf((sh.red[0][i] + sh.red[1][i] + sh.red[2][i] + sh.red[3][i]) / (float)D + P.eps);
      float mpart = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float gf[8], df[8], dg8[8];
        unpack8(*tile_at(Qt, i, 4 * qd + u), gf);
        unpack8(dyr[u], df);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float nv = ov[8 * u + e] * ro;
          const float z = sigmoid_fast(gf[e]);
          const float dn = df[e] * z;
          dg8[e] = dn * nv * (1.f - z);
          mpart = fmaf(dn, nv, mpart);
          ov[8 * u + e] = dn;  // keep dn; n is recomputed below
        }
        *tile_at(PM, i, 4 * qd + u) = pack8(dg8);
      }
      sh.red2[qd][i] = mpart;
      __syncthreads();
      const float mean = (sh.red2[0][i] + sh.red2[1][i] + sh.red2[2][i] + sh.red2[3][i]) / (float)D;
      // n = o ro again from TMEM (cheaper than holding both o and dn in registers)
      float o2[32];
      umma::tmem_ld2x16(tO + col, o2);
#pragma unroll
      for (int e = 0; e < 32; ++e) ov[e] = valid ? ro * (ov[e] - o2[e] * ro * mean) : 0.f;
      {  // v_i . do_i in fp32: do_i is orthogonal to o_i, so this nearly cancels
         // wherever o_i is close to a multiple of v_i, and bf16 do loses it
        float vd = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float vf[8];
          unpack8(*tile_at(Vt, i, 4 * qd + u), vf);
#pragma unroll
          for (int e = 0; e < 8; ++e) vd = fmaf(vf[e], ov[8 * u + e], vd);
        }
        sh.vd_diag[qd][i] = vd;
      }
      store_quarter(Qt, i, qd, ov);
    }
    umma::fence_async_smem();
    sync_tc();
    if (tid == 0) {
      tma_store_tile(&tmdg, PM, b, h, c0);
      tma_store_tile(&tmo, Qt, b, h, c0);
      umma::bulk_commit();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // MMA5: dP = dO V^T
        umma::mma_ss(tm, umma::desc_kmajor(aQ, kk, ROWS), umma::desc_kmajor(aV, kk, ROWS), id_kk, kk > 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // MMA6: I = dO S^T
        umma::mma_ss(tm + 256, umma::desc_kmajor(aQ, kk, ROWS), umma::desc_kmajor(aSB, kk, ROWS), id_kk, kk > 0);
      umma::commit(&sh.bar_mma[3]);
      umma::bulk_wait_read();  // dgate and dO have left PM and Q before [4] reuses them
    }

    // [4] dPm = bf16(dP (.) D) into PM (Pm is dead once MMA3 is done)
    BWD_WAIT(&sh.bar_mma[3], ph);

    if (tid == 0 && n + 1 < ntile) {  // the Q tile (dO) is free: next q
      umma::mbar_expect_tx(bar_q, tile_bytes);
      tma_tile(Qt, &tmq, b, h, c0 + CV, bar_q);
    }
    {
      float pv[32];
      const float vd = diag_sum(sh.vd_diag, i);
      if (qd == sub && valid) P.ddiag[((size_t)b * P.T + c0 + i) * P.H + h] = vd;
      mask_lower_block(tP + col, pv, i, sub, qd, valid, gm, sh.pw, true, vd);
      store_quarter(PM, i, qd, pv);
    }
    uint4 qraw[4];  // raw q pairs of row i for the dq epilogue (in flight during MMA7)
    load_pairs(qraw, row_ptr(P.q, P, b, h, valid ? c0 + i : c0), qd, valid);
    umma::fence_async_smem();
    sync_tc();
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // MMA7: O-columns <- dPm K~
        umma::mma_ss(tm + 128, umma::desc_kmajor(aPM, kk, ROWS), umma::desc_mnmajor(aK, kk, ROWS), id_kmn, kk > 0);
      umma::commit(&sh.bar_mma[4]);
    }

    // [5] k~dec (in place), MMA4 (state carry); dq epilogue overlaps MMA4
    BWD_WAIT(&sh.bar_mma[4], ph);
    rescale_quarter(Kt, i, qd, valid ? sh.pw[c - 1 - i] : 0.f, false);
    umma::fence_async_smem();
    sync_tc();
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // MMA4: S += K~dec^T V
        umma::mma_ss(tm + 384, umma::desc_mnmajor(aK, kk, ROWS), umma::desc_mnmajor(aV, kk, ROWS), id_mnmn, 1u);
      umma::commit(&sh.bar_mma[5]);
    }
    {
      // dQ~ = intra + gamma^{i+1} inter, for this thread's 16 RoPE pairs
      float alo[16], ahi[16];
      const float wi = sh.pw[i + 1];
      {
        float t[16];
        umma::tmem_ld16(tO + 16 * qd, alo);
        umma::tmem_ld16(tI + 16 * qd, t);
#pragma unroll
        for (int e = 0; e < 16; ++e) alo[e] = fmaf(wi, t[e], alo[e]);
        umma::tmem_ld16(tO + 64 + 16 * qd, ahi);
        umma::tmem_ld16(tI + 64 + 16 * qd, t);
#pragma unroll
        for (int e = 0; e < 16; ++e) ahi[e] = fmaf(wi, t[e], ahi[e]);
      }
      feature_grad_row(alo, ahi, qraw, rq, pos, i, qd, valid, sh.ru, sh.red, SB);  // S is dead
    }
    umma::fence_async_smem();
    BWD_WAIT(&sh.bar_mma[5], ph);
    if (tid == 0) {  // dq out; MMA4 done: V and this K buffer are free
      tma_store_tile(&tmdq, SB, b, h, c0);
      umma::bulk_commit();
      if (n + 1 < ntile) {
        umma::mbar_expect_tx(bar_v, tile_bytes);
        tma_tile(Vt, &tmv, b, h, c0 + CV, bar_v);
      }
      if (n + 2 < ntile) {
        umma::mbar_expect_tx(&bar_k[buf], tile_bytes);
        tma_tile(Kt, &tmk, b, h, c0 + 2 * CV, &bar_k[buf]);
      }
    }
  }
  if (tid == 0) umma::bulk_wait_all();
  if (failed && tid == 0 && P.err) atomicOr(P.err, 4u);
  sync_tc();
  if (warp == 0) umma::tmem_dealloc(tm, 512);
}

// ------------------------------------------------------------------ dk / dv pass

__global__ void __launch_bounds__(NT, 1)
    tc_bwd_dkdv_kernel(const __grid_constant__ MixerParams P, const __grid_constant__ CUtensorMap tmq,
                       const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                       const __grid_constant__ CUtensorMap tmo, const __grid_constant__ CUtensorMap tmdk,
                       const __grid_constant__ CUtensorMap tmdv) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  // Q: raw q -> q~ (fp16) -> q~ (bf16) -> q~w.  K: raw k -> k~ (fp16) -> k~dec,
  // then dv (TMA-stored).  V: v -> vdec, then dk (TMA-stored).  DO: do.
  // EB: E (bf16).  X: M1 (.) D^T, then M2 (.) D^T.
  unsigned char *Qt = base, *Kt = base + TILE, *Vt = base + 2 * TILE, *DOt = base + 3 * TILE;
  unsigned char *EB = base + 4 * TILE, *X = base + 5 * TILE;
  BwdShared &sh = *reinterpret_cast<BwdShared *>(base + 6 * TILE);
  uint64_t *bar_q = &sh.bar_tma[0], *bar_k = &sh.bar_tma[1], *bar_v = &sh.bar_tma[2],
           *bar_do = &sh.bar_tma[3];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sub = warp & 3, qd = warp >> 2, i = 32 * sub + lane;
  const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int t0 = g * P.seg_len, t1 = min(P.T, t0 + P.seg_len);
  const int CV = P.chunk;
  const int ntile = ceil_div(t1 - t0, CV);
  const float gm = P.gamma[h];
  const float l2g = log2f(gm);
  const uint32_t tile_bytes = (uint32_t)CV * D * 2;

  if (tid == 0) {
    for (int j = 0; j < 5; ++j) umma::mbar_init(&sh.bar_tma[j], 1);
    for (int j = 0; j < 6; ++j) umma::mbar_init(&sh.bar_mma[j], 1);
    umma::mbar_fence_init();
  }
  if (tid <= ROWS) sh.pw[tid] = exp2f((float)tid * l2g);
  load_rope_table(sh.ru, P, tid);
  if (warp == 0) umma::tmem_alloc(&sh.tmem_base, 512);
  if (CV < ROWS)  // rows [CV, 128) of V and DO are never written by TMA: clear them once
    for (int e = tid; e < 2 * (ROWS - CV) * 16; e += NT) {
      const int r = e % ((ROWS - CV) * 16);
      *tile_at(e < (ROWS - CV) * 16 ? Vt : DOt, CV + r / 16, r % 16) = make_uint4(0, 0, 0, 0);
    }
  sync_tc();
  const uint32_t tm = sh.tmem_base;
  const uint32_t lb = (uint32_t)(32 * sub) << 16, col = 32 * qd;
  const uint32_t tA = tm + lb, tB = tm + 128 + lb, tE = tm + 256 + lb;
  {  // gradient reaching the segment's last state from later tokens -> TMEM
    const float *ein = P.seg2 + (((size_t)b * P.H + h) * P.nseg + g) * (size_t)D * D;
    const float4 *s4 = reinterpret_cast<const float4 *>(ein + (size_t)i * D + col);
    float v[32];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float4 x = s4[u];
      v[4 * u] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
    }
    umma::tmem_st32(tE + col, v);
    umma::tmem_wait_st();
  }
  if (tid == 0) {
    const int cl = t0 + (ntile - 1) * CV;
    umma::mbar_expect_tx(bar_q, tile_bytes);
    tma_tile(Qt, &tmq, b, h, cl, bar_q);
    umma::mbar_expect_tx(bar_k, tile_bytes);
    tma_tile(Kt, &tmk, b, h, cl, bar_k);
    umma::mbar_expect_tx(bar_v, tile_bytes);
    tma_tile(Vt, &tmv, b, h, cl, bar_v);
    umma::mbar_expect_tx(bar_do, tile_bytes);
    tma_tile(DOt, &tmo, b, h, cl, bar_do);
  }
  const uint32_t id_kq16 = umma::idesc_bf16(128, 128, false, false, true);
  const uint32_t id_kmn = umma::idesc_bf16(128, 128, false, true);
  const uint32_t id_kk = umma::idesc_bf16(128, 128, false, false);
  const uint32_t id_mnmn = umma::idesc_bf16(128, 128, true, true);
  const uint32_t aQ = umma::smem_u32(Qt), aK = umma::smem_u32(Kt), aV = umma::smem_u32(Vt),
                 aDO = umma::smem_u32(DOt), aE = umma::smem_u32(EB), aX = umma::smem_u32(X);

  bool failed = false;
  for (int it = 0; it < ntile; ++it) {
    const int n = ntile - 1 - it;
    const uint32_t ph = it & 1;
    const int c0 = t0 + n * CV, c = min(CV, t1 - c0);
    const bool valid = i < c;
    const long long pos = P.pos_offset + c0 + i;
    const float wdec = valid ? sh.pw[c - 1 - i] : 0.f;

    // [1] q~, k~ (fp16, in place); EB = bf16(E); E <- gamma^c E
    BWD_WAIT(bar_q, ph);
    BWD_WAIT(bar_k, ph);
    float rk;
    {
      uint4 qr[4], kr[4];
      ld_pairs(Qt, i, qd, qr);
      ld_pairs(Kt, i, qd, kr);
      if (!valid) qr[0] = qr[1] = qr[2] = qr[3] = kr[0] = kr[1] = kr[2] = kr[3] = make_uint4(0, 0, 0, 0);
      sh.red[qd][i] = sumsq_pairs(qr);
      sh.red2[qd][i] = sumsq_pairs(kr);
      float ev[32];
      umma::tmem_ld2x16(tE + col, ev);
      store_quarter(EB, i, qd, ev);
      const float carry = sh.pw[c];
#pragma unroll
      for (int e = 0; e < 32; ++e) ev[e] *= carry;
      umma::tmem_st32(tE + col, ev);
      __syncthreads();
      const float rq = rsqrtf((sh.red[0][i] + sh.red[1][i] + sh.red[2][i] + sh.red[3][i]) / (float)D + P.eps);
      rk = rsqrtf((sh.red2[0][i] + sh.red2[1][i] + sh.red2[2][i] + sh.red2[3][i]) / (float)D + P.eps);
      sh.qk_diag[qd][i] = feature_qk_store(qr, kr, rq, rk * P.kscale, pos, qd, sh.ru, Qt, Kt, i);
      umma::tmem_wait_st();
    }
    umma::fence_async_smem();
    umma::fence_before();
    BWD_WAIT(bar_v, ph);
    BWD_WAIT(bar_do, ph);
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // M1 = K~ Q~^T (fp16)
        umma::mma_ss(tm, umma::desc_kmajor(aK, kk, ROWS), umma::desc_kmajor(aQ, kk, ROWS), id_kq16, kk > 0);
      umma::commit(&sh.bar_mma[0]);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // M2 = V dO^T
        umma::mma_ss(tm + 128, umma::desc_kmajor(aV, kk, ROWS), umma::desc_kmajor(aDO, kk, ROWS), id_kk, kk > 0);
      umma::commit(&sh.bar_mma[1]);
    }

    // [2] X = bf16(M1 (.) D^T); k~ -> k~dec
    BWD_WAIT(&sh.bar_mma[0], ph);
    {
      float v[32];
      mask_upper_block(tA + col, v, i, sub, qd, c, valid, gm, sh.pw, true,
                       diag_sum(sh.qk_diag, i));  // fp32 k~_i . q~_i on the diagonal
      store_quarter(X, i, qd, v);
      rescale_quarter(Kt, i, qd, wdec, true);
    }
    umma::fence_async_smem();
    sync_tc();
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // dV = X dO
        umma::mma_ss(tm, umma::desc_kmajor(aX, kk, ROWS), umma::desc_mnmajor(aDO, kk, ROWS), id_kmn, kk > 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // dV += K~dec E
        umma::mma_ss(tm, umma::desc_kmajor(aK, kk, ROWS), umma::desc_mnmajor(aE, kk, ROWS), id_kmn, 1u);
      umma::commit(&sh.bar_mma[2]);
    }

    // [3] M2 (.) D^T (held in registers until X is free); v -> vdec; q~ -> bf16
    BWD_WAIT(&sh.bar_mma[1], ph);
    uint4 kraw[4];  // raw k pairs of row i for the dk epilogue
    load_pairs(kraw, row_ptr(P.k, P, b, h, valid ? c0 + i : c0), qd, valid);
    {
      float v[32];
      // fp32 v_i . do_i on the diagonal, kept by the dq pass
      const float vd = (qd == sub && valid) ? P.ddiag[((size_t)b * P.T + c0 + i) * P.H + h] : 0.f;
      mask_upper_block(tB + col, v, i, sub, qd, c, valid, gm, sh.pw, true, vd);
      rescale_quarter(Vt, i, qd, wdec, false);
      rescale_quarter(Qt, i, qd, 1.f, true);
      BWD_WAIT(&sh.bar_mma[2], ph);  // dV done: X and K are free
      store_quarter(X, i, qd, v);
    }
    {  // dv of this tile (dV is complete) -> K, for a TMA store
      float v[32];
      umma::tmem_ld2x16(tA + col, v);
      store_quarter(Kt, i, qd, v);
    }
    umma::fence_async_smem();
    sync_tc();
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // dK~ = X Q~
        umma::mma_ss(tm + 128, umma::desc_kmajor(aX, kk, ROWS), umma::desc_mnmajor(aQ, kk, ROWS), id_kmn, kk > 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // dK~ += V~dec E^T
        umma::mma_ss(tm + 128, umma::desc_kmajor(aV, kk, ROWS), umma::desc_kmajor(aE, kk, ROWS), id_kk, 1u);
      umma::commit(&sh.bar_mma[3]);
      tma_store_tile(&tmdv, Kt, b, h, c0);
      umma::bulk_commit();
    }

    // [4] q~ -> q~w = gamma^{i+1} q~; E += q~w^T dO; dk epilogue overlaps it
    BWD_WAIT(&sh.bar_mma[3], ph);
    rescale_quarter(Qt, i, qd, sh.pw[i + 1], false);
    umma::fence_async_smem();
    sync_tc();
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // E += Q~w^T dO
        umma::mma_ss(tm + 256, umma::desc_mnmajor(aQ, kk, ROWS), umma::desc_mnmajor(aDO, kk, ROWS), id_mnmn, 1u);
      umma::commit(&sh.bar_mma[4]);
      umma::bulk_wait_read();  // dv has left K
      if (n > 0) {
        umma::mbar_expect_tx(bar_k, tile_bytes);
        tma_tile(Kt, &tmk, b, h, c0 - CV, bar_k);
      }
    }
    {
      float glo[16], ghi[16];
      tmem_ld_pairs(tB, qd, glo, ghi);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        glo[e] *= P.kscale;
        ghi[e] *= P.kscale;
      }
      feature_grad_row(glo, ghi, kraw, rk, pos, i, qd, valid, sh.ru, sh.red, Vt);  // v~dec is dead
    }
    umma::fence_async_smem();
    BWD_WAIT(&sh.bar_mma[4], ph);
    if (tid == 0) {  // E update done: Q and DO are free; dk out, then V is free
      if (n > 0) {
        umma::mbar_expect_tx(bar_q, tile_bytes);
        tma_tile(Qt, &tmq, b, h, c0 - CV, bar_q);
        umma::mbar_expect_tx(bar_do, tile_bytes);
        tma_tile(DOt, &tmo, b, h, c0 - CV, bar_do);
      }
      tma_store_tile(&tmdk, Vt, b, h, c0);
      umma::bulk_commit();
      umma::bulk_wait_read();
      if (n > 0) {
        umma::mbar_expect_tx(bar_v, tile_bytes);
        tma_tile(Vt, &tmv, b, h, c0 - CV, bar_v);
      }
    }
  }
  if (tid == 0) umma::bulk_wait_all();
  if (failed && tid == 0 && P.err) atomicOr(P.err, 8u);
  sync_tc();
  if (warp == 0) umma::tmem_dealloc(tm, 512);
}

#undef BWD_WAIT

constexpr size_t kBwdSmem = 6 * TILE + sizeof(BwdShared) + 1024;

}  // namespace
}  // namespace tc

cudaError_t launch_tc_bwd_dq(const MixerParams &P, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mg, mo, mdg, mdq;
  cudaError_t e;
  if ((e = tc::make_map(&mq, P.q, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mk, P.k, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mv, P.v, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mg, P.g, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mo, P.dO, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mdg, P.dg, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mdq, P.dq, P, P.chunk)) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc::tc_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)tc::kBwdSmem);
  if (e != cudaSuccess) return e;
  tc::tc_bwd_dq_kernel<<<dim3(P.nseg, P.H, P.B), tc::NT, tc::kBwdSmem, st>>>(P, mq, mk, mv, mg, mo, mdg, mdq);
  return cudaGetLastError();
}

cudaError_t launch_tc_bwd_dkdv(const MixerParams &P, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mo, mdk, mdv;
  cudaError_t e;
  if ((e = tc::make_map(&mq, P.q, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mk, P.k, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mv, P.v, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mo, P.dO, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mdk, P.dk, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mdv, P.dv, P, P.chunk)) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc::tc_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)tc::kBwdSmem);
  if (e != cudaSuccess) return e;
  tc::tc_bwd_dkdv_kernel<<<dim3(P.nseg, P.H, P.B), tc::NT, tc::kBwdSmem, st>>>(P, mq, mk, mv, mo, mdk, mdv);
  return cudaGetLastError();
}

}  // namespace hla
