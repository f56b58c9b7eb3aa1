// tc_prefill.cu — tensor-core (tcgen05) prefill for bf16 inputs at d = 128.
//
// The chunked form of Eq. 18 (arXiv 2601.22156, Appendix A): for a tile of
// c <= 128 tokens entering with state S,
//   P     = Q~ K~^T                                  MMA1  (M=128, N=128, K=d)
//   O     = Q~ S                                     MMA2  (K = d_k)
//   O    <- diag(gamma^{i+1}) O  (in TMEM), then
//   O    += (P (.) D) V,   D_ij = gamma^{i-j}, i >= j MMA3
//   S    <- gamma^c S + (diag(gamma^{c-1-j}) K~)^T V  MMA4  (accumulated onto S in TMEM)
//   y_i   = Norm(o_i) * sigmoid(gate_i)
// Accumulators live in the 512 columns of tensor memory: P, two O buffers
// (tile n accumulates while tile n - 1 drains) and the fp32 state S.
// Operands are 16-bit tiles in shared memory in the 128-byte-swizzled layout
// of umma.cuh.  Raw q, k and v tiles arrive by TMA straight into the operand
// buffers and are transformed in place (q -> q~, k -> k~ -> k~dec), so no
// register ever waits on a global load.
//
// Precision: Q~, K~ and S enter MMA1/MMA2 as fp16 (11-bit significand).  With
// bf16 there, the rounding of q~ . k~ dominates the error of y wherever o
// nearly cancels (fast-decaying heads); fp16 cuts that fourfold.  S is scaled
// by a power of two into fp16 range each tile and the scale is undone on O.
// P (.) D, K~dec and V stay bf16 (V is a bf16 input; MMA3/MMA4 run bf16).
//
// Threads: both kernels run CTAs of 640 threads (NTO), warp-specialized: 16
// worker warps (0..15) own the CUDA-core phases and one issuer warpgroup
// (warps 16..19), whose first lane issues every TMA copy and MMA; workers and
// issuer hand each phase over through mbarriers.  In the phases that touch
// TMEM, worker thread (warp w, lane l) owns tile row i = 32 (w % 4) + l and
// column quarter qd = w / 4, which is also the TMEM lane and column block that
// warp may access; the feature map uses row 8 w + l / 4 and pair quarter l % 4.
//
//   tc_state_kernel:  one CTA per piece of a segment's local state, the sum
//                     over its tokens of gamma^{end-s} k~_s^T v_s, one MMA per
//                     tile accumulated in TMEM (the decay weight of each key
//                     row is folded into K~); also, for the backward, the
//                     mirror sum of q~^T do.
//   tc_output_kernel: one CTA per (b, h, segment): the outputs of the segment
//                     from the entering state written by the fp32 scan
//                     (scan.cu).
#include "tc_common.cuh"

namespace hla {
namespace tc {

namespace {

// ------------------------------------------------------------------ local state pass

constexpr int kStages = 3;             // (k, v) tile pairs of the local-state pass in flight

struct StateShared {
  unsigned long long ru[kMaxPairs];  // RoPE phase increments (load_rope_table)
  uint64_t bar_tma[kStages];   // TMA of the (k, v) pair in stage j
  uint64_t bar_feat[kStages];  // workers: k~dec of stage j written (one arrive per warp)
  uint64_t bar_mma[kStages];   // MMA of stage j done (commit)
  uint32_t tmem_base;
  uint32_t failed;
};

// kGrad = false: Delta_seg = sum_s gamma^{end-s} k~_s^T v_s   (k~ = RoPE(Norm(k)) / sqrt(d))
// kGrad = true:  DeltaG_seg = sum_s gamma^{s-start+1} q~_s^T do_s, the backward's
//                per-segment state gradient (q~ = RoPE(Norm(q)), do a bf16 tensor);
//                tmk then maps q and tmv maps do.
// One CTA per piece of a segment (piece_tiles): only the tiles within the
// decay horizon decay_rows() are read (the weights beyond it sum to at most
// 2^-40), cut into pieces of at most kPieceTiles, and each piece's sum goes to
// its own slot of P.part.
// Warp-specialized: 16 worker warps turn raw k rows into decay-weighted k~
// in place (row norms from the four lanes that share a row); the issuer warp
// issues one MMA per tile as soon as the workers are done with it and refills
// the stage once that MMA has read it, three tiles ahead.  Workers never wait
// for the tensor core.
// kSaved: tmk maps saved fp16 features (q~ of the forward, with kGrad; k~
// given to hla_prefill_features, without), so the workers only weight them
// and convert them to bf16 (the MMA's type, that of do or v).
template <bool kGrad, bool kSaved = false>
__global__ void __launch_bounds__(NTO, 1)
    tc_state_kernel(const __grid_constant__ MixerParams P, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  // stage j: K at base + 2 j TILE, V at base + (2 j + 1) TILE
  StateShared &sh = *reinterpret_cast<StateShared *>(base + 2 * kStages * TILE);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int np = P.npart > 1 ? P.npart : 1;
  // heads in reverse launch order: under the paper's schedule gamma_h grows with
  // h, so the slowest-decaying heads, whose pieces are the longest, start first
  const int g = P.state_seg0 + blockIdx.x / np, piece = blockIdx.x % np;
  const int h = P.H - 1 - blockIdx.y, b = blockIdx.z;
  const int t0 = g * P.seg_len, t1 = min(P.T, t0 + P.seg_len);
  const int CV = P.chunk;
  const int L = t1 - t0;
  const float l2g = log2f(P.gamma[h]);
  int lo, hi;
  piece_tiles(decay_rows(l2g), L, CV, piece, kGrad, lo, hi);
  float *out = P.part ? P.part + ((((size_t)b * P.H + h) * P.nseg + g) * P.npart + piece) * (size_t)D * D
                      : (kGrad ? P.seg2 : P.seg) + (((size_t)b * P.H + h) * P.nseg + g) * (size_t)D * D;
  if (lo >= hi) {  // nothing within the decay horizon (uniform: the CTA leaves before any barrier)
    if (!P.part)   // the segment's only piece: its sum is zero
      for (int e = threadIdx.x; e < D * D; e += NTO) out[e] = 0.f;
    return;
  }
  const int ntile = hi - lo;       // tiles of this piece
  const int tb = t0 + lo * CV;     // its first token
  const uint32_t tile_bytes = (uint32_t)CV * D * 2;

  if (tid == 0) {
    for (int j = 0; j < kStages; ++j) {
      umma::mbar_init(&sh.bar_tma[j], 1);
      umma::mbar_init(&sh.bar_feat[j], NWORK);
      umma::mbar_init(&sh.bar_mma[j], 1);
    }
    umma::mbar_fence_init();
    sh.failed = 0;
  }
  load_rope_table(sh.ru, P, tid);
  if (warp == 0) umma::tmem_alloc(&sh.tmem_base, 128);
  // rows [CV, 128) of the V buffers are never written by TMA: clear them once
  if (CV < ROWS)
    for (int e = tid; e < kStages * (ROWS - CV) * 16; e += NTO) {
      const int j = e / ((ROWS - CV) * 16), r = e % ((ROWS - CV) * 16);
      *tile_at(base + (2 * j + 1) * TILE, CV + r / 16, r % 16) = make_uint4(0, 0, 0, 0);
    }
  sync_tc();
  const uint32_t tm = sh.tmem_base;
  bool failed = false;

  if (warp >= NWORK) {
    // ---------------------------------------------------------------- issuer
    if (warp == NWORK && lane == 0) {
      const uint32_t idesc = umma::idesc_bf16(128, 128, true, true);
      for (int n = 0; n < kStages && n < ntile; ++n) {
        umma::mbar_expect_tx(&sh.bar_tma[n], 2 * tile_bytes);
        tma_tile(base + 2 * n * TILE, &tmk, b, h, tb + n * CV, &sh.bar_tma[n]);
        tma_tile(base + (2 * n + 1) * TILE, &tmv, b, h, tb + n * CV, &sh.bar_tma[n]);
      }
      for (int n = 0; n < ntile; ++n) {
        const int st = n % kStages;
        const uint32_t par = (n / kStages) & 1;
        unsigned char *Kt = base + 2 * st * TILE;
        wait_plain(&sh.bar_feat[st], par, failed);
        if (!failed) {
          umma::fence_after();
          const uint32_t a = umma::smem_u32(Kt), bv = a + TILE;
#pragma unroll
          for (int kk = 0; kk < ROWS / 16; ++kk)
            umma::mma_ss(tm, umma::desc_mnmajor(a, kk, ROWS), umma::desc_mnmajor(bv, kk, ROWS), idesc,
                         (n > 0 || kk > 0) ? 1u : 0u);
          umma::commit(&sh.bar_mma[st]);
        }
        if (n + kStages < ntile) {  // the stage takes tile n + 3 once MMA n has read it
          wait_plain(&sh.bar_mma[st], par, failed);
          if (!failed) {
            const int cn = tb + (n + kStages) * CV;
            umma::mbar_expect_tx(&sh.bar_tma[st], 2 * tile_bytes);
            tma_tile(Kt, &tmk, b, h, cn, &sh.bar_tma[st]);
            tma_tile(Kt + TILE, &tmv, b, h, cn, &sh.bar_tma[st]);
          }
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- workers
    const int fr = 8 * warp + (lane >> 2), fu = lane & 3;  // row, pair quarter
    const float scale = kGrad ? 1.f : P.kscale;
    for (int n = 0; n < ntile; ++n) {
      const int st = n % kStages;
      unsigned char *Kt = base + 2 * st * TILE;
      const int c0 = tb + n * CV, c = min(CV, t1 - c0);
      wait_plain(&sh.bar_tma[st], (n / kStages) & 1, failed);
      const bool valid = fr < c;
      if (kSaved) {  // q~ -> gamma^{s+1} q~ or k~ -> gamma^{L-1-s} k~ (fp16 -> bf16) in
                     // place; zeros past the tile
        const int s_rel = c0 - t0 + fr;
        const f2 w = dup2(exp2f((float)(kGrad ? s_rel + 1 : L - 1 - s_rel) * l2g));
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint4 *p = tile_at(Kt, fr, (u < 2 ? 0 : 8) + 2 * fu + (u & 1));
          f2 f[4];
          unpack4x2h(*p, f);
#pragma unroll
          for (int e = 0; e < 4; ++e) f[e] = mul2(f[e], w);
          *p = valid ? pack4x2(f) : make_uint4(0, 0, 0, 0);
        }
        warp_arrive(&sh.bar_feat[st], lane);
        continue;
      }
      uint4 kr[4];
      ld_pairs(Kt, fr, fu, kr);
      if (!valid)  // rows past the tile hold stale bytes: use zeros
        kr[0] = kr[1] = kr[2] = kr[3] = make_uint4(0, 0, 0, 0);
      float sk = sumsq_pairs(kr);
      sk += __shfl_xor_sync(0xffffffffu, sk, 1);
      sk += __shfl_xor_sync(0xffffffffu, sk, 2);
      const float rk = rsqrtf(sk / (float)D + P.eps);
      // decay weight of this row towards the end (forward) or from the start
      // (gradient) of the segment; 0 past the tile
      const int s_rel = c0 - t0 + fr;
      const float wgt = valid ? exp2f((float)(kGrad ? s_rel + 1 : L - 1 - s_rel) * l2g) : 0.f;
      feature_store(kr, rk * scale * wgt, P.pos_offset + c0 + fr, fu, sh.ru, Kt, fr, false);
      warp_arrive(&sh.bar_feat[st], lane);
    }
  }
  // the last MMA's completion covers all earlier ones
  {
    const int nl = ntile - 1;
    if (!failed && !umma::mbar_wait(&sh.bar_mma[nl % kStages], (nl / kStages) & 1)) failed = true;
    umma::fence_after();
    if (failed) atomicOr(&sh.failed, 1u);
  }
  sync_tc();
  if (warp < NWORK) {
    const int sub = warp & 3, qd = warp >> 2, i = 32 * sub + lane;
    if (!sh.failed) {
      float v[32];
      umma::tmem_ld32(tm + ((uint32_t)(32 * sub) << 16) + 32 * qd, v);
      float4 *o4 = reinterpret_cast<float4 *>(out + (size_t)i * D + 32 * qd);
#pragma unroll
      for (int u = 0; u < 8; ++u) o4[u] = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
    } else {
      const float nan = __int_as_float(0x7fc00000);
      for (int e = tid; e < D * D; e += NWORK * 32) out[e] = nan;
      if (tid == 0 && P.err) atomicOr(P.err, 1u);
    }
  }
  sync_tc();
  if (warp == 0) umma::tmem_dealloc(tm, 128);
}

// ------------------------------------------------------------------ output pass

struct OutShared {
  RopeTab rope_small[8];             // RoPE angles of the offsets 0..7 (fill_rope_small)
  RopeTab rope_base[NWORK];          // per worker warp: angles at its first feature row
  unsigned long long ru[kMaxPairs];  // RoPE phase increments (load_rope_table)
  float red_o[4][ROWS];
  float pw[ROWS + 1];
  alignas(16) float dm[4][DM_STRIDE];  // causal-mask decay table (fill_mask_table)
  float qk_diag[2][ROWS];  // fp32 q~_i . k~_i of tiles n (n & 1)
  float smax[NWORK];
  uint64_t bar_mma[2];  // [0]: MMA1 + MMA2 of a tile done, [1]: MMA3 + MMA4 done (commits)
  uint64_t bar_p;       // MMA1 (P) of a tile done
  uint64_t bar_q;       // TMA of raw q
  uint64_t bar_k[2];    // TMA of raw k into buffer 0 / 1
  uint64_t bar_v;       // TMA of raw v
  uint64_t bar_g;       // TMA of the gate tile
  uint64_t bar_feat;    // workers: q~, k~ of the tile written (one arrive per warp)
  uint64_t bar_sb;      // workers: Sb written and S rescaled
  uint64_t bar_pm;      // workers: Pm, scaled O and k~dec written
  uint64_t bar_epi;     // workers: y of the previous tile written over its gate tile
  uint64_t bar_sv;      // saving: the TMA stores of q~, k~ have read Q and K (issuer)
  uint64_t bar_wtma[3];   // one launch: TMA of the (k, v) window tile in stage j
  uint64_t bar_wfeat[3];  // one launch: workers wrote k~dec of stage j (one arrive per warp)
  uint64_t bar_wmma[3];   // one launch: MMA of stage j done (commit)
  uint64_t bar_wdone;     // one launch: every window MMA done (commit)
  uint64_t bar_drain;     // after a wait gave up: every MMA the issuer issued is done (commit)
  uint32_t tmem_base;
  uint32_t failed;
};


// ------------------------------------------------------------------ one launch: the window phase
// The state entering a segment, formed by its own output CTA (kWin below):
// gamma^t0 state_in, plus S += K~dec^T V over the window_tiles() tiles before
// t0, with three (k, v) stages in flight over the six tile buffers.  Kept out
// of line (one call per CTA) so that the tile loop's registers are allocated
// as in the other variants.  Both return whether a bounded wait gave up.

// Issuer side: copies and one MMA per window tile into S (tS).
__device__ __noinline__ bool window_issue(const CUtensorMap &tmk, const CUtensorMap &tmv, OutShared &sh,
                                          unsigned char *base, uint32_t tS, int b, int h, int t0,
                                          int CV, float l2g) {
  bool failed = false;
  const uint32_t tile_bytes = (uint32_t)CV * D * 2;
  const uint32_t id_mn = umma::idesc_bf16(128, 128, true, true);  // bf16 K~dec^T V
  const int nw = window_tiles(l2g, t0, CV), ws = t0 - nw * CV;
  int armed[3] = {0, 0, 0};  // copies issued per stage (each stage has at most one in flight)
  for (int w = 0; w < 3 && w < nw; ++w) {
    umma::mbar_expect_tx(&sh.bar_wtma[w], 2 * tile_bytes);
    tma_tile(base + 2 * w * TILE, &tmk, b, h, ws + w * CV, &sh.bar_wtma[w]);
    tma_tile(base + (2 * w + 1) * TILE, &tmv, b, h, ws + w * CV, &sh.bar_wtma[w]);
    ++armed[w];
  }
  for (int w = 0; w < nw; ++w) {
    const int st = w % 3;
    const uint32_t par = (w / 3) & 1;
    unsigned char *Kw = base + 2 * st * TILE;
    wait_plain(&sh.bar_wfeat[st], par, failed);
    if (!failed) {
      umma::fence_after();
      const uint32_t a = umma::smem_u32(Kw), bv = a + TILE;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma::mma_ss(tS, umma::desc_mnmajor(a, kk, ROWS), umma::desc_mnmajor(bv, kk, ROWS), id_mn, 1u);
      umma::commit(&sh.bar_wmma[st]);
    }
    if (w + 3 < nw) {  // the stage takes tile w + 3 once MMA w has read it
      wait_plain(&sh.bar_wmma[st], par, failed);
      if (!failed) {
        umma::mbar_expect_tx(&sh.bar_wtma[st], 2 * tile_bytes);
        tma_tile(Kw, &tmk, b, h, ws + (w + 3) * CV, &sh.bar_wtma[st]);
        tma_tile(Kw + TILE, &tmv, b, h, ws + (w + 3) * CV, &sh.bar_wtma[st]);
        ++armed[st];
      }
    }
  }
  if (nw > 0) {
    // every window MMA done before the buffers take the tile loop's copies (the
    // commit covers whatever was issued, also after a wait gave up)
    umma::commit(&sh.bar_wdone);
    if (!umma::mbar_wait(&sh.bar_wdone, 0)) failed = true;
    umma::fence_after();
    // after a wait gave up, every copy issued lands before anything else
    // reuses the stage buffers (the normal budget; copies complete on their own)
    if (failed)
      for (int st = 0; st < 3; ++st)
        if (armed[st]) umma::mbar_wait(&sh.bar_wtma[st], (armed[st] - 1) & 1);
  }
  return failed;
}

// Worker side: gamma^t0 state_in into S (TMEM), each window tile's raw k (or
// given fp16 k~, kFeat) turned into K~dec in place with weights
// gamma^{t0-1-s}, and, once every window MMA is done, the entering state out
// to seg_in (row i, columns [col, col + 32)), where the backward can read it.
template <bool kFeat>
__device__ __noinline__ bool window_work(const MixerParams &P, OutShared &sh, unsigned char *base,
                                         uint32_t myS, float *seg_in, int b, int h, int t0, int CV,
                                         float l2g, int i, uint32_t col, int warp, int lane) {
  bool failed = false;
  const int fr = 8 * warp + (lane >> 2), fu = lane & 3;  // feature map: row, pair quarter
  {
    const float w0 = exp2f((float)t0 * l2g);
    float v[32];
    if (P.state_in && w0 > 0.f) {
      const float4 *s4 =
          reinterpret_cast<const float4 *>(P.state_in + (((size_t)b * P.H + h) * D + i) * D + col);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 x = s4[u];
        v[4 * u] = w0 * x.x; v[4 * u + 1] = w0 * x.y; v[4 * u + 2] = w0 * x.z; v[4 * u + 3] = w0 * x.w;
      }
    } else {
#pragma unroll
      for (int u = 0; u < 32; ++u) v[u] = 0.f;
    }
    umma::tmem_st32(myS, v);
    umma::tmem_wait_st();
  }
  const int nw = window_tiles(l2g, t0, CV), ws = t0 - nw * CV;
  const bool wvalid = fr < CV;  // window tiles are always full
  for (int w = 0; w < nw; ++w) {
    const int st = w % 3;
    unsigned char *Kw = base + 2 * st * TILE;
    wait_plain(&sh.bar_wtma[st], (w / 3) & 1, failed);
    const int s_tok = ws + w * CV + fr;
    const float wgt = wvalid ? exp2f((float)(t0 - 1 - s_tok) * l2g) : 0.f;
    if (kFeat) {  // given k~ (fp16): weight and convert
      const f2 wk = dup2(wgt);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint4 *pk = tile_at(Kw, fr, (u < 2 ? 0 : 8) + 2 * fu + (u & 1));
        f2 f[4];
        unpack4x2h(*pk, f);
#pragma unroll
        for (int e = 0; e < 4; ++e) f[e] = mul2(f[e], wk);
        *pk = wvalid ? pack4x2(f) : make_uint4(0, 0, 0, 0);
      }
    } else {
      uint4 kr[4];
      ld_pairs(Kw, fr, fu, kr);
      if (!wvalid) kr[0] = kr[1] = kr[2] = kr[3] = make_uint4(0, 0, 0, 0);
      float sk = sumsq_pairs(kr);
      sk += __shfl_xor_sync(0xffffffffu, sk, 1);
      sk += __shfl_xor_sync(0xffffffffu, sk, 2);
      const float rk = rsqrtf(sk / (float)D + P.eps);
      feature_store(kr, rk * P.kscale * wgt, P.pos_offset + s_tok, fu, sh.ru, Kw, fr, false);
    }
    warp_arrive(&sh.bar_wfeat[st], lane);
  }
  if (nw > 0) wait_or_fail(&sh.bar_wdone, 0, failed);
  float v[32];
  umma::tmem_ld2x16(myS, v);
  float4 *o4 = reinterpret_cast<float4 *>(seg_in + (size_t)i * D + col);
#pragma unroll
  for (int u = 0; u < 8; ++u) o4[u] = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
  return failed;
}

// Output pass over the tiles of one segment, warp-specialized.
//   Issuer warp (warp 16): per tile n, waits for the workers' barriers and
//   issues MMA1 (P = Q~ K~^T), MMA2 (O = Q~ Sb), MMA3 (O += Pm V) and MMA4
//   (S += K~dec^T V), the TMA store of y of tile n - 1 (written over its gate
//   tile by the workers) and the TMA copies that refill the freed buffers.
//   Every global access of the tile loop is a TMA bulk copy.
//   Worker warps (0..15), per tile n:
//     [A]/[D] raw q, k -> row norms (warp shuffles) -> q~, k~ fp16 in place
//     [B]/[C] after MMA3/MMA4 of tile n - 1: Sb = fp16(S 2^-e) with one power
//             of two per column quarter, S <- gamma^c S
//     [F]     after MMA1/MMA2: mask P -> Pm, O <- gamma^{i+1} 2^e O, k~ -> k~dec
//     [E]     epilogue of tile n - 1, while MMA3/MMA4 of tile n run and q of
//             tile n + 1 is copied into the Q buffer MMA2 has just freed; when
//             saving or given the features (kEpiFirst) it runs before [F]
//             instead, right after [C], and the issuer stores y of tile n - 1
//             before it waits for [F]
// The only CTA-wide barriers are outside the tile loop; the two reductions
// (max |S| per column quarter, the RMS of o per row) use 4-warp named barriers.
// kSave: the features are also saved for the backward.  Once q~, k~ of a tile
// are in place the issuer stores both tiles by TMA (fp16 maps tmsq / tmsk)
// and, when the stores have read them, lets the workers turn k~ into k~dec
// (bar_sv); the [A]/[D] warps write 1/RMS(q), 1/RMS(k) and q~_i . k~_i.
// kFeat (hla_prefill_features): tmq / tmk map given fp16 q~ and k~ (the saved
// layout), so [A]/[D] are skipped: MMA1 waits for their copies, and the
// diagonal warps load q~_i . k~_i from the saved scalars by cp.async into the
// qk_diag slot only they read.
// kWin (the prefill in one launch): the CTA forms the state entering its
// segment itself instead of reading it from the scan: gamma^t0 state_in, plus
// the window of window_tiles() tiles before t0, each (k, v) tile turned into
// K~dec by the workers (weights gamma^{t0-1-s}) and accumulated into S in TMEM
// by one MMA, through three (k, v) stages over the six tile buffers before the
// tile loop takes them.  Tokens before the window carry weights that sum to at
// most 2^-40 (decay_rows).  No CTA waits for another; the entering state is
// also written to P.seg, where the backward can read it.
template <bool kSave, bool kFeat = false, bool kWin = false>
__global__ void __launch_bounds__(NTO, 1)
    tc_output_kernel(const __grid_constant__ MixerParams P, const __grid_constant__ CUtensorMap tmq,
                     const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ CUtensorMap tmg, const __grid_constant__ CUtensorMap tmy,
                     const __grid_constant__ CUtensorMap tmsq, const __grid_constant__ CUtensorMap tmsk) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  // Q: raw q -> q~ (free once MMA2 has read it: the next q lands there).
  // K buffer j at base + (1 + j) TILE: raw k -> k~ -> k~dec (double-buffered).
  // G: gate of the tile being drained -> its y, stored from there by TMA.
  unsigned char *Qs = base, *Vs = base + 3 * TILE, *SP = base + 4 * TILE, *Gs = base + 5 * TILE;
  OutShared &sh = *reinterpret_cast<OutShared *>(base + 6 * TILE);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int t0 = g * P.seg_len, t1 = min(P.T, t0 + P.seg_len);
  const int CV = P.chunk;
  const int ntile = ceil_div(t1 - t0, CV);
  const float gm = P.gamma[h];
  const float l2g = log2f(gm);
  const uint32_t tile_bytes = (uint32_t)CV * D * 2;
  // order of a tile's worker phases: [E] of the tile before ahead of [F] when
  // saving or given the features, after it otherwise (both issuer and workers)
  constexpr bool kEpiFirst = kSave || kFeat;

  if (tid == 0) {
    for (int j = 0; j < 2; ++j) {
      umma::mbar_init(&sh.bar_mma[j], 1);
      umma::mbar_init(&sh.bar_k[j], 1);
    }
    umma::mbar_init(&sh.bar_q, 1);
    umma::mbar_init(&sh.bar_v, 1);
    umma::mbar_init(&sh.bar_g, 1);
    umma::mbar_init(&sh.bar_p, 1);
    umma::mbar_init(&sh.bar_sv, 1);
    umma::mbar_init(&sh.bar_feat, NWORK);
    umma::mbar_init(&sh.bar_sb, NWORK);
    umma::mbar_init(&sh.bar_pm, NWORK);
    umma::mbar_init(&sh.bar_epi, NWORK);
    for (int j = 0; j < 3; ++j) {
      umma::mbar_init(&sh.bar_wtma[j], 1);
      umma::mbar_init(&sh.bar_wfeat[j], NWORK);
      umma::mbar_init(&sh.bar_wmma[j], 1);
    }
    umma::mbar_init(&sh.bar_wdone, 1);
    umma::mbar_init(&sh.bar_drain, 1);
    umma::mbar_fence_init();
    sh.failed = 0;
  }
  if (tid <= ROWS) sh.pw[tid] = exp2f((float)tid * l2g);
  fill_mask_table(sh.dm, l2g, tid, NTO);
  load_rope_table(sh.ru, P, tid);
  fill_rope_small(sh.rope_small, P.rope_u, tid, NTO);
  if (warp == 0) umma::tmem_alloc(&sh.tmem_base, 512);
  if (CV < ROWS) {  // rows [CV, 128) that TMA never writes and no phase rewrites: clear
                    // them once.  V; with given features Q and both K buffers (which [D]
                    // would have written); in one launch the window stages' V buffers.
    const unsigned clear = (1u << 3) | (kFeat ? 7u : 0u) | (kWin ? (1u << 1) | (1u << 5) : 0u);
    for (int e = tid; e < 6 * (ROWS - CV) * 16; e += NTO) {
      const int t = e / ((ROWS - CV) * 16), r = e % ((ROWS - CV) * 16);
      if (clear & (1u << t)) *tile_at(base + t * TILE, CV + r / 16, r % 16) = make_uint4(0, 0, 0, 0);
    }
  }
  sync_tc();
  const uint32_t tm = sh.tmem_base;
  const uint32_t tP = tm, tS = tm + 384;
  bool failed = false;

  if (warp >= NWORK) {
    // ---------------------------------------------------------------- issuer warpgroup
    if (warp == NWORK && lane == 0) {
      const uint32_t id_qk = umma::idesc_bf16(128, 128, false, false, true);  // fp16 Q~ K~^T
      const uint32_t id_qs = umma::idesc_bf16(128, 128, false, true, true);   // fp16 Q~ S
      const uint32_t id_pv = umma::idesc_bf16(128, 128, false, true);         // bf16 Pm V
      const uint32_t id_mn = umma::idesc_bf16(128, 128, true, true);          // bf16 K~dec^T V
      if (kWin) failed = window_issue(tmk, tmv, sh, base, tS, b, h, t0, CV, l2g);
      // copies issued per barrier: after a wait gave up, the drain below waits
      // for the last of each (no barrier ever has two copies in flight)
      int armed_q = 0, armed_k[2] = {0, 0}, armed_v = 0, armed_g = 0;
      umma::mbar_expect_tx(&sh.bar_q, tile_bytes);
      tma_tile(Qs, &tmq, b, h, t0, &sh.bar_q);
      ++armed_q;
      for (int n = 0; n < 2 && n < ntile; ++n) {
        umma::mbar_expect_tx(&sh.bar_k[n], tile_bytes);
        tma_tile(base + (1 + n) * TILE, &tmk, b, h, t0 + n * CV, &sh.bar_k[n]);
        ++armed_k[n];
      }
      umma::mbar_expect_tx(&sh.bar_v, tile_bytes);
      tma_tile(Vs, &tmv, b, h, t0, &sh.bar_v);
      ++armed_v;
      umma::mbar_expect_tx(&sh.bar_g, tile_bytes);
      tma_tile(Gs, &tmg, b, h, t0, &sh.bar_g);
      ++armed_g;
      const uint32_t aq = umma::smem_u32(Qs);
      for (int n = 0; n < ntile; ++n) {
        const int buf = n & 1;
        const int c0 = t0 + n * CV;
        const uint32_t ak = umma::smem_u32(base + (1 + buf) * TILE);
        const uint32_t as = umma::smem_u32(SP), av = umma::smem_u32(Vs);
        const uint32_t ocur = tm + 128 + 128 * buf;
        // (one tcgen05 fence before each group of MMAs covers the waits before it)
        if (kFeat) {  // q~, k~ given: MMA1 once their copies are in
          wait_plain(&sh.bar_q, n & 1, failed);
          wait_plain(&sh.bar_k[buf], (n >> 1) & 1, failed);
        } else {
          if (n == 0 && P.test_wait_cycles > 0) {  // testing the expiry path
            if (!failed && !umma::mbar_wait(&sh.bar_feat, 0, P.test_wait_cycles)) failed = true;
          } else {
            wait_plain(&sh.bar_feat, n & 1, failed);
          }
        }
        if (!failed) {
          if (kSave) {  // q~, k~ of the tile out for the backward
            tma_store_tile(&tmsq, Qs, b, h, c0);
            tma_store_tile(&tmsk, base + (1 + buf) * TILE, b, h, c0);
            umma::bulk_commit();
          }
          umma::fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma::mma_ss(tP, umma::desc_kmajor(aq, kk, ROWS), umma::desc_kmajor(ak, kk, ROWS),
                         id_qk, kk > 0);
          umma::commit(&sh.bar_p);
        }
        wait_plain(&sh.bar_sb, n & 1, failed);
        if (!failed) {
          umma::fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma::mma_ss(ocur, umma::desc_kmajor(aq, kk, ROWS), umma::desc_mnmajor(as, kk, ROWS),
                         id_qs, kk > 0);
          umma::commit(&sh.bar_mma[0]);
        }
        if (kSave) {  // the saving stores have read Q and K: K may become k~dec
          if (!failed) umma::bulk_wait_read();
          umma::mbar_arrive(&sh.bar_sv);
        }
        // MMA2 done: Q is free for the next q (as early as possible: the
        // workers need it right after this tile's mask)
        wait_plain(&sh.bar_mma[0], n & 1, failed);
        if (!failed && n + 1 < ntile) {
          umma::mbar_expect_tx(&sh.bar_q, tile_bytes);
          tma_tile(Qs, &tmq, b, h, c0 + CV, &sh.bar_q);
          ++armed_q;
        }
        // the q tile after that into L2, so that its copy (issued one tile
        // from now, on the workers' critical path) does not wait on HBM
        if (!failed && n + 2 < ntile) tma_prefetch_tile(&tmq, b, h, c0 + 2 * CV);
        // kEpiFirst: y of tile n - 1 is in G right after this tile's Sb: store
        // it, then G takes the gate of tile n
        if constexpr (kEpiFirst) {
          if (n >= 1) {
            wait_plain(&sh.bar_epi, (n - 1) & 1, failed);
            if (!failed) {
              tma_store_tile(&tmy, Gs, b, h, c0 - CV);
              umma::bulk_commit();
              umma::bulk_wait_read();
              umma::mbar_expect_tx(&sh.bar_g, tile_bytes);
              tma_tile(Gs, &tmg, b, h, c0, &sh.bar_g);
              ++armed_g;
            }
          }
        }
        wait_plain(&sh.bar_pm, n & 1, failed);
        wait_plain(&sh.bar_v, n & 1, failed);
        if (!failed) {
          umma::fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma::mma_ss(ocur, umma::desc_kmajor(as, kk, ROWS), umma::desc_mnmajor(av, kk, ROWS),
                         id_pv, 1u);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma::mma_ss(tS, umma::desc_mnmajor(ak, kk, ROWS), umma::desc_mnmajor(av, kk, ROWS),
                         id_mn, 1u);
          umma::commit(&sh.bar_mma[1]);
        }
        // MMA3 / MMA4 done: V and K buffer `buf` are free for the next copies
        wait_plain(&sh.bar_mma[1], n & 1, failed);
        if (!failed) {
          if (n + 1 < ntile) {
            umma::mbar_expect_tx(&sh.bar_v, tile_bytes);
            tma_tile(Vs, &tmv, b, h, c0 + CV, &sh.bar_v);
            ++armed_v;
          }
          if (n + 2 < ntile) {
            umma::mbar_expect_tx(&sh.bar_k[buf], tile_bytes);
            tma_tile(base + (1 + buf) * TILE, &tmk, b, h, c0 + 2 * CV, &sh.bar_k[buf]);
            ++armed_k[buf];
          }
        }
        // y of tile n - 1 is in G once the workers' epilogue (after this
        // tile's mask) is done: store it, then G takes the gate of tile n
        if (!kEpiFirst && n >= 1) {
          wait_plain(&sh.bar_epi, (n - 1) & 1, failed);
          if (!failed) {
            tma_store_tile(&tmy, Gs, b, h, c0 - CV);
            umma::bulk_commit();
            umma::bulk_wait_read();
            umma::mbar_expect_tx(&sh.bar_g, tile_bytes);
            tma_tile(Gs, &tmg, b, h, c0, &sh.bar_g);
            ++armed_g;
          }
        }
      }
      // y of the last tile
      wait_plain(&sh.bar_epi, (ntile - 1) & 1, failed);
      if (!failed) {
        tma_store_tile(&tmy, Gs, b, h, t0 + (ntile - 1) * CV);
        umma::bulk_commit();
      }
      if (failed) {
        // a wait gave up: before the CTA leaves (and frees its shared and tensor
        // memory) every MMA this thread issued completes, and every copy it
        // armed lands; those complete on their own, so the normal budget ends
        // each wait
        umma::commit(&sh.bar_drain);
        umma::mbar_wait(&sh.bar_drain, 0);
        if (armed_q) umma::mbar_wait(&sh.bar_q, (armed_q - 1) & 1);
        for (int j = 0; j < 2; ++j)
          if (armed_k[j]) umma::mbar_wait(&sh.bar_k[j], (armed_k[j] - 1) & 1);
        if (armed_v) umma::mbar_wait(&sh.bar_v, (armed_v - 1) & 1);
        if (armed_g) umma::mbar_wait(&sh.bar_g, (armed_g - 1) & 1);
        umma::fence_after();
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
    float *seg_in = P.seg + (((size_t)b * P.H + h) * P.nseg + g) * (size_t)D * D;
    if (!kWin) {
      // entering state of the segment (from the scan) -> TMEM (fp32)
      const float4 *s4 = reinterpret_cast<const float4 *>(seg_in + (size_t)i * D + col);
      float v[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 x = s4[u];
        v[4 * u] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
      }
      umma::tmem_st32(myS, v);
      umma::tmem_wait_st();
    } else {
      failed = window_work<kFeat>(P, sh, base, myS, seg_in, b, h, t0, CV, l2g, i, col, warp, lane);
    }
    int prev_c0 = 0, prev_c = 0;
    for (int n = 0; n <= ntile; ++n) {
      const bool have = n < ntile, drain = n >= 1;
      const int c0 = t0 + n * CV, c = have ? min(CV, t1 - c0) : 0;
      const int buf = n & 1;
      const bool valid = i < c;
      const uint32_t ocur = tm + 128 + 128 * buf;        // O buffer of tile n
      const uint32_t oprev = tm + 128 + 128 * (buf ^ 1); // O buffer of tile n - 1
      unsigned char *Qt = Qs, *Kt = base + (1 + buf) * TILE;
      if (have && kFeat) {
        // q~ . k~ of row i from the given scalars, into the slot only this
        // thread reads (in [F], on the diagonal warps)
        if (qd == sub) {
          if (valid) cp_async4(&sh.qk_diag[buf][i], saved_scalar(P, kSavedDiag, b, h, c0 + i));
          else sh.qk_diag[buf][i] = 0.f;
        }
      }
      if (have && !kFeat) {
        // this warp's RoPE angles at row 8 warp of the tile (its rows are 8 warp + 0..7),
        // two per lane, into its own table (rope8_tab)
        __syncwarp();
        sh.rope_base[warp].v[lane >> 3][lane & 7] =
            rope_entry(P.pos_offset + c0 + 8 * warp, sh.ru, lane >> 3, lane & 7);
        __syncwarp();
        // [A] raw q, k of tile n: row fr, pairs [16 fu, 16 fu + 16); norms by shuffles
        wait_plain(&sh.bar_q, n & 1, failed);
        wait_plain(&sh.bar_k[buf], (n >> 1) & 1, failed);
        uint4 qr[4], kr[4];
        ld_pairs(Qt, fr, fu, qr);
        ld_pairs(Kt, fr, fu, kr);
        const bool fvalid = fr < c;
        if (!fvalid)  // rows past the tile hold stale bytes: use zeros
          qr[0] = qr[1] = qr[2] = qr[3] = kr[0] = kr[1] = kr[2] = kr[3] = make_uint4(0, 0, 0, 0);
        float sq, sk, qk;
        norms_and_dot(qr, kr, sq, sk, qk);
        sq += __shfl_xor_sync(0xffffffffu, sq, 1);
        sk += __shfl_xor_sync(0xffffffffu, sk, 1);
        qk += __shfl_xor_sync(0xffffffffu, qk, 1);
        sq += __shfl_xor_sync(0xffffffffu, sq, 2);
        sk += __shfl_xor_sync(0xffffffffu, sk, 2);
        qk += __shfl_xor_sync(0xffffffffu, qk, 2);
        // [D] q~ = RoPE(Norm(q)), k~ = RoPE(Norm(k)) / sqrt(d), fp16, in place
        const float rq = rsqrtf(sq / (float)D + P.eps);
        const float rk0 = rsqrtf(sk / (float)D + P.eps), rk = rk0 * P.kscale;
        // q~_i . k~_i in fp32 (one rotation acts on both, so RoPE drops out);
        // zero on rows past the tile.  Read in [F] by the diagonal warps.
        if (fu == 0) sh.qk_diag[buf][fr] = qk * rq * rk;
        if (kSave && fu == 0 && fvalid) {
          *saved_scalar(P, kSavedRq, b, h, c0 + fr) = rq;
          *saved_scalar(P, kSavedRk, b, h, c0 + fr) = rk0;
          *saved_scalar(P, kSavedDiag, b, h, c0 + fr) = qk * rq * rk;
        }
        feature_qk_store_tab(qr, kr, rq, rk, &sh.rope_base[warp].v[fu][0],
                             &sh.rope_small[lane >> 2].v[fu][0], fu, Qt, Kt, fr);
        warp_arrive(&sh.bar_feat, lane);
      }
      if (drain) wait_or_fail(&sh.bar_mma[1], (n - 1) & 1, failed);  // O(n-1), S, SP ready
      float s_inv = 1.f;
      if (have) {
        // [B] max |S| over this column quarter (4 warps)
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
        // [C] Sb = fp16(S 2^-e) with 2^e >= max |S| of the quarter, then S <- gamma^c S
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
          *tile_at(SP, i, 4 * qd + u) = pack4x2h(t);
        }
        const f2 carry = dup2(sh.pw[c]);
#pragma unroll
        for (int e2 = 0; e2 < 16; ++e2) x[e2] = mul2(x[e2], carry);
        floats_of(x, sv);
        umma::tmem_st32(myS, sv);
        umma::tmem_wait_st();
        warp_arrive(&sh.bar_sb, lane);
      }
      // [E] for the saving and given-features variants: the epilogue of tile
      // n - 1 right after this tile's Sb, so that MMA2 of tile n is done by the
      // time [F] needs it (1.349 -> 1.315 ms for the saving pass at 8 x 16K x 32).
      // The plain variant runs its epilogue after [F] (below), which measured
      // faster there; the two are written out separately (their sigmoid forms
      // differ, and one inlined lambda shared by both places cost the plain
      // pass 0.2%).
      if constexpr (kEpiFirst) {
        if (drain) {
          float o[32];
          umma::tmem_ld2x16(oprev + lane_base + col, o);
          if (P.o && i < prev_c) {
            const size_t row = (((size_t)b * P.T + prev_c0 + i) * P.H + h) * D + col;
            float4 *o4 = reinterpret_cast<float4 *>(P.o + row);
#pragma unroll
            for (int u = 0; u < 8; ++u)
              o4[u] = make_float4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
          }
          f2 ox[16];
          pairs_of(o, ox);
          f2 ss = 0ull;
#pragma unroll
          for (int e = 0; e < 16; ++e) ss = fma2(ox[e], ox[e], ss);
          sh.red_o[qd][i] = hsum2(ss);
          named_sync(5 + sub, 128);
          // gate of tile n - 1 (TMA) -> y, in place; the issuer stores the tile
          wait_plain(&sh.bar_g, (n - 1) & 1, failed);
          {
            const float ro1 = rsqrtf((sh.red_o[0][i] + sh.red_o[1][i] + sh.red_o[2][i] +
                                      sh.red_o[3][i]) / (float)D + P.eps);
            // 1/RMS(o) for the backward, with the features it was given or saves
            if (qd == 0 && i < prev_c) *saved_scalar(P, kSavedRo, b, h, prev_c0 + i) = ro1;
            const f2 ro = dup2(ro1);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              uint4 *p = tile_at(Gs, i, 4 * qd + u);
              f2 g[4], t[4];
              unpack4x2(*p, g);
              // the sigmoid in the form the backward divides y by again (sigmoid_e2)
#pragma unroll
              for (int e = 0; e < 4; ++e) t[e] = mul2(mul2(ox[4 * u + e], ro), sigmoid_e2(g[e]));
              *p = pack4x2(t);
            }
          }
          warp_arrive(&sh.bar_epi, lane);
        }
      }
      if (have) {
        // [F] MMA1 of tile n done: mask P
        wait_or_fail(&sh.bar_p, n & 1, failed);
        {
          // k~dec = gamma^{c-1-i} k~ as bf16, in place (K~ is dead once MMA1 is done,
          // and, when saving, once its store has read it).  When saving, the row
          // is read and weighted before the TMEM load of P and written after the
          // mask (measured faster there; without saving the registers it holds
          // made the kernel spill and run slower, so that variant keeps the
          // rewrite after the mask)
          const f2 wk = dup2(valid ? sh.pw[c - 1 - i] : 0.f);
          uint4 kdnew[4];
          if (kSave) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              f2 f[4];
              unpack4x2h(*tile_at(Kt, i, 4 * qd + u), f);
#pragma unroll
              for (int e = 0; e < 4; ++e) f[e] = mul2(f[e], wk);
              kdnew[u] = pack4x2(f);
            }
          }
          float pv[32];
          umma::tmem_ld2x16(myP, pv);
          // mask: Pm = bf16((Q~ K~^T) (.) D) into SP (Sb is dead once MMA2 is done),
          // D_ij = gamma^(i-j) for j <= i, else 0.  Rows and columns past the
          // tile are zero already (their q~, k~ are zero).
          f2 x[16];
          pairs_of(pv, x);
          mask_lower_table(x, sh.dm, i, (int)col);
          if (kSave) {
            wait_plain(&sh.bar_sv, n & 1, failed);
#pragma unroll
            for (int u = 0; u < 4; ++u) *tile_at(Kt, i, 4 * qd + u) = kdnew[u];
          } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              uint4 *p = tile_at(Kt, i, 4 * qd + u);
              f2 f[4];
              unpack4x2h(*p, f);
#pragma unroll
              for (int e = 0; e < 4; ++e) f[e] = mul2(f[e], wk);
              *p = pack4x2(f);
            }
          }
          // MMA2 of tile n done: Sb is dead and the Q~ S part of O is ready
          wait_or_fail(&sh.bar_mma[0], n & 1, failed);
          if (kFeat) cp_async_wait();
#pragma unroll
          for (int u = 0; u < 4; ++u) *tile_at(SP, i, 4 * qd + u) = pack4x2(&x[4 * u]);
          // the diagonal of Pm from fp32 features: where q~_i . k~_i nearly
          // cancels (a row whose output is almost only its own term: t = 0, or
          // gamma near 0) the fp16 operands of MMA1 lose it; its weight is
          // gamma^0 = 1.  Rows 32 qd .. 32 qd + 31 of qk_diag were written by
          // warps 4 qd .. 4 qd + 3, which met this warp at [B]'s barrier
          // (given features: by this thread's own copy).
          if (qd == sub)
            *(reinterpret_cast<__nv_bfloat16 *>(tile_at(SP, i, i >> 3)) + (i & 7)) =
                __float2bfloat16_rn(sh.qk_diag[buf][i]);
          // O <- gamma^{i+1} 2^e O  (the Q~ S part, before MMA3 adds Pm V)
          float ov[32];
          umma::tmem_ld2x16(ocur + lane_base + col, ov);
          const f2 f = dup2(sh.pw[i + 1] * s_inv);
          f2 y2[16];
          pairs_of(ov, y2);
#pragma unroll
          for (int e = 0; e < 16; ++e) y2[e] = mul2(y2[e], f);
          floats_of(y2, ov);
          umma::tmem_st32(ocur + lane_base + col, ov);
        }
        umma::tmem_wait_st();
        warp_arrive(&sh.bar_pm, lane);
      }
      // [E] plain variant: epilogue of tile n - 1 (overlaps MMA3 / MMA4 of tile n
      // and the copy of q of tile n + 1)
      if (!kEpiFirst && drain) {
        float o[32];
        umma::tmem_ld2x16(oprev + lane_base + col, o);
        if (P.o && i < prev_c) {
          const size_t row = (((size_t)b * P.T + prev_c0 + i) * P.H + h) * D + col;
          float4 *o4 = reinterpret_cast<float4 *>(P.o + row);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            o4[u] = make_float4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
        }
        f2 ox[16];
        pairs_of(o, ox);
        f2 ss = 0ull;
#pragma unroll
        for (int e = 0; e < 16; ++e) ss = fma2(ox[e], ox[e], ss);
        sh.red_o[qd][i] = hsum2(ss);
        named_sync(5 + sub, 128);
        // gate of tile n - 1 (TMA) -> y, in place; the issuer stores the tile
        wait_plain(&sh.bar_g, (n - 1) & 1, failed);
        {
          const float ro1 = rsqrtf((sh.red_o[0][i] + sh.red_o[1][i] + sh.red_o[2][i] +
                                    sh.red_o[3][i]) / (float)D + P.eps);
          const f2 ro = dup2(ro1), half = dup2(0.5f);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 *p = tile_at(Gs, i, 4 * qd + u);
            f2 g[4], t[4];
            unpack4x2(*p, g);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              // sigmoid(z) = 0.5 + 0.5 tanh(z / 2): one special-function op
              float za, zb;
              split2(mul2(g[e], half), za, zb);
              const f2 sg = fma2(mk2(tanh_fast(za), tanh_fast(zb)), half, half);
              t[e] = mul2(mul2(ox[4 * u + e], ro), sg);
            }
            *p = pack4x2(t);
          }
        }
        warp_arrive(&sh.bar_epi, lane);
      }
      prev_c0 = c0;
      prev_c = c;
    }
  }
  if (failed) atomicOr(&sh.failed, 1u);
  sync_tc();
  if (sh.failed && tid == 0 && P.err) atomicOr(P.err, 2u);
  // the last segment's S after its last tile (its MMA4 was waited for in the
  // workers' drain step) is the sequence's final state
  // (by the issuer warpgroup, idle by now: row i = its TMEM lane, all columns)
  if (P.state_out && g == P.nseg - 1 && warp >= NWORK) {
    const int i = 32 * (warp & 3) + lane;
    float *row = P.state_out + (((size_t)b * P.H + h) * D + i) * D;
#pragma unroll 1
    for (int qd = 0; qd < 4; ++qd) {
      float sv[32];
      umma::tmem_ld2x16(tS + ((uint32_t)(32 * (warp & 3)) << 16) + 32 * qd, sv);
      float4 *o4 = reinterpret_cast<float4 *>(row + 32 * qd);
#pragma unroll
      for (int u = 0; u < 8; ++u) o4[u] = make_float4(sv[4 * u], sv[4 * u + 1], sv[4 * u + 2], sv[4 * u + 3]);
    }
  }
  if (warp == 0) umma::tmem_dealloc(tm, 512);
}

constexpr size_t kStateSmem = 2 * kStages * TILE + sizeof(StateShared) + 1024;
static_assert(kStateSmem <= 232448, "local-state pass exceeds 227 KiB of shared memory per CTA");
constexpr size_t kOutputSmem = 6 * TILE + sizeof(OutShared) + 1024;
static_assert(kOutputSmem <= 232448, "output pass exceeds 227 KiB of shared memory per CTA");

}  // namespace
}  // namespace tc

bool tc_supported(const MixerParams &P, int dtype) { return dtype == HLA_BF16 && P.D == 128; }

namespace {
template <bool kGrad, bool kSaved = false>
cudaError_t launch_state_variant(const MixerParams &P, const void *a, const void *bsrc,
                                 cudaStream_t st) {
  CUtensorMap ma, mb;
  cudaError_t e;
  if ((e = tc::make_map(&ma, a, P, P.chunk,
                        kSaved ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)) !=
      cudaSuccess)
    return e;
  if ((e = tc::make_map(&mb, bsrc, P, P.chunk)) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc::tc_state_kernel<kGrad, kSaved>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc::kStateSmem);
  if (e != cudaSuccess) return e;
  const int np = P.npart > 1 ? P.npart : 1;
  if (P.state_nseg == 0) return cudaSuccess;  // one segment: its sums feed no other
  tc::tc_state_kernel<kGrad, kSaved><<<dim3(P.state_nseg * np, P.H, P.B), tc::NTO, tc::kStateSmem,
                                       st>>>(P, ma, mb);
  if (cudaGetLastError() != cudaSuccess) return cudaErrorLaunchFailure;
  return P.part ? launch_part_sum(P, kGrad, st) : cudaSuccess;
}
}  // namespace

cudaError_t launch_tc_seg_state(const MixerParams &P, cudaStream_t st) {
  // k~ from given features (hla_prefill_features) when there are some
  return P.features_in
             ? launch_state_variant<false, true>(P, P.saved + saved_k_offset(P.B, P.T, P.H, P.D), P.v, st)
             : launch_state_variant<false>(P, P.k, P.v, st);
}

cudaError_t launch_tc_seg_gstate(const MixerParams &P, cudaStream_t st) {
  // q~ from the forward's saved features when there are some
  return P.saved ? launch_state_variant<true, true>(P, P.saved, P.dO, st)
                 : launch_state_variant<true>(P, P.q, P.dO, st);
}

namespace {
template <bool kSave, bool kFeat = false, bool kWin = false>
cudaError_t launch_output_variant(const MixerParams &P, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mg, my, msq, msk;
  cudaError_t e;
  if (kFeat) {  // q~ and k~ given (fp16, the saved layout)
    if ((e = tc::make_map(&mq, P.saved, P, P.chunk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != cudaSuccess)
      return e;
    if ((e = tc::make_map(&mk, P.saved + saved_k_offset(P.B, P.T, P.H, P.D), P, P.chunk,
                          CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != cudaSuccess)
      return e;
  } else {
    if ((e = tc::make_map(&mq, P.q, P, P.chunk)) != cudaSuccess) return e;
    if ((e = tc::make_map(&mk, P.k, P, P.chunk)) != cudaSuccess) return e;
  }
  if ((e = tc::make_map(&mv, P.v, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&mg, P.g, P, P.chunk)) != cudaSuccess) return e;
  if ((e = tc::make_map(&my, P.y, P, P.chunk)) != cudaSuccess) return e;
  if (kSave) {
    if ((e = tc::make_map(&msq, P.saved, P, P.chunk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != cudaSuccess)
      return e;
    if ((e = tc::make_map(&msk, P.saved + saved_k_offset(P.B, P.T, P.H, P.D), P, P.chunk,
                          CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != cudaSuccess)
      return e;
  } else {
    msq = mq;  // not read
    msk = mk;
  }
  e = cudaFuncSetAttribute(tc::tc_output_kernel<kSave, kFeat, kWin>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc::kOutputSmem);
  if (e != cudaSuccess) return e;
  tc::tc_output_kernel<kSave, kFeat, kWin><<<dim3(P.nseg, P.H, P.B), tc::NTO, tc::kOutputSmem, st>>>(
      P, mq, mk, mv, mg, my, msq, msk);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_tc_seg_output(const MixerParams &P, cudaStream_t st) {
  if (P.fused) {
    if (P.features_in) return launch_output_variant<false, true, true>(P, st);
    return P.saved ? launch_output_variant<true, false, true>(P, st)
                   : launch_output_variant<false, false, true>(P, st);
  }
  if (P.features_in) return launch_output_variant<false, true>(P, st);
  return P.saved ? launch_output_variant<true>(P, st) : launch_output_variant<false>(P, st);
}

}  // namespace hla
