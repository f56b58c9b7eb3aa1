// tc_attention.cu — tensor-core (tcgen05) causal softmax attention of the
// hybrid's attention layers, bf16 at d = 128.
//
// arXiv 2601.22156, Section 5.1 "Attention Logits Scaling" (Eq. 11) and
// Appendix A "Attention Layers" (Eq. 17): per query head h (key/value head
// h / (Hq / Hkv)) and query token t at position p = pos_offset + t,
//   logit_ti = s_p (q_t . k_i) / sqrt(d),   s_p = log_a(p + 1 + a),   i <= t
//   o_t = sum_i softmax_i(logit_ti) v_i,    y_t = Norm(o_t) * sigmoid(gate_t).
//
// One CTA per (128-query tile, query head, sequence), query tiles longest
// first.  Per key tile j = 0 .. (the query tile's own index):
//   MMA1  S_j = Q K_j^T            (raw bf16 q, k; fp32 in TMEM, two buffers)
//   workers: x = S_j row, masked above the diagonal on the last tile; the
//            row's running maximum m (shared by the row's four quarter threads
//            through shared memory); p = 2^(c_t x - m) with c_t = s_p log2(e) /
//            sqrt(d) folded into the exponent's FMA (so q is never rounded
//            after scaling); the row sum kept as one partial per quarter; P as
//            packed bf16 over the S columns it came from; O <- 2^(m_old -
//            m) O in TMEM once the previous MMA2 is done (skipped where no row
//            of the warp changed its maximum)
//   MMA2  O += P V_j               (A = P from tensor memory)
// The issuer issues MMA1 of tile j + 1 before waiting for the workers' P of
// tile j, so the QK^T product of the next tile runs under this tile's
// softmax; k and v are double-buffered by TMA, k refilled as soon as MMA1 of
// the tile before has read it and v once MMA2 has.  The epilogue divides by the
// row sum, takes the output RMSNorm and the gate (tile loaded at the start)
// and writes y over the gate tile for a TMA store.
#include "tc_common.cuh"

namespace hla {

struct AttnParams {
  int B, T, Hq, Hkv, group, nqt;
  long long pos_offset;
  float a;          // logit-scale base
  float inv_log2a;  // 1 / log2(a)
  float eps;
  float *o;           // optional fp32 [B, T, Hq, d]
  unsigned int *err;  // device status word
};

namespace tc {
namespace {

struct AttnShared {
  float red_m[2][4][ROWS];  // quarter maxima of each row, by key-tile parity
  float red_e[2][4][ROWS];  // epilogue: quarter parts of the row sum and of sum O^2
  uint64_t bar_q, bar_g;    // TMA: q tile, gate tile
  uint64_t bar_k[2];        // TMA: k tile into buffer 0 / 1
  uint64_t bar_v[2];        // TMA: v tile into buffer 0 / 1
  uint64_t bar_s[2];        // MMA1 done (S buffer 0 / 1)
  uint64_t bar_o[2];        // MMA2 of tile j done, on barrier j & 1: the workers wait only
                            // for some of them, and a parity wait is exact only while it
                            // is at most one phase behind its barrier
  uint64_t bar_p;           // workers: P written, O rescaled (one arrive per warp)
  uint64_t bar_epi;         // workers: y written over the gate tile
  uint32_t tmem_base;
  uint32_t failed;
};

__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(NTO, 1)
    tc_attention_kernel(const __grid_constant__ AttnParams A, const __grid_constant__ CUtensorMap tmq,
                        const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                        const __grid_constant__ CUtensorMap tmg, const __grid_constant__ CUtensorMap tmy) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  // Q: q.  K j / V j at base + (1 + j) TILE / base + (3 + j) TILE.  G: gate -> y.
  unsigned char *Qs = base, *Gs = base + 5 * TILE;
  AttnShared &sh = *reinterpret_cast<AttnShared *>(base + 6 * TILE);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = A.nqt - 1 - (int)blockIdx.x;  // longest rows first
  const int h = blockIdx.y, b = blockIdx.z, hk = h / A.group;
  const int q0 = qt * ROWS;
  const int nkt = qt + 1;
  const uint32_t tile_bytes = (uint32_t)ROWS * D * 2;

  if (tid == 0) {
    uint64_t *bars[] = {&sh.bar_q,    &sh.bar_g,    &sh.bar_k[0], &sh.bar_k[1], &sh.bar_v[0],
                        &sh.bar_v[1], &sh.bar_s[0], &sh.bar_s[1], &sh.bar_o[0], &sh.bar_o[1]};
    for (uint64_t *bar : bars) umma::mbar_init(bar, 1);
    umma::mbar_init(&sh.bar_p, NWORK);
    umma::mbar_init(&sh.bar_epi, NWORK);
    umma::mbar_fence_init();
    sh.failed = 0;
  }
  if (warp == 0) umma::tmem_alloc(&sh.tmem_base, 512);
  sync_tc();
  const uint32_t tm = sh.tmem_base;
  const uint32_t tS0 = tm, tO = tm + 256;  // S buffer j at tm + 128 j
  bool failed = false;

  if (warp >= NWORK) {
    // ---------------------------------------------------------------- issuer
    if (warp == NWORK && lane == 0) {
      const uint32_t id_qk = umma::idesc_bf16(128, 128, false, false);  // Q K^T, both K-major
      const uint32_t id_pv = umma::idesc_bf16(128, 128, false, true);   // P (TMEM) V
      const uint32_t aq = umma::smem_u32(Qs);
      umma::mbar_expect_tx(&sh.bar_q, tile_bytes);
      tma_tile(Qs, &tmq, b, h, q0, &sh.bar_q);
      umma::mbar_expect_tx(&sh.bar_g, tile_bytes);
      tma_tile(Gs, &tmg, b, h, q0, &sh.bar_g);
      for (int n = 0; n < 2 && n < nkt; ++n) {
        umma::mbar_expect_tx(&sh.bar_k[n], tile_bytes);
        tma_tile(base + (1 + n) * TILE, &tmk, b, hk, n * ROWS, &sh.bar_k[n]);
        umma::mbar_expect_tx(&sh.bar_v[n], tile_bytes);
        tma_tile(base + (3 + n) * TILE, &tmv, b, hk, n * ROWS, &sh.bar_v[n]);
      }
      wait_or_fail(&sh.bar_q, 0, failed);
      for (int j = 0; j <= nkt; ++j) {
        if (j < nkt) {  // MMA1 of tile j as soon as its k has landed
          const int buf = j & 1;
          wait_or_fail(&sh.bar_k[buf], (j >> 1) & 1, failed);
          if (!failed) {
            const uint32_t ak = umma::smem_u32(base + (1 + buf) * TILE);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma::mma_ss(tS0 + 128 * buf, umma::desc_kmajor(aq, kk, ROWS), umma::desc_kmajor(ak, kk, ROWS),
                           id_qk, kk > 0);
            umma::commit(&sh.bar_s[buf]);
          }
        }
        // MMA1 of tile j - 1 is done (its softmax has started or finished): that
        // k buffer takes tile j + 1, a whole tile before MMA1 needs it
        if (j >= 1 && j + 1 < nkt) {
          const int pb = (j - 1) & 1;
          wait_or_fail(&sh.bar_s[pb], ((j - 1) >> 1) & 1, failed);
          if (!failed) {
            umma::mbar_expect_tx(&sh.bar_k[pb], tile_bytes);
            tma_tile(base + (1 + pb) * TILE, &tmk, b, hk, (j + 1) * ROWS, &sh.bar_k[pb]);
          }
        }
        if (j >= 1) {  // MMA2 of tile j - 1 once its P is in place
          const int jp = j - 1, pb = jp & 1;
          wait_or_fail(&sh.bar_p, jp & 1, failed);
          wait_or_fail(&sh.bar_v[pb], (jp >> 1) & 1, failed);
          if (!failed) {
            const uint32_t av = umma::smem_u32(base + (3 + pb) * TILE);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma::mma_ts(tO, tS0 + 128 * pb + 32 * (kk >> 1) + 8 * (kk & 1),
                           umma::desc_mnmajor(av, kk, ROWS), id_pv, (jp > 0 || kk > 0) ? 1u : 0u);
            umma::commit(&sh.bar_o[pb]);
          }
          // MMA2 of tile j - 1 done: its v buffer takes tile j + 1
          wait_or_fail(&sh.bar_o[pb], (jp >> 1) & 1, failed);
          if (!failed && j + 1 < nkt) {
            umma::mbar_expect_tx(&sh.bar_v[pb], tile_bytes);
            tma_tile(base + (3 + pb) * TILE, &tmv, b, hk, (j + 1) * ROWS, &sh.bar_v[pb]);
          }
        }
      }
      // y out of G
      wait_or_fail(&sh.bar_epi, 0, failed);
      if (!failed) {
        tma_store_tile(&tmy, Gs, b, h, q0);
        umma::bulk_commit();
      }
      umma::bulk_wait_all();
    }
  } else {
    // ---------------------------------------------------------------- workers
    const int sub = warp & 3, qd = warp >> 2, i = 32 * sub + lane;
    const uint32_t lane_base = (uint32_t)(32 * sub) << 16;
    const uint32_t col = 32 * qd;
    // c_t = s_p log2(e) / sqrt(d): logits in units of log2, for ex2
    const float ct = log2f((float)(A.pos_offset + q0 + i) + 1.f + A.a) * A.inv_log2a *
                     (1.4426950408889634f / 11.313708498984761f);
    float m_run = -INFINITY, l_part = 0.f;
    for (int j = 0; j < nkt; ++j) {
      const int buf = j & 1;
      const uint32_t ts = tS0 + 128 * buf + lane_base + col;
      wait_or_fail(&sh.bar_s[buf], (j >> 1) & 1, failed);
      float x[32];
      umma::tmem_ld2x16(ts, x);
      if (j == qt) {  // the diagonal tile: keys after the query are masked
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = (int)col + e > i ? -INFINITY : x[e];
      }
      float mx = x[0];
#pragma unroll
      for (int e = 1; e < 32; ++e) mx = fmaxf(mx, x[e]);
      sh.red_m[j & 1][qd][i] = mx;
      named_sync(5 + sub, 128);
      const float mt = fmaxf(fmaxf(sh.red_m[j & 1][0][i], sh.red_m[j & 1][1][i]),
                             fmaxf(sh.red_m[j & 1][2][i], sh.red_m[j & 1][3][i]));
      // The exponent's offset m moves only when the row's maximum exceeds it by
      // more than 8 (log2 units): until then p <= 2^8, which fp32 sums and bf16
      // operands hold as well as p <= 1, and the final division by the row sum
      // cancels whichever offset was used.  So O needs rescaling only on the
      // few tiles where some row of the warp moves m.
      const float m_tile = ct * mt;  // every row has a key: finite
      const bool upd = m_tile > m_run + 8.f;  // always on the first tile
      const float m_new = upd ? m_tile : m_run;
      const float alpha = ex2_fast(m_run - m_new);  // 1 without a move; 0 on the first tile
      // p = 2^(c_t x - m), two lanes per FMA; masked entries (-inf) give 0
      uint32_t pw[16];
      f2 s2 = 0ull;
      {
        const f2 c2 = dup2(ct), nm = dup2(-m_new), one = dup2(1.f);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float lo, hi;
          split2(fma2(mk2(x[2 * e], x[2 * e + 1]), c2, nm), lo, hi);
          const f2 pp = mk2(ex2_fast(lo), ex2_fast(hi));
          s2 = fma2(pp, one, s2);
          pw[e] = bf_of_f2(pp);
        }
      }
      l_part = fmaf(l_part, alpha, hsum2(s2));
      umma::tmem_st16u(ts, pw);
      if (j > 0 && !__all_sync(0xffffffffu, !upd)) {  // O <- alpha O once MMA2 of tile j - 1 is done
        wait_or_fail(&sh.bar_o[(j - 1) & 1], ((j - 1) >> 1) & 1, failed);
        {
          float ov[32];
          umma::tmem_ld2x16(tO + lane_base + col, ov);
          f2 y2[16];
          pairs_of(ov, y2);
          const f2 al = dup2(alpha);
#pragma unroll
          for (int e = 0; e < 16; ++e) y2[e] = mul2(y2[e], al);
          floats_of(y2, ov);
          umma::tmem_st32(tO + lane_base + col, ov);
        }
      }
      m_run = m_new;
      umma::tmem_wait_st();
      warp_arrive(&sh.bar_p, lane);
    }
    // epilogue: o = O / l, y = Norm(o) sigmoid(gate) over the gate tile
    // the last MMA2's completion covers every earlier one
    wait_or_fail(&sh.bar_o[(nkt - 1) & 1], ((nkt - 1) >> 1) & 1, failed);
    float ov[32];
    umma::tmem_ld2x16(tO + lane_base + col, ov);
    f2 o2[16];
    pairs_of(ov, o2);
    f2 ss = 0ull;
#pragma unroll
    for (int e = 0; e < 16; ++e) ss = fma2(o2[e], o2[e], ss);
    sh.red_e[0][qd][i] = l_part;
    sh.red_e[1][qd][i] = hsum2(ss);
    named_sync(5 + sub, 128);
    const float l = sh.red_e[0][0][i] + sh.red_e[0][1][i] + sh.red_e[0][2][i] + sh.red_e[0][3][i];
    const float so = sh.red_e[1][0][i] + sh.red_e[1][1][i] + sh.red_e[1][2][i] + sh.red_e[1][3][i];
    const float inv_l = 1.f / l;
    const float ro = rsqrtf(so * inv_l * inv_l / (float)D + A.eps);
    const f2 il = dup2(inv_l);
#pragma unroll
    for (int e = 0; e < 16; ++e) o2[e] = mul2(o2[e], il);
    const bool valid = q0 + i < A.T;
    if (A.o && valid) {
      float4 *o4 = reinterpret_cast<float4 *>(A.o + (((size_t)b * A.T + q0 + i) * A.Hq + h) * D + col);
      floats_of(o2, ov);
#pragma unroll
      for (int u = 0; u < 8; ++u) o4[u] = make_float4(ov[4 * u], ov[4 * u + 1], ov[4 * u + 2], ov[4 * u + 3]);
    }
    wait_or_fail(&sh.bar_g, 0, failed);
    {
      const f2 r2 = dup2(ro), half = dup2(0.5f);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint4 *p = tile_at(Gs, i, 4 * qd + u);
        f2 g[4], t[4];
        unpack4x2(*p, g);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float za, zb;  // sigmoid(z) = 0.5 + 0.5 tanh(z / 2)
          split2(mul2(g[e], half), za, zb);
          const f2 sg = fma2(mk2(tanh_fast(za), tanh_fast(zb)), half, half);
          t[e] = mul2(mul2(o2[4 * u + e], r2), sg);
        }
        *p = pack4x2(t);
      }
    }
    warp_arrive(&sh.bar_epi, lane);
  }
  if (failed) atomicOr(&sh.failed, 1u);
  sync_tc();
  if (sh.failed && tid == 0 && A.err) atomicOr(A.err, 16u);
  if (warp == 0) umma::tmem_dealloc(tm, 512);
}

constexpr size_t kAttnSmem = 6 * TILE + sizeof(AttnShared) + 1024;
static_assert(kAttnSmem <= 232448, "attention exceeds 227 KiB of shared memory per CTA");

}  // namespace
}  // namespace tc

namespace {

// TMA map of a [B, T, H, 128] bf16 tensor with 128-token boxes.
cudaError_t attn_map(CUtensorMap *map, const void *ptr, int B, int T, int H) {
  MixerParams P;
  memset(&P, 0, sizeof(P));
  P.B = B;
  P.T = T;
  P.H = H;
  return tc::make_map(map, ptr, P, tc::ROWS);
}

hla_status check_attn_shape(const hla_attn_shape *s) {
  if (!s) return HLA_ERR_INVALID_ARG;
  if (s->B < 0 || s->T < 0 || s->Hq < 1 || s->Hkv < 1 || s->pos_offset < 0 ||
      !(s->a > 1.0) || !(s->a < 1e30) || !(s->norm_eps >= 0.f) || !(s->norm_eps < 1.f))
    return HLA_ERR_INVALID_ARG;
  if (s->pos_offset > (1LL << 62) - (long long)s->T) return HLA_ERR_INVALID_ARG;
  if (s->Hq % s->Hkv) return HLA_ERR_INVALID_ARG;
  if (s->dtype != HLA_BF16 || s->d != 128 || s->Hq > kMaxHeads) return HLA_ERR_UNSUPPORTED;
  return HLA_OK;
}

}  // namespace
}  // namespace hla

using namespace hla;

extern "C" {

size_t hla_attention_workspace_size(const hla_attn_shape *s) {
  return check_attn_shape(s) == HLA_OK ? kStatusBytes : 0;
}

hla_status hla_attention_prefill(const hla_attn_shape *s, const void *q, const void *k,
                                 const void *v, const void *gate, void *y, float *o, void *ws,
                                 size_t ws_bytes, hla_stream stream) {
  hla_status st = check_attn_shape(s);
  if (st != HLA_OK) return st;
  const bool empty = s->B == 0 || s->T == 0;
  const void *acts[] = {q, k, v, gate, y};
  for (const void *p : acts)
    if ((st = need_unless(empty, p)) != HLA_OK) return st;
  if ((st = maybe(o)) != HLA_OK) return st;
  if (!ws || !aligned16(ws) || ws_bytes < kStatusBytes) return HLA_ERR_WORKSPACE;
  cudaStream_t cs = (cudaStream_t)stream;
  unsigned int *err = (unsigned int *)ws;
  if (cudaMemsetAsync(err, 0, sizeof(unsigned int), cs) != cudaSuccess) return HLA_ERR_CUDA;
  if (empty) return HLA_OK;

  AttnParams A;
  A.B = s->B;
  A.T = s->T;
  A.Hq = s->Hq;
  A.Hkv = s->Hkv;
  A.group = s->Hq / s->Hkv;
  A.nqt = ceil_div(s->T, tc::ROWS);
  A.pos_offset = s->pos_offset;
  A.a = (float)s->a;
  A.inv_log2a = (float)(1.0 / log2(s->a));
  A.eps = s->norm_eps;
  A.o = o;
  A.err = err;
  CUtensorMap mq, mk, mv, mg, my;
  if (attn_map(&mq, q, s->B, s->T, s->Hq) != cudaSuccess ||
      attn_map(&mk, k, s->B, s->T, s->Hkv) != cudaSuccess ||
      attn_map(&mv, v, s->B, s->T, s->Hkv) != cudaSuccess ||
      attn_map(&mg, gate, s->B, s->T, s->Hq) != cudaSuccess ||
      attn_map(&my, y, s->B, s->T, s->Hq) != cudaSuccess)
    return HLA_ERR_CUDA;
  if (cudaFuncSetAttribute(tc::tc_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)tc::kAttnSmem) != cudaSuccess)
    return HLA_ERR_CUDA;
  tc::tc_attention_kernel<<<dim3(A.nqt, s->Hq, s->B), tc::NTO, tc::kAttnSmem, cs>>>(A, mq, mk, mv, mg,
                                                                                    my);
  return cudaGetLastError() == cudaSuccess ? HLA_OK : HLA_ERR_CUDA;
}

}  // extern "C"
