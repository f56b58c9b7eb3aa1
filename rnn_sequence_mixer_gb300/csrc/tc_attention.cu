// tc_attention.cu — tensor-core (tcgen05) causal softmax attention of the
// hybrid's attention layers, bf16 at d = 128.
//
// arXiv 2601.22156, Section 5.1 "Attention Logits Scaling" (Eq. 11) and
// Appendix A "Attention Layers" (Eq. 17): per query head h (key/value head
// h / (Hq / Hkv)) and query token t at position p = pos_offset + t,
//   logit_ti = s_p (q_t . k_i) / sqrt(d),   s_p = log_a(p + 1 + a),   i <= t
//   o_t = sum_i softmax_i(logit_ti) v_i,    y_t = Norm(o_t) * sigmoid(gate_t).
//
// One CTA per pair of adjacent 128-query tiles (query head, sequence), the
// longest pairs first.  Per query tile X and key tile j = 0 .. X:
//   MMA1  S_j = Q K_j^T            (raw bf16 q, k; fp32 in TMEM)
//   softmax: one thread per score row; x = S_j row, masked above the diagonal
//            on the last tile; p = 2^(c_t x - m) with c_t = s_p log2(e) /
//            sqrt(d) folded into the exponent's FMA (so q is never rounded
//            after scaling) and an offset m that moves only when the row's
//            maximum outgrows it; P as packed bf16 over the S columns it came
//            from; O <- 2^(m_old - m) O in TMEM once the previous MMA2 is done
//            (skipped where no row of the warp moved m)
//   MMA2  O += P V_j               (A = P from tensor memory)
// MMA1 of tile j + 1 is issued right behind MMA2 of tile j, so the next QK^T
// product runs under this tile's softmax, and the two query tiles' softmaxes
// alternate on the tensor core.  k and v are double-buffered by TMA from a
// warp of their own.  The epilogue divides by the row sum, takes the output
// RMSNorm and the gate (loaded into the q buffer once its last MMA1 is done)
// and writes y over the gate tile for a TMA store.
#include <type_traits>

#include "tc_common.cuh"

namespace hla {

struct AttnParams {
  int B, T, Hq, Hkv, group, nqt;
  int npairs;       // CTAs per (sequence, head): pairs of adjacent query tiles
  int pad;
  long long pos_offset;
  float a;          // logit-scale base
  float inv_log2a;  // 1 / log2(a)
  float eps;
  float *o;           // optional fp32 [B, T, Hq, d]
  unsigned int *err;  // device status word
};

namespace tc {
namespace {

constexpr int kAttnThreads = 352;  // two softmax warpgroups, the copy warp, one MMA warp per query tile

struct AttnShared {
  uint64_t bar_q;     // TMA: the two q tiles
  uint64_t bar_k[2];  // TMA: k tile into buffer 0 / 1
  uint64_t bar_v[2];  // TMA: v tile into buffer 0 / 1
  uint64_t bar_s[2];  // MMA1 of query tile X done (S_X written), one phase per key tile
  uint64_t bar_p[2];  // softmax X: P_X written (one arrive per warp), one phase per key tile
  uint64_t bar_o[2];  // MMA2 of query tile X done, one phase per key tile
  uint64_t bar_g[2];  // TMA: gate of query tile X, into its q buffer
  uint64_t bar_e[2];  // softmax X: y written over that gate (one arrive per warp)
  uint64_t bar_kfree[2];  // MMA1 of each query tile reading k buffer n done (one commit per tile), one phase per key tile held
  uint64_t bar_vfree[2];  // MMA2 of each query tile reading v buffer n done (one commit per tile), one phase per key tile held
  uint64_t bar_drain[2];  // after a wait gave up: every MMA issued for tile X is done (commit)
  uint64_t bar_turn[2];   // the other tile's MMA thread has issued its products: tile X's turn
  uint32_t tmem_base;
  uint32_t failed;
};

__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// A bounded wait (as wait_or_fail) that tries the phase once before reading
// the clock: the phases waited on here have mostly completed already.
__device__ __forceinline__ void attn_wait(uint64_t *bar, uint32_t parity, bool &failed) {
  if (!failed && !umma::mbar_wait_tryfirst(bar, parity)) failed = true;
  umma::fence_after();
}

// 128 consecutive fp32 columns of this thread's TMEM lane under one wait.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&x)[128]) {
  uint32_t r[8][16];
#pragma unroll
  for (int c = 0; c < 8; ++c) umma::tmem_ld16_nowait(taddr + 16 * c, r[c]);
  umma::tmem_wait_ld();
#pragma unroll
  for (int c = 0; c < 8; ++c)
#pragma unroll
    for (int e = 0; e < 16; ++e) x[16 * c + e] = __uint_as_float(r[c][e]);
}

// One CTA takes two adjacent query tiles of one head, A = 2 pr and B = 2 pr + 1
// (B absent past the sequence), and streams their key/value tiles 0..B once
// for both.  Tensor memory: S_A, S_B (128 columns each; P_X is written as
// packed bf16 over the first 64 columns of S_X, MMA2's A operand) and O_A,
// O_B.  Warps 0..3 run the softmax of A, warps 4..7 that of B, one thread per
// score row (the row's maximum and sum stay in the thread).  The first lane of
// warp 9 (10) issues the MMAs of A (B): once its softmax has written P_X(j), it
// issues MMA2_X(j) = O_X += P_X V_j and MMA1_X(j + 1) (ordered behind it by the
// tensor pipe, although it writes the columns that MMA2 reads P from).  A
// thread that issues MMAs stalls while the tensor pipe is busy, so each tile
// has a thread of its own: while one waits for the pipe the other's products
// are already queued, and the pipe runs one tile's products while the other
// tile's softmax works.  Each MMA thread commits to a buffer's "free" barrier
// after its last MMA that reads the buffer, and warp 8's first lane refills the
// buffer with the key tile two ahead once both have, so the copies run a whole
// tile ahead.
__global__ void __launch_bounds__(kAttnThreads, 1)
    tc_attention_kernel(const __grid_constant__ AttnParams A, const __grid_constant__ CUtensorMap tmq,
                        const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                        const __grid_constant__ CUtensorMap tmg, const __grid_constant__ CUtensorMap tmy) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  // Q X at base + X TILE (q, then the gate and y of tile X); K j at base + (2 + j) TILE;
  // V j at base + (4 + j) TILE.
  AttnShared &sh = *reinterpret_cast<AttnShared *>(base + 6 * TILE);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pr = A.npairs - 1 - (int)blockIdx.x;  // longest pairs first
  const int qa = 2 * pr, qb = 2 * pr + 1;
  const bool hasB = qb < A.nqt;
  const int last = hasB ? qb : qa;  // key tiles 0..last (A uses 0..qa)
  const int h = blockIdx.y, b = blockIdx.z, hk = h / A.group;
  const uint32_t tile_bytes = (uint32_t)ROWS * D * 2;

  if (tid == 0) {
    uint64_t *bars[] = {&sh.bar_q, &sh.bar_k[0], &sh.bar_k[1], &sh.bar_v[0], &sh.bar_v[1],
                        &sh.bar_s[0], &sh.bar_s[1], &sh.bar_o[0], &sh.bar_o[1], &sh.bar_g[0],
                        &sh.bar_g[1], &sh.bar_drain[0], &sh.bar_drain[1], &sh.bar_turn[0],
                        &sh.bar_turn[1]};
    for (uint64_t *bar : bars) umma::mbar_init(bar, 1);
    for (int x = 0; x < 2; ++x) {
      umma::mbar_init(&sh.bar_p[x], 4);
      umma::mbar_init(&sh.bar_e[x], 4);
      // the tiles that wait on a free barrier (key tiles 0 .. qa - 1) are read by both query tiles
      umma::mbar_init(&sh.bar_kfree[x], hasB ? 2 : 1);
      umma::mbar_init(&sh.bar_vfree[x], hasB ? 2 : 1);
    }
    umma::mbar_fence_init();
    sh.failed = 0;
  }
  if (warp == 0) umma::tmem_alloc(&sh.tmem_base, 512);
  sync_tc();
  const uint32_t tm = sh.tmem_base;
  bool failed = false;

  if (warp == 8) {
    // ---------------------------------------------------------------- copies
    if (lane == 0) {
      int armed_k[2] = {0, 0}, armed_v[2] = {0, 0};
      umma::mbar_expect_tx(&sh.bar_q, (hasB ? 2 : 1) * tile_bytes);
      tma_tile(base, &tmq, b, h, qa * ROWS, &sh.bar_q);
      if (hasB) tma_tile(base + TILE, &tmq, b, h, qb * ROWS, &sh.bar_q);
      for (int n = 0; n < 2 && n <= last; ++n) {
        umma::mbar_expect_tx(&sh.bar_k[n], tile_bytes);
        tma_tile(base + (2 + n) * TILE, &tmk, b, hk, n * ROWS, &sh.bar_k[n]);
        ++armed_k[n];
        umma::mbar_expect_tx(&sh.bar_v[n], tile_bytes);
        tma_tile(base + (4 + n) * TILE, &tmv, b, hk, n * ROWS, &sh.bar_v[n]);
        ++armed_v[n];
      }
      // key tile j + 2 into the buffers of tile j once every MMA reading them is
      // done (each free barrier completes one phase per tile the buffer held)
      for (int j = 0; j + 2 <= last; ++j) {
        const int kb = j & 1;
        if (j + 3 <= last) tma_prefetch_tile(&tmk, b, hk, (j + 3) * ROWS);
        attn_wait(&sh.bar_kfree[kb], (j >> 1) & 1, failed);
        if (!failed) {
          umma::mbar_expect_tx(&sh.bar_k[kb], tile_bytes);
          tma_tile(base + (2 + kb) * TILE, &tmk, b, hk, (j + 2) * ROWS, &sh.bar_k[kb]);
          ++armed_k[kb];
        }
        attn_wait(&sh.bar_vfree[kb], (j >> 1) & 1, failed);
        if (!failed) {
          umma::mbar_expect_tx(&sh.bar_v[kb], tile_bytes);
          tma_tile(base + (4 + kb) * TILE, &tmv, b, hk, (j + 2) * ROWS, &sh.bar_v[kb]);
          ++armed_v[kb];
        }
      }
      if (failed) {
        // a wait gave up: every copy armed lands before the CTA leaves (they
        // complete on their own: normal budgets)
        umma::mbar_wait(&sh.bar_q, 0);
        for (int n = 0; n < 2; ++n) {
          if (armed_k[n]) umma::mbar_wait(&sh.bar_k[n], (armed_k[n] - 1) & 1);
          if (armed_v[n]) umma::mbar_wait(&sh.bar_v[n], (armed_v[n] - 1) & 1);
        }
      }
    }
  } else if (warp == 9 || warp == 10) {
    // ---------------------------------------------------------------- MMAs of tile X
    const int x = warp - 9, qx = x ? qb : qa;
    if (lane == 0 && (x == 0 || hasB)) {
      const uint32_t id_qk = umma::idesc_bf16(128, 128, false, false);  // Q K^T, both K-major
      const uint32_t id_pv = umma::idesc_bf16(128, 128, false, true);   // P (TMEM) V
      const uint32_t aq = umma::smem_u32(base + x * TILE);
      const uint32_t tS = tm + 128 * x, tO = tm + 256 + 128 * x;
      bool armed_g = false;
      // Buffers enter as compile-time constants (N = j & 1), so every operand
      // descriptor is loop-invariant and computed once: recomputing them for a
      // runtime buffer index between MMAs holds the issuing thread behind the
      // tensor pipe (measured: 72-80 cycles per 128x128x16 MMA instead of 64).
      // S_X = Q_X K_j^T; then this tile is done with k buffer N
      auto mma1 = [&](int j, auto nbuf) {
        constexpr int N = decltype(nbuf)::value;
        const uint32_t ak = umma::smem_u32(base + (2 + N) * TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma::mma_ss(tS, umma::desc_kmajor(aq, kk, ROWS), umma::desc_kmajor(ak, kk, ROWS), id_qk,
                       kk > 0);
        umma::commit(&sh.bar_s[x]);
        umma::commit(&sh.bar_kfree[N]);
      };
      // O_X += P_X V_j, P_X from the first 64 columns of S_X; then this tile is
      // done with v buffer N
      auto mma2 = [&](int j, auto nbuf) {
        constexpr int N = decltype(nbuf)::value;
        const uint32_t av = umma::smem_u32(base + (4 + N) * TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma::mma_ts(tO, tS + 8 * kk, umma::desc_mnmajor(av, kk, ROWS), id_pv,
                       (j > 0 || kk > 0) ? 1u : 0u);
        umma::commit(&sh.bar_o[x]);
        umma::commit(&sh.bar_vfree[N]);
      };
      // The two threads take turns: A's first product, B's, then per key tile j
      // A's MMA2 + MMA1 and B's.  A thread stalls while the tensor pipe is
      // busy, so the one whose turn comes next makes its checks (P written, v
      // and k in) meanwhile and issues as soon as the other has issued, and the
      // products of the two tiles never share the pipe: each tile's S is ready
      // as early as it can be and the two softmaxes take turns too.
      // turn(n): wait for the other thread's n-th hand-over (0 = its first
      // product); tile A has no turn to wait for without B, nor B past A's last
      auto wait_plain = [&](uint64_t *bar, uint32_t parity) {
        if (!failed && !umma::mbar_wait_tryfirst(bar, parity)) failed = true;
      };
      auto turn = [&](int n) {
        if (hasB && (x == 0 || n <= qa + 1) && !failed) {  // polled: the turn comes soon
          const long long t0 = clock64();
          while (!umma::mbar_test(&sh.bar_turn[x], n & 1))
            if (clock64() - t0 > 4000000000LL) {
              failed = true;
              break;
            }
        }
      };
      auto hand_over = [&]() { umma::mbar_arrive(&sh.bar_turn[x ^ 1]); };
      constexpr std::integral_constant<int, 0> kBuf0{};
      constexpr std::integral_constant<int, 1> kBuf1{};
      attn_wait(&sh.bar_q, 0, failed);
      attn_wait(&sh.bar_k[0], 0, failed);
      if (x == 1) turn(0);
      if (!failed) mma1(0, kBuf0);
      hand_over();
      // key tile j with its v in buffer N = j & 1 and the next k in buffer N ^ 1
      auto step = [&](int j, auto nbuf) {
        constexpr int N = decltype(nbuf)::value;
        // one tcgen05 fence after the last of these waits, before the MMAs
        wait_plain(&sh.bar_p[x], j & 1);
        wait_plain(&sh.bar_v[N], (j >> 1) & 1);
        if (j < qx) wait_plain(&sh.bar_k[N ^ 1], ((j + 1) >> 1) & 1);
        turn(x == 0 ? j : j + 1);  // A's batch j follows B's hand-over j, B's follows A's j + 1
        if (failed) return;
        umma::fence_after();
        mma2(j, nbuf);
        if (j == qx) {  // MMA1_X is done for good: Q_X takes the gate of tile X
          umma::mbar_expect_tx(&sh.bar_g[x], tile_bytes);
          tma_tile(base + x * TILE, &tmg, b, h, j * ROWS, &sh.bar_g[x]);
          armed_g = true;
        } else {
          mma1(j + 1, std::integral_constant<int, N ^ 1>{});
        }
        hand_over();
      };
      for (int j = 0; j <= qx && !failed; j += 2) {
        step(j, kBuf0);
        if (j + 1 <= qx && !failed) step(j + 1, kBuf1);
      }
      // y of tile X out of its q buffer
      attn_wait(&sh.bar_e[x], 0, failed);
      if (!failed) {
        tma_store_tile(&tmy, base + x * TILE, b, h, qx * ROWS);
        umma::bulk_commit();
      }
      if (failed) {
        // a wait gave up: every MMA this thread issued completes and its gate lands
        umma::commit(&sh.bar_drain[x]);
        umma::mbar_wait(&sh.bar_drain[x], 0);
        if (armed_g) umma::mbar_wait(&sh.bar_g[x], 0);
        umma::fence_after();
      }
      umma::bulk_wait_all();
    }
  } else if (warp < 4 || hasB) {
    // ---------------------------------------------------------------- softmax of tile X
    const int x = warp >> 2, sub = warp & 3, i = 32 * sub + lane;  // score row = TMEM lane
    const int qx = x ? qb : qa, q = qx * ROWS + i;
    const uint32_t lane_base = (uint32_t)(32 * sub) << 16;
    const uint32_t tS = tm + 128 * x + lane_base, tO = tm + 256 + 128 * x + lane_base;
    // c_t = s_p log2(e) / sqrt(d): logits in units of log2, for ex2
    const float ct = log2f((float)(A.pos_offset + q) + 1.f + A.a) * A.inv_log2a *
                     (1.4426950408889634f / 11.313708498984761f);
    float m_run = -INFINITY, l = 0.f;
    for (int j = 0; j <= qx; ++j) {
      attn_wait(&sh.bar_s[x], j & 1, failed);
      float s[128];
      tmem_ld128(tS, s);
      if (j == qx) {  // the diagonal tile: keys after the query are masked
#pragma unroll
        for (int e = 0; e < 128; ++e) s[e] = e > i ? -INFINITY : s[e];
      }
      // the row maximum as a tree (eight independent chains, not one of 128)
      float m8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) m8[e] = s[e];
#pragma unroll
      for (int e = 8; e < 128; ++e) m8[e & 7] = fmaxf(m8[e & 7], s[e]);
      const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      // The exponent's offset m moves only when the row's maximum exceeds it by
      // more than 8 (log2 units): until then p <= 2^8, which fp32 sums and bf16
      // operands hold as well as p <= 1, and the final division by the row sum
      // cancels whichever offset was used.  So O needs rescaling only on the
      // few tiles where some row of the warp moves m.
      const float m_tile = ct * mx;  // every row has a key: finite
      const bool upd = m_tile > m_run + 8.f;  // always on the first tile
      const float m_new = upd ? m_tile : m_run;
      const float alpha = ex2_fast(m_run - m_new);  // 1 without a move; 0 on the first tile
      // p = 2^(c_t x - m) as packed bf16 over S's first 64 columns (all of S is
      // in registers already); masked entries (-inf) give 0
      f2 s4[4] = {0ull, 0ull, 0ull, 0ull};  // the row sum in four independent chains
      const f2 c2 = dup2(ct), nm = dup2(-m_new), one = dup2(1.f);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pw[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float lo, hi;
          split2(fma2(mk2(s[32 * c + 2 * e], s[32 * c + 2 * e + 1]), c2, nm), lo, hi);
          const f2 pp = mk2(ex2_fast(lo), ex2_fast(hi));
          s4[e & 3] = fma2(pp, one, s4[e & 3]);
          pw[e] = bf_of_f2(pp);
        }
        umma::tmem_st16u(tS + 16 * c, pw);
      }
      l = fmaf(l, alpha, hsum2(s4[0]) + hsum2(s4[1]) + (hsum2(s4[2]) + hsum2(s4[3])));
      if (j > 0 && __any_sync(0xffffffffu, upd)) {  // O <- alpha O once MMA2_X(j - 1) is done
        attn_wait(&sh.bar_o[x], (j - 1) & 1, failed);
        const f2 al = dup2(alpha);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float ov[32];
          umma::tmem_ld2x16(tO + 32 * c, ov);
          f2 y2[16];
          pairs_of(ov, y2);
#pragma unroll
          for (int e = 0; e < 16; ++e) y2[e] = mul2(y2[e], al);
          floats_of(y2, ov);
          umma::tmem_st32(tO + 32 * c, ov);
        }
      }
      m_run = m_new;
      umma::tmem_wait_st();
      warp_arrive(&sh.bar_p[x], lane);
    }
    // epilogue: o = O / l, y = Norm(o) sigmoid(gate) over the gate tile in Q_X;
    // the last MMA2_X's completion covers every earlier one
    attn_wait(&sh.bar_o[x], qx & 1, failed);
    float o[128];
    tmem_ld128(tO, o);
    const float inv_l = 1.f / l;
    float s8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 128; ++e) {
      o[e] *= inv_l;
      s8[e & 7] = fmaf(o[e], o[e], s8[e & 7]);
    }
    const float ss = ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
    const float ro = rsqrtf(ss / (float)D + A.eps);
    const bool valid = q < A.T;
    if (A.o && valid) {
      float4 *o4 = reinterpret_cast<float4 *>(A.o + (((size_t)b * A.T + q) * A.Hq + h) * D);
#pragma unroll
      for (int u = 0; u < 32; ++u) o4[u] = make_float4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
    }
    attn_wait(&sh.bar_g[x], 0, failed);
    {
      unsigned char *G = base + x * TILE;
      const f2 r2 = dup2(ro), half = dup2(0.5f);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        uint4 *p = tile_at(G, i, c);
        f2 g[4], t[4];
        unpack4x2(*p, g);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float za, zb;  // sigmoid(z) = 0.5 + 0.5 tanh(z / 2)
          split2(mul2(g[e], half), za, zb);
          const f2 sg = fma2(mk2(tanh_fast(za), tanh_fast(zb)), half, half);
          t[e] = mul2(mul2(mk2(o[8 * c + 2 * e], o[8 * c + 2 * e + 1]), r2), sg);
        }
        *p = pack4x2(t);
      }
    }
    warp_arrive(&sh.bar_e[x], lane);
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
  A.npairs = (A.nqt + 1) / 2;
  tc::tc_attention_kernel<<<dim3(A.npairs, s->Hq, s->B), tc::kAttnThreads, tc::kAttnSmem, cs>>>(
      A, mq, mk, mv, mg, my);
  return cudaGetLastError() == cudaSuccess ? HLA_OK : HLA_ERR_CUDA;
}

}  // extern "C"
