// tc_proj.cu — the projections around the RNN mixer as tcgen05 GEMMs: bf16
// operands, fp32 accumulation in tensor memory (arXiv 2601.22156, Appendix A,
// Eq. 18, "RNN Layers").
//
//   projection in:  per head h, q = x W_q,h, k = x W_k,h, v = x W_v,h and the
//                   gate logit x W_z,h, all heads in one product, with the
//                   mixer's feature map fused into the epilogue: from the fp32
//                   q and k rows it writes q~ = RoPE(Norm(q)) and
//                   k~ = RoPE(Norm(k)) / sqrt(d) as fp16, 1/RMS(q), 1/RMS(k)
//                   and the fp32 q~ . k~ (the saved-feature layout of hla.h),
//                   and v and the gate logit as bf16.  Raw q and k never
//                   reach global memory.
//   projection out: out = u W_o^T, u the gated mixer rows of all heads side
//                   by side (bf16 out).
//
// Both are C[M, N] = A[M, K] W[N, K]^T with A and W row-major bf16 (W is a
// linear layer's output-feature-major weight).  One persistent CTA per SM walks
// output tiles of 128 x 256, N fastest (the CTAs running at once share their A
// rows, and W stays in L2).  K advances in blocks of 64 through a ring of
// kStages shared-memory stages, each an A tile (128 x 64) and a W tile
// (256 x 64) filled by TMA with the 128-byte swizzle that the MMA descriptors
// read.  Warp roles (12 warps, 384 threads):
//   warp 0, lane 0   TMA producer: fills stage s once the MMAs of the K block
//                    kStages earlier have read it (mbarrier `empty`)
//   warp 1           allocates the 512 TMEM columns; lane 0 issues the MMAs
//                    (M = 128, N = 256, K = 16, four per K block) into one of
//                    two 256-column fp32 accumulators, so the epilogue of tile
//                    i overlaps the MMAs of tile i + 1
//   warps 4..11      the epilogue: two warpgroups; thread (warp w, lane l) owns
//                    output row i = 32 (w % 4) + l, its TMEM lane
// Every wait is bounded: after the budget the thread records the failure in
// the status word and stops waiting, so a lost arrival never hangs the GPU.
#include "tc_common.cuh"

namespace hla {

namespace tc {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr int kATile = kBM * kBK * 2;    // 16 KiB
constexpr int kBTile = kBN * kBK * 2;    // 32 KiB
constexpr int kStageBytes = kATile + kBTile;
constexpr int kProjThreads = 384;
constexpr int kEpiWarp0 = 4;             // first epilogue warp
constexpr int kEpiWarps = 8;

struct ProjShared {
  uint64_t full[kStages];    // TMA -> MMA: stage s filled
  uint64_t empty[kStages];   // MMA -> TMA: stage s read (commit)
  uint64_t tfull[2];         // MMA -> epilogue: accumulator a complete (commit)
  uint64_t tempty[2];        // epilogue -> MMA: accumulator a drained (one arrive per warp)
  float red[2][2][3][kBM];   // projection in: [tile parity][warpgroup][sum][row] partial row sums
  uint32_t tmem_base;
};

constexpr size_t kProjSmem = kStages * kStageBytes + sizeof(ProjShared) + 1024;
static_assert(kProjSmem <= 232448, "projection GEMM exceeds 227 KiB of shared memory per CTA");

__device__ __forceinline__ void wait_bounded(uint64_t *bar, uint32_t parity, bool &failed) {
  if (!failed && !umma::mbar_wait(bar, parity)) failed = true;
  umma::fence_after();
}

// Four 16-column TMEM loads under one wait.
__device__ __forceinline__ void tmem_ld4x16(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            float (&x0)[16], float (&x1)[16], float (&x2)[16],
                                            float (&x3)[16]) {
  uint32_t r0[16], r1[16], r2[16], r3[16];
  umma::tmem_ld16_nowait(a0, r0);
  umma::tmem_ld16_nowait(a1, r1);
  umma::tmem_ld16_nowait(a2, r2);
  umma::tmem_ld16_nowait(a3, r3);
  umma::tmem_wait_ld();
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    x0[e] = __uint_as_float(r0[e]);
    x1[e] = __uint_as_float(r1[e]);
    x2[e] = __uint_as_float(r2[e]);
    x3[e] = __uint_as_float(r3[e]);
  }
}

// 128 fp32 columns of this thread's row from TMEM at taddr, as bf16, to dst
// (256 contiguous bytes).
__device__ __forceinline__ void store_row_bf16(uint32_t taddr, __nv_bfloat16 *dst, bool valid) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float x[32];
    umma::tmem_ld2x16(taddr + 32 * c, x);
    if (valid) {
      uint4 *d4 = reinterpret_cast<uint4 *>(dst + 32 * c);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        d4[u] = make_uint4(pack2(x[8 * u], x[8 * u + 1]), pack2(x[8 * u + 2], x[8 * u + 3]),
                           pack2(x[8 * u + 4], x[8 * u + 5]), pack2(x[8 * u + 6], x[8 * u + 7]));
    }
  }
}

// kQKVZ: the projection-in epilogue (N tile 2h: q | k of head h; 2h + 1: v | z);
// otherwise the plain bf16 epilogue of the projection out.
template <bool kQKVZ>
__global__ void __launch_bounds__(kProjThreads, 1)
    tc_proj_kernel(const __grid_constant__ ProjParams P, const __grid_constant__ CUtensorMap tma,
                   const __grid_constant__ CUtensorMap tmw) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  ProjShared &sh = *reinterpret_cast<ProjShared *>(base + kStages * kStageBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntiles = P.n_mt * P.n_nt;
  const int nk = P.K / kBK;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      umma::mbar_init(&sh.full[s], 1);
      umma::mbar_init(&sh.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      umma::mbar_init(&sh.tfull[a], 1);
      umma::mbar_init(&sh.tempty[a], kEpiWarps);
    }
    umma::mbar_fence_init();
  }
  if (warp == 1) umma::tmem_alloc(&sh.tmem_base, 512);
  sync_tc();
  const uint32_t tm = sh.tmem_base;
  bool failed = false;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int it = 0;
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int m0 = (tile / P.n_nt) * kBM, n0 = (tile % P.n_nt) * kBN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages;
          if (it >= kStages) wait_plain(&sh.empty[s], ((it / kStages) & 1) ^ 1, failed);
          if (failed) continue;
          unsigned char *st = base + s * kStageBytes;
          umma::mbar_expect_tx(&sh.full[s], kStageBytes);
          umma::tma_load_2d(st, &tma, kb * kBK, m0, &sh.full[s]);
          umma::tma_load_2d(st + kATile, &tmw, kb * kBK, n0, &sh.full[s]);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = umma::idesc_bf16(kBM, kBN, false, false);
      const uint32_t a0 = umma::smem_u32(base);
      int it = 0, i = 0;
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++i) {
        const int ab = i & 1;
        const uint32_t acc = tm + 256 * ab;
        // the fence after this wait orders the tile's MMAs after the epilogue's
        // reads of the accumulator; the stage waits need none (TMA data)
        if (i >= 2) wait_bounded(&sh.tempty[ab], ((i >> 1) - 1) & 1, failed);
        // K block kb from stage S: the four MMAs and the stage's release
        auto kblock = [&](int kb, int s, uint32_t par) {
          wait_plain(&sh.full[s], par, failed);
          if (failed) return;
          const uint32_t a = a0 + s * kStageBytes, w = a + kATile;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma::mma_ss(acc, umma::make_desc(a + 32 * kk, 16, 1024),
                         umma::make_desc(w + 32 * kk, 16, 1024), idesc, (kb | kk) ? 1u : 0u);
          umma::commit(&sh.empty[s]);
        };
        if (nk % kStages == 0) {
          // every tile starts at stage 0: stages as compile-time constants, so
          // each MMA's descriptors are loop-invariant (computing them between
          // MMAs holds the issuing thread behind the tensor pipe)
          for (int kb = 0; kb < nk; kb += kStages, it += kStages) {
            const uint32_t par = (it / kStages) & 1;
#pragma unroll
            for (int s = 0; s < kStages; ++s) kblock(kb + s, s, par);
          }
        } else {
          for (int kb = 0; kb < nk; ++kb, ++it) kblock(kb, it % kStages, (it / kStages) & 1);
        }
        if (!failed) umma::commit(&sh.tfull[ab]);
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - kEpiWarp0, grp = ew >> 2, sub = warp & 3;
    const int i_row = 32 * sub + lane;
    const uint32_t lane_base = (uint32_t)(32 * sub) << 16;
    int i = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++i) {
      const int ab = i & 1;
      const int m0 = (tile / P.n_nt) * kBM, nt = tile % P.n_nt;
      const int m = m0 + i_row;
      const bool valid = m < P.M;
      const uint32_t acc = tm + lane_base + 256 * ab;
      wait_bounded(&sh.tfull[ab], (i >> 1) & 1, failed);
      if (!kQKVZ) {
        // warpgroup grp: columns [128 grp, 128 grp + 128) of the tile
        const int n = nt * kBN + 128 * grp;
        store_row_bf16(acc + 128 * grp, reinterpret_cast<__nv_bfloat16 *>(P.out) + (size_t)m * P.N + n,
                       valid && n < P.N);
      } else {
        const int h = nt >> 1;
        const size_t row = ((size_t)m * P.H + h) * 128;  // [M, H, d]
        if (nt & 1) {
          // v (warpgroup 0) and the gate logit (warpgroup 1), bf16
          store_row_bf16(acc + 128 * grp, reinterpret_cast<__nv_bfloat16 *>(grp ? P.g : P.v) + row, valid);
        } else {
          // q in columns 0..127, k in 128..255.  Warpgroup grp takes RoPE pairs
          // [32 grp, 32 grp + 32): columns j and 64 + j of both.
          float sq = 0.f, sk = 0.f, sqk = 0.f;
#pragma unroll
          for (int pc = 0; pc < 2; ++pc) {
            const int j0 = 32 * grp + 16 * pc;
            float q0[16], q1[16], k0[16], k1[16];
            tmem_ld4x16(acc + j0, acc + 64 + j0, acc + 128 + j0, acc + 192 + j0, q0, q1, k0, k1);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              sq = fmaf(q0[e], q0[e], fmaf(q1[e], q1[e], sq));
              sk = fmaf(k0[e], k0[e], fmaf(k1[e], k1[e], sk));
              sqk = fmaf(q0[e], k0[e], fmaf(q1[e], k1[e], sqk));
            }
          }
          float(*red)[3][kBM] = sh.red[ab];
          red[grp][0][i_row] = sq;
          red[grp][1][i_row] = sk;
          red[grp][2][i_row] = sqk;
          named_sync(1, 32 * kEpiWarps);
          sq = red[0][0][i_row] + red[1][0][i_row];
          sk = red[0][1][i_row] + red[1][1][i_row];
          sqk = red[0][2][i_row] + red[1][2][i_row];
          const float rq = rsqrtf(sq / 128.f + P.eps), rk0 = rsqrtf(sk / 128.f + P.eps);
          const float rk = rk0 * P.kscale;
          const int b = m / P.T, t = m - b * P.T;
          if (grp == 0 && valid) {
            // [3, B, H, T]: 1/RMS(q), 1/RMS(k), q~ . k~ (RoPE rotates q and k by
            // the same angle, so it drops out of their dot product)
            const size_t plane = (size_t)(P.M / P.T) * P.H * P.T;
            const size_t si = ((size_t)b * P.H + h) * P.T + t;
            P.scal[si] = rq;
            P.scal[plane + si] = rk0;
            P.scal[2 * plane + si] = sqk * rq * rk;
          }
          const long long pos = P.pos_offset + t;
#pragma unroll
          for (int pc = 0; pc < 2; ++pc) {
            const int j0 = 32 * grp + 16 * pc;
            float q0[16], q1[16], k0[16], k1[16];
            tmem_ld4x16(acc + j0, acc + 64 + j0, acc + 128 + j0, acc + 192 + j0, q0, q1, k0, k1);
            uint32_t qlo[8], qhi[8], klo[8], khi[8];
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              float c0, s0, c1, s1;
              rope_fast(pos, P.rope_u[j0 + e], c0, s0);
              rope_fast(pos, P.rope_u[j0 + e + 1], c1, s1);
              // (x0, x1) -> (x0 c - x1 s, x0 s + x1 c), times the row's scale
              qlo[e / 2] = pack2h((q0[e] * c0 - q1[e] * s0) * rq, (q0[e + 1] * c1 - q1[e + 1] * s1) * rq);
              qhi[e / 2] = pack2h((q0[e] * s0 + q1[e] * c0) * rq, (q0[e + 1] * s1 + q1[e + 1] * c1) * rq);
              klo[e / 2] = pack2h((k0[e] * c0 - k1[e] * s0) * rk, (k0[e + 1] * c1 - k1[e + 1] * s1) * rk);
              khi[e / 2] = pack2h((k0[e] * s0 + k1[e] * c0) * rk, (k0[e + 1] * s1 + k1[e + 1] * c1) * rk);
            }
            if (valid) {
              __half *qt = reinterpret_cast<__half *>(P.qt) + row, *kt = reinterpret_cast<__half *>(P.kt) + row;
              uint4 *ql = reinterpret_cast<uint4 *>(qt + j0), *qh = reinterpret_cast<uint4 *>(qt + 64 + j0);
              uint4 *kl = reinterpret_cast<uint4 *>(kt + j0), *kh = reinterpret_cast<uint4 *>(kt + 64 + j0);
              ql[0] = make_uint4(qlo[0], qlo[1], qlo[2], qlo[3]);
              ql[1] = make_uint4(qlo[4], qlo[5], qlo[6], qlo[7]);
              qh[0] = make_uint4(qhi[0], qhi[1], qhi[2], qhi[3]);
              qh[1] = make_uint4(qhi[4], qhi[5], qhi[6], qhi[7]);
              kl[0] = make_uint4(klo[0], klo[1], klo[2], klo[3]);
              kl[1] = make_uint4(klo[4], klo[5], klo[6], klo[7]);
              kh[0] = make_uint4(khi[0], khi[1], khi[2], khi[3]);
              kh[1] = make_uint4(khi[4], khi[5], khi[6], khi[7]);
            }
          }
        }
      }
      // accumulator ab drained: the MMAs of tile i + 2 may overwrite it
      umma::fence_before();
      __syncwarp();
      if (lane == 0) umma::mbar_arrive(&sh.tempty[ab]);
    }
  }
  if (failed && P.err) atomicOr(P.err, 16u);
  sync_tc();
  if (warp == 1) umma::tmem_dealloc(tm, 512);
}

// 2-D map over a row-major bf16 [rows, cols] matrix with a box of 64 columns x
// box_rows rows, 128-byte swizzled (the MMA operand layout).  Out-of-range rows
// read as zeros.
cudaError_t make_map_2d(CUtensorMap *map, const void *ptr, long long rows, long long cols,
                        int box_rows) {
  EncodeFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  if (!ptr) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <bool kQKVZ>
cudaError_t run_proj(const ProjParams &P, const void *a, const void *w, cudaStream_t st) {
  CUtensorMap ma, mw;
  cudaError_t e;
  if ((e = make_map_2d(&ma, a, P.M, P.K, kBM)) != cudaSuccess) return e;
  if ((e = make_map_2d(&mw, w, P.N, P.K, kBN)) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc_proj_kernel<kQKVZ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kProjSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int ntiles = P.n_mt * P.n_nt;
  const int grid = ntiles < sms ? ntiles : sms;
  tc_proj_kernel<kQKVZ><<<grid, kProjThreads, kProjSmem, st>>>(P, ma, mw);
  return cudaGetLastError();
}

}  // namespace
}  // namespace tc

cudaError_t launch_proj_in(ProjParams &P, const void *x, const void *w, cudaStream_t st) {
  P.n_mt = ceil_div(P.M, tc::kBM);
  P.n_nt = ceil_div(P.N, tc::kBN);
  return tc::run_proj<true>(P, x, w, st);
}

cudaError_t launch_proj_out(ProjParams &P, const void *u, const void *w, cudaStream_t st) {
  P.n_mt = ceil_div(P.M, tc::kBM);
  P.n_nt = ceil_div(P.N, tc::kBN);
  return tc::run_proj<false>(P, u, w, st);
}

}  // namespace hla
