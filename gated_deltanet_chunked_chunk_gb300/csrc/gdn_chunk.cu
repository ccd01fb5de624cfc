// gdn_chunk.cu -- chunked prefill for sm_103a: a parallel per-chunk prep
// kernel followed by the serial state walk.
//
// Algorithm: the six steps of "NPU Training Operators - GDN", section
// "Operator semantics", with chunk size 64: chunk-local cumsum of g, beta K K^T
// with gate decay, triangular solve, w/u recompute, inter-chunk state
// propagation, output.  Steps 1-4 (and the h-independent half of step 6)
// depend on one chunk only, so they run in a separate, fully parallel kernel;
// only the state recurrence is serial.
//
// Notation for one chunk of one value head (rows i, j in [0, 64), L valid
// rows, gamma = cumsum g, rk / rq = 1/||k||, 1/||q|| (1 without the L2 norm),
// raw bf16 k, q, v; rows >= L behave as g = beta = k = q = v = 0):
//   A  = strictly-lower beta_i e^{gamma_i-gamma_j} rk_i rk_j (k_i.k_j)
//   P  = causal e^{gamma_i-gamma_j} rq_i rk_j (q_i.k_j)
//   T  = (I + A)^{-1}
//   W  = [T diag(beta e^gamma rk)] K          (w of the WY form, raw K)
//   Ts = (T - I) diag(beta)                   (so that u = beta v + Ts V)
// and, per 32-column slice of V with the state slice h:
//   v_new = u - W h
//   o     = scale (e^gamma rq (Q h) + P v_new)
//   h    <- e^{gamma_L} h + K^T diag(e^{gamma_L-gamma} rk) v_new
//
// gdn_chunk_prep (one CTA per (chunk, value head), four CTAs per SM): TMA loads
// K and Q; one thread issues tcgen05.mma for [K;Q][K;Q]^T (M = N = 128,
// 128B-swizzled smem operands, fp32 accumulator in TMEM), whose diagonal gives
// the row norms; A and P are built from TMEM; T by 16x16 diagonal-block
// substitution plus tf32 mma.sync for the off-diagonal blocks, in place; W by
// one more tcgen05 product.  The CTA writes one record [W | P hi | P lo | Ts^T |
// scalars] per (chunk, value head) to the workspace, laid out exactly as the
// walk kernel wants it in shared memory.
//
// gdn_chunk_walk (one CTA per (32-column slice, value head, sequence)): keeps
// the fp32 state slice in registers; a producer warp streams K, Q, a 64-column
// V box and the record into a two-stage ring with TMA / bulk copies; eight
// compute warps issue the serial chain's products on tcgen05 (TMEM
// accumulators, smem operands), W h, Ts V and K^T (s v_new), and run v_new,
// the state update and o in the epilogues; two more warps issue Q h and
// P v_new off the chain.  One long sequence is walked in up to four chunk
// ranges, each later range's prep running beside the previous range's walk.
//
// Precision: the main terms of o (P v_new and Q h) and the state update split
// their computed factor into bf16 hi + lo parts (the raw bf16 q, k, v are
// exact), and W h takes h as hi + lo too; W and Ts are plain bf16;
// accumulation is fp32, and h, A, T stay fp32.  Every mbarrier wait is bounded;
// on expiry a CTA records GDN_DEV_WAIT_TIMEOUT, drains its outstanding copies
// and leaves.
#include <cuda.h>
#include <string.h>

#include <mutex>

#include "gdn_chunk_shared.cuh"
#include "gdn_common.cuh"
#include "gdn_sm103.cuh"

namespace {

using namespace gdn;
using namespace gdnc;

constexpr int VT = 32;
constexpr int NW = 8;
constexpr int NTH = NW * 32;
constexpr int FROW = 68;                        // floats per padded fp32 row of 64

// [K; Q] tile as two TMA boxes per 64-key atom column: rows 0-63 K, 64-127 Q.
template <int K>
struct KQ {
  static constexpr int KA = K / 64;
  static constexpr int BYTES = KA * 16384;
};

__device__ __forceinline__ unsigned char *align1024(unsigned char *p) {
  return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}
// acc (16 x 16 as two 16x8 tiles) += A (16 x 16) * B (16 x 16), fp32 row-major in
// shared memory; fp32 bits go straight to the tf32 unit (low mantissa bits ignored).
__device__ __forceinline__ void mm16_tf32(const float *A, int lda, const float *B, int ldb, float acc[2][4], int g4,
                                          int t4) {
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    const uint32_t a0 = __float_as_uint(A[g4 * lda + 8 * ks + t4]);
    const uint32_t a1 = __float_as_uint(A[(g4 + 8) * lda + 8 * ks + t4]);
    const uint32_t a2 = __float_as_uint(A[g4 * lda + 8 * ks + t4 + 4]);
    const uint32_t a3 = __float_as_uint(A[(g4 + 8) * lda + 8 * ks + t4 + 4]);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const uint32_t b0 = __float_as_uint(B[(8 * ks + t4) * ldb + 8 * nt + g4]);
      const uint32_t b1 = __float_as_uint(B[(8 * ks + t4 + 4) * ldb + 8 * nt + g4]);
      asm volatile(
          "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
          "{%0,%1,%2,%3};"
          : "+f"(acc[nt][0]), "+f"(acc[nt][1]), "+f"(acc[nt][2]), "+f"(acc[nt][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
  }
}

// ============================================================== prep kernel
template <int K>
struct PrepLay {
  // The Q rows of the [K;Q] tile are dead once [K;Q][K;Q]^T has completed: the
  // bf16 T diag(beta e^g rk) tile and the fp32 scratch of the solve reuse them,
  // which keeps a CTA small enough for four per SM.
  static constexpr int OFF_KQ = 0;                              // [K;Q] tile
  static constexpr int OFF_TP = 8192;                           // T diag(beta e^g rk), bf16 SW128 (Q rows, atom 0)
  static constexpr int OFF_AT = KQ<K>::BYTES;                   // A then T, fp32 [64][FROW], in place
  static constexpr int OFF_X = K >= 128 ? 16384 + 8192          // 4 x [16][17] fp32 (Q rows, atom 1)
                                        : OFF_AT + 64 * FROW * 4;
  static constexpr int OFF_SC = K >= 128 ? OFF_AT + 64 * FROW * 4 : OFF_X + 4352;  // gl, bet, rk, rq, rowA, rowP, colf, ftp
  static constexpr int OFF_BAR = OFF_SC + 8 * 256;
  static constexpr int OFF_MISC = OFF_BAR + 16;
  static constexpr int BYTES = OFF_MISC + 16;
  // Staging of the record for bulk stores (K = 128; at K = 64 P and Ts^T are
  // stored directly): P hi and P lo in the two Q-row blocks (dead after the
  // first product, read back by the bulk copies before Tp and the solve's
  // scratch reuse them), Ts^T in the second Q-row block after the solve, and
  // W in the K rows of the tile once W = Tp K has completed.
  static constexpr int OFF_PH = 8192, OFF_PL = 16384 + 8192, OFF_TSS = 16384 + 8192;
  static_assert(K < 128 || (OFF_PH + 8192 <= 16384 && OFF_PL + 8192 <= OFF_AT && OFF_TSS + 8192 <= OFF_AT),
                "record staging inside the [K;Q] tile");
  static_assert(OFF_TP % 1024 == 0, "swizzled tile alignment");
  static_assert(4 * (BYTES + 1024 + 1024) <= 228 * 1024, "four CTAs per SM");
};
enum { PS_GL = 0, PS_BET = 1, PS_RK = 2, PS_RQ = 3, PS_RA = 4, PS_RP = 5, PS_CF = 6, PS_FTP = 7 };

// Raw gate inputs when the gating is fused into the prep (A_log == NULL: g and
// beta are given instead).
struct PrepGates {
  const float *A_log;
  const uint16_t *a, *b;
  const float *dt_bias;
  float *g_out, *beta_out;  // optional copies of the computed gates
};

template <int K>
__global__ void __launch_bounds__(NTH, 4) chunk_prep_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k, const float *__restrict__ g,
    const float *__restrict__ beta, const PrepGates gt, const int32_t *__restrict__ cu,
    const int32_t *__restrict__ cs, int N, int T, int H, int HV, int l2, unsigned char *__restrict__ ws,
    int32_t *dev_status, int slot0) {
  using Ly = PrepLay<K>;
  using R = Rec<K>;
  constexpr int KA = K / 64;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = align1024(smem_raw);
  const uint32_t sb = smem_u32(sm);
  // Value head fastest: the G value heads of a key head run side by side and
  // share the K, Q tile through L2.  The grid covers the chunk slots from slot0
  // on.
  const int gc = slot0 + static_cast<int>(blockIdx.x / HV), hv = static_cast<int>(blockIdx.x % HV);
  const int h = hv / (HV / H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g4 = lane >> 2, t4 = lane & 3;

  // Which sequence / chunk is this?
  int n = 0, c = 0;
  int64_t tok0 = 0, len = 0;
  if (!slot_chunk(cs, N, T, gc, n, c) || !seq_bounds(cu, n, T, tok0, len))
    return;  // past the last chunk (the grid is an upper bound)
  const int64_t rem = len - static_cast<int64_t>(c) * C;
  const int L = static_cast<int>(rem < C ? rem : C);
  const int64_t trow0 = tok0 + static_cast<int64_t>(c) * C;

  float *scal = reinterpret_cast<float *>(sm + Ly::OFF_SC);
  float *gl = scal + PS_GL * 64, *bet = scal + PS_BET * 64, *rk = scal + PS_RK * 64, *rq = scal + PS_RQ * 64;
  float *rowA = scal + PS_RA * 64, *rowP = scal + PS_RP * 64, *colf = scal + PS_CF * 64, *ftp = scal + PS_FTP * 64;
  float *AT = reinterpret_cast<float *>(sm + Ly::OFF_AT);
  float *Xs = reinterpret_cast<float *>(sm + Ly::OFF_X);
  // Every byte of the record the walk reads is written below: P, Ts^T and W
  // through shared-memory staging and bulk stores (P and Ts^T directly at
  // K = 64), the scalars directly.
  unsigned char *rec = ws + (static_cast<size_t>(gc) * HV + hv) * R::BYTES;
  float *rsc = reinterpret_cast<float *>(rec + R::SC);
  uint32_t *misc = reinterpret_cast<uint32_t *>(sm + Ly::OFF_MISC);
  const uint32_t b_tma = sb + Ly::OFF_BAR, b_mma = sb + Ly::OFF_BAR + 8;
  const uint32_t kq = sb + Ly::OFF_KQ;

  if (tid == 0) {
    mbar_init(b_tma, 1);
    mbar_init(b_mma, 1);
    misc[1] = 0;
    mbar_fence_init();
    // The loads go out first: they overlap the TMEM allocation and the gates.
    mbar_arrive_expect_tx(b_tma, KQ<K>::BYTES);
#pragma unroll
    for (int a = 0; a < KA; ++a) {
      tma_load_3d(kq + a * 16384, &tm_k, b_tma, 64 * a, h, static_cast<int>(trow0));
      tma_load_3d(kq + a * 16384 + 8192, &tm_q, b_tma, 64 * a, h, static_cast<int>(trow0));
    }
  }
  if (warp == 0) tmem_alloc(sb + Ly::OFF_MISC, 128);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  // Gates (rows >= L read as 0) and their chunk-local cumsum in base 2 (warp 4).
  // Fused gating follows FastDeploy PR "support fla triton kernel for qwen3.5",
  // Usage section 5: g = -e^{A_log} softplus(a + dt_bias), beta = sigmoid(b).
  if (warp == 4) {
    float x[2], bb[2];
    const float na = gt.A_log ? -expf(gt.A_log[hv]) : 0.f;
    const float db = gt.A_log ? gt.dt_bias[hv] : 0.f;
#pragma unroll
    for (int u2 = 0; u2 < 2; ++u2) {
      const int r = 2 * lane + u2;
      const int64_t gi = (trow0 + r) * HV + hv;
      x[u2] = 0.f;
      bb[u2] = 0.f;
      if (r < L) {
        if (gt.A_log) {
          x[u2] = na * softplus_fast(bf2f(gt.a[gi]) + db);  // as gdn_gating computes them
          bb[u2] = sigmoid_fast(bf2f(gt.b[gi]));
          if (gt.g_out) {
            gt.g_out[gi] = x[u2];
            gt.beta_out[gi] = bb[u2];
          }
        } else {
          x[u2] = g[gi];
          bb[u2] = beta[gi];
        }
      }
    }
    bet[2 * lane] = bb[0];
    bet[2 * lane + 1] = bb[1];
    float sum = x[0] + x[1];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, sum, off);
      if (lane >= off) sum += y;
    }
    const float excl = sum - (x[0] + x[1]);
    gl[2 * lane] = (excl + x[0]) * kLog2e;
    gl[2 * lane + 1] = sum * kLog2e;
  }
  bool ok = true;
  if (tid == 0) {
    ok = mbar_wait_bounded(b_tma, 0, kWaitLimit);
    if (ok) {
      tc_fence_after();
      constexpr uint32_t idesc = umma_idesc_bf16(128, 128);
#pragma unroll
      for (int kk = 0; kk < K / 16; ++kk) {
        const uint64_t d = umma_desc_sw128(kq + (kk >> 2) * 16384 + (kk & 3) * 32);
        umma_bf16(tmem, d, d, idesc, kk > 0 ? 1u : 0u);
      }
      umma_commit(b_mma);
      ok = mbar_wait_bounded(b_mma, 0, kWaitLimit);
    }
    if (!ok) {
      misc[1] = 1;
      set_status(dev_status, GDN_DEV_WAIT_TIMEOUT);
    }
  }
  __syncthreads();
  if (misc[1]) {
    if (warp == 0) tmem_dealloc(tmem, 128);
    return;
  }
  tc_fence_after();

  // Row norms from the diagonal of [K;Q][K;Q]^T; this thread's 32 columns.
  const int quad = warp & 3, half = warp >> 2;
  const int row = 32 * quad + lane;
  float vals[32];
  {
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * quad) << 16);
    tmem_ld32(tl + half * 32, vals);
    if (l2) {
      const bool kdiag = (quad < 2) && (half == quad);
      const bool qdiag = (warp == 2) || (warp == 7);
      if (kdiag || qdiag) {
        float d = vals[0];
        if (kdiag) {
#pragma unroll
          for (int m = 1; m < 32; ++m) d = (lane == m) ? vals[m] : d;
        } else {
          // The Q Q^T diagonal, 16 columns at a time (fewer live registers).
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            uint32_t dv[16];
            tmem_ld16_issue(tl + 64 + 32 * (quad - 2) + 16 * p, dv);
            tmem_ld_wait16(dv);
#pragma unroll
            for (int m = 0; m < 16; ++m) d = (lane == 16 * p + m) ? __uint_as_float(dv[m]) : d;
          }
        }
        const float rn = rsqrtf(d + GDN_L2_EPS);
        if (kdiag) rk[row] = rn; else rq[row - 64] = rn;
      }
    } else if (tid < 64) {
      rk[tid] = 1.f;
      rq[tid] = 1.f;
    }
  }
  tc_fence_before();
  __syncthreads();  // every read of [K;Q][K;Q]^T from TMEM is done: W reuses the columns

  // Per-row factors; the decay e^{gamma_i-gamma_j} is factored when the chunk's
  // total decay fits the fp32 range, else taken element by element.
  const bool fact = (gl[0] - gl[63]) < 120.f;
  if (tid < 64) {
    const float gi = gl[tid];
    const float e = ex2(gi);
    const float er = ex2(gi - gl[0]);
    rsc[RS_OG + tid] = e * rq[tid];
    rsc[RS_SV + tid] = ex2(gl[63] - gi) * rk[tid];
    rsc[RS_BET + tid] = bet[tid];
    ftp[tid] = bet[tid] * e * rk[tid];
    rowA[tid] = bet[tid] * rk[tid] * er;
    rowP[tid] = rq[tid] * er;
    colf[tid] = fact ? rk[tid] * ex2(gl[0] - gi) : 0.f;
    if (tid == 0) rsc[RS_DL] = ex2(gl[63]);
  }
  __syncthreads();

  // A (fp32, only j < i stored: the solve reads nothing else) and P (bf16 hi + lo).
  if (row < 64) {
    const int i = row;
    const float ra = rowA[i], gi = gl[i], ci = bet[i] * rk[i];
    const bool live = i < L;
#pragma unroll
    for (int q4 = 0; q4 < 8; ++q4) {
      const int j0 = half * 32 + 4 * q4;
      if (j0 < i) {
        float a4[4];
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
          const int j = j0 + u4;
          const float x = vals[4 * q4 + u4];
          const float a = fact ? ra * colf[j] * x : ci * rk[j] * ex2(gi - gl[j]) * x;
          a4[u4] = (live && j < i) ? a : 0.f;
        }
        *reinterpret_cast<float4 *>(AT + i * FROW + j0) = make_float4(a4[0], a4[1], a4[2], a4[3]);
      }
    }
  } else {
    const int i = row - 64;
    const float rp = rowP[i], gi = gl[i], ci = rq[i];
    const bool live = i < L;
#pragma unroll
    for (int q8 = 0; q8 < 4; ++q8) {
      const int j0 = half * 32 + q8 * 8;
      uint4 vh = make_uint4(0, 0, 0, 0), vl = make_uint4(0, 0, 0, 0);
      if (live && j0 <= i) {
        uint32_t ph[4], pl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float pv[2];
#pragma unroll
          for (int u2 = 0; u2 < 2; ++u2) {
            const int j = j0 + 2 * e + u2;
            const float x = vals[q8 * 8 + 2 * e + u2];
            const float p = fact ? rp * colf[j] * x : ci * rk[j] * ex2(gi - gl[j]) * x;
            pv[u2] = (j <= i) ? p : 0.f;
          }
          ph[e] = pack_bf16(pv[0], pv[1]);
          pl[e] = pack_bf16(pv[0] - bf16lo_f(ph[e]), pv[1] - bf16hi_f(ph[e]));
        }
        vh = make_uint4(ph[0], ph[1], ph[2], ph[3]);
        vl = make_uint4(pl[0], pl[1], pl[2], pl[3]);
      }
      const int chunk = half * 4 + q8;
      if constexpr (K >= 128) {
        *reinterpret_cast<uint4 *>(sm + Ly::OFF_PH + sw128(i, chunk)) = vh;
        *reinterpret_cast<uint4 *>(sm + Ly::OFF_PL + sw128(i, chunk)) = vl;
      } else {
        *reinterpret_cast<uint4 *>(rec + R::PH + sw128(i, chunk)) = vh;
        *reinterpret_cast<uint4 *>(rec + R::PL + sw128(i, chunk)) = vl;
      }
    }
  }
  if constexpr (K >= 128) fence_proxy_async_smem();  // P, for the bulk copies
  __syncthreads();
  if constexpr (K >= 128) {
    if (tid == 0) {
      bulk_store(rec + R::PH, sb + Ly::OFF_PH, 8192);
      bulk_store(rec + R::PL, sb + Ly::OFF_PL, 8192);
      bulk_commit();
    }
  }

  // T = (I + A)^{-1}, in place.  Diagonal 16x16 blocks: warps 0-3, lanes 0-15,
  // one column each (right-looking substitution).  Warps 4-7 zero the K rows
  // >= L (they multiply zero columns of the next products).
  if (warp < 4) {
    const int b0 = 16 * warp, col = lane & 15;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (i == col) ? 1.f : 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
#pragma unroll
      for (int i = j + 1; i < 16; ++i) x[i] = fmaf(-AT[(b0 + i) * FROW + b0 + j], x[j], x[i]);
    __syncwarp();
    if (lane < 16) {
#pragma unroll
      for (int i = 0; i < 16; ++i) AT[(b0 + i) * FROW + b0 + col] = x[i];
    }
  } else if (L < C) {
    for (int e = tid - 128; e < (C - L) * 8 * KA; e += 128) {
      const int zr = L + e / (8 * KA), kc = e % (8 * KA);
      *reinterpret_cast<uint4 *>(sm + Ly::OFF_KQ + (kc >> 3) * 16384 + sw128(zr, kc & 7)) = make_uint4(0, 0, 0, 0);
    }
  }
  if constexpr (K >= 128) {
    if (tid == 0) bulk_wait_read();  // the solve's scratch and Tp reuse P's staging
  }
  __syncthreads();
  {
    auto blk = [&](int bi, int bj) { return AT + 16 * bi * FROW + 16 * bj; };
    auto store_c = [&](float *dst, int ld, float acc[2][4], float sgn) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        dst[g4 * ld + 8 * nt + 2 * t4] = sgn * acc[nt][0];
        dst[g4 * ld + 8 * nt + 2 * t4 + 1] = sgn * acc[nt][1];
        dst[(g4 + 8) * ld + 8 * nt + 2 * t4] = sgn * acc[nt][2];
        dst[(g4 + 8) * ld + 8 * nt + 2 * t4 + 1] = sgn * acc[nt][3];
      }
    };
    // T10 = -D1 (A10 D0), T32 = -D3 (A32 D2)
    if (warp < 2) {
      const int bj = 2 * warp, bi = bj + 1;
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      mm16_tf32(blk(bi, bj), FROW, blk(bj, bj), FROW, acc, g4, t4);
      float *X = Xs + warp * 272;
      store_c(X, 17, acc, 1.f);
      __syncwarp();
      float tt[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      mm16_tf32(blk(bi, bi), FROW, X, 17, tt, g4, t4);
      __syncwarp();
      store_c(blk(bi, bj), FROW, tt, -1.f);
    }
    __syncthreads();
    // Y = A[32:64, 0:32] T11, with T11 = [[D0, 0], [T10, D1]]
    if (warp < 4) {
      const int a = warp >> 1, b = warp & 1;
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      for (int kb = b; kb < 2; ++kb) mm16_tf32(blk(2 + a, kb), FROW, blk(kb, b), FROW, acc, g4, t4);
      store_c(Xs + warp * 272, 17, acc, 1.f);
    }
    __syncthreads();
    // T[32:64, 0:32] = -T22 Y, with T22 = [[D2, 0], [T32, D3]]
    if (warp < 4) {
      const int a = warp >> 1, b = warp & 1;
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      for (int kb = 0; kb <= a; ++kb) mm16_tf32(blk(2 + a, 2 + kb), FROW, Xs + (2 * kb + b) * 272, 17, acc, g4, t4);
      store_c(blk(2 + a, b), FROW, acc, -1.f);
    }
    __syncthreads();
  }

  // Tp = T diag(beta e^gamma rk) (j <= i, for W), bf16 SW128 in shared memory.
  for (int e = tid; e < 64 * 8; e += NTH) {
    const int i = e >> 3, ch = e & 7;
    uint4 tpv = make_uint4(0, 0, 0, 0);
    if (8 * ch <= i) {
      const float4 t0 = *reinterpret_cast<const float4 *>(AT + i * FROW + 8 * ch);
      const float4 t1 = *reinterpret_cast<const float4 *>(AT + i * FROW + 8 * ch + 4);
      const float4 f0 = *reinterpret_cast<const float4 *>(ftp + 8 * ch);
      const float4 f1 = *reinterpret_cast<const float4 *>(ftp + 8 * ch + 4);
      const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
      const float fv[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
      uint32_t tp[4];
#pragma unroll
      for (int q2 = 0; q2 < 4; ++q2) {
        float a2[2];
#pragma unroll
        for (int u2 = 0; u2 < 2; ++u2) {
          const int jj = 2 * q2 + u2, j = 8 * ch + jj;
          a2[u2] = (j <= i) ? tv[jj] * fv[jj] : 0.f;
        }
        tp[q2] = pack_bf16(a2[0], a2[1]);
      }
      tpv = make_uint4(tp[0], tp[1], tp[2], tp[3]);
    }
    *reinterpret_cast<uint4 *>(sm + Ly::OFF_TP + sw128(i, ch)) = tpv;
  }
  // W = Tp K (64 x K) on tcgen05: A = Tp (K-major, its rows 64-127 whatever
  // follows the tile: those accumulator lanes are not read), B = the K rows of
  // the [K;Q] tile as an MN-major operand (keys contiguous, 64-key atoms 16 KB
  // apart), fp32 accumulator in the TMEM columns of the first product.  It runs
  // while the threads build Ts^T, whose staging block (the Q rows of the second
  // atom) neither operand reads.  The warps of TMEM lanes 0-63 then turn it
  // into the record's bf16 W, one row and 64 keys per thread, staged in the K
  // rows for two bulk stores.
  fence_proxy_async_smem();  // Tp and the zeroed K rows, for the async proxy
  __syncthreads();
  if (tid == 0) {
    tc_fence_after();
    constexpr uint32_t idw = umma_idesc_bf16(128, K, 0, 1);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      umma_bf16(tmem, umma_desc_sw128(sb + Ly::OFF_TP + kk * 32), umma_desc_sw128_mn(kq + kk * 2048, 16384), idw,
                kk > 0 ? 1u : 0u);
    umma_commit(b_mma);
  }
  // Ts = (T - I) diag(beta) (j < i), written transposed (row j holds column j
  // of Ts): the MN-major A operand of the walk's u = Ts V product.  A warp
  // takes 32 consecutive columns j, so its reads of T hit distinct banks.
  for (int e = tid; e < 64 * 8; e += NTH) {
    const int j = e & 63, ich = e >> 6;
    const float bj = bet[j];
    uint32_t w[4];
#pragma unroll
    for (int q2 = 0; q2 < 4; ++q2) {
      float v2[2];
#pragma unroll
      for (int u2 = 0; u2 < 2; ++u2) {
        const int i = 8 * ich + 2 * q2 + u2;
        v2[u2] = (j < i) ? AT[i * FROW + j] * bj : 0.f;
      }
      w[q2] = pack_bf16(v2[0], v2[1]);
    }
    if constexpr (K >= 128)
      *reinterpret_cast<uint4 *>(sm + Ly::OFF_TSS + sw128(j, ich)) = make_uint4(w[0], w[1], w[2], w[3]);
    else
      *reinterpret_cast<uint4 *>(rec + R::TS + sw128(j, ich)) = make_uint4(w[0], w[1], w[2], w[3]);
  }

  if constexpr (K >= 128) fence_proxy_async_smem();  // Ts^T, for the bulk copy
  __syncthreads();
  if (tid == 0) {
    if constexpr (K >= 128) {
      bulk_store(rec + R::TS, sb + Ly::OFF_TSS, 8192);
      bulk_commit();
    }
    if (!mbar_wait_bounded(b_mma, 1, kWaitLimit)) {
      misc[1] = 1;
      set_status(dev_status, GDN_DEV_WAIT_TIMEOUT);
    }
  }
  __syncthreads();
  if (!misc[1] && (warp & 3) < 2 && (warp >> 2) < KA) {
    tc_fence_after();
    const int i = 32 * (warp & 3) + lane, a = warp >> 2;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + 64 * a;
    unsigned char *wrow = sm + Ly::OFF_KQ + a * 16384;  // the K rows of atom a: dead now
    // Two 16-column loads in flight per round trip.
#pragma unroll
    for (int q8 = 0; q8 < 2; ++q8) {
      uint32_t x[2][16];
      tmem_ld16_issue(tl + 32 * q8, x[0]);
      tmem_ld16_issue(tl + 32 * q8 + 16, x[1]);
      tmem_ld_wait16(x[0]);
      tmem_ld_wait16(x[1]);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w[e] = pack_bf16(__uint_as_float(x[c4 >> 1][8 * (c4 & 1) + 2 * e]),
                           __uint_as_float(x[c4 >> 1][8 * (c4 & 1) + 2 * e + 1]));
        *reinterpret_cast<uint4 *>(wrow + sw128(i, 4 * q8 + c4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    fence_proxy_async_smem();  // W, for the bulk copies
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
  if (tid == 0) {
    if (!misc[1]) {
#pragma unroll
      for (int a = 0; a < KA; ++a) bulk_store(rec + R::W + a * 8192, sb + Ly::OFF_KQ + a * 16384, 8192);
      bulk_commit();
    }
    // Shared memory must outlive the copies' reads of it; their global writes
    // are performed before the grid completes, which orders them before the
    // walk on the stream.
    bulk_wait_read();
  }
}

// ============================================================== walk kernel
// Eleven warps.  Every product runs on tcgen05 with fp32 accumulators in TMEM.
// A thread needs about 100 cycles to issue one tcgen05.mma while issues from
// different warps overlap, and every wait on an mbarrier costs several hundred
// cycles while the tensor core and TMA keep shared memory busy; so the serial
// products are split over several issuing warps into partial accumulators
// that the epilogues add up, the products off the serial chain are issued by
// warps of their own, and completions that are always needed together share
// one barrier.
//
// Products whose rows are the chunk's 64 tokens use M = 64.  Row i of such an
// accumulator sits in TMEM lane 32 (i / 16) + i % 16, so each of the four lane
// quarters holds 16 rows and the token-row epilogues run on all four SM
// sub-partitions (an M = 128 accumulator would put them in lanes 0-63, which
// only two of them reach).
//  * Compute warps 0-7.  Token-row work: thread t of warp w takes row
//    16 (w & 3) + t % 16 and the 8 columns 16 (w >> 2) + 8 (t / 16) .. + 7 of
//    the slice's 32.  State work: the thread owns TMEM lane r = 32 (w & 3) + t
//    (key r) and the 16 columns 16 (w >> 2) .. + 15, and holds the fp32 state
//    h[r][16 columns] in registers.  Per chunk c:
//      W [h_hi | h_lo] -> ACC1 (4 partials, warps 0-3) and u(c) = Ts V -> ACC4
//      (warp 7, on the SM sub-partition no other issuing warp uses); meanwhile
//      the output of chunk c - 1;
//      v_new = beta v + u - W h -> s v_new, v_new (bf16 hi | lo);
//      K^T [s v_new hi | lo] -> ACC2 (2 partials, warps 0-1);
//      h <- e^{gamma_L} h + ACC2, written back as [h_hi | h_lo], and
//      e^gamma rq (Q h) of chunk c from ACCQ into registers for its output.
//  * Warp 8: TMA / bulk loads of chunk c + 2 into the stage chunk c released.
//  * Warps 9 and 10, off the serial chain: Q [h_hi | h_lo] -> ACCQ (warp 9,
//    once W h is done), then P_hi [v_new hi | lo] -> ACC3 (warp 9) and
//    P_lo [v_new hi | lo] -> ACC3L (warp 10) once the state product is done.
template <int K>
struct WalkLay {
  static constexpr int KA = K / 64;
  static constexpr int KT = 0;                           // K tile [token][key], KA x 8 KB (TMA)
  static constexpr int WQ = KT + KA * 8192;              // [W; Q], KA x 16 KB (W: record, Q: TMA)
  static constexpr int VB = WQ + KA * 16384;             // V [token][64 columns] SW128 (TMA)
  static constexpr int RR = VB + 8192;                   // record from P hi on: PH | PL | TS | SC
  static constexpr int RR_BYTES = Rec<K>::BYTES - Rec<K>::PH;
  static constexpr int STAGE = RR + RR_BYTES;
  static constexpr int NS = 2;
  static constexpr int OFF_H = NS * STAGE;               // [K][64] bf16 (h hi | h lo), MN-major SW128
  static constexpr int OFF_VS = OFF_H + K * 128;         // [64][64] bf16 (s v_new hi | lo), MN-major SW128
  static constexpr int OFF_VN = OFF_VS + 8192;           // [64][64] bf16 (v_new hi | lo), MN-major SW128
  static constexpr int OFF_Z = OFF_VN + 8192;            // 8 KB of zeros: keys 64-127 of the state product for K = 64
  static constexpr int OFF_BAR = OFF_Z + 8192;
  static constexpr int NBAR = 12;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr uint32_t TX = STAGE;                  // every byte of a stage is loaded per chunk
  // TMEM columns: ACC1 four M = 64 partials of 64 columns; ACC2 (M = 128, two
  // partials) reuses ACC1's first two, which the v_new epilogue has read before
  // the state product is issued; ACC3, ACC3L, ACC4 and ACCQ one M = 64 block each.
  static constexpr uint32_t ACC1 = 0, ACC2 = 0, ACC3 = 256, ACC3L = 320, ACC4 = 384, ACCQ = 448;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(STAGE % 1024 == 0 && OFF_H % 1024 == 0 && OFF_VS % 1024 == 0 && OFF_Z % 1024 == 0,
                "swizzled tile alignment");
  static_assert(BYTES + 1024 <= 232448, "shared memory budget (227 KB per CTA)");
};
constexpr int WALK_COMPUTE = 256;
constexpr int WALK_THREADS = WALK_COMPUTE + 96;

template <int K>
__global__ void __launch_bounds__(WALK_THREADS, 1) chunk_walk_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, float scale, const float *__restrict__ h0,
    const int32_t *__restrict__ cu, int T, int H, int HV, int V, const unsigned char *__restrict__ ws,
    uint16_t *__restrict__ o, float *__restrict__ ht, float *__restrict__ hsave, const int32_t *__restrict__ cs,
    int32_t *dev_status, int force_expiry, int c_begin, int c_end) {
  using Ly = WalkLay<K>;
  using R = Rec<K>;
  // A kernel launched as this grid's programmatic dependent (the next range's
  // prep) may start once every CTA of this grid is resident; it reads nothing
  // this grid writes.  Without such a dependent this does nothing.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int KA = K / 64;
  constexpr int NS = Ly::NS;
  constexpr int TSO = Ly::RR + (R::TS - R::PH);          // Ts^T within a stage
  constexpr int SCO = Ly::RR + (R::SC - R::PH);          // scalars within a stage
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = align1024(smem_raw);
  const uint32_t sb = smem_u32(sm);
  const int vt0 = blockIdx.x * VT, hv = blockIdx.y, n = blockIdx.z;
  const int vhalf = vt0 & 32;                            // this slice within its 64-column V box
  const int h = hv / (HV / H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  int64_t tok0, len;
  if (!seq_bounds(cu, n, T, tok0, len)) {
    if (tid == 0) set_status(dev_status, GDN_DEV_BAD_CU_SEQLENS);
    return;
  }
  int64_t cb = chunk_base(cs, n, T);
  {
    // This launch walks chunks [c_begin, c_end) of the sequence, starting from
    // the state h0 and leaving the state after its last chunk in ht: chunk c
    // below is chunk c_begin + c of the sequence.
    const int64_t skip = c_begin < chunks_of(len) ? c_begin : chunks_of(len);
    tok0 += skip * C;
    len -= skip * C;
    cb += skip;
  }
  const int NC = chunks_of(len) < c_end - c_begin ? chunks_of(len) : c_end - c_begin;
  uint32_t *misc = reinterpret_cast<uint32_t *>(sm + Ly::OFF_MISC);
  volatile uint32_t *abort_flag = misc + 1;
  // Two-slot barriers, slot c & 1 serving chunk c:
  //   FULL(c):  the loads of chunk c landed (the producer's arrive with the
  //             byte count; nothing else, so that a drain after an abort
  //             waits for the copies alone);
  //   OUT(c):   the two output products of chunk c are done (the commits of
  //             warps 9 and 10);
  //   CDONE(c): no warp and no product but the output products (which OUT(c)
  //             covers) reads chunk c's stage any more.
  // Single-slot: M1 (phase c: u(c) and the four parts of W h of chunk c are
  // done), M2 (phase c: K^T (s v_new) of chunk c is done) and QD (phase c:
  // Q h of chunk c is done).
  enum { FULL = 0, CDONE = 1 };
  auto bar = [&](int kind, int b) { return sb + Ly::OFF_BAR + 8 * (2 * kind + b); };
  const uint32_t b_m1 = sb + Ly::OFF_BAR + 32, b_m2 = sb + Ly::OFF_BAR + 40, b_drain = sb + Ly::OFF_BAR + 48;
  const uint32_t b_never = sb + Ly::OFF_BAR + 56;  // nothing arrives: the testing hook's wait
  const uint32_t b_qd = sb + Ly::OFF_BAR + 64;
  auto b_out = [&](int c) { return sb + Ly::OFF_BAR + 72 + 8 * (c & 1); };
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(FULL, b), 1);
      mbar_init(bar(CDONE, b), 1);
      mbar_init(sb + Ly::OFF_BAR + 72 + 8 * b, 2);
    }
    mbar_init(b_m1, 5);
    mbar_init(b_m2, 2);
    mbar_init(b_drain, 7);
    mbar_init(b_never, 1);
    mbar_init(b_qd, 1);
    misc[1] = 0;
    mbar_fence_init();
  }
  for (int e = tid; e < 8192 / 16; e += WALK_THREADS)
    reinterpret_cast<uint4 *>(sm + Ly::OFF_Z)[e] = make_uint4(0, 0, 0, 0);
  if (warp == 0) tmem_alloc(sb + Ly::OFF_MISC, Ly::TMEM_COLS);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  // Bounded wait; lane 0 polls and the result is warp-uniform.  After an
  // expired wait every later wait of this warp returns false at once (loops
  // run to their end without work but still pass every named barrier).  A
  // wait also gives up once another warp has recorded an abort in the shared
  // flag (read every 64 polls only: reading it on every poll would queue
  // behind the TMA traffic).
  bool dead = false;
  auto waitl = [&](uint32_t b, uint32_t parity, long long limit) -> bool {
    uint32_t ok = 0;
    if (lane == 0 && !dead) {
      const long long t0 = clock64();
      for (int it = 1;; ++it) {
        if (mbar_try_wait(b, parity)) { ok = 1; break; }
        if ((it & 63) == 0) {
          if (*abort_flag) break;
          if (clock64() - t0 > limit) { *abort_flag = 1; break; }
        }
      }
    }
    __syncwarp();
    ok = __shfl_sync(0xffffffffu, ok, 0);
    dead = dead || !ok;
    return ok != 0;
  };
  auto waitb = [&](uint32_t b, uint32_t parity) { return waitl(b, parity, kWaitLimit); };
  auto waitc = [&](int kind, int c) { return waitb(bar(kind, c & 1), (c >> 1) & 1); };
  auto wait_out = [&](int c) { return waitb(b_out(c), (c >> 1) & 1); };
  auto chunk_rows = [&](int c) {
    const int64_t rem = len - static_cast<int64_t>(c) * C;
    return static_cast<int>(rem < C ? rem : C);
  };
  const int64_t sbase = (static_cast<int64_t>(n) * HV + hv) * K;

  if (warp < 8) {
    // ------------------------------------------------------- compute warps
    const int q4 = warp & 3;                             // TMEM lane quarter
    const int hs = warp >> 2;                            // column half of the state work
    const int r = 32 * q4 + lane;                        // state work: TMEM lane, key r
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    const bool krow = r < K;
    const int ti = 16 * q4 + (lane & 15);                // token-row work: row ti, columns tc .. tc + 7
    const int tc = 16 * hs + 8 * (lane >> 4);
    float hr[16], qh[8];
#pragma unroll
    for (int j = 0; j < 16; ++j) hr[j] = (h0 && krow) ? h0[(sbase + r) * V + vt0 + 16 * hs + j] : 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) qh[j] = 0.f;
    // Row r of h -> columns [16 hs, 16 hs + 16) of the hi and lo halves of the
    // MN-major SW128 H tile.
    auto write_h = [&]() {
      if (!krow) return;
      unsigned char *row = sm + Ly::OFF_H + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = hr[8 * m + 2 * e], x1 = hr[8 * m + 2 * e + 1];
          hi[e] = pack_bf16(x0, x1);
          lo[e] = pack_bf16(x0 - bf16lo_f(hi[e]), x1 - bf16hi_f(hi[e]));
        }
        const int chh = 2 * hs + m;
        *reinterpret_cast<uint4 *>(row + ((chh ^ (r & 7)) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(row + (((4 + chh) ^ (r & 7)) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    };
    // Output of chunk c for row ti, columns tc .. tc + 7: ACC3 holds
    // P_hi [v_new hi | lo], ACC3L P_lo [v_new hi | lo] (of which the v_new hi
    // block is used), qh the e^gamma rq Q h of chunk c; the caller has seen
    // both output products complete.
    auto output = [&](int c, bool go) {
      if (go) {
        tc_fence_after();
        uint32_t a[8], b[8], l[8];
        tmem_ld8x2_issue(tl + Ly::ACC3 + 16 * hs, a);
        tmem_ld8x2_issue(tl + Ly::ACC3 + 32 + 16 * hs, b);
        tmem_ld8x2_issue(tl + Ly::ACC3L + 16 * hs, l);
        tmem_ld_wait8(a);
        tmem_ld_wait8(b);
        tmem_ld_wait8(l);
        if (o && ti < chunk_rows(c)) {
          const int64_t trow = tok0 + static_cast<int64_t>(c) * C + ti;
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 2 * e;
            w[e] = pack_bf16(scale * (qh[j] + (__uint_as_float(a[j]) + __uint_as_float(b[j])) + __uint_as_float(l[j])),
                             scale * (qh[j + 1] + (__uint_as_float(a[j + 1]) + __uint_as_float(b[j + 1])) +
                                      __uint_as_float(l[j + 1])));
          }
          *reinterpret_cast<uint4 *>(o + (trow * HV + hv) * V + vt0 + tc) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      return go;
    };
    // u(c) = Ts V into ACC4 (M = 64), completing on phase c of M1; Ts^T is
    // the MN-major A operand.
    auto issue_u = [&](int c) {
      const int s = c % NS;
      const uint32_t st = sb + s * Ly::STAGE;
      tc_fence_after();
      constexpr uint32_t id4 = umma_idesc_bf16(64, 64, 1, 1);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t a = umma_desc_sw128_mn(st + TSO + kk * 2048, 8192);
        const uint64_t b = umma_desc_sw128_mn(st + Ly::VB + kk * 2048, 8192);
        umma_bf16(tmem + Ly::ACC4, a, b, id4, kk > 0 ? 1u : 0u);
      }
      umma_commit(b_m1);
    };
    write_h();
    fence_proxy_async_smem();
    named_bar_sync(1, WALK_COMPUTE);
    bool go = true;
    for (int c = 0; c < NC; ++c) {
      const int s = c % NS;
      const uint32_t st = sb + s * Ly::STAGE;
      const unsigned char *stp = sm + s * Ly::STAGE;
      const float *rsc = reinterpret_cast<const float *>(stp + SCO);
      if (hsave && krow) {
        // The state entering chunk c (the backward pass reads it back).
        float *dst = hsave + ((((cb + c) * HV + hv) * K + r) * V + vt0 + 16 * hs);
#pragma unroll
        for (int j = 0; j < 16; j += 4) *reinterpret_cast<float4 *>(dst + j) = make_float4(hr[j], hr[j + 1], hr[j + 2], hr[j + 3]);
      }
      // The loads of chunk c.  The testing hook replaces the first wait by one
      // on a barrier nothing completes.
      go = ((force_expiry && c == 0) ? waitl(b_never, 0, kTestWaitLimit) : waitc(FULL, c)) && go;
      // W [h_hi | h_lo] (M = 64): warp p < 4 takes k-steps [p KA, p KA + KA).
      if (warp < 4 && lane == 0 && go) {
        tc_fence_after();
        constexpr uint32_t id1 = umma_idesc_bf16(64, 64, 0, 1);
#pragma unroll
        for (int m = 0; m < KA; ++m) {
          const int kk = warp * KA + m;
          const uint64_t a = umma_desc_sw128(st + Ly::WQ + (kk >> 2) * 16384 + (kk & 3) * 32);
          const uint64_t b = umma_desc_sw128_mn(sb + Ly::OFF_H + kk * 2048, 8192);
          umma_bf16(tmem + Ly::ACC1 + 64 * warp, a, b, id1, m > 0 ? 1u : 0u);
        }
        umma_commit(b_m1);
      } else if (warp == 7 && lane == 0 && go) {
        issue_u(c);  // ACC4 was last read for chunk c - 1, before its v_new barrier
      }
      __syncwarp();
      // Output of the previous chunk while these products run.
      if (c >= 1) {
        go = wait_out(c - 1) && go;
        go = output(c - 1, go);
      }
      go = waitb(b_m1, c & 1) && go;  // W h and u of this chunk
      const float dL = go ? rsc[RS_DL] : 0.f;
      float og = 0.f;
      if (go) {
        // v_new = beta v + u - W (h_hi + h_lo) for row ti; s v_new and v_new
        // as bf16 hi | lo.
        tc_fence_after();
        const int i = ti;
        uint32_t pw[8][8], u[8];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          tmem_ld8x2_issue(tl + Ly::ACC1 + 64 * p + 16 * hs, pw[2 * p]);
          tmem_ld8x2_issue(tl + Ly::ACC1 + 64 * p + 32 + 16 * hs, pw[2 * p + 1]);
        }
        tmem_ld8x2_issue(tl + Ly::ACC4 + vhalf + 16 * hs, u);
        const float bt = rsc[RS_BET + i], sv = rsc[RS_SV + i];
        og = rsc[RS_OG + i];
        const uint4 vv = *reinterpret_cast<const uint4 *>(stp + Ly::VB + i * 128 + ((((vhalf + tc) >> 3) ^ (i & 7)) << 4));
#pragma unroll
        for (int p = 0; p < 8; ++p) tmem_ld_wait8(pw[p]);
        tmem_ld_wait8(u);
        float wh[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          wh[j] = ((__uint_as_float(pw[0][j]) + __uint_as_float(pw[1][j])) + (__uint_as_float(pw[2][j]) + __uint_as_float(pw[3][j]))) +
                  ((__uint_as_float(pw[4][j]) + __uint_as_float(pw[5][j])) + (__uint_as_float(pw[6][j]) + __uint_as_float(pw[7][j])));
        const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
        uint32_t yh[4], yl[4], xh[4], xl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = 2 * e;
          const float x0 = fmaf(bt, bf16lo_f(vw[e]), __uint_as_float(u[j])) - wh[j];
          const float x1 = fmaf(bt, bf16hi_f(vw[e]), __uint_as_float(u[j + 1])) - wh[j + 1];
          xh[e] = pack_bf16(x0, x1);
          xl[e] = pack_bf16(x0 - bf16lo_f(xh[e]), x1 - bf16hi_f(xh[e]));
          const float y0 = sv * x0, y1 = sv * x1;
          yh[e] = pack_bf16(y0, y1);
          yl[e] = pack_bf16(y0 - bf16lo_f(yh[e]), y1 - bf16hi_f(yh[e]));
        }
        const int chh = tc >> 3;
        unsigned char *vsr = sm + Ly::OFF_VS + (i >> 3) * 1024 + (i & 7) * 128;
        unsigned char *vnr = sm + Ly::OFF_VN + (i >> 3) * 1024 + (i & 7) * 128;
        *reinterpret_cast<uint4 *>(vsr + ((chh ^ (i & 7)) << 4)) = make_uint4(yh[0], yh[1], yh[2], yh[3]);
        *reinterpret_cast<uint4 *>(vsr + (((4 + chh) ^ (i & 7)) << 4)) = make_uint4(yl[0], yl[1], yl[2], yl[3]);
        *reinterpret_cast<uint4 *>(vnr + ((chh ^ (i & 7)) << 4)) = make_uint4(xh[0], xh[1], xh[2], xh[3]);
        *reinterpret_cast<uint4 *>(vnr + (((4 + chh) ^ (i & 7)) << 4)) = make_uint4(xl[0], xl[1], xl[2], xl[3]);
      }
      tc_fence_before();
      fence_proxy_async_smem();
      named_bar_sync(1, WALK_COMPUTE);
      // K^T [s v_new hi | lo]: warp q < 2 takes k-steps 2q, 2q + 1.  For K = 64
      // the keys 64-127 of the M = 128 operand come from the zero block.
      if (warp < 2 && lane == 0 && go) {
        tc_fence_after();
        constexpr uint32_t id2 = umma_idesc_bf16(128, 64, 1, 1);
        const uint32_t lbo = (K == 64) ? static_cast<uint32_t>(Ly::OFF_Z - s * Ly::STAGE - Ly::KT) : 8192u;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const int kk = 2 * warp + m;
          const uint64_t a = umma_desc_sw128_mn(st + Ly::KT + kk * 2048, lbo);
          const uint64_t b = umma_desc_sw128_mn(sb + Ly::OFF_VS + kk * 2048, 8192);
          umma_bf16(tmem + Ly::ACC2 + 64 * warp, a, b, id2, m > 0 ? 1u : 0u);
        }
        umma_commit(b_m2);
      }
      __syncwarp();
      go = waitb(b_m2, c & 1) && go;
      go = waitb(b_qd, c & 1) && go;  // Q h: it read the stage's Q tile and the H tile
      if (tid == 0 && go) mbar_arrive(bar(CDONE, c & 1));
      if (go) {
        tc_fence_after();
        uint32_t x0[16], y0[16], x1[16], y1[16], qa[8], qb[8];
        tmem_ld16_issue(tl + Ly::ACC2 + 16 * hs, x0);
        tmem_ld16_issue(tl + Ly::ACC2 + 32 + 16 * hs, y0);
        tmem_ld16_issue(tl + Ly::ACC2 + 64 + 16 * hs, x1);
        tmem_ld16_issue(tl + Ly::ACC2 + 96 + 16 * hs, y1);
        tmem_ld8x2_issue(tl + Ly::ACCQ + 16 * hs, qa);
        tmem_ld8x2_issue(tl + Ly::ACCQ + 32 + 16 * hs, qb);
        tmem_ld_wait16(x0);
        tmem_ld_wait16(y0);
        tmem_ld_wait16(x1);
        tmem_ld_wait16(y1);
        tmem_ld_wait8(qa);
        tmem_ld_wait8(qb);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          hr[j] = fmaf(dL, hr[j], (__uint_as_float(x0[j]) + __uint_as_float(y0[j])) + (__uint_as_float(x1[j]) + __uint_as_float(y1[j])));
#pragma unroll
        for (int j = 0; j < 8; ++j) qh[j] = og * (__uint_as_float(qa[j]) + __uint_as_float(qb[j]));
        write_h();
      }
      tc_fence_before();
      fence_proxy_async_smem();
      named_bar_sync(1, WALK_COMPUTE);
    }
    if (NC > 0) {
      go = wait_out(NC - 1) && go;
      go = output(NC - 1, go);
    }
    if (lane == 0 && *abort_flag) {
      // After an abort products may still be in flight: one more commit by
      // each issuing thread completes once all of that thread's products have.
      if (warp < 4 || warp == 7) {
        tc_fence_after();
        umma_commit(b_drain);
        if (!mbar_wait_bounded(b_drain, 0, kWaitLimit)) set_status(dev_status, GDN_DEV_DRAIN_TIMEOUT);
      }
    }
    if (ht && krow && !*abort_flag) {
#pragma unroll
      for (int j = 0; j < 16; j += 4)
        *reinterpret_cast<float4 *>(ht + (sbase + r) * V + vt0 + 16 * hs + j) =
            make_float4(hr[j], hr[j + 1], hr[j + 2], hr[j + 3]);
    }
  } else if (warp >= 9) {
    // ------------------------------------------------- off-chain products
    bool go = true;
    for (int c = 0; c < NC; ++c) {
      const int s = c % NS;
      const uint32_t st = sb + s * Ly::STAGE;
      if (warp == 9) {
        // Q [h_hi | h_lo] (M = 64) once W h is done: h_c and Q are in shared
        // memory, and ACCQ of chunk c - 1 was read before W h was issued.
        go = waitc(FULL, c) && go;
        go = waitb(b_m1, c & 1) && go;
        if (lane == 0 && go) {
          tc_fence_after();
          constexpr uint32_t idq = umma_idesc_bf16(64, 64, 0, 1);
#pragma unroll
          for (int kk = 0; kk < 4 * KA; ++kk) {
            const uint64_t a = umma_desc_sw128(st + Ly::WQ + (kk >> 2) * 16384 + 8192 + (kk & 3) * 32);
            const uint64_t b = umma_desc_sw128_mn(sb + Ly::OFF_H + kk * 2048, 8192);
            umma_bf16(tmem + Ly::ACCQ, a, b, idq, kk > 0 ? 1u : 0u);
          }
          umma_commit(b_qd);
        }
        __syncwarp();
      }
      // [P_hi | P_lo] [v_new hi | lo] once the state product is done: v_new of
      // chunk c is in shared memory and ACC3 / ACC3L of chunk c - 1 were read
      // before it was issued.  Both complete on OUT(c).
      go = waitb(b_m2, c & 1) && go;
      if (lane == 0 && go) {
        tc_fence_after();
        constexpr uint32_t id3 = umma_idesc_bf16(64, 64, 0, 1);
        const uint32_t pa = st + Ly::RR + (warp - 9) * 8192;
        const uint32_t acc = tmem + (warp == 9 ? Ly::ACC3 : Ly::ACC3L);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t a = umma_desc_sw128(pa + kk * 32);
          const uint64_t b = umma_desc_sw128_mn(sb + Ly::OFF_VN + kk * 2048, 8192);
          umma_bf16(acc, a, b, id3, kk > 0 ? 1u : 0u);
        }
        umma_commit(b_out(c));
      }
      __syncwarp();
    }
    if (lane == 0 && *abort_flag) {
      tc_fence_after();
      umma_commit(b_drain);
      if (!mbar_wait_bounded(b_drain, 0, kWaitLimit)) set_status(dev_status, GDN_DEV_DRAIN_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------- producer
    int issued = 0;
    auto issue = [&](int c) {
      const int s = c % NS;
      const uint32_t st = sb + s * Ly::STAGE;
      const int trow = static_cast<int>(tok0) + c * C;
      const unsigned char *rec = ws + (static_cast<size_t>(cb + c) * HV + hv) * R::BYTES;
      mbar_arrive_expect_tx(bar(FULL, s), Ly::TX);
#pragma unroll
      for (int a = 0; a < KA; ++a) {
        tma_load_3d(st + Ly::KT + a * 8192, &tm_k, bar(FULL, s), 64 * a, h, trow);
        tma_load_3d(st + Ly::WQ + a * 16384 + 8192, &tm_q, bar(FULL, s), 64 * a, h, trow);
        bulk_load(st + Ly::WQ + a * 16384, rec + R::W + a * 8192, 8192, bar(FULL, s));
      }
      tma_load_3d(st + Ly::VB, &tm_v, bar(FULL, s), vt0 - vhalf, hv, trow);
      bulk_load(st + Ly::RR, rec + R::PH, Ly::RR_BYTES, bar(FULL, s));
      issued = c + 1;
    };
    if (lane == 0)
      for (int c = 0; c < NS && c < NC; ++c) issue(c);
    __syncwarp();
    for (int c = 0; c + NS < NC; ++c) {
      bool can = waitc(CDONE, c);
      can = wait_out(c) && can;  // the output products of chunk c read P hi / lo
      if (can && lane == 0) issue(c + NS);
      __syncwarp();
    }
    if (lane == 0 && *abort_flag) {
      // Nothing of this CTA may still be in flight at exit.
      for (int k = (issued > NS ? issued - NS : 0); k < issued; ++k)
        if (!mbar_wait_bounded(bar(FULL, k % NS), (k / NS) & 1, kWaitLimit))
          set_status(dev_status, GDN_DEV_DRAIN_TIMEOUT);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, Ly::TMEM_COLS);
  }
  if (tid == 0 && *abort_flag) set_status(dev_status, GDN_DEV_WAIT_TIMEOUT);
}

// ------------------------------------------------------------- chunk starts
// cs[n] = number of chunks of the sequences before n (cu_seqlens input; a
// sequence whose offsets break the rules has none), cs[N] = the total: one
// block, each thread summing a contiguous run of sequences, then a block scan.
__global__ void __launch_bounds__(1024) chunk_starts_kernel(const int32_t *__restrict__ cu, int N, int T,
                                                            int32_t *__restrict__ cs) {
  __shared__ int32_t part[1024];
  const int tid = threadIdx.x;
  const int per = (N + 1023) / 1024;
  const int n0 = min(N, tid * per), n1 = min(N, n0 + per);
  int32_t sum = 0;
  for (int n = n0; n < n1; ++n) {
    int64_t t0, l0;
    if (seq_bounds(cu, n, T, t0, l0)) sum += chunks_of(l0);
  }
  part[tid] = sum;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {  // inclusive scan
    const int32_t y = tid >= off ? part[tid - off] : 0;
    __syncthreads();
    part[tid] += y;
    __syncthreads();
  }
  int32_t run = part[tid] - sum;  // exclusive
  for (int n = n0; n < n1; ++n) {
    cs[n] = run;
    int64_t t0, l0;
    if (seq_bounds(cu, n, T, t0, l0)) run += chunks_of(l0);
  }
  if (tid == 1023) cs[N] = part[1023];
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 3-D map over a [rows][heads][dim] bf16 tensor, box {box0, 1 head, 64 rows}.
bool make_map(CUtensorMap *m, const void *ptr, int dim, int heads, int64_t rows, int box0, bool swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[3] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstr[2] = {static_cast<cuuint64_t>(dim) * 2, static_cast<cuuint64_t>(dim) * heads * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box0), 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), gdim, gstr, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int K>
size_t records_bytes(int B, int T, int HV, int N, bool varlen) {
  return static_cast<size_t>(total_chunk_slots(B, T, N, varlen)) * HV * Rec<K>::BYTES;
}
// A long single sequence (N = 1, dense or cu_seqlens) is walked in several chunk ranges.
// While the walk of one range runs, the prep of the next runs on the SMs the
// walk leaves free (a walk CTA fills an SM): it is launched as a programmatic
// dependent of that walk, whose CTAs release it once they are all resident,
// so it can never take the walk's SMs first.  The walk of the next range,
// launched normally after it, waits for both and starts from the state the
// previous walk left in the workspace (each CTA reads and later writes only
// its own slice there, so one buffer serves every hand-over).  Only the first
// range's prep is not hidden behind a walk.
constexpr int kSplitMinChunks = 64;
constexpr int kSplitMinFreeSMs = 16;
constexpr int kMaxRanges = 4;
constexpr int kMinRangeChunks = 32;
inline bool split_shape(int N, int T, bool varlen) {
  (void)varlen;  // with cu_seqlens, N = 1 means the one sequence spans [0, T)
  return N == 1 && (static_cast<int64_t>(T) + C - 1) / C >= kSplitMinChunks;
}
// Bytes of the state handed from the first range's walk to the second's.
inline size_t handoff_bytes(int N, int T, int HV, int K, int V, bool varlen) {
  return split_shape(N, T, varlen) ? static_cast<size_t>(N) * HV * K * V * 4 : 0;
}
template <int K>
size_t ws_bytes(int B, int T, int HV, int V, int N, bool varlen) {
  return records_bytes<K>(B, T, HV, N, varlen) + chunk_starts_bytes(N, varlen) + handoff_bytes(N, T, HV, K, V, varlen);
}
// The chunk ranges of this call on the current device: bounds[0] = 0 <
// bounds[1] < ... < bounds[R] = number of chunks; R = 1 when it is walked in
// one range.  A range's walk should take as long as the next range's prep on
// the F free SMs of S.  Measured at K = V = 128, a chunk's prep on the whole
// GPU costs 1 / 3.1 of its walk, and a prep CTA beside a walk runs about 8 %
// faster than in a full prep grid, so each range has q = 3.3 F / S times the
// chunks of the one before it; the count is the largest (up to kMaxRanges)
// whose last range keeps kMinRangeChunks chunks.
cudaError_t chunk_ranges(int N, int T, int HV, int V, bool varlen, bool hsave, int *bounds, int *R) {
  const int64_t nc = (static_cast<int64_t>(T) > 0 ? (static_cast<int64_t>(T) + C - 1) / C : 0);
  *R = 1;
  bounds[0] = 0;
  bounds[1] = static_cast<int>(nc);
  (void)hsave;  // a walk that saves the chunk states splits the same way (each range saves its own)
  if (T <= 0 || !split_shape(N, T, varlen)) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int free_sms = sms - (V / VT) * HV;
  if (free_sms < kSplitMinFreeSMs) return cudaSuccess;
  const double q = free_sms * 3.3 < sms ? free_sms * 3.3 / sms : 0.9;
  for (int r = kMaxRanges; r >= 2; --r) {
    // Range k has about nc * q^k (1 - q) / (1 - q^r) chunks.
    double w = 1.0, wsum = 0.0;
    for (int k = 0; k < r; ++k, w *= q) wsum += w;
    double acc = 0.0;
    w = 1.0;
    bool ok = true;
    for (int k = 0; k < r; ++k, w *= q) {
      acc += w;
      bounds[k + 1] = k + 1 == r ? static_cast<int>(nc) : static_cast<int>(nc * acc / wsum + 0.5);
      if (bounds[k + 1] - bounds[k] < kMinRangeChunks) ok = false;
    }
    if (ok) {
      *R = r;
      return cudaSuccess;
    }
  }
  bounds[1] = static_cast<int>(nc);
  return cudaSuccess;
}

template <int K>
cudaError_t launch_k(const gdn_host::ChunkArgs &a, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(a.B) * a.T;
  CUtensorMap mq, mk, mv;
  memset(&mq, 0, sizeof(mq));
  memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv));
  // With no tokens every sequence is empty: the walk only copies states and
  // never touches the (then unused) maps.
  if (rows > 0 && (!make_map(&mq, a.q, K, a.H, rows, 64, true) || !make_map(&mk, a.k, K, a.H, rows, 64, true) ||
                   !make_map(&mv, a.v, a.V, a.HV, rows, 64, true)))
    return cudaErrorInvalidValue;
  const int64_t slots = total_chunk_slots(a.B, a.T, a.N, a.cu != nullptr);
  // cu_seqlens: the chunk starts of the sequences, after the records.
  const int32_t *cs = nullptr;
  if (a.cu) {
    int32_t *csw = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(a.ws) +
                                               records_bytes<K>(a.B, a.T, a.HV, a.N, true));
    chunk_starts_kernel<<<1, 1024, 0, s>>>(a.cu, a.N, a.T, csw);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cs = csw;
  }
  const int psmem = PrepLay<K>::BYTES + 1024;
  const int wsmem = WalkLay<K>::BYTES + 1024;
  cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, psmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(chunk_walk_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, wsmem);
  if (e != cudaSuccess) return e;
  const PrepGates gt{a.A_log, a.ga, a.gb, a.dt_bias, a.g_out, a.beta_out};
  // The prep of chunk slots [slot_begin, slot_begin + nslots).
  auto prep = [&](int slot_begin, int64_t nslots, cudaStream_t st) {
    if (rows <= 0 || nslots <= 0) return cudaSuccess;
    dim3 pgrid(static_cast<unsigned>(nslots * a.HV));
    chunk_prep_kernel<K><<<pgrid, NTH, psmem, st>>>(mq, mk, a.g, a.beta, gt, a.cu, cs, a.N, a.T, a.H, a.HV, a.l2,
                                                    static_cast<unsigned char *>(a.ws), a.dev_status, slot_begin);
    return cudaGetLastError();
  };
  // The walk of chunks [c_begin, c_end) of every sequence, from state hin to hout.
  auto walk = [&](int c_begin, int c_end, const float *hin, float *hout, cudaStream_t st) {
    dim3 grid(a.V / VT, a.HV, a.N);
    chunk_walk_kernel<K><<<grid, WALK_THREADS, wsmem, st>>>(mq, mk, mv, a.scale, hin, a.cu, a.T, a.H, a.HV, a.V,
                                                   static_cast<const unsigned char *>(a.ws), a.o, hout, a.hsave,
                                                   cs, a.dev_status, a.force_expiry, c_begin, c_end);
    return cudaGetLastError();
  };
  int bounds[kMaxRanges + 1], R = 1;
  if ((e = chunk_ranges(a.N, a.T, a.HV, a.V, a.cu != nullptr, a.hsave != nullptr, bounds, &R)) != cudaSuccess)
    return e;
  if (R == 1) {
    if ((e = prep(0, slots, s)) != cudaSuccess) return e;
    return walk(0, bounds[1], a.h0, a.ht, s);
  }
  float *hmid = reinterpret_cast<float *>(static_cast<unsigned char *>(a.ws) +
                                          records_bytes<K>(a.B, a.T, a.HV, a.N, a.cu != nullptr) +
                                          chunk_starts_bytes(a.N, a.cu != nullptr));
  if ((e = prep(0, bounds[1], s)) != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  for (int r = 0; r < R; ++r) {
    e = walk(bounds[r], bounds[r + 1], r == 0 ? a.h0 : hmid, r + 1 == R ? a.ht : hmid, s);
    if (e != cudaSuccess || r + 1 == R) return e;
    // The next range's prep, beside this walk.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(static_cast<int64_t>(bounds[r + 2] - bounds[r + 1]) * a.HV));
    cfg.blockDim = dim3(NTH);
    cfg.dynamicSmemBytes = psmem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, chunk_prep_kernel<K>, mq, mk, a.g, a.beta, gt, a.cu, cs, a.N, a.T, a.H, a.HV, a.l2,
                           static_cast<unsigned char *>(a.ws), a.dev_status, bounds[r + 1]);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

namespace gdn_host {

size_t chunk_workspace_bytes(int B, int T, int H, int HV, int K, int V, int N, int varlen) {
  (void)H;
  if (K == 128) return ws_bytes<128>(B, T, HV, V, N, varlen != 0);
  if (K == 64) return ws_bytes<64>(B, T, HV, V, N, varlen != 0);
  return 0;
}

int chunk_fwd_launches(int B, int T, int H, int HV, int K, int V, int N, int varlen) {
  (void)H;
  (void)K;
  if (N <= 0) return 0;
  int bounds[kMaxRanges + 1], R = 1;
  if (chunk_ranges(N, T, HV, V, varlen != 0, false, bounds, &R) != cudaSuccess) return -1;
  if (R > 1) return 2 * R + (varlen ? 1 : 0);
  const bool prep = static_cast<int64_t>(B) * T > 0 && total_chunk_slots(B, T, N, varlen != 0) > 0;
  return (varlen ? 1 : 0) + (prep ? 1 : 0) + 1;
}

cudaError_t launch_chunk(const ChunkArgs &a, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  if (a.K == 128) return launch_k<128>(a, s);
  if (a.K == 64) return launch_k<64>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace gdn_host

// ------------------------------------------------ no-allocation entry point
//
// Some callers cannot allocate device memory at call time: serving runtimes
// that hand all device memory to their own pool at start-up and forbid any
// later cudaMalloc, and hot loops that must not take the driver's allocation
// path.  For them gdn_chunk_fwd_noalloc runs the same two kernels with the
// workspace in a fixed buffer compiled into this library instead of a
// caller-provided one.
//
// The buffer is a file-scope __device__ array: every GPU that loads the
// library holds GDN_NOALLOC_SCRATCH_BYTES of it until the process exits.  In
// host code the array's name is only a host-side stand-in, so its device
// address is looked up once per device (with that device current) through
// cudaGetSymbolAddress and cached.  Every call on a device shares the buffer
// and leaves the last call's contents in it; nothing in it must start at zero
// (each record the walk kernel reads is written by the prep kernel of the same
// call), but two calls that overlap on the GPU race on it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch buffer on the current device (set-up on the
// first call per device).
int noalloc_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ECUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GDN_ECUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return GDN_OK;
}
}  // namespace

extern "C" int gdn_chunk_fwd_noalloc(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *g,
                                     const float *beta, float scale, const float *initial_state,
                                     const int32_t *cu_seqlens, int N, int B, int T, int H, int HV, int K, int V,
                                     int use_qk_l2norm, uint16_t *o, float *final_state, int32_t *dev_status,
                                     void *stream) {
  if (B < 0 || T < 0 || N < 0 || HV <= 0 || K <= 0) return GDN_EINVAL;
  const size_t need = gdn_chunk_fwd_workspace_size(B, T, H, HV, K, V, N, cu_seqlens != nullptr);
  if (need > GDN_NOALLOC_SCRATCH_BYTES) return GDN_ESCRATCH_LIMIT;
  void *ws = nullptr;
  if (need > 0) {
    const int rc = noalloc_scratch(&ws);
    if (rc != GDN_OK) return rc;
  }
  return gdn_chunk_fwd(q, k, v, g, beta, scale, initial_state, cu_seqlens, N, B, T, H, HV, K, V, use_qk_l2norm, o,
                       final_state, ws, need > 0 ? GDN_NOALLOC_SCRATCH_BYTES : 0, dev_status, stream);
}
