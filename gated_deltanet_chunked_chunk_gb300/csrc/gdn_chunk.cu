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
// gdn_chunk_prep (one CTA per (chunk, value head), two CTAs per SM): TMA loads
// K and Q; one thread issues tcgen05.mma for [K;Q][K;Q]^T (M = N = 128,
// 128B-swizzled smem operands, fp32 accumulator in TMEM), whose diagonal gives
// the row norms; A and P are built from TMEM; T by 16x16 diagonal-block
// substitution plus tf32 mma.sync for the off-diagonal blocks, in place; W by
// mma.sync.  The CTA writes one record [W | P hi | P lo | Ts | scalars] per
// (chunk, value head) to the workspace, laid out exactly as the walk kernel
// wants it in shared memory.
//
// gdn_chunk_walk (one CTA per (32-column slice, value head, sequence)): keeps
// the fp32 state slice in registers; per chunk one thread issues the TMA
// loads of K, Q, the V slice and a bulk copy of the record into a two-stage
// ring, and the eight warps run u, [Q; W] h, v_new, the state update and o
// with mma.sync, two CTA barriers per chunk.
//
// Precision: the main terms of o (P v_new and Q h) and the state update split
// their computed factor into bf16 hi + lo parts (the raw bf16 q, k, v are
// exact); W, Ts and the h in W h are plain bf16; accumulation is fp32, and h,
// A, T stay fp32.  Every mbarrier wait is bounded; on expiry a CTA records
// GDN_DEV_WAIT_TIMEOUT, drains its outstanding copies and leaves.
#include <cuda.h>
#include <string.h>

#include <mutex>

#include "gdn_common.cuh"
#include "gdn_sm103.cuh"

namespace {

using namespace gdn;

constexpr int C = 64;
constexpr int VT = 32;
constexpr int NW = 8;
constexpr int NTH = NW * 32;
constexpr long long kWaitLimit = 2000000000LL;  // clock cycles (about 1 s) before a wait gives up
constexpr int HROW = 80;                        // bytes per padded row of 32 bf16
constexpr int FROW = 68;                        // floats per padded fp32 row of 64
constexpr float kLog2e = 1.4426950408889634f;

// Per-(chunk, value head) record, byte offsets; also its shared-memory image.
template <int K>
struct Rec {
  static constexpr int KA = K / 64;
  static constexpr int W = 0;               // [64][K] bf16, 64-key SW128 atom columns
  static constexpr int PH = KA * 8192;      // [64][64] bf16 SW128
  static constexpr int PL = PH + 8192;
  static constexpr int TS = PL + 8192;
  static constexpr int SC = TS + 8192;      // og[64], sv[64], beta[64], e^{gamma_L} (fp32)
  static constexpr int BYTES = SC + 1024;
  static_assert(BYTES % 1024 == 0, "record alignment");
};
enum { RS_OG = 0, RS_SV = 64, RS_BET = 128, RS_DL = 192 };

// [K; Q] tile as two TMA boxes per 64-key atom column: rows 0-63 K, 64-127 Q.
template <int K>
struct KQ {
  static constexpr int KA = K / 64;
  static constexpr int BYTES = KA * 16384;
};

__device__ __forceinline__ unsigned char *align1024(unsigned char *p) {
  return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}
// Address of the 16-byte chunk holding keys [8 kc, 8 kc + 8) of row `row` in a
// [rows][K] bf16 tile stored as 64-key SW128 atom columns of `rows` rows.
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int rows, int row, int kc) {
  return base + (kc >> 3) * (rows * 128) + sw128(row, kc & 7);
}
// 2^x with the hardware approximation (relative error around 2^-22).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Sequence bounds (dense or cu_seqlens); false for offsets that break the rules.
__device__ __forceinline__ bool seq_bounds(const int32_t *cu, int n, int T, int64_t &tok0, int64_t &len) {
  if (cu) {
    const int32_t a0 = cu[n], a1 = cu[n + 1];
    if (a0 < 0 || a1 < a0 || a1 > T || (n == 0 && a0 != 0)) return false;
    tok0 = a0;
    len = a1 - a0;
  } else {
    tok0 = static_cast<int64_t>(n) * T;
    len = T;
  }
  return true;
}
__device__ __forceinline__ int chunks_of(int64_t len) { return static_cast<int>((len + C - 1) / C); }
// Index of the first chunk of sequence n in the workspace: sum of the chunk
// counts of the sequences before it (offsets that break the rules count 0).
__device__ __forceinline__ int64_t chunk_base(const int32_t *cu, int n, int T) {
  if (!cu) return static_cast<int64_t>(n) * chunks_of(T);
  int64_t b = 0;
  for (int m = 0; m < n; ++m) {
    int64_t t0, l0;
    if (seq_bounds(cu, m, T, t0, l0)) b += chunks_of(l0);
  }
  return b;
}

// ============================================================== prep kernel
template <int K>
struct PrepLay {
  static constexpr int OFF_KQ = 0;                              // [K;Q] tile
  static constexpr int OFF_REC = KQ<K>::BYTES;                  // record image
  static constexpr int OFF_AT = OFF_REC + Rec<K>::BYTES;        // A then T, fp32 [64][FROW], in place
  static constexpr int OFF_TP = OFF_AT + 64 * FROW * 4;         // T diag(beta e^g rk), bf16 SW128
  static constexpr int OFF_X = OFF_TP + 8192;                   // 4 x [16][17] fp32
  static constexpr int OFF_SC = OFF_X + 4352;                   // gl, bet, rk, rq, rowA, rowP, colf, ftp
  static constexpr int OFF_BAR = OFF_SC + 8 * 256;
  static constexpr int OFF_MISC = OFF_BAR + 16;
  static constexpr int BYTES = OFF_MISC + 16;
  static_assert(OFF_TP % 1024 == 0, "swizzled tile alignment");
};
enum { PS_GL = 0, PS_BET = 1, PS_RK = 2, PS_RQ = 3, PS_RA = 4, PS_RP = 5, PS_CF = 6, PS_FTP = 7 };

template <int K>
__global__ void __launch_bounds__(NTH, 2) chunk_prep_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k, const float *__restrict__ g,
    const float *__restrict__ beta, const int32_t *__restrict__ cu, int N, int T, int H, int HV, int l2,
    unsigned char *__restrict__ ws, int32_t *dev_status) {
  using Ly = PrepLay<K>;
  using R = Rec<K>;
  constexpr int KA = K / 64;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = align1024(smem_raw);
  const uint32_t sb = smem_u32(sm);
  const int gc = blockIdx.x, hv = blockIdx.y;
  const int h = hv / (HV / H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g4 = lane >> 2, t4 = lane & 3;

  // Which sequence / chunk is this?
  int n = 0, c = 0;
  int64_t tok0 = 0, len = 0;
  {
    int64_t base = 0;
    bool found = false;
    for (int m = 0; m < N && !found; ++m) {
      int64_t t0, l0;
      if (!seq_bounds(cu, m, T, t0, l0)) continue;
      const int nc = chunks_of(l0);
      if (gc < base + nc) {
        found = true;
        n = m;
        c = static_cast<int>(gc - base);
        tok0 = t0;
        len = l0;
      }
      base += nc;
    }
    if (!found) return;  // past the last chunk (the grid is an upper bound)
  }
  (void)n;
  const int64_t rem = len - static_cast<int64_t>(c) * C;
  const int L = static_cast<int>(rem < C ? rem : C);
  const int64_t trow0 = tok0 + static_cast<int64_t>(c) * C;

  float *scal = reinterpret_cast<float *>(sm + Ly::OFF_SC);
  float *gl = scal + PS_GL * 64, *bet = scal + PS_BET * 64, *rk = scal + PS_RK * 64, *rq = scal + PS_RQ * 64;
  float *rowA = scal + PS_RA * 64, *rowP = scal + PS_RP * 64, *colf = scal + PS_CF * 64, *ftp = scal + PS_FTP * 64;
  float *AT = reinterpret_cast<float *>(sm + Ly::OFF_AT);
  float *Xs = reinterpret_cast<float *>(sm + Ly::OFF_X);
  unsigned char *rec = sm + Ly::OFF_REC;
  float *rsc = reinterpret_cast<float *>(rec + R::SC);
  uint32_t *misc = reinterpret_cast<uint32_t *>(sm + Ly::OFF_MISC);
  const uint32_t b_tma = sb + Ly::OFF_BAR, b_mma = sb + Ly::OFF_BAR + 8;
  const uint32_t kq = sb + Ly::OFF_KQ;

  if (tid == 0) {
    mbar_init(b_tma, 1);
    mbar_init(b_mma, 1);
    misc[1] = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(sb + Ly::OFF_MISC, 128);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  if (tid == 0) {
    mbar_arrive_expect_tx(b_tma, KQ<K>::BYTES);
#pragma unroll
    for (int a = 0; a < KA; ++a) {
      tma_load_3d(kq + a * 16384, &tm_k, b_tma, 64 * a, h, static_cast<int>(trow0));
      tma_load_3d(kq + a * 16384 + 8192, &tm_q, b_tma, 64 * a, h, static_cast<int>(trow0));
    }
  }
  // Gates (rows >= L read as 0) and their chunk-local cumsum in base 2 (warp 4).
  if (warp == 4) {
    float x[2], bb[2];
#pragma unroll
    for (int u2 = 0; u2 < 2; ++u2) {
      const int r = 2 * lane + u2;
      x[u2] = r < L ? g[(trow0 + r) * HV + hv] : 0.f;
      bb[u2] = r < L ? beta[(trow0 + r) * HV + hv] : 0.f;
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
        float dv[32];
        if (qdiag) tmem_ld32(tl + 64 + 32 * (quad - 2), dv);
        float d = kdiag ? vals[0] : dv[0];
#pragma unroll
        for (int m = 1; m < 32; ++m) d = (lane == m) ? (kdiag ? vals[m] : dv[m]) : d;
        const float rn = rsqrtf(d + GDN_L2_EPS);
        if (kdiag) rk[row] = rn; else rq[row - 64] = rn;
      }
    } else if (tid < 64) {
      rk[tid] = 1.f;
      rq[tid] = 1.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);  // every TMEM read is done

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
      *reinterpret_cast<uint4 *>(rec + R::PH + sw128(i, chunk)) = vh;
      *reinterpret_cast<uint4 *>(rec + R::PL + sw128(i, chunk)) = vl;
    }
  }
  __syncthreads();

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

  // Tp = T diag(beta e^gamma rk) (j <= i, for W) and Ts = (T - I) diag(beta) (j < i), bf16.
  for (int e = tid; e < 64 * 8; e += NTH) {
    const int i = e >> 3, ch = e & 7;
    uint4 tpv = make_uint4(0, 0, 0, 0), tsv = make_uint4(0, 0, 0, 0);
    if (8 * ch <= i) {
      const float4 t0 = *reinterpret_cast<const float4 *>(AT + i * FROW + 8 * ch);
      const float4 t1 = *reinterpret_cast<const float4 *>(AT + i * FROW + 8 * ch + 4);
      const float4 f0 = *reinterpret_cast<const float4 *>(ftp + 8 * ch);
      const float4 f1 = *reinterpret_cast<const float4 *>(ftp + 8 * ch + 4);
      const float4 c0 = *reinterpret_cast<const float4 *>(bet + 8 * ch);
      const float4 c1 = *reinterpret_cast<const float4 *>(bet + 8 * ch + 4);
      const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
      const float fv[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
      const float bv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      uint32_t tp[4], ts[4];
#pragma unroll
      for (int q2 = 0; q2 < 4; ++q2) {
        float a2[2], b2[2];
#pragma unroll
        for (int u2 = 0; u2 < 2; ++u2) {
          const int jj = 2 * q2 + u2, j = 8 * ch + jj;
          a2[u2] = (j <= i) ? tv[jj] * fv[jj] : 0.f;
          b2[u2] = (j < i) ? tv[jj] * bv[jj] : 0.f;
        }
        tp[q2] = pack_bf16(a2[0], a2[1]);
        ts[q2] = pack_bf16(b2[0], b2[1]);
      }
      tpv = make_uint4(tp[0], tp[1], tp[2], tp[3]);
      tsv = make_uint4(ts[0], ts[1], ts[2], ts[3]);
    }
    *reinterpret_cast<uint4 *>(sm + Ly::OFF_TP + sw128(i, ch)) = tpv;
    *reinterpret_cast<uint4 *>(rec + R::TS + sw128(i, ch)) = tsv;
  }
  __syncthreads();

  // W = Tp K (64 x K): warp -> 16 rows (mi) x half of the keys (nh).
  {
    const int mi = warp & 3, nh = warp >> 2;
    constexpr int WN = K / 16;
    float acc[WN][4];
#pragma unroll
    for (int j = 0; j < WN; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t a[4];
      ldsm_x4(sb + Ly::OFF_TP + sw128(16 * mi + (lane & 15), 2 * kk + (lane >> 4)), a);
      const int mq = lane >> 3;
      const int trow = 16 * kk + (lane & 7) + 8 * (mq & 1);
#pragma unroll
      for (int j = 0; j < WN; j += 2) {
        uint32_t b[4];
        ldsm_x4_t(tile_addr(kq, 128, trow, nh * WN + j + (mq >> 1)), b);
        mma_bf16(acc[j], a, b[0], b[1]);
        mma_bf16(acc[j + 1], a, b[2], b[3]);
      }
    }
#pragma unroll
    for (int j = 0; j < WN; ++j) {
      const int key = 8 * (nh * WN + j) + 2 * t4;
      const int r0 = 16 * mi + g4;
      unsigned char *base = rec + R::W + (key >> 6) * 8192 + (key & 7) * 2;
      *reinterpret_cast<uint32_t *>(base + sw128(r0, (key & 63) >> 3)) = pack_bf16(acc[j][0], acc[j][1]);
      *reinterpret_cast<uint32_t *>(base + sw128(r0 + 8, (key & 63) >> 3)) = pack_bf16(acc[j][2], acc[j][3]);
    }
  }
  __syncthreads();

  // Record -> workspace (16-byte coalesced stores).
  uint4 *dst = reinterpret_cast<uint4 *>(ws + (static_cast<size_t>(gc) * HV + hv) * R::BYTES);
  const uint4 *src = reinterpret_cast<const uint4 *>(rec);
  for (int e = tid; e < R::BYTES / 16; e += NTH) dst[e] = src[e];
}

// ============================================================== walk kernel
// Sixteen warps in two groups that hand data to each other through mbarriers:
//   chain (warps 0-7): u = beta v + Ts V, W h, v_new = u - W h, the state update
//     h <- e^{gamma_L} h + K^T (s v_new) and the bf16 copy of h;
//   side (warps 8-15): Q h (hi + lo) while the chain works, o = scale (e^gamma rq
//     Q h + P v_new) once v_new is out, and (thread 256) the TMA / bulk loads of
//     chunk c+2 once both groups are done with chunk c.
template <int K>
struct WalkLay {
  static constexpr int KQB = KQ<K>::BYTES;
  static constexpr int V_BYTES = C * VT * 2;
  static constexpr int STAGE = KQB + V_BYTES + Rec<K>::BYTES;  // [K;Q] | V slice | record
  static constexpr int NS = 2;
  static constexpr int OFF_H = NS * STAGE;                     // h bf16 hi [K][HROW] then lo
  static constexpr int OFF_VS = OFF_H + 2 * K * HROW;          // s v_new hi, lo (chain only)
  static constexpr int OFF_VH = OFF_VS + 2 * 64 * HROW;        // v_new hi, lo (chain -> side)
  static constexpr int OFF_BAR = OFF_VH + 2 * 64 * HROW;
  static constexpr int NBAR = 2 * 7;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr uint32_t TX = KQB + V_BYTES + Rec<K>::BYTES;
  static_assert(STAGE % 1024 == 0, "stage alignment");
  static_assert(BYTES + 1024 <= 232448, "shared memory budget (227 KB per CTA)");
};
constexpr int WNTH = 2 * NTH;  // 512 threads

template <int K>
__global__ void __launch_bounds__(WNTH, 1) chunk_walk_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, float scale, const float *__restrict__ h0,
    const int32_t *__restrict__ cu, int T, int H, int HV, int V, const unsigned char *__restrict__ ws,
    uint16_t *__restrict__ o, float *__restrict__ ht, int32_t *dev_status) {
  using Ly = WalkLay<K>;
  using R = Rec<K>;
  constexpr int KA = K / 64;
  constexpr int NS = Ly::NS;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = align1024(smem_raw);
  const uint32_t sb = smem_u32(sm);
  const int vt0 = blockIdx.x * VT, hv = blockIdx.y, n = blockIdx.z;
  const int h = hv / (HV / H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g4 = lane >> 2, t4 = lane & 3;
  const bool chain = warp < 8;
  const int gw = warp & 7;                  // warp index within its group
  const int mi = gw & 3, nh = gw >> 2;      // 16-row tile, 16-column half (64-row products)

  int64_t tok0, len;
  if (!seq_bounds(cu, n, T, tok0, len)) {
    if (tid == 0) set_status(dev_status, GDN_DEV_BAD_CU_SEQLENS);
    return;
  }
  const int NC = chunks_of(len);
  const int64_t cb = chunk_base(cu, n, T);
  uint32_t *misc = reinterpret_cast<uint32_t *>(sm + Ly::OFF_MISC);
  volatile uint32_t *abort_flag = misc + 1;
  // Barriers, two of each (indexed by chunk parity): TMA full; (unused); h ready;
  // v_new ready; chain done with the stage; side done with h; side done with v_new.
  auto bar = [&](int kind, int b) { return sb + Ly::OFF_BAR + 8 * (2 * kind + b); };
  enum { FULL = 0, HREADY = 2, VREADY = 3, CDONE = 4, SHDONE = 5, SVDONE = 6 };
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(FULL, b), 1);
      for (int kd = 1; kd < 7; ++kd) mbar_init(bar(kd, b), 8);
    }
    misc[1] = 0;
    mbar_fence_init();
  }
  __syncthreads();
  // Waits on chunk c's use of a barrier (each barrier serves every other chunk).
  // Lane 0 polls; __syncwarp orders the other lanes' later reads after its
  // acquire, and the result is warp-uniform.  After any expired wait every
  // later wait returns false at once: the loops then run to their end without
  // work but still pass every named barrier, so no warp is left waiting.
  auto waitc = [&](int kind, int c) -> bool {
    uint32_t ok = 0;
    if (lane == 0) {
      ok = !*abort_flag;
      if (ok && !mbar_wait_bounded(bar(kind, c & 1), (c >> 1) & 1, kWaitLimit)) {
        *abort_flag = 1;
        ok = 0;
      }
    }
    __syncwarp();
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
  };
  auto arrive = [&](int kind, int c) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kind, c & 1));
  };

  const uint32_t aH = sb + Ly::OFF_H, aHL = aH + K * HROW;
  const uint32_t aVS = sb + Ly::OFF_VS, aVSL = aVS + 64 * HROW;
  const uint32_t aVH = sb + Ly::OFF_VH, aVL = aVH + 64 * HROW;
  const int64_t sbase = (static_cast<int64_t>(n) * HV + hv) * K;

  if (chain) {
    // ---------------------------------------------------------------- chain
    constexpr int NT8 = (K / 16) * 4 / 8;  // state n-tiles per warp
    const int hm = gw % (K / 16);
    const int hn0 = (gw / (K / 16)) * NT8;
    float hf[NT8][4];
#pragma unroll
    for (int j = 0; j < NT8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = 16 * hm + g4 + 8 * (e >> 1);
        const int col = 8 * (hn0 + j) + 2 * t4 + (e & 1);
        hf[j][e] = h0 ? h0[(sbase + key) * V + vt0 + col] : 0.f;
      }
    unsigned char *Hb = sm + Ly::OFF_H;
    auto write_h = [&]() {
#pragma unroll
      for (int j = 0; j < NT8; ++j)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int key = 16 * hm + g4 + 8 * hh;
          const int col = 8 * (hn0 + j) + 2 * t4;
          const float x0 = hf[j][2 * hh], x1 = hf[j][2 * hh + 1];
          const uint32_t hi = pack_bf16(x0, x1);
          *reinterpret_cast<uint32_t *>(Hb + key * HROW + col * 2) = hi;
          *reinterpret_cast<uint32_t *>(Hb + (K + key) * HROW + col * 2) = pack_bf16(x0 - bf16lo_f(hi), x1 - bf16hi_f(hi));
        }
    };
    write_h();
    named_bar_sync(1, NTH);
    arrive(HREADY, 0);

    for (int c = 0; c < NC; ++c) {
      const int s = c % NS;
      const uint32_t st = sb + s * Ly::STAGE;
      const uint32_t rc = st + Ly::KQB + Ly::V_BYTES;
      const float *rsc = reinterpret_cast<const float *>(sm + s * Ly::STAGE + Ly::KQB + Ly::V_BYTES + R::SC);
      bool go = waitc(FULL, c);
      if (go) {
      // u = beta v + Ts V for rows 16 mi.., columns 16 nh.. (registers).  Rows >= L
      // of the V slice may hold the next sequence's values; beta and the Ts
      // columns are zero there, so they do not contribute.
      float u[2][4];
      {
        const uint32_t stV = st + Ly::KQB;
        const unsigned char *stp = sm + s * Ly::STAGE;
        float au[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t as[4], bv[4];
          ldsm_x4(rc + R::TS + sw128(16 * mi + (lane & 15), 2 * kk + (lane >> 4)), as);
          const int mq = lane >> 3;
          ldsm_x4_t(stV + (16 * kk + (lane & 7) + 8 * (mq & 1)) * 64 + (2 * nh + (mq >> 1)) * 16, bv);
          mma_bf16(au[0], as, bv[0], bv[1]);
          mma_bf16(au[1], as, bv[2], bv[3]);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int r = 16 * mi + g4 + 8 * hh;
            const int col = 16 * nh + 8 * j + 2 * t4;
            const float bt = rsc[RS_BET + r];
            float v0 = 0.f, v1 = 0.f;
            if (bt != 0.f) {
              const uint32_t vv = *reinterpret_cast<const uint32_t *>(stp + Ly::KQB + r * 64 + col * 2);
              v0 = bf16lo_f(vv);
              v1 = bf16hi_f(vv);
            }
            u[j][2 * hh] = fmaf(bt, v0, au[j][2 * hh]);
            u[j][2 * hh + 1] = fmaf(bt, v1, au[j][2 * hh + 1]);
          }
      }

      // W h (hi part of h): rows 16 mi.., columns 16 nh..
      float aw[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < K / 16; ++kk) {
        uint32_t fw[4], b[4];
        ldsm_x4(tile_addr(rc + R::W, 64, 16 * mi + (lane & 15), 2 * kk + (lane >> 4)), fw);
        const int mq = lane >> 3;
        ldsm_x4_t(aH + (16 * kk + (lane & 7) + 8 * (mq & 1)) * HROW + (2 * nh + (mq >> 1)) * 16, b);
        mma_bf16(aw[0], fw, b[0], b[1]);
        mma_bf16(aw[1], fw, b[2], b[3]);
      }
      // v_new = u - W h; s v_new (hi, lo) for the state update, v_new (hi, lo) for o.
      if (c >= 1) go = waitc(SVDONE, c - 1) && go;
      if (go) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int col = 16 * nh + 8 * j + 2 * t4;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int r = 16 * mi + g4 + 8 * hh;
          const float x0 = u[j][2 * hh] - aw[j][2 * hh], x1 = u[j][2 * hh + 1] - aw[j][2 * hh + 1];
          const uint32_t hi = pack_bf16(x0, x1);
          const uint32_t lo = pack_bf16(x0 - bf16lo_f(hi), x1 - bf16hi_f(hi));
          const float sr = rsc[RS_SV + r];
          const float y0 = sr * x0, y1 = sr * x1;
          const uint32_t yh = pack_bf16(y0, y1);
          const uint32_t yl = pack_bf16(y0 - bf16lo_f(yh), y1 - bf16hi_f(yh));
          unsigned char *vs = sm + Ly::OFF_VS + r * HROW + col * 2;
          *reinterpret_cast<uint32_t *>(vs) = yh;
          *reinterpret_cast<uint32_t *>(vs + 64 * HROW) = yl;
          unsigned char *vh = sm + Ly::OFF_VH + r * HROW + col * 2;
          *reinterpret_cast<uint32_t *>(vh) = hi;
          *reinterpret_cast<uint32_t *>(vh + 64 * HROW) = lo;
        }
      }
      }
      }
      named_bar_sync(1, NTH);
      if (go) arrive(VREADY, c);

      // h = e^{gamma_L} h + K^T (s v_new), hi and lo parts.
      if (go) {
        const float dL = rsc[RS_DL];
        float hl[NT8][4];
#pragma unroll
        for (int j = 0; j < NT8; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            hf[j][e] *= dL;
            hl[j][e] = 0.f;
          }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int mq = lane >> 3;
          uint32_t a[4];
          ldsm_x4_t(tile_addr(st, 128, 16 * kk + (lane & 7) + 8 * (mq >> 1), 2 * hm + (mq & 1)), a);
#pragma unroll
          for (int j = 0; j < NT8; j += 2) {
            uint32_t b[4], bl[4];
            const uint32_t ro = (16 * kk + (lane & 7) + 8 * (mq & 1)) * HROW + (hn0 + j + (mq >> 1)) * 16;
            ldsm_x4_t(aVS + ro, b);
            ldsm_x4_t(aVSL + ro, bl);
            mma_bf16(hf[j], a, b[0], b[1]);
            mma_bf16(hf[j + 1], a, b[2], b[3]);
            mma_bf16(hl[j], a, bl[0], bl[1]);
            mma_bf16(hl[j + 1], a, bl[2], bl[3]);
          }
        }
#pragma unroll
        for (int j = 0; j < NT8; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) hf[j][e] += hl[j][e];
      }
      if (go) arrive(CDONE, c);  // this chunk's stage is no longer read by the chain
      go = waitc(SHDONE, c) && go;  // the side group has read h_c
      if (go) write_h();
      named_bar_sync(1, NTH);
      if (go) arrive(HREADY, c + 1);
    }
    if (ht && !*abort_flag) {
#pragma unroll
      for (int j = 0; j < NT8; ++j)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int key = 16 * hm + g4 + 8 * hh;
          const int col = 8 * (hn0 + j) + 2 * t4;
          *reinterpret_cast<float2 *>(ht + (sbase + key) * V + vt0 + col) = make_float2(hf[j][2 * hh], hf[j][2 * hh + 1]);
        }
    }
  } else {
    // ----------------------------------------------------------------- side
    const bool issuer = (tid == NTH);
    int tma_hi = 0;
    auto issue = [&](int c) {
      const int s = c % NS;
      const uint32_t st = sb + s * Ly::STAGE;
      const int trow = static_cast<int>(tok0) + c * C;
      mbar_arrive_expect_tx(bar(FULL, s), Ly::TX);
#pragma unroll
      for (int a = 0; a < KA; ++a) {
        tma_load_3d(st + a * 16384, &tm_k, bar(FULL, s), 64 * a, h, trow);
        tma_load_3d(st + a * 16384 + 8192, &tm_q, bar(FULL, s), 64 * a, h, trow);
      }
      tma_load_3d(st + Ly::KQB, &tm_v, bar(FULL, s), vt0, hv, trow);
      bulk_load(st + Ly::KQB + Ly::V_BYTES, ws + (static_cast<size_t>(cb + c) * HV + hv) * R::BYTES, R::BYTES,
                bar(FULL, s));
      tma_hi = c + 1;
    };
    if (issuer)
      for (int c = 0; c < NS && c < NC; ++c) issue(c);
    __syncwarp();
    const float dscale = scale;
    for (int c = 0; c < NC; ++c) {
      const int s = c % NS;
      const uint32_t st = sb + s * Ly::STAGE;
      const uint32_t rc = st + Ly::KQB + Ly::V_BYTES;
      const float *rsc = reinterpret_cast<const float *>(sm + s * Ly::STAGE + Ly::KQB + Ly::V_BYTES + R::SC);
      const int64_t remc = len - static_cast<int64_t>(c) * C;
      const int L = static_cast<int>(remc < C ? remc : C);
      const int64_t trow0 = tok0 + static_cast<int64_t>(c) * C;
      // Q h_c, h as hi + lo.
      bool go = waitc(FULL, c);
      go = waitc(HREADY, c) && go;
      float aq[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      float aql[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if (go) {
#pragma unroll
      for (int kk = 0; kk < K / 16; ++kk) {
        uint32_t fq[4], b[4], bl[4];
        ldsm_x4(tile_addr(st, 128, 64 + 16 * mi + (lane & 15), 2 * kk + (lane >> 4)), fq);
        const int mq = lane >> 3;
        const uint32_t ho = (16 * kk + (lane & 7) + 8 * (mq & 1)) * HROW + (2 * nh + (mq >> 1)) * 16;
        ldsm_x4_t(aH + ho, b);
        ldsm_x4_t(aHL + ho, bl);
        mma_bf16(aq[0], fq, b[0], b[1]);
        mma_bf16(aq[1], fq, b[2], b[3]);
        mma_bf16(aql[0], fq, bl[0], bl[1]);
        mma_bf16(aql[1], fq, bl[2], bl[3]);
      }
      arrive(SHDONE, c);
      }
      // o = scale (e^gamma rq (Q h) + P v_new), P and v_new as bf16 hi + lo.
      go = waitc(VREADY, c) && go;
      float ac[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if (go) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t ph[4], pl[4], bh[4], bl[4];
        ldsm_x4(rc + R::PH + sw128(16 * mi + (lane & 15), 2 * kk + (lane >> 4)), ph);
        ldsm_x4(rc + R::PL + sw128(16 * mi + (lane & 15), 2 * kk + (lane >> 4)), pl);
        const int mq = lane >> 3;
        const uint32_t ro = (16 * kk + (lane & 7) + 8 * (mq & 1)) * HROW + (2 * nh + (mq >> 1)) * 16;
        ldsm_x4_t(aVH + ro, bh);
        ldsm_x4_t(aVL + ro, bl);
        mma_bf16(ac[0], ph, bh[0], bh[1]);
        mma_bf16(ac[1], ph, bh[2], bh[3]);
        mma_bf16(ac[0], ph, bl[0], bl[1]);
        mma_bf16(ac[1], ph, bl[2], bl[3]);
        mma_bf16(ac[0], pl, bh[0], bh[1]);
        mma_bf16(ac[1], pl, bh[2], bh[3]);
      }
      arrive(SVDONE, c);
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int r = 16 * mi + g4 + 8 * hh;
          if (r < L) {
            const int col = 16 * nh + 8 * j + 2 * t4;
            const float ogr = rsc[RS_OG + r];
            const float o0 = dscale * (ogr * (aq[j][2 * hh] + aql[j][2 * hh]) + ac[j][2 * hh]);
            const float o1 = dscale * (ogr * (aq[j][2 * hh + 1] + aql[j][2 * hh + 1]) + ac[j][2 * hh + 1]);
            *reinterpret_cast<uint32_t *>(o + ((trow0 + r) * HV + hv) * V + vt0 + col) = pack_bf16(o0, o1);
          }
        }
      }
      // Both groups are done with stage s once the chain has signalled and every
      // side warp is past this point: refill it with chunk c + 2.
      named_bar_sync(2, NTH);
      if (warp == 8 && c + NS < NC) {
        const bool can = waitc(CDONE, c) && go;
        if (issuer && can) issue(c + NS);
        __syncwarp();
      }
    }
    if (issuer && *abort_flag) {
      // Nothing of this CTA may still be in flight at exit.
      for (int k = (tma_hi > NS ? tma_hi - NS : 0); k < tma_hi; ++k)
        mbar_wait_bounded(bar(FULL, k % NS), (k / NS) & 1, kWaitLimit);
    }
  }
  __syncthreads();
  if (tid == 0 && *abort_flag) set_status(dev_status, GDN_DEV_WAIT_TIMEOUT);
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

int64_t total_chunk_slots(int B, int T, int N, bool varlen) {
  const int64_t per = (static_cast<int64_t>(T) + C - 1) / C;
  return varlen ? per + N : static_cast<int64_t>(B) * per;
}

template <int K>
size_t ws_bytes(int B, int T, int HV, int N, bool varlen) {
  return static_cast<size_t>(total_chunk_slots(B, T, N, varlen)) * HV * Rec<K>::BYTES;
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
                   !make_map(&mv, a.v, a.V, a.HV, rows, VT, false)))
    return cudaErrorInvalidValue;
  const int64_t slots = total_chunk_slots(a.B, a.T, a.N, a.cu != nullptr);
  if (rows > 0 && slots > 0) {
    const int psmem = PrepLay<K>::BYTES + 1024;
    cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, psmem);
    if (e != cudaSuccess) return e;
    dim3 pgrid(static_cast<unsigned>(slots), a.HV);
    chunk_prep_kernel<K><<<pgrid, NTH, psmem, s>>>(mq, mk, a.g, a.beta, a.cu, a.N, a.T, a.H, a.HV, a.l2,
                                                   static_cast<unsigned char *>(a.ws), a.dev_status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int wsmem = WalkLay<K>::BYTES + 1024;
  cudaError_t e = cudaFuncSetAttribute(chunk_walk_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, wsmem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.V / VT, a.HV, a.N);
  chunk_walk_kernel<K><<<grid, WNTH, wsmem, s>>>(mq, mk, mv, a.scale, a.h0, a.cu, a.T, a.H, a.HV, a.V,
                                                static_cast<const unsigned char *>(a.ws), a.o, a.ht, a.dev_status);
  return cudaGetLastError();
}

}  // namespace

namespace gdn_host {

size_t chunk_workspace_bytes(int B, int T, int H, int HV, int K, int V, int N, int varlen) {
  (void)H;
  (void)V;
  if (K == 128) return ws_bytes<128>(B, T, HV, N, varlen != 0);
  if (K == 64) return ws_bytes<64>(B, T, HV, N, varlen != 0);
  return 0;
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
