// gdn_chunk_tc.cu -- fused chunked prefill for sm_103a (tensor cores).
//
// Algorithm: the six steps of "NPU Training Operators - GDN", section
// "Operator semantics", for chunk size 64 (chunk-local cumsum of g, beta K K^T
// with gate decay, triangular solve, w/u recompute, inter-chunk state
// propagation, output), computed for one (sequence, value head, 32-column
// slice of V) per CTA.  The CTA walks the chunks of its sequence in order and
// keeps its K x 32 slice of the fp32 state h in registers for the whole walk;
// no per-chunk intermediate ever reaches global memory.
//
// Per chunk (rows i, j in [0, 64), L valid rows, gamma = cumsum g,
// rk/rq = 1/||k||, 1/||q|| (or 1 without the L2 norm), raw bf16 k, q, v):
//   [K;Q][K;Q]^T         tcgen05.mma, M=128 N=128, TMA-fed smem -> TMEM     (issued ahead by one thread;
//                        its diagonal gives ||k||^2 and ||q||^2)
//   A_ij = beta_i e^{gamma_i-gamma_j} rk_i rk_j (k_i.k_j)     i > j         (from TMEM)
//   P_ij = e^{gamma_i-gamma_j} rq_i rk_j (q_i.k_j)            j <= i        (from TMEM)
//   T    = (I + A)^{-1}                    16x16 diagonal blocks by substitution (fp32),
//                                          off-diagonal blocks by tf32 mma.sync
//   W    = [T diag(beta e^gamma rk)] K     (w of the WY form)               mma.sync
//   U    = beta v + [(T - I) diag(beta)] V (u of the WY form)               mma.sync
//   Z    = [Q; W] h                        (one product for Q h and W h)    mma.sync
//   v_new = U - W h,  o = scale (e^gamma rq Q h + P v_new)
//   h    = e^{gamma_L} h + K^T diag(e^{gamma_L-gamma} rk) v_new             mma.sync
// Precision: the main terms of o (P v_new and Q h) and the state update get
// their computed factor split into bf16 hi + lo parts (the raw bf16 q, k, v
// are exact); W, T diag(.) and the h in W h are plain bf16; fp32 accumulation
// throughout, and h, A, T stay fp32.
//
// Roles: eight warps compute; thread 0 also issues, at each chunk boundary,
// the TMA loads of chunk c+2 (three-stage ring) and the tcgen05.mma of chunk
// c+1, so copies and the K K^T / Q K^T product run ahead of the walk.  Every
// mbarrier wait is bounded; on expiry the CTA records GDN_DEV_WAIT_TIMEOUT,
// drains its outstanding copies and leaves.
#include <cuda.h>

#include "gdn_common.cuh"
#include "gdn_sm103.cuh"

namespace {

using namespace gdn;

constexpr int C = 64;
constexpr int VT = 32;
constexpr int NCW = 8;                    // compute warps
constexpr int NTH = NCW * 32;
constexpr long long kWaitLimit = 2000000000LL;  // clock cycles (about 1 s) before a wait gives up
constexpr int HROW = 80;                  // bytes per padded row of 32 bf16 (64 B + 16 B pad)
constexpr int FROW = 68;                  // floats per padded fp32 row of 64

template <int K>
struct Lay {
  static constexpr int KA = K / 64;                // 64-key atom columns
  static constexpr int KQ_BYTES = KA * 16384;      // [K;Q]: 128 rows x 128 B per atom column
  static constexpr int V_BYTES = C * VT * 2;       // 64 x 32 bf16, unswizzled
  static constexpr int STAGE = KQ_BYTES + V_BYTES;
  static constexpr int NS = 3;                     // stages in the TMA ring
  static constexpr int OFF_W = NS * STAGE;         // W [64][K] bf16, SW128, KA x 8 KB
  static constexpr int OFF_PH = OFF_W + KA * 8192; // P hi [64][64] bf16, SW128
  static constexpr int OFF_PL = OFF_PH + 8192;     // P lo
  static constexpr int OFF_TP = OFF_PL + 8192;     // T diag(beta e^g rk) bf16, SW128
  static constexpr int OFF_TS = OFF_TP + 8192;     // (T - I) diag(beta) bf16, SW128
  static constexpr int OFF_A = OFF_TS + 8192;      // A fp32 [64][FROW]
  static constexpr int OFF_T = OFF_A + 64 * FROW * 4;
  static constexpr int OFF_X = OFF_T + 64 * FROW * 4;     // 4 x [16][17] fp32 scratch
  static constexpr int OFF_H = OFF_X + 4352;              // h as bf16 hi [K][HROW] then lo [K][HROW]
  // The four v_new tiles [64][HROW] live in the A / T scratch, which is dead
  // from the end of step 6 until the next chunk's step 3.
  static constexpr int OFF_VS = OFF_A;                    // s * v_new, bf16 hi
  static constexpr int OFF_VSL = OFF_VS + 64 * HROW;      // s * v_new, bf16 lo
  static constexpr int OFF_VH = OFF_VSL + 64 * HROW;      // v_new hi
  static constexpr int OFF_VL = OFF_VH + 64 * HROW;       // v_new lo
  static constexpr int OFF_SC = OFF_H + 2 * K * HROW;     // scalars: 10 x 64 fp32
  static constexpr int OFF_BAR = OFF_SC + 10 * 64 * 4;    // 4 x NS mbarriers
  static constexpr int OFF_MISC = OFF_BAR + 4 * NS * 8;   // tmem base, abort flag
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr uint32_t TX = KQ_BYTES + V_BYTES;      // bytes per stage fill
  static_assert(STAGE % 1024 == 0, "stage alignment");
  static_assert(4 * 64 * HROW <= 2 * 64 * FROW * 4, "v_new tiles fit in the A/T scratch");
  static_assert(BYTES + 1024 <= 232448, "shared memory budget (227 KB per CTA)");
};

// Per-row scalars of a chunk: gamma * log2(e), beta, 1/||k||, 1/||q||,
// e^gamma / ||q||, e^{gamma_L - gamma} / ||k||, beta e^gamma / ||k||.
// When the chunk's total decay fits the fp32 range, e^{gamma_i - gamma_j} is
// factored as row * column factors relative to gamma_0 (rowA, rowP, colf);
// otherwise every element takes its own exponential.
enum { SC_GL = 0, SC_BET = 1, SC_RK = 2, SC_RQ = 3, SC_OG = 4, SC_SV = 5, SC_FTP = 6, SC_RA = 7, SC_RP = 8,
       SC_CF = 9 };
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ unsigned char *align1024(unsigned char *p) {
  return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

// Address of the 16-byte chunk holding keys [8*kc, 8*kc+8) of row `row` in a
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
// fp32 bits fed straight to a tf32 mma (the unit ignores the low mantissa bits).
__device__ __forceinline__ uint32_t to_tf32(float x) { return __float_as_uint(x); }

// acc (16 x 16 as two 16x8 tf32 mma tiles) += A (16 x 16) * B (16 x 16), both
// fp32 row-major in shared memory with leading dimensions lda / ldb.
__device__ __forceinline__ void mm16_tf32(const float *A, int lda, const float *B, int ldb, float acc[2][4], int g4,
                                          int t4) {
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    const uint32_t a0 = to_tf32(A[g4 * lda + 8 * ks + t4]);
    const uint32_t a1 = to_tf32(A[(g4 + 8) * lda + 8 * ks + t4]);
    const uint32_t a2 = to_tf32(A[g4 * lda + 8 * ks + t4 + 4]);
    const uint32_t a3 = to_tf32(A[(g4 + 8) * lda + 8 * ks + t4 + 4]);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const uint32_t b0 = to_tf32(B[(8 * ks + t4) * ldb + 8 * nt + g4]);
      const uint32_t b1 = to_tf32(B[(8 * ks + t4 + 4) * ldb + 8 * nt + g4]);
      asm volatile(
          "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
          "{%0,%1,%2,%3};"
          : "+f"(acc[nt][0]), "+f"(acc[nt][1]), "+f"(acc[nt][2]), "+f"(acc[nt][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
  }
}

template <int K>
__global__ void __launch_bounds__(NTH, 1) chunk_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const float *__restrict__ g, const float *__restrict__ beta,
    float scale, const float *__restrict__ h0, const int32_t *__restrict__ cu, int T, int H, int HV, int V, int l2,
    uint16_t *__restrict__ o, float *__restrict__ ht, int32_t *dev_status) {
  using Ly = Lay<K>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = align1024(smem_raw);
  const uint32_t sb = smem_u32(sm);
  const int vt0 = blockIdx.x * VT, hv = blockIdx.y, n = blockIdx.z;
  const int h = hv / (HV / H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  int64_t tok0, len;
  if (cu) {
    const int32_t a0 = cu[n], a1 = cu[n + 1];
    if (a0 < 0 || a1 < a0 || a1 > T || (n == 0 && a0 != 0)) {
      if (tid == 0) set_status(dev_status, GDN_DEV_BAD_CU_SEQLENS);
      return;
    }
    tok0 = a0;
    len = a1 - a0;
  } else {
    tok0 = static_cast<int64_t>(n) * T;
    len = T;
  }
  const int NC = static_cast<int>((len + C - 1) / C);

  float *scal = reinterpret_cast<float *>(sm + Ly::OFF_SC);
  float *Am = reinterpret_cast<float *>(sm + Ly::OFF_A);
  float *Tm = reinterpret_cast<float *>(sm + Ly::OFF_T);
  float *Xs = reinterpret_cast<float *>(sm + Ly::OFF_X);
  uint32_t *misc = reinterpret_cast<uint32_t *>(sm + Ly::OFF_MISC);
  volatile uint32_t *abort_flag = misc + 1;
  const uint32_t bar0 = sb + Ly::OFF_BAR;
  constexpr int NS = Ly::NS;
  auto b_full = [&](int s) { return bar0 + 8 * s; };
  auto b_kqf = [&](int s) { return bar0 + 8 * (NS + s); };

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(b_full(s), 1);
      mbar_init(b_kqf(s), 1);
    }
    misc[1] = 0;
    misc[2] = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(sb + Ly::OFF_MISC, 512);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  {
    // ------------------------------------------------------------ compute
    constexpr int MTH = K / 16;             // m-tiles of the state (16 keys each)
    constexpr int NTH_ = (K / 16) * 4 / NCW; // n-tiles (8 columns) of the state per warp
    const int g4 = lane >> 2, t4 = lane & 3;
    const int hm = warp % MTH;               // state m-tile of this warp
    const int hn0 = (warp / MTH) * NTH_;     // first state n-tile of this warp
    const int mi = warp & 3;                 // 16-row tile for the 64-row products
    const int nh = warp >> 2;                // which 16-column half of the 32-column slice
    const float dscale = scale;
    float hf[NTH_][4];
    const int64_t sbase = (static_cast<int64_t>(n) * HV + hv) * K;  // state row base
#pragma unroll
    for (int j = 0; j < NTH_; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = 16 * hm + g4 + 8 * (e >> 1);
        const int col = 8 * (hn0 + j) + 2 * t4 + (e & 1);
        hf[j][e] = h0 ? h0[(sbase + key) * V + vt0 + col] : 0.f;
      }
    unsigned char *Hb = sm + Ly::OFF_H;
    // h goes to shared memory as bf16 hi + lo planes (the B operand of [Q; W] h).
    auto write_h = [&]() {
#pragma unroll
      for (int j = 0; j < NTH_; ++j)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int key = 16 * hm + g4 + 8 * hh;
          const int col = 8 * (hn0 + j) + 2 * t4;
          const float x0 = hf[j][2 * hh], x1 = hf[j][2 * hh + 1];
          const uint32_t hi = pack_bf16(x0, x1);
          *reinterpret_cast<uint32_t *>(Hb + key * HROW + col * 2) = hi;
          *reinterpret_cast<uint32_t *>(Hb + (K + key) * HROW + col * 2) =
              pack_bf16(x0 - bf16lo_f(hi), x1 - bf16hi_f(hi));
        }
    };
    write_h();
    named_bar_sync(1, NCW * 32);

    const uint32_t aW = sb + Ly::OFF_W, aPH = sb + Ly::OFF_PH, aPL = sb + Ly::OFF_PL;
    const uint32_t aTP = sb + Ly::OFF_TP, aTS = sb + Ly::OFF_TS;
    const uint32_t aH = sb + Ly::OFF_H, aHL = sb + Ly::OFF_H + K * HROW;
    const uint32_t aVS = sb + Ly::OFF_VS, aVSL = sb + Ly::OFF_VSL, aVH = sb + Ly::OFF_VH, aVL = sb + Ly::OFF_VL;
    float *gl = scal + SC_GL * 64, *bet = scal + SC_BET * 64, *rk = scal + SC_RK * 64;
    float *rq = scal + SC_RQ * 64, *og = scal + SC_OG * 64, *sv = scal + SC_SV * 64;
    float *ftp = scal + SC_FTP * 64;
    auto rows_of = [&](int c) {
      const int64_t rem = len - static_cast<int64_t>(c) * C;
      return static_cast<int>(rem < C ? rem : C);
    };
    // Gates of the next chunk are loaded one chunk ahead by warp 4 (two rows per lane).
    float g_nx[2] = {0.f, 0.f}, b_nx[2] = {0.f, 0.f};
    if (warp == 4 && NC > 0) {
      const int L0 = rows_of(0);
#pragma unroll
      for (int u2 = 0; u2 < 2; ++u2) {
        const int r = 2 * lane + u2;
        if (r < L0) {
          g_nx[u2] = g[(tok0 + r) * HV + hv];
          b_nx[u2] = beta[(tok0 + r) * HV + hv];
        }
      }
    }
    const int quad = warp & 3, half = warp >> 2;
    const int row = 32 * quad + lane;  // row of [K; Q] served by this thread in TMEM

    // Thread 0 drives the copies and the tensor-core product: chunk c lives in
    // stage / TMEM buffer c % NS.  At the start of chunk c (all warps are past
    // chunk c-1) it refills the stage chunk c-1 used with chunk c+NS-1 and
    // issues [K;Q][K;Q]^T for chunk c+1, so both run a chunk or more ahead.
    int tma_hi = 0, mma_hi = 0, c_waited = 0;
    auto issue_tma = [&](int c) {
      const int s = c % NS;
      const uint32_t st = sb + s * Ly::STAGE;
      const int trow = static_cast<int>(tok0) + c * C;
      mbar_arrive_expect_tx(b_full(s), Ly::TX);
#pragma unroll
      for (int a = 0; a < Ly::KA; ++a) {
        tma_load_3d(st + a * 16384, &tm_k, b_full(s), 64 * a, h, trow);
        tma_load_3d(st + a * 16384 + 8192, &tm_q, b_full(s), 64 * a, h, trow);
      }
      tma_load_3d(st + Ly::KQ_BYTES, &tm_v, b_full(s), vt0, hv, trow);
      tma_hi = c + 1;
    };
    // [K; Q] [K; Q]^T: rows 0-63 hold K K^T | K Q^T, rows 64-127 Q K^T | Q Q^T.
    auto issue_mma = [&](int c) {
      const int s = c % NS;
      if (!mbar_wait_bounded(b_full(s), (c / NS) & 1, kWaitLimit)) {
        *abort_flag = 1;
        return;
      }
      tc_fence_after();
      constexpr uint32_t idesc = umma_idesc_bf16(128, 128);
      const uint32_t st = sb + s * Ly::STAGE;
#pragma unroll
      for (int kk = 0; kk < K / 16; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint64_t d = umma_desc_sw128(st + off);
        umma_bf16(tmem + s * 128, d, d, idesc, kk > 0 ? 1u : 0u);
      }
      umma_commit(b_kqf(s));
      mma_hi = c + 1;
    };
    const bool issuer = (tid == 128);  // warp 4, lane 0 (idle while warps 0-3 run step 4a)
    if (issuer && NC > 0) {
      for (int c = 0; c < NS - 1 && c < NC; ++c) issue_tma(c);
      issue_mma(0);
    }

    for (int c = 0; c < NC; ++c) {
      const int s = c % NS;
      const uint32_t par = (c / NS) & 1;
      unsigned char *stp = sm + s * Ly::STAGE;
      const uint32_t st = sb + s * Ly::STAGE;
      const uint32_t stV = st + Ly::KQ_BYTES;
      const int L = rows_of(c);
      const int64_t trow0 = tok0 + static_cast<int64_t>(c) * C;

      // 1. warp 4: this chunk's gates, chunk-local cumsum of g (in base 2), next
      //    chunk's gates requested.  Every warp: tiles landed, 32 columns of
      //    [K;Q][K;Q]^T from TMEM; the row norms are its diagonal.
      if (!mbar_wait_bounded(b_full(s), par, kWaitLimit)) *abort_flag = 1;
      if (warp == 4) {
        const float x0 = g_nx[0], x1 = g_nx[1];
        bet[2 * lane] = b_nx[0];
        bet[2 * lane + 1] = b_nx[1];
        float sum = x0 + x1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, sum, off);
          if (lane >= off) sum += y;
        }
        const float excl = sum - (x0 + x1);
        gl[2 * lane] = (excl + x0) * kLog2e;
        gl[2 * lane + 1] = sum * kLog2e;
        const int Ln = (c + 1 < NC) ? rows_of(c + 1) : 0;
#pragma unroll
        for (int u2 = 0; u2 < 2; ++u2) {
          const int r = 2 * lane + u2;
          g_nx[u2] = 0.f;
          b_nx[u2] = 0.f;
          if (r < Ln) {
            g_nx[u2] = g[(trow0 + C + r) * HV + hv];
            b_nx[u2] = beta[(trow0 + C + r) * HV + hv];
          }
        }
      }
      if (!mbar_wait_bounded(b_kqf(s), par, kWaitLimit)) *abort_flag = 1;
      tc_fence_after();
      const uint32_t tl = tmem + (static_cast<uint32_t>(32 * quad) << 16) + s * 128;
      float vals[32];
      tmem_ld32(tl + half * 32, vals);
      if (l2) {
        // K K^T diagonal: warps (quad 0, half 0) and (quad 1, half 1);
        // Q Q^T diagonal (columns 64..127): warps 2 and 7 load it separately.
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
      tc_fence_before();
      if (tid == 0) misc[2] = *abort_flag;  // one snapshot, read by every warp after the barrier
      named_bar_sync(1, NCW * 32);
      if (misc[2]) break;

      // 2. per-row factors.
      const bool fact = (gl[0] - gl[63]) < 120.f;  // chunk decay fits the fp32 range
      if (tid < 64) {
        const float gi = gl[tid];
        const float e = ex2(gi);
        og[tid] = e * rq[tid];
        sv[tid] = ex2(gl[63] - gi) * rk[tid];
        ftp[tid] = bet[tid] * e * rk[tid];
        const float er = ex2(gi - gl[0]);
        scal[SC_RA * 64 + tid] = bet[tid] * rk[tid] * er;
        scal[SC_RP * 64 + tid] = rq[tid] * er;
        scal[SC_CF * 64 + tid] = fact ? rk[tid] * ex2(gl[0] - gi) : 0.f;
      }
      named_bar_sync(1, NCW * 32);

      // 3. A = strictly-lower beta_i e^{gamma_i-gamma_j} rk_i rk_j (k_i.k_j) (fp32; only
      //    j < i is stored, the solve reads nothing else) and
      //    P = causal e^{gamma_i-gamma_j} rq_i rk_j (q_i.k_j) as bf16 hi + lo.
      {
        const float *colf = scal + SC_CF * 64;
        if (row < 64) {
          const int i = row;
          const float ra = scal[SC_RA * 64 + i], gi = gl[i], ci = bet[i] * rk[i];
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
              *reinterpret_cast<float4 *>(Am + i * FROW + j0) = make_float4(a4[0], a4[1], a4[2], a4[3]);
            }
          }
        } else {
          const int i = row - 64;
          const float rp = scal[SC_RP * 64 + i], gi = gl[i], ci = rq[i];
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
            *reinterpret_cast<uint4 *>(sm + Ly::OFF_PH + sw128(i, chunk)) = vh;
            *reinterpret_cast<uint4 *>(sm + Ly::OFF_PL + sw128(i, chunk)) = vl;
          }
        }
      }
      named_bar_sync(1, NCW * 32);

      // 4a. diagonal 16x16 blocks D_b of T = (I + A)^{-1} (warps 0-3, lanes 0-15: one
      //     column each, right-looking substitution); warps 4-7 zero the rows >= L
      //     of this stage's tiles.
      if (warp < 4) {
        if (lane < 16) {
          const int b0 = 16 * warp, col = lane;
          float x[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] = (i == col) ? 1.f : 0.f;
#pragma unroll
          for (int j = 0; j < 16; ++j)
#pragma unroll
            for (int i = j + 1; i < 16; ++i) x[i] = fmaf(-Am[(b0 + i) * FROW + b0 + j], x[j], x[i]);
#pragma unroll
          for (int i = 0; i < 16; ++i) Tm[(b0 + i) * FROW + b0 + col] = x[i];
        }
      } else {
        if (issuer) {
          // Chunk c-1 is done: its stage takes chunk c+2, and TMEM buffer
          // (c+1) % NS (last read in chunk c-2) takes the product of chunk c+1.
          if (c + NS - 1 < NC) issue_tma(c + NS - 1);
          if (c + 1 < NC && !*abort_flag) issue_mma(c + 1);
          c_waited = c + 1;
        }
        const int t2 = tid - 128;
        for (int e = t2; e < (C - L) * 8 * Ly::KA * 2; e += 128) {
          const int rr = e / (8 * Ly::KA * 2), rem = e % (8 * Ly::KA * 2);
          const int which = rem / (8 * Ly::KA), kc = rem % (8 * Ly::KA);
          const int zr = L + rr + 64 * which;
          *reinterpret_cast<uint4 *>(stp + (kc >> 3) * 16384 + sw128(zr, kc & 7)) = make_uint4(0, 0, 0, 0);
        }
        for (int e = t2; e < (C - L) * 4; e += 128) {
          const int zr = L + e / 4, q = e % 4;
          *reinterpret_cast<uint4 *>(stp + Ly::KQ_BYTES + zr * 64 + q * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      named_bar_sync(1, NCW * 32);
      // 4b. off-diagonal blocks, tf32 mma.sync on 16x16 tiles (one warp per tile):
      //     T10 = -D1 A10 D0, T32 = -D3 A32 D2; then the lower-left 32x32 block
      //     T[32:64, 0:32] = -T22 (A[32:64, 0:32] T11).
      {
        auto blk = [&](float *base, int bi, int bj) { return base + 16 * bi * FROW + 16 * bj; };
        auto store_c = [&](float *dst, int ld, float acc[2][4], float sgn) {
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            dst[g4 * ld + 8 * nt + 2 * t4] = sgn * acc[nt][0];
            dst[g4 * ld + 8 * nt + 2 * t4 + 1] = sgn * acc[nt][1];
            dst[(g4 + 8) * ld + 8 * nt + 2 * t4] = sgn * acc[nt][2];
            dst[(g4 + 8) * ld + 8 * nt + 2 * t4 + 1] = sgn * acc[nt][3];
          }
        };
        if (warp < 2) {
          const int bj = 2 * warp, bi = bj + 1;  // (1,0) and (3,2)
          float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
          mm16_tf32(blk(Am, bi, bj), FROW, blk(Tm, bj, bj), FROW, acc, g4, t4);
          float *X = Xs + warp * 272;
          store_c(X, 17, acc, 1.f);
          __syncwarp();
          float tt[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
          mm16_tf32(blk(Tm, bi, bi), FROW, X, 17, tt, g4, t4);
          store_c(blk(Tm, bi, bj), FROW, tt, -1.f);
        }
        named_bar_sync(1, NCW * 32);
        if (warp < 4) {
          // Y_{a,b} = sum_k A[2+a][k] T11[k][b]  (T11 = [[D0, 0], [T10, D1]])
          const int a = warp >> 1, b = warp & 1;
          float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
          for (int kb = b; kb < 2; ++kb) mm16_tf32(blk(Am, 2 + a, kb), FROW, blk(Tm, kb, b), FROW, acc, g4, t4);
          store_c(Xs + warp * 272, 17, acc, 1.f);
        }
        named_bar_sync(1, NCW * 32);
        if (warp < 4) {
          // T[2+a][b] = -sum_k T22[a][k] Y_{k,b}  (T22 = [[D2, 0], [T32, D3]])
          const int a = warp >> 1, b = warp & 1;
          float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
          for (int kb = 0; kb <= a; ++kb) mm16_tf32(blk(Tm, 2 + a, 2 + kb), FROW, Xs + (2 * kb + b) * 272, 17, acc, g4, t4);
          store_c(blk(Tm, 2 + a, b), FROW, acc, -1.f);
        }
        named_bar_sync(1, NCW * 32);
      }

      // 5. Tp = T diag(beta e^gamma rk) (j <= i), Ts = (T - I) diag(beta) (j < i), bf16.
      for (int e = tid; e < 64 * 8; e += NCW * 32) {
        const int i = e >> 3, ch = e & 7;
        uint4 tpv = make_uint4(0, 0, 0, 0), tsv = make_uint4(0, 0, 0, 0);
        if (8 * ch <= i) {
          const float4 t0 = *reinterpret_cast<const float4 *>(Tm + i * FROW + 8 * ch);
          const float4 t1 = *reinterpret_cast<const float4 *>(Tm + i * FROW + 8 * ch + 4);
          const float4 f0 = *reinterpret_cast<const float4 *>(ftp + 8 * ch);
          const float4 f1 = *reinterpret_cast<const float4 *>(ftp + 8 * ch + 4);
          const float4 b0 = *reinterpret_cast<const float4 *>(bet + 8 * ch);
          const float4 b1 = *reinterpret_cast<const float4 *>(bet + 8 * ch + 4);
          const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
          const float fv[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
          const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
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
        *reinterpret_cast<uint4 *>(sm + Ly::OFF_TS + sw128(i, ch)) = tsv;
      }
      named_bar_sync(1, NCW * 32);

      // 6. W = Tp K (64 x K) and U = beta v + Ts V (64 x 32, kept in registers).
      float u[2][4];
      {
        constexpr int WN = K / 16;  // n-tiles of W per warp (half of K / 8)
        float acc[WN][4];
#pragma unroll
        for (int j = 0; j < WN; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
        float au[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t a[4], as[4];
          ldsm_x4(aTP + sw128(16 * mi + (lane & 15), 2 * kk + (lane >> 4)), a);
          ldsm_x4(aTS + sw128(16 * mi + (lane & 15), 2 * kk + (lane >> 4)), as);
          const int mq = lane >> 3;
          const int trow = 16 * kk + (lane & 7) + 8 * (mq & 1);
#pragma unroll
          for (int j = 0; j < WN; j += 2) {
            const int kc = (nh * WN + j) + (mq >> 1);  // 8-key chunk index
            uint32_t b[4];
            ldsm_x4_t(tile_addr(st, 128, trow, kc), b);
            mma_bf16(acc[j], a, b[0], b[1]);
            mma_bf16(acc[j + 1], a, b[2], b[3]);
          }
          uint32_t bv[4];
          ldsm_x4_t(stV + trow * 64 + (2 * nh + (mq >> 1)) * 16, bv);
          mma_bf16(au[0], as, bv[0], bv[1]);
          mma_bf16(au[1], as, bv[2], bv[3]);
        }
#pragma unroll
        for (int j = 0; j < WN; ++j) {
          const int key = 8 * (nh * WN + j) + 2 * t4;
          const int r0 = 16 * mi + g4;
          const uint32_t base = Ly::OFF_W + (key >> 6) * 8192;
          *reinterpret_cast<uint32_t *>(sm + base + sw128(r0, (key & 63) >> 3) + (key & 7) * 2) =
              pack_bf16(acc[j][0], acc[j][1]);
          *reinterpret_cast<uint32_t *>(sm + base + sw128(r0 + 8, (key & 63) >> 3) + (key & 7) * 2) =
              pack_bf16(acc[j][2], acc[j][3]);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = 16 * mi + g4 + 8 * (e >> 1);
            const int col = 16 * nh + 8 * j + 2 * t4 + (e & 1);
            const float vv = bf2f(*reinterpret_cast<const uint16_t *>(stp + Ly::KQ_BYTES + r * 64 + col * 2));
            u[j][e] = fmaf(bet[r], vv, au[j][e]);
          }
      }
      named_bar_sync(1, NCW * 32);

      // 7. Z = [Q; W] h for rows 16 mi.. and columns 16 nh..: W h with the bf16 hi
      //    part of h (it only corrects U), Q h with hi + lo (it is a main term of o).
      float aq[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      float aql[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        float aw[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < K / 16; ++kk) {
          uint32_t fq[4], fw[4], b[4], bl[4];
          const int kc = 2 * kk + (lane >> 4);
          ldsm_x4(tile_addr(aW, 64, 16 * mi + (lane & 15), kc), fw);
          ldsm_x4(tile_addr(st, 128, 64 + 16 * mi + (lane & 15), kc), fq);
          const int mq = lane >> 3;
          const uint32_t ho = (16 * kk + (lane & 7) + 8 * (mq & 1)) * HROW + (2 * nh + (mq >> 1)) * 16;
          ldsm_x4_t(aH + ho, b);
          ldsm_x4_t(aHL + ho, bl);
          mma_bf16(aw[0], fw, b[0], b[1]);
          mma_bf16(aw[1], fw, b[2], b[3]);
          mma_bf16(aq[0], fq, b[0], b[1]);
          mma_bf16(aq[1], fq, b[2], b[3]);
          mma_bf16(aql[0], fq, bl[0], bl[1]);
          mma_bf16(aql[1], fq, bl[2], bl[3]);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int col = 16 * nh + 8 * j + 2 * t4;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int r = 16 * mi + g4 + 8 * hh;
            const float x0 = u[j][2 * hh] - aw[j][2 * hh], x1 = u[j][2 * hh + 1] - aw[j][2 * hh + 1];
            const uint32_t hi = pack_bf16(x0, x1);
            const uint32_t lo = pack_bf16(x0 - bf16lo_f(hi), x1 - bf16hi_f(hi));
            const float sr = sv[r];
            const float y0 = sr * x0, y1 = sr * x1;
            const uint32_t yh = pack_bf16(y0, y1);
            const uint32_t yl = pack_bf16(y0 - bf16lo_f(yh), y1 - bf16hi_f(yh));
            *reinterpret_cast<uint32_t *>(sm + Ly::OFF_VS + r * HROW + col * 2) = yh;
            *reinterpret_cast<uint32_t *>(sm + Ly::OFF_VSL + r * HROW + col * 2) = yl;
            *reinterpret_cast<uint32_t *>(sm + Ly::OFF_VH + r * HROW + col * 2) = hi;
            *reinterpret_cast<uint32_t *>(sm + Ly::OFF_VL + r * HROW + col * 2) = lo;
          }
        }
      }
      named_bar_sync(1, NCW * 32);

      // 8. h = e^{gamma_L} h + K^T (s v_new)  (state walk), then the bf16 copy for the next chunk.
      {
        const float dL = ex2(gl[63]);
        float hl[NTH_][4];
#pragma unroll
        for (int j = 0; j < NTH_; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            hf[j][e] *= dL;
            hl[j][e] = 0.f;
          }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int mq = lane >> 3;
          uint32_t a[4];
          // A = K^T: rows = keys 16 hm.., k = tokens 16 kk..; K is stored [token][key].
          ldsm_x4_t(tile_addr(st, 128, 16 * kk + (lane & 7) + 8 * (mq >> 1), 2 * hm + (mq & 1)), a);
#pragma unroll
          for (int j = 0; j < NTH_; j += 2) {
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
        for (int j = 0; j < NTH_; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) hf[j][e] += hl[j][e];
        write_h();
      }

      // 9. o = scale (o_inter + P v_new) with P and v_new split into bf16 hi + lo.
      {
        float ac[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t ph[4], pl[4], bh[4], bl[4];
          ldsm_x4(aPH + sw128(16 * mi + (lane & 15), 2 * kk + (lane >> 4)), ph);
          ldsm_x4(aPL + sw128(16 * mi + (lane & 15), 2 * kk + (lane >> 4)), pl);
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
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int r = 16 * mi + g4 + 8 * hh;
            if (r < L) {
              const int col = 16 * nh + 8 * j + 2 * t4;
              const float ogr = og[r];
              const float o0 = dscale * (ogr * (aq[j][2 * hh] + aql[j][2 * hh]) + ac[j][2 * hh]);
              const float o1 = dscale * (ogr * (aq[j][2 * hh + 1] + aql[j][2 * hh + 1]) + ac[j][2 * hh + 1]);
              *reinterpret_cast<uint32_t *>(o + ((trow0 + r) * HV + hv) * V + vt0 + col) = pack_bf16(o0, o1);
            }
          }
      }
      // 10. this stage is free for the next TMA fill (generic writes ordered before async-proxy ones).
      fence_proxy_async_smem();
      named_bar_sync(1, NCW * 32);
    }
    if (issuer) {
      // Nothing of this CTA may still be in flight at exit (only after an abort
      // can a copy or product be outstanding here).
      for (int k = c_waited; k < tma_hi; ++k) mbar_wait_bounded(b_full(k % NS), (k / NS) & 1, kWaitLimit);
      if (mma_hi > 0) mbar_wait_bounded(b_kqf((mma_hi - 1) % NS), ((mma_hi - 1) / NS) & 1, kWaitLimit);
      if (*abort_flag) set_status(dev_status, GDN_DEV_WAIT_TIMEOUT);
    }
    if (ht && !misc[2]) {
#pragma unroll
      for (int j = 0; j < NTH_; ++j)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int key = 16 * hm + g4 + 8 * hh;
          const int col = 8 * (hn0 + j) + 2 * t4;
          *reinterpret_cast<float2 *>(ht + (sbase + key) * V + vt0 + col) = make_float2(hf[j][2 * hh], hf[j][2 * hh + 1]);
        }
    }
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
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

// 3-D map over a [rows][heads][dim] bf16 tensor with a box of
// {box0 elements, 1 head, 64 rows}.
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
cudaError_t launch_k(const gdn_host::ChunkArgs &a, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(a.B) * a.T;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, K, a.H, rows, 64, true) || !make_map(&mk, a.k, K, a.H, rows, 64, true) ||
      !make_map(&mv, a.v, a.V, a.HV, rows, VT, false))
    return cudaErrorInvalidValue;
  const int smem = Lay<K>::BYTES + 1024;
  cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.V / VT, a.HV, a.N);
  chunk_tc_kernel<K><<<grid, NTH, smem, s>>>(mq, mk, mv, a.g, a.beta, a.scale, a.h0, a.cu, a.T,
                                             a.H, a.HV, a.V, a.l2, a.o, a.ht, a.dev_status);
  return cudaGetLastError();
}

}  // namespace

namespace gdn_host {

size_t chunk_workspace_bytes(int, int, int, int, int, int, int, int) { return 0; }

cudaError_t launch_chunk(const ChunkArgs &a, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  if (a.K == 128) return launch_k<128>(a, s);
  if (a.K == 64) return launch_k<64>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace gdn_host
