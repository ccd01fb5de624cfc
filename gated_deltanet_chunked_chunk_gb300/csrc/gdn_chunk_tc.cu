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
//   [K;Q] K^T            tcgen05.mma, M=128 N=64, TMA-fed smem -> TMEM      (issued ahead by one thread)
//   A_ij = beta_i e^{gamma_i-gamma_j} rk_i rk_j (k_i.k_j)     i > j         (from TMEM)
//   P_ij = e^{gamma_i-gamma_j} rq_i rk_j (q_i.k_j)            j <= i        (from TMEM)
//   T    = (I + A)^{-1}                    blocked 16x16 forward substitution, fp32
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
// Roles: warps 0-7 compute; warp 8 lane 0 issues the TMA loads (three-stage
// ring) and the tcgen05.mma for chunk c as soon as its tiles land, so the
// K K^T / Q K^T product of the next chunk runs while the current one is
// being walked.  Every mbarrier wait is bounded; on expiry the CTA records
// GDN_DEV_WAIT_TIMEOUT, drains its outstanding copies and leaves.
#include <cuda.h>

#include "gdn_common.cuh"
#include "gdn_sm103.cuh"

namespace {

using namespace gdn;

constexpr int C = 64;
constexpr int VT = 32;
constexpr int NCW = 8;                    // compute warps
constexpr int NTH = (NCW + 1) * 32;       // + one control warp
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
  static constexpr int OFF_X = OFF_T + 64 * FROW * 4;     // 3 x [16][17] fp32 scratch
  static constexpr int OFF_H = OFF_X + 3328;              // h as bf16 hi [K][HROW] then lo [K][HROW]
  // The four v_new tiles [64][HROW] live in the A / T scratch, which is dead
  // from the end of step 6 until the next chunk's step 3.
  static constexpr int OFF_VS = OFF_A;                    // s * v_new, bf16 hi
  static constexpr int OFF_VSL = OFF_VS + 64 * HROW;      // s * v_new, bf16 lo
  static constexpr int OFF_VH = OFF_VSL + 64 * HROW;      // v_new hi
  static constexpr int OFF_VL = OFF_VH + 64 * HROW;       // v_new lo
  static constexpr int OFF_SC = OFF_H + 2 * K * HROW;     // scalars: 6 x 64 fp32
  static constexpr int OFF_BAR = OFF_SC + 6 * 64 * 4;     // 4 x NS mbarriers
  static constexpr int OFF_MISC = OFF_BAR + 4 * NS * 8;   // tmem base, abort flag
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr uint32_t TX = KQ_BYTES + V_BYTES;      // bytes per stage fill
  static_assert(STAGE % 1024 == 0, "stage alignment");
  static_assert(4 * 64 * HROW <= 2 * 64 * FROW * 4, "v_new tiles fit in the A/T scratch");
  static_assert(BYTES + 1024 <= 232448, "shared memory budget (227 KB per CTA)");
};

enum { SC_GAM = 0, SC_BET = 1, SC_RK = 2, SC_RQ = 3, SC_OG = 4, SC_SV = 5 };

__device__ __forceinline__ unsigned char *align1024(unsigned char *p) {
  return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

// Address of the 16-byte chunk holding keys [8*kc, 8*kc+8) of row `row` in a
// [rows][K] bf16 tile stored as 64-key SW128 atom columns of `rows` rows.
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int rows, int row, int kc) {
  return base + (kc >> 3) * (rows * 128) + sw128(row, kc & 7);
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
  auto b_empty = [&](int s) { return bar0 + 8 * (NS + s); };
  auto b_kqf = [&](int s) { return bar0 + 8 * (2 * NS + s); };
  auto b_kqe = [&](int s) { return bar0 + 8 * (3 * NS + s); };

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(b_full(s), 1);
      mbar_init(b_empty(s), NCW);
      mbar_init(b_kqf(s), 1);
      mbar_init(b_kqe(s), NCW);
    }
    misc[1] = 0;
    misc[2] = 0;
    mbar_fence_init();
  }
  if (warp == NCW) tmem_alloc(sb + Ly::OFF_MISC, 256);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  if (warp == NCW) {
    // ------------------------------------------------------------ control
    if (lane == 0 && NC > 0) {
      // Chunk c lives in stage / TMEM buffer c % NS.  The product for chunk c is
      // issued as soon as its tiles land; the refill of chunk c + NS - 1 waits
      // for chunk c - 1 to be released, so the ring runs NS - 1 chunks ahead.
      bool pend_tma[NS];
      uint32_t pend_par[NS];
      for (int s = 0; s < NS; ++s) { pend_tma[s] = false; pend_par[s] = 0; }
      int last_mma = -1;
      auto issue = [&](int c) {
        const int s = c % NS;
        const uint32_t st = sb + s * Ly::STAGE;
        const int row = static_cast<int>(tok0) + c * C;
        mbar_arrive_expect_tx(b_full(s), Ly::TX);
#pragma unroll
        for (int a = 0; a < Ly::KA; ++a) {
          tma_load_3d(st + a * 16384, &tm_k, b_full(s), 64 * a, h, row);
          tma_load_3d(st + a * 16384 + 8192, &tm_q, b_full(s), 64 * a, h, row);
        }
        tma_load_3d(st + Ly::KQ_BYTES, &tm_v, b_full(s), vt0, hv, row);
        pend_tma[s] = true;
        pend_par[s] = (c / NS) & 1;
      };
      for (int c = 0; c < NS - 1 && c < NC; ++c) issue(c);
      constexpr uint32_t idesc = umma_idesc_bf16(128, 64);
      for (int c = 0; c < NC; ++c) {
        const int s = c % NS;
        if (*abort_flag) break;
        if (!mbar_wait_bounded(b_full(s), (c / NS) & 1, kWaitLimit)) { *abort_flag = 1; break; }
        pend_tma[s] = false;
        if (c >= NS && !mbar_wait_bounded(b_kqe(s), ((c - NS) / NS) & 1, kWaitLimit)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t st = sb + s * Ly::STAGE;
#pragma unroll
        for (int kk = 0; kk < K / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint64_t d = umma_desc_sw128(st + off);
          umma_bf16(tmem + s * 64, d, d, idesc, kk > 0 ? 1u : 0u);
        }
        umma_commit(b_kqf(s));
        last_mma = c;
        const int nxt = c + NS - 1;  // refill the stage that chunk c - 1 used
        if (nxt < NC) {
          if (c >= 1 && !mbar_wait_bounded(b_empty((c - 1) % NS), ((c - 1) / NS) & 1, kWaitLimit)) {
            *abort_flag = 1;
            break;
          }
          issue(nxt);
        }
      }
      // Drain: no copy or MMA of this CTA may still be in flight at exit.
      for (int s = 0; s < NS; ++s)
        if (pend_tma[s]) mbar_wait_bounded(b_full(s), pend_par[s], kWaitLimit);
      if (last_mma >= 0) mbar_wait_bounded(b_kqf(last_mma % NS), (last_mma / NS) & 1, kWaitLimit);
      if (*abort_flag) set_status(dev_status, GDN_DEV_WAIT_TIMEOUT);
    }
    __syncwarp();
  } else {
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
    float *gam = scal + SC_GAM * 64, *bet = scal + SC_BET * 64, *rk = scal + SC_RK * 64;
    float *rq = scal + SC_RQ * 64, *og = scal + SC_OG * 64, *sv = scal + SC_SV * 64;

    for (int c = 0; c < NC; ++c) {
      const int s = c % NS;
      const uint32_t par = (c / NS) & 1;
      unsigned char *stp = sm + s * Ly::STAGE;
      const uint32_t st = sb + s * Ly::STAGE;
      const uint32_t stV = st + Ly::KQ_BYTES;
      const int L = static_cast<int>(len - static_cast<int64_t>(c) * C < C ? len - static_cast<int64_t>(c) * C : C);
      const int64_t trow0 = tok0 + static_cast<int64_t>(c) * C;

      // 1. tiles landed; gates of this chunk (rows >= L read as 0).
      if (!mbar_wait_bounded(b_full(s), par, kWaitLimit)) *abort_flag = 1;
      if (tid < 64) {
        const bool ok = tid < L;
        gam[tid] = ok ? g[(trow0 + tid) * HV + hv] : 0.f;
        bet[tid] = ok ? beta[(trow0 + tid) * HV + hv] : 0.f;
      }
      if (tid == 0) misc[2] = *abort_flag;  // one snapshot, read by every warp after the barrier
      named_bar_sync(1, NCW * 32);
      if (misc[2]) break;

      // 2. row norms of k (threads 0-63) and q (64-127); chunk-local cumsum of g (warp 4).
      if (tid < 128) {
        const int r = tid;  // row of the stacked [K; Q] tile
        float ss = 0.f;
#pragma unroll
        for (int kc = 0; kc < K / 8; ++kc) {
          const uint4 v4 = *reinterpret_cast<const uint4 *>(stp + (kc >> 3) * 16384 + sw128(r, kc & 7));
          const uint32_t w4[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
          for (int q2 = 0; q2 < 4; ++q2) {
            const float lo = bf16lo_f(w4[q2]), hi = bf16hi_f(w4[q2]);
            ss = fmaf(lo, lo, fmaf(hi, hi, ss));
          }
        }
        const float rn = l2 ? rsqrtf(ss + GDN_L2_EPS) : 1.f;
        if (r < 64) rk[r] = rn; else rq[r - 64] = rn;
      } else if (warp == 4) {
        const float x0 = gam[2 * lane], x1 = gam[2 * lane + 1];
        float sum = x0 + x1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, sum, off);
          if (lane >= off) sum += y;
        }
        const float excl = sum - (x0 + x1);
        gam[2 * lane] = excl + x0;
        gam[2 * lane + 1] = sum;
      }
      named_bar_sync(1, NCW * 32);
      if (tid < 64) {
        og[tid] = expf(gam[tid]) * rq[tid];
        sv[tid] = expf(gam[63] - gam[tid]) * rk[tid];
      }

      // 3. K K^T and Q K^T from TMEM -> A (fp32) and P hi/lo (bf16).
      if (!mbar_wait_bounded(b_kqf(s), par, kWaitLimit)) *abort_flag = 1;
      tc_fence_after();
      {
        const int quad = warp & 3, half = warp >> 2;
        float vals[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(32 * quad) << 16) + s * 64 + half * 32, vals);
        const int row = 32 * quad + lane;
        if (row < 64) {
          const int i = row;
          const float gi = gam[i], ci = bet[i] * rk[i];
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int j = half * 32 + jj;
            Am[i * FROW + j] = (j < i && i < L) ? ci * expf(gi - gam[j]) * rk[j] * vals[jj] : 0.f;
          }
        } else {
          const int i = row - 64;
          const float gi = gam[i], ci = rq[i];
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            uint32_t ph[4], pl[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float pv[2];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int jj = q8 * 8 + 2 * e + u;
                const int j = half * 32 + jj;
                pv[u] = (j <= i && i < L) ? ci * expf(gi - gam[j]) * rk[j] * vals[jj] : 0.f;
              }
              ph[e] = pack_bf16(pv[0], pv[1]);
              pl[e] = pack_bf16(pv[0] - bf16lo_f(ph[e]), pv[1] - bf16hi_f(ph[e]));
            }
            const int chunk = half * 4 + q8;
            *reinterpret_cast<uint4 *>(sm + Ly::OFF_PH + sw128(i, chunk)) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
            *reinterpret_cast<uint4 *>(sm + Ly::OFF_PL + sw128(i, chunk)) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_kqe(s));
      if (tid == 0) misc[2] = *abort_flag;
      named_bar_sync(1, NCW * 32);
      if (misc[2]) break;

      // 4a. diagonal 16x16 blocks of T (warps 0-3, lanes 0-15: one column each);
      //     warps 4-7 zero the rows >= L of this stage's tiles.
      if (warp < 4) {
        if (lane < 16) {
          const int b0 = 16 * warp, col = lane;
          float x[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float acc = (i == col) ? 1.f : 0.f;
#pragma unroll
            for (int j = 0; j < i; ++j) acc = fmaf(-Am[(b0 + i) * FROW + b0 + j], x[j], acc);
            x[i] = (i < col) ? 0.f : acc;
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) Tm[(b0 + i) * FROW + b0 + col] = x[i];
        }
      } else if (L < C) {
        const int t2 = tid - 128;
        for (int e = t2; e < (C - L) * 8 * Ly::KA * 2; e += 128) {
          const int rr = e / (8 * Ly::KA * 2), rem = e % (8 * Ly::KA * 2);
          const int which = rem / (8 * Ly::KA), kc = rem % (8 * Ly::KA);
          const int row = L + rr + 64 * which;
          *reinterpret_cast<uint4 *>(stp + (kc >> 3) * 16384 + sw128(row, kc & 7)) = make_uint4(0, 0, 0, 0);
        }
        for (int e = t2; e < (C - L) * 4; e += 128) {
          const int row = L + e / 4, q = e % 4;
          *reinterpret_cast<uint4 *>(stp + Ly::KQ_BYTES + row * 64 + q * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      named_bar_sync(1, NCW * 32);
      // 4b. off-diagonal blocks: T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj, by block distance.
#pragma unroll
      for (int d = 1; d <= 3; ++d) {
        const int nb = 4 - d;  // blocks at this distance: i = d .. 3, j = i - d
        for (int e = tid; e < nb * 256; e += NCW * 32) {
          const int bi = e >> 8, r = (e >> 4) & 15, cc = e & 15;
          const int i = bi + d, j = i - d;
          float acc = 0.f;
          for (int kb = j; kb < i; ++kb) {
#pragma unroll
            for (int k2 = 0; k2 < 16; ++k2)
              acc = fmaf(Am[(16 * i + r) * FROW + 16 * kb + k2], Tm[(16 * kb + k2) * FROW + 16 * j + cc], acc);
          }
          Xs[bi * 272 + r * 17 + cc] = acc;
        }
        named_bar_sync(1, NCW * 32);
        for (int e = tid; e < nb * 256; e += NCW * 32) {
          const int bi = e >> 8, r = (e >> 4) & 15, cc = e & 15;
          const int i = bi + d, j = i - d;
          float acc = 0.f;
#pragma unroll
          for (int k2 = 0; k2 < 16; ++k2) acc = fmaf(Tm[(16 * i + r) * FROW + 16 * i + k2], Xs[bi * 272 + k2 * 17 + cc], acc);
          Tm[(16 * i + r) * FROW + 16 * j + cc] = -acc;
        }
        named_bar_sync(1, NCW * 32);
      }

      // 5. Tp = T diag(beta e^gamma rk) (j <= i), Ts = (T - I) diag(beta) (j < i), bf16.
      for (int e = tid; e < 64 * 8; e += NCW * 32) {
        const int i = e >> 3, ch = e & 7;
        uint32_t tp[4], ts[4];
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2) {
          float a2[2], b2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int j = ch * 8 + 2 * q2 + u;
            const float tv = Tm[i * FROW + j];
            a2[u] = (j <= i) ? tv * bet[j] * expf(gam[j]) * rk[j] : 0.f;
            b2[u] = (j < i) ? tv * bet[j] : 0.f;
          }
          tp[q2] = pack_bf16(a2[0], a2[1]);
          ts[q2] = pack_bf16(b2[0], b2[1]);
        }
        *reinterpret_cast<uint4 *>(sm + Ly::OFF_TP + sw128(i, ch)) = make_uint4(tp[0], tp[1], tp[2], tp[3]);
        *reinterpret_cast<uint4 *>(sm + Ly::OFF_TS + sw128(i, ch)) = make_uint4(ts[0], ts[1], ts[2], ts[3]);
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
        const float dL = expf(gam[63]);
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
      __syncwarp();
      if (lane == 0) mbar_arrive(b_empty(s));
      named_bar_sync(1, NCW * 32);
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
  if (warp == NCW) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
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
