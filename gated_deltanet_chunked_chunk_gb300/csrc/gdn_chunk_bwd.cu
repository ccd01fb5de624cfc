// gdn_chunk_bwd.cu -- backward of the chunked Gated DeltaNet forward.
//
// "NPU Training Operators - GDN" pairs the chunked forward with its backward
// (gradients of q, k, v, beta, g and the initial state) for training; the
// pages give no backward formulas, so this is reverse-mode differentiation of
// the chunked form the forward computes.  For one chunk of one value head
// (rows i, j < 64; gamma = chunk-local cumsum of g; q^, k^ the normalised
// q, k; og_i = e^{gamma_i}; s_j = e^{gamma_L - gamma_j}; h the state entering
// the chunk, h' the state leaving it):
//   A = strictly-lower beta_i e^{gamma_i-gamma_j} k^_i.k^_j,  T = (I + A)^-1
//   U = T diag(beta) V,  v_new = U - T diag(beta og) K^ h
//   o_i = scale (og_i q^_i^T h + sum_{j<=i} e^{gamma_i-gamma_j} (q^_i.k^_j) v_new_j)
//   h' = e^{gamma_L} h + sum_j s_j k^_j v_new_j^T
// Given do and dh' (the gradient of the state leaving the chunk):
//   dv_new_j = s_j dh'^T k^_j + scale sum_{i>=j} P_ij do_i            (P as above)
//   dh       = e^{gamma_L} dh' + scale sum_i og_i q^_i do_i^T - W^T dv_new
// which is serial over chunks (chunk_dh_kernel, last chunk first, the
// gradient of the final state seeding it), and then, per chunk in parallel
// (chunk_grad_kernel), the gradients through U, W, T (dA = -T^T dT T^T), A, P,
// the decays (reverse cumsum into dg) and the L2 norms.
//
// The forward is re-run first (prep + walk kernels of gdn_chunk.cu) with the
// walk saving the state entering every chunk; the dh walk saves dh' of every
// chunk.  The dh walk runs on tcgen05 at K = 128 (chunk_dh_tc_kernel, TMEM
// accumulators) and on warp-level mma.sync otherwise; the per-chunk gradients
// run on mma.sync (computed operands split hi + lo; see the helpers).
#include <math.h>
#include <string.h>

#include "gdn_chunk_shared.cuh"
#include "gdn_common.cuh"
#include "gdn_sm103.cuh"

namespace {

using namespace gdn;
using namespace gdnc;

constexpr int BT = 256;  // threads per CTA for both kernels

__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool valid) {
  const uint32_t d = smem_u32(dst);
  const int n = valid ? 16 : 0;  // 0: zero-fill
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Element (row, key) of the record's W: 64-key SW128 atom columns of 64 rows.
__device__ __forceinline__ float rec_w(const unsigned char *w, int row, int key) {
  const uint16_t x =
      *reinterpret_cast<const uint16_t *>(w + (key >> 6) * 8192 + sw128(row, (key & 63) >> 3) + (key & 7) * 2);
  return bf2f(x);
}
// Element (i, j) of a [64][64] SW128 bf16 tile.
__device__ __forceinline__ float tile64(const unsigned char *t, int i, int j) {
  return bf2f(*reinterpret_cast<const uint16_t *>(t + sw128(i, j >> 3) + (j & 7) * 2));
}

// ------------------------------------------------------------- mma helpers
// Warp-level mma.sync m16n8k16 in bf16 with fp32 accumulation (wgemm_bf,
// wgemm_bf_pb below).  A computed fp32 operand is split into bf16 hi + lo parts
// and a product takes hi*hi + hi*lo + lo*hi (relative error near 2^-17); an
// operand holding raw bf16 values is exact and has no low part.
// f(rh, r, n, x) for every accumulator element: row r = g + 8 rh, column n.
template <int NT, class F>
__device__ __forceinline__ void cvisit(float (&c)[NT][4], F f) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) f(e >> 1, g + 8 * (e >> 1), 8 * n + 2 * t + (e & 1), c[n][e]);
}
__device__ __forceinline__ void prefetch_l2(const void *p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  return x + __shfl_xor_sync(0xffffffffu, x, 2);
}

constexpr int VS = 32;  // V columns per slice
constexpr int MS = 68;  // fp32 row stride of a 64 x 64 tile
constexpr int SS = 36;  // fp32 row stride of a 32-column slice

// c (16 x 8 NT) += A (16 x [k0, k1)) B ([k0, k1) x 8 NT) for one warp on
// mma.sync m16n8k16 in bf16: a computed operand is split into bf16 hi + lo
// (about 16 bits kept; hi*hi + hi*lo + lo*hi leaves a relative error near
// 2^-17), an operand of raw bf16 values has no low part (AX / BX).  fa2(r, k)
// and fb2(k, n) return the pairs (A[r][k], A[r][k + 1]) and (B[k][n],
// B[k + 1][n]); k0, k1 are multiples of 16.
__device__ __forceinline__ void split_bf16(float2 v, uint32_t &hi, uint32_t &lo) {
  hi = pack_bf16(v.x, v.y);
  lo = pack_bf16(v.x - bf16lo_f(hi), v.y - bf16hi_f(hi));
}
template <int NT, bool AX, bool BX, class FA2, class FB2>
__device__ __forceinline__ void wgemm_bf(float (&c)[NT][4], int k0, int k1, FA2 fa2, FB2 fb2) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll 2
  for (int k = k0; k < k1; k += 16) {
    const float2 av[4] = {fa2(g, k + 2 * t), fa2(g + 8, k + 2 * t), fa2(g, k + 2 * t + 8), fa2(g + 8, k + 2 * t + 8)};
    uint32_t ah[4], al[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (AX) {
        ah[e] = pack_bf16(av[e].x, av[e].y);
        al[e] = 0u;
      } else {
        split_bf16(av[e], ah[e], al[e]);
      }
    }
    uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const float2 b0 = fb2(k + 2 * t, 8 * n + g), b1 = fb2(k + 2 * t + 8, 8 * n + g);
      if (BX) {
        bh[n][0] = pack_bf16(b0.x, b0.y);
        bh[n][1] = pack_bf16(b1.x, b1.y);
        bl[n][0] = bl[n][1] = 0u;
      } else {
        split_bf16(b0, bh[n][0], bl[n][0]);
        split_bf16(b1, bh[n][1], bl[n][1]);
      }
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) mma_bf16(c[n], ah, bh[n][0], bh[n][1]);
    if (!BX) {
#pragma unroll
      for (int n = 0; n < NT; ++n) mma_bf16(c[n], ah, bl[n][0], bl[n][1]);
    }
    if (!AX) {
#pragma unroll
      for (int n = 0; n < NT; ++n) mma_bf16(c[n], al, bh[n][0], bh[n][1]);
    }
  }
}
// wgemm_bf with a B operand stored already split: fbp(k, n) returns the bf16
// pairs {hi (B[k][n], B[k + 1][n]), lo (B[k][n], B[k + 1][n])}.
template <int NT, bool AX, class FA2, class FBP>
__device__ __forceinline__ void wgemm_bf_pb(float (&c)[NT][4], int k0, int k1, FA2 fa2, FBP fbp) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll 2
  for (int k = k0; k < k1; k += 16) {
    const float2 av[4] = {fa2(g, k + 2 * t), fa2(g + 8, k + 2 * t), fa2(g, k + 2 * t + 8), fa2(g + 8, k + 2 * t + 8)};
    uint32_t ah[4], al[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (AX) {
        ah[e] = pack_bf16(av[e].x, av[e].y);
        al[e] = 0u;
      } else {
        split_bf16(av[e], ah[e], al[e]);
      }
    }
    uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const uint2 b0 = fbp(k + 2 * t, 8 * n + g), b1 = fbp(k + 2 * t + 8, 8 * n + g);
      bh[n][0] = b0.x;
      bl[n][0] = b0.y;
      bh[n][1] = b1.x;
      bl[n][1] = b1.y;
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) mma_bf16(c[n], ah, bh[n][0], bh[n][1]);
#pragma unroll
    for (int n = 0; n < NT; ++n) mma_bf16(c[n], ah, bl[n][0], bl[n][1]);
    if (!AX) {
#pragma unroll
      for (int n = 0; n < NT; ++n) mma_bf16(c[n], al, bh[n][0], bh[n][1]);
    }
  }
}
// ------------------------------------------------------------------ dh walk
// One CTA per (64-column slice of V, value head, sequence), last chunk first
// (64 columns: at V = 128 the grid of HV x N x 2 CTAs fits one wave of SMs for
// the usual head counts, where 32-column slices needed two).
// dh (K x 64 fp32) lives in the mma accumulators of the eight warps (warp w:
// rows of tile w % (K / 16), a share of the columns); per chunk K, Q, W, P,
// the scalars and the do slice are staged in shared memory (cp.async, double
// buffered).  Both products of a chunk run on mma.sync m16n8k16 in bf16: the
// raw k, q, W, P hi / lo and do are exact, the computed dh' and dv_new are
// split hi + lo.
constexpr int DVC = 64;  // V columns per dh-walk CTA

template <int K>
struct DhLay {
  static constexpr int KROW = K * 2 + 16;             // padded bf16 row of K keys
  static constexpr int OFF_K = 0;                     // raw K [64][KROW]
  static constexpr int OFF_Q = OFF_K + 64 * KROW;     // raw Q [64][KROW]
  static constexpr int OFF_REC = OFF_Q + 64 * KROW;   // record bytes W | PH | PL (contiguous in the record)
  static constexpr int REC_BYTES = Rec<K>::TS;        // W + PH + PL
  static constexpr int OFF_SC = OFF_REC + REC_BYTES;  // record scalars (1 KB)
  static constexpr int DOROW = DVC * 2 + 16;          // padded bf16 row of the do slice (bytes)
  static constexpr int OFF_DO = OFF_SC + 1024;        // do slice [64][DOROW bytes]
  static constexpr int STAGE = OFF_DO + 64 * DOROW;
  // dh', dv_new and do are read as bf16 B operands (rows k + 2t and k + 2t + 1,
  // column g of a fragment): a row stride of 4 (mod 16) words keeps those reads
  // free of bank conflicts (DOROW = 144 bytes = 36 words as well).
  static constexpr int BS = DVC + 4;
  static constexpr int OFF_DHS = 2 * STAGE;           // dh' [K][BS] fp32
  static constexpr int OFF_DVN = OFF_DHS + K * BS * 4;  // dv_new [64][BS] fp32
  static constexpr int BYTES = OFF_DVN + 64 * BS * 4;
  static_assert(STAGE % 16 == 0, "16-byte copies");
};

template <int K>
__global__ void __launch_bounds__(BT, 1) chunk_dh_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ k, const uint16_t *__restrict__ dout,
    const unsigned char *__restrict__ ws, float *__restrict__ DH, const float *__restrict__ dht,
    float *__restrict__ dh0, float scale, const int32_t *__restrict__ cu, const int32_t *__restrict__ cs, int T,
    int H, int HV, int V, int32_t *dev_status) {
  using Ly = DhLay<K>;
  using R = Rec<K>;
  constexpr int KE = Ly::KROW / 2;  // bf16 elements per staged K / Q row
  constexpr int MTK = K / 16;       // row tiles of dh
  constexpr int WPM = 8 / MTK;      // warps per row tile
  constexpr int NTD = DVC / 8 / WPM;  // n-tiles (8 columns) per warp
  extern __shared__ __align__(16) unsigned char smem[];
  const int vt0 = blockIdx.x * DVC, hv = blockIdx.y, n = blockIdx.z;
  const int h = hv / (HV / H);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int dm0 = 16 * (warp % MTK), dc0 = 8 * NTD * (warp / MTK);  // this warp's block of dh
  const int mt = warp & 3, r0 = 16 * mt, hf = warp >> 2;              // its block of dv_new

  int64_t tok0, len;
  if (!seq_bounds(cu, n, T, tok0, len)) {
    if (tid == 0) set_status(dev_status, GDN_DEV_BAD_CU_SEQLENS);
    return;
  }
  const int NC = chunks_of(len);
  const int64_t cb = chunk_base(cs, n, T);
  const int64_t sbase = ((int64_t)n * HV + hv) * K;
  float dh[NTD][4];
  cvisit(dh, [&](int, int r, int c, float &x) {
    x = dht ? dht[(sbase + dm0 + r) * V + vt0 + dc0 + c] : 0.f;
  });

  auto issue = [&](int c, int st) {
    unsigned char *S = smem + st * Ly::STAGE;
    const int64_t trow = tok0 + (int64_t)c * C;
    const int64_t rem = len - (int64_t)c * C;
    const int L = rem < C ? (int)rem : C;
    for (int e = tid; e < 64 * (K / 8); e += BT) {
      const int row = e / (K / 8), ch = e % (K / 8);
      const bool ok = row < L;
      const int64_t g = ok ? ((trow + row) * H + h) * K + ch * 8 : 0;
      cp_async16(S + Ly::OFF_K + row * Ly::KROW + ch * 16, k + g, ok);
      cp_async16(S + Ly::OFF_Q + row * Ly::KROW + ch * 16, q + g, ok);
    }
    const unsigned char *rec = ws + ((size_t)(cb + c) * HV + hv) * R::BYTES;
    for (int e = tid; e < Ly::REC_BYTES / 16; e += BT) cp_async16(S + Ly::OFF_REC + e * 16, rec + e * 16, true);
    for (int e = tid; e < 1024 / 16; e += BT) cp_async16(S + Ly::OFF_SC + e * 16, rec + R::SC + e * 16, true);
    for (int e = tid; e < 64 * (DVC / 8); e += BT) {
      const int row = e / (DVC / 8), ch = e % (DVC / 8);
      const bool ok = row < L;
      const int64_t g = ok ? ((trow + row) * HV + hv) * V + vt0 + ch * 8 : 0;
      cp_async16(S + Ly::OFF_DO + row * Ly::DOROW + ch * 16, dout + g, ok);
    }
    cp_async_commit();
  };

  float *dhs = reinterpret_cast<float *>(smem + Ly::OFF_DHS);
  float *dvn = reinterpret_cast<float *>(smem + Ly::OFF_DVN);
  if (NC > 0) issue(NC - 1, 0);
  for (int c = NC - 1; c >= 0; --c) {
    const int st = (NC - 1 - c) & 1;
    if (c > 0) {
      issue(c - 1, st ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    // dh' of this chunk: to shared memory, then from there to the workspace
    // with coalesced 16-byte stores (rows of DVC consecutive floats).
    cvisit(dh, [&](int, int r, int cc, float x) { dhs[(dm0 + r) * Ly::BS + dc0 + cc] = x; });
    __syncthreads();
    {
      float *dst = DH + (((cb + c) * HV + hv) * K) * (int64_t)V + vt0;
      for (int e = tid; e < K * (DVC / 4); e += BT) {
        const int row = e / (DVC / 4), c4 = e % (DVC / 4);
        *reinterpret_cast<float4 *>(dst + (int64_t)row * V + 4 * c4) =
            *reinterpret_cast<const float4 *>(dhs + row * Ly::BS + 4 * c4);
      }
    }
    const unsigned char *S = smem + st * Ly::STAGE;
    const float *sc = reinterpret_cast<const float *>(S + Ly::OFF_SC);
    const uint16_t *Ks = reinterpret_cast<const uint16_t *>(S + Ly::OFF_K);
    const uint16_t *Qs = reinterpret_cast<const uint16_t *>(S + Ly::OFF_Q);
    const uint16_t *Ds = reinterpret_cast<const uint16_t *>(S + Ly::OFF_DO);
    const unsigned char *Wt = S + Ly::OFF_REC;
    const unsigned char *PH = S + Ly::OFF_REC + (R::PH - R::W);
    const unsigned char *PL = S + Ly::OFF_REC + (R::PL - R::W);
    // dv_new = diag(sv) K dh' + scale (P_hi + P_lo)^T do   (sv carries 1/||k||)
    {
      constexpr int NTV = DVC / 16;  // n-tiles of a warp's half of the columns
      float ca[NTV][4] = {}, cp[NTV][4] = {};
      const int n0 = (DVC / 2) * hf;
      // bf16 m16n8k16: raw k, P halves and do exact, dh' split hi + lo
      auto fk = [&](int r, int x) {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(Ks + (r0 + r) * KE + x);
        return make_float2(bf16lo_f(w), bf16hi_f(w));
      };
      auto fd = [&](int x, int nn) { return make_float2(dhs[x * Ly::BS + n0 + nn], dhs[(x + 1) * Ly::BS + n0 + nn]); };
      wgemm_bf<NTV, true, false>(ca, 0, K, fk, fd);
      auto fph = [&](int r, int i) { return make_float2(tile64(PH, i, r0 + r), tile64(PH, i + 1, r0 + r)); };
      auto fpl = [&](int r, int i) { return make_float2(tile64(PL, i, r0 + r), tile64(PL, i + 1, r0 + r)); };
      auto fo = [&](int i, int nn) {
        return make_float2(bf2f(Ds[i * (Ly::DOROW / 2) + n0 + nn]), bf2f(Ds[(i + 1) * (Ly::DOROW / 2) + n0 + nn]));
      };
      wgemm_bf<NTV, true, true>(cp, r0, 64, fph, fo);
      wgemm_bf<NTV, true, true>(cp, r0, 64, fpl, fo);
      const int g = (tid & 31) >> 2, t = tid & 3;
#pragma unroll
      for (int nt = 0; nt < NTV; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = r0 + g + 8 * (e >> 1);
          dvn[j * Ly::BS + n0 + 8 * nt + 2 * t + (e & 1)] = fmaf(sc[RS_SV + j], ca[nt][e], scale * cp[nt][e]);
        }
    }
    __syncthreads();
    // dh = e^{gamma_L} dh' + Q^T diag(scale og) do - W^T dv_new   (og carries 1/||q||)
    {
      const float dL = sc[RS_DL];
      float t1[NTD][4] = {}, t2[NTD][4] = {};  // separate accumulators: independent mma chains
      auto fq = [&](int r, int i) { return make_float2(bf2f(Qs[i * KE + dm0 + r]), bf2f(Qs[(i + 1) * KE + dm0 + r])); };
      auto fo = [&](int i, int cc) {
        return make_float2(scale * sc[RS_OG + i] * bf2f(Ds[i * (Ly::DOROW / 2) + dc0 + cc]),
                           scale * sc[RS_OG + i + 1] * bf2f(Ds[(i + 1) * (Ly::DOROW / 2) + dc0 + cc]));
      };
      wgemm_bf<NTD, true, false>(t1, 0, 64, fq, fo);
      auto fw = [&](int r, int j) { return make_float2(rec_w(Wt, j, dm0 + r), rec_w(Wt, j + 1, dm0 + r)); };
      auto fv = [&](int j, int cc) { return make_float2(dvn[j * Ly::BS + dc0 + cc], dvn[(j + 1) * Ly::BS + dc0 + cc]); };
      wgemm_bf<NTD, true, false>(t2, 0, 64, fw, fv);
#pragma unroll
      for (int nt = 0; nt < NTD; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) dh[nt][e] = fmaf(dL, dh[nt][e], t1[nt][e] - t2[nt][e]);
    }
    __syncthreads();  // this stage is refilled by the next issue
  }
  if (dh0) {
    cvisit(dh, [&](int, int r, int cc, float x) { dh0[(sbase + dm0 + r) * V + vt0 + dc0 + cc] = x; });
  }
}

// ---------------------------------------------------------- chunk gradients
// One CTA per (chunk, value head); every product on the tensor cores with the
// helpers above (raw q, k, v, do exact, computed operands split).  Warp w owns
// the 16-row tile mt = w & 3 of a 64-row result and, where the result is wider
// than one warp's share, the column half hf = w >> 2.

template <int K>
struct GradLay {
  static constexpr int BROW = K + 8;                     // bf16 row stride of raw q, k
  static constexpr int M64 = 64 * MS * 4;
  static constexpr int HSB = VS + 8;                     // bf16 row stride of a split h / dh' slice
  static constexpr int HS = K * HSB * 2, RS = 64 * SS * 4;
  static constexpr int OFF_QB = 0;                       // raw q [64][BROW] bf16
  static constexpr int OFF_KB = OFF_QB + 64 * BROW * 2;  // raw k
  static constexpr int OFF_T = OFF_KB + 64 * BROW * 2;   // A, then T = (I + A)^-1
  static constexpr int OFF_P = OFF_T + M64;              // P_ij = e^{gamma_i-gamma_j} q^_i.k^_j (j <= i)
  static constexpr int OFF_EK = OFF_P + M64;             // e^{gamma_i-gamma_j} k^_i.k^_j (j < i)
  static constexpr int OFF_SL = OFF_EK + M64;            // V-slice buffers, reused afterwards
  static constexpr int OFF_H = OFF_SL;                   // h slice [K][HSB] as bf16 hi, then lo
  static constexpr int OFF_DH = OFF_H + 2 * HS;          // dh' slice, hi then lo
  static constexpr int OFF_V = OFF_DH + 2 * HS;          // v slice [64][SS]
  static constexpr int OFF_DO = OFF_V + RS;              // do slice
  static constexpr int OFF_KH = OFF_DO + RS;             // k^ h
  static constexpr int OFF_KDH = OFF_KH + RS;            // k^ dh'
  static constexpr int OFF_MV = OFF_KDH + RS;            // diag(beta) (v - diag(og) k^ h)
  static constexpr int OFF_VN = OFF_MV + RS;             // v_new
  static constexpr int OFF_DVN = OFF_VN + RS;            // dv_new
  static constexpr int OFF_TU = OFF_DVN + RS;            // T^T dv_new
  static constexpr int SL_END = OFF_TU + RS;
  static constexpr int OFF_DT = OFF_SL;                  // after the slices: dT, then dA
  static constexpr int OFF_DP = OFF_DT + M64;            // scale dP
  static constexpr int OFF_X = OFF_DP + M64;             // dT T^T
  static constexpr int OFF_S1 = OFF_X + M64;             // (A-bar + A-bar^T) diag(rk)
  static constexpr int OFF_S2 = OFF_S1 + M64;            // P-bar^T diag(rq)
  static constexpr int OFF_S3 = OFF_S2 + M64;            // P-bar diag(rk)
  static constexpr int END_END = OFF_S3 + M64;
  static constexpr int OFF_VEC = SL_END > END_END ? SL_END : END_END;
  static constexpr int NVEC = 14;
  static constexpr int BYTES = OFF_VEC + NVEC * 64 * 4;
  static_assert(BYTES <= 227 * 1024, "one CTA per SM");
};
enum { GV_GAM = 0, GV_OG, GV_SV, GV_BET, GV_RQ, GV_RK, GV_DB, GV_DG, GV_SQ, GV_SG, GV_SL, GV_PQ, GV_PK, GV_MISC };

template <int K>
__global__ void __launch_bounds__(BT, 1) chunk_grad_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
    const float *__restrict__ g, const float *__restrict__ beta, const uint16_t *__restrict__ dout,
    const float *__restrict__ Hs, const float *__restrict__ DH, float scale, const int32_t *__restrict__ cu,
    const int32_t *__restrict__ cs, int N, int T, int H, int HV, int V, int l2, float *__restrict__ dq,
    float *__restrict__ dk, float *__restrict__ dqk_part, int64_t part_stride,
    float *__restrict__ dv, float *__restrict__ dg, float *__restrict__ dbeta, int32_t *dev_status) {
  using Ly = GradLay<K>;
  constexpr int BR = Ly::BROW;
  constexpr int NH = K / 16;  // n-tiles of a warp's half of K columns
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t *Qb = reinterpret_cast<uint16_t *>(smem + Ly::OFF_QB);
  uint16_t *Kb = reinterpret_cast<uint16_t *>(smem + Ly::OFF_KB);
  float *Tm = reinterpret_cast<float *>(smem + Ly::OFF_T);
  float *Pm = reinterpret_cast<float *>(smem + Ly::OFF_P);
  float *EK = reinterpret_cast<float *>(smem + Ly::OFF_EK);
  // h, dh' of the current slice, split once into bf16 hi + lo when loaded
  uint16_t *Hhi = reinterpret_cast<uint16_t *>(smem + Ly::OFF_H);
  uint16_t *Hlo = reinterpret_cast<uint16_t *>(smem + Ly::OFF_H + Ly::HS);
  uint16_t *DHhi = reinterpret_cast<uint16_t *>(smem + Ly::OFF_DH);
  uint16_t *DHlo = reinterpret_cast<uint16_t *>(smem + Ly::OFF_DH + Ly::HS);
  constexpr int HSB = Ly::HSB;
  auto pair16 = [](const uint16_t *p, int stride) {  // (p[0], p[stride]) as a bf16 pair
    return static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[stride]) << 16);
  };
  auto word16 = [](const uint16_t *p) { return *reinterpret_cast<const uint32_t *>(p); };
  float *vS = reinterpret_cast<float *>(smem + Ly::OFF_V);
  float *doS = reinterpret_cast<float *>(smem + Ly::OFF_DO);
  float *KhS = reinterpret_cast<float *>(smem + Ly::OFF_KH);
  float *KdhS = reinterpret_cast<float *>(smem + Ly::OFF_KDH);
  float *MvS = reinterpret_cast<float *>(smem + Ly::OFF_MV);
  float *vnS = reinterpret_cast<float *>(smem + Ly::OFF_VN);
  float *dvnS = reinterpret_cast<float *>(smem + Ly::OFF_DVN);
  float *TuS = reinterpret_cast<float *>(smem + Ly::OFF_TU);
  float *DT = reinterpret_cast<float *>(smem + Ly::OFF_DT);
  float *DP = reinterpret_cast<float *>(smem + Ly::OFF_DP);
  float *Xm = reinterpret_cast<float *>(smem + Ly::OFF_X);
  float *S1 = reinterpret_cast<float *>(smem + Ly::OFF_S1);
  float *S2 = reinterpret_cast<float *>(smem + Ly::OFF_S2);
  float *S3 = reinterpret_cast<float *>(smem + Ly::OFF_S3);
  float *vec = reinterpret_cast<float *>(smem + Ly::OFF_VEC);
  float *gam = vec + GV_GAM * 64, *og = vec + GV_OG * 64, *sv = vec + GV_SV * 64, *bet = vec + GV_BET * 64;
  float *rq = vec + GV_RQ * 64, *rk = vec + GV_RK * 64, *DB = vec + GV_DB * 64, *DG = vec + GV_DG * 64;
  float *SQ = vec + GV_SQ * 64, *SG = vec + GV_SG * 64, *SLv = vec + GV_SL * 64;
  float *PQ = vec + GV_PQ * 64, *PK = vec + GV_PK * 64, *misc = vec + GV_MISC * 64;

  // Value head fastest, so that the value heads of a key head share q, k through L2.
  const int gc = static_cast<int>(blockIdx.x / HV), hv = static_cast<int>(blockIdx.x % HV);
  const int h = hv / (HV / H);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int mt = warp & 3, hf = warp >> 2, r0 = 16 * mt;

  // Which sequence / chunk?
  int n = 0, c = 0;
  int64_t tok0 = 0, len = 0;
  const int64_t slot = gc;
  if (!slot_chunk(cs, N, T, gc, n, c) || !seq_bounds(cu, n, T, tok0, len)) return;
  const int64_t rem = len - (int64_t)c * C;
  const int L = rem < C ? (int)rem : C;
  const int64_t trow0 = tok0 + (int64_t)c * C;
  auto qv = [&](int i, int x) { return bf2f(Qb[i * BR + x]); };
  auto kv = [&](int i, int x) { return bf2f(Kb[i * BR + x]); };
  // (x, x + 1) of a raw row, x even: one 32-bit load
  auto pair_of = [](const uint16_t *p) {
    const uint32_t w = *reinterpret_cast<const uint32_t *>(p);
    return make_float2(bf16lo_f(w), bf16hi_f(w));
  };
  auto ld2 = [](const float *p) { return *reinterpret_cast<const float2 *>(p); };

  // The rows of a V slice (h, dh': K rows of 128 bytes; v, do: L rows of 64)
  // into L2, one line per thread; slice 0 lands while the chunk's own
  // products run, slice s + 1 during slice s.
  auto prefetch_slice = [&](int v0) {
    const int64_t hb = ((slot * HV + hv) * K) * (int64_t)V + v0;
    if (tid < 2 * K) prefetch_l2((tid < K ? Hs : DH) + hb + (int64_t)(tid % K) * V);
    const int i = tid & 63;
    if (tid < 128 && i < L) prefetch_l2((tid < 64 ? v : dout) + ((trow0 + i) * HV + hv) * V + v0);
  };
  prefetch_slice(0);
  // ---- raw q, k rows (zero past L), gates and their cumsum
  // (asynchronous 16-byte copies, zero-filled past L: every copy in flight at once)
  for (int e = tid; e < 64 * (K / 8); e += BT) {
    const int i = e / (K / 8), ch = e % (K / 8);
    const bool ok = i < L;
    const int64_t off = ok ? ((trow0 + i) * H + h) * K + ch * 8 : 0;
    cp_async16(Qb + i * BR + ch * 8, q + off, ok);
    cp_async16(Kb + i * BR + ch * 8, k + off, ok);
  }
  cp_async_commit();
  if (warp == 0) {
    float x[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int i = 2 * lane + u;
      x[u] = i < L ? g[(trow0 + i) * HV + hv] : 0.f;
      bet[i] = i < L ? beta[(trow0 + i) * HV + hv] : 0.f;
    }
    float sum = x[0] + x[1];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, sum, off);
      if (lane >= off) sum += y;
    }
    gam[2 * lane] = sum - x[1];
    gam[2 * lane + 1] = sum;
  }
  for (int e = tid; e < 64 * (GV_MISC - GV_DB + 1); e += BT) vec[GV_DB * 64 + e] = 0.f;
  cp_async_wait<0>();
  __syncthreads();
  {  // norms: four threads per row
    const int i = tid >> 2, p = tid & 3;
    float sq = 0.f, sk = 0.f;
    for (int x = p * (K / 4); x < (p + 1) * (K / 4); ++x) {
      const float a = qv(i, x), b = kv(i, x);
      sq = fmaf(a, a, sq);
      sk = fmaf(b, b, sk);
    }
    sq = quad_sum(sq);
    sk = quad_sum(sk);
    if (p == 0) {
      rq[i] = l2 ? rsqrtf(sq + GDN_L2_EPS) : 1.f;
      rk[i] = l2 ? rsqrtf(sk + GDN_L2_EPS) : 1.f;
    }
    if (tid < 64) {
      og[tid] = expf(gam[tid]);
      sv[tid] = expf(gam[63] - gam[tid]);
    }
  }
  __syncthreads();

  // ---- k k^T and q k^T (exact bf16 operands): EK, A (into Tm), P
  {
    float ck[4][4] = {}, cq[4][4] = {};
    auto fk = [&](int r, int x) { return pair_of(Kb + (r0 + r) * BR + x); };
    auto fq = [&](int r, int x) { return pair_of(Qb + (r0 + r) * BR + x); };
    auto fkt = [&](int x, int n) { return pair_of(Kb + (32 * hf + n) * BR + x); };
    wgemm_bf<4, true, true>(ck, 0, K, fk, fkt);
    wgemm_bf<4, true, true>(cq, 0, K, fq, fkt);
    cvisit(ck, [&](int, int r, int n, float x) {
      const int i = r0 + r, j = 32 * hf + n;
      const float ek = (j < i) ? expf(gam[i] - gam[j]) * x * rk[i] * rk[j] : 0.f;
      EK[i * MS + j] = ek;
      Tm[i * MS + j] = bet[i] * ek;
    });
    cvisit(cq, [&](int, int r, int n, float x) {
      const int i = r0 + r, j = 32 * hf + n;
      Pm[i * MS + j] = (j <= i) ? expf(gam[i] - gam[j]) * x * rq[i] * rk[j] : 0.f;
    });
  }
  __syncthreads();

  // ---- T = (I + A)^-1 in place: 16 x 16 diagonal blocks by substitution
  // (thread = one column of one block), then block rows 1..3:
  // T_ij = -D_i sum_{m=j}^{i-1} A_im T_mj.
  if (tid < 64) {
    const int b0 = 16 * (tid >> 4), col = tid & 15;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (i == col) ? 1.f : 0.f;
#pragma unroll
    for (int j = 0; j < 15; ++j)
#pragma unroll
      for (int i = j + 1; i < 16; ++i) x[i] = fmaf(-Tm[(b0 + i) * MS + b0 + j], x[j], x[i]);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 16; ++i) Tm[(b0 + i) * MS + b0 + col] = x[i];
  }
  __syncthreads();
  for (int bi = 1; bi < 4; ++bi) {
    float *Xs = DT + warp * 16 * 17;  // the slice area is free here
    if (warp < bi) {
      float cs[2][4] = {};
      auto fa = [&](int r, int m) { return ld2(Tm + (16 * bi + r) * MS + m); };
      auto fb = [&](int m, int n) { return make_float2(Tm[m * MS + 16 * warp + n], Tm[(m + 1) * MS + 16 * warp + n]); };
      wgemm_bf<2, false, false>(cs, 16 * warp, 16 * bi, fa, fb);
      cvisit(cs, [&](int, int r, int n, float x) { Xs[r * 17 + n] = x; });
    }
    __syncthreads();
    if (warp < bi) {
      float ct[2][4] = {};
      auto fa = [&](int r, int m) { return ld2(Tm + (16 * bi + r) * MS + 16 * bi + m); };
      auto fb = [&](int m, int n) { return make_float2(Xs[m * 17 + n], Xs[(m + 1) * 17 + n]); };
      wgemm_bf<2, false, false>(ct, 0, 16, fa, fb);
      cvisit(ct, [&](int, int r, int n, float x) { Tm[(16 * bi + r) * MS + 16 * warp + n] = -x; });
    }
    __syncthreads();
  }

  // ---- V slices
  float accK[NH][4] = {}, accQ[NH][4] = {};  // dk^, and do h^T (dq^ before its row scale)
  float accT[4][4] = {}, accP[4][4] = {};    // dT, dP (rows r0.., columns 32 hf..)
  const int x0 = hf * (K / 2);
  for (int v0 = 0; v0 < V; v0 += VS) {
    const int64_t hb = ((slot * HV + hv) * K) * (int64_t)V + v0;
    if (v0 + VS < V) prefetch_slice(v0 + VS);
    for (int e = tid; e < K * (VS / 4); e += BT) {
      const int x = e / (VS / 4), c4 = e % (VS / 4);
      const float4 hv4 = *reinterpret_cast<const float4 *>(Hs + hb + (int64_t)x * V + 4 * c4);
      const float4 dv4 = *reinterpret_cast<const float4 *>(DH + hb + (int64_t)x * V + 4 * c4);
      uint32_t hi[2], lo[2];
      split_bf16(make_float2(hv4.x, hv4.y), hi[0], lo[0]);
      split_bf16(make_float2(hv4.z, hv4.w), hi[1], lo[1]);
      *reinterpret_cast<uint2 *>(Hhi + x * HSB + 4 * c4) = make_uint2(hi[0], hi[1]);
      *reinterpret_cast<uint2 *>(Hlo + x * HSB + 4 * c4) = make_uint2(lo[0], lo[1]);
      split_bf16(make_float2(dv4.x, dv4.y), hi[0], lo[0]);
      split_bf16(make_float2(dv4.z, dv4.w), hi[1], lo[1]);
      *reinterpret_cast<uint2 *>(DHhi + x * HSB + 4 * c4) = make_uint2(hi[0], hi[1]);
      *reinterpret_cast<uint2 *>(DHlo + x * HSB + 4 * c4) = make_uint2(lo[0], lo[1]);
    }
    for (int e = tid; e < 64 * (VS / 8); e += BT) {
      const int i = e / (VS / 8), c8 = e % (VS / 8);
      uint4 a = make_uint4(0, 0, 0, 0), b = a;
      if (i < L) {
        const int64_t off = ((trow0 + i) * HV + hv) * V + v0 + 8 * c8;
        a = *reinterpret_cast<const uint4 *>(v + off);
        b = *reinterpret_cast<const uint4 *>(dout + off);
      }
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
      float *vd = vS + i * SS + 8 * c8, *dd = doS + i * SS + 8 * c8;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        vd[2 * u] = bf16lo_f(aw[u]);
        vd[2 * u + 1] = bf16hi_f(aw[u]);
        dd[2 * u] = bf16lo_f(bw[u]);
        dd[2 * u + 1] = bf16hi_f(bw[u]);
      }
    }
    __syncthreads();
    // k^ h and k^ dh' (columns 16 hf ..): k exact, h, dh' split.  (The q^ h of
    // d gamma's output term is not needed: sum_c (q^_i . h_c) do_ic equals
    // q^_i . (do h^T)_i, formed from the dq^ accumulator after the slices.)
    {
      float ckh[2][4] = {}, ckd[2][4] = {};
      const int n0 = 16 * hf;
      // one pass over K for the two products (shared fragments, four accumulators),
      // bf16 m16n8k16: k raw (exact), h and dh' split hi + lo
      {
        const int fr = lane >> 2, ft = lane & 3;
#pragma unroll 2
        for (int kk = 0; kk < K; kk += 16) {
          uint32_t ak[4];
          ak[0] = *reinterpret_cast<const uint32_t *>(Kb + (r0 + fr) * BR + kk + 2 * ft);
          ak[1] = *reinterpret_cast<const uint32_t *>(Kb + (r0 + fr + 8) * BR + kk + 2 * ft);
          ak[2] = *reinterpret_cast<const uint32_t *>(Kb + (r0 + fr) * BR + kk + 2 * ft + 8);
          ak[3] = *reinterpret_cast<const uint32_t *>(Kb + (r0 + fr + 8) * BR + kk + 2 * ft + 8);
          uint32_t hh[2][2], hl[2][2], dh_[2][2], dl[2][2];
#pragma unroll
          for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int x = kk + 2 * ft + 8 * u, c = n0 + 8 * n + fr;
              hh[n][u] = pair16(Hhi + x * HSB + c, HSB);
              hl[n][u] = pair16(Hlo + x * HSB + c, HSB);
              dh_[n][u] = pair16(DHhi + x * HSB + c, HSB);
              dl[n][u] = pair16(DHlo + x * HSB + c, HSB);
            }
#pragma unroll
          for (int n = 0; n < 2; ++n) {
            mma_bf16(ckh[n], ak, hh[n][0], hh[n][1]);
            mma_bf16(ckd[n], ak, dh_[n][0], dh_[n][1]);
          }
#pragma unroll
          for (int n = 0; n < 2; ++n) {
            mma_bf16(ckh[n], ak, hl[n][0], hl[n][1]);
            mma_bf16(ckd[n], ak, dl[n][0], dl[n][1]);
          }
        }
      }
      cvisit(ckh, [&](int, int r, int n, float x) {
        const int i = r0 + r, cc = n0 + n;
        const float kh = x * rk[i];
        KhS[i * SS + cc] = kh;
        MvS[i * SS + cc] = bet[i] * (vS[i * SS + cc] - og[i] * kh);
      });
      cvisit(ckd, [&](int, int r, int n, float x) { KdhS[(r0 + r) * SS + n0 + n] = x * rk[r0 + r]; });
    }
    __syncthreads();
    if (warp < 4) {
      // v_new = T Mv (T lower)
      float cc[4][4] = {};
      auto fa = [&](int r, int m) { return ld2(Tm + (r0 + r) * MS + m); };
      auto fb = [&](int m, int n) { return make_float2(MvS[m * SS + n], MvS[(m + 1) * SS + n]); };
      wgemm_bf<4, false, false>(cc, 0, r0 + 16, fa, fb);
      cvisit(cc, [&](int, int r, int n, float x) { vnS[(r0 + r) * SS + n] = x; });
    } else {
      // dv_new = diag(sv) k^ dh' + scale P^T do (P^T upper)
      float cc[4][4] = {};
      auto fa = [&](int r, int m) { return make_float2(Pm[m * MS + r0 + r], Pm[(m + 1) * MS + r0 + r]); };
      auto fb = [&](int m, int n) { return make_float2(doS[m * SS + n], doS[(m + 1) * SS + n]); };
      wgemm_bf<4, false, true>(cc, r0, 64, fa, fb);
      cvisit(cc, [&](int, int r, int n, float x) {
        const int i = r0 + r;
        dvnS[i * SS + n] = fmaf(sv[i], KdhS[i * SS + n], scale * x);
      });
    }
    __syncthreads();
    if (warp < 4) {
      // Tu = T^T dv_new (T^T upper); dv = diag(beta) Tu; d beta, d gamma row sums
      float cc[4][4] = {};
      auto fa = [&](int r, int m) { return make_float2(Tm[m * MS + r0 + r], Tm[(m + 1) * MS + r0 + r]); };
      auto fb = [&](int m, int n) { return make_float2(dvnS[m * SS + n], dvnS[(m + 1) * SS + n]); };
      wgemm_bf<4, false, false>(cc, r0, 64, fa, fb);
      float sb[2] = {0.f, 0.f}, sg[2] = {0.f, 0.f};
      cvisit(cc, [&](int rh, int r, int n, float x) {
        const int i = r0 + r;
        TuS[i * SS + n] = x;
        if (i < L) dv[((trow0 + i) * HV + hv) * V + v0 + n] = bet[i] * x;
        const float kh = KhS[i * SS + n];
        sb[rh] = fmaf(x, vS[i * SS + n] - og[i] * kh, sb[rh]);
        sg[rh] = fmaf(x, kh, sg[rh]);
      });
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        sb[u] = quad_sum(sb[u]);
        sg[u] = quad_sum(sg[u]);
      }
      if (t4 == 0) {
        DB[r0 + g8] += sb[0];
        DB[r0 + g8 + 8] += sb[1];
        SG[r0 + g8] += sg[0];
        SG[r0 + g8 + 8] += sg[1];
      }
    } else {
      // state terms: sum_c k^dh'_ic v_new_ic per row, and <dh', h> for d gamma_L
      const int tt = tid - 128, i = tt >> 1, cb = (tt & 1) * (VS / 2);
      float s = 0.f;
#pragma unroll 4
      for (int u = 0; u < VS / 2; ++u) s = fmaf(KdhS[i * SS + cb + u], vnS[i * SS + cb + u], s);
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      if ((tt & 1) == 0) SLv[i] += s;
      float hh = 0.f;
      for (int e = tt; e < K * VS; e += 128) {
        const int o16 = (e / VS) * HSB + e % VS;
        hh = fmaf(bf2f(DHhi[o16]) + bf2f(DHlo[o16]), bf2f(Hhi[o16]) + bf2f(Hlo[o16]), hh);
      }
      hh = warp_sum(hh);
      if (lane == 0) misc[warp - 4] += hh;  // one slot per warp, summed in a fixed order below
    }
    __syncthreads();
    {
      // dT += dv_new Mv^T ; dP += do v_new^T (j <= i)   (bf16 m16n8k16, pairs along the slice)
      auto fa1 = [&](int r, int u) { return ld2(dvnS + (r0 + r) * SS + u); };
      auto fb1 = [&](int u, int n) { return ld2(MvS + (32 * hf + n) * SS + u); };
      wgemm_bf<4, false, false>(accT, 0, VS, fa1, fb1);
      if (!(hf == 1 && mt < 2)) {
        auto fa2 = [&](int r, int u) { return ld2(doS + (r0 + r) * SS + u); };
        auto fb2 = [&](int u, int n) { return ld2(vnS + (32 * hf + n) * SS + u); };
        wgemm_bf<4, true, false>(accP, 0, VS, fa2, fb2);
      }
      // dk^ += [-diag(beta og) Tu | diag(sv) v_new] [h | dh']^T ; do h^T
      auto fa3 = [&](int r, int u) {
        const int i = r0 + r;
        if (u < VS) {
          const float f = -bet[i] * og[i];
          const float2 x = ld2(TuS + i * SS + u);
          return make_float2(f * x.x, f * x.y);
        }
        const float2 x = ld2(vnS + i * SS + u - VS);
        return make_float2(sv[i] * x.x, sv[i] * x.y);
      };
      auto fb3 = [&](int u, int n) {
        const int o16 = (x0 + n) * HSB + (u < VS ? u : u - VS);
        return u < VS ? make_uint2(word16(Hhi + o16), word16(Hlo + o16)) : make_uint2(word16(DHhi + o16), word16(DHlo + o16));
      };
      wgemm_bf_pb<NH, false>(accK, 0, 2 * VS, fa3, fb3);
      auto fa4 = [&](int r, int u) { return ld2(doS + (r0 + r) * SS + u); };
      auto fb4 = [&](int u, int n) {
        const int o16 = (x0 + n) * HSB + u;
        return make_uint2(word16(Hhi + o16), word16(Hlo + o16));
      };
      wgemm_bf_pb<NH, true>(accQ, 0, VS, fa4, fb4);
    }
    __syncthreads();
  }

  // ---- dA = -T^T (dT T^T) (strictly lower)
  cvisit(accT, [&](int, int r, int n, float x) { DT[(r0 + r) * MS + 32 * hf + n] = x; });
  cvisit(accP, [&](int, int r, int n, float x) {
    const int i = r0 + r, j = 32 * hf + n;
    DP[i * MS + j] = (j <= i) ? scale * x : 0.f;
  });
  __syncthreads();
  {
    float cc[4][4] = {};
    auto fa = [&](int r, int m) { return ld2(DT + (r0 + r) * MS + m); };
    auto fb = [&](int m, int n) { return ld2(Tm + (32 * hf + n) * MS + m); };
    wgemm_bf<4, false, false>(cc, 0, 32 * hf + 32, fa, fb);
    cvisit(cc, [&](int, int r, int n, float x) { Xm[(r0 + r) * MS + 32 * hf + n] = x; });
  }
  __syncthreads();
  {
    float cc[4][4] = {};
    if (!(hf == 1 && mt < 2)) {
      auto fa = [&](int r, int m) { return make_float2(Tm[m * MS + r0 + r], Tm[(m + 1) * MS + r0 + r]); };
      auto fb = [&](int m, int n) { return make_float2(Xm[m * MS + 32 * hf + n], Xm[(m + 1) * MS + 32 * hf + n]); };
      wgemm_bf<4, false, false>(cc, r0, 64, fa, fb);
    }
    cvisit(cc, [&](int, int r, int n, float x) {
      const int i = r0 + r, j = 32 * hf + n;
      DT[i * MS + j] = (j < i) ? -x : 0.f;
    });
  }
  __syncthreads();
  // ---- through A_ij = beta_i EK_ij and P_ij: d beta, d gamma (row +, column -),
  // and the coefficient tiles of the last products.  Thread (i, q4) takes
  // elements (i, j) and (j, i) for j = q4 + 4 m, so both the row and the column
  // sums of row / column i reduce within its quad (no shared atomics).
  {
    const int i = tid >> 2, q4 = tid & 3;
    float sb = 0.f, sr = 0.f, sc = 0.f;
#pragma unroll 4
    for (int m = 0; m < 16; ++m) {
      const int j = q4 + 4 * m;
      const float da = DT[i * MS + j], dp = DP[i * MS + j], ek = EK[i * MS + j];
      const float daT = DT[j * MS + i], dpT = DP[j * MS + i];
      sb = fmaf(da, ek, sb);
      sr += fmaf(da * bet[i], ek, dp * Pm[i * MS + j]);
      sc += fmaf(daT * bet[j], EK[j * MS + i], dpT * Pm[j * MS + i]);
      float s1 = 0.f, s2 = 0.f, s3 = 0.f;
      if (j < i) {
        const float e = expf(gam[i] - gam[j]);
        s1 = da * bet[i] * e * rk[j];
        s3 = dp * e * rk[j];
      } else if (j > i) {
        const float e = expf(gam[j] - gam[i]);
        s1 = daT * bet[j] * e * rk[j];
        s2 = dpT * e * rq[j];
      } else {
        s2 = dp * rq[j];
        s3 = dp * rk[j];
      }
      S1[i * MS + j] = s1;
      S2[i * MS + j] = s2;
      S3[i * MS + j] = s3;
    }
    sb = quad_sum(sb);
    sr = quad_sum(sr);
    sc = quad_sum(sc);
    if (q4 == 0) {
      DB[i] += sb;
      DG[i] += sr - sc;
    }
  }
  __syncthreads();
  // ---- dk^ += [S1 | S2] [k; q] ; dq^ = scale og (do h^T) + S3 k
  {
    auto fa = [&](int r, int m) { return m < 64 ? ld2(S1 + (r0 + r) * MS + m) : ld2(S2 + (r0 + r) * MS + m - 64); };
    auto fb = [&](int m, int n) {
      return m < 64 ? make_float2(kv(m, x0 + n), kv(m + 1, x0 + n)) : make_float2(qv(m - 64, x0 + n), qv(m - 63, x0 + n));
    };
    wgemm_bf<NH, false, true>(accK, 0, 128, fa, fb);
    // d gamma's output term: sum_c (q^_i . h_c) do_ic = q^_i . (do h^T)_i
    // (each element of SQ, PQ, PK below gets exactly two adds, one per warp of
    // a row block, so their order cannot change the sum)
    {
      float sq[2] = {0.f, 0.f};
      cvisit(accQ, [&](int rh, int r, int n, float x) { sq[rh] = fmaf(qv(r0 + r, x0 + n), x, sq[rh]); });
#pragma unroll
      for (int u = 0; u < 2; ++u) sq[u] = quad_sum(sq[u]);
      if (t4 == 0) {
        atomicAdd(&SQ[r0 + g8], rq[r0 + g8] * sq[0]);
        atomicAdd(&SQ[r0 + g8 + 8], rq[r0 + g8 + 8] * sq[1]);
      }
    }
    cvisit(accQ, [&](int, int r, int, float &x) { x *= scale * og[r0 + r]; });
    auto fa2 = [&](int r, int m) { return ld2(S3 + (r0 + r) * MS + m); };
    auto fb2 = [&](int m, int n) { return make_float2(kv(m, x0 + n), kv(m + 1, x0 + n)); };
    wgemm_bf<NH, false, true>(accQ, 0, r0 + 16, fa2, fb2);
  }
  // ---- through the L2 norms (dx = r (dx^ - x^ (x^ . dx^))).  The group's first
  // value head writes its share into dq, dk, the j-th later one into slot j - 1
  // of dqk_part (dq shares, then dk shares, part_stride floats apart); a
  // second pass adds the slots in head order, so two runs agree bit for bit.
  {
    float pq[2] = {0.f, 0.f}, pk[2] = {0.f, 0.f};
    cvisit(accQ, [&](int rh, int r, int n, float x) { pq[rh] = fmaf(qv(r0 + r, x0 + n), x, pq[rh]); });
    cvisit(accK, [&](int rh, int r, int n, float x) { pk[rh] = fmaf(kv(r0 + r, x0 + n), x, pk[rh]); });
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      pq[u] = quad_sum(pq[u]);
      pk[u] = quad_sum(pk[u]);
    }
    if (t4 == 0) {
      atomicAdd(&PQ[r0 + g8], pq[0]);
      atomicAdd(&PQ[r0 + g8 + 8], pq[1]);
      atomicAdd(&PK[r0 + g8], pk[0]);
      atomicAdd(&PK[r0 + g8 + 8], pk[1]);
    }
  }
  __syncthreads();
  const int gj = hv % (HV / H);  // this value head's place in its group
  float *dq_dst = gj == 0 ? dq : dqk_part + (int64_t)(gj - 1) * 2 * part_stride;
  float *dk_dst = gj == 0 ? dk : dqk_part + ((int64_t)(gj - 1) * 2 + 1) * part_stride;
  // A thread's accumulator holds two adjacent columns of a row per 8-column
  // tile and row half: one 8-byte store each.
#pragma unroll
  for (int nt = 0; nt < NH; ++nt) {
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
      const int i = r0 + g8 + 8 * rh, xx = x0 + 8 * nt + 2 * t4;
      if (i < L) {
        float gq[2], gk[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float xq = accQ[nt][2 * rh + e], xk = accK[nt][2 * rh + e];
          gq[e] = l2 ? rq[i] * (xq - rq[i] * rq[i] * qv(i, xx + e) * PQ[i]) : xq;
          gk[e] = l2 ? rk[i] * (xk - rk[i] * rk[i] * kv(i, xx + e) * PK[i]) : xk;
        }
        const int64_t off = ((trow0 + i) * H + h) * K + xx;
        *reinterpret_cast<float2 *>(dq_dst + off) = make_float2(gq[0], gq[1]);
        *reinterpret_cast<float2 *>(dk_dst + off) = make_float2(gk[0], gk[1]);
      }
    }
  }
  // ---- d gamma, then dg = reverse cumsum over the chunk; d beta
  if (warp == 0) {
    float d[2], dl = 0.f;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int i = 2 * lane + u;
      d[u] = DG[i] - bet[i] * og[i] * SG[i] + scale * og[i] * SQ[i] - sv[i] * SLv[i];
      dl = fmaf(sv[i], SLv[i], dl);
    }
    dl = warp_sum(dl) + og[63] * (((misc[0] + misc[1]) + misc[2]) + misc[3]);  // d gamma_L
    if (lane == 31) d[1] += dl;
    float s = d[0] + d[1];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_down_sync(0xffffffffu, s, off);
      if (lane + off < 32) s += y;
    }
    const float s1 = s - d[0];  // rows >= 2 lane + 1
    if (2 * lane < L) {
      dg[(trow0 + 2 * lane) * HV + hv] = s;
      dbeta[(trow0 + 2 * lane) * HV + hv] = DB[2 * lane];
    }
    if (2 * lane + 1 < L) {
      dg[(trow0 + 2 * lane + 1) * HV + hv] = s1;
      dbeta[(trow0 + 2 * lane + 1) * HV + hv] = DB[2 * lane + 1];
    }
  }
}

// -------------------------------------------- state-gradient walk, tcgen05
// The same recurrence as chunk_dh_kernel for K = 128 and 64-column slices of
// V, on tcgen05 with TMEM accumulators, built like the forward walk: one CTA
// per (64-column slice, value head, sequence) walks the chunks last to first;
// the fp32 dh' lives in registers of eight chain warps (thread = TMEM lane,
// i.e. key, x 32 columns) and is written back as bf16 hi | lo as the B operand
// of the next chunk's first product.  Per chunk (operands from the record and
// raw bf16 tiles, 128-byte swizzled shared memory, fp32 accumulators):
//   D1 = K [dh'_hi | dh'_lo]               M=128 (rows 64-127 not read) N=128, two partials (warps 0, 1)
//   D2 = P_hi^T do + P_lo^T do             M=128 (rows 64-127 not read) N=64  (converter warp, early)
//   dv_new = diag(sv) (D1 hi + lo) + scale D2     (rows 0-63), as bf16 hi | lo
//   D34 = Q^T [s do_hi | s do_lo]          s = scale e^gamma / ||q||, rows >= L zero (converter, early)
//   D34 -= W^T [dv_new hi | lo]            the A operand negated in the instruction (warp 0)
//   dh = e^{gamma_L} dh' + D34 hi + lo
// Rows >= L of a chunk: W, P rows are zero in the record and the scaled do
// rows are zeroed here, so the K, Q and do rows that TMA brings in from the
// next sequence never reach dh.
struct DhtLay {
  static constexpr int KT = 0;          // K tile [64 tokens][128 keys]: two 64-key atoms of 8 KB (TMA)
  static constexpr int QT = 16384;      // Q tile, the same (TMA)
  static constexpr int WR = 32768;      // record W | P hi | P lo (bulk, 32 KB)
  static constexpr int PH = WR + 16384, PL = WR + 24576;
  static constexpr int DO = 65536;      // do box [64 tokens][64 columns] (TMA)
  static constexpr int SC = 73728;      // record scalars (1 KB)
  static constexpr int STAGE = 74752;
  static constexpr int OFF_H = 2 * STAGE;          // [dh'_hi | dh'_lo]: two N atoms [128 keys][64] of 16 KB
  static constexpr int OFF_DV = OFF_H + 32768;     // [dv_new hi | lo]: two N atoms [64 tokens][64] of 8 KB
  static constexpr int OFF_DS = OFF_DV + 16384;    // [s do hi | lo]: the same
  static constexpr int OFF_BAR = OFF_DS + 16384;
  static constexpr int NBAR = 16;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr uint32_t TX = 4 * 8192 + 32768 + 8192 + 1024;
  static_assert(STAGE % 1024 == 0 && SC + 1024 <= STAGE && OFF_H % 1024 == 0, "stage layout");
  static_assert(BYTES + 1024 <= 232448, "shared memory budget (227 KB per CTA)");
};
// TMEM columns.
constexpr uint32_t DT_D1A = 0, DT_D1B = 128, DT_D2 = 256, DT_D34 = 384;
constexpr int DT_THREADS = 11 * 32;
enum { DB_FULL = 0, DB_EMPTY = 2, DB_D2R = 4, DB_CHD = 6, DB_M1 = 8, DB_M3 = 9, DB_D4R = 10, DB_DRAIN = 11,
       DB_CONV = 12 };

__global__ void __launch_bounds__(DT_THREADS, 1) chunk_dh_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_do, const unsigned char *__restrict__ ws, float *__restrict__ DH,
    const float *__restrict__ dht, float *__restrict__ dh0, float scale, const int32_t *__restrict__ cu,
    const int32_t *__restrict__ cs, int T, int H, int HV, int V, int32_t *dev_status) {
  constexpr int K = 128;
  using Ly = DhtLay;
  using R = Rec<K>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                        ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  const int vt0 = blockIdx.x * DVC, hv = blockIdx.y, n = blockIdx.z;
  const int h = hv / (HV / H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int64_t tok0, len;
  if (!seq_bounds(cu, n, T, tok0, len)) {
    if (tid == 0) set_status(dev_status, GDN_DEV_BAD_CU_SEQLENS);
    return;
  }
  const int NC = chunks_of(len);
  const int64_t cb = chunk_base(cs, n, T);
  const int64_t sbase = ((int64_t)n * HV + hv) * K;
  uint32_t *misc = reinterpret_cast<uint32_t *>(sm + Ly::OFF_MISC);
  volatile uint32_t *abort_flag = misc + 1;
  auto bar = [&](int i) { return sb + Ly::OFF_BAR + 8 * i; };
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(DB_FULL + b), 1);
      mbar_init(bar(DB_EMPTY + b), 1);
      mbar_init(bar(DB_D2R + b), 1);
      mbar_init(bar(DB_CHD + b), 1);
    }
    mbar_init(bar(DB_M1), 2);
    mbar_init(bar(DB_M3), 1);
    mbar_init(bar(DB_D4R), 1);
    mbar_init(bar(DB_CONV), 2);
    mbar_init(bar(DB_DRAIN), 4);  // warps 0, 1 and 9, and the producer's stand-in
    misc[1] = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(sb + Ly::OFF_MISC, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  bool dead = false;
  auto waitl = [&](uint32_t b, uint32_t parity) -> bool {
    uint32_t ok = 0;
    if (lane == 0 && !dead) {
      const long long t0 = clock64();
      for (int it = 1;; ++it) {
        if (mbar_try_wait(b, parity)) { ok = 1; break; }
        if ((it & 63) == 0) {
          if (*abort_flag) break;
          if (clock64() - t0 > kWaitLimit) { *abort_flag = 1; break; }
        }
      }
    }
    __syncwarp();
    ok = __shfl_sync(0xffffffffu, ok, 0);
    dead = dead || !ok;
    return ok != 0;
  };
  auto wait2 = [&](int slot, int it) { return waitl(bar(slot + (it & 1)), (it >> 1) & 1); };
  auto stage = [&](int it) { return sb + (it & 1) * Ly::STAGE; };
  auto chunk_of = [&](int it) { return NC - 1 - it; };
  auto rows_of = [&](int c) {
    const int64_t rem = len - (int64_t)c * C;
    return rem < C ? (int)rem : C;
  };
  constexpr uint32_t ID1 = umma_idesc_bf16(128, 128, 0, 1);
  constexpr uint32_t ID2 = umma_idesc_bf16(128, 64, 1, 1);
  constexpr uint32_t ID4 = umma_idesc_bf16(128, 128, 1, 1);
  constexpr uint32_t ID3N = umma_idesc_bf16(128, 128, 1, 1) | (1u << 13);  // A negated
  int issued = 0;

  if (warp < 8) {
    // ------------------------------------------------------- chain warps
    const int r = 32 * (warp & 3) + lane;  // TMEM lane: key (dh) or token (dv_new, r < 64)
    const int hs = warp >> 2;              // columns 32 hs .. 32 hs + 31 of the slice
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    float dh[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) dh[j] = dht ? dht[(sbase + r) * V + vt0 + 32 * hs + j] : 0.f;
    // Row r of a two-atom MN-major SW128 tile (atom = 64 columns): columns
    // [32 hs, 32 hs + 32) of the hi and the lo atom.
    auto write_split = [&](uint32_t off, int atom_bytes, const float *x) {
      unsigned char *base = sm + off + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = x[8 * m + 2 * e], x1 = x[8 * m + 2 * e + 1];
          hi[e] = pack_bf16(x0, x1);
          lo[e] = pack_bf16(x0 - bf16lo_f(hi[e]), x1 - bf16hi_f(hi[e]));
        }
        const int chk = (4 * hs + m) ^ (r & 7);
        *reinterpret_cast<uint4 *>(base + (chk << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(base + atom_bytes + (chk << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    };
    bool go = true;
    for (int it = 0; it < NC; ++it) {
      const int c = chunk_of(it);
      // dh' of chunk c: to the workspace and, split, to the H tile (its last
      // reader, the first product of the chunk before, has completed).
      {
        float *dst = DH + (((cb + c) * HV + hv) * K + r) * (int64_t)V + vt0 + 32 * hs;
#pragma unroll
        for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4 *>(dst + j) = make_float4(dh[j], dh[j + 1], dh[j + 2], dh[j + 3]);
        write_split(Ly::OFF_H, 16384, dh);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 256);
      go = wait2(DB_FULL, it) && go;
      const unsigned char *scp = sm + (it & 1) * Ly::STAGE + Ly::SC;
      const float dL = go ? reinterpret_cast<const float *>(scp)[RS_DL] : 0.f;
      const float svr = (go && r < 64) ? reinterpret_cast<const float *>(scp)[RS_SV + r] : 0.f;
      if (warp < 2 && lane == 0 && go) {
        tc_fence_after();
        const uint32_t st = stage(it);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int kk = 4 * warp + m;  // keys 16 kk .. 16 kk + 15
          const uint64_t a = umma_desc_sw128(st + Ly::KT + (kk >> 2) * 8192 + (kk & 3) * 32);
          const uint64_t b = umma_desc_sw128_mn(sb + Ly::OFF_H + kk * 2048, 16384);
          umma_bf16(tmem + (warp ? DT_D1B : DT_D1A), a, b, ID1, m > 0 ? 1u : 0u);
        }
        umma_commit(bar(DB_M1));
      }
      __syncwarp();
      go = waitl(bar(DB_M1), it & 1) && go;
      go = wait2(DB_D2R, it) && go;
      if (go && r < 64) {
        // dv_new rows 0-63 (warps 0, 1, 4, 5), 16 columns at a time.
        tc_fence_after();
        float dv[32];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint32_t col = 32 * hs + 16 * q;
          uint32_t a0[16], a1[16], b0[16], b1[16], p[16];
          tmem_ld16_issue(tl + DT_D1A + col, a0);
          tmem_ld16_issue(tl + DT_D1A + 64 + col, a1);
          tmem_ld16_issue(tl + DT_D1B + col, b0);
          tmem_ld16_issue(tl + DT_D1B + 64 + col, b1);
          tmem_ld16_issue(tl + DT_D2 + 64 * (it & 1) + col, p);
          tmem_ld_wait16(a0);
          tmem_ld_wait16(a1);
          tmem_ld_wait16(b0);
          tmem_ld_wait16(b1);
          tmem_ld_wait16(p);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float kd = (__uint_as_float(a0[j]) + __uint_as_float(a1[j])) + (__uint_as_float(b0[j]) + __uint_as_float(b1[j]));
            dv[16 * q + j] = fmaf(svr, kd, scale * __uint_as_float(p[j]));
          }
        }
        write_split(Ly::OFF_DV, 8192, dv);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(1, 256);
      if (warp == 0) {
        go = waitl(bar(DB_D4R), it & 1) && go;  // Q^T (s do) is in D34: accumulate onto it
        if (lane == 0 && go) {
          tc_fence_after();
          const uint32_t st = stage(it);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = umma_desc_sw128_mn(st + Ly::WR + kk * 2048, 8192);
            const uint64_t b = umma_desc_sw128_mn(sb + Ly::OFF_DV + kk * 2048, 8192);
            umma_bf16(tmem + DT_D34, a, b, ID3N, 1u);
          }
          umma_commit(bar(DB_M3));
          umma_commit(bar(DB_EMPTY + (it & 1)));  // every product that reads the stage is done then
        }
        __syncwarp();
      }
      go = waitl(bar(DB_M3), it & 1) && go;
      if (go) {
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint32_t col = 32 * hs + 16 * q;
          uint32_t x0[16], x1[16];
          tmem_ld16_issue(tl + DT_D34 + col, x0);
          tmem_ld16_issue(tl + DT_D34 + 64 + col, x1);
          tmem_ld_wait16(x0);
          tmem_ld_wait16(x1);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            dh[16 * q + j] = fmaf(dL, dh[16 * q + j], __uint_as_float(x0[j]) + __uint_as_float(x1[j]));
        }
      }
      tc_fence_before();
      named_bar_sync(1, 256);
      if (tid == 0) mbar_arrive(bar(DB_CHD + (it & 1)));
    }
    if (dh0 && !*abort_flag) {
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4 *>(dh0 + (sbase + r) * V + vt0 + 32 * hs + j) =
            make_float4(dh[j], dh[j + 1], dh[j + 2], dh[j + 3]);
    }
  } else if (warp == 8) {
    // ----------------------------------------------------------- producer
    for (int it = 0; it < NC; ++it) {
      if (it >= 2 && !wait2(DB_EMPTY, it - 2)) break;
      if (lane == 0) {
        const int c = chunk_of(it);
        const uint32_t st = stage(it), fb = bar(DB_FULL + (it & 1));
        const int trow = static_cast<int>(tok0) + c * C;
        const unsigned char *rec = ws + (static_cast<size_t>(cb + c) * HV + hv) * R::BYTES;
        mbar_arrive_expect_tx(fb, Ly::TX);
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          tma_load_3d(st + Ly::KT + a * 8192, &tm_k, fb, 64 * a, h, trow);
          tma_load_3d(st + Ly::QT + a * 8192, &tm_q, fb, 64 * a, h, trow);
        }
#pragma unroll
        for (int p = 0; p < 4; ++p) bulk_load(st + Ly::WR + p * 8192, rec + R::W + p * 8192, 8192, fb);
        tma_load_3d(st + Ly::DO, &tm_do, fb, vt0, hv, trow);
        bulk_load(st + Ly::SC, rec + R::SC, 1024, fb);
      }
      issued = it + 1;
      __syncwarp();
    }
  } else if (warp == 9 || warp == 10) {
    // ------------- converters: P^T do into D2 (warp 9), the scaled do tile
    // (rows 0-31 warp 9, rows 32-63 warp 10), Q^T (s do) into D34 (warp 9)
    const int cw = warp - 9;
    for (int it = 0; it < NC; ++it) {
      const int c = chunk_of(it);
      const uint32_t st = stage(it);
      bool ok = wait2(DB_FULL, it);
      if (cw == 0 && it >= 2) ok = ok && wait2(DB_CHD, it - 2);  // the chain has read D2 of chunk it - 2
      if (!ok) break;
      if (cw == 0 && lane == 0) {
        tc_fence_after();
        const uint32_t d2 = tmem + DT_D2 + 64 * (it & 1);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(d2, umma_desc_sw128_mn(st + Ly::PH + kk * 2048, 8192), umma_desc_sw128_mn(st + Ly::DO + kk * 2048, 8192),
                    ID2, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(d2, umma_desc_sw128_mn(st + Ly::PL + kk * 2048, 8192), umma_desc_sw128_mn(st + Ly::DO + kk * 2048, 8192),
                    ID2, 1u);
        umma_commit(bar(DB_D2R + (it & 1)));
      }
      __syncwarp();
      // The scaled do tile and D34 of chunk it - 1 are free once the chain has
      // finished that chunk.
      if (it >= 1 && !wait2(DB_CHD, it - 1)) break;
      {
        const int L = rows_of(c);
        const float *scf = reinterpret_cast<const float *>(sm + (it & 1) * Ly::STAGE + Ly::SC);
        const unsigned char *dop = sm + (it & 1) * Ly::STAGE + Ly::DO;
        {
          const int i = lane + 32 * cw;
          const float s = i < L ? scale * scf[RS_OG + i] : 0.f;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint4 x = *reinterpret_cast<const uint4 *>(dop + sw128(i, ch));
            const uint32_t xv[4] = {x.x, x.y, x.z, x.w};
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float y0 = s * bf16lo_f(xv[e]), y1 = s * bf16hi_f(xv[e]);
              hi[e] = pack_bf16(y0, y1);
              lo[e] = pack_bf16(y0 - bf16lo_f(hi[e]), y1 - bf16hi_f(hi[e]));
            }
            *reinterpret_cast<uint4 *>(sm + Ly::OFF_DS + sw128(i, ch)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(sm + Ly::OFF_DS + 8192 + sw128(i, ch)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(DB_CONV));
      if (cw == 1) continue;
      if (!waitl(bar(DB_CONV), it & 1)) break;  // both halves of the scaled do tile are written
      if (lane == 0) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(tmem + DT_D34, umma_desc_sw128_mn(st + Ly::QT + kk * 2048, 8192),
                    umma_desc_sw128_mn(sb + Ly::OFF_DS + kk * 2048, 8192), ID4, kk > 0 ? 1u : 0u);
        umma_commit(bar(DB_D4R));
      }
      __syncwarp();
    }
  }
  // After an abort: the producer waits for its last loads; the issuing threads
  // commit once more to DRAIN (warps 0, 1, 9, plus thread 0 for the producer's
  // share), completing when their products have.
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    if (warp == 8 && lane == 0)
      for (int k2 = (issued > 2 ? issued - 2 : 0); k2 < issued; ++k2)
        if (!mbar_wait_bounded(bar(DB_FULL + (k2 & 1)), (k2 >> 1) & 1, kWaitLimit))
          set_status(dev_status, GDN_DEV_DRAIN_TIMEOUT);
    if (lane == 0 && (warp < 2 || warp == 9)) {
      tc_fence_after();
      umma_commit(bar(DB_DRAIN));
    }
    if (tid == 0) {
      mbar_arrive(bar(DB_DRAIN));
      if (!mbar_wait_bounded(bar(DB_DRAIN), 0, kWaitLimit)) set_status(dev_status, GDN_DEV_DRAIN_TIMEOUT);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (tid == 0 && *abort_flag) set_status(dev_status, GDN_DEV_WAIT_TIMEOUT);
}

typedef CUresult (*DhEncodeFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                               const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                               CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// 3-D map over a [rows][heads][dim] bf16 tensor, box {64, 1 head, 64 rows}, 128-byte swizzle.
bool dh_map(CUtensorMap *m, const void *ptr, int dim, int heads, int64_t rows) {
  static DhEncodeFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) != cudaSuccess ||
        qr != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<DhEncodeFn>(p);
  }
  cuuint64_t gdim[3] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstr[2] = {static_cast<cuuint64_t>(dim) * 2, static_cast<cuuint64_t>(dim) * heads * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), gdim, gstr, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// dq, dk += the shares of a group's later value heads, added in head order
// (part holds nparts pairs of [rows, H, K] shares: dq's, then dk's).
__global__ void __launch_bounds__(256) dqk_sum_kernel(float *__restrict__ dq, float *__restrict__ dk,
                                                      const float *__restrict__ part, int64_t n4,
                                                      int64_t part_stride, int nparts) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
    float4 a = reinterpret_cast<const float4 *>(dq)[i], b = reinterpret_cast<const float4 *>(dk)[i];
    for (int j = 0; j < nparts; ++j) {
      const float4 pa = reinterpret_cast<const float4 *>(part + 2 * j * part_stride)[i];
      const float4 pb = reinterpret_cast<const float4 *>(part + (2 * j + 1) * part_stride)[i];
      a = make_float4(a.x + pa.x, a.y + pa.y, a.z + pa.z, a.w + pa.w);
      b = make_float4(b.x + pb.x, b.y + pb.y, b.z + pb.z, b.w + pb.w);
    }
    reinterpret_cast<float4 *>(dq)[i] = a;
    reinterpret_cast<float4 *>(dk)[i] = b;
  }
}

template <int K>
cudaError_t launch_bwd_k(const gdn_host::ChunkBwdArgs &a, cudaStream_t s) {
  const int64_t slots = total_chunk_slots(a.B, a.T, a.N, a.cu != nullptr);
  const size_t hbytes = (size_t)slots * a.HV * K * a.V * sizeof(float);
  unsigned char *wsb = static_cast<unsigned char *>(a.ws);
  const size_t rec_bytes = gdn_host::chunk_workspace_bytes(a.B, a.T, a.H, a.HV, K, a.V, a.N, a.cu != nullptr);
  float *Hs = reinterpret_cast<float *>(wsb + rec_bytes);
  float *DH = reinterpret_cast<float *>(wsb + rec_bytes + hbytes);
  // The forward below writes the chunk starts of cu_seqlens input right after its records.
  const int32_t *cs =
      a.cu ? reinterpret_cast<const int32_t *>(wsb + (size_t)slots * a.HV * Rec<K>::BYTES) : nullptr;
  const int64_t rows = (int64_t)a.B * a.T;
  // dq, dk shares of the later value heads of each group, after the states.
  const int nparts = a.HV / a.H - 1;
  const int64_t part_stride = rows * a.H * K;
  float *part = reinterpret_cast<float *>(wsb + rec_bytes + 2 * hbytes);
  cudaError_t e;
  if (rows > 0 && a.cu) {
    // Every token of every sequence gets its dq, dk (and shares) written;
    // tokens that cu_seqlens leaves outside all sequences stay zero.
    e = cudaMemsetAsync(a.dq, 0, (size_t)part_stride * sizeof(float), s);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(a.dk, 0, (size_t)part_stride * sizeof(float), s);
    if (e != cudaSuccess) return e;
    if (nparts > 0) {
      e = cudaMemsetAsync(part, 0, (size_t)nparts * 2 * part_stride * sizeof(float), s);
      if (e != cudaSuccess) return e;
    }
  }
  // 1. forward again, saving the state entering every chunk (no output needed)
  gdn_host::ChunkArgs f{};
  f.q = a.q; f.k = a.k; f.v = a.v; f.g = a.g; f.beta = a.beta; f.scale = a.scale; f.h0 = a.h0; f.cu = a.cu;
  f.N = a.N; f.B = a.B; f.T = a.T; f.H = a.H; f.HV = a.HV; f.K = K; f.V = a.V; f.l2 = a.l2;
  f.o = nullptr; f.ht = nullptr; f.hsave = Hs; f.ws = a.ws; f.ws_bytes = rec_bytes; f.dev_status = a.dev_status;
  e = gdn_host::launch_chunk(f, s);
  if (e != cudaSuccess) return e;
  // 2. state gradients, last chunk first (tcgen05 walk at K = 128 and 64-column slices)
  if (K == 128 && a.V % DVC == 0 && rows > 0) {
    CUtensorMap mq, mk, md;
    memset(&mq, 0, sizeof(mq));
    memset(&mk, 0, sizeof(mk));
    memset(&md, 0, sizeof(md));
    if (!dh_map(&mq, a.q, K, a.H, rows) || !dh_map(&mk, a.k, K, a.H, rows) || !dh_map(&md, a.dout, a.V, a.HV, rows))
      return cudaErrorInvalidValue;
    const int smem = DhtLay::BYTES + 1024;
    e = cudaFuncSetAttribute(chunk_dh_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    chunk_dh_tc_kernel<<<dim3(a.V / DVC, a.HV, a.N), DT_THREADS, smem, s>>>(
        mq, mk, md, static_cast<const unsigned char *>(a.ws), DH, a.dht, a.dh0, a.scale, a.cu, cs, a.T, a.H, a.HV,
        a.V, a.dev_status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  } else {
    const int smem = DhLay<K>::BYTES;
    e = cudaFuncSetAttribute(chunk_dh_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    chunk_dh_kernel<K><<<dim3(a.V / DVC, a.HV, a.N), BT, smem, s>>>(
        a.q, a.k, a.dout, static_cast<const unsigned char *>(a.ws), DH, a.dht, a.dh0, a.scale, a.cu, cs, a.T,
        a.H, a.HV, a.V, a.dev_status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // 3. per-chunk gradients
  if (rows > 0 && slots > 0) {
    const int smem = GradLay<K>::BYTES;
    e = cudaFuncSetAttribute(chunk_grad_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    chunk_grad_kernel<K><<<dim3((unsigned)(slots * a.HV)), BT, smem, s>>>(
        a.q, a.k, a.v, a.g, a.beta, a.dout, Hs, DH, a.scale, a.cu, cs, a.N, a.T, a.H, a.HV, a.V, a.l2, a.dq,
        a.dk, part, part_stride, a.dv, a.dg, a.dbeta, a.dev_status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (nparts > 0) {
      int dev = 0, sms = 148;
      cudaGetDevice(&dev);
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      const int64_t n4 = part_stride / 4;
      const int64_t want = (n4 + 255) / 256;
      const int blocks = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
      dqk_sum_kernel<<<blocks, 256, 0, s>>>(a.dq, a.dk, part, n4, part_stride, nparts);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace

namespace gdn_host {

size_t chunk_bwd_workspace_bytes(int B, int T, int H, int HV, int K, int V, int N, int varlen) {
  const size_t rec = chunk_workspace_bytes(B, T, H, HV, K, V, N, varlen);
  const size_t st = (size_t)total_chunk_slots(B, T, N, varlen != 0) * HV * K * V * sizeof(float);
  // the dq, dk shares of each group's later value heads
  const size_t parts = H > 0 ? (size_t)(HV / H - 1) * 2 * B * T * H * K * sizeof(float) : 0;
  return rec + 2 * st + parts;
}

cudaError_t launch_chunk_bwd(const ChunkBwdArgs &a, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  if (a.K == 128) return launch_bwd_k<128>(a, s);
  if (a.K == 64) return launch_bwd_k<64>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace gdn_host
