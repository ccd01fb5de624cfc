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
// chunk.  Both kernels here compute in fp32 on the CUDA cores.
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

// ------------------------------------------------------------------ dh walk
// One CTA per (32-column slice of V, value head, sequence): dh (K x 32 fp32)
// lives in registers, thread (row r, columns c0 .. c0 + CPT); per chunk, last
// first, K, Q, W, P, the scalars and the do slice are staged in shared memory
// (cp.async, double buffered).
template <int K>
struct DhLay {
  static constexpr int KROW = K * 2 + 16;             // padded bf16 row of K keys
  static constexpr int OFF_K = 0;                     // raw K [64][KROW]
  static constexpr int OFF_Q = OFF_K + 64 * KROW;     // raw Q [64][KROW]
  static constexpr int OFF_REC = OFF_Q + 64 * KROW;   // record bytes W | PH | PL (contiguous in the record)
  static constexpr int REC_BYTES = Rec<K>::TS;        // W + PH + PL
  static constexpr int OFF_SC = OFF_REC + REC_BYTES;  // record scalars (1 KB)
  static constexpr int OFF_DO = OFF_SC + 1024;        // do slice [64][32] bf16
  static constexpr int STAGE = OFF_DO + 64 * 64;
  static constexpr int OFF_DHS = 2 * STAGE;           // dh' [K][32] fp32
  static constexpr int OFF_DVN = OFF_DHS + K * 32 * 4;  // dv_new [64][32] fp32
  static constexpr int BYTES = OFF_DVN + 64 * 32 * 4;
  static_assert(STAGE % 16 == 0, "16-byte copies");
};

template <int K>
__global__ void __launch_bounds__(BT, 1) chunk_dh_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ k, const uint16_t *__restrict__ dout,
    const unsigned char *__restrict__ ws, float *__restrict__ DH, const float *__restrict__ dht,
    float *__restrict__ dh0, float scale, const int32_t *__restrict__ cu, int T, int H, int HV, int V,
    int32_t *dev_status) {
  using Ly = DhLay<K>;
  using R = Rec<K>;
  constexpr int TPR = BT / K;   // threads per state row
  constexpr int CPT = 32 / TPR; // columns per thread
  extern __shared__ __align__(16) unsigned char smem[];
  const int vt0 = blockIdx.x * 32, hv = blockIdx.y, n = blockIdx.z;
  const int h = hv / (HV / H);
  const int tid = threadIdx.x;
  const int r = tid / TPR, c0 = (tid % TPR) * CPT;

  int64_t tok0, len;
  if (!seq_bounds(cu, n, T, tok0, len)) {
    if (tid == 0) set_status(dev_status, GDN_DEV_BAD_CU_SEQLENS);
    return;
  }
  const int NC = chunks_of(len);
  const int64_t cb = chunk_base(cu, n, T);
  const int64_t sidx = ((int64_t)n * HV + hv) * K + r;
  float dh[CPT];
#pragma unroll
  for (int j = 0; j < CPT; ++j) dh[j] = dht ? dht[sidx * V + vt0 + c0 + j] : 0.f;

  auto issue = [&](int c, int st) {
    unsigned char *S = smem + st * Ly::STAGE;
    const int64_t trow = tok0 + (int64_t)c * C;
    const int64_t rem = len - (int64_t)c * C;
    const int L = rem < C ? (int)rem : C;
    // K and Q rows: K * 2 bytes = K / 8 chunks of 16 bytes each
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
    for (int e = tid; e < 64 * 4; e += BT) {
      const int row = e >> 2, ch = e & 3;
      const bool ok = row < L;
      const int64_t g = ok ? ((trow + row) * HV + hv) * V + vt0 + ch * 8 : 0;
      cp_async16(S + Ly::OFF_DO + row * 64 + ch * 16, dout + g, ok);
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
    // dh' of this chunk: to the workspace and to shared memory.
    {
      float *dst = DH + (((cb + c) * HV + hv) * K + r) * (int64_t)V + vt0 + c0;
#pragma unroll
      for (int j = 0; j < CPT; ++j) {
        dst[j] = dh[j];
        dhs[r * 32 + c0 + j] = dh[j];
      }
    }
    __syncthreads();
    const unsigned char *S = smem + st * Ly::STAGE;
    const float *sc = reinterpret_cast<const float *>(S + Ly::OFF_SC);
    const uint16_t *Ks = reinterpret_cast<const uint16_t *>(S + Ly::OFF_K);
    const uint16_t *Qs = reinterpret_cast<const uint16_t *>(S + Ly::OFF_Q);
    const uint16_t *Ds = reinterpret_cast<const uint16_t *>(S + Ly::OFF_DO);
    const unsigned char *PH = S + Ly::OFF_REC + (R::PH - R::W);
    const unsigned char *PL = S + Ly::OFF_REC + (R::PL - R::W);
    // dv_new[j][8 columns] = sv_j (k_j . dh'[:, c]) + scale sum_{i >= j} P_ij do_i[c]
    {
      const int j = tid >> 2, cq = (tid & 3) * 8;
      float a[8], b[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) a[x] = b[x] = 0.f;
      const uint16_t *kr = Ks + j * (Ly::KROW / 2);
      for (int key = 0; key < K; ++key) {
        const float kv = bf2f(kr[key]);
        const float *dr = dhs + key * 32 + cq;
#pragma unroll
        for (int x = 0; x < 8; ++x) a[x] = fmaf(kv, dr[x], a[x]);
      }
      for (int i = j; i < 64; ++i) {
        const float p = tile64(PH, i, j) + tile64(PL, i, j);
        const uint16_t *dr = Ds + i * 32 + cq;
#pragma unroll
        for (int x = 0; x < 8; ++x) b[x] = fmaf(p, bf2f(dr[x]), b[x]);
      }
      const float sv = sc[RS_SV + j];
#pragma unroll
      for (int x = 0; x < 8; ++x) dvn[j * 32 + cq + x] = fmaf(sv, a[x], scale * b[x]);
    }
    __syncthreads();
    // dh = e^{gamma_L} dh' + scale sum_i og_i q_i[r] do_i - sum_j W_j[r] dv_new_j
    {
      float a[CPT], b[CPT];
#pragma unroll
      for (int x = 0; x < CPT; ++x) a[x] = b[x] = 0.f;
      const unsigned char *Wt = S + Ly::OFF_REC;
      for (int i = 0; i < 64; ++i) {
        const float qo = sc[RS_OG + i] * bf2f(Qs[i * (Ly::KROW / 2) + r]);
        const float wv = rec_w(Wt, i, r);
        const uint16_t *dr = Ds + i * 32 + c0;
        const float *vr = dvn + i * 32 + c0;
#pragma unroll
        for (int x = 0; x < CPT; ++x) {
          a[x] = fmaf(qo, bf2f(dr[x]), a[x]);
          b[x] = fmaf(wv, vr[x], b[x]);
        }
      }
      const float dL = sc[RS_DL];
#pragma unroll
      for (int x = 0; x < CPT; ++x) dh[x] = fmaf(dL, dh[x], fmaf(scale, a[x], -b[x]));
    }
    __syncthreads();  // this stage is refilled by the next issue
  }
  if (dh0) {
#pragma unroll
    for (int j = 0; j < CPT; ++j) dh0[sidx * V + vt0 + c0 + j] = dh[j];
  }
}

// ---------------------------------------------------------- chunk gradients
// One CTA per (chunk, value head), fp32 throughout.  Thread t owns row
// i = t / 4 of every 64-row result and a quarter of its columns.
constexpr int VS = 16;  // V columns per slice

template <int K>
struct GradLay {
  static constexpr int QROW = K + 4;                        // padded fp32 rows
  static constexpr int OFF_Q = 0;                           // q^ [64][QROW]
  static constexpr int OFF_K = OFF_Q + 64 * QROW * 4;       // k^ [64][QROW]
  static constexpr int M64 = 64 * 65 * 4;                   // a padded 64 x 64 fp32 tile
  static constexpr int OFF_KK = OFF_K + 64 * QROW * 4;      // k^ k^T
  static constexpr int OFF_QK = OFF_KK + M64;               // q^ k^T
  static constexpr int OFF_T = OFF_QK + M64;                // T
  static constexpr int OFF_DT = OFF_T + M64;                // dT
  static constexpr int OFF_DP = OFF_DT + M64;               // dP
  static constexpr int OFF_X = OFF_DP + M64;                // scratch 64 x 64
  static constexpr int SROW = VS + 1;
  static constexpr int OFF_H = OFF_X + M64;                 // h slice [K][SROW]
  static constexpr int OFF_DH = OFF_H + K * SROW * 4;       // dh' slice [K][SROW]
  static constexpr int OFF_V = OFF_DH + K * SROW * 4;       // v slice [64][SROW]
  static constexpr int OFF_DO = OFF_V + 64 * SROW * 4;      // do slice
  static constexpr int OFF_KH = OFF_DO + 64 * SROW * 4;     // k^ h
  static constexpr int OFF_QH = OFF_KH + 64 * SROW * 4;     // q^ h
  static constexpr int OFF_KDH = OFF_QH + 64 * SROW * 4;    // k^ dh'
  static constexpr int OFF_VN = OFF_KDH + 64 * SROW * 4;    // v_new
  static constexpr int OFF_DVN = OFF_VN + 64 * SROW * 4;    // dv_new
  static constexpr int OFF_TU = OFF_DVN + 64 * SROW * 4;    // T^T dv_new
  static constexpr int OFF_VEC = OFF_TU + 64 * SROW * 4;    // per-row vectors
  static constexpr int NVEC = 12;
  static constexpr int BYTES = OFF_VEC + NVEC * 64 * 4 + 16;
};
enum { GV_GAM = 0, GV_BET, GV_RQ, GV_RK, GV_OG, GV_SV, GV_DB, GV_DG, GV_DGL, GV_TMP, GV_TMP2, GV_L };

template <int K>
__global__ void __launch_bounds__(BT, 1) chunk_grad_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
    const float *__restrict__ g, const float *__restrict__ beta, const uint16_t *__restrict__ dout,
    const float *__restrict__ Hs, const float *__restrict__ DH, float scale, const int32_t *__restrict__ cu,
    int N, int T, int H, int HV, int V, int l2, float *__restrict__ dq, float *__restrict__ dk,
    float *__restrict__ dv, float *__restrict__ dg, float *__restrict__ dbeta, int32_t *dev_status) {
  using Ly = GradLay<K>;
  constexpr int QR = Ly::QROW, SR = Ly::SROW;
  extern __shared__ __align__(16) unsigned char smem[];
  float *Qh = reinterpret_cast<float *>(smem + Ly::OFF_Q);
  float *Kh = reinterpret_cast<float *>(smem + Ly::OFF_K);
  float *KK = reinterpret_cast<float *>(smem + Ly::OFF_KK);
  float *QK = reinterpret_cast<float *>(smem + Ly::OFF_QK);
  float *Tm = reinterpret_cast<float *>(smem + Ly::OFF_T);
  float *dT = reinterpret_cast<float *>(smem + Ly::OFF_DT);
  float *dP = reinterpret_cast<float *>(smem + Ly::OFF_DP);
  float *X = reinterpret_cast<float *>(smem + Ly::OFF_X);
  float *hS = reinterpret_cast<float *>(smem + Ly::OFF_H);
  float *dhS = reinterpret_cast<float *>(smem + Ly::OFF_DH);
  float *vS = reinterpret_cast<float *>(smem + Ly::OFF_V);
  float *doS = reinterpret_cast<float *>(smem + Ly::OFF_DO);
  float *KhS = reinterpret_cast<float *>(smem + Ly::OFF_KH);
  float *QhS = reinterpret_cast<float *>(smem + Ly::OFF_QH);
  float *KdhS = reinterpret_cast<float *>(smem + Ly::OFF_KDH);
  float *vnS = reinterpret_cast<float *>(smem + Ly::OFF_VN);
  float *dvnS = reinterpret_cast<float *>(smem + Ly::OFF_DVN);
  float *TuS = reinterpret_cast<float *>(smem + Ly::OFF_TU);
  float *vec = reinterpret_cast<float *>(smem + Ly::OFF_VEC);
  float *gam = vec + GV_GAM * 64, *bet = vec + GV_BET * 64, *rq = vec + GV_RQ * 64, *rk = vec + GV_RK * 64;
  float *og = vec + GV_OG * 64, *sv = vec + GV_SV * 64, *dbv = vec + GV_DB * 64, *dgam = vec + GV_DG * 64;
  float *tmp = vec + GV_TMP * 64;
  constexpr int M = 65;  // padded 64 x 64 stride

  const int gc = blockIdx.x, hv = blockIdx.y;
  const int h = hv / (HV / H);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ri = tid >> 2, qd = tid & 3;  // row and column quarter of 64-row results

  // Which sequence / chunk?
  int c = 0;
  int64_t tok0 = 0, len = 0, slot = gc;
  {
    int64_t base = 0;
    bool found = false;
    for (int m = 0; m < N && !found; ++m) {
      int64_t t0, l0;
      if (!seq_bounds(cu, m, T, t0, l0)) continue;
      const int nc = chunks_of(l0);
      if (gc < base + nc) {
        found = true;
        c = (int)(gc - base);
        tok0 = t0;
        len = l0;
      }
      base += nc;
    }
    if (!found) return;
  }
  const int64_t rem = len - (int64_t)c * C;
  const int L = rem < C ? (int)rem : C;
  const int64_t trow0 = tok0 + (int64_t)c * C;

  // ---- q^, k^, gates, decays
  for (int e = tid; e < 64 * K; e += BT) {
    const int i = e / K, x = e % K;
    const bool live = i < L;
    Qh[i * QR + x] = live ? bf2f(q[((trow0 + i) * H + h) * K + x]) : 0.f;
    Kh[i * QR + x] = live ? bf2f(k[((trow0 + i) * H + h) * K + x]) : 0.f;
  }
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
  __syncthreads();
  if (tid < 128) {  // norms: 2 threads per row (q for tid < 64, k otherwise)
    const int i = tid & 63;
    const float *row = (tid < 64 ? Qh : Kh) + i * QR;
    float s2 = 0.f;
    for (int x = 0; x < K; ++x) s2 = fmaf(row[x], row[x], s2);
    const float rn = l2 ? rsqrtf(s2 + GDN_L2_EPS) : 1.f;
    (tid < 64 ? rq : rk)[i] = rn;
  }
  __syncthreads();
  for (int e = tid; e < 64 * K; e += BT) {
    const int i = e / K, x = e % K;
    Qh[i * QR + x] *= rq[i];
    Kh[i * QR + x] *= rk[i];
  }
  if (tid < 64) {
    og[tid] = expf(gam[tid]);
    sv[tid] = expf(gam[63] - gam[tid]);
    dbv[tid] = 0.f;
    dgam[tid] = 0.f;
  }
  __syncthreads();
  // ---- KK = k^ k^T, QK = q^ k^T (full 64 x 64)
  for (int e = tid; e < 64 * 64; e += BT) {
    const int i = e >> 6, j = e & 63;
    float a = 0.f, b = 0.f;
    for (int x = 0; x < K; ++x) {
      a = fmaf(Kh[i * QR + x], Kh[j * QR + x], a);
      b = fmaf(Qh[i * QR + x], Kh[j * QR + x], b);
    }
    KK[i * M + j] = a;
    QK[i * M + j] = b;
  }
  __syncthreads();
  // ---- T = (I + A)^-1: column j by forward substitution (64 threads)
  if (tid < 64) {
    const int j = tid;
    for (int i = 0; i < 64; ++i) {
      float x = (i == j) ? 1.f : 0.f;
      if (i > j) {
        const float ci = bet[i];
        float s = 0.f;
        for (int m = j; m < i; ++m) s = fmaf(ci * expf(gam[i] - gam[m]) * KK[i * M + m], Tm[m * M + j], s);
        x = -s;
      }
      Tm[i * M + j] = (i >= j) ? x : 0.f;
    }
  }
  for (int e = tid; e < 64 * 64; e += BT) {
    const int i = e >> 6, j = e & 63;
    dT[i * M + j] = 0.f;
    dP[i * M + j] = 0.f;
  }
  float dQa[K / 4], dKa[K / 4];  // this thread's quarter of row ri of dq^, dk^
#pragma unroll
  for (int x = 0; x < K / 4; ++x) dQa[x] = dKa[x] = 0.f;
  float dgl = 0.f;  // this thread's part of d gamma_L
  __syncthreads();

  // ---- V slices
  for (int v0 = 0; v0 < V; v0 += VS) {
    const int64_t hb = ((int64_t)(slot * HV + hv) * K) * V + v0;
    for (int e = tid; e < K * VS; e += BT) {
      const int x = e / VS, cc = e % VS;
      hS[x * SR + cc] = Hs[hb + (int64_t)x * V + cc];
      dhS[x * SR + cc] = DH[hb + (int64_t)x * V + cc];
    }
    for (int e = tid; e < 64 * VS; e += BT) {
      const int i = e / VS, cc = e % VS;
      const bool live = i < L;
      vS[i * SR + cc] = live ? bf2f(v[((trow0 + i) * HV + hv) * V + v0 + cc]) : 0.f;
      doS[i * SR + cc] = live ? bf2f(dout[((trow0 + i) * HV + hv) * V + v0 + cc]) : 0.f;
    }
    __syncthreads();
    // k^ h, q^ h, k^ dh' (64 x VS): thread (ri, 4 columns)
    {
      float a[4] = {0, 0, 0, 0}, b[4] = {0, 0, 0, 0}, d[4] = {0, 0, 0, 0};
      for (int x = 0; x < K; ++x) {
        const float kv = Kh[ri * QR + x], qv = Qh[ri * QR + x];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float hv_ = hS[x * SR + qd * 4 + u], dv_ = dhS[x * SR + qd * 4 + u];
          a[u] = fmaf(kv, hv_, a[u]);
          b[u] = fmaf(qv, hv_, b[u]);
          d[u] = fmaf(kv, dv_, d[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        KhS[ri * SR + qd * 4 + u] = a[u];
        QhS[ri * SR + qd * 4 + u] = b[u];
        KdhS[ri * SR + qd * 4 + u] = d[u];
      }
    }
    __syncthreads();
    // v_new = T (diag(beta) V - diag(beta og) K^h);  dv_new = diag(sv) K^dh' + scale P^T do
    {
      float a[4] = {0, 0, 0, 0}, b[4] = {0, 0, 0, 0};
      for (int m = 0; m <= ri; ++m) {
        const float t = Tm[ri * M + m] * bet[m];
        const float tg = t * og[m];
#pragma unroll
        for (int u = 0; u < 4; ++u) a[u] = fmaf(t, vS[m * SR + qd * 4 + u], fmaf(-tg, KhS[m * SR + qd * 4 + u], a[u]));
      }
      for (int i = ri; i < 64; ++i) {
        const float p = expf(gam[i] - gam[ri]) * QK[i * M + ri];
#pragma unroll
        for (int u = 0; u < 4; ++u) b[u] = fmaf(p, doS[i * SR + qd * 4 + u], b[u]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        vnS[ri * SR + qd * 4 + u] = a[u];
        dvnS[ri * SR + qd * 4 + u] = fmaf(sv[ri], KdhS[ri * SR + qd * 4 + u], scale * b[u]);
      }
    }
    __syncthreads();
    // T^T dv_new; dv = diag(beta) T^T dv_new (output)
    {
      float a[4] = {0, 0, 0, 0};
      for (int m = ri; m < 64; ++m) {
        const float t = Tm[m * M + ri];
#pragma unroll
        for (int u = 0; u < 4; ++u) a[u] = fmaf(t, dvnS[m * SR + qd * 4 + u], a[u]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) TuS[ri * SR + qd * 4 + u] = a[u];
      if (ri < L) {
#pragma unroll
        for (int u = 0; u < 4; ++u) dv[((trow0 + ri) * HV + hv) * V + v0 + qd * 4 + u] = bet[ri] * a[u];
      }
    }
    __syncthreads();
    // dT += dv_new (diag(beta) V - diag(beta og) K^h)^T ;  dP += scale do v_new^T (j <= i)
    for (int e = tid; e < 64 * 64; e += BT) {
      const int i = e >> 6, j = e & 63;
      float a = 0.f, b = 0.f;
#pragma unroll
      for (int u = 0; u < VS; ++u) {
        a = fmaf(dvnS[i * SR + u], bet[j] * (vS[j * SR + u] - og[j] * KhS[j * SR + u]), a);
        b = fmaf(doS[i * SR + u], vnS[j * SR + u], b);
      }
      dT[i * M + j] += a;
      if (j <= i) dP[i * M + j] += scale * b;
    }
    // per-row sums (thread ri, columns of its quarter, reduced over the 4 threads of the row)
    {
      float sb = 0.f, sg = 0.f, sq = 0.f, sl = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int cc = qd * 4 + u;
        const float tu = TuS[ri * SR + cc], khv = KhS[ri * SR + cc];
        sb = fmaf(tu, vS[ri * SR + cc] - og[ri] * khv, sb);   // d beta
        sg = fmaf(tu, khv, sg);                                // -> d gamma (W term)
        sq = fmaf(QhS[ri * SR + cc], doS[ri * SR + cc], sq);   // og term
        sl = fmaf(KdhS[ri * SR + cc], vnS[ri * SR + cc], sl);  // state term
      }
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        sb += __shfl_xor_sync(0xffffffffu, sb, off);
        sg += __shfl_xor_sync(0xffffffffu, sg, off);
        sq += __shfl_xor_sync(0xffffffffu, sq, off);
        sl += __shfl_xor_sync(0xffffffffu, sl, off);
      }
      if (qd == 0) {
        dbv[ri] += sb;
        dgam[ri] += -bet[ri] * og[ri] * sg + scale * og[ri] * sq - sv[ri] * sl;
      }
      if (qd == 0) dgl += sv[ri] * sl;
    }
    // e^{gamma_L} <dh', h> for this slice
    {
      float s = 0.f;
      for (int e = tid; e < K * VS; e += BT) s = fmaf(dhS[(e / VS) * SR + e % VS], hS[(e / VS) * SR + e % VS], s);
      if (tid < 64) tmp[tid] = 0.f;
      s = warp_sum(s);
      __syncthreads();
      if (lane == 0) atomicAdd(&tmp[0], s);
      __syncthreads();
      if (tid == 0) dgl += og[63] * tmp[0];
    }
    // dk^ += -diag(beta og) T^T dv_new h^T + diag(sv) v_new dh'^T ;  dq^ += scale diag(og) do h^T
#pragma unroll
    for (int xq = 0; xq < K / 4; ++xq) {
      const int x = qd * (K / 4) + xq;
      float a = 0.f, b = 0.f, d = 0.f;
#pragma unroll
      for (int u = 0; u < VS; ++u) {
        a = fmaf(TuS[ri * SR + u], hS[x * SR + u], a);
        b = fmaf(vnS[ri * SR + u], dhS[x * SR + u], b);
        d = fmaf(doS[ri * SR + u], hS[x * SR + u], d);
      }
      dKa[xq] += -bet[ri] * og[ri] * a + sv[ri] * b;
      dQa[xq] += scale * og[ri] * d;
    }
    __syncthreads();
  }

  // ---- dA = -(T^T dT T^T), strictly lower.  X = dT T^T, then dA = -T^T X.
  for (int e = tid; e < 64 * 64; e += BT) {
    const int i = e >> 6, j = e & 63;
    float a = 0.f;
    for (int m = 0; m <= j; ++m) a = fmaf(dT[i * M + m], Tm[j * M + m], a);  // (T^T)_{mj} = T_{jm}, m <= j
    X[i * M + j] = a;
  }
  __syncthreads();
  for (int e = tid; e < 64 * 64; e += BT) {
    const int i = e >> 6, j = e & 63;
    float a = 0.f;
    if (j < i)
      for (int m = i; m < 64; ++m) a = fmaf(Tm[m * M + i], X[m * M + j], a);
    dT[i * M + j] = -a;  // dT now holds dA (zero outside j < i)
  }
  __syncthreads();
  // ---- from A_ij = beta_i e^{gamma_i-gamma_j} KK_ij (j < i) and P_ij = e^{gamma_i-gamma_j} QK_ij (j <= i)
  // row terms (thread ri): d beta_i, d gamma_i (+), dk^_i, dq^_i
  {
    float sb = 0.f, sgr = 0.f;
    for (int j = qd; j < 64; j += 4) {
      const float e = expf(gam[ri] - gam[j]);
      if (j < ri) {
        const float da = dT[ri * M + j];
        sb = fmaf(da, e * KK[ri * M + j], sb);
        sgr = fmaf(da, bet[ri] * e * KK[ri * M + j], sgr);
      }
      if (j <= ri) sgr = fmaf(dP[ri * M + j], e * QK[ri * M + j], sgr);
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      sb += __shfl_xor_sync(0xffffffffu, sb, off);
      sgr += __shfl_xor_sync(0xffffffffu, sgr, off);
    }
    if (qd == 0) {
      dbv[ri] += sb;
      dgam[ri] += sgr;
    }
  }
  __syncthreads();
  // column terms: d gamma_j (-)
  if (tid < 64) {
    const int j = tid;
    float s = 0.f;
    for (int i = j; i < 64; ++i) {
      const float e = expf(gam[i] - gam[j]);
      if (j < i) s = fmaf(dT[i * M + j], bet[i] * e * KK[i * M + j], s);
      s = fmaf(dP[i * M + j], e * QK[i * M + j], s);
    }
    dgam[j] -= s;
  }
  // dk^_i += sum_{j<i} dA_ij beta_i e_ij k^_j + sum_{m>i} dA_mi beta_m e_mi k^_m + sum_{m>=i} dP_mi e_mi q^_m
  // dq^_i += sum_{j<=i} dP_ij e_ij k^_j
  for (int j = 0; j < 64; ++j) {
    const float eij = expf(gam[ri] - gam[j]);
    const float cA = (j < ri) ? dT[ri * M + j] * bet[ri] * eij : 0.f;
    const float cP = (j <= ri) ? dP[ri * M + j] * eij : 0.f;
    const float eji = expf(gam[j] - gam[ri]);
    const float cA2 = (j > ri) ? dT[j * M + ri] * bet[j] * eji : 0.f;
    const float cP2 = (j >= ri) ? dP[j * M + ri] * eji : 0.f;
#pragma unroll
    for (int xq = 0; xq < K / 4; ++xq) {
      const int x = qd * (K / 4) + xq;
      dKa[xq] = fmaf(cA, Kh[j * QR + x], fmaf(cA2, Kh[j * QR + x], fmaf(cP2, Qh[j * QR + x], dKa[xq])));
      dQa[xq] = fmaf(cP, Kh[j * QR + x], dQa[xq]);
    }
  }
  __syncthreads();
  // ---- d gamma_L, then dg = reverse cumsum of d gamma over the chunk
  dgl = warp_sum(dgl);
  if (tid < 64) tmp[tid] = 0.f;
  __syncthreads();
  if (lane == 0) atomicAdd(&tmp[0], dgl);
  __syncthreads();
  if (tid == 0) dgam[63] += tmp[0];
  __syncthreads();
  if (warp == 0) {
    // reverse inclusive scan over 64 rows, two per lane
    const float x0 = dgam[2 * lane], x1 = dgam[2 * lane + 1];
    float s = x0 + x1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_down_sync(0xffffffffu, s, off);
      if (lane + off < 32) s += y;
    }
    const float r1 = s - x0;  // sum over rows >= 2 lane + 1
    if (2 * lane < L) {
      dg[(trow0 + 2 * lane) * HV + hv] = s;
      dbeta[(trow0 + 2 * lane) * HV + hv] = dbv[2 * lane];
    }
    if (2 * lane + 1 < L) {
      dg[(trow0 + 2 * lane + 1) * HV + hv] = r1;
      dbeta[(trow0 + 2 * lane + 1) * HV + hv] = dbv[2 * lane + 1];
    }
  }
  // ---- through the L2 norms: dx = r (dx^ - x^ (x^ . dx^)); summed over the group's value heads
  {
    float pq = 0.f, pk = 0.f;
#pragma unroll
    for (int xq = 0; xq < K / 4; ++xq) {
      const int x = qd * (K / 4) + xq;
      pq = fmaf(Qh[ri * QR + x], dQa[xq], pq);
      pk = fmaf(Kh[ri * QR + x], dKa[xq], pk);
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      pq += __shfl_xor_sync(0xffffffffu, pq, off);
      pk += __shfl_xor_sync(0xffffffffu, pk, off);
    }
    if (ri < L) {
      float *dqr = dq + ((trow0 + ri) * H + h) * K + qd * (K / 4);
      float *dkr = dk + ((trow0 + ri) * H + h) * K + qd * (K / 4);
#pragma unroll
      for (int xq = 0; xq < K / 4; ++xq) {
        const int x = qd * (K / 4) + xq;
        const float gq = l2 ? rq[ri] * (dQa[xq] - Qh[ri * QR + x] * pq) : dQa[xq];
        const float gk = l2 ? rk[ri] * (dKa[xq] - Kh[ri * QR + x] * pk) : dKa[xq];
        atomicAdd(dqr + xq, gq);
        atomicAdd(dkr + xq, gk);
      }
    }
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
  const int64_t rows = (int64_t)a.B * a.T;
  cudaError_t e;
  if (rows > 0) {
    e = cudaMemsetAsync(a.dq, 0, (size_t)rows * a.H * K * sizeof(float), s);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(a.dk, 0, (size_t)rows * a.H * K * sizeof(float), s);
    if (e != cudaSuccess) return e;
  }
  // 1. forward again, saving the state entering every chunk (no output needed)
  gdn_host::ChunkArgs f{};
  f.q = a.q; f.k = a.k; f.v = a.v; f.g = a.g; f.beta = a.beta; f.scale = a.scale; f.h0 = a.h0; f.cu = a.cu;
  f.N = a.N; f.B = a.B; f.T = a.T; f.H = a.H; f.HV = a.HV; f.K = K; f.V = a.V; f.l2 = a.l2;
  f.o = nullptr; f.ht = nullptr; f.hsave = Hs; f.ws = a.ws; f.ws_bytes = rec_bytes; f.dev_status = a.dev_status;
  e = gdn_host::launch_chunk(f, s);
  if (e != cudaSuccess) return e;
  // 2. state gradients, last chunk first
  {
    const int smem = DhLay<K>::BYTES;
    e = cudaFuncSetAttribute(chunk_dh_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    chunk_dh_kernel<K><<<dim3(a.V / 32, a.HV, a.N), BT, smem, s>>>(
        a.q, a.k, a.dout, static_cast<const unsigned char *>(a.ws), DH, a.dht, a.dh0, a.scale, a.cu, a.T, a.H,
        a.HV, a.V, a.dev_status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // 3. per-chunk gradients
  if (rows > 0 && slots > 0) {
    const int smem = GradLay<K>::BYTES;
    e = cudaFuncSetAttribute(chunk_grad_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    chunk_grad_kernel<K><<<dim3((unsigned)slots, a.HV), BT, smem, s>>>(
        a.q, a.k, a.v, a.g, a.beta, a.dout, Hs, DH, a.scale, a.cu, a.N, a.T, a.H, a.HV, a.V, a.l2, a.dq, a.dk,
        a.dv, a.dg, a.dbeta, a.dev_status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

namespace gdn_host {

size_t chunk_bwd_workspace_bytes(int B, int T, int H, int HV, int K, int V, int N, int varlen) {
  const size_t rec = chunk_workspace_bytes(B, T, H, HV, K, V, N, varlen);
  const size_t st = (size_t)total_chunk_slots(B, T, N, varlen != 0) * HV * K * V * sizeof(float);
  return rec + 2 * st;
}

cudaError_t launch_chunk_bwd(const ChunkBwdArgs &a, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  if (a.K == 128) return launch_bwd_k<128>(a, s);
  if (a.K == 64) return launch_bwd_k<64>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace gdn_host
