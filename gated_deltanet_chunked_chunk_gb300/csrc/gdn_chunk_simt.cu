// gdn_chunk_simt.cu -- chunked WY prefill on CUDA cores, fp32 throughout.
//
// The six steps of "NPU Training Operators - GDN", section "Operator
// semantics", for chunk size 64, one block per (value-head column tile of 32,
// value head, sequence).  The block walks the chunks of its sequence in order
// with its K x 32 slice of the state in shared memory:
//
//   gamma = chunk-local cumsum of g
//   A_ij  = beta_i e^{gamma_i - gamma_j} k_i.k_j  (i > j)      (KK^T with decay)
//   Tm    = (I + A)^{-1}                          (forward substitution)
//   w     = Tm diag(beta e^gamma) K,  u = Tm diag(beta) V     (WY recompute)
//   v_new = u - w h
//   o     = scale (diag(e^gamma) Q h + (Q K^T * causal decay) v_new)
//   h     = e^{gamma_last} h + K^T diag(e^{gamma_last - gamma}) v_new
//
// This kernel is the straightforward fp32 form of the algorithm; it keeps the
// library correct for every supported shape and is the yardstick for the
// tensor-core kernel.
#include "gdn_common.cuh"

namespace {

constexpr int C = GDN_CHUNK;
constexpr int VT = 32;       // value columns per block
constexpr int NT = 256;      // threads per block

template <int K>
struct Smem {
  float kn[C][K + 1];
  float qn[C][K + 1];
  float w[C][K + 1];
  float A[C][C + 1];     // A, then P = causal(decay * Q K^T)
  float Tm[C][C + 1];
  float h[K][VT + 1];
  float vt[C][VT + 1];
  float u[C][VT + 1];
  float vn[C][VT + 1];
  float gam[C], bet[C], egam[C];
};

template <int K, int V>
__global__ void __launch_bounds__(NT) chunk_simt_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ k,
    const uint16_t *__restrict__ v, const float *__restrict__ g,
    const float *__restrict__ beta, float scale, const float *__restrict__ h0,
    const int32_t *__restrict__ cu, int T, int H, int HV, int l2,
    uint16_t *__restrict__ o, float *__restrict__ ht, int32_t *dev_status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem<K> &sm = *reinterpret_cast<Smem<K> *>(smem_raw);
  const int vt0 = blockIdx.x * VT, hv = blockIdx.y, n = blockIdx.z;
  const int h = hv / (HV / H);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  int64_t tok0, len;
  if (cu) {
    const int32_t a0 = cu[n], a1 = cu[n + 1];
    if (a0 < 0 || a1 < a0 || a1 > T || (n == 0 && a0 != 0)) {
      if (tid == 0) gdn::set_status(dev_status, GDN_DEV_BAD_CU_SEQLENS);
      return;
    }
    tok0 = a0;
    len = a1 - a0;
  } else {
    tok0 = (int64_t)n * T;
    len = T;
  }

  // State slice h[:, vt0:vt0+32].
  for (int e = tid; e < K * VT; e += NT) {
    const int r = e / VT, c = e % VT;
    sm.h[r][c] = h0 ? h0[((int64_t)(n * HV + hv) * K + r) * V + vt0 + c] : 0.f;
  }

  for (int64_t c0 = 0; c0 < len; c0 += C) {
    const int L = (int)(len - c0 < C ? len - c0 : C);
    __syncthreads();
    // 1. Load q, k (key head h), the value tile, g and beta; rows >= L are zero.
    for (int e = tid; e < C * K; e += NT) {
      const int i = e / K, c = e % K;
      float kx = 0.f, qx = 0.f;
      if (i < L) {
        const int64_t off = ((tok0 + c0 + i) * H + h) * K + c;
        kx = gdn::bf2f(k[off]);
        qx = gdn::bf2f(q[off]);
      }
      sm.kn[i][c] = kx;
      sm.qn[i][c] = qx;
    }
    for (int e = tid; e < C * VT; e += NT) {
      const int i = e / VT, c = e % VT;
      sm.vt[i][c] = i < L ? gdn::bf2f(v[((tok0 + c0 + i) * HV + hv) * V + vt0 + c]) : 0.f;
    }
    if (tid < C) {
      const bool ok = tid < L;
      sm.gam[tid] = ok ? g[(tok0 + c0 + tid) * HV + hv] : 0.f;
      sm.bet[tid] = ok ? beta[(tok0 + c0 + tid) * HV + hv] : 0.f;
    }
    __syncthreads();
    // 2. Row norms (one warp per row) and the chunk-local cumsum of g.
    if (l2) {
      for (int i = warp; i < C; i += NT / 32) {
        float sk = 0.f, sq = 0.f;
        for (int c = lane; c < K; c += 32) {
          sk += sm.kn[i][c] * sm.kn[i][c];
          sq += sm.qn[i][c] * sm.qn[i][c];
        }
        sk = rsqrtf(gdn::warp_sum(sk) + GDN_L2_EPS);
        sq = rsqrtf(gdn::warp_sum(sq) + GDN_L2_EPS);
        for (int c = lane; c < K; c += 32) {
          sm.kn[i][c] *= sk;
          sm.qn[i][c] *= sq;
        }
      }
    }
    if (tid == 0) {
      float acc = 0.f;
      for (int i = 0; i < C; ++i) {
        acc += sm.gam[i];
        sm.gam[i] = acc;
        sm.egam[i] = expf(acc);
      }
    }
    __syncthreads();
    // 3. A = strictly-lower beta_i e^{gamma_i - gamma_j} k_i.k_j
    for (int e = tid; e < C * C; e += NT) {
      const int i = e / C, j = e % C;
      float val = 0.f;
      if (j < i) {
        float d = 0.f;
        for (int c = 0; c < K; ++c) d = fmaf(sm.kn[i][c], sm.kn[j][c], d);
        val = sm.bet[i] * expf(sm.gam[i] - sm.gam[j]) * d;
      }
      sm.A[i][j] = val;
    }
    __syncthreads();
    // 4. Tm = (I + A)^{-1}: column c by forward substitution in one thread.
    if (tid < C) {
      const int c = tid;
      for (int i = 0; i < C; ++i) {
        float x = (i == c) ? 1.f : 0.f;
        for (int j = c; j < i; ++j) x = fmaf(-sm.A[i][j], sm.Tm[j][c], x);
        sm.Tm[i][c] = (i < c) ? 0.f : x;
      }
    }
    __syncthreads();
    // 5. P = causal(e^{gamma_i - gamma_j} q_i.k_j) into A; w and u.
    for (int e = tid; e < C * C; e += NT) {
      const int i = e / C, j = e % C;
      float val = 0.f;
      if (j <= i) {
        float d = 0.f;
        for (int c = 0; c < K; ++c) d = fmaf(sm.qn[i][c], sm.kn[j][c], d);
        val = expf(sm.gam[i] - sm.gam[j]) * d;
      }
      sm.A[i][j] = val;
    }
    for (int e = tid; e < C * K; e += NT) {
      const int i = e / K, c = e % K;
      float acc = 0.f;
      for (int j = 0; j <= i; ++j) acc = fmaf(sm.Tm[i][j] * sm.bet[j] * sm.egam[j], sm.kn[j][c], acc);
      sm.w[i][c] = acc;
    }
    for (int e = tid; e < C * VT; e += NT) {
      const int i = e / VT, c = e % VT;
      float acc = 0.f;
      for (int j = 0; j <= i; ++j) acc = fmaf(sm.Tm[i][j] * sm.bet[j], sm.vt[j][c], acc);
      sm.u[i][c] = acc;
    }
    __syncthreads();
    // 6. v_new = u - w h
    for (int e = tid; e < C * VT; e += NT) {
      const int i = e / VT, c = e % VT;
      float acc = sm.u[i][c];
      for (int r = 0; r < K; ++r) acc = fmaf(-sm.w[i][r], sm.h[r][c], acc);
      sm.vn[i][c] = acc;
    }
    __syncthreads();
    // 7. o = scale (e^gamma Q h + P v_new)
    for (int e = tid; e < C * VT; e += NT) {
      const int i = e / VT, c = e % VT;
      if (i >= L) continue;
      float inter = 0.f, intra = 0.f;
      for (int r = 0; r < K; ++r) inter = fmaf(sm.qn[i][r], sm.h[r][c], inter);
      for (int j = 0; j <= i; ++j) intra = fmaf(sm.A[i][j], sm.vn[j][c], intra);
      const float ov = scale * (sm.egam[i] * inter + intra);
      o[((tok0 + c0 + i) * HV + hv) * V + vt0 + c] = gdn::f2bf(ov);
    }
    __syncthreads();
    // 8. h = e^{gamma_last} h + K^T diag(e^{gamma_last - gamma}) v_new
    {
      const float gl = sm.gam[C - 1];
      for (int e = tid; e < K * VT; e += NT) {
        const int r = e / VT, c = e % VT;
        float acc = sm.egam[C - 1] * sm.h[r][c];
        for (int j = 0; j < L; ++j) acc = fmaf(sm.kn[j][r] * expf(gl - sm.gam[j]), sm.vn[j][c], acc);
        sm.h[r][c] = acc;
      }
    }
  }
  __syncthreads();
  if (ht) {
    for (int e = tid; e < K * VT; e += NT) {
      const int r = e / VT, c = e % VT;
      ht[((int64_t)(n * HV + hv) * K + r) * V + vt0 + c] = sm.h[r][c];
    }
  }
}

template <int K, int V>
cudaError_t launch_kv(const gdn_host::ChunkArgs &a, cudaStream_t s) {
  const size_t smem = sizeof(Smem<K>);
  cudaError_t e = cudaFuncSetAttribute(chunk_simt_kernel<K, V>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(V / VT, a.HV, a.N);
  chunk_simt_kernel<K, V><<<grid, NT, smem, s>>>(a.q, a.k, a.v, a.g, a.beta, a.scale, a.h0,
                                                 a.cu, a.T, a.H, a.HV, a.l2, a.o, a.ht,
                                                 a.dev_status);
  return cudaGetLastError();
}

}  // namespace

namespace gdn_host {

size_t chunk_workspace_bytes(int, int, int, int, int, int, int, int) { return 0; }

cudaError_t launch_chunk(const ChunkArgs &a, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  if (a.K == 128 && a.V == 128) return launch_kv<128, 128>(a, s);
  if (a.K == 64 && a.V == 64) return launch_kv<64, 64>(a, s);
  if (a.K == 64 && a.V == 128) return launch_kv<64, 128>(a, s);
  if (a.K == 128 && a.V == 64) return launch_kv<128, 64>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace gdn_host
