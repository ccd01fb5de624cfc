// gdn_decode.cu -- pool-indexed one-token decode with optional fused gating.
//
// FastDeploy PR "support fla triton kernel for qwen3.5", Usage section 2
// ("Decode (fused recurrent, pool-index)"): the state pool [P, HV, K, V] is
// read and written in place through per-request slot indices, PAD_SLOT_ID = -1
// is skipped.  The LightLLM "gdn.py" decode path hands A_log, dt_bias and the
// raw a, b to the same kernel, so the gates are computed in-kernel.
//
// Design: the op moves 2 x K x V x 4 bytes of state per (request, value head)
// and does ~6 K V flops on it, so it is HBM-bound.  One 256-thread block owns
// one (value head, request) state.  Lane l holds V/32 consecutive columns of
// K/8 rows (warp w owns rows [w K/8, (w+1) K/8)), so every warp-wide load or
// store is one contiguous 512-byte (V = 128) row segment, issued as 16-byte
// streaming loads all at once before any arithmetic.  The two reductions over
// K (S^T k and S^T q) go through shared memory across the 8 warps.  The
// updated state is written back with streaming stores.
#include "gdn_common.cuh"

namespace {

constexpr int kWarps = 8;

template <int N> struct VecF;
template <> struct VecF<4> { using T = float4; };
template <> struct VecF<2> { using T = float2; };

__device__ __forceinline__ void unpack(const float4 &x, float *o) { o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w; }
__device__ __forceinline__ void unpack(const float2 &x, float *o) { o[0] = x.x; o[1] = x.y; }
__device__ __forceinline__ float4 pack4(const float *o) { return make_float4(o[0], o[1], o[2], o[3]); }
__device__ __forceinline__ float2 pack2(const float *o) { return make_float2(o[0], o[1]); }
template <int N> __device__ __forceinline__ typename VecF<N>::T packv(const float *o);
template <> __device__ __forceinline__ float4 packv<4>(const float *o) { return pack4(o); }
template <> __device__ __forceinline__ float2 packv<2>(const float *o) { return pack2(o); }

// State storage: fp32, or bf16 (the step runs in fp32 on the stored values;
// the new state is rounded to bf16 when stored).
template <typename ST, int N> struct StateIO;
template <int N> struct StateIO<float, N> {
  static __device__ __forceinline__ void load(const float *p, float *o) {
    unpack(__ldcs(reinterpret_cast<const typename VecF<N>::T *>(p)), o);
  }
  static __device__ __forceinline__ void store(float *p, const float *o) {
    __stcs(reinterpret_cast<typename VecF<N>::T *>(p), packv<N>(o));
  }
};
template <> struct StateIO<uint16_t, 4> {
  static __device__ __forceinline__ void load(const uint16_t *p, float *o) {
    const uint2 u = __ldcs(reinterpret_cast<const uint2 *>(p));
    o[0] = gdn::bf2f((uint16_t)(u.x & 0xffff)); o[1] = gdn::bf2f((uint16_t)(u.x >> 16));
    o[2] = gdn::bf2f((uint16_t)(u.y & 0xffff)); o[3] = gdn::bf2f((uint16_t)(u.y >> 16));
  }
  static __device__ __forceinline__ void store(uint16_t *p, const float *o) {
    const uint2 u = make_uint2((uint32_t)gdn::f2bf(o[0]) | ((uint32_t)gdn::f2bf(o[1]) << 16),
                               (uint32_t)gdn::f2bf(o[2]) | ((uint32_t)gdn::f2bf(o[3]) << 16));
    __stcs(reinterpret_cast<uint2 *>(p), u);
  }
};
template <> struct StateIO<uint16_t, 2> {
  static __device__ __forceinline__ void load(const uint16_t *p, float *o) {
    const uint32_t u = __ldcs(reinterpret_cast<const unsigned int *>(p));
    o[0] = gdn::bf2f((uint16_t)(u & 0xffff)); o[1] = gdn::bf2f((uint16_t)(u >> 16));
  }
  static __device__ __forceinline__ void store(uint16_t *p, const float *o) {
    __stcs(reinterpret_cast<unsigned int *>(p), (uint32_t)gdn::f2bf(o[0]) | ((uint32_t)gdn::f2bf(o[1]) << 16));
  }
};

// One block per (value head, request).  A request owns tokens [t0, t1)
// (t0 = n, t1 = n + 1 without cu); it starts from
// pool[read_idx[n * ld + num_acc[n] - 1]] (column 0 without num_acc) and
// stores the state after its i-th token into pool[write_idx[n * ld + i]]
// (-1: not stored).  The state stays in registers across the tokens.
template <int K, int V, typename ST>
__global__ void __launch_bounds__(kWarps * 32, 2) decode_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ k,
    const uint16_t *__restrict__ v, const float *__restrict__ g_in,
    const float *__restrict__ beta_in, const float *__restrict__ A_log,
    const uint16_t *__restrict__ a_raw, const uint16_t *__restrict__ b_raw,
    const float *__restrict__ dt_bias, float scale, int l2, ST *pool, int P,
    const int32_t *__restrict__ cu, int Ttot, const int32_t *__restrict__ read_idx,
    const int32_t *__restrict__ write_idx, int ld, const int32_t *__restrict__ num_acc,
    int H, int HV, uint16_t *__restrict__ o, int32_t *dev_status) {
  constexpr int VPL = V / 32;        // columns per lane
  constexpr int RPW = K / kWarps;    // rows per warp

  __shared__ float qn[K], kn[K];
  __shared__ float red[2][kWarps][V];
  __shared__ float sh_norm[2];

  const int hv = blockIdx.x, n = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  int t0 = n, t1 = n + 1;
  if (cu) {
    t0 = cu[n];
    t1 = cu[n + 1];
    if (t0 < 0 || t1 < t0 || t1 > Ttot || t1 - t0 > ld) {
      if (tid == 0) gdn::set_status(dev_status, GDN_DEV_BAD_CU_SEQLENS);
      return;
    }
  }
  const int acc = num_acc ? num_acc[n] : 1;
  int s = -1;
  if (acc >= 1 && acc <= ld) {
    s = read_idx[(int64_t)n * ld + acc - 1];
  } else if (tid == 0) {
    gdn::set_status(dev_status, GDN_DEV_BAD_SLOT);
  }
  if (s < 0 || s >= P) {
    if (s != -1 && tid == 0) gdn::set_status(dev_status, GDN_DEV_BAD_SLOT);
    for (int t = t0; t < t1; ++t)
      for (int j = tid; j < V; j += blockDim.x) o[((int64_t)t * HV + hv) * V + j] = 0;
    return;
  }
  const int h = hv / (HV / H);

  // Issue every state load before any other work.
  float Sf[RPW][VPL];
  {
    const ST *S = pool + ((int64_t)s * HV + hv) * (int64_t)K * V;
#pragma unroll
    for (int i = 0; i < RPW; ++i) StateIO<ST, VPL>::load(S + (int64_t)(w * RPW + i) * V + lane * VPL, Sf[i]);
  }

  for (int t = t0; t < t1; ++t) {
    if (t > t0) __syncthreads();  // the previous token's readers of the shared buffers are done
    // q, k rows and their norms.
    const uint16_t *qr = q + ((int64_t)t * H + h) * K;
    const uint16_t *kr = k + ((int64_t)t * H + h) * K;
    float qx = 0.f, kx = 0.f;
    if (tid < K) { qx = gdn::bf2f(qr[tid]); kx = gdn::bf2f(kr[tid]); }
    if (l2) {
      float qs = gdn::warp_sum(qx * qx), ks = gdn::warp_sum(kx * kx);
      if (lane == 0 && w < K / 32) { red[0][w][0] = qs; red[1][w][0] = ks; }
      __syncthreads();
      if (tid == 0) {
        float a0 = 0.f, b0 = 0.f;
        for (int i = 0; i < K / 32; ++i) { a0 += red[0][i][0]; b0 += red[1][i][0]; }
        sh_norm[0] = rsqrtf(a0 + GDN_L2_EPS);
        sh_norm[1] = rsqrtf(b0 + GDN_L2_EPS);
      }
      __syncthreads();
      if (tid < K) { qn[tid] = qx * sh_norm[0]; kn[tid] = kx * sh_norm[1]; }
    } else if (tid < K) {
      qn[tid] = qx;
      kn[tid] = kx;
    }

    // Gates.
    float gg, bb;
    const int64_t gi = (int64_t)t * HV + hv;
    if (g_in) {
      gg = g_in[gi];
      bb = beta_in[gi];
    } else {
      gg = -expf(A_log[hv]) * gdn::softplus_f(gdn::bf2f(a_raw[gi]) + dt_bias[hv]);
      bb = gdn::sigmoid_f(gdn::bf2f(b_raw[gi]));
    }
    const float decay = expf(gg);

    // Value columns of this lane.
    float vv[VPL];
    const uint16_t *vr = v + ((int64_t)t * HV + hv) * V + lane * VPL;
#pragma unroll
    for (int c = 0; c < VPL; ++c) vv[c] = gdn::bf2f(vr[c]);
    __syncthreads();  // qn / kn visible; red reusable

    // r = S^T k (partial over this warp's rows).
    float part[VPL];
#pragma unroll
    for (int c = 0; c < VPL; ++c) part[c] = 0.f;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const float kk = kn[w * RPW + i];
#pragma unroll
      for (int c = 0; c < VPL; ++c) part[c] = fmaf(Sf[i][c], kk, part[c]);
    }
#pragma unroll
    for (int c = 0; c < VPL; ++c) red[0][w][lane * VPL + c] = part[c];
    __syncthreads();
    float delta[VPL];
#pragma unroll
    for (int c = 0; c < VPL; ++c) {
      float rs = 0.f;
#pragma unroll
      for (int j = 0; j < kWarps; ++j) rs += red[0][j][lane * VPL + c];
      delta[c] = bb * (vv[c] - decay * rs);
    }

    // S <- a S + k delta^T, then o partial = S^T q.
#pragma unroll
    for (int c = 0; c < VPL; ++c) part[c] = 0.f;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const float kk = kn[w * RPW + i], qq = qn[w * RPW + i];
#pragma unroll
      for (int c = 0; c < VPL; ++c) {
        Sf[i][c] = fmaf(decay, Sf[i][c], kk * delta[c]);
        part[c] = fmaf(Sf[i][c], qq, part[c]);
      }
    }
    const int ws = write_idx[(int64_t)n * ld + (t - t0)];
    if (ws >= 0 && ws < P) {
      ST *D = pool + ((int64_t)ws * HV + hv) * (int64_t)K * V;
#pragma unroll
      for (int i = 0; i < RPW; ++i) StateIO<ST, VPL>::store(D + (int64_t)(w * RPW + i) * V + lane * VPL, Sf[i]);
    } else if (ws != -1 && tid == 0) {
      gdn::set_status(dev_status, GDN_DEV_BAD_SLOT);
    }
#pragma unroll
    for (int c = 0; c < VPL; ++c) red[1][w][lane * VPL + c] = part[c];
    __syncthreads();
    if (w == 0) {
      uint16_t *orow = o + ((int64_t)t * HV + hv) * V;
#pragma unroll
      for (int c = 0; c < VPL; ++c) {
        float os = 0.f;
#pragma unroll
        for (int j = 0; j < kWarps; ++j) os += red[1][j][lane * VPL + c];
        orow[lane * VPL + c] = gdn::f2bf(scale * os);
      }
    }
  }
}

template <int K, int V, typename ST>
cudaError_t launch_kv(const gdn_host::DecodeArgs &a, ST *pool, cudaStream_t s) {
  dim3 grid(a.HV, a.N);
  decode_kernel<K, V, ST><<<grid, kWarps * 32, 0, s>>>(
      a.q, a.k, a.v, a.g, a.beta, a.A_log, a.a, a.b, a.dt_bias, a.scale, a.l2, pool, a.P, a.cu, a.Ttot,
      a.read_idx, a.write_idx, a.ld, a.num_acc, a.H, a.HV, a.o, a.dev_status);
  return cudaGetLastError();
}

template <typename ST>
cudaError_t launch_any(const gdn_host::DecodeArgs &a, ST *pool, cudaStream_t s) {
#define GDN_DEC(KK, VV) \
  if (a.K == KK && a.V == VV) return launch_kv<KK, VV, ST>(a, pool, s);
  GDN_DEC(128, 128)
  GDN_DEC(64, 64)
  GDN_DEC(64, 128)
  GDN_DEC(128, 64)
#undef GDN_DEC
  return cudaErrorInvalidValue;
}

}  // namespace

namespace gdn_host {

cudaError_t launch_decode_general(const DecodeArgs &a, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  if (a.pool_bf16) return launch_any<uint16_t>(a, static_cast<uint16_t *>(a.pool), s);
  return launch_any<float>(a, static_cast<float *>(a.pool), s);
}

}  // namespace gdn_host
