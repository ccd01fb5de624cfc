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

template <int K, int V>
__global__ void __launch_bounds__(kWarps * 32, 2) decode_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ k,
    const uint16_t *__restrict__ v, const float *__restrict__ g_in,
    const float *__restrict__ beta_in, const float *__restrict__ A_log,
    const uint16_t *__restrict__ a_raw, const uint16_t *__restrict__ b_raw,
    const float *__restrict__ dt_bias, float scale, int l2, float *pool, int P,
    const int32_t *__restrict__ idx, int H, int HV, uint16_t *__restrict__ o,
    int32_t *dev_status) {
  constexpr int VPL = V / 32;        // columns per lane
  constexpr int RPW = K / kWarps;    // rows per warp
  using VT = typename VecF<VPL>::T;

  __shared__ float qn[K], kn[K];
  __shared__ float red[2][kWarps][V];
  __shared__ float sh_norm[2];

  const int hv = blockIdx.x, r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int s = idx[r];
  uint16_t *orow = o + ((int64_t)r * HV + hv) * V;
  if (s < 0 || s >= P) {
    if (s != -1 && tid == 0) gdn::set_status(dev_status, GDN_DEV_BAD_SLOT);
    for (int j = tid; j < V; j += blockDim.x) orow[j] = 0;
    return;
  }
  const int h = hv / (HV / H);

  // Issue every state load before any other work.
  float *S = pool + ((int64_t)s * HV + hv) * (int64_t)K * V;
  VT Sv[RPW];
#pragma unroll
  for (int i = 0; i < RPW; ++i)
    Sv[i] = __ldcs(reinterpret_cast<const VT *>(S + (int64_t)(w * RPW + i) * V) + lane);

  // q, k rows and their norms.
  const uint16_t *qr = q + ((int64_t)r * H + h) * K;
  const uint16_t *kr = k + ((int64_t)r * H + h) * K;
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
  const int64_t gi = (int64_t)r * HV + hv;
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
  const uint16_t *vr = v + ((int64_t)r * HV + hv) * V + lane * VPL;
#pragma unroll
  for (int c = 0; c < VPL; ++c) vv[c] = gdn::bf2f(vr[c]);
  __syncthreads();  // qn / kn visible; red reusable

  // r = S^T k (partial over this warp's rows).
  float Sf[RPW][VPL];
#pragma unroll
  for (int i = 0; i < RPW; ++i) unpack(Sv[i], Sf[i]);
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
#pragma unroll
  for (int i = 0; i < RPW; ++i)
    __stcs(reinterpret_cast<VT *>(S + (int64_t)(w * RPW + i) * V) + lane, packv<VPL>(Sf[i]));
#pragma unroll
  for (int c = 0; c < VPL; ++c) red[1][w][lane * VPL + c] = part[c];
  __syncthreads();
  if (w == 0) {
#pragma unroll
    for (int c = 0; c < VPL; ++c) {
      float os = 0.f;
#pragma unroll
      for (int j = 0; j < kWarps; ++j) os += red[1][j][lane * VPL + c];
      orow[lane * VPL + c] = gdn::f2bf(scale * os);
    }
  }
}

template <int K, int V>
cudaError_t launch_kv(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const float *g, const float *beta, const float *A_log,
                      const uint16_t *a, const uint16_t *b,
                      const float *dt_bias, float scale, int l2, float *pool,
                      int P, const int32_t *idx, int R, int H, int HV,
                      uint16_t *o, int32_t *st, cudaStream_t s) {
  dim3 grid(HV, R);
  decode_kernel<K, V><<<grid, kWarps * 32, 0, s>>>(q, k, v, g, beta, A_log, a, b, dt_bias,
                                                   scale, l2, pool, P, idx, H, HV, o, st);
  return cudaGetLastError();
}

}  // namespace

namespace gdn_host {

cudaError_t launch_decode(const uint16_t *q, const uint16_t *k,
                          const uint16_t *v, const float *g, const float *beta,
                          const float *A_log, const uint16_t *a,
                          const uint16_t *b, const float *dt_bias, float scale,
                          int l2, float *pool, int P, const int32_t *idx, int R,
                          int H, int HV, int K, int V, uint16_t *o,
                          int32_t *st, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
#define GDN_DEC(KK, VV)                                                          \
  if (K == KK && V == VV)                                                        \
    return launch_kv<KK, VV>(q, k, v, g, beta, A_log, a, b, dt_bias, scale, l2, \
                             pool, P, idx, R, H, HV, o, st, s);
  GDN_DEC(128, 128)
  GDN_DEC(64, 64)
  GDN_DEC(64, 128)
  GDN_DEC(128, 64)
#undef GDN_DEC
  return cudaErrorInvalidValue;
}

}  // namespace gdn_host
