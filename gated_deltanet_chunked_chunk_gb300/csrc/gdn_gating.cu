// gdn_gating.cu -- fused gate kernel.
//
// FastDeploy PR "support fla triton kernel for qwen3.5", Usage section 5
// ("Fused GDN Gating"): g = -exp(A_log) * softplus(a + dt_bias) and
// beta = sigmoid(b), both fp32, in one launch.
//
// The op is elementwise and HBM-bound (4 bytes in, 8 bytes out per element).
// Each thread handles 4 consecutive elements of the flattened [Ttok, HV]
// array: one 8-byte load each of a and b, one 16-byte store each of g and
// beta.  The grid is a multiple of the SM count and strides over the array.
#include "gdn_common.cuh"

namespace {

__global__ void __launch_bounds__(256) gating_kernel(
    const float *__restrict__ A_log, const uint16_t *__restrict__ a,
    const uint16_t *__restrict__ b, const float *__restrict__ dt_bias,
    int64_t n_elem, int HV, float *__restrict__ g, float *__restrict__ beta) {
  const int64_t n4 = n_elem / 4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 7) == 0 &&
                      ((reinterpret_cast<uintptr_t>(g) | reinterpret_cast<uintptr_t>(beta)) & 15) == 0;
  int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (vec_ok) {
    for (int64_t i = i0; i < n4; i += stride) {
      uint2 av = __ldcs(reinterpret_cast<const uint2 *>(a) + i);
      uint2 bv = __ldcs(reinterpret_cast<const uint2 *>(b) + i);
      uint16_t as[4] = {(uint16_t)(av.x & 0xffff), (uint16_t)(av.x >> 16),
                        (uint16_t)(av.y & 0xffff), (uint16_t)(av.y >> 16)};
      uint16_t bs[4] = {(uint16_t)(bv.x & 0xffff), (uint16_t)(bv.x >> 16),
                        (uint16_t)(bv.y & 0xffff), (uint16_t)(bv.y >> 16)};
      float go[4], bo[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        int h = (int)((i * 4 + j) % HV);
        go[j] = -expf(__ldg(A_log + h)) * gdn::softplus_f(gdn::bf2f(as[j]) + __ldg(dt_bias + h));
        bo[j] = gdn::sigmoid_f(gdn::bf2f(bs[j]));
      }
      __stcs(reinterpret_cast<float4 *>(g) + i, make_float4(go[0], go[1], go[2], go[3]));
      __stcs(reinterpret_cast<float4 *>(beta) + i, make_float4(bo[0], bo[1], bo[2], bo[3]));
    }
    for (int64_t i = n4 * 4 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_elem; i += stride) {
      int h = (int)(i % HV);
      g[i] = -expf(A_log[h]) * gdn::softplus_f(gdn::bf2f(a[i]) + dt_bias[h]);
      beta[i] = gdn::sigmoid_f(gdn::bf2f(b[i]));
    }
  } else {
    for (int64_t i = i0; i < n_elem; i += stride) {
      int h = (int)(i % HV);
      g[i] = -expf(A_log[h]) * gdn::softplus_f(gdn::bf2f(a[i]) + dt_bias[h]);
      beta[i] = gdn::sigmoid_f(gdn::bf2f(b[i]));
    }
  }
}

}  // namespace

namespace gdn_host {

cudaError_t launch_gating(const float *A_log, const uint16_t *a,
                          const uint16_t *b, const float *dt_bias,
                          int64_t Ttok, int HV, float *g, float *beta,
                          cudaStream_t s) {
  const int64_t n = Ttok * (int64_t)HV;
  if (n == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int threads = 256;
  int64_t want = (n / 4 + threads - 1) / threads;
  int64_t cap = (int64_t)sms * 8;  // 8 resident 256-thread blocks per SM
  int blocks = (int)(want < cap ? (want < 1 ? 1 : want) : cap);
  gating_kernel<<<blocks, threads, 0, s>>>(A_log, a, b, dt_bias, n, HV, g, beta);
  return cudaGetLastError();
}

}  // namespace gdn_host
