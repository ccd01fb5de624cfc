// gdn_gating.cu -- fused gate kernel.
//
// FastDeploy PR "support fla triton kernel for qwen3.5", Usage section 5
// ("Fused GDN Gating"): g = -exp(A_log) * softplus(a + dt_bias) and
// beta = sigmoid(b), both fp32, in one launch.
//
// The op is elementwise and HBM-bound (4 bytes in, 8 bytes out per element).
// Fast path (HV % 8 == 0, 16-byte aligned buffers): a thread owns 8
// consecutive elements of one row of the [Ttok, HV] array -- one 16-byte load
// each of a and b, two 16-byte stores each of g and beta.  The grid-stride is
// a multiple of the HV / 8 groups of a row, so a thread always meets the same
// 8 heads and reads their -exp(A_log) and dt_bias once.  Other shapes take a
// plain one-element-per-thread loop.
#include "gdn_common.cuh"

namespace {

// softplus / sigmoid take the hardware exponential (gdn::softplus_fast,
// gdn::sigmoid_fast), which keeps the kernel on the memory roofline.
__global__ void __launch_bounds__(256) gating_kernel_v8(
    const float *__restrict__ A_log, const uint16_t *__restrict__ a,
    const uint16_t *__restrict__ b, const float *__restrict__ dt_bias,
    int64_t n8, int groups, float *__restrict__ g, float *__restrict__ beta) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;  // a multiple of `groups`
  const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i0 >= n8) return;
  const int h0 = (int)(i0 % groups) * 8;
  float na[8], db[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    na[j] = -expf(__ldg(A_log + h0 + j));
    db[j] = __ldg(dt_bias + h0 + j);
  }
  // Two rows of 8 per trip, both loads issued before either is used.
  auto compute = [&](const uint4 av, const uint4 bv, int64_t i) {
    const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
    const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
    float go[8], bo[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint16_t ah = (uint16_t)((j & 1) ? (aw[j >> 1] >> 16) : (aw[j >> 1] & 0xffff));
      const uint16_t bh = (uint16_t)((j & 1) ? (bw[j >> 1] >> 16) : (bw[j >> 1] & 0xffff));
      go[j] = na[j] * gdn::softplus_fast(gdn::bf2f(ah) + db[j]);
      bo[j] = gdn::sigmoid_fast(gdn::bf2f(bh));
    }
    float4 *gp = reinterpret_cast<float4 *>(g) + 2 * i;
    float4 *bp = reinterpret_cast<float4 *>(beta) + 2 * i;
    __stcs(gp, make_float4(go[0], go[1], go[2], go[3]));
    __stcs(gp + 1, make_float4(go[4], go[5], go[6], go[7]));
    __stcs(bp, make_float4(bo[0], bo[1], bo[2], bo[3]));
    __stcs(bp + 1, make_float4(bo[4], bo[5], bo[6], bo[7]));
  };
  int64_t i = i0;
  for (; i + stride < n8; i += 2 * stride) {
    const uint4 a0 = __ldcs(reinterpret_cast<const uint4 *>(a) + i);
    const uint4 b0 = __ldcs(reinterpret_cast<const uint4 *>(b) + i);
    const uint4 a1 = __ldcs(reinterpret_cast<const uint4 *>(a) + i + stride);
    const uint4 b1 = __ldcs(reinterpret_cast<const uint4 *>(b) + i + stride);
    compute(a0, b0, i);
    compute(a1, b1, i + stride);
  }
  if (i < n8) compute(__ldcs(reinterpret_cast<const uint4 *>(a) + i), __ldcs(reinterpret_cast<const uint4 *>(b) + i), i);
}

__global__ void __launch_bounds__(256) gating_kernel_any(
    const float *__restrict__ A_log, const uint16_t *__restrict__ a,
    const uint16_t *__restrict__ b, const float *__restrict__ dt_bias,
    int64_t n_elem, int HV, float *__restrict__ g, float *__restrict__ beta) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_elem; i += stride) {
    const int h = (int)(i % HV);
    g[i] = -expf(A_log[h]) * gdn::softplus_fast(gdn::bf2f(a[i]) + dt_bias[h]);
    beta[i] = gdn::sigmoid_fast(gdn::bf2f(b[i]));
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
  const bool aligned = ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) |
                         reinterpret_cast<uintptr_t>(g) | reinterpret_cast<uintptr_t>(beta)) & 15) == 0;
  if (HV % 8 == 0 && aligned) {
    const int groups = HV / 8;
    const int64_t n8 = n / 8;
    // Enough threads for one pass when that fits 8 resident blocks per SM;
    // otherwise a grid whose thread count is a multiple of `groups`.
    int64_t blocks = (n8 + threads - 1) / threads;
    const int64_t cap = (int64_t)sms * 8;
    if (blocks > cap) {
      blocks = cap;
      while ((blocks * threads) % groups != 0) --blocks;
    }
    gating_kernel_v8<<<(int)blocks, threads, 0, s>>>(A_log, a, b, dt_bias, n8, groups, g, beta);
  } else {
    int64_t want = (n + threads - 1) / threads;
    const int64_t cap = (int64_t)sms * 8;
    const int blocks = (int)(want < cap ? want : cap);
    gating_kernel_any<<<blocks, threads, 0, s>>>(A_log, a, b, dt_bias, n, HV, g, beta);
  }
  return cudaGetLastError();
}

}  // namespace gdn_host
