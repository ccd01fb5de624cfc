// gdn_common.cuh -- small device helpers shared by the libgdn kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn.h"

#define GDN_CHUNK 64
#define GDN_L2_EPS 1e-6f

namespace gdn {

__device__ __forceinline__ float bf2f(uint16_t x) {
  return __uint_as_float(static_cast<uint32_t>(x) << 16);
}

__device__ __forceinline__ uint16_t f2bf(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t *>(&h);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// softplus(x) = log1p(exp(x)), and x itself above 20 (where the two agree
// to well under one fp32 ulp).
__device__ __forceinline__ float softplus_f(float x) {
  return x > 20.f ? x : log1pf(expf(x));
}

__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

// The same two functions in a few fused multiply-adds, for the streaming gate
// kernels.  softplus(x) = max(x, 0) + log1p(e^-|x|), and for y = e^-|x| in
// (0, 1], log1p(y) = 2 artanh(s) with s = y / (2 + y) in (0, 1/3], taken as
// the odd Taylor series of artanh, 2 s (1 + s^2/3 + s^4/5 + ... + s^14/15):
// the first omitted term is below 1e-9 of the sum.  The exponential is the
// hardware one and the divisions are the fast ones (errors of a few ulp, far
// inside the 1e-5 relative budget of the gates).  gdn_gating and the fused
// gating of the prefill both use these, so their gates agree bit for bit.
__device__ __forceinline__ float log1p_unit(float y) {  // y in [0, 1]
  const float s = __fdividef(y, 2.f + y);
  const float t = s * s;
  float p = 1.f / 15.f;
  p = fmaf(p, t, 1.f / 13.f);
  p = fmaf(p, t, 1.f / 11.f);
  p = fmaf(p, t, 1.f / 9.f);
  p = fmaf(p, t, 1.f / 7.f);
  p = fmaf(p, t, 1.f / 5.f);
  p = fmaf(p, t, 1.f / 3.f);
  p = fmaf(p, t, 1.f);
  return 2.f * s * p;
}
__device__ __forceinline__ float softplus_fast(float x) {
  return x > 20.f ? x : fmaxf(x, 0.f) + log1p_unit(__expf(-fabsf(x)));
}
__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }

__device__ __forceinline__ void set_status(int32_t *st, int bits) {
  if (st) atomicOr(st, bits);
}

}  // namespace gdn

// Host-side launchers implemented in the kernel translation units.
namespace gdn_host {
cudaError_t launch_gating(const float *A_log, const uint16_t *a,
                          const uint16_t *b, const float *dt_bias,
                          int64_t Ttok, int HV, float *g, float *beta,
                          cudaStream_t s);
// Recurrent decode over N requests: request n owns tokens [cu[n], cu[n+1])
// (token n when cu is NULL), starts from pool[read_idx[n*ld + num_acc[n]-1]]
// (column 0 when num_acc is NULL) and stores the state after its i-th token
// into pool[write_idx[n*ld + i]].  pool is float* or bf16 (uint16_t*).
struct DecodeArgs {
  const uint16_t *q, *k, *v;
  const float *g, *beta, *A_log;
  const uint16_t *a, *b;
  const float *dt_bias;
  float scale;
  int l2;
  void *pool;
  int pool_bf16;
  int P;
  const int32_t *cu;
  int N, Ttot;
  const int32_t *read_idx, *write_idx;
  int ld;
  const int32_t *num_acc;
  int H, HV, K, V;
  uint16_t *o;
  int32_t *dev_status;
  int force_expiry;  // testing hook: the first bounded wait of every block runs out
};
cudaError_t launch_decode_general(const DecodeArgs &a, cudaStream_t s);
struct ChunkArgs {
  const uint16_t *q, *k, *v;
  const float *g, *beta;
  float scale;
  const float *h0;
  const int32_t *cu;
  int N, B, T, H, HV, K, V, l2;
  uint16_t *o;   // may be NULL (no output written)
  float *ht;
  float *hsave;  // NULL, or [chunk slots][HV][K][V]: the state entering every chunk
  // Fused gating (A_log != NULL; g, beta then NULL): the prep kernel computes
  // g = -e^{A_log} softplus(a + dt_bias), beta = sigmoid(b) itself and, when
  // g_out / beta_out are set, stores them ([B, T, HV] fp32).
  const float *A_log;
  const uint16_t *ga, *gb;
  const float *dt_bias;
  float *g_out, *beta_out;
  void *ws;
  size_t ws_bytes;
  int32_t *dev_status;
  int force_expiry;  // testing hook: the first bounded wait of every chain runs out
};
size_t chunk_workspace_bytes(int B, int T, int H, int HV, int K, int V, int N,
                             int varlen);
cudaError_t launch_chunk(const ChunkArgs &a, cudaStream_t s);
// Kernel launches of launch_chunk for these sizes on the current device (-1: no device).
int chunk_fwd_launches(int B, int T, int H, int HV, int K, int V, int N, int varlen);
struct ChunkBwdArgs {
  const uint16_t *q, *k, *v;
  const float *g, *beta;
  float scale;
  const float *h0;
  const int32_t *cu;
  int N, B, T, H, HV, K, V, l2;
  const uint16_t *dout;
  const float *dht;
  float *dq, *dk, *dv, *dg, *dbeta, *dh0;
  void *ws;
  size_t ws_bytes;
  int32_t *dev_status;
};
size_t chunk_bwd_workspace_bytes(int B, int T, int H, int HV, int K, int V, int N, int varlen);
cudaError_t launch_chunk_bwd(const ChunkBwdArgs &a, cudaStream_t s);
}  // namespace gdn_host
