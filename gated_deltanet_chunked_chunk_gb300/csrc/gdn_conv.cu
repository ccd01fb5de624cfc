// gdn_conv.cu -- causal depthwise conv1d in front of Gated DeltaNet, and its
// C ABI (gdn_causal_conv1d_fwd, gdn_causal_conv1d_update, gdn_conv_decode_pack).
//
// FastDeploy PR "support fla triton kernel for qwen3.5": Modifications table
// (causal_conv1d.py: causal_conv1d_update for decode against a conv-state pool
// addressed by slot ids, causal_conv1d_fn for varlen prefill with
// query_start_loc / has_initial_state) and Usage sections 3 and 4; LightLLM
// "gdn.py": the prefill backend convolves the packed q | k | v channels, the
// decode backend fuses the conv with the split into q, k, v.
//
// Per channel d, with the input stream history ++ x of a sequence (history =
// the slot's state, or zeros), out[d, p] = act(bias[d] + sum_j w[d, j] *
// stream[d, p + j]) where the last tap multiplies the current token; the slot
// then holds the last S entries of the stream.  act is identity or SiLU.
//
// All three ops are memory-bound (a few multiply-adds per element).
//  * conv_prefill_kernel: x is channel-first [dim, total]; a CTA takes one
//    channel and 32768 tokens, a thread 16 consecutive tokens per step with
//    16-byte loads and stores (the general per-token path, with a binary
//    search in query_start_loc, serves sequence starts and unaligned rows).
//  * conv_state_kernel (same stream, after the prefill kernel, so every read
//    of the old states precedes the writes): one thread per (sequence,
//    channel) writes the slot's new last-S inputs.
//  * conv_update_kernel: x is token-major [R, dim]; one thread per (request,
//    channel), consecutive threads on consecutive channels; the output goes to
//    up to three destination arrays split by channel range (the q | k | v
//    split of the fused decode form).
#include <math.h>

#include "gdn_common.cuh"

namespace {

constexpr int kConvMaxW = 8;
constexpr int kConvMaxS = 64;
constexpr int kPrefillTile = 32768;
constexpr int kGroup = 16;  // tokens a thread takes per step on the vector path

// Two floats to a bf16 pair (round to nearest even, as __float2bfloat16_rn),
// lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// SiLU with the hardware exponential and a fast divide: a few ulp of fp32,
// far below the bf16 rounding of the output (for x < -87 the divisor is huge
// and the result is 0, as SiLU underflows there anyway).
__device__ __forceinline__ float conv_act(float x, int act) { return act ? __fdividef(x, 1.f + __expf(-x)) : x; }

// Largest n in [0, N] with qsl[n] <= t (qsl non-decreasing), or -1.
__device__ __forceinline__ int seq_of(const int32_t *qsl, int N, int64_t t) {
  if (qsl[0] > t) return -1;
  int lo = 0, hi = N;  // invariant: qsl[lo] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (qsl[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Output of token t (one element), general path: sequence by binary search,
// taps before the sequence start read the slot's state or zero.
__device__ __forceinline__ float conv_prefill_one(const uint16_t *__restrict__ xr, const float *wf, float b0,
                                                  const uint16_t *__restrict__ states, int P, int S,
                                                  const int32_t *__restrict__ qsl, const int32_t *__restrict__ cache,
                                                  const uint8_t *__restrict__ has_init, int N, int dim, int d,
                                                  int64_t t, int W, int32_t *dev_status, bool &ok) {
  ok = false;
  const int n = seq_of(qsl, N, t);
  if (n < 0 || n >= N || qsl[n] < 0) {  // offsets that do not cover this token
    gdn::set_status(dev_status, GDN_DEV_BAD_CU_SEQLENS);
    return 0.f;
  }
  const int64_t s0 = qsl[n], p = t - s0;
  const int slot = cache ? cache[n] : -1;
  if (slot < -1 || slot >= P) gdn::set_status(dev_status, GDN_DEV_BAD_SLOT);
  const bool hist = slot >= 0 && slot < P && has_init && has_init[n];
  const uint16_t *srow = hist ? states + ((int64_t)slot * dim + d) * S : nullptr;
  float acc = b0;
#pragma unroll
  for (int j = 0; j < kConvMaxW; ++j) {
    if (j < W) {
      const int64_t src = p - (W - 1) + j;
      float v = 0.f;
      if (src >= 0) v = gdn::bf2f(xr[s0 + src]);
      else if (hist) v = gdn::bf2f(srow[S + src]);
      acc = fmaf(wf[j], v, acc);
    }
  }
  ok = true;
  return acc;
}

// One CTA per (channel, 32768-token tile).  Vector path (rows 16-byte aligned):
// a thread takes 16 consecutive tokens, loads them and the 8 before them with
// three 16-byte loads (the last mostly an L1 hit) and stores 32 bytes; tokens
// within W - 1 of a sequence start, or sharing the 16 with a boundary, take the
// general path.  Without aligned rows every token takes the general path.
// WT > 0 fixes the width at compile time (so the 24-value window stays in
// registers); WT = 0 takes it from W at run time.
template <int WT>
__global__ void __launch_bounds__(256) conv_prefill_kernel(
    const uint16_t *__restrict__ x, const uint16_t *__restrict__ w, const uint16_t *__restrict__ bias,
    const uint16_t *__restrict__ states, int P, int S, const int32_t *__restrict__ qsl,
    const int32_t *__restrict__ cache, const uint8_t *__restrict__ has_init, int N, int dim, int64_t total,
    int W_rt, int act, uint16_t *__restrict__ out, int32_t *dev_status, int vec) {
  const int W = WT > 0 ? WT : W_rt;
  const int d = blockIdx.x;
  float wf[kConvMaxW];
#pragma unroll
  for (int j = 0; j < kConvMaxW; ++j) wf[j] = j < W ? gdn::bf2f(w[(int64_t)d * W + j]) : 0.f;
  const float b0 = bias ? gdn::bf2f(bias[d]) : 0.f;
  const uint16_t *xr = x + (int64_t)d * total;
  uint16_t *orow = out + (int64_t)d * total;
  const int64_t tile0 = (int64_t)blockIdx.y * kPrefillTile;
  const int64_t t_end = min(total, tile0 + kPrefillTile);
  if (!vec) {
    for (int64_t t = tile0 + threadIdx.x; t < t_end; t += blockDim.x) {
      bool ok;
      const float acc = conv_prefill_one(xr, wf, b0, states, P, S, qsl, cache, has_init, N, dim, d, t, W,
                                         dev_status, ok);
      orow[t] = ok ? gdn::f2bf(conv_act(acc, act)) : (uint16_t)0;
    }
    return;
  }
  // The sequence [s_lo, s_hi) holding the last group looked up: the thread's
  // groups are kGroup blockDim tokens apart, so the binary search runs only
  // when a group leaves it.
  int64_t s_lo = 1, s_hi = 0;
  for (int64_t t0 = tile0 + kGroup * threadIdx.x; t0 < t_end; t0 += kGroup * blockDim.x) {
  // Fast path: all kGroup tokens in one sequence, at least W - 1 tokens past its start.
  bool fast = t0 + kGroup <= t_end;
  if (fast) {
    if (t0 < s_lo || t0 >= s_hi) {
      const int n = seq_of(qsl, N, t0);
      if (n >= 0 && n < N && qsl[n] >= 0) {
        s_lo = qsl[n];
        s_hi = qsl[n + 1];
      } else {
        s_lo = 1;
        s_hi = 0;
      }
    }
    fast = t0 >= s_lo && t0 - s_lo >= W - 1 && s_hi >= t0 + kGroup;
  }
  if (fast) {
    // The group's tokens and the 8 before it (W - 1 <= 7 of them are taps).
    const uint4 c0 = *reinterpret_cast<const uint4 *>(xr + t0);
    const uint4 c1 = *reinterpret_cast<const uint4 *>(xr + t0 + 8);
    uint4 prv = make_uint4(0, 0, 0, 0);
    if (t0 >= 8) prv = *reinterpret_cast<const uint4 *>(xr + t0 - 8);
    const uint32_t wv[12] = {prv.x, prv.y, prv.z, prv.w, c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    float v[24];
#pragma unroll
    for (int i = 0; i < 12; ++i) {
      v[2 * i] = gdn::bf2f(static_cast<uint16_t>(wv[i] & 0xFFFFu));
      v[2 * i + 1] = gdn::bf2f(static_cast<uint16_t>(wv[i] >> 16));
    }
    uint32_t o[8];
#pragma unroll
    for (int e = 0; e < kGroup; e += 2) {
      float a0 = b0, a1 = b0;
#pragma unroll
      for (int j = 0; j < kConvMaxW; ++j) {
        if (j < W) {
          a0 = fmaf(wf[j], v[8 + e - (W - 1) + j], a0);
          a1 = fmaf(wf[j], v[9 + e - (W - 1) + j], a1);
        }
      }
      o[e / 2] = pack_bf16x2(conv_act(a0, act), conv_act(a1, act));
    }
    *reinterpret_cast<uint4 *>(orow + t0) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4 *>(orow + t0 + 8) = make_uint4(o[4], o[5], o[6], o[7]);
    continue;
  }
  for (int64_t t = t0; t < t0 + kGroup && t < t_end; ++t) {
    bool ok;
    const float acc = conv_prefill_one(xr, wf, b0, states, P, S, qsl, cache, has_init, N, dim, d, t, W,
                                       dev_status, ok);
    orow[t] = ok ? gdn::f2bf(conv_act(acc, act)) : (uint16_t)0;
  }
  }
}

__global__ void __launch_bounds__(256) conv_state_kernel(
    const uint16_t *__restrict__ x, uint16_t *__restrict__ states, int P, int S, const int32_t *__restrict__ qsl,
    const int32_t *__restrict__ cache, const uint8_t *__restrict__ has_init, int N, int dim, int64_t total,
    int32_t *dev_status) {
  const int d = blockIdx.x * blockDim.x + threadIdx.x;
  const int n = blockIdx.y;
  if (d >= dim) return;
  const int64_t s0 = qsl[n], s1 = qsl[n + 1];
  if (s0 < 0 || s1 < s0 || s1 > total || (n == 0 && s0 != 0)) {
    if (d == 0) gdn::set_status(dev_status, GDN_DEV_BAD_CU_SEQLENS);
    return;
  }
  const int slot = cache ? cache[n] : -1;
  if (slot < 0 || slot >= P) return;  // no slot (PAD), or a bad one (flagged by the prefill kernel)
  const bool hist = has_init && has_init[n];
  uint16_t *srow = states + ((int64_t)slot * dim + d) * S;
  const int64_t len = s1 - s0;
  // New state j = stream position len + j of old (S entries, or zeros) ++ x
  // (len entries).  Going upward, entry len + j of the old row is read before
  // any write reaches it.
  for (int j = 0; j < S; ++j) {
    const int64_t pos = len + j;
    srow[j] = pos >= S ? x[(int64_t)d * total + s0 + (pos - S)] : (hist ? srow[pos] : (uint16_t)0);
  }
}

__global__ void __launch_bounds__(256) conv_update_kernel(
    const uint16_t *__restrict__ x, uint16_t *__restrict__ states, int P, int S, const uint16_t *__restrict__ w,
    const uint16_t *__restrict__ bias, const int32_t *__restrict__ idx, int dim, int W, int act,
    uint16_t *__restrict__ o0, uint16_t *__restrict__ o1, uint16_t *__restrict__ o2, int c1, int c2,
    int32_t *dev_status) {
  const int d = blockIdx.x * blockDim.x + threadIdx.x;
  const int r = blockIdx.y;
  if (d >= dim) return;
  uint16_t *dst = d < c1 ? o0 + (int64_t)r * c1 + d
                : d < c2 ? o1 + (int64_t)r * (c2 - c1) + (d - c1)
                         : o2 + (int64_t)r * (dim - c2) + (d - c2);
  const int slot = idx[r];
  if (slot < 0 || slot >= P) {
    if (slot != -1 && d == 0) gdn::set_status(dev_status, GDN_DEV_BAD_SLOT);
    *dst = 0;  // PAD (or a bad slot treated as PAD): zero row, pool untouched
    return;
  }
  uint16_t *srow = states + ((int64_t)slot * dim + d) * S;
  const uint16_t xv = x[(int64_t)r * dim + d];
  float acc = bias ? gdn::bf2f(bias[d]) : 0.f;
#pragma unroll
  for (int j = 0; j < kConvMaxW; ++j) {
    if (j < W) {
      // tap j reads stream position S - (W - 1) + j of history (S) ++ x
      const int pos = S - (W - 1) + j;
      const float v = gdn::bf2f(pos < S ? srow[pos] : xv);
      acc = fmaf(gdn::bf2f(w[(int64_t)d * W + j]), v, acc);
    }
  }
  *dst = gdn::f2bf(conv_act(acc, act));
  // Shift the row by one (reads run ahead of writes) and append x.
  for (int j = 0; j + 1 < S; ++j) srow[j] = srow[j + 1];
  srow[S - 1] = xv;
}

// Multi-token (speculative / MTP) decode, the LightLLM "gdn.py" MTP path's
// causal_conv1d_update with mtp_step, num_accepted_tokens and query_start_loc.
// A slot holds the last S inputs of its request's stream as of the previous
// step, whose last m + 1 entries were that step's tokens; of those only A =
// num_accepted_tokens[n] were accepted, so the accepted stream is the first
// S - (m + 1 - A) entries.  The request's tokens follow it (each output uses
// the W - 1 inputs before it) and the slot then holds the last S entries of
// accepted ++ tokens (zeros in front if that is shorter).  One thread per
// (request, channel); the accepted part of the row is read before the row is
// rewritten.
__global__ void __launch_bounds__(256) conv_update_spec_kernel(
    const uint16_t *__restrict__ x, uint16_t *__restrict__ states, int P, int S, const uint16_t *__restrict__ w,
    const uint16_t *__restrict__ bias, const int32_t *__restrict__ idx, const int32_t *__restrict__ num_acc,
    const int32_t *__restrict__ qsl, int Ttot, int m, int dim, int W, int act, uint16_t *__restrict__ out,
    int32_t *dev_status) {
  const int d = blockIdx.x * blockDim.x + threadIdx.x;
  const int n = blockIdx.y;
  if (d >= dim) return;
  const int t0 = qsl[n], t1 = qsl[n + 1];
  if (t0 < 0 || t1 < t0 || t1 > Ttot || t1 - t0 > m + 1) {
    if (d == 0) gdn::set_status(dev_status, GDN_DEV_BAD_CU_SEQLENS);
    return;
  }
  const int slot = idx[n];
  const int A = num_acc ? num_acc[n] : 1;
  const bool bad_acc = A < 1 || A > m + 1;
  if (slot < 0 || slot >= P || bad_acc) {
    if ((slot != -1 || bad_acc) && d == 0) gdn::set_status(dev_status, GDN_DEV_BAD_SLOT);
    for (int t = t0; t < t1; ++t) out[(int64_t)t * dim + d] = 0;  // PAD: zero rows, pool untouched
    return;
  }
  uint16_t *srow = states + ((int64_t)slot * dim + d) * S;
  const int la = S - (m + 1 - A);  // accepted entries (>= W - 1)
  uint16_t hist[kConvMaxS];
#pragma unroll
  for (int j = 0; j < kConvMaxS; ++j)
    if (j < la) hist[j] = srow[j];
  float wf[kConvMaxW];
#pragma unroll
  for (int j = 0; j < kConvMaxW; ++j) wf[j] = j < W ? gdn::bf2f(w[(int64_t)d * W + j]) : 0.f;
  const float b0 = bias ? gdn::bf2f(bias[d]) : 0.f;
  auto at = [&](int p) -> uint16_t { return p < la ? hist[p] : x[(int64_t)(t0 + p - la) * dim + d]; };
  const int nt = t1 - t0;
  for (int i = 0; i < nt; ++i) {
    float acc = b0;
#pragma unroll
    for (int j = 0; j < kConvMaxW; ++j)
      if (j < W) acc = fmaf(wf[j], gdn::bf2f(at(la - (W - 1) + i + j)), acc);
    out[(int64_t)(t0 + i) * dim + d] = gdn::f2bf(conv_act(acc, act));
  }
  const int len = la + nt;
  for (int k = 0; k < S; ++k) {
    const int p = len - S + k;
    srow[k] = p < 0 ? (uint16_t)0 : at(p);
  }
}

bool conv_dims_ok(int dim, int W, int S) {
  return dim > 0 && W >= 1 && W <= kConvMaxW && S >= W - 1 && S >= 1 && S <= kConvMaxS;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ECUDA; }

}  // namespace

extern "C" {

int gdn_causal_conv1d_fwd(const uint16_t *x, const uint16_t *weight, const uint16_t *bias,
                          uint16_t *conv_states, int P, int state_len, const int32_t *query_start_loc,
                          const int32_t *cache_indices, const uint8_t *has_initial_state, int N, int dim,
                          int64_t total, int width, int activation, uint16_t *out, int32_t *dev_status,
                          void *stream) {
  if (N < 0 || P < 0 || total < 0 || dim <= 0 || (activation != 0 && activation != 1)) return GDN_EINVAL;
  if (!conv_dims_ok(dim, width, state_len)) return GDN_EUNSUPPORTED;
  if (N == 0) return total == 0 ? GDN_OK : GDN_EINVAL;  // tokens need a sequence
  if (!query_start_loc || !weight) return GDN_EINVAL;
  if (total > 0 && (!x || !out)) return GDN_EINVAL;
  if (P > 0 && !conv_states) return GDN_EINVAL;
  if (cache_indices && !conv_states) return GDN_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (total > 0) {
    const int64_t tiles = (total + kPrefillTile - 1) / kPrefillTile;
    if (tiles > 65535) return GDN_EUNSUPPORTED;
    // 16-byte vector access needs every row start 16-byte aligned.
    const int vec = (total % 8 == 0) && ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15) == 0;
    const dim3 grid(dim, (unsigned)tiles);
    if (width == 4)
      conv_prefill_kernel<4><<<grid, 256, 0, s>>>(x, weight, bias, conv_states, P, state_len, query_start_loc,
                                                  cache_indices, has_initial_state, N, dim, total, width,
                                                  activation, out, dev_status, vec);
    else
      conv_prefill_kernel<0><<<grid, 256, 0, s>>>(x, weight, bias, conv_states, P, state_len, query_start_loc,
                                                  cache_indices, has_initial_state, N, dim, total, width,
                                                  activation, out, dev_status, vec);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return GDN_ECUDA;
  }
  if (N > 0 && cache_indices && P > 0) {
    if (N > 65535) return GDN_EUNSUPPORTED;
    conv_state_kernel<<<dim3((dim + 255) / 256, N), 256, 0, s>>>(
        x, conv_states, P, state_len, query_start_loc, cache_indices, has_initial_state, N, dim, total, dev_status);
    return cuda_rc(cudaGetLastError());
  }
  return GDN_OK;
}

int gdn_causal_conv1d_update(const uint16_t *x, uint16_t *conv_state, int P, int state_len,
                             const uint16_t *weight, const uint16_t *bias, const int32_t *conv_state_indices,
                             int R, int dim, int width, int activation, uint16_t *out, int32_t *dev_status,
                             void *stream) {
  if (R < 0 || P < 0 || dim <= 0 || (activation != 0 && activation != 1)) return GDN_EINVAL;
  if (!conv_dims_ok(dim, width, state_len)) return GDN_EUNSUPPORTED;
  if (R == 0) return GDN_OK;
  if (R > 65535) return GDN_EUNSUPPORTED;
  if (!x || !conv_state || !weight || !conv_state_indices || !out) return GDN_EINVAL;
  conv_update_kernel<<<dim3((dim + 255) / 256, R), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      x, conv_state, P, state_len, weight, bias, conv_state_indices, dim, width, activation, out, out, out, dim,
      dim, dev_status);
  return cuda_rc(cudaGetLastError());
}

int gdn_causal_conv1d_update_spec(const uint16_t *x, uint16_t *conv_state, int P, int state_len,
                                  const uint16_t *weight, const uint16_t *bias, const int32_t *conv_state_indices,
                                  const int32_t *num_accepted_tokens, const int32_t *query_start_loc, int N,
                                  int Ttot, int mtp_step, int dim, int width, int activation, uint16_t *out,
                                  int32_t *dev_status, void *stream) {
  if (N < 0 || P < 0 || Ttot < 0 || dim <= 0 || mtp_step < 0 || (activation != 0 && activation != 1))
    return GDN_EINVAL;
  if (!conv_dims_ok(dim, width, state_len) || state_len < width - 1 + mtp_step) return GDN_EUNSUPPORTED;
  if (N == 0) return GDN_OK;
  if (N > 65535) return GDN_EUNSUPPORTED;
  if (!x || !conv_state || !weight || !conv_state_indices || !query_start_loc || !out) return GDN_EINVAL;
  conv_update_spec_kernel<<<dim3((dim + 255) / 256, N), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      x, conv_state, P, state_len, weight, bias, conv_state_indices, num_accepted_tokens, query_start_loc, Ttot,
      mtp_step, dim, width, activation, out, dev_status);
  return cuda_rc(cudaGetLastError());
}

int gdn_conv_decode_pack(const uint16_t *mixed_qkv, uint16_t *conv_state, int P, int state_len,
                         const uint16_t *weight, const uint16_t *bias, const int32_t *conv_state_indices, int R,
                         int H, int HV, int K, int V, int width, int activation, uint16_t *q, uint16_t *k,
                         uint16_t *v, int32_t *dev_status, void *stream) {
  if (R < 0 || P < 0 || H <= 0 || HV <= 0 || K <= 0 || V <= 0 || (activation != 0 && activation != 1))
    return GDN_EINVAL;
  const int64_t dim64 = 2LL * H * K + (int64_t)HV * V;
  if (dim64 > (1LL << 30)) return GDN_EUNSUPPORTED;
  const int dim = static_cast<int>(dim64);
  if (!conv_dims_ok(dim, width, state_len)) return GDN_EUNSUPPORTED;
  if (R == 0) return GDN_OK;
  if (R > 65535) return GDN_EUNSUPPORTED;
  if (!mixed_qkv || !conv_state || !weight || !conv_state_indices || !q || !k || !v) return GDN_EINVAL;
  conv_update_kernel<<<dim3((dim + 255) / 256, R), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      mixed_qkv, conv_state, P, state_len, weight, bias, conv_state_indices, dim, width, activation, q, k, v,
      H * K, 2 * H * K, dev_status);
  return cuda_rc(cudaGetLastError());
}

}  // extern "C"
