// gdn_chunk_shared.cuh -- pieces shared by the chunked forward (gdn_chunk.cu)
// and backward (gdn_chunk_bwd.cu): chunk size, the per-(chunk, value head)
// record layout the prep kernel writes, and the sequence / chunk indexing.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdnc {

constexpr int C = 64;                           // chunk length
constexpr long long kWaitLimit = 2000000000LL;  // clock cycles (about 1 s) before a wait gives up
constexpr long long kTestWaitLimit = 4000;       // the testing hook's wait on a barrier nothing completes
constexpr float kLog2e = 1.4426950408889634f;

// Per-(chunk, value head) record, byte offsets; also its shared-memory image.
//   W   = [T diag(beta e^gamma / ||k||)] K   [64][K] bf16, 64-key SW128 atom columns
//   P   = causal e^{gamma_i - gamma_j} (q_i . k_j) / (||q_i|| ||k_j||) as bf16 hi + lo, [64][64] SW128
//   TS  = ((T - I) diag(beta))^T                [64][64] bf16 SW128 (row j = column j)
//   SC  = e^gamma / ||q||, e^{gamma_L - gamma} / ||k||, beta, e^{gamma_L} (fp32)
template <int K>
struct Rec {
  static constexpr int KA = K / 64;
  static constexpr int W = 0;
  static constexpr int PH = KA * 8192;
  static constexpr int PL = PH + 8192;
  static constexpr int TS = PL + 8192;
  static constexpr int SC = TS + 8192;
  static constexpr int BYTES = SC + 1024;
  static_assert(BYTES % 1024 == 0, "record alignment");
};
enum { RS_OG = 0, RS_SV = 64, RS_BET = 128, RS_DL = 192 };

// 2^x with the hardware approximation (relative error around 2^-22).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Sequence bounds (dense or cu_seqlens); false for offsets that break the rules.
__device__ __forceinline__ bool seq_bounds(const int32_t *cu, int n, int T, int64_t &tok0, int64_t &len) {
  if (cu) {
    const int32_t a0 = cu[n], a1 = cu[n + 1];
    if (a0 < 0 || a1 < a0 || a1 > T || (n == 0 && a0 != 0)) return false;
    tok0 = a0;
    len = a1 - a0;
  } else {
    tok0 = static_cast<int64_t>(n) * T;
    len = T;
  }
  return true;
}
__device__ __forceinline__ int chunks_of(int64_t len) { return static_cast<int>((len + C - 1) / C); }
// Index of the first chunk of sequence n in the workspace: cs[n], the prefix
// sums of the sequences' chunk counts (written by the chunk-starts kernel for
// cu_seqlens input; offsets that break the rules count 0 chunks), or
// n * chunks_of(T) for dense input (cs == NULL).
__device__ __forceinline__ int64_t chunk_base(const int32_t *cs, int n, int T) {
  return cs ? static_cast<int64_t>(cs[n]) : static_cast<int64_t>(n) * chunks_of(T);
}
// Sequence n and chunk c of chunk slot gc (false past the last chunk): for
// cu_seqlens input the largest n with cs[n] <= gc, by binary search.
__device__ __forceinline__ bool slot_chunk(const int32_t *cs, int N, int T, int64_t gc, int &n, int &c) {
  if (!cs) {
    const int nc = chunks_of(T);
    if (nc == 0 || gc >= static_cast<int64_t>(N) * nc) return false;
    n = static_cast<int>(gc / nc);
    c = static_cast<int>(gc % nc);
    return true;
  }
  if (N <= 0 || gc >= cs[N]) return false;
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cs[mid] <= gc) lo = mid; else hi = mid - 1;
  }
  n = lo;
  c = static_cast<int>(gc - cs[lo]);
  return true;
}

// Upper bound on the number of chunk slots of a call (varlen: one ragged chunk
// per sequence on top of T / C).
inline int64_t total_chunk_slots(int B, int T, int N, bool varlen) {
  const int64_t per = (static_cast<int64_t>(T) + C - 1) / C;
  return varlen ? per + N : static_cast<int64_t>(B) * per;
}
// Bytes of the chunk-starts array (N + 1 int32, cu_seqlens input only), kept
// in the workspace right after the records, in whole KB.
inline size_t chunk_starts_bytes(int N, bool varlen) {
  return varlen ? ((static_cast<size_t>(N) + 1) * 4 + 1023) / 1024 * 1024 : 0;
}

}  // namespace gdnc
