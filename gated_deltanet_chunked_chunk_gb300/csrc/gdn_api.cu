// gdn_api.cu -- the C ABI of libgdn: argument checks, then stream-ordered
// launches.  No entry point allocates device memory or synchronises.
#include <math.h>

#include "gdn_common.cuh"

namespace {

bool head_dim_ok(int d) { return d == 64 || d == 128; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ECUDA; }

}  // namespace

extern "C" {

const char *gdn_status_string(int status) {
  switch (status) {
    case GDN_OK: return "ok";
    case GDN_EINVAL: return "invalid argument (null pointer, inconsistent shape, HV % H != 0, or B != 1 with cu_seqlens)";
    case GDN_EUNSUPPORTED: return "unsupported configuration (head dims K and V must be 64 or 128)";
    case GDN_ECUDA: return "CUDA error while launching";
    case GDN_EWORKSPACE: return "workspace missing or too small";
    case GDN_ESCRATCH_LIMIT: return "input needs more workspace than the fixed no-allocation scratch holds; call gdn_chunk_fwd with a workspace";
    default: return "unknown status";
  }
}

int gdn_version(void) { return 100; }

int gdn_gating(const float *A_log, const uint16_t *a, const uint16_t *b,
               const float *dt_bias, int64_t Ttok, int HV, float *g,
               float *beta, void *stream) {
  if (Ttok < 0 || HV <= 0) return GDN_EINVAL;
  if (Ttok == 0) return GDN_OK;
  if (!A_log || !a || !b || !dt_bias || !g || !beta) return GDN_EINVAL;
  return cuda_status(gdn_host::launch_gating(A_log, a, b, dt_bias, Ttok, HV, g, beta,
                                             static_cast<cudaStream_t>(stream)));
}

size_t gdn_chunk_fwd_workspace_size(int B, int T, int H, int HV, int K, int V,
                                    int N, int varlen) {
  return gdn_host::chunk_workspace_bytes(B, T, H, HV, K, V, N, varlen);
}

int gdn_chunk_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                  const float *g, const float *beta, float scale,
                  const float *initial_state, const int32_t *cu_seqlens, int N,
                  int B, int T, int H, int HV, int K, int V, int use_qk_l2norm,
                  uint16_t *o, float *final_state, void *workspace,
                  size_t workspace_bytes, int32_t *dev_status, void *stream) {
  if (B < 0 || T < 0 || H <= 0 || HV <= 0 || K <= 0 || V <= 0 || N < 0) return GDN_EINVAL;
  if (HV % H != 0) return GDN_EINVAL;
  if (cu_seqlens) {
    if (B != 1) return GDN_EINVAL;
  } else if (N != B) {
    return GDN_EINVAL;
  }
  if (!head_dim_ok(K) || !head_dim_ok(V)) return GDN_EUNSUPPORTED;
  const bool has_tokens = (int64_t)B * T > 0;
  if (has_tokens && (!q || !k || !v || !g || !beta || !o)) return GDN_EINVAL;
  if (N == 0) return GDN_OK;
  const size_t need = gdn_host::chunk_workspace_bytes(B, T, H, HV, K, V, N, cu_seqlens != nullptr);
  if (need > 0 && (!workspace || workspace_bytes < need)) return GDN_EWORKSPACE;
  if (!(scale > 0.f)) scale = 1.f / sqrtf((float)K);  // also catches NaN
  gdn_host::ChunkArgs a;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.scale = scale;
  a.h0 = initial_state; a.cu = cu_seqlens;
  a.N = N; a.B = B; a.T = T; a.H = H; a.HV = HV; a.K = K; a.V = V;
  a.l2 = use_qk_l2norm ? 1 : 0;
  a.o = o; a.ht = final_state; a.ws = workspace; a.ws_bytes = workspace_bytes;
  a.dev_status = dev_status;
  return cuda_status(gdn_host::launch_chunk(a, static_cast<cudaStream_t>(stream)));
}

int gdn_recurrent_decode(const uint16_t *q, const uint16_t *k,
                         const uint16_t *v, const float *g, const float *beta,
                         const float *A_log, const uint16_t *a,
                         const uint16_t *b, const float *dt_bias, float scale,
                         int use_qk_l2norm, float *ssm_pool, int P,
                         const int32_t *ssm_indices, int R, int H, int HV,
                         int K, int V, uint16_t *o, int32_t *dev_status,
                         void *stream) {
  if (R < 0 || P < 0 || H <= 0 || HV <= 0 || K <= 0 || V <= 0) return GDN_EINVAL;
  if (HV % H != 0) return GDN_EINVAL;
  if (!head_dim_ok(K) || !head_dim_ok(V)) return GDN_EUNSUPPORTED;
  if (R == 0) return GDN_OK;
  if (!q || !k || !v || !o || !ssm_indices || !ssm_pool) return GDN_EINVAL;
  const bool given = g || beta;
  const bool fused = A_log || a || b || dt_bias;
  if (given == fused) return GDN_EINVAL;  // exactly one gate group
  if (given && !(g && beta)) return GDN_EINVAL;
  if (fused && !(A_log && a && b && dt_bias)) return GDN_EINVAL;
  if (!(scale > 0.f)) scale = 1.f / sqrtf((float)K);
  return cuda_status(gdn_host::launch_decode(q, k, v, g, beta, A_log, a, b, dt_bias, scale,
                                             use_qk_l2norm ? 1 : 0, ssm_pool, P, ssm_indices,
                                             R, H, HV, K, V, o, dev_status,
                                             static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
