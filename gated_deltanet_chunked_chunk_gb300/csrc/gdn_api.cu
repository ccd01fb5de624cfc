// gdn_api.cu -- the C ABI of libgdn: argument checks, then stream-ordered
// launches.  No entry point allocates device memory or synchronises.
#include <cuda.h>
#include <math.h>

#include <atomic>
#include <initializer_list>

#include "gdn_common.cuh"

namespace {

bool head_dim_ok(int d) { return d == 64 || d == 128; }

// Testing hook (gdn_testing_force_wait_expiry): read at every launch.
std::atomic<int> g_force_wait_expiry{0};

int cuda_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ECUDA; }

// Buffers that the chunk kernels move with TMA, bulk copies or 16-byte
// accesses must start on a 16-byte boundary; a view at an odd offset is refused
// on the host instead of faulting on the device.  Null pointers pass.
bool aligned16(std::initializer_list<const void *> ptrs) {
  for (const void *p : ptrs)
    if (reinterpret_cast<uintptr_t>(p) & 15u) return false;
  return true;
}

// The chunk entry points encode TMA tensor maps with a driver call, which needs
// a context current on the calling thread.  A thread whose first CUDA work this
// is (a framework's worker thread, say) may have none: then setting the
// thread's device makes that device's primary context current.  A context the
// caller made current is left in place.
bool bind_context() {
  using GetCurrentFn = CUresult (*)(CUcontext *);
  static const GetCurrentFn get_current = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    const bool ok = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                        cudaSuccess &&
                    q == cudaDriverEntryPointSuccess;
    return ok ? reinterpret_cast<GetCurrentFn>(p) : nullptr;
  }();
  CUcontext ctx = nullptr;
  if (get_current && get_current(&ctx) == CUDA_SUCCESS && ctx) return true;
  int dev = 0;
  return cudaGetDevice(&dev) == cudaSuccess && cudaSetDevice(dev) == cudaSuccess;
}

}  // namespace

extern "C" {

const char *gdn_status_string(int status) {
  switch (status) {
    case GDN_OK: return "ok";
    case GDN_EINVAL: return "invalid argument (null pointer, inconsistent shape, HV % H != 0, or B != 1 with cu_seqlens)";
    case GDN_EUNSUPPORTED: return "unsupported configuration (head dims K and V must be 64 or 128; at most 65535 sequences or requests per call)";
    case GDN_ECUDA: return "CUDA error while launching";
    case GDN_EWORKSPACE: return "workspace missing or too small";
    case GDN_ESCRATCH_LIMIT: return "input needs more workspace than the fixed no-allocation scratch holds; call gdn_chunk_fwd with a workspace";
    default: return "unknown status";
  }
}

int gdn_version(void) { return 200; }

int gdn_testing_force_wait_expiry(int on) { return g_force_wait_expiry.exchange(on ? 1 : 0); }

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

int gdn_chunk_fwd_kernel_launches(int B, int T, int H, int HV, int K, int V, int N, int varlen) {
  if (B < 0 || T < 0 || N < 0 || HV <= 0 || (K != 64 && K != 128) || (V != 64 && V != 128)) return -1;
  return gdn_host::chunk_fwd_launches(B, T, H, HV, K, V, N, varlen);
}

namespace {
// Shared checks and launch of the two prefill entry points; `a` arrives with
// its gate fields set.
int chunk_fwd_common(gdn_host::ChunkArgs &a, const uint16_t *q, const uint16_t *k, const uint16_t *v, float scale,
                     const float *initial_state, const int32_t *cu_seqlens, int N, int B, int T, int H, int HV,
                     int K, int V, int use_qk_l2norm, uint16_t *o, float *final_state, void *workspace,
                     size_t workspace_bytes, int32_t *dev_status, void *stream) {
  if (B < 0 || T < 0 || H <= 0 || HV <= 0 || K <= 0 || V <= 0 || N < 0) return GDN_EINVAL;
  if (HV % H != 0) return GDN_EINVAL;
  if (cu_seqlens) {
    if (B != 1) return GDN_EINVAL;
  } else if (N != B) {
    return GDN_EINVAL;
  }
  if (!head_dim_ok(K) || !head_dim_ok(V)) return GDN_EUNSUPPORTED;
  if (N > 65535) return GDN_EUNSUPPORTED;
  const bool has_tokens = (int64_t)B * T > 0;
  const bool gates = a.A_log ? (a.ga && a.gb && a.dt_bias) : (a.g && a.beta);
  if (has_tokens && (!q || !k || !v || !gates || !o)) return GDN_EINVAL;
  if (!aligned16({q, k, v, o, initial_state, final_state, workspace})) return GDN_EINVAL;
  if (N == 0) return GDN_OK;
  const size_t need = gdn_host::chunk_workspace_bytes(B, T, H, HV, K, V, N, cu_seqlens != nullptr);
  if (need > 0 && (!workspace || workspace_bytes < need)) return GDN_EWORKSPACE;
  if (!(scale > 0.f)) scale = 1.f / sqrtf((float)K);  // also catches NaN
  a.q = q; a.k = k; a.v = v; a.scale = scale;
  a.h0 = initial_state; a.cu = cu_seqlens;
  a.N = N; a.B = B; a.T = T; a.H = H; a.HV = HV; a.K = K; a.V = V;
  a.l2 = use_qk_l2norm ? 1 : 0;
  a.o = o; a.ht = final_state; a.ws = workspace; a.ws_bytes = workspace_bytes;
  a.dev_status = dev_status;
  a.force_expiry = g_force_wait_expiry.load();
  if (!bind_context()) return GDN_ECUDA;
  return cuda_status(gdn_host::launch_chunk(a, static_cast<cudaStream_t>(stream)));
}
}  // namespace

int gdn_chunk_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                  const float *g, const float *beta, float scale,
                  const float *initial_state, const int32_t *cu_seqlens, int N,
                  int B, int T, int H, int HV, int K, int V, int use_qk_l2norm,
                  uint16_t *o, float *final_state, void *workspace,
                  size_t workspace_bytes, int32_t *dev_status, void *stream) {
  gdn_host::ChunkArgs a{};
  a.g = g; a.beta = beta;
  return chunk_fwd_common(a, q, k, v, scale, initial_state, cu_seqlens, N, B, T, H, HV, K, V, use_qk_l2norm, o,
                          final_state, workspace, workspace_bytes, dev_status, stream);
}

int gdn_chunk_fwd_gated(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *A_log,
                        const uint16_t *a_raw, const uint16_t *b_raw, const float *dt_bias, float scale,
                        const float *initial_state, const int32_t *cu_seqlens, int N, int B, int T, int H,
                        int HV, int K, int V, int use_qk_l2norm, uint16_t *o, float *final_state, float *g_out,
                        float *beta_out, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                        void *stream) {
  if ((g_out == nullptr) != (beta_out == nullptr)) return GDN_EINVAL;  // both or neither
  gdn_host::ChunkArgs a{};
  a.A_log = A_log; a.ga = a_raw; a.gb = b_raw; a.dt_bias = dt_bias; a.g_out = g_out; a.beta_out = beta_out;
  return chunk_fwd_common(a, q, k, v, scale, initial_state, cu_seqlens, N, B, T, H, HV, K, V, use_qk_l2norm, o,
                          final_state, workspace, workspace_bytes, dev_status, stream);
}

size_t gdn_chunk_bwd_workspace_size(int B, int T, int H, int HV, int K, int V, int N, int varlen) {
  if ((K != 64 && K != 128) || (V != 64 && V != 128) || B < 0 || T < 0 || HV <= 0 || N < 0) return 0;
  return gdn_host::chunk_bwd_workspace_bytes(B, T, H, HV, K, V, N, varlen);
}

int gdn_chunk_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *g, const float *beta,
                  float scale, const float *initial_state, const int32_t *cu_seqlens, int N, int B, int T, int H,
                  int HV, int K, int V, int use_qk_l2norm, const uint16_t *dout, const float *dht, float *dq,
                  float *dk, float *dv, float *dg, float *dbeta, float *dh0, void *workspace,
                  size_t workspace_bytes, int32_t *dev_status, void *stream) {
  if (B < 0 || T < 0 || H <= 0 || HV <= 0 || K <= 0 || V <= 0 || N < 0) return GDN_EINVAL;
  if (HV % H != 0) return GDN_EINVAL;
  if (cu_seqlens) {
    if (B != 1) return GDN_EINVAL;
  } else if (N != B) {
    return GDN_EINVAL;
  }
  if (!head_dim_ok(K) || !head_dim_ok(V)) return GDN_EUNSUPPORTED;
  if (N > 65535) return GDN_EUNSUPPORTED;
  const bool has_tokens = (int64_t)B * T > 0;
  if (has_tokens && (!q || !k || !v || !g || !beta || !dout || !dq || !dk || !dv || !dg || !dbeta))
    return GDN_EINVAL;
  if (!aligned16({q, k, v, dout, dht, initial_state, dq, dk, dh0, workspace})) return GDN_EINVAL;
  if (N == 0) return GDN_OK;
  const size_t need = gdn_host::chunk_bwd_workspace_bytes(B, T, H, HV, K, V, N, cu_seqlens != nullptr);
  if (!workspace || workspace_bytes < need) return GDN_EWORKSPACE;
  if (!(scale > 0.f)) scale = 1.f / sqrtf((float)K);
  gdn_host::ChunkBwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.scale = scale; a.h0 = initial_state; a.cu = cu_seqlens;
  a.N = N; a.B = B; a.T = T; a.H = H; a.HV = HV; a.K = K; a.V = V; a.l2 = use_qk_l2norm ? 1 : 0;
  a.dout = dout; a.dht = dht; a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dbeta = dbeta; a.dh0 = dh0;
  a.ws = workspace; a.ws_bytes = workspace_bytes; a.dev_status = dev_status;
  if (!bind_context()) return GDN_ECUDA;
  return cuda_status(gdn_host::launch_chunk_bwd(a, static_cast<cudaStream_t>(stream)));
}

namespace {
// Shared checks of the decode entry points; fills the gate part of `d`.
int decode_common(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *g, const float *beta,
                  const float *A_log, const uint16_t *a, const uint16_t *b, const float *dt_bias, float scale,
                  int use_qk_l2norm, const void *pool, int H, int HV, int K, int V, const uint16_t *o,
                  gdn_host::DecodeArgs &d) {
  if (H <= 0 || HV <= 0 || K <= 0 || V <= 0) return GDN_EINVAL;
  if (HV % H != 0) return GDN_EINVAL;
  if (!head_dim_ok(K) || !head_dim_ok(V)) return GDN_EUNSUPPORTED;
  if (!q || !k || !v || !o || !pool) return GDN_EINVAL;
  // The state moves in 16-byte vectors and bulk copies: a misaligned pool (a
  // view at an odd offset) is refused here instead of faulting on the device.
  if (reinterpret_cast<uintptr_t>(pool) & 15u) return GDN_EINVAL;
  const bool given = g || beta;
  const bool fused = A_log || a || b || dt_bias;
  if (given == fused) return GDN_EINVAL;  // exactly one gate group
  if (given && !(g && beta)) return GDN_EINVAL;
  if (fused && !(A_log && a && b && dt_bias)) return GDN_EINVAL;
  d.q = q; d.k = k; d.v = v; d.g = g; d.beta = beta; d.A_log = A_log; d.a = a; d.b = b; d.dt_bias = dt_bias;
  d.scale = (scale > 0.f) ? scale : 1.f / sqrtf((float)K);  // also catches NaN
  d.l2 = use_qk_l2norm ? 1 : 0;
  d.H = H; d.HV = HV; d.K = K; d.V = V;
  d.force_expiry = g_force_wait_expiry.load();
  return GDN_OK;
}
}  // namespace

int gdn_recurrent_decode(const uint16_t *q, const uint16_t *k,
                         const uint16_t *v, const float *g, const float *beta,
                         const float *A_log, const uint16_t *a,
                         const uint16_t *b, const float *dt_bias, float scale,
                         int use_qk_l2norm, float *ssm_pool, int P,
                         const int32_t *ssm_indices, int R, int H, int HV,
                         int K, int V, uint16_t *o, int32_t *dev_status,
                         void *stream) {
  if (R < 0 || P < 0) return GDN_EINVAL;
  if (H <= 0 || HV <= 0 || K <= 0 || V <= 0 || HV % H != 0) return GDN_EINVAL;
  if (!head_dim_ok(K) || !head_dim_ok(V)) return GDN_EUNSUPPORTED;
  if (R == 0) return GDN_OK;
  if (R > 65535) return GDN_EUNSUPPORTED;  // requests index the grid's y dimension
  if (!ssm_indices) return GDN_EINVAL;
  gdn_host::DecodeArgs d{};
  const int rc = decode_common(q, k, v, g, beta, A_log, a, b, dt_bias, scale, use_qk_l2norm, ssm_pool, H, HV,
                               K, V, o, d);
  if (rc != GDN_OK) return rc;
  d.pool = ssm_pool; d.pool_bf16 = 0; d.P = P;
  d.cu = nullptr; d.N = R; d.Ttot = R;
  d.read_idx = ssm_indices; d.write_idx = ssm_indices; d.ld = 1; d.num_acc = nullptr;
  d.o = o; d.dev_status = dev_status;
  return cuda_status(gdn_host::launch_decode_general(d, static_cast<cudaStream_t>(stream)));
}

int gdn_recurrent_decode_bf16(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *g,
                              const float *beta, const float *A_log, const uint16_t *a, const uint16_t *b,
                              const float *dt_bias, float scale, int use_qk_l2norm, uint16_t *ssm_pool, int P,
                              const int32_t *ssm_indices, int R, int H, int HV, int K, int V, uint16_t *o,
                              int32_t *dev_status, void *stream) {
  if (R < 0 || P < 0) return GDN_EINVAL;
  if (H <= 0 || HV <= 0 || K <= 0 || V <= 0 || HV % H != 0) return GDN_EINVAL;
  if (!head_dim_ok(K) || !head_dim_ok(V)) return GDN_EUNSUPPORTED;
  if (R == 0) return GDN_OK;
  if (R > 65535) return GDN_EUNSUPPORTED;  // requests index the grid's y dimension
  if (!ssm_indices) return GDN_EINVAL;
  gdn_host::DecodeArgs d{};
  const int rc = decode_common(q, k, v, g, beta, A_log, a, b, dt_bias, scale, use_qk_l2norm, ssm_pool, H, HV,
                               K, V, o, d);
  if (rc != GDN_OK) return rc;
  d.pool = ssm_pool; d.pool_bf16 = 1; d.P = P;
  d.cu = nullptr; d.N = R; d.Ttot = R;
  d.read_idx = ssm_indices; d.write_idx = ssm_indices; d.ld = 1; d.num_acc = nullptr;
  d.o = o; d.dev_status = dev_status;
  return cuda_status(gdn_host::launch_decode_general(d, static_cast<cudaStream_t>(stream)));
}

int gdn_recurrent_decode_mtp(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *g,
                             const float *beta, const float *A_log, const uint16_t *a, const uint16_t *b,
                             const float *dt_bias, float scale, int use_qk_l2norm, float *ssm_pool, int P,
                             const int32_t *cu_seqlens, int N, int Ttot, const int32_t *read_indices,
                             const int32_t *write_indices, int ld, const int32_t *num_accepted_tokens, int H,
                             int HV, int K, int V, uint16_t *o, int32_t *dev_status, void *stream) {
  if (N < 0 || P < 0 || Ttot < 0 || ld <= 0) return GDN_EINVAL;
  if (H <= 0 || HV <= 0 || K <= 0 || V <= 0 || HV % H != 0) return GDN_EINVAL;
  if (!head_dim_ok(K) || !head_dim_ok(V)) return GDN_EUNSUPPORTED;
  if (N == 0) return GDN_OK;
  if (N > 65535) return GDN_EUNSUPPORTED;
  if (!cu_seqlens || !read_indices || !write_indices) return GDN_EINVAL;
  if (Ttot == 0) return GDN_OK;
  gdn_host::DecodeArgs d{};
  const int rc = decode_common(q, k, v, g, beta, A_log, a, b, dt_bias, scale, use_qk_l2norm, ssm_pool, H, HV,
                               K, V, o, d);
  if (rc != GDN_OK) return rc;
  d.pool = ssm_pool; d.pool_bf16 = 0; d.P = P;
  d.cu = cu_seqlens; d.N = N; d.Ttot = Ttot;
  d.read_idx = read_indices; d.write_idx = write_indices; d.ld = ld; d.num_acc = num_accepted_tokens;
  d.o = o; d.dev_status = dev_status;
  return cuda_status(gdn_host::launch_decode_general(d, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
