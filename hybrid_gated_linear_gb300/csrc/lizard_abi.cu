// lizard_abi.cu -- the C ABI: host-side validation, workspace sizing and dispatch.
//
// Every entry point checks its arguments before enqueuing anything, then launches the
// kernels on the caller's stream and returns without synchronising.
#include <math.h>
#include <stdint.h>

#include "lizard_internal.h"

namespace {

thread_local int32_t g_last_launches = 0;

// The per-query window backward keeps one row of logits per warp in shared memory.
constexpr int kMaxBwdWindow = 4096;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A null pointer is allowed only where `optional` is true.
bool ptr_ok(const void* p, bool optional) { return p ? aligned16(p) : optional; }

bool dims_ok(const lizard_dims* d) {
  if (!d) return false;
  if (d->B < 1 || d->H < 1 || d->L < 0) return false;
  if (d->M < 0 || d->M > 16) return false;
  if (d->dtype != LIZARD_F32 && d->dtype != LIZARD_BF16) return false;
  if ((long long)d->B * d->H > 65535LL * 1024LL) return false;
  if ((long long)d->B * d->H * (long long)d->L > (1LL << 40)) return false;
  if (!isfinite(d->scale)) return false;
  return d->dk >= 1 && d->dv >= 1;
}

lizard_status shape_supported(int dk, int dv) {
  if (dk != dv) return LIZARD_ERR_UNSUPPORTED;
  if (dk != 64 && dk != 128) return LIZARD_ERR_UNSUPPORTED;
  return LIZARD_OK;
}

float resolve_scale(float scale, int dk) { return scale > 0.f ? scale : 1.0f / sqrtf((float)dk); }

size_t elem_size(lizard_dtype t) { return t == LIZARD_F32 ? 4 : 2; }

// [a, a+na) and [b, b+nb) overlap?
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

lizard_status cuda_status(cudaError_t e) { return e == cudaSuccess ? LIZARD_OK : LIZARD_ERR_CUDA; }

}  // namespace

extern "C" {

int32_t lizard_abi_version(void) { return LIZARD_ABI_VERSION; }

int32_t lizard_last_launch_count(void) { return g_last_launches; }

const char* lizard_status_string(lizard_status s) {
  switch (s) {
    case LIZARD_OK: return "ok";
    case LIZARD_ERR_INVALID_ARG: return "invalid argument";
    case LIZARD_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case LIZARD_ERR_CUDA: return "CUDA error";
    case LIZARD_ERR_TIMEOUT: return "device-side wait timed out";
    case LIZARD_ERR_DEVICE_CHECK: return "device-side check failed";
    case LIZARD_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

size_t lizard_fwd_workspace_bytes(const lizard_dims* dims, int32_t W) {
  if (!dims_ok(dims) || W < 1) return 0;
  const int W_eff = dims->L > 0 && W > dims->L ? dims->L : W;
  if (lz::fwd_chunk_tc_supported(dims->dk, dims->dv, dims->L, W_eff, dims->M, dims->dtype))
    return lz::kWsHeader + lz::fwd_chunk_tc_workspace(dims->B * dims->H, dims->L);
  return lz::kWsHeader;
}

size_t lizard_bwd_workspace_bytes(const lizard_dims* dims, int32_t W) {
  if (!dims_ok(dims) || W < 1) return 0;
  if (shape_supported(dims->dk, dims->dv) != LIZARD_OK) return 0;
  return lz::kWsHeader + lz::bwd_simt_workspace(dims->B, dims->H, dims->L, dims->dk, dims->dv,
                                               dims->M);
}

size_t lizard_decode_workspace_bytes(const lizard_decode_dims* dims) {
  if (!dims || dims->N < 1) return 0;
  return lz::kWsHeader + lz::align_up(sizeof(unsigned) * (size_t)dims->N, 256);
}

lizard_status lizard_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  g_last_launches = 0;
  if (!workspace || workspace_bytes == 0) return LIZARD_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream));
}

lizard_status lizard_check_device_errors(void* workspace, void* stream) {
  g_last_launches = 0;
  if (!workspace) return LIZARD_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LIZARD_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return LIZARD_ERR_CUDA;
  if (word != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(workspace, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return LIZARD_ERR_CUDA;
  }
  if (word & lz::kDevTimeout) return LIZARD_ERR_TIMEOUT;
  if (word & lz::kDevCheck) return LIZARD_ERR_DEVICE_CHECK;
  return LIZARD_OK;
}

lizard_status lizard_chunk_cumsum(int32_t units, int32_t L, int32_t dk, int32_t chunk,
                                  const float* log_gamma, float* b, float* gamma_chunk,
                                  void* stream) {
  g_last_launches = 0;
  if (units < 1 || units > 65535 || L < 0 || dk < 1 || dk > 1024 || chunk < 1 || chunk > 1024)
    return LIZARD_ERR_INVALID_ARG;
  if (!ptr_ok(log_gamma, false) || !ptr_ok(b, false) || !ptr_ok(gamma_chunk, true))
    return LIZARD_ERR_INVALID_ARG;
  const size_t n = (size_t)units * L * dk * sizeof(float);
  if (overlap(log_gamma, n, b, n)) return LIZARD_ERR_INVALID_ARG;
  int launches = 0;
  cudaError_t e = lz::launch_chunk_cumsum(units, L, dk, chunk, log_gamma, b, gamma_chunk,
                                          (cudaStream_t)stream, &launches);
  g_last_launches = launches;
  return cuda_status(e);
}

lizard_status lizard_attn_fwd(const lizard_dims* dims, const void* phi_q, const void* phi_k,
                              const void* v, const float* log_gamma, const void* q,
                              const void* k, const void* meta_k, const void* meta_v,
                              int32_t W, float alpha, void* y, const float* h0,
                              float* h_final, void* workspace, size_t workspace_bytes,
                              void* stream) {
  g_last_launches = 0;
  if (!dims_ok(dims) || W < 1 || !isfinite(alpha)) return LIZARD_ERR_INVALID_ARG;
  const lizard_dims& d = *dims;
  const bool tok = d.L > 0;
  if (!ptr_ok(phi_q, !tok) || !ptr_ok(phi_k, !tok) || !ptr_ok(v, !tok) ||
      !ptr_ok(log_gamma, !tok) || !ptr_ok(q, !tok) || !ptr_ok(k, !tok) || !ptr_ok(y, !tok))
    return LIZARD_ERR_INVALID_ARG;
  if (!ptr_ok(meta_k, d.M == 0) || !ptr_ok(meta_v, d.M == 0)) return LIZARD_ERR_INVALID_ARG;
  if (!ptr_ok(h0, true) || !ptr_ok(h_final, true)) return LIZARD_ERR_INVALID_ARG;
  lizard_status st = shape_supported(d.dk, d.dv);
  if (st != LIZARD_OK) return st;
  const size_t need = lizard_fwd_workspace_bytes(dims, W);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return LIZARD_ERR_WORKSPACE;
  const size_t es = elem_size(d.dtype);
  const size_t ny = (size_t)d.B * d.H * d.L * d.dv * es;
  const size_t nk = (size_t)d.B * d.H * d.L * d.dk * es;
  const size_t nh = (size_t)d.B * d.H * d.dk * d.dv * sizeof(float);
  const void* ins[] = {phi_q, phi_k, q, k};
  for (const void* p : ins)
    if (overlap(y, ny, p, nk) || overlap(h_final, nh, p, nk)) return LIZARD_ERR_INVALID_ARG;
  if (overlap(y, ny, v, ny) || overlap(y, ny, log_gamma, nk / es * 4) ||
      overlap(y, ny, h0, nh) || overlap(h_final, nh, h0, nh) || overlap(y, ny, h_final, nh) ||
      overlap(y, ny, workspace, workspace_bytes) || overlap(h_final, nh, workspace, workspace_bytes))
    return LIZARD_ERR_INVALID_ARG;

  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemsetAsync(workspace, 0, lz::kWsHeader, s);
  if (e != cudaSuccess) return LIZARD_ERR_CUDA;
  // A window longer than the sequence sees the same keys as one of length L.
  const int W_eff = d.L > 0 && W > d.L ? d.L : W;
  lz::FwdArgs a{d.B, d.H, d.L, d.dk, d.dv, d.M, W_eff, resolve_scale(d.scale, d.dk), alpha,
                phi_q, phi_k, v, log_gamma, q, k, meta_k, meta_v, y, h0, h_final,
                static_cast<unsigned*>(workspace),
                static_cast<unsigned char*>(workspace) + lz::kWsHeader};
  int launches = 0;
  e = lz::fwd_chunk_tc_supported(d.dk, d.dv, d.L, W_eff, d.M, d.dtype)
          ? lz::launch_fwd_chunk_tc(a, a.ws, s, &launches)
          : lz::launch_fwd_simt(a, d.dtype, s, &launches);
  g_last_launches = launches;
  return cuda_status(e);
}

lizard_status lizard_attn_bwd(const lizard_dims* dims, const void* phi_q, const void* phi_k,
                              const void* v, const float* log_gamma, const void* q,
                              const void* k, const void* meta_k, const void* meta_v,
                              int32_t W, float alpha, const float* h0, const void* dy,
                              void* d_phi_q, void* d_phi_k, void* d_v, float* d_log_gamma,
                              void* d_q, void* d_k, float* d_meta_k, float* d_meta_v,
                              float* d_h0, void* workspace, size_t workspace_bytes,
                              void* stream) {
  g_last_launches = 0;
  if (!dims_ok(dims) || W < 1 || !isfinite(alpha)) return LIZARD_ERR_INVALID_ARG;
  const lizard_dims& d = *dims;
  const bool tok = d.L > 0;
  const void* tok_ptrs[] = {phi_q, phi_k, v, log_gamma, q, k, dy,
                            d_phi_q, d_phi_k, d_v, d_log_gamma, d_q, d_k};
  for (const void* p : tok_ptrs)
    if (!ptr_ok(p, !tok)) return LIZARD_ERR_INVALID_ARG;
  if (!ptr_ok(meta_k, d.M == 0) || !ptr_ok(meta_v, d.M == 0) ||
      !ptr_ok(d_meta_k, d.M == 0) || !ptr_ok(d_meta_v, d.M == 0))
    return LIZARD_ERR_INVALID_ARG;
  if (!ptr_ok(h0, true) || !ptr_ok(d_h0, true)) return LIZARD_ERR_INVALID_ARG;
  lizard_status st = shape_supported(d.dk, d.dv);
  if (st != LIZARD_OK) return st;
  const size_t need = lizard_bwd_workspace_bytes(dims, W);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return LIZARD_ERR_WORKSPACE;
  const size_t es = elem_size(d.dtype);
  const size_t nt = (size_t)d.B * d.H * d.L * d.dk * es;  // dk == dv
  const size_t nf = (size_t)d.B * d.H * d.L * d.dk * sizeof(float);
  const size_t nm = (size_t)d.H * d.M * d.dk * sizeof(float);
  const size_t nh = (size_t)d.B * d.H * d.dk * d.dv * sizeof(float);
  struct Span { const void* p; size_t n; };
  const Span outs[] = {{d_phi_q, nt}, {d_phi_k, nt}, {d_v, nt}, {d_log_gamma, nf}, {d_q, nt},
                       {d_k, nt}, {d_meta_k, nm}, {d_meta_v, nm}, {d_h0, nh},
                       {workspace, workspace_bytes}};
  const Span ins[] = {{phi_q, nt}, {phi_k, nt}, {v, nt}, {log_gamma, nf}, {q, nt}, {k, nt},
                      {meta_k, nm / 4 * es}, {meta_v, nm / 4 * es}, {h0, nh}, {dy, nt}};
  const int nouts = sizeof(outs) / sizeof(outs[0]);
  for (int i = 0; i < nouts; ++i) {
    for (const Span& in : ins)
      if (overlap(outs[i].p, outs[i].n, in.p, in.n)) return LIZARD_ERR_INVALID_ARG;
    for (int j = i + 1; j < nouts; ++j)
      if (overlap(outs[i].p, outs[i].n, outs[j].p, outs[j].n)) return LIZARD_ERR_INVALID_ARG;
  }

  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemsetAsync(workspace, 0, lz::kWsHeader, s);
  if (e != cudaSuccess) return LIZARD_ERR_CUDA;
  const int W_eff = d.L > 0 && W > d.L ? d.L : W;
  if (W_eff > kMaxBwdWindow) return LIZARD_ERR_UNSUPPORTED;
  lz::BwdArgs a{d.B, d.H, d.L, d.dk, d.dv, d.M, W_eff, resolve_scale(d.scale, d.dk), alpha,
                phi_q, phi_k, v, log_gamma, q, k, meta_k, meta_v, h0, dy,
                d_phi_q, d_phi_k, d_v, d_log_gamma, d_q, d_k, d_meta_k, d_meta_v, d_h0,
                static_cast<unsigned*>(workspace),
                static_cast<unsigned char*>(workspace) + lz::kWsHeader,
                workspace_bytes - lz::kWsHeader};
  int launches = 0;
  e = lz::launch_bwd_simt(a, d.dtype, s, &launches);
  g_last_launches = launches;
  return cuda_status(e);
}

lizard_status lizard_decode_step(const lizard_decode_dims* dims, const void* phi_q,
                                 const void* phi_k, const void* v, const float* log_gamma,
                                 const void* q, const void* k, const void* meta_k,
                                 const void* meta_v, int32_t W, float alpha, float* h,
                                 void* k_ring, void* v_ring, int64_t* pos, void* y,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  g_last_launches = 0;
  if (!dims) return LIZARD_ERR_INVALID_ARG;
  const lizard_decode_dims& d = *dims;
  if (d.N < 1 || d.H < 1 || d.M < 0 || d.M > 16 || W < 1 || W > 1024 || !isfinite(alpha) ||
      !isfinite(d.scale) || (long long)d.N * d.H > 2147483647LL)
    return LIZARD_ERR_INVALID_ARG;
  if (d.dtype != LIZARD_F32 && d.dtype != LIZARD_BF16) return LIZARD_ERR_INVALID_ARG;
  const void* ptrs[] = {phi_q, phi_k, v, log_gamma, q, k, h, k_ring, v_ring, pos, y};
  for (const void* p : ptrs)
    if (!ptr_ok(p, false)) return LIZARD_ERR_INVALID_ARG;
  if (!ptr_ok(meta_k, d.M == 0) || !ptr_ok(meta_v, d.M == 0)) return LIZARD_ERR_INVALID_ARG;
  lizard_status st = shape_supported(d.dk, d.dv);
  if (st != LIZARD_OK) return st;
  const size_t need = lizard_decode_workspace_bytes(dims);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return LIZARD_ERR_WORKSPACE;
  const size_t es = elem_size(d.dtype);
  const size_t nh = (size_t)d.N * d.H * d.dk * d.dv * sizeof(float);
  const size_t nr = (size_t)d.N * d.H * W * d.dk * es;
  const size_t ny = (size_t)d.N * d.H * d.dv * es;
  const size_t nt = (size_t)d.N * d.H * d.dk * es;
  struct Span { const void* p; size_t n; };
  const Span outs[] = {{h, nh}, {k_ring, nr}, {v_ring, nr}, {pos, (size_t)d.N * 8}, {y, ny},
                       {workspace, workspace_bytes}};
  const Span ins[] = {{phi_q, nt}, {phi_k, nt}, {v, nt}, {log_gamma, nt / es * 4}, {q, nt}, {k, nt},
                      {meta_k, (size_t)d.H * d.M * d.dk * es}, {meta_v, (size_t)d.H * d.M * d.dv * es}};
  const int nouts = sizeof(outs) / sizeof(outs[0]);
  for (int i = 0; i < nouts; ++i) {
    for (const Span& in : ins)
      if (overlap(outs[i].p, outs[i].n, in.p, in.n)) return LIZARD_ERR_INVALID_ARG;
    for (int j = i + 1; j < nouts; ++j)
      if (overlap(outs[i].p, outs[i].n, outs[j].p, outs[j].n)) return LIZARD_ERR_INVALID_ARG;
  }
  lz::DecArgs a{d.N, d.H, d.dk, d.dv, d.M, W, resolve_scale(d.scale, d.dk), alpha,
                phi_q, phi_k, v, log_gamma, q, k, meta_k, meta_v, h, k_ring, v_ring, pos, y,
                reinterpret_cast<unsigned*>(static_cast<unsigned char*>(workspace) + lz::kWsHeader),
                static_cast<unsigned*>(workspace)};
  int launches = 0;
  cudaError_t e = lz::launch_decode(a, d.dtype, (cudaStream_t)stream, &launches);
  g_last_launches = launches;
  return cuda_status(e);
}

}  // extern "C"
