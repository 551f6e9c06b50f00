// lizard_abi.cu -- the C ABI: host-side validation, workspace sizing and dispatch.
//
// Every entry point checks its arguments before enqueuing anything, then launches the
// kernels on the caller's stream and returns without synchronising.
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "lizard_dev.cuh"
#include "lizard_internal.h"

namespace {

// Clears the workspace header (status word and counters) in stream order.  A one-CTA
// kernel launched as a programmatic dependent: it waits for the previous kernel on the
// stream like a memset would, but its launch overlaps that kernel's tail and the next
// kernel can be launched before it ends, which a memset node prevents.
__global__ void header_reset_kernel(unsigned* w) {
  lz::pdl_wait();
  for (int i = threadIdx.x; i < (int)(lz::kWsHeader / sizeof(unsigned)); i += blockDim.x) w[i] = 0u;
  lz::pdl_trigger();
}

cudaError_t reset_header(void* workspace, cudaStream_t s, int* launches) {
  lz::trace_begin("header_reset", s);
  const cudaError_t e = lz::launch_pdl(header_reset_kernel, dim3(1), dim3(64), 0, s,
                                       static_cast<unsigned*>(workspace));
  lz::trace_end(s);
  ++*launches;
  return e;
}

}  // namespace

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

cudaError_t dispatch_fwd(const lz::FwdArgs& a, lizard_dtype dt, cudaStream_t s, int* launches) {
  return lz::fwd_chunk_tc_supported(a.dk, a.dv, a.L, a.W, a.M, dt)
             ? lz::launch_fwd_chunk_tc(a, a.ws, s, launches)
             : lz::launch_fwd_simt(a, dt, s, launches);
}

// ---------------------------------------------------------------------------------------
// Host-memory forward + backward: head slices pipelined over three streams.
// ---------------------------------------------------------------------------------------
int host_slice_heads(int H) { return (H + 7) / 8; }  // the widest slice

// Head slices of the host-memory pipeline: the first and the last hold a quarter of the
// widest slice, so that the copy-in before the first compute and the compute and copy-out
// after the last copy-in are short; the slices between hold up to the widest.  Returns
// the count and fills starts (head of each slice) and the end in starts[count].
int host_slice_plan(int H, int* starts, int max_slices) {
  const int Hs = host_slice_heads(H);
  const int edge = (Hs + 3) / 4;
  int n = 0, h = 0;
  if (H > 2 * edge + Hs) {
    starts[n++] = 0;
    h = edge;
    const int mid = H - 2 * edge;
    const int nmid = (mid + Hs - 1) / Hs;
    for (int k = 0; k < nmid; ++k) {
      starts[n++] = h;
      h += mid / nmid + (k < mid % nmid ? 1 : 0);
    }
    starts[n++] = h;
  } else {
    for (; h < H && n < max_slices; h += Hs) starts[n++] = h;
  }
  starts[n] = H;
  return n;
}

struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, ev_in[2] = {}, ev_comp[2] = {}, ev_out[2] = {};
  bool ready = false;
};
std::mutex g_pipe_mu;
HostPipe g_pipe[64];

// The copy streams and events of the current device, created on first use and kept for
// the life of the process.  Called with g_pipe_mu held.
HostPipe* host_pipe() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  HostPipe& p = g_pipe[dev];
  if (!p.ready) {
    bool ok = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming) == cudaSuccess;
    for (int b = 0; b < 2 && ok; ++b)
      ok = cudaEventCreateWithFlags(&p.ev_in[b], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&p.ev_comp[b], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&p.ev_out[b], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) return nullptr;
    p.ready = true;
  }
  return &p;
}

// Byte offsets of one slice buffer (device) for Hs heads.
struct SliceLayout {
  enum { PQ, PK, V, Q, K, DY, LG, H0, MK, MV, Y, DPQ, DPK, DV, DQ, DK, DLG, HF, DH0, DMK, DMV, N };
  size_t off[N];
  size_t bytes;
};

SliceLayout slice_layout(const lizard_dims& d, int Hs, bool h0, bool hf, bool dh0) {
  const size_t es = elem_size(d.dtype);
  const size_t tokT = (size_t)d.B * Hs * d.L * d.dk * es, tokF = (size_t)d.B * Hs * d.L * d.dk * 4;
  const size_t st = (size_t)d.B * Hs * d.dk * d.dv * 4;
  const size_t meT = (size_t)Hs * d.M * d.dk * es, meF = (size_t)Hs * d.M * d.dk * 4;
  const size_t sz[SliceLayout::N] = {tokT, tokT, tokT, tokT, tokT, tokT, tokF, h0 ? st : 0, meT, meT,
                                     tokT, tokT, tokT, tokT, tokT, tokT, tokF, hf ? st : 0,
                                     dh0 ? st : 0, meF, meF};
  SliceLayout l;
  size_t o = 0;
  for (int i = 0; i < SliceLayout::N; ++i) {
    l.off[i] = o;
    o += lz::align_up(sz[i], 256);
  }
  l.bytes = o;
  return l;
}

// Scratch of the forward (kept for the backward, which reuses it) and of the backward for
// one slice of Hs heads, without their headers.
size_t host_fwd_scratch(const lizard_dims& d, int W, int Hs) {
  lizard_dims ds = d;
  ds.H = Hs;
  return lizard_fwd_workspace_bytes(&ds, W) - lz::kWsHeader;
}

size_t host_bwd_scratch(const lizard_dims& d, int W, int Hs) {
  lizard_dims ds = d;
  ds.H = Hs;
  return lizard_bwd_workspace_bytes(&ds, W) - lz::kWsHeader;
}

// Copies heads [h0, h0+hs) of a [B, H, rows] tensor (rows bytes per head) between host and
// a [B, hs, rows] device buffer.
cudaError_t copy_heads(void* dst, const void* src, const lizard_dims& d, int h0, int hs,
                       size_t row, bool to_device, cudaStream_t s) {
  if (!dst || !src || row == 0) return cudaSuccess;
  if (to_device)
    return cudaMemcpy2DAsync(dst, hs * row, static_cast<const char*>(src) + h0 * row, d.H * row,
                             hs * row, d.B, cudaMemcpyHostToDevice, s);
  return cudaMemcpy2DAsync(static_cast<char*>(dst) + h0 * row, d.H * row, src, hs * row, hs * row,
                           d.B, cudaMemcpyDeviceToHost, s);
}

}  // namespace

void lz::set_last_launches(int n) { g_last_launches = n; }

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
  int launches = 0;
  cudaError_t e = reset_header(workspace, s, &launches);
  if (e != cudaSuccess) return LIZARD_ERR_CUDA;
  // A window longer than the sequence sees the same keys as one of length L.
  const int W_eff = d.L > 0 && W > d.L ? d.L : W;
  lz::FwdArgs a{d.B, d.H, d.L, d.dk, d.dv, d.M, W_eff, resolve_scale(d.scale, d.dk), alpha,
                phi_q, phi_k, v, log_gamma, q, k, meta_k, meta_v, y, h0, h_final,
                static_cast<unsigned*>(workspace),
                static_cast<unsigned char*>(workspace) + lz::kWsHeader};
  e = dispatch_fwd(a, d.dtype, s, &launches);
  g_last_launches = launches;
  return cuda_status(e);
}

lizard_status lizard_attn_fwd_fmap(const lizard_dims* dims, const void* x_q, const void* x_k,
                                   const void* w_q, const void* w_k, const void* v,
                                   const float* log_gamma, const void* q, const void* k,
                                   const void* meta_k, const void* meta_v, int32_t W,
                                   float alpha, void* y, const float* h0, float* h_final,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  g_last_launches = 0;
  if (!dims_ok(dims) || W < 1 || !isfinite(alpha)) return LIZARD_ERR_INVALID_ARG;
  const lizard_dims& d = *dims;
  const bool tok = d.L > 0;
  if (!ptr_ok(x_q, !tok) || !ptr_ok(x_k, !tok) || !ptr_ok(w_q, false) || !ptr_ok(w_k, false) ||
      !ptr_ok(v, !tok) || !ptr_ok(log_gamma, !tok) || !ptr_ok(q, !tok) || !ptr_ok(k, !tok) ||
      !ptr_ok(y, !tok))
    return LIZARD_ERR_INVALID_ARG;
  if (!ptr_ok(meta_k, d.M == 0) || !ptr_ok(meta_v, d.M == 0)) return LIZARD_ERR_INVALID_ARG;
  if (!ptr_ok(h0, true) || !ptr_ok(h_final, true)) return LIZARD_ERR_INVALID_ARG;
  const int W_eff = d.L > 0 && W > d.L ? d.L : W;
  // the fused prologue exists on the tensor-core path only (bf16, x and phi of width 128);
  // L = 0 has no tokens and only carries h0 to h_final
  if (d.dtype != LIZARD_BF16 || d.dk != 128 || d.dv != 128) return LIZARD_ERR_UNSUPPORTED;
  if (tok && !lz::fwd_chunk_tc_supported(d.dk, d.dv, d.L, W_eff, d.M, d.dtype))
    return LIZARD_ERR_UNSUPPORTED;
  const size_t need = lizard_fwd_workspace_bytes(dims, W);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return LIZARD_ERR_WORKSPACE;
  const size_t nt = (size_t)d.B * d.H * d.L * 128 * 2;
  const size_t nw = (size_t)d.H * 128 * 64 * 2;
  const size_t nh = (size_t)d.B * d.H * 128 * 128 * sizeof(float);
  const size_t nm = (size_t)d.H * d.M * 128 * 2;
  struct Span { const void* p; size_t n; };
  const Span ins[] = {{x_q, nt}, {x_k, nt}, {w_q, nw}, {w_k, nw}, {v, nt}, {log_gamma, nt * 2},
                      {q, nt}, {k, nt}, {meta_k, nm}, {meta_v, nm}, {h0, nh},
                      {workspace, workspace_bytes}};
  for (const Span& in : ins)
    if (overlap(y, nt, in.p, in.n) || overlap(h_final, nh, in.p, in.n)) return LIZARD_ERR_INVALID_ARG;
  if (overlap(y, nt, h_final, nh)) return LIZARD_ERR_INVALID_ARG;

  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(workspace, 0, lz::kWsHeader, s) != cudaSuccess) return LIZARD_ERR_CUDA;
  lz::FwdArgs a{d.B, d.H, d.L, d.dk, d.dv, d.M, W_eff, resolve_scale(d.scale, d.dk), alpha,
                nullptr, nullptr, v, log_gamma, q, k, meta_k, meta_v, y, h0, h_final,
                static_cast<unsigned*>(workspace),
                static_cast<unsigned char*>(workspace) + lz::kWsHeader};
  a.xq = x_q;
  a.xk = x_k;
  a.wq = w_q;
  a.wk = w_k;
  int launches = 0;
  // with no tokens the CUDA-core forward only copies h0 to h_final and reads no phi
  const cudaError_t e = tok ? lz::launch_fwd_chunk_tc(a, a.ws, s, &launches)
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
                              float* d_h0, const void* fwd_workspace, void* workspace,
                              size_t workspace_bytes, void* stream) {
  g_last_launches = 0;
  if (!dims_ok(dims) || W < 1 || !isfinite(alpha)) return LIZARD_ERR_INVALID_ARG;
  const lizard_dims& d = *dims;
  const bool tok = d.L > 0;
  const int W_eff = d.L > 0 && W > d.L ? d.L : W;
  // phi_q / phi_k may be NULL when the forward's saved context stands in for them: the
  // tensor-core GLA backward given fwd_workspace reads Qt, Kt and e^b, never phi.
  const bool ctx = fwd_workspace && lz::bwd_gla_tc_supported(d.dk, d.dv, d.L, d.dtype) &&
                   lz::fwd_ctx_usable(d.dk, d.dv, d.L, W_eff, d.M, d.dtype);
  if (!ptr_ok(phi_q, !tok || ctx) || !ptr_ok(phi_k, !tok || ctx)) return LIZARD_ERR_INVALID_ARG;
  const void* tok_ptrs[] = {v, log_gamma, q, k, dy, d_phi_q, d_phi_k, d_v, d_log_gamma, d_q, d_k};
  for (const void* p : tok_ptrs)
    if (!ptr_ok(p, !tok)) return LIZARD_ERR_INVALID_ARG;
  if (!ptr_ok(meta_k, d.M == 0) || !ptr_ok(meta_v, d.M == 0) ||
      !ptr_ok(d_meta_k, d.M == 0) || !ptr_ok(d_meta_v, d.M == 0))
    return LIZARD_ERR_INVALID_ARG;
  if (!ptr_ok(h0, true) || !ptr_ok(d_h0, true) || !ptr_ok(fwd_workspace, true))
    return LIZARD_ERR_INVALID_ARG;
  if (fwd_workspace && fwd_workspace == workspace) return LIZARD_ERR_INVALID_ARG;
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

  if (W_eff > kMaxBwdWindow) return LIZARD_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  int launches = 0;
  cudaError_t e = reset_header(workspace, s, &launches);
  if (e != cudaSuccess) return LIZARD_ERR_CUDA;
  lz::BwdArgs a{d.B, d.H, d.L, d.dk, d.dv, d.M, W_eff, resolve_scale(d.scale, d.dk), alpha,
                phi_q, phi_k, v, log_gamma, q, k, meta_k, meta_v, h0, dy,
                d_phi_q, d_phi_k, d_v, d_log_gamma, d_q, d_k, d_meta_k, d_meta_v, d_h0,
                static_cast<unsigned*>(workspace),
                static_cast<unsigned char*>(workspace) + lz::kWsHeader,
                workspace_bytes - lz::kWsHeader,
                fwd_workspace ? static_cast<unsigned char*>(const_cast<void*>(fwd_workspace)) +
                                    lz::kWsHeader
                              : nullptr};
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

lizard_status lizard_decode_ring_fill(const lizard_decode_dims* dims, int32_t L, int32_t W,
                                      const void* k, const void* v, void* k_ring, void* v_ring,
                                      int64_t* pos, void* stream) {
  g_last_launches = 0;
  if (!dims || dims->N < 1 || dims->H < 1 || L < 0 || W < 1) return LIZARD_ERR_INVALID_ARG;
  if (dims->dtype != LIZARD_F32 && dims->dtype != LIZARD_BF16) return LIZARD_ERR_INVALID_ARG;
  const lizard_status st = shape_supported(dims->dk, dims->dv);
  if (st != LIZARD_OK) return st;
  if (!ptr_ok(k, L == 0) || !ptr_ok(v, L == 0) || !ptr_ok(k_ring, false) ||
      !ptr_ok(v_ring, false) || !ptr_ok(pos, false))
    return LIZARD_ERR_INVALID_ARG;
  const size_t es = elem_size(dims->dtype);
  const size_t nr = (size_t)dims->N * dims->H * W * dims->dk * es;
  const size_t nt = (size_t)dims->N * dims->H * L * dims->dk * es;
  if (overlap(k_ring, nr, v_ring, nr) || overlap(k_ring, nr, k, nt) || overlap(k_ring, nr, v, nt) ||
      overlap(v_ring, nr, k, nt) || overlap(v_ring, nr, v, nt) ||
      overlap(pos, 8 * (size_t)dims->N, k_ring, nr) || overlap(pos, 8 * (size_t)dims->N, v_ring, nr))
    return LIZARD_ERR_INVALID_ARG;
  int launches = 0;
  const cudaError_t e = lz::launch_ring_fill(dims->N, dims->H, L, W, dims->dk, dims->dv,
                                             dims->dtype, k, v, k_ring, v_ring, pos,
                                             (cudaStream_t)stream, &launches);
  g_last_launches = launches;
  return cuda_status(e);
}

lizard_status lizard_state_combine(int32_t units, int32_t dk, int32_t dv, const float* gamma_a,
                                   const float* h_a, const float* gamma_b, const float* h_b,
                                   float* gamma_out, float* h_out, void* stream) {
  g_last_launches = 0;
  if (units < 0 || dk < 1 || dk > 1024 || dv < 4 || dv > 1024 || dv % 4 != 0)
    return LIZARD_ERR_INVALID_ARG;
  const bool any = units > 0;
  if (!ptr_ok(gamma_a, !any || !gamma_out) || !ptr_ok(h_a, !any) || !ptr_ok(gamma_b, !any) ||
      !ptr_ok(h_b, !any) || !ptr_ok(gamma_out, true) || !ptr_ok(h_out, !any))
    return LIZARD_ERR_INVALID_ARG;
  const size_t ng = (size_t)units * dk * 4, nh = ng * dv;
  if (overlap(gamma_out, ng, gamma_a, ng) || overlap(gamma_out, ng, gamma_b, ng) ||
      overlap(gamma_out, ng, h_a, nh) || overlap(gamma_out, ng, h_b, nh) ||
      overlap(gamma_out, ng, h_out, nh) || overlap(h_out, nh, gamma_a, ng) ||
      overlap(h_out, nh, gamma_b, ng))
    return LIZARD_ERR_INVALID_ARG;
  // h_out may coincide with h_a or h_b exactly (elementwise), not partially
  if ((overlap(h_out, nh, h_a, nh) && h_out != h_a) || (overlap(h_out, nh, h_b, nh) && h_out != h_b))
    return LIZARD_ERR_INVALID_ARG;
  int launches = 0;
  const cudaError_t e = lz::launch_state_combine(units, dk, dv, gamma_a, h_a, gamma_b, h_b,
                                                 gamma_out, h_out, (cudaStream_t)stream, &launches);
  g_last_launches = launches;
  return cuda_status(e);
}

namespace {
bool fmap_dims_ok(const lizard_fmap_dims* d) {
  if (!d || d->B < 1 || d->H < 1 || d->L < 0) return false;
  if (d->dtype != LIZARD_F32 && d->dtype != LIZARD_BF16) return false;
  if ((long long)d->B * d->H > 65535LL) return false;
  if ((long long)d->B * d->H * (long long)d->L > (1LL << 40)) return false;
  return lz::fmap_simt_supported(d->D, d->F);
}
}  // namespace

size_t lizard_feature_map_workspace_bytes(const lizard_fmap_dims* dims, int32_t is_bwd) {
  if (!fmap_dims_ok(dims)) return 0;
  if (!is_bwd) return lz::kWsHeader;
  return lz::kWsHeader + lz::fmap_bwd_workspace(dims->B, dims->H, dims->L, dims->D, dims->F,
                                               dims->dtype);
}

lizard_status lizard_feature_map_fwd(const lizard_fmap_dims* dims, const void* x, const void* w,
                                     void* phi, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  g_last_launches = 0;
  if (!fmap_dims_ok(dims)) return LIZARD_ERR_INVALID_ARG;
  const lizard_fmap_dims& d = *dims;
  const bool tok = d.L > 0;
  if (!ptr_ok(x, !tok) || !ptr_ok(w, false) || !ptr_ok(phi, !tok)) return LIZARD_ERR_INVALID_ARG;
  const size_t need = lizard_feature_map_workspace_bytes(dims, 0);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return LIZARD_ERR_WORKSPACE;
  const size_t es = elem_size(d.dtype), rows = (size_t)d.B * d.H * d.L;
  const size_t nphi = rows * 2 * d.F * es;
  if (overlap(phi, nphi, x, rows * d.D * es) || overlap(phi, nphi, w, (size_t)d.H * d.D * d.F * es) ||
      overlap(phi, nphi, workspace, workspace_bytes))
    return LIZARD_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(workspace, 0, lz::kWsHeader, s) != cudaSuccess) return LIZARD_ERR_CUDA;
  int launches = 0;
  const cudaError_t e = lz::launch_fmap_fwd(d.B, d.H, d.L, d.D, d.F, d.dtype, x, w, phi,
                                            static_cast<unsigned*>(workspace), s, &launches);
  g_last_launches = launches;
  return cuda_status(e);
}

lizard_status lizard_feature_map_bwd(const lizard_fmap_dims* dims, const void* x, const void* w,
                                     const void* d_phi, void* d_x, float* d_w, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  g_last_launches = 0;
  if (!fmap_dims_ok(dims)) return LIZARD_ERR_INVALID_ARG;
  const lizard_fmap_dims& d = *dims;
  const bool tok = d.L > 0;
  if (!ptr_ok(x, !tok) || !ptr_ok(w, false) || !ptr_ok(d_phi, !tok) || !ptr_ok(d_x, !tok) ||
      !ptr_ok(d_w, false))
    return LIZARD_ERR_INVALID_ARG;
  const size_t need = lizard_feature_map_workspace_bytes(dims, 1);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return LIZARD_ERR_WORKSPACE;
  const size_t es = elem_size(d.dtype), rows = (size_t)d.B * d.H * d.L;
  const size_t nx = rows * d.D * es, nw = (size_t)d.H * d.D * d.F * es, np = rows * 2 * d.F * es;
  const size_t ndw = (size_t)d.H * d.D * d.F * sizeof(float);
  const struct { const void* p; size_t n; } ins[] = {{x, nx}, {w, nw}, {d_phi, np},
                                                     {workspace, workspace_bytes}};
  for (const auto& in : ins)
    if (overlap(d_x, nx, in.p, in.n) || overlap(d_w, ndw, in.p, in.n)) return LIZARD_ERR_INVALID_ARG;
  if (overlap(d_x, nx, d_w, ndw)) return LIZARD_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(workspace, 0, lz::kWsHeader, s) != cudaSuccess) return LIZARD_ERR_CUDA;
  int launches = 0;
  const cudaError_t e = lz::launch_fmap_bwd(
      d.B, d.H, d.L, d.D, d.F, d.dtype, x, w, d_phi, d_x, d_w,
      static_cast<unsigned char*>(workspace) + lz::kWsHeader, static_cast<unsigned*>(workspace),
      s, &launches);
  g_last_launches = launches;
  return cuda_status(e);
}

namespace {
bool gate_dims_ok(const lizard_gate_dims* d) {
  if (!d || d->B < 1 || d->H < 1 || d->L < 0 || d->D < 1 || d->D > 256) return false;
  if (d->dk != 64 && d->dk != 128) return false;
  if (d->dtype != LIZARD_F32 && d->dtype != LIZARD_BF16) return false;
  if ((long long)d->B * d->H > 65535LL) return false;
  if ((long long)d->B * d->H * (long long)d->L > (1LL << 40)) return false;
  return isfinite(d->tau);
}
float resolve_tau(float tau) { return tau > 0.f ? tau : 16.f; }
}  // namespace

size_t lizard_gate_workspace_bytes(const lizard_gate_dims* dims) {
  if (!gate_dims_ok(dims)) return 0;
  return lz::align_up(lz::gate_bwd_workspace(dims->B, dims->H, dims->L, dims->D, dims->dk), 256);
}

lizard_status lizard_gate_fwd(const lizard_gate_dims* dims, const void* x, const void* w,
                              float* log_gamma, void* stream) {
  g_last_launches = 0;
  if (!gate_dims_ok(dims)) return LIZARD_ERR_INVALID_ARG;
  const lizard_gate_dims& d = *dims;
  const bool tok = d.L > 0;
  if (!ptr_ok(x, !tok) || !ptr_ok(w, false) || !ptr_ok(log_gamma, !tok)) return LIZARD_ERR_INVALID_ARG;
  const size_t es = elem_size(d.dtype);
  const size_t nx = (size_t)d.B * d.H * d.L * d.D * es, nw = (size_t)d.H * d.D * d.dk * es;
  const size_t nl = (size_t)d.B * d.H * d.L * d.dk * sizeof(float);
  if (overlap(log_gamma, nl, x, nx) || overlap(log_gamma, nl, w, nw)) return LIZARD_ERR_INVALID_ARG;
  int launches = 0;
  const cudaError_t e = lz::launch_gate_fwd(d.B, d.H, d.L, d.D, d.dk, d.dtype, resolve_tau(d.tau),
                                            x, w, log_gamma, (cudaStream_t)stream, &launches);
  g_last_launches = launches;
  return cuda_status(e);
}

lizard_status lizard_gate_bwd(const lizard_gate_dims* dims, const void* x, const void* w,
                              const float* d_log_gamma, void* d_x, float* d_w, void* workspace,
                              size_t workspace_bytes, void* stream) {
  g_last_launches = 0;
  if (!gate_dims_ok(dims)) return LIZARD_ERR_INVALID_ARG;
  const lizard_gate_dims& d = *dims;
  const bool tok = d.L > 0;
  if (!ptr_ok(x, !tok) || !ptr_ok(w, false) || !ptr_ok(d_log_gamma, !tok) || !ptr_ok(d_x, !tok) ||
      !ptr_ok(d_w, false))
    return LIZARD_ERR_INVALID_ARG;
  const size_t need = lizard_gate_workspace_bytes(dims);
  if (tok && (!workspace || workspace_bytes < need || !aligned16(workspace))) return LIZARD_ERR_WORKSPACE;
  const size_t es = elem_size(d.dtype);
  const size_t nx = (size_t)d.B * d.H * d.L * d.D * es, nw = (size_t)d.H * d.D * d.dk * es;
  const size_t nl = (size_t)d.B * d.H * d.L * d.dk * sizeof(float);
  const size_t ndw = (size_t)d.H * d.D * d.dk * sizeof(float);
  struct Span { const void* p; size_t n; };
  const Span ins[] = {{x, nx}, {w, nw}, {d_log_gamma, nl}, {workspace, workspace_bytes}};
  for (const Span& in : ins)
    if (overlap(d_x, nx, in.p, in.n) || overlap(d_w, ndw, in.p, in.n)) return LIZARD_ERR_INVALID_ARG;
  if (overlap(d_x, nx, d_w, ndw)) return LIZARD_ERR_INVALID_ARG;
  int launches = 0;
  const cudaError_t e = lz::launch_gate_bwd(d.B, d.H, d.L, d.D, d.dk, d.dtype, resolve_tau(d.tau),
                                            x, w, d_log_gamma, d_x, d_w,
                                            static_cast<unsigned char*>(workspace),
                                            (cudaStream_t)stream, &launches);
  g_last_launches = launches;
  return cuda_status(e);
}

size_t lizard_gla_std_workspace_bytes(const lizard_dims* dims) {
  if (!dims_ok(dims) || shape_supported(dims->dk, dims->dv) != LIZARD_OK) return 0;
  return lz::kWsHeader + lz::gla_std_workspace(dims->B * dims->H, dims->L, dims->dk);
}

lizard_status lizard_gla_std_fwd(const lizard_dims* dims, const void* phi_q, const void* phi_k,
                                 const void* v, const float* log_gamma, void* y, const float* h0,
                                 float* h_final, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  g_last_launches = 0;
  if (!dims_ok(dims)) return LIZARD_ERR_INVALID_ARG;
  const lizard_dims& d = *dims;
  const bool tok = d.L > 0;
  if (!ptr_ok(phi_q, !tok) || !ptr_ok(phi_k, !tok) || !ptr_ok(v, !tok) ||
      !ptr_ok(log_gamma, !tok) || !ptr_ok(y, !tok) || !ptr_ok(h0, true) || !ptr_ok(h_final, true))
    return LIZARD_ERR_INVALID_ARG;
  lizard_status st = shape_supported(d.dk, d.dv);
  if (st != LIZARD_OK) return st;
  if ((long long)d.B * d.H > 65535LL) return LIZARD_ERR_UNSUPPORTED;
  const size_t need = lizard_gla_std_workspace_bytes(dims);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return LIZARD_ERR_WORKSPACE;
  const size_t es = elem_size(d.dtype);
  const size_t ny = (size_t)d.B * d.H * d.L * d.dv * es;
  const size_t nk = (size_t)d.B * d.H * d.L * d.dk * es;
  const size_t nh = (size_t)d.B * d.H * d.dk * d.dv * sizeof(float);
  struct Span { const void* p; size_t n; };
  const Span ins[] = {{phi_q, nk}, {phi_k, nk}, {v, ny}, {log_gamma, nk / es * 4}, {h0, nh},
                      {workspace, workspace_bytes}};
  for (const Span& in : ins)
    if (overlap(y, ny, in.p, in.n) || overlap(h_final, nh, in.p, in.n)) return LIZARD_ERR_INVALID_ARG;
  if (overlap(y, ny, h_final, nh)) return LIZARD_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(workspace, 0, lz::kWsHeader, s) != cudaSuccess) return LIZARD_ERR_CUDA;
  int launches = 0;
  const cudaError_t e = lz::launch_gla_std_fwd(
      d.B * d.H, d.L, d.dk, d.dtype, phi_q, phi_k, v, log_gamma, h0, h_final, y,
      static_cast<unsigned*>(workspace), static_cast<unsigned char*>(workspace) + lz::kWsHeader, s,
      &launches);
  g_last_launches = launches;
  return cuda_status(e);
}

size_t lizard_fwd_bwd_host_workspace_bytes(const lizard_dims* dims, int32_t W) {
  if (!dims_ok(dims) || W < 1 || shape_supported(dims->dk, dims->dv) != LIZARD_OK) return 0;
  const int Hs = host_slice_heads(dims->H);
  const SliceLayout l = slice_layout(*dims, Hs, true, true, true);
  return 2 * lz::kWsHeader + lz::align_up(host_fwd_scratch(*dims, W, Hs), 256) +
         lz::align_up(host_bwd_scratch(*dims, W, Hs), 256) + 2 * l.bytes;
}

lizard_status lizard_attn_fwd_bwd_host(const lizard_dims* dims, const void* phi_q,
                                       const void* phi_k, const void* v, const float* log_gamma,
                                       const void* q, const void* k, const void* meta_k,
                                       const void* meta_v, int32_t W, float alpha,
                                       const float* h0, const void* dy, void* y, float* h_final,
                                       void* d_phi_q, void* d_phi_k, void* d_v,
                                       float* d_log_gamma, void* d_q, void* d_k, float* d_meta_k,
                                       float* d_meta_v, float* d_h0, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  g_last_launches = 0;
  if (!dims_ok(dims) || W < 1 || !isfinite(alpha)) return LIZARD_ERR_INVALID_ARG;
  const lizard_dims& d = *dims;
  const bool tok = d.L > 0;
  const void* tok_ptrs[] = {phi_q, phi_k, v, log_gamma, q, k, dy, y,
                            d_phi_q, d_phi_k, d_v, d_log_gamma, d_q, d_k};
  for (const void* p : tok_ptrs)
    if (!ptr_ok(p, !tok)) return LIZARD_ERR_INVALID_ARG;
  if (!ptr_ok(meta_k, d.M == 0) || !ptr_ok(meta_v, d.M == 0) ||
      !ptr_ok(d_meta_k, d.M == 0) || !ptr_ok(d_meta_v, d.M == 0))
    return LIZARD_ERR_INVALID_ARG;
  if (!ptr_ok(h0, true) || !ptr_ok(h_final, true) || !ptr_ok(d_h0, true))
    return LIZARD_ERR_INVALID_ARG;
  lizard_status st = shape_supported(d.dk, d.dv);
  if (st != LIZARD_OK) return st;
  const size_t need = lizard_fwd_bwd_host_workspace_bytes(dims, W);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return LIZARD_ERR_WORKSPACE;
  const int W_eff = d.L > 0 && W > d.L ? d.L : W;
  if (W_eff > kMaxBwdWindow) return LIZARD_ERR_UNSUPPORTED;

  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe* pp = host_pipe();
  if (!pp) return LIZARD_ERR_CUDA;
  HostPipe& P = *pp;
  cudaStream_t s = (cudaStream_t)stream;
  const int Hs = host_slice_heads(d.H);
  int starts[64];
  const int nslices = host_slice_plan(d.H, starts, 62);
  const SliceLayout l = slice_layout(d, Hs, h0 != nullptr, h_final != nullptr, d_h0 != nullptr);
  unsigned char* base = static_cast<unsigned char*>(workspace);
  // [status header][forward header + scratch][backward scratch][two slice buffers]; the
  // forward's header slot only gives its scratch the offset the backward expects.
  unsigned char* fwd_ws = base + lz::kWsHeader;
  unsigned char* fscratch = fwd_ws + lz::kWsHeader;
  unsigned char* bscratch = fscratch + lz::align_up(host_fwd_scratch(d, W, Hs), 256);
  const size_t bbytes = host_bwd_scratch(d, W, Hs);
  unsigned char* bufs = bscratch + lz::align_up(bbytes, 256);
  const size_t es = elem_size(d.dtype);
  const size_t rowT = (size_t)d.L * d.dk * es, rowF = (size_t)d.L * d.dk * 4;
  const size_t rowS = (size_t)d.dk * d.dv * 4;
  const size_t metaT = (size_t)d.M * d.dk * es, metaF = (size_t)d.M * d.dk * 4;
  const float scale = resolve_scale(d.scale, d.dk);

  cudaError_t e = cudaMemsetAsync(workspace, 0, lz::kWsHeader, s);
  // the copy streams start after the work already queued on `stream`
  if (e == cudaSuccess) e = cudaEventRecord(P.start, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(P.in, P.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(P.out, P.start, 0);
  int launches = 0;
  for (int si = 0; si < nslices && e == cudaSuccess; ++si) {
    const int b = si & 1, hb = starts[si], hs = starts[si + 1] - starts[si];
    unsigned char* buf = bufs + b * l.bytes;
    auto at = [&](int i) { return static_cast<void*>(buf + l.off[i]); };
    // copy in (after the compute of the slice that used this buffer two slices ago)
    if (si >= 2) e = cudaStreamWaitEvent(P.in, P.ev_comp[b], 0);
    const void* ins[] = {phi_q, phi_k, v, q, k, dy};
    const int in_ix[] = {SliceLayout::PQ, SliceLayout::PK, SliceLayout::V, SliceLayout::Q,
                         SliceLayout::K, SliceLayout::DY};
    for (int i = 0; i < 6 && e == cudaSuccess; ++i)
      e = copy_heads(at(in_ix[i]), ins[i], d, hb, hs, rowT, true, P.in);
    if (e == cudaSuccess) e = copy_heads(at(SliceLayout::LG), log_gamma, d, hb, hs, rowF, true, P.in);
    if (e == cudaSuccess && h0) e = copy_heads(at(SliceLayout::H0), h0, d, hb, hs, rowS, true, P.in);
    if (e == cudaSuccess && d.M > 0) {
      e = cudaMemcpyAsync(at(SliceLayout::MK), static_cast<const char*>(meta_k) + hb * metaT,
                          hs * metaT, cudaMemcpyHostToDevice, P.in);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(at(SliceLayout::MV), static_cast<const char*>(meta_v) + hb * metaT,
                            hs * metaT, cudaMemcpyHostToDevice, P.in);
    }
    if (e == cudaSuccess) e = cudaEventRecord(P.ev_in[b], P.in);
    // compute on `stream` (after this slice's inputs and the copy-out two slices ago)
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, P.ev_in[b], 0);
    if (e == cudaSuccess && si >= 2) e = cudaStreamWaitEvent(s, P.ev_out[b], 0);
    // every slice lists its own wide chunks: the forward's counter (read back by the
    // backward from the header slot in front of the forward's scratch) and the
    // backward's own start from zero
    unsigned* fwd_wcount = reinterpret_cast<unsigned*>(fwd_ws) + lz::kWsWideCount;
    if (e == cudaSuccess) e = cudaMemsetAsync(fwd_wcount, 0, sizeof(unsigned), s);
    if (e == cudaSuccess)
      e = cudaMemsetAsync(static_cast<unsigned*>(workspace) + lz::kWsWideCount, 0, sizeof(unsigned), s);
    if (e == cudaSuccess) {
      lz::FwdArgs fa{d.B, hs, d.L, d.dk, d.dv, d.M, W_eff, scale, alpha,
                     at(SliceLayout::PQ), at(SliceLayout::PK), at(SliceLayout::V),
                     static_cast<const float*>(at(SliceLayout::LG)), at(SliceLayout::Q),
                     at(SliceLayout::K), d.M ? at(SliceLayout::MK) : nullptr,
                     d.M ? at(SliceLayout::MV) : nullptr, at(SliceLayout::Y),
                     h0 ? static_cast<const float*>(at(SliceLayout::H0)) : nullptr,
                     h_final ? static_cast<float*>(at(SliceLayout::HF)) : nullptr,
                     static_cast<unsigned*>(workspace), fscratch};
      fa.wcount = fwd_wcount;
      if (d.L > 0 || h_final) e = dispatch_fwd(fa, d.dtype, s, &launches);
    }
    if (e == cudaSuccess) {
      lz::BwdArgs ba{d.B, hs, d.L, d.dk, d.dv, d.M, W_eff, scale, alpha,
                     at(SliceLayout::PQ), at(SliceLayout::PK), at(SliceLayout::V),
                     static_cast<const float*>(at(SliceLayout::LG)), at(SliceLayout::Q),
                     at(SliceLayout::K), d.M ? at(SliceLayout::MK) : nullptr,
                     d.M ? at(SliceLayout::MV) : nullptr,
                     h0 ? static_cast<const float*>(at(SliceLayout::H0)) : nullptr,
                     at(SliceLayout::DY), at(SliceLayout::DPQ), at(SliceLayout::DPK),
                     at(SliceLayout::DV), static_cast<float*>(at(SliceLayout::DLG)),
                     at(SliceLayout::DQ), at(SliceLayout::DK),
                     d.M ? static_cast<float*>(at(SliceLayout::DMK)) : nullptr,
                     d.M ? static_cast<float*>(at(SliceLayout::DMV)) : nullptr,
                     d_h0 ? static_cast<float*>(at(SliceLayout::DH0)) : nullptr,
                     static_cast<unsigned*>(workspace), bscratch, bbytes, fscratch};
      e = lz::launch_bwd_simt(ba, d.dtype, s, &launches);
    }
    if (e == cudaSuccess) e = cudaEventRecord(P.ev_comp[b], s);
    // copy out
    if (e == cudaSuccess) e = cudaStreamWaitEvent(P.out, P.ev_comp[b], 0);
    void* outs[] = {y, d_phi_q, d_phi_k, d_v, d_q, d_k};
    const int out_ix[] = {SliceLayout::Y, SliceLayout::DPQ, SliceLayout::DPK, SliceLayout::DV,
                          SliceLayout::DQ, SliceLayout::DK};
    for (int i = 0; i < 6 && e == cudaSuccess; ++i)
      e = copy_heads(outs[i], at(out_ix[i]), d, hb, hs, rowT, false, P.out);
    if (e == cudaSuccess) e = copy_heads(d_log_gamma, at(SliceLayout::DLG), d, hb, hs, rowF, false, P.out);
    if (e == cudaSuccess && h_final) e = copy_heads(h_final, at(SliceLayout::HF), d, hb, hs, rowS, false, P.out);
    if (e == cudaSuccess && d_h0) e = copy_heads(d_h0, at(SliceLayout::DH0), d, hb, hs, rowS, false, P.out);
    if (e == cudaSuccess && d.M > 0) {
      e = cudaMemcpyAsync(static_cast<char*>(static_cast<void*>(d_meta_k)) + hb * metaF,
                          at(SliceLayout::DMK), hs * metaF, cudaMemcpyDeviceToHost, P.out);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(static_cast<char*>(static_cast<void*>(d_meta_v)) + hb * metaF,
                            at(SliceLayout::DMV), hs * metaF, cudaMemcpyDeviceToHost, P.out);
    }
    if (e == cudaSuccess) e = cudaEventRecord(P.ev_out[b], P.out);
  }
  // `stream` covers every copy once it has passed the last copy-out
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, P.ev_out[(nslices - 1) & 1], 0);
  if (e == cudaSuccess && nslices > 1) e = cudaStreamWaitEvent(s, P.ev_out[nslices & 1], 0);
  g_last_launches = launches;
  return cuda_status(e);
}

}  // extern "C"
