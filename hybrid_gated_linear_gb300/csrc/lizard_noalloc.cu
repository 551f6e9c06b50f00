// lizard_noalloc.cu -- a decode step for callers that cannot allocate device memory.
//
// lizard_decode_step needs a small caller-provided workspace (a status word and one
// counter per sequence, used to advance pos from the last CTA of each sequence).  Some
// callers have no way to provide it: for example a plain-C host program or language
// binding that embeds this library without any device allocator of its own, or a serving
// runtime whose device memory is entirely owned by its own pool and which may not call
// cudaMalloc on the per-token path (a cudaMalloc can synchronise the device and can fail
// once the pool has reserved everything).  For them this file keeps the scratch in a
// fixed, file-scope device array and runs the same decode kernel with it.
//
// The array is loaded with the library on every GPU that uses it and stays there until
// the process exits.  Its size caps the number of sequences per call.
#include <mutex>

#include "lizard_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kScratchBytes =
    lz::kWsHeader + sizeof(unsigned) * (size_t)LIZARD_NOALLOC_MAX_SEQUENCES;

// Status word (first 256 bytes) and per-sequence counters.  Host code must not use this
// name as an address; it uses the device address fetched below.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device, fetched once per device.
lizard_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LIZARD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LIZARD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return LIZARD_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return LIZARD_OK;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool disjoint(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return true;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return !(x < y + nb && y < x + na);
}

}  // namespace

extern "C" lizard_status lizard_decode_step_noalloc(
    const lizard_decode_dims* dims, const void* phi_q, const void* phi_k, const void* v,
    const float* log_gamma, const void* q, const void* k, const void* meta_k,
    const void* meta_v, int32_t W, float alpha, float* h, void* k_ring, void* v_ring,
    int64_t* pos, void* y, void* stream) {
  lz::set_last_launches(0);
  if (!dims) return LIZARD_ERR_INVALID_ARG;
  const lizard_decode_dims& d = *dims;
  if (d.N < 1 || d.H < 1 || d.M < 0 || d.M > 16 || W < 1 || W > 1024 || !isfinite(alpha) ||
      !isfinite(d.scale) || (long long)d.N * d.H > 2147483647LL)
    return LIZARD_ERR_INVALID_ARG;
  if (d.dtype != LIZARD_F32 && d.dtype != LIZARD_BF16) return LIZARD_ERR_INVALID_ARG;
  if (d.dk != d.dv || (d.dk != 64 && d.dk != 128)) return LIZARD_ERR_UNSUPPORTED;
  if (d.N > LIZARD_NOALLOC_MAX_SEQUENCES) return LIZARD_ERR_UNSUPPORTED;
  const void* ptrs[] = {phi_q, phi_k, v, log_gamma, q, k, h, k_ring, v_ring, pos, y};
  for (const void* p : ptrs)
    if (!aligned16(p)) return LIZARD_ERR_INVALID_ARG;
  if (d.M > 0 && (!aligned16(meta_k) || !aligned16(meta_v))) return LIZARD_ERR_INVALID_ARG;
  const size_t es = d.dtype == LIZARD_F32 ? 4 : 2;
  const size_t nh = (size_t)d.N * d.H * d.dk * d.dv * sizeof(float);
  const size_t nr = (size_t)d.N * d.H * W * d.dk * es;
  const size_t ny = (size_t)d.N * d.H * d.dv * es;
  const size_t nt = (size_t)d.N * d.H * d.dk * es;
  struct Span { const void* p; size_t n; };
  const Span outs[] = {{h, nh}, {k_ring, nr}, {v_ring, nr}, {pos, (size_t)d.N * 8}, {y, ny}};
  const Span ins[] = {{phi_q, nt}, {phi_k, nt}, {v, nt}, {log_gamma, nt / es * 4}, {q, nt},
                      {k, nt}, {meta_k, (size_t)d.H * d.M * d.dk * es},
                      {meta_v, (size_t)d.H * d.M * d.dv * es}};
  for (int i = 0; i < 5; ++i) {
    for (const Span& in : ins)
      if (!disjoint(outs[i].p, outs[i].n, in.p, in.n)) return LIZARD_ERR_INVALID_ARG;
    for (int j = i + 1; j < 5; ++j)
      if (!disjoint(outs[i].p, outs[i].n, outs[j].p, outs[j].n)) return LIZARD_ERR_INVALID_ARG;
  }

  void* scratch = nullptr;
  lizard_status st = scratch_address(&scratch);
  if (st != LIZARD_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  // The counters must start at zero; clear them (and the status word) on the stream.
  if (cudaMemsetAsync(scratch, 0, lz::kWsHeader + sizeof(unsigned) * (size_t)d.N, s) !=
      cudaSuccess)
    return LIZARD_ERR_CUDA;
  unsigned char* base = static_cast<unsigned char*>(scratch);
  lz::DecArgs a{d.N, d.H, d.dk, d.dv, d.M, W, d.scale > 0.f ? d.scale : 1.0f / sqrtf((float)d.dk),
                alpha, phi_q, phi_k, v, log_gamma, q, k, meta_k, meta_v, h, k_ring, v_ring, pos,
                y, reinterpret_cast<unsigned*>(base + lz::kWsHeader),
                reinterpret_cast<unsigned*>(base)};
  int launches = 0;
  const cudaError_t e = lz::launch_decode(a, d.dtype, s, &launches);
  lz::set_last_launches(launches);
  return e == cudaSuccess ? LIZARD_OK : LIZARD_ERR_CUDA;
}
