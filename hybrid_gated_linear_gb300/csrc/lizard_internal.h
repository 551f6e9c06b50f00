// lizard_internal.h -- shared declarations of the CUDA library (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lizard.h"

namespace lz {

// Device status word bits (first word of every workspace).
enum : unsigned { kDevTimeout = 1u, kDevCheck = 2u };

// Every workspace starts with this many bytes: the status word, then zero padding.
constexpr size_t kWsHeader = 256;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Arguments of one forward call after validation (device pointers).
struct FwdArgs {
  int B, H, L, dk, dv, M, W;
  float scale, alpha;
  const void *pq, *pk, *v;
  const float* lg;
  const void *q, *k, *mk, *mv;
  void* y;
  const float* h0;
  float* hf;
  unsigned* status;
};

struct BwdArgs {
  int B, H, L, dk, dv, M, W;
  float scale, alpha;
  const void *pq, *pk, *v;
  const float* lg;
  const void *q, *k, *mk, *mv;
  const float* h0;
  const void* dy;
  void *dpq, *dpk, *dvv;
  float* dlg;
  void *dq, *dk_;
  float *dmk, *dmv, *dh0;
  unsigned* status;
  unsigned char* ws;  // workspace after the header
  size_t ws_bytes;
};

struct DecArgs {
  int N, H, dk, dv, M, W;
  float scale, alpha;
  const void *pq, *pk, *v;
  const float* lg;
  const void *q, *k, *mk, *mv;
  float* h;
  void *kr, *vr;
  int64_t* pos;
  void* y;
  unsigned* counters;  // N zero-initialised words
  unsigned* status;
};

// Optional per-kernel event tracing (no-ops unless enabled on this host thread).
void trace_begin(const char* name, cudaStream_t s);
void trace_end(cudaStream_t s);

// Launchers: return the first CUDA error and add the number of kernels they enqueued
// to *launches.
cudaError_t launch_chunk_cumsum(int units, int L, int dk, int chunk, const float* lg, float* b,
                                float* gamma_chunk, cudaStream_t s, int* launches);
cudaError_t launch_fwd_simt(const FwdArgs& a, lizard_dtype dt, cudaStream_t s, int* launches);
// Tensor-core forward (bf16, dk = dv = 128, W <= 129, M <= 16).
bool fwd_tc_supported(const FwdArgs& a, lizard_dtype dt);
cudaError_t launch_fwd_tc(const FwdArgs& a, cudaStream_t s, int* launches);
size_t bwd_simt_workspace(int B, int H, int L, int dk, int dv, int M);
cudaError_t launch_bwd_simt(const BwdArgs& a, lizard_dtype dt, cudaStream_t s, int* launches);
cudaError_t launch_decode(const DecArgs& a, lizard_dtype dt, cudaStream_t s, int* launches);

}  // namespace lz
