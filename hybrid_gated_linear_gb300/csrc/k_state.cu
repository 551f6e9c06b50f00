// k_state.cu -- state plumbing around the hot path: the associative combine of segment
// states used by a sequence split, and the prefill -> decode handoff of the window ring.
//
// Combine ("Lizard", arXiv 2507.09025, Preliminaries: recurrent form).  A segment of the
// recurrence h_i = diag(gamma_i) h_{i-1} + phi_k_i v_i^T maps its initial state h to
// diag(e^Gamma) h + h_seg, where Gamma is the sum of log gamma over the segment and h_seg
// its final state from a zero start.  Two consecutive segments compose as
//   (Gamma_1, h_1) o (Gamma_2, h_2) = (Gamma_1 + Gamma_2, diag(e^Gamma_2) h_1 + h_2),
// an associative operation, so the initial states of many segments follow from one
// exclusive scan.
//
// Ring fill (papernotes.org note on Lizard, 关键设计: Anchor Window Attention): after a
// prefill of L tokens the decode step at position L needs the keys and values of tokens
// max(0, L-W) .. L-1 in ring slots (t mod W), and pos = L.
#include "lizard_dev.cuh"
#include "lizard_internal.h"

namespace lz {
namespace {

// One thread per (unit, row, 4 columns).
__global__ void combine_kernel(int units, int dk, int dv, const float* __restrict__ ga,
                               const float* __restrict__ ha, const float* __restrict__ gb,
                               const float* __restrict__ hb, float* __restrict__ go,
                               float* __restrict__ ho) {
  const long n4 = (long)units * dk * (dv / 4);
  for (long e = blockIdx.x * (long)blockDim.x + threadIdx.x; e < n4; e += (long)gridDim.x * blockDim.x) {
    const long row = e / (dv / 4);  // unit * dk + k
    const float f = expf(gb[row]);
    const float4 a = reinterpret_cast<const float4*>(ha)[e];
    const float4 b = reinterpret_cast<const float4*>(hb)[e];
    reinterpret_cast<float4*>(ho)[e] =
        make_float4(fmaf(f, a.x, b.x), fmaf(f, a.y, b.y), fmaf(f, a.z, b.z), fmaf(f, a.w, b.w));
    if (go && e % (dv / 4) == 0) go[row] = ga[row] + gb[row];
  }
}

// One CTA per (sequence, head, ring slot), one thread per 16 bytes of a row.
template <typename T>
__global__ void ring_fill_kernel(int H, int L, int W, int dk, int dv, const T* __restrict__ k,
                                 const T* __restrict__ v, T* __restrict__ kr, T* __restrict__ vr,
                                 int64_t* __restrict__ pos) {
  const int slot = blockIdx.x % W;
  const long nh = blockIdx.x / W;  // sequence * H + head
  // the token that sits in this slot: the latest t < L with t mod W == slot
  const int last = L - 1 - ((L - 1 - slot) % W + W) % W;
  const bool have = L > 0 && last >= 0 && last >= L - W;
  constexpr int kPer = 16 / sizeof(T);
  for (int c = threadIdx.x * kPer; c < dk; c += blockDim.x * kPer) {
    uint4 val = make_uint4(0, 0, 0, 0);
    if (have) val = *reinterpret_cast<const uint4*>(k + ((size_t)nh * L + last) * dk + c);
    *reinterpret_cast<uint4*>(kr + ((size_t)nh * W + slot) * dk + c) = val;
  }
  for (int c = threadIdx.x * kPer; c < dv; c += blockDim.x * kPer) {
    uint4 val = make_uint4(0, 0, 0, 0);
    if (have) val = *reinterpret_cast<const uint4*>(v + ((size_t)nh * L + last) * dv + c);
    *reinterpret_cast<uint4*>(vr + ((size_t)nh * W + slot) * dv + c) = val;
  }
  if (blockIdx.x % (W * H) == 0 && threadIdx.x == 0) pos[nh / H] = L;
}

}  // namespace

cudaError_t launch_state_combine(int units, int dk, int dv, const float* ga, const float* ha,
                                 const float* gb, const float* hb, float* go, float* ho,
                                 cudaStream_t s, int* launches) {
  const long n4 = (long)units * dk * (dv / 4);
  if (n4 == 0) return cudaSuccess;
  const int threads = 256;
  const long blocks = (n4 + threads - 1) / threads;
  const int grid = (int)(blocks < 4L * ctas_per_wave(8) ? blocks : 4L * ctas_per_wave(8));
  trace_begin("state_combine", s);
  combine_kernel<<<grid, threads, 0, s>>>(units, dk, dv, ga, ha, gb, hb, go, ho);
  trace_end(s);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_ring_fill(int N, int H, int L, int W, int dk, int dv, lizard_dtype dt,
                             const void* k, const void* v, void* kr, void* vr, int64_t* pos,
                             cudaStream_t s, int* launches) {
  const long blocks = (long)N * H * W;
  if (blocks == 0) return cudaSuccess;
  trace_begin("ring_fill", s);
  if (dt == LIZARD_F32)
    ring_fill_kernel<float><<<(unsigned)blocks, 32, 0, s>>>(
        H, L, W, dk, dv, static_cast<const float*>(k), static_cast<const float*>(v),
        static_cast<float*>(kr), static_cast<float*>(vr), pos);
  else
    ring_fill_kernel<bf16><<<(unsigned)blocks, 32, 0, s>>>(
        H, L, W, dk, dv, static_cast<const bf16*>(k), static_cast<const bf16*>(v),
        static_cast<bf16*>(kr), static_cast<bf16*>(vr), pos);
  trace_end(s);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace lz
