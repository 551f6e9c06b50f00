// k_cumsum.cu -- chunk-local inclusive cumulative sum of log gamma (standalone form).
//
// "Lizard: An Efficient Linearization Framework for Large Language Models" (arXiv
// 2507.09025), Method: the parallel GLA form multiplies by cumulative gate products
// c_t; taking them in log space relative to the start of each chunk keeps exp(+-b)
// inside the fp32/bf16 range.  b_t = sum of log gamma from the chunk start to t
// (inclusive); Gamma_c = b at the chunk's last token.  Chunks are independent, so one
// CTA scans one chunk of one unit; each thread owns key dimensions (coalesced rows).
// The production forward kernels fuse this scan into their prologue.
#include "lizard_internal.h"

namespace lz {
namespace {

__global__ void chunk_cumsum_kernel(int L, int dk, int chunk, int nchunks, const float* lg,
                                    float* b, float* gamma_chunk) {
  const int c = blockIdx.x;
  const size_t u = blockIdx.y;
  const int t0 = c * chunk;
  const int t1 = min(L, t0 + chunk);
  for (int k = threadIdx.x; k < dk; k += blockDim.x) {
    float run = 0.f;
    for (int t = t0; t < t1; ++t) {
      const size_t idx = (u * L + t) * dk + k;
      run += lg[idx];
      b[idx] = run;
    }
    if (gamma_chunk) gamma_chunk[(u * nchunks + c) * dk + k] = run;
  }
}

}  // namespace

cudaError_t launch_chunk_cumsum(int units, int L, int dk, int chunk, const float* lg, float* b,
                                float* gamma_chunk, cudaStream_t s, int* launches) {
  if (L == 0) return cudaSuccess;
  const int nchunks = (L + chunk - 1) / chunk;
  const int threads = dk >= 256 ? 256 : ((dk + 31) / 32) * 32;
  dim3 grid(nchunks, units);
  trace_begin("chunk_cumsum", s);
  chunk_cumsum_kernel<<<grid, threads, 0, s>>>(L, dk, chunk, nchunks, lg, b, gamma_chunk);
  trace_end(s);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace lz
