// k_gate.cu -- the gate projection in front of the operator and its backward.
//
// The gate is data dependent and trained through a projection W_gamma ("Lizard", arXiv
// 2507.09025, Method / Stage 1: the gate projection is trained; papernotes.org note,
// 关键设计: gamma_i is computed by W_gamma).  The pages fix neither the projection's
// input nor its nonlinearity; the reading taken here (that of the workloads' gates) is
//   log gamma[b,h,t,k] = logsigmoid( sum_d x[b,h,t,d] W[h,d,k] ) / tau,   tau = 16 by default,
// so that gamma is in (0, 1) and tau sets how slowly the state decays.  Backward, with
// z = x W recomputed and d/dz logsigmoid(z) = sigmoid(-z):
//   dz = d_log_gamma sigmoid(-z) / tau,   dx = dz W^T,   dW[h] = sum over batch and tokens x^T dz
// CUDA cores, fp32 arithmetic, x and dx in the operator's element type, W in the element
// type, dW fp32.  The dW partials of every (b, h, group of kGroupTok tokens) are summed
// afterwards in a fixed order, so dW is run-to-run identical.
#include <type_traits>

#include "lizard_dev.cuh"
#include "lizard_internal.h"

namespace lz {
namespace {

constexpr int kTok = 32;         // tokens per tile
constexpr int kThreads = 256;
constexpr int kDc = 32;          // input features staged per step
constexpr int kGroupTok = 512;   // tokens per backward CTA (one dW partial each)

// log sigmoid(z) = min(z, 0) - log(1 + e^-|z|), finite for every finite z
__device__ __forceinline__ float logsigmoid(float z) {
  return fminf(z, 0.f) - log1pf(expf(-fabsf(z)));
}

__device__ __forceinline__ float sigmoid_neg(float z) {  // sigmoid(-z) = 1 - sigmoid(z)
  return z >= 0.f ? expf(-z) / (1.f + expf(-z)) : 1.f / (1.f + expf(z));
}

// z = x W for a tile of kTok tokens x DK columns: thread (row group rg = tid / 32 -> rows
// 4 rg .. 4 rg + 3, lane -> columns lane + 32 j).  xs [kTok][kDc + 1], ws [kDc][DK] staged.
template <typename T, int DK>
__device__ void tile_z(const T* x, const T* w, int D, int t0, int n, float* xs, float* ws,
                       float (&acc)[4][DK / 32]) {
  const int tid = threadIdx.x, lane = tid & 31, rg = tid >> 5;
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int j = 0; j < DK / 32; ++j) acc[r][j] = 0.f;
  for (int d0 = 0; d0 < D; d0 += kDc) {
    const int dn = min(kDc, D - d0);
    __syncthreads();
    for (int e = tid; e < kTok * kDc; e += kThreads) {
      const int t = e / kDc, d = e % kDc;
      xs[t * (kDc + 1) + d] = (t < n && d < dn) ? ld_f(x + (size_t)(t0 + t) * D + d0 + d) : 0.f;
    }
    for (int e = tid; e < kDc * DK; e += kThreads) {
      const int d = e / DK, k = e % DK;
      ws[e] = d < dn ? ld_f(w + (size_t)(d0 + d) * DK + k) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int d = 0; d < kDc; ++d) {
      float wv[DK / 32];
#pragma unroll
      for (int j = 0; j < DK / 32; ++j) wv[j] = ws[d * DK + lane + 32 * j];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float xv = xs[(4 * rg + r) * (kDc + 1) + d];
#pragma unroll
        for (int j = 0; j < DK / 32; ++j) acc[r][j] = fmaf(xv, wv[j], acc[r][j]);
      }
    }
  }
}

template <typename T, int DK>
__global__ void __launch_bounds__(kThreads) gate_fwd_kernel(int H, int L, int D, float inv_tau,
                                                            const T* x, const T* w, float* lg) {
  __shared__ float xs[kTok * (kDc + 1)];
  __shared__ float ws[kDc * DK];
  const int bh = blockIdx.y, hh = bh % H, t0 = blockIdx.x * kTok, n = min(kTok, L - t0);
  const int lane = threadIdx.x & 31, rg = threadIdx.x >> 5;
  pdl_wait();
  float acc[4][DK / 32];
  tile_z<T, DK>(x + (size_t)bh * L * D, w + (size_t)hh * D * DK, D, t0, n, xs, ws, acc);
  float* out = lg + ((size_t)bh * L + t0) * DK;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int t = 4 * rg + r;
    if (t < n) {
#pragma unroll
      for (int j = 0; j < DK / 32; ++j) out[(size_t)t * DK + lane + 32 * j] = logsigmoid(acc[r][j]) * inv_tau;
    }
  }
  pdl_trigger();
}

// One CTA per (b, h, group of kGroupTok tokens): tiles of kTok tokens in order; dx per tile,
// this group's dW partial accumulated in registers (thread: input features tid / (DK/4)
// ... strided) and written once.
template <typename T, int DK>
__global__ void __launch_bounds__(kThreads) gate_bwd_kernel(int H, int L, int D, int groups,
                                                            float inv_tau, const T* x, const T* w,
                                                            const float* dlg, T* dx, float* dw_part) {
  extern __shared__ float sm[];
  float* xs = sm;                              // [kTok][kDc + 1] (z), then [kTok][D + 1] (x tile)
  float* ws = xs + kTok * (256 + 1);           // [kDc][DK]
  float* dzs = ws + kDc * DK;                  // [kTok][DK]
  const int g = blockIdx.x, bh = blockIdx.y, hh = bh % H;
  const int tid = threadIdx.x, lane = tid & 31, rg = tid >> 5;
  const T* xb = x + (size_t)bh * L * D;
  const T* wh = w + (size_t)hh * D * DK;
  pdl_wait();
  // dW partial: element e = tid + kThreads m of the [D][DK] block
  constexpr int kMaxAcc = 256 * DK / kThreads;
  float dwa[kMaxAcc];
#pragma unroll
  for (int m = 0; m < kMaxAcc; ++m) dwa[m] = 0.f;
  const int tend = min(L, (g + 1) * kGroupTok);
  for (int t0 = g * kGroupTok; t0 < tend; t0 += kTok) {
    const int n = min(kTok, L - t0);
    float acc[4][DK / 32];
    tile_z<T, DK>(xb, wh, D, t0, n, xs, ws, acc);
    // dz = d log gamma sigmoid(-z) / tau  (rows beyond L: 0)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int t = 4 * rg + r;
#pragma unroll
      for (int j = 0; j < DK / 32; ++j) {
        const int k = lane + 32 * j;
        dzs[t * DK + k] = t < n ? dlg[((size_t)bh * L + t0 + t) * DK + k] * sigmoid_neg(acc[r][j]) * inv_tau : 0.f;
      }
    }
    __syncthreads();
    // x tile in full [kTok][D] for dW (over the z staging, no longer needed)
    for (int e = tid; e < kTok * D; e += kThreads) {
      const int t = e / D, d = e % D;
      xs[t * (D + 1) + d] = t < n ? ld_f(xb + (size_t)(t0 + t) * D + d) : 0.f;
    }
    __syncthreads();
    // dx[t][d] = sum_k dz[t][k] W[d][k]; thread: token t = tid / 8 ... (kTok * D outputs)
    for (int e = tid; e < n * D; e += kThreads) {
      const int t = e / D, d = e % D;
      const T* wr = wh + (size_t)d * DK;
      float s = 0.f;
      for (int k = 0; k < DK; k += 4) {
        const float4 wv = ld4(wr + k);
        s = fmaf(dzs[t * DK + k], wv.x, s);
        s = fmaf(dzs[t * DK + k + 1], wv.y, s);
        s = fmaf(dzs[t * DK + k + 2], wv.z, s);
        s = fmaf(dzs[t * DK + k + 3], wv.w, s);
      }
      dx[((size_t)bh * L + t0 + t) * D + d] = cvt_out<T>(s);
    }
    // dW[d][k] += sum_t x[t][d] dz[t][k], tokens in order
#pragma unroll
    for (int m = 0; m < kMaxAcc; ++m) {
      const int e = tid + kThreads * m;
      if (e < D * DK) {
        const int d = e / DK, k = e % DK;
        float s = dwa[m];
        for (int t = 0; t < kTok; ++t) s = fmaf(xs[t * (D + 1) + d], dzs[t * DK + k], s);
        dwa[m] = s;
      }
    }
    __syncthreads();
  }
  float* part = dw_part + ((size_t)bh * groups + g) * D * DK;
#pragma unroll
  for (int m = 0; m < kMaxAcc; ++m) {
    const int e = tid + kThreads * m;
    if (e < D * DK) part[e] = dwa[m];
  }
  pdl_trigger();
}

// dW[h] = sum over b, then groups, of the partials (fixed order).
__global__ void __launch_bounds__(256) gate_dw_kernel(int B, int H, int groups, int DDK,
                                                      const float* part, float* dw) {
  const int hh = blockIdx.y, e = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_wait();
  if (e < DDK) {
    float s = 0.f;
    for (int b = 0; b < B; ++b)
      for (int g = 0; g < groups; ++g) s += part[(((size_t)b * H + hh) * groups + g) * DDK + e];
    dw[(size_t)hh * DDK + e] = s;
  }
  pdl_trigger();
}

int gate_groups(int L) { return (L + kGroupTok - 1) / kGroupTok; }

template <typename T, int DK>
cudaError_t gate_fwd_t(int B, int H, int L, int D, float tau, const void* x, const void* w,
                       float* lg, cudaStream_t s) {
  const dim3 grid((L + kTok - 1) / kTok, B * H);
  return launch_pdl(gate_fwd_kernel<T, DK>, grid, dim3(kThreads), 0, s, H, L, D, 1.f / tau,
                    static_cast<const T*>(x), static_cast<const T*>(w), lg);
}

template <typename T, int DK>
cudaError_t gate_bwd_t(int B, int H, int L, int D, float tau, const void* x, const void* w,
                       const float* dlg, void* dx, float* part, cudaStream_t s) {
  const int groups = gate_groups(L);
  const size_t smem = ((size_t)kTok * (256 + 1) + (size_t)kDc * DK + (size_t)kTok * DK) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(gate_bwd_kernel<T, DK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(gate_bwd_kernel<T, DK>, dim3(groups, B * H), dim3(kThreads), smem, s, H, L, D,
                    groups, 1.f / tau, static_cast<const T*>(x), static_cast<const T*>(w), dlg,
                    static_cast<T*>(dx), part);
}

}  // namespace

size_t gate_bwd_workspace(int B, int H, int L, int D, int dk) {
  return (size_t)B * H * gate_groups(L) * D * dk * sizeof(float);
}

cudaError_t launch_gate_fwd(int B, int H, int L, int D, int dk, lizard_dtype dt, float tau,
                            const void* x, const void* w, float* lg, cudaStream_t s, int* launches) {
  if (L == 0) return cudaSuccess;
  trace_begin("gate_fwd", s);
  cudaError_t e;
  if (dt == LIZARD_F32)
    e = dk == 64 ? gate_fwd_t<float, 64>(B, H, L, D, tau, x, w, lg, s)
                 : gate_fwd_t<float, 128>(B, H, L, D, tau, x, w, lg, s);
  else
    e = dk == 64 ? gate_fwd_t<bf16, 64>(B, H, L, D, tau, x, w, lg, s)
                 : gate_fwd_t<bf16, 128>(B, H, L, D, tau, x, w, lg, s);
  trace_end(s);
  ++*launches;
  return e;
}

cudaError_t launch_gate_bwd(int B, int H, int L, int D, int dk, lizard_dtype dt, float tau,
                            const void* x, const void* w, const float* dlg, void* dx, float* dw,
                            unsigned char* ws, cudaStream_t s, int* launches) {
  if (L == 0) return cudaMemsetAsync(dw, 0, (size_t)H * D * dk * sizeof(float), s);
  float* part = reinterpret_cast<float*>(ws);
  trace_begin("gate_bwd", s);
  cudaError_t e;
  if (dt == LIZARD_F32)
    e = dk == 64 ? gate_bwd_t<float, 64>(B, H, L, D, tau, x, w, dlg, dx, part, s)
                 : gate_bwd_t<float, 128>(B, H, L, D, tau, x, w, dlg, dx, part, s);
  else
    e = dk == 64 ? gate_bwd_t<bf16, 64>(B, H, L, D, tau, x, w, dlg, dx, part, s)
                 : gate_bwd_t<bf16, 128>(B, H, L, D, tau, x, w, dlg, dx, part, s);
  trace_end(s);
  ++*launches;
  if (e != cudaSuccess) return e;
  const int DDK = D * dk;
  trace_begin("gate_dw", s);
  e = launch_pdl(gate_dw_kernel, dim3((DDK + 255) / 256, H), dim3(256), 0, s, B, H, gate_groups(L),
                 DDK, static_cast<const float*>(part), dw);
  trace_end(s);
  ++*launches;
  return e;
}

}  // namespace lz
