// k_fwd_simt.cu -- forward pass on CUDA cores (fp32 FMA), any dtype.
//
// The exact-arithmetic path: it is the one used for fp32 inputs (no tf32 tensor
// cores, which could not meet a 1e-5 relative error) and for shapes the tensor-core
// kernels do not cover.
//
// GLA branch, chunkwise form of the recurrence ("Lizard", arXiv 2507.09025, Method:
// parallel form with cumulative gate products, absorbed into query/key features):
// per chunk of C tokens starting at t0, with b_t the chunk-local inclusive cumsum of
// log gamma and Gamma its last value,
//   Qt_t = phi_q_t * exp(b_t),  Kt_s = phi_k_s * exp(-b_s)
//   y_gla_t = Qt_t . h_prev + sum_{s<=t} (Qt_t . Kt_s) v_s
//   h_next  = diag(exp(Gamma)) (h_prev + Kt^T V)
// Window branch (papernotes.org note on Lizard, 关键设计: Anchor Window Attention):
// one warp per query, lanes take 32 keys at a time (M meta keys first, then tokens
// [max(0, t-W+1), t]), online softmax with warp-shuffle max/sum, then lanes take the
// value columns.  y = y_gla + alpha * y_win, rounded once.
//
// Grid: one CTA per (b, h, 32-column slice of dv); the state slice lives in shared
// memory for the whole walk over the chunks.
#include "lizard_dev.cuh"
#include "lizard_internal.h"

namespace lz {
namespace {

constexpr int kC = 64;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kDVS = 32;

template <int DK>
constexpr size_t fwd_simt_smem_floats() {
  return (size_t)DK * kDVS          // state slice
         + 2 * kC * (DK + 1)        // Qt, Kt
         + kC * kDVS                // V slice
         + kC * (kC + 1)            // S
         + DK                       // exp(Gamma)
         + kWarps * DK;             // per-warp query rows
}

template <typename T, int DK>
__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(FwdArgs a) {
  extern __shared__ float sm[];
  float* hs = sm;
  float* Qt = hs + DK * kDVS;
  float* Kt = Qt + kC * (DK + 1);
  float* Vs = Kt + kC * (DK + 1);
  float* S = Vs + kC * kDVS;
  float* eG = S + kC * (kC + 1);
  float* qw = eG + DK;

  const int dv = a.dv;
  const int nslice = dv / kDVS;
  const int bh = blockIdx.x / nslice;
  const int c0 = (blockIdx.x % nslice) * kDVS;
  const int hh = bh % a.H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = a.L;

  const T* pq = static_cast<const T*>(a.pq) + (size_t)bh * L * DK;
  const T* pk = static_cast<const T*>(a.pk) + (size_t)bh * L * DK;
  const T* qg = static_cast<const T*>(a.q) + (size_t)bh * L * DK;
  const T* kg = static_cast<const T*>(a.k) + (size_t)bh * L * DK;
  const T* vg = static_cast<const T*>(a.v) + (size_t)bh * L * dv;
  const float* lg = a.lg + (size_t)bh * L * DK;
  const T* mk = a.M ? static_cast<const T*>(a.mk) + (size_t)hh * a.M * DK : nullptr;
  const T* mv = a.M ? static_cast<const T*>(a.mv) + (size_t)hh * a.M * dv : nullptr;
  T* y = static_cast<T*>(a.y) + (size_t)bh * L * dv;

  for (int e = tid; e < DK * kDVS; e += kThreads) {
    const int r = e / kDVS, c = e % kDVS;
    hs[e] = a.h0 ? a.h0[((size_t)bh * DK + r) * dv + c0 + c] : 0.f;
  }
  __syncthreads();

  const int nchunks = (L + kC - 1) / kC;
  for (int ch = 0; ch < nchunks; ++ch) {
    const int t0 = ch * kC;
    const int n = min(kC, L - t0);

    // A: chunk-local cumsum of log gamma; absorb exp(+-b) into the features.
    if (tid < DK) {
      const int kk = tid;
      float run = 0.f;
#pragma unroll 4
      for (int t = 0; t < kC; ++t) {
        float qv = 0.f, kv = 0.f;
        if (t < n) {
          const size_t idx = (size_t)(t0 + t) * DK + kk;
          run += lg[idx];
          qv = ld_f(pq + idx) * expf(run);
          kv = ld_f(pk + idx) * expf(-run);
        }
        Qt[t * (DK + 1) + kk] = qv;
        Kt[t * (DK + 1) + kk] = kv;
      }
      eG[kk] = expf(run);
    } else {
      for (int e = tid - DK; e < kC * kDVS; e += kThreads - DK) {
        const int t = e / kDVS, c = e % kDVS;
        Vs[e] = (t < n) ? ld_f(vg + (size_t)(t0 + t) * dv + c0 + c) : 0.f;
      }
    }
    __syncthreads();

    // B: S = (Qt Kt^T) masked to s <= t.
    {
      const int ty = tid >> 4, tx = tid & 15;
      float acc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
      for (int kk = 0; kk < DK; ++kk) {
        float qa[4], kb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) qa[i] = Qt[(ty + 16 * i) * (DK + 1) + kk];
#pragma unroll
        for (int j = 0; j < 4; ++j) kb[j] = Kt[(tx + 16 * j) * (DK + 1) + kk];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(qa[i], kb[j], acc[i][j]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int t = ty + 16 * i, s = tx + 16 * j;
          S[t * (kC + 1) + s] = (s <= t) ? acc[i][j] : 0.f;
        }
    }
    __syncthreads();

    // C: O = S V + Qt h_prev for rows t = warp + 8 i, column c0 + lane.
    float o[kC / kWarps];
#pragma unroll
    for (int i = 0; i < kC / kWarps; ++i) o[i] = 0.f;
    for (int s = 0; s < kC; ++s) {
      const float vsc = Vs[s * kDVS + lane];
#pragma unroll
      for (int i = 0; i < kC / kWarps; ++i) o[i] = fmaf(S[(warp + kWarps * i) * (kC + 1) + s], vsc, o[i]);
    }
    for (int kk = 0; kk < DK; ++kk) {
      const float hv = hs[kk * kDVS + lane];
#pragma unroll
      for (int i = 0; i < kC / kWarps; ++i) o[i] = fmaf(Qt[(warp + kWarps * i) * (DK + 1) + kk], hv, o[i]);
    }
    __syncthreads();

    // D: h_next = diag(exp(Gamma)) (h_prev + Kt^T V).
    for (int i = 0; i < DK / kWarps; ++i) {
      const int kk = warp + kWarps * i;
      float acc = hs[kk * kDVS + lane];
      for (int s = 0; s < kC; ++s) acc = fmaf(Kt[s * (DK + 1) + kk], Vs[s * kDVS + lane], acc);
      hs[kk * kDVS + lane] = eG[kk] * acc;
    }

    // E: window branch for the same rows, then the merged store.
    float* qs = qw + warp * DK;
    for (int i = 0; i < kC / kWarps; ++i) {
      const int t = warp + kWarps * i;
      if (t >= n) break;
      const int tq = t0 + t;
      for (int d = lane; d < DK; d += 32) qs[d] = ld_f(qg + (size_t)tq * DK + d);
      __syncwarp();
      const int j_lo = max(0, tq - a.W + 1);
      const int nkeys = a.M + (tq - j_lo + 1);
      float m_run = -INFINITY, l_run = 0.f, acc = 0.f;
      for (int kb = 0; kb < nkeys; kb += 32) {
        const int j = kb + lane;
        float z = -INFINITY;
        if (j < nkeys) {
          const T* key = (j < a.M) ? mk + (size_t)j * DK : kg + (size_t)(j_lo + j - a.M) * DK;
          float d = 0.f;
#pragma unroll 8
          for (int e = 0; e < DK; e += 4) {
            const float4 kv = ld4(key + e);
            d = fmaf(qs[e], kv.x, d);
            d = fmaf(qs[e + 1], kv.y, d);
            d = fmaf(qs[e + 2], kv.z, d);
            d = fmaf(qs[e + 3], kv.w, d);
          }
          z = d * a.scale;
        }
        const float m_new = fmaxf(m_run, warp_max(z));
        const float p = (j < nkeys) ? expf(z - m_new) : 0.f;
        const float corr = (m_run == -INFINITY) ? 0.f : expf(m_run - m_new);
        l_run = l_run * corr + warp_sum(p);
        acc *= corr;
        const int nb = min(32, nkeys - kb);
        for (int jj = 0; jj < nb; ++jj) {
          const float pj = __shfl_sync(0xffffffffu, p, jj);
          const int ja = kb + jj;
          const T* vrow = (ja < a.M) ? mv + (size_t)ja * dv : vg + (size_t)(j_lo + ja - a.M) * dv;
          acc = fmaf(pj, ld_f(vrow + c0 + lane), acc);
        }
        m_run = m_new;
      }
      y[(size_t)tq * dv + c0 + lane] = cvt_out<T>(o[i] + a.alpha * (acc / l_run));
      __syncwarp();
    }
    __syncthreads();
  }

  if (a.hf) {
    for (int e = tid; e < DK * kDVS; e += kThreads) {
      const int r = e / kDVS, c = e % kDVS;
      a.hf[((size_t)bh * DK + r) * dv + c0 + c] = hs[e];
    }
  }
}

template <typename T, int DK>
cudaError_t launch_typed(const FwdArgs& a, cudaStream_t s, int* launches) {
  const size_t smem = fwd_simt_smem_floats<DK>() * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(fwd_simt_kernel<T, DK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = a.B * a.H * (a.dv / kDVS);
  trace_begin("fwd_simt", s);
  fwd_simt_kernel<T, DK><<<grid, kThreads, smem, s>>>(a);
  trace_end(s);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt(const FwdArgs& a, lizard_dtype dt, cudaStream_t s, int* launches) {
  if (dt == LIZARD_F32) {
    return a.dk == 64 ? launch_typed<float, 64>(a, s, launches)
                      : launch_typed<float, 128>(a, s, launches);
  }
  return a.dk == 64 ? launch_typed<bf16, 64>(a, s, launches)
                    : launch_typed<bf16, 128>(a, s, launches);
}

}  // namespace lz
