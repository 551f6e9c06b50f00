// k_fwd_simt.cu -- forward pass on CUDA cores (fp32 FMA), any dtype, and the exact
// recomputation of the tensor-core forward's "wide" chunks.
//
// GLA branch: the token recurrence itself (papernotes.org note on Lizard, 关键设计;
// "Lizard", arXiv 2507.09025, Preliminaries: recurrent form)
//   h_t = diag(gamma_t) h_{t-1} + phi_k_t v_t^T,   y_gla_t = phi_q_t^T h_t,
// with gamma_t = exp(log gamma_t) formed per token.  No cumulative product of gates is
// ever formed, so every finite gate gives a finite, exact-in-fp32 result however strong
// the decay.  One CTA per (b, h, 32 value columns): warp w carries state rows
// [w K, (w+1) K) (K = dk / 8) of the CTA's columns in registers, lane = value column;
// tokens are staged 64 at a time, each warp walks them without synchronising, and the
// per-warp partial readouts are summed after the walk.
//
// Window branch (papernotes.org note on Lizard, 关键设计: Anchor Window Attention): one
// warp per query, lanes take 32 keys at a time (the M meta keys first, then tokens
// [max(0, t-W+1), t]), online softmax with warp-shuffle max/sum, then lanes take the value
// columns.  y = y_gla + alpha * y_win, rounded once.
//
// The tensor-core forward (k_fwd_chunk_tc.cu) factorises the gate of a 128-token chunk as
// e^{+b} e^{-b}, which is exact only while e^{-b} stays finite; its prep pass lists the
// chunks where it does not ("wide" chunks).  fwd_wide_kernel recomputes every listed chunk
// here from the chunk-start state the bounded state scan left, and overwrites its y.
#include <type_traits>

#include "lizard_dev.cuh"
#include "lizard_internal.h"

namespace lz {
namespace {

constexpr int kC = 64;  // tokens staged per step
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kDVS = 32;  // value columns per CTA

// Shared-memory layout (floats).
template <int DK>
struct FsLayout {
  static constexpr int KPW = DK / kWarps;  // state rows per warp
  static constexpr int PQ = 0;                                // phi_q   [kC][DK]
  static constexpr int PK = PQ + kC * DK;                     // phi_k   [kC][DK]
  static constexpr int GM = PK + kC * DK;                     // gamma   [kC][DK]
  static constexpr int VS = GM + kC * DK;                     // v slice [kC][32]
  static constexpr int PART = VS + kC * kDVS;                 // [kC][kWarps][32] partial readouts
  static constexpr int QW = PART + kC * kWarps * kDVS;        // [kWarps][DK] query rows
  static constexpr int TOTAL = QW + kWarps * DK;
  static_assert(KPW % 4 == 0, "rows per warp");
  static_assert(2 * 64 * 128 <= kC * kWarps * kDVS, "feature-map weights fit the partials");
};

// One range of tokens of one (b, h) unit for the CTA's 32 value columns.
struct Range {
  int t_begin, t_end;
  const float* h0;        // fp32 [dk][dv] state before t_begin (null: zeros) ...
  const bf16* hc;         // ... or a bf16 [128][128] chunk-start state
  float* hf;              // fp32 [dk][dv] state after t_end - 1 (null: not written)
  bf16 *phq_out, *phk_out;  // [BH][L][dk]: phi_q, phi_k of the range written here (or null)
};

// phi_q and phi_k of tokens [t0, t0 + n) from the raw projections and the Hedgehog map,
// phi(x) = [exp(x W), exp(-x W)] (bf16 x [.., 128], W [128][64] per head), into the PQ
// and PK tiles (fp32).  The W tiles are staged in the PART region, which is free here.
template <int DK>
__device__ void load_phi_fmap(const FwdArgs& a, float* sm, int bh, int t0, int n) {
  using Lay = FsLayout<DK>;
  constexpr int kF = 64;
  const int tid = threadIdx.x, hh = bh % a.H;
  const bf16* xs[2] = {static_cast<const bf16*>(a.xq), static_cast<const bf16*>(a.xk)};
  const bf16* ws[2] = {static_cast<const bf16*>(a.wq), static_cast<const bf16*>(a.wk)};
  float* dst[2] = {sm + Lay::PQ, sm + Lay::PK};
  float* wsm = sm + Lay::PART;  // [2][128][64]
  for (int u = 0; u < 2; ++u) {
    const bf16* x = xs[u] + ((size_t)bh * a.L + t0) * 128;
    for (int e4 = tid; e4 < kC * 128 / 4; e4 += kThreads) {
      const int t = (4 * e4) / 128;
      const float4 v = t < n ? ld4(x + 4 * e4) : make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(dst[u] + 4 * e4) = v;  // x staged where phi goes
    }
    const bf16* w = ws[u] + (size_t)hh * 128 * kF;
    for (int e4 = tid; e4 < 128 * kF / 4; e4 += kThreads)
      *reinterpret_cast<float4*>(wsm + u * 128 * kF + 4 * e4) = ld4(w + 4 * e4);
  }
  __syncthreads();
  // thread: token t = tid / 4, features 16 (tid % 4) .. + 15 of both maps
  const int t = tid >> 2, f0 = (tid & 3) * 16;
  float z[2][16];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
#pragma unroll
    for (int f = 0; f < 16; ++f) z[u][f] = 0.f;
    const float* xr = dst[u] + t * 128;
    const float* wu = wsm + u * 128 * kF + f0;
    for (int d = 0; d < 128; ++d) {
      const float xv = xr[d];
#pragma unroll
      for (int f = 0; f < 16; f += 4) {
        const float4 wv = *reinterpret_cast<const float4*>(wu + d * kF + f);
        z[u][f] = fmaf(xv, wv.x, z[u][f]);
        z[u][f + 1] = fmaf(xv, wv.y, z[u][f + 1]);
        z[u][f + 2] = fmaf(xv, wv.z, z[u][f + 2]);
        z[u][f + 3] = fmaf(xv, wv.w, z[u][f + 3]);
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < 2; ++u) {
#pragma unroll
    for (int f = 0; f < 16; ++f) {
      const bool ok = t < n;
      dst[u][t * DK + f0 + f] = ok ? expf(z[u][f]) : 0.f;
      dst[u][t * DK + kF + f0 + f] = ok ? expf(-z[u][f]) : 0.f;
    }
  }
}

// The forward over tokens [r.t_begin, r.t_end) of unit bh for value columns
// [32 slice, 32 slice + 32): GLA by the recurrence, window, merge, store.
template <typename T, int DK>
__device__ void fwd_range(const FwdArgs& a, float* sm, int bh, int slice, const Range& r) {
  using Lay = FsLayout<DK>;
  constexpr int KPW = Lay::KPW;
  const int dv = a.dv, L = a.L;
  const int c0 = slice * kDVS;
  const int hh = bh % a.H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k0 = warp * KPW;  // this warp's first state row

  const T* pq = static_cast<const T*>(a.pq) + (size_t)bh * L * DK;
  const T* pk = static_cast<const T*>(a.pk) + (size_t)bh * L * DK;
  const T* qg = static_cast<const T*>(a.q) + (size_t)bh * L * DK;
  const T* kg = static_cast<const T*>(a.k) + (size_t)bh * L * DK;
  const T* vg = static_cast<const T*>(a.v) + (size_t)bh * L * dv;
  const float* lg = a.lg + (size_t)bh * L * DK;
  const T* mk = a.M ? static_cast<const T*>(a.mk) + (size_t)hh * a.M * DK : nullptr;
  const T* mv = a.M ? static_cast<const T*>(a.mv) + (size_t)hh * a.M * dv : nullptr;
  T* y = static_cast<T*>(a.y) + (size_t)bh * L * dv;

  float h[KPW];
#pragma unroll
  for (int j = 0; j < KPW; ++j) {
    const int k = k0 + j;
    h[j] = r.h0 ? r.h0[((size_t)bh * DK + k) * dv + c0 + lane]
         : r.hc ? __bfloat162float(r.hc[(size_t)k * 128 + c0 + lane])
                : 0.f;
  }

  for (int t0 = r.t_begin; t0 < r.t_end; t0 += kC) {
    const int n = min(kC, r.t_end - t0);

    // A: stage phi_q, phi_k (fp32), gamma = exp(log gamma) and the value slice.
    bool fmap = false;
    if constexpr (DK == 128 && std::is_same<T, bf16>::value) fmap = a.xq != nullptr;
    if (fmap) {
      if constexpr (DK == 128) load_phi_fmap<DK>(a, sm, bh, t0, n);
    } else {
      for (int e4 = tid; e4 < kC * DK / 4; e4 += kThreads) {
        const int t = (4 * e4) / DK;
        const size_t idx = (size_t)(t0 + t) * DK + (4 * e4) % DK;
        const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(sm + Lay::PQ + 4 * e4) = t < n ? ld4(pq + idx) : z4;
        *reinterpret_cast<float4*>(sm + Lay::PK + 4 * e4) = t < n ? ld4(pk + idx) : z4;
      }
    }
    for (int e4 = tid; e4 < kC * DK / 4; e4 += kThreads) {
      const int t = (4 * e4) / DK;
      float4 g = make_float4(1.f, 1.f, 1.f, 1.f);
      if (t < n) {
        const float4 l = *reinterpret_cast<const float4*>(lg + (size_t)(t0 + t) * DK + (4 * e4) % DK);
        g = make_float4(expf(l.x), expf(l.y), expf(l.z), expf(l.w));
      }
      *reinterpret_cast<float4*>(sm + Lay::GM + 4 * e4) = g;
    }
    for (int e = tid; e < kC * kDVS; e += kThreads) {
      const int t = e / kDVS, c = e % kDVS;
      sm[Lay::VS + e] = t < n ? ld_f(vg + (size_t)(t0 + t) * dv + c0 + c) : 0.f;
    }
    __syncthreads();

    // The features of a recomputed chunk are kept for a later backward (32 of the
    // dk columns per CTA).
    if (r.phq_out) {
      for (int e = tid; e < n * kDVS; e += kThreads) {
        const int t = e / kDVS, k = slice * kDVS + e % kDVS;
        const size_t o = ((size_t)bh * L + t0 + t) * DK + k;
        r.phq_out[o] = __float2bfloat16_rn(sm[Lay::PQ + t * DK + k]);
        r.phk_out[o] = __float2bfloat16_rn(sm[Lay::PK + t * DK + k]);
      }
    }

    // B: the recurrence; each warp walks all n tokens over its own state rows.
    for (int t = 0; t < n; ++t) {
      const float vt = sm[Lay::VS + t * kDVS + lane];
      const float* gq = sm + Lay::PQ + t * DK + k0;
      const float* gk = sm + Lay::PK + t * DK + k0;
      const float* gg = sm + Lay::GM + t * DK + k0;
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < KPW; j += 4) {
        const float4 g4 = *reinterpret_cast<const float4*>(gg + j);
        const float4 k4 = *reinterpret_cast<const float4*>(gk + j);
        const float4 q4 = *reinterpret_cast<const float4*>(gq + j);
        h[j] = fmaf(g4.x, h[j], k4.x * vt);
        h[j + 1] = fmaf(g4.y, h[j + 1], k4.y * vt);
        h[j + 2] = fmaf(g4.z, h[j + 2], k4.z * vt);
        h[j + 3] = fmaf(g4.w, h[j + 3], k4.w * vt);
        acc = fmaf(q4.x, h[j], acc);
        acc = fmaf(q4.y, h[j + 1], acc);
        acc = fmaf(q4.z, h[j + 2], acc);
        acc = fmaf(q4.w, h[j + 3], acc);
      }
      sm[Lay::PART + (t * kWarps + warp) * kDVS + lane] = acc;
    }
    __syncthreads();

    // C: window branch for rows t = warp + 8 i, the GLA readout summed over the warps'
    // partials in a fixed order, then the merged store.
    float* qs = sm + Lay::QW + warp * DK;
    for (int t = warp; t < n; t += kWarps) {
      const int tq = t0 + t;
      float o = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) o += sm[Lay::PART + (t * kWarps + w) * kDVS + lane];
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
      y[(size_t)tq * dv + c0 + lane] = cvt_out<T>(o + a.alpha * (acc / l_run));
      __syncwarp();
    }
    __syncthreads();
  }

  if (r.hf) {
#pragma unroll
    for (int j = 0; j < KPW; ++j) r.hf[((size_t)bh * DK + k0 + j) * dv + c0 + lane] = h[j];
  }
}

template <typename T, int DK>
__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(FwdArgs a) {
  extern __shared__ float sm[];
  const int nslice = a.dv / kDVS;
  const int bh = blockIdx.x / nslice, slice = blockIdx.x % nslice;
  const Range r{0, a.L, a.h0, nullptr, a.hf, nullptr, nullptr};
  fwd_range<T, DK>(a, sm, bh, slice, r);
}

// Wide chunks of the tensor-core forward: work item = (listed chunk, 32-column slice).
// When no chunk is listed every CTA returns after one load.
__global__ void __launch_bounds__(kThreads) fwd_wide_kernel(FwdArgs a, WideFix w) {
  extern __shared__ float sm[];
  pdl_wait();
  const int total = a.B * a.H * w.nc;  // the list's capacity
  const int items = (int)min(*w.count, (unsigned)total) * 4;
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int chunk = w.list[it >> 2], slice = it & 3;
    if (chunk < 0 || chunk >= total) continue;
    const int bh = chunk / w.nc, c = chunk % w.nc;
    const int tb = c * kGlaChunk, te = min(a.L, tb + kGlaChunk);
    const Range r{tb, te, nullptr, w.hs + (size_t)chunk * 128 * 128, nullptr, w.phq, w.phk};
    fwd_range<bf16, 128>(a, sm, bh, slice, r);
  }
  pdl_trigger();
}

template <typename T, int DK>
cudaError_t launch_typed(const FwdArgs& a, cudaStream_t s, int* launches) {
  const size_t smem = FsLayout<DK>::TOTAL * sizeof(float);
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

cudaError_t launch_fwd_wide_fix(const FwdArgs& a, const WideFix& w, cudaStream_t s, int* launches) {
  const size_t smem = FsLayout<128>::TOTAL * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(fwd_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int items = a.B * a.H * w.nc * 4;
  const int grid = items < ctas_per_wave(1) ? items : ctas_per_wave(1);
  trace_begin("fwd_wide_fix", s);
  e = launch_pdl(fwd_wide_kernel, dim3(grid), dim3(kThreads), smem, s, a, w);
  trace_end(s);
  ++*launches;
  return e;
}

}  // namespace lz
