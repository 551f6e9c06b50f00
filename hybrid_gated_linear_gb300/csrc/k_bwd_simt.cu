// k_bwd_simt.cu -- backward pass on CUDA cores (fp32 FMA), any dtype.
//
// The pages give no backward formulas; these are the exact adjoints of the chunkwise
// forward (see k_fwd_simt.cu).  Per chunk (C tokens, b chunk-local cumsum, Gamma its
// last value, Qt = phi_q exp(b), Kt = phi_k exp(-b), h_prev the state at the chunk
// start, G the adjoint of the state at the chunk end coming from later chunks):
//   A[t][s] = dy_t . v_s,   P[t][s] = Qt_t . Kt_s          (s <= t)
//   dQt_t = h_prev dy_t + sum_{s<=t} A[t][s] Kt_s          d_phi_q = dQt * exp(b)
//   dKt_s = sum_{t>=s} A[t][s] Qt_t + exp(Gamma) (.) (G v_s)  d_phi_k = dKt * exp(-b)
//   dv_s  = sum_{t>=s} P[t][s] dy_t + (Kt_s (.) exp(Gamma))^T G
//   G    <- diag(exp(Gamma)) G + Qt^T dY                     (moving one chunk back)
//   d log_gamma_t = sum_{t'>=t} (phi_q (.) d_phi_q - phi_k (.) d_phi_k)_{t'}
// (the gate enters only through cumulative sums b, and d/db of Qt, Kt gives the
// per-token term).  After the walk G is the adjoint of h0.
//
// Window branch: textbook softmax backward in two deterministic kernels, one per
// query (dq, and the row statistics lse_i and D_i = dyw_i . y_win_i) and one per key
// (dk, dv, visiting the <= W queries that see the key); meta-key/value gradients are
// per-token terms reduced over (batch, token) in a fixed order.
#include <type_traits>

#include "lizard_dev.cuh"
#include "lizard_internal.h"

namespace lz {
namespace {

constexpr int kCB = 32;  // chunk of the backward walk
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct BwdWs {
  float* states;   // [BH][nc][DK][DV] state at the start of each chunk (CUDA-core path)
  unsigned char* gla_tc;  // scratch of the tensor-core GLA path
  float* dvacc;    // [BH][L][DV] GLA part of dv
  float* lse;      // [BH][L]
  float* Dw;       // [BH][L]
  float* ds_meta;  // [BH][L][M]
  float* p_meta;   // [BH][L][M]
  float* dmeta_part;  // [nsplit][H][M][DK+DV]
  float* mpart;       // per-block meta partials of the tensor-core window path
  int nsplit;
};

// Token splits of the meta-gradient reduction: a function of the tokens only, so that a
// head's sums do not depend on how many heads share the call.
inline int bwd_nsplit(int B, int H, int L) {
  (void)H;
  long tokens = (long)B * L;
  int ns = 128;
  if (ns > tokens) ns = (int)tokens;
  return ns < 1 ? 1 : ns;
}

// Window scratch and the GLA part of dv first, then the GLA path's own scratch: the
// chunk states (CUDA cores) or bwd_gla_tc_workspace bytes (tensor cores).
BwdWs carve(unsigned char* p, int B, int H, int L, int dk, int dv, int M, bool tc) {
  BwdWs w;
  const size_t BH = (size_t)B * H;
  const size_t nc = (L + kCB - 1) / kCB;
  size_t off = 0;
  auto take = [&](size_t floats) {
    float* r = reinterpret_cast<float*>(p + off);
    off += align_up(floats * sizeof(float) + 1, 256);
    return r;
  };
  w.dvacc = take(BH * (size_t)L * dv);
  w.lse = take(BH * (size_t)L);
  w.Dw = take(BH * (size_t)L);
  w.ds_meta = take(BH * (size_t)L * M);
  w.p_meta = take(BH * (size_t)L * M);
  w.nsplit = bwd_nsplit(B, H, L);
  w.dmeta_part = take((size_t)w.nsplit * H * M * (dk + dv));
  w.mpart = dk == 128 && dv == 128 ? take(bwd_win_tc_meta_floats((int)BH, L, M)) : nullptr;
  w.states = nullptr;
  w.gla_tc = nullptr;
  if (tc) w.gla_tc = p + off;
  else w.states = take(BH * nc * dk * dv);
  return w;
}

size_t carve_bytes(int B, int H, int L, int dk, int dv, int M) {
  const size_t BH = (size_t)B * H;
  const size_t nc = (L + kCB - 1) / kCB;
  size_t off = 0;
  auto take = [&](size_t floats) { off += align_up(floats * sizeof(float) + 1, 256); };
  take(BH * (size_t)L * dv);
  take(BH * (size_t)L);
  take(BH * (size_t)L);
  take(BH * (size_t)L * M);
  take(BH * (size_t)L * M);
  take((size_t)bwd_nsplit(B, H, L) * H * M * (dk + dv));
  if (dk == 128 && dv == 128) take(bwd_win_tc_meta_floats((int)BH, L, M));
  const size_t simt = align_up(BH * nc * dk * dv * sizeof(float) + 1, 256);
  const size_t tc = dk == 128 && dv == 128 && L > 0 ? bwd_gla_tc_workspace((int)BH, L) : 0;
  return off + (simt > tc ? simt : tc);
}

// ------------------------------------------------------------------------------------
// GLA adjoint: one CTA per (b, h), full state in shared memory.
// ------------------------------------------------------------------------------------
template <int DK, int DV>
constexpr size_t gla_bwd_smem_floats() {
  return 2 * (size_t)DK * (DV + 1)      // G, Hs
         + 3 * (size_t)kCB * (DK + 1)   // Qt, Kt, Eb
         + 2 * (size_t)kCB * (DV + 1)   // Vs, dYs
         + 2 * (size_t)kCB * (kCB + 1)  // A, P
         + DK;                          // exp(Gamma)
}

template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThreads) gla_bwd_kernel(BwdArgs a, BwdWs w) {
  extern __shared__ float sm[];
  float* G = sm;
  float* Hs = G + DK * (DV + 1);
  float* Qt = Hs + DK * (DV + 1);
  float* Kt = Qt + kCB * (DK + 1);
  float* Eb = Kt + kCB * (DK + 1);
  float* Vs = Eb + kCB * (DK + 1);
  float* dYs = Vs + kCB * (DV + 1);
  float* A = dYs + kCB * (DV + 1);
  float* P = A + kCB * (kCB + 1);
  float* eG = P + kCB * (kCB + 1);

  const int bh = blockIdx.x;
  const int tid = threadIdx.x;
  const int L = a.L;
  const int nc = (L + kCB - 1) / kCB;
  const T* pq = static_cast<const T*>(a.pq) + (size_t)bh * L * DK;
  const T* pk = static_cast<const T*>(a.pk) + (size_t)bh * L * DK;
  const T* vg = static_cast<const T*>(a.v) + (size_t)bh * L * DV;
  const T* dyg = static_cast<const T*>(a.dy) + (size_t)bh * L * DV;
  const float* lg = a.lg + (size_t)bh * L * DK;
  T* dpq = static_cast<T*>(a.dpq) + (size_t)bh * L * DK;
  T* dpk = static_cast<T*>(a.dpk) + (size_t)bh * L * DK;
  float* dlg = a.dlg + (size_t)bh * L * DK;
  float* states = w.states + (size_t)bh * nc * DK * DV;
  float* dvacc = w.dvacc + (size_t)bh * L * DV;

  // Loads chunk ch: cumsum, exp(+-b), features, values (and dy when want_dy).
  auto load_chunk = [&](int ch, bool want_dy) {
    const int t0 = ch * kCB;
    const int n = min(kCB, L - t0);
    if (tid < DK) {
      const int kk = tid;
      float run = 0.f;
      // eight tokens' loads in flight at a time
      for (int t8 = 0; t8 < kCB; t8 += 8) {
        float lv[8], qv[8], kv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const bool ok = t8 + i < n;
          const size_t idx = (size_t)(t0 + t8 + i) * DK + kk;
          lv[i] = ok ? lg[idx] : 0.f;
          qv[i] = ok ? ld_f(pq + idx) : 0.f;
          kv[i] = ok ? ld_f(pk + idx) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int t = t8 + i;
          run += lv[i];
          const float e = t < n ? expf(run) : 1.f;
          Qt[t * (DK + 1) + kk] = qv[i] * e;
          Kt[t * (DK + 1) + kk] = t < n ? kv[i] * expf(-run) : 0.f;
          Eb[t * (DK + 1) + kk] = e;
        }
      }
      eG[kk] = expf(run);
    }
    constexpr int kPer = kCB * DV / kThreads;  // elements per thread
    float vv[kPer], dd[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = tid + i * kThreads;
      const int t = e / DV, c = e % DV;
      const bool ok = t < n;
      vv[i] = ok ? ld_f(vg + (size_t)(t0 + t) * DV + c) : 0.f;
      dd[i] = (ok && want_dy) ? ld_f(dyg + (size_t)(t0 + t) * DV + c) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = tid + i * kThreads;
      const int t = e / DV, c = e % DV;
      Vs[t * (DV + 1) + c] = vv[i];
      if (want_dy) dYs[t * (DV + 1) + c] = dd[i];
    }
  };

  // Forward walk: record the state at the start of every chunk.
  for (int e = tid; e < DK * DV; e += kThreads) {
    const int r = e / DV, c = e % DV;
    Hs[r * (DV + 1) + c] = a.h0 ? a.h0[(size_t)bh * DK * DV + e] : 0.f;
  }
  __syncthreads();
  for (int ch = 0; ch < nc; ++ch) {
    {
      float4* dst = reinterpret_cast<float4*>(states + (size_t)ch * DK * DV);
      for (int e4 = tid; e4 < DK * DV / 4; e4 += kThreads) {
        const int e = 4 * e4, r = e / DV, c = e % DV;
        const float* src = Hs + r * (DV + 1) + c;
        dst[e4] = make_float4(src[0], src[1], src[2], src[3]);
      }
    }
    load_chunk(ch, false);
    __syncthreads();
    for (int e = tid; e < DK * DV; e += kThreads) {
      const int r = e / DV, c = e % DV;
      float acc = Hs[r * (DV + 1) + c];
      for (int s = 0; s < kCB; ++s) acc = fmaf(Kt[s * (DK + 1) + r], Vs[s * (DV + 1) + c], acc);
      Hs[r * (DV + 1) + c] = eG[r] * acc;
    }
    __syncthreads();
  }

  // Reverse walk.
  for (int e = tid; e < DK * DV; e += kThreads) G[(e / DV) * (DV + 1) + e % DV] = 0.f;
  float carry = 0.f;  // running suffix sum of the log-gate term (threads < DK)
  for (int ch = nc - 1; ch >= 0; --ch) {
    const int t0 = ch * kCB;
    const int n = min(kCB, L - t0);
    {
      // the saved state of this chunk: 16-byte loads, eight in flight per thread
      const float4* src = reinterpret_cast<const float4*>(states + (size_t)ch * DK * DV);
      constexpr int kN4 = DK * DV / 4 / kThreads;
#pragma unroll
      for (int b8 = 0; b8 < kN4; b8 += 8) {
        float4 r4[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) r4[i] = src[tid + (b8 + i) * kThreads];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int e = 4 * (tid + (b8 + i) * kThreads);
          const int r = e / DV, c = e % DV;
          float* dst = Hs + r * (DV + 1) + c;
          dst[0] = r4[i].x;
          dst[1] = r4[i].y;
          dst[2] = r4[i].z;
          dst[3] = r4[i].w;
        }
      }
    }
    load_chunk(ch, true);
    __syncthreads();

    // A = dY V^T, P = Qt Kt^T, both masked to s <= t.
    for (int e = tid; e < kCB * kCB; e += kThreads) {
      const int t = e / kCB, s = e % kCB;
      float x = 0.f, p = 0.f;
      if (s <= t) {
        for (int c = 0; c < DV; ++c) x = fmaf(dYs[t * (DV + 1) + c], Vs[s * (DV + 1) + c], x);
        for (int kk = 0; kk < DK; ++kk) p = fmaf(Qt[t * (DK + 1) + kk], Kt[s * (DK + 1) + kk], p);
      }
      A[t * (kCB + 1) + s] = x;
      P[t * (kCB + 1) + s] = p;
    }
    __syncthreads();

    // d_phi_q, d_phi_k, and the per-token log-gate term (stored over Eb).
    {
      constexpr int kRowsPerThread = kCB * DK / kThreads;
      constexpr int kRowStep = kThreads / DK;
      const int kk = tid % DK;
      const int r0 = tid / DK;
      float aq[kRowsPerThread], ak[kRowsPerThread];
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) aq[i] = ak[i] = 0.f;
      for (int c = 0; c < DV; ++c) {
        const float hv = Hs[kk * (DV + 1) + c];
        const float gv = G[kk * (DV + 1) + c];
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i) {
          const int t = r0 + kRowStep * i;
          aq[i] = fmaf(hv, dYs[t * (DV + 1) + c], aq[i]);
          ak[i] = fmaf(gv, Vs[t * (DV + 1) + c], ak[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        const int t = r0 + kRowStep * i;
        float q = aq[i], k = eG[kk] * ak[i];
        for (int s = 0; s <= t; ++s) q = fmaf(A[t * (kCB + 1) + s], Kt[s * (DK + 1) + kk], q);
        for (int u = t; u < kCB; ++u) k = fmaf(A[u * (kCB + 1) + t], Qt[u * (DK + 1) + kk], k);
        const float eb = Eb[t * (DK + 1) + kk];
        const float dphq = q * eb;
        const float dphk = k * __frcp_rn(eb);
        float term = 0.f;
        if (t < n) {
          const size_t idx = (size_t)(t0 + t) * DK + kk;
          dpq[idx] = cvt_out<T>(dphq);
          dpk[idx] = cvt_out<T>(dphk);
          term = ld_f(pq + idx) * dphq - ld_f(pk + idx) * dphk;
        }
        Eb[t * (DK + 1) + kk] = term;
      }
    }
    __syncthreads();
    if (tid < DK) {
      for (int t = n - 1; t >= 0; --t) {
        carry += Eb[t * (DK + 1) + tid];
        dlg[(size_t)(t0 + t) * DK + tid] = carry;
      }
    }

    // GLA part of dv.
    {
      constexpr int kRowsPerThread = kCB * DV / kThreads;
      constexpr int kRowStep = kThreads / DV;
      const int c = tid % DV;
      const int r0 = tid / DV;
      float acc[kRowsPerThread];
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) acc[i] = 0.f;
      for (int kk = 0; kk < DK; ++kk) {
        const float g = eG[kk] * G[kk * (DV + 1) + c];
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i)
          acc[i] = fmaf(Kt[(r0 + kRowStep * i) * (DK + 1) + kk], g, acc[i]);
      }
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        const int s = r0 + kRowStep * i;
        float x = acc[i];
        for (int t = s; t < kCB; ++t) x = fmaf(P[t * (kCB + 1) + s], dYs[t * (DV + 1) + c], x);
        if (s < n) dvacc[(size_t)(t0 + s) * DV + c] = x;
      }
    }
    __syncthreads();

    // Move the state adjoint to the start of this chunk.
    for (int e = tid; e < DK * DV; e += kThreads) {
      const int r = e / DV, c = e % DV;
      float acc = eG[r] * G[r * (DV + 1) + c];
      for (int t = 0; t < kCB; ++t) acc = fmaf(Qt[t * (DK + 1) + r], dYs[t * (DV + 1) + c], acc);
      G[r * (DV + 1) + c] = acc;
    }
    __syncthreads();
  }
  if (a.dh0) {
    for (int e = tid; e < DK * DV; e += kThreads)
      a.dh0[(size_t)bh * DK * DV + e] = G[(e / DV) * (DV + 1) + e % DV];
  }
}

// ------------------------------------------------------------------------------------
// Window adjoint, per query: dq, lse, D = dyw . y_win, meta terms.  Warp per query.
// ------------------------------------------------------------------------------------
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThreads) win_bwd_query_kernel(BwdArgs a, BwdWs w, int zcap) {
  extern __shared__ float sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* qs = sm + warp * (DK + DV + zcap);
  float* dys = qs + DK;
  float* z = dys + DV;  // logits, then probabilities, then ds
  const int bh = blockIdx.x;
  const int hh = bh % a.H;
  const int i = blockIdx.y * kWarps + warp;
  if (i >= a.L) return;
  const int L = a.L, M = a.M;
  const T* qg = static_cast<const T*>(a.q) + (size_t)bh * L * DK;
  const T* kg = static_cast<const T*>(a.k) + (size_t)bh * L * DK;
  const T* vg = static_cast<const T*>(a.v) + (size_t)bh * L * DV;
  const T* dyg = static_cast<const T*>(a.dy) + (size_t)bh * L * DV;
  const T* mk = M ? static_cast<const T*>(a.mk) + (size_t)hh * M * DK : nullptr;
  const T* mv = M ? static_cast<const T*>(a.mv) + (size_t)hh * M * DV : nullptr;

  for (int d = lane; d < DK; d += 32) qs[d] = ld_f(qg + (size_t)i * DK + d);
  for (int c = lane; c < DV; c += 32) dys[c] = a.alpha * ld_f(dyg + (size_t)i * DV + c);
  __syncwarp();
  const int j_lo = max(0, i - a.W + 1);
  const int nkeys = M + (i - j_lo + 1);
  auto key_of = [&](int j) { return (j < M) ? mk + (size_t)j * DK : kg + (size_t)(j_lo + j - M) * DK; };
  auto val_of = [&](int j) { return (j < M) ? mv + (size_t)j * DV : vg + (size_t)(j_lo + j - M) * DV; };

  float mx = -INFINITY;
  for (int j = lane; j < nkeys; j += 32) {
    const T* key = key_of(j);
    float d = 0.f;
    for (int e = 0; e < DK; e += 4) {
      const float4 kv = ld4(key + e);
      d = fmaf(qs[e], kv.x, d); d = fmaf(qs[e + 1], kv.y, d);
      d = fmaf(qs[e + 2], kv.z, d); d = fmaf(qs[e + 3], kv.w, d);
    }
    z[j] = d * a.scale;
    mx = fmaxf(mx, z[j]);
  }
  mx = warp_max(mx);
  float sum = 0.f;
  for (int j = lane; j < nkeys; j += 32) sum += expf(z[j] - mx);
  sum = warp_sum(sum);
  const float lse = mx + logf(sum);
  for (int j = lane; j < nkeys; j += 32) z[j] = expf(z[j] - lse);
  __syncwarp();
  // y_win columns (lanes take columns) and D = dyw . y_win.
  float dloc = 0.f;
  for (int c = lane; c < DV; c += 32) {
    float yc = 0.f;
    for (int j = 0; j < nkeys; ++j) yc = fmaf(z[j], ld_f(val_of(j) + c), yc);
    dloc = fmaf(dys[c], yc, dloc);
  }
  const float D = warp_sum(dloc);
  __syncwarp();
  // ds_j = p_j (dyw . value_j - D), in place.
  for (int j = lane; j < nkeys; j += 32) {
    const T* val = val_of(j);
    float dp = 0.f;
    for (int c = 0; c < DV; c += 4) {
      const float4 vv = ld4(val + c);
      dp = fmaf(dys[c], vv.x, dp); dp = fmaf(dys[c + 1], vv.y, dp);
      dp = fmaf(dys[c + 2], vv.z, dp); dp = fmaf(dys[c + 3], vv.w, dp);
    }
    const float p = z[j];
    if (j < M) w.p_meta[((size_t)bh * L + i) * M + j] = p;
    z[j] = p * (dp - D);
    if (j < M) w.ds_meta[((size_t)bh * L + i) * M + j] = z[j];
  }
  __syncwarp();
  for (int d = lane; d < DK; d += 32) {
    float acc = 0.f;
    for (int j = 0; j < nkeys; ++j) acc = fmaf(z[j], ld_f(key_of(j) + d), acc);
    static_cast<T*>(a.dq)[((size_t)bh * L + i) * DK + d] = cvt_out<T>(a.scale * acc);
  }
  if (lane == 0) {
    w.lse[(size_t)bh * L + i] = lse;
    w.Dw[(size_t)bh * L + i] = D;
  }
}

// ------------------------------------------------------------------------------------
// Window adjoint, per key j: dk_j and dv_j (plus the GLA part of dv).  Warp per key.
// ------------------------------------------------------------------------------------
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThreads) win_bwd_key_kernel(BwdArgs a, BwdWs w) {
  __shared__ float ks[kWarps][DK];
  __shared__ float vs[kWarps][DV];
  __shared__ float ps[kWarps][32];
  __shared__ float dss[kWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int j = blockIdx.y * kWarps + warp;
  if (j >= a.L) return;
  const int L = a.L;
  const T* qg = static_cast<const T*>(a.q) + (size_t)bh * L * DK;
  const T* kg = static_cast<const T*>(a.k) + (size_t)bh * L * DK;
  const T* vg = static_cast<const T*>(a.v) + (size_t)bh * L * DV;
  const T* dyg = static_cast<const T*>(a.dy) + (size_t)bh * L * DV;
  for (int d = lane; d < DK; d += 32) ks[warp][d] = ld_f(kg + (size_t)j * DK + d);
  for (int c = lane; c < DV; c += 32) vs[warp][c] = ld_f(vg + (size_t)j * DV + c);
  __syncwarp();
  const int i_hi = min(L - 1, j + a.W - 1);
  float dk_acc[DK / 32], dv_acc[DV / 32];
#pragma unroll
  for (int e = 0; e < DK / 32; ++e) dk_acc[e] = 0.f;
#pragma unroll
  for (int e = 0; e < DV / 32; ++e) dv_acc[e] = 0.f;
  for (int ib = j; ib <= i_hi; ib += 32) {
    const int i = ib + lane;
    float p = 0.f, ds = 0.f;
    if (i <= i_hi) {
      const T* qrow = qg + (size_t)i * DK;
      const T* dyrow = dyg + (size_t)i * DV;
      float zz = 0.f, dp = 0.f;
      for (int e = 0; e < DK; e += 4) {
        const float4 qv = ld4(qrow + e);
        zz = fmaf(qv.x, ks[warp][e], zz); zz = fmaf(qv.y, ks[warp][e + 1], zz);
        zz = fmaf(qv.z, ks[warp][e + 2], zz); zz = fmaf(qv.w, ks[warp][e + 3], zz);
      }
      for (int c = 0; c < DV; c += 4) {
        const float4 dv4 = ld4(dyrow + c);
        dp = fmaf(dv4.x, vs[warp][c], dp); dp = fmaf(dv4.y, vs[warp][c + 1], dp);
        dp = fmaf(dv4.z, vs[warp][c + 2], dp); dp = fmaf(dv4.w, vs[warp][c + 3], dp);
      }
      dp *= a.alpha;
      p = expf(zz * a.scale - w.lse[(size_t)bh * L + i]);
      ds = p * (dp - w.Dw[(size_t)bh * L + i]);
    }
    ps[warp][lane] = p;
    dss[warp][lane] = ds;
    __syncwarp();
    const int nb = min(32, i_hi - ib + 1);
    for (int u = 0; u < nb; ++u) {
      const int iq = ib + u;
      const float pu = ps[warp][u], du = dss[warp][u];
#pragma unroll
      for (int e = 0; e < DK / 32; ++e)
        dk_acc[e] = fmaf(du, ld_f(qg + (size_t)iq * DK + lane + 32 * e), dk_acc[e]);
#pragma unroll
      for (int e = 0; e < DV / 32; ++e)
        dv_acc[e] = fmaf(pu, ld_f(dyg + (size_t)iq * DV + lane + 32 * e), dv_acc[e]);
    }
    __syncwarp();
  }
#pragma unroll
  for (int e = 0; e < DK / 32; ++e)
    static_cast<T*>(a.dk_)[((size_t)bh * L + j) * DK + lane + 32 * e] = cvt_out<T>(a.scale * dk_acc[e]);
#pragma unroll
  for (int e = 0; e < DV / 32; ++e) {
    const size_t idx = ((size_t)bh * L + j) * DV + lane + 32 * e;
    static_cast<T*>(a.dvv)[idx] = cvt_out<T>(w.dvacc[idx] + a.alpha * dv_acc[e]);
  }
}

// ------------------------------------------------------------------------------------
// Meta gradients: per (head, token split) partial sums in a fixed order, then a final
// ordered sum over splits.
// ------------------------------------------------------------------------------------
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(128) dmeta_partial_kernel(BwdArgs a, BwdWs w) {
  const int hh = blockIdx.x, split = blockIdx.y;
  const int d = threadIdx.x;
  const int M = a.M, L = a.L;
  const long tokens = (long)a.B * L;
  const long per = (tokens + w.nsplit - 1) / w.nsplit;
  const long u0 = split * per, u1 = min(tokens, u0 + per);
  float ak[16], av[16];
#pragma unroll
  for (int m = 0; m < 16; ++m) ak[m] = av[m] = 0.f;
  for (long u = u0; u < u1; ++u) {
    const int b = (int)(u / L), i = (int)(u % L);
    const size_t bh = (size_t)b * a.H + hh;
    const size_t row = bh * L + i;
    const float qd = d < DK ? ld_f(static_cast<const T*>(a.q) + row * DK + d) : 0.f;
    const float dyd = d < DV ? a.alpha * ld_f(static_cast<const T*>(a.dy) + row * DV + d) : 0.f;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      if (m < M) {
        ak[m] = fmaf(w.ds_meta[row * M + m], qd, ak[m]);
        av[m] = fmaf(w.p_meta[row * M + m], dyd, av[m]);
      }
    }
  }
  float* part = w.dmeta_part + ((size_t)split * a.H + hh) * M * (DK + DV);
#pragma unroll
  for (int m = 0; m < 16; ++m) {
    if (m < M) {
      if (d < DK) part[m * (DK + DV) + d] = ak[m];
      if (d < DV) part[m * (DK + DV) + DK + d] = av[m];
    }
  }
}

template <int DK, int DV>
__global__ void dmeta_final_kernel(BwdArgs a, BwdWs w) {
  const int hh = blockIdx.x;
  const int M = a.M;
  for (int e = threadIdx.x; e < M * (DK + DV); e += blockDim.x) {
    float s = 0.f;
    for (int sp = 0; sp < w.nsplit; ++sp) s += w.dmeta_part[((size_t)sp * a.H + hh) * M * (DK + DV) + e];
    const int m = e / (DK + DV), d = e % (DK + DV);
    if (d < DK) a.dmk[((size_t)hh * M + m) * DK + d] = a.scale * s;
    else a.dmv[((size_t)hh * M + m) * DV + (d - DK)] = s;
  }
}

template <typename T, int D>
cudaError_t launch_typed(const BwdArgs& a, cudaStream_t s, int* launches) {
  constexpr lizard_dtype kDt = std::is_same<T, bf16>::value ? LIZARD_BF16 : LIZARD_F32;
  const bool tc = bwd_gla_tc_supported(D, D, a.L, kDt);
  BwdWs w = carve(a.ws, a.B, a.H, a.L, D, D, a.M, tc);
  const int BH = a.B * a.H;
  cudaError_t e;
  if (tc && bwd_win_tc_supported(D, D, a.L, a.W, a.M, kDt)) {
    // The query half of the window backward and the meta-gradient sum do not depend on the
    // GLA branch: they run on a second stream beside the GLA kernels.  The key half waits
    // for the GLA branch and the query half; the caller's stream waits for the meta sum
    // at the end.
    std::lock_guard<std::mutex> lock(side_stream_lock());
    SideStream* ss = side_stream();
    if (!ss) return cudaErrorNotReady;
    if ((e = cudaEventRecord(ss->fork, s)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(ss->stream, ss->fork, 0)) != cudaSuccess) return e;
    if ((e = launch_bwd_win_q_tc(a, w.dvacc, w.lse, w.Dw, w.mpart, ss->stream, launches)) != cudaSuccess)
      return e;
    if ((e = cudaEventRecord(ss->join, ss->stream)) != cudaSuccess) return e;
    if ((e = launch_bwd_win_meta_tc(a, w.mpart, ss->stream, launches)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(ss->done, ss->stream)) != cudaSuccess) return e;
    if ((e = launch_bwd_gla_tc(a, w.dvacc, w.gla_tc, s, launches)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(s, ss->join, 0)) != cudaSuccess) return e;
    if ((e = launch_bwd_win_k_tc(a, w.dvacc, w.lse, w.Dw, w.mpart, s, launches)) != cudaSuccess)
      return e;
    return cudaStreamWaitEvent(s, ss->done, 0);
  }
  if (tc) {
    if ((e = launch_bwd_gla_tc(a, w.dvacc, w.gla_tc, s, launches)) != cudaSuccess) return e;
  } else {
    const size_t smem = gla_bwd_smem_floats<D, D>() * sizeof(float);
    e = cudaFuncSetAttribute(gla_bwd_kernel<T, D, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    trace_begin("gla_bwd_simt", s);
    gla_bwd_kernel<T, D, D><<<BH, kThreads, smem, s>>>(a, w);
    trace_end(s);
    ++*launches;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (bwd_win_tc_supported(D, D, a.L, a.W, a.M, kDt)) {
    if ((e = launch_bwd_win_q_tc(a, w.dvacc, w.lse, w.Dw, w.mpart, s, launches)) != cudaSuccess) return e;
    if ((e = launch_bwd_win_meta_tc(a, w.mpart, s, launches)) != cudaSuccess) return e;
    return launch_bwd_win_k_tc(a, w.dvacc, w.lse, w.Dw, w.mpart, s, launches);
  }
  if (a.L > 0) {
    const int zcap = a.M + a.W + 1;
    const size_t smem = (size_t)kWarps * (2 * D + zcap) * sizeof(float);
    e = cudaFuncSetAttribute(win_bwd_query_kernel<T, D, D>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(BH, (a.L + kWarps - 1) / kWarps);
    trace_begin("win_bwd_query", s);
    win_bwd_query_kernel<T, D, D><<<grid, kThreads, smem, s>>>(a, w, zcap);
    trace_end(s);
    ++*launches;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    trace_begin("win_bwd_key", s);
    win_bwd_key_kernel<T, D, D><<<grid, kThreads, 0, s>>>(a, w);
    trace_end(s);
    ++*launches;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (a.M > 0) {
    if (a.L > 0) {
      trace_begin("dmeta_partial", s);
      dmeta_partial_kernel<T, D, D><<<dim3(a.H, w.nsplit), 128, 0, s>>>(a, w);
      trace_end(s);
      ++*launches;
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      trace_begin("dmeta_final", s);
      dmeta_final_kernel<D, D><<<a.H, 256, 0, s>>>(a, w);
      trace_end(s);
      ++*launches;
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    } else {
      e = cudaMemsetAsync(a.dmk, 0, sizeof(float) * a.H * a.M * D, s);
      if (e == cudaSuccess) e = cudaMemsetAsync(a.dmv, 0, sizeof(float) * a.H * a.M * D, s);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace

size_t bwd_simt_workspace(int B, int H, int L, int dk, int dv, int M) {
  return carve_bytes(B, H, L, dk, dv, M);
}

cudaError_t launch_bwd_simt(const BwdArgs& a, lizard_dtype dt, cudaStream_t s, int* launches) {
  if (dt == LIZARD_F32) {
    return a.dk == 64 ? launch_typed<float, 64>(a, s, launches)
                      : launch_typed<float, 128>(a, s, launches);
  }
  return a.dk == 64 ? launch_typed<bf16, 64>(a, s, launches)
                    : launch_typed<bf16, 128>(a, s, launches);
}

}  // namespace lz
