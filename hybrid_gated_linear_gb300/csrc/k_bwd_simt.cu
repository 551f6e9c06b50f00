// k_bwd_simt.cu -- backward pass on CUDA cores (fp32 FMA), any dtype, and the exact
// recomputation of the tensor-core backward's "wide" chunks.
//
// The pages give no backward formulas; these are the exact adjoints of the recurrence
// the forward computes (papernotes.org note on Lizard, 关键设计;
// "Lizard", arXiv 2507.09025, Preliminaries: recurrent form)
//   h_t = diag(gamma_t) h_{t-1} + phi_k_t v_t^T,   y_t = phi_q_t^T h_t,   gamma_t = e^{log gamma_t}.
// GLA branch, one CTA per (b, h) with the whole dk x dv state in registers (warp w: state
// rows [w K, (w+1) K), K = dk / 16; lane: value columns lane + 32 j), two walks:
//   forward:  h_t as above;                      d phi_q_t = h_t dy_t
//   reverse:  dh_t = phi_q_t dy_t^T + diag(gamma_{t+1}) dh_{t+1}   (dh after the last
//             token = 0, or the adjoint coming from later tokens);
//             d phi_k_t = dh_t v_t,   dv_t = dh_t^T phi_k_t (the GLA part of dv)
//   d log gamma_t = sum_{t' >= t} (phi_q (.) d phi_q - phi_k (.) d phi_k)_{t'}
// The last line holds because log gamma_t enters every later state only through the
// cumulative log decay, which multiplies the query side by e^{+sum} and the key side by
// e^{-sum}.  Every factor is a gate in (0, 1] or an input: the result is finite for every
// finite gate.  The adjoint of h0 is dh before token 0.  Reductions over the value
// columns run inside a warp (shuffles in a fixed pattern), over the state rows through
// shared memory in a fixed order, so every result is run-to-run deterministic.
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

constexpr int kThreads = 256;  // window kernels
constexpr int kWarps = kThreads / 32;

constexpr int kSub = 32;  // tokens per checkpoint of the GLA adjoint's forward walk

// Scratch of one GLA adjoint walker (floats): the state at every kSub-th token of its range
// and the kSub states of the sub-range the reverse walk is in.
__host__ __device__ inline size_t walk_scratch_floats(int D, int tokens) {
  return ((size_t)(tokens + kSub - 1) / kSub + kSub) * D * D;
}

struct BwdWs {
  unsigned char* gla_tc;  // scratch of the tensor-core GLA path
  float* dvacc;    // [BH][L][DV] GLA part of dv
  float* lse;      // [BH][L]
  float* Dw;       // [BH][L]
  float* ds_meta;  // [BH][L][M]
  float* p_meta;   // [BH][L][M]
  float* dmeta_part;  // [nsplit][H][M][DK+DV]
  float* mpart;       // per-block meta partials of the tensor-core window path
  float* walk;        // scratch of the CUDA-core GLA walks (checkpoints and sub-range states)
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

// Window scratch and the GLA part of dv first, then the tensor-core GLA path's scratch.
BwdWs carve(unsigned char* p, int B, int H, int L, int dk, int dv, int M, bool tc) {
  BwdWs w;
  const size_t BH = (size_t)B * H;
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
  w.gla_tc = tc ? p + off : nullptr;
  w.walk = tc ? nullptr : take(BH * walk_scratch_floats(dk, L));
  return w;
}

size_t carve_bytes(int B, int H, int L, int dk, int dv, int M) {
  const size_t BH = (size_t)B * H;
  size_t off = 0;
  auto take = [&](size_t floats) { off += align_up(floats * sizeof(float) + 1, 256); };
  take(BH * (size_t)L * dv);
  take(BH * (size_t)L);
  take(BH * (size_t)L);
  take(BH * (size_t)L * M);
  take(BH * (size_t)L * M);
  take((size_t)bwd_nsplit(B, H, L) * H * M * (dk + dv));
  if (dk == 128 && dv == 128) take(bwd_win_tc_meta_floats((int)BH, L, M));
  const size_t tc = dk == 128 && dv == 128 && L > 0 ? bwd_gla_tc_workspace((int)BH, L) : 0;
  const size_t simt = align_up(BH * walk_scratch_floats(dk, L) * sizeof(float) + 1, 256);
  return off + (tc > simt ? tc : simt);
}

// ------------------------------------------------------------------------------------
// GLA adjoint by the recurrence: one CTA of 512 threads per (b, h) (or per wide chunk).
// ------------------------------------------------------------------------------------
constexpr int kGThreads = 512;
constexpr int kGWarps = kGThreads / 32;
constexpr int kTB = 8;    // tokens staged per step

template <int D>
struct GbLayout {
  static constexpr int KPW = D / kGWarps;  // state rows per warp: 8 or 4
  static constexpr int VPL = D / 32;       // value columns per lane: 4 or 2
  // floats
  static constexpr int PQ = 0, PK = PQ + kTB * D, GM = PK + kTB * D, VS = GM + kTB * D,
                       DY = VS + kTB * D, PV = DY + kTB * D;  // PV: [kTB][kGWarps][D]
  static constexpr int TOTAL = PV + kTB * kGWarps * D;
  static_assert(KPW == 4 || KPW == 8, "rows per warp");
};

// Sum over the 32 lanes of each of the R values every lane holds (R = 4 or 8), in a fixed
// butterfly pattern.  Returns, in every lane, the total of row row_of_lane(lane).
template <int R>
__device__ __forceinline__ float warp_sum_rows(float (&v)[R]) {
  const int lane = threadIdx.x & 31;
  float w[R];
#pragma unroll
  for (int m = 0; m < R; ++m) w[m] = v[m];
  int off = 16;
#pragma unroll
  for (int n = R; n > 1; n >>= 1, off >>= 1) {
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int m = 0; m < n / 2; ++m) {
      const float send = up ? w[m] : w[m + n / 2];
      const float keep = up ? w[m + n / 2] : w[m];
      w[m] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float x = w[0];
  for (; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// The row (0 .. R-1) whose total warp_sum_rows leaves in `lane`; lanes with
// lane % (32 / R) == 0 hold each row once.
template <int R>
__device__ __forceinline__ int row_of_lane(int lane) {
  return R == 8 ? ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1)
                : ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
}

// What one pair of walks covers: tokens [t_begin, t_end) of unit bh.
template <typename T>
struct GlaWalk {
  int t_begin, t_end;
  const T *pq, *pk;          // [BH][L][D] features
  const float* h_init;       // fp32 [D][D] state before t_begin (null: zeros) ...
  const bf16* hb_init;       // ... or bf16 [128][128]
  const bf16* gb_init;       // bf16 [128][128] adjoint after t_end - 1 (null: zeros)
  float* dh_out;             // fp32 [D][D]: adjoint of the state before t_begin (or null)
  float* rtot;               // [D]: the range's total of the per-token log-gate term
                             // phi_q (.) d phi_q - phi_k (.) d phi_k (or null)
  float* scratch;            // walk_scratch_floats(D, t_end - t_begin) floats
};

// d log gamma_t = gamma_t <dh_t, h_{t-1}> row by row (the adjoint of h_t against the state
// before token t): no cancellation between large terms, so the result keeps its relative
// accuracy however small gamma is.  h_{t-1} comes from a second forward pass over each
// kSub-token sub-range, started from the checkpoint the first forward walk left and
// written to scratch; every scratch element is written and read back by the same thread.
template <typename T, int D>
__device__ void gla_bwd_walks(const BwdArgs& a, float* sm, int bh, const GlaWalk<T>& g,
                              float* dvacc) {
  using Lay = GbLayout<D>;
  constexpr int KPW = Lay::KPW, VPL = Lay::VPL;
  constexpr size_t kS = (size_t)D * D;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = a.L, k0 = warp * KPW;
  const int myrow = row_of_lane<KPW>(lane);
  const bool writer = (lane % (32 / KPW)) == 0;  // holds row myrow's total
  const int kw = k0 + myrow;
  const T* pq = g.pq + (size_t)bh * L * D;
  const T* pk = g.pk + (size_t)bh * L * D;
  const T* vg = static_cast<const T*>(a.v) + (size_t)bh * L * D;
  const T* dyg = static_cast<const T*>(a.dy) + (size_t)bh * L * D;
  const float* lg = a.lg + (size_t)bh * L * D;
  T* dpq = static_cast<T*>(a.dpq) + (size_t)bh * L * D;
  T* dpk = static_cast<T*>(a.dpk) + (size_t)bh * L * D;
  float* dlg = a.dlg + (size_t)bh * L * D;
  float* dva = dvacc + (size_t)bh * L * D;
  const int nsub = (g.t_end - g.t_begin + kSub - 1) / kSub;
  float* ckpt = g.scratch;                    // [nsub][D][D]
  float* subst = g.scratch + (size_t)nsub * kS;  // [kSub][D][D]
  // element (i, j) of this thread in a [D][D] state
  auto eo = [&](int i, int j) { return (size_t)(k0 + i) * D + lane + 32 * j; };

  // tokens [t0, t0 + n) into shared memory (fp32; gamma = exp(log gamma))
  auto stage = [&](int t0, int n) {
    for (int e4 = tid; e4 < kTB * D / 4; e4 += kGThreads) {
      const int t = (4 * e4) / D;
      const size_t idx = (size_t)(t0 + t) * D + (4 * e4) % D;
      const bool ok = t < n;
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(sm + Lay::PQ + 4 * e4) = ok ? ld4(pq + idx) : z;
      *reinterpret_cast<float4*>(sm + Lay::PK + 4 * e4) = ok ? ld4(pk + idx) : z;
      *reinterpret_cast<float4*>(sm + Lay::VS + 4 * e4) = ok ? ld4(vg + idx) : z;
      *reinterpret_cast<float4*>(sm + Lay::DY + 4 * e4) = ok ? ld4(dyg + idx) : z;
      float4 gm = make_float4(1.f, 1.f, 1.f, 1.f);
      if (ok) {
        const float4 l = *reinterpret_cast<const float4*>(lg + idx);
        gm = make_float4(expf(l.x), expf(l.y), expf(l.z), expf(l.w));
      }
      *reinterpret_cast<float4*>(sm + Lay::GM + 4 * e4) = gm;
    }
  };
  // h <- diag(gamma_t) h + phi_k_t v_t^T for staged token t
  auto advance = [&](float (&h)[KPW][VPL], int t) {
    float vv[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j) vv[j] = sm[Lay::VS + t * D + lane + 32 * j];
#pragma unroll
    for (int i = 0; i < KPW; i += 4) {
      const float4 g4 = *reinterpret_cast<const float4*>(sm + Lay::GM + t * D + k0 + i);
      const float4 k4 = *reinterpret_cast<const float4*>(sm + Lay::PK + t * D + k0 + i);
      const float gg[4] = {g4.x, g4.y, g4.z, g4.w}, kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int j = 0; j < VPL; ++j) h[i + u][j] = fmaf(gg[u], h[i + u][j], kk[u] * vv[j]);
    }
  };

  float x[KPW][VPL];
  // ---- forward walk: d phi_q_t = h_t dy_t (and phi_q_t (.) d phi_q_t parked in
  //      d log gamma_t); the state before every kSub-th token goes to the checkpoints
#pragma unroll
  for (int i = 0; i < KPW; ++i)
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      x[i][j] = g.h_init ? g.h_init[eo(i, j)]
              : g.hb_init ? __bfloat162float(g.hb_init[(size_t)(k0 + i) * 128 + lane + 32 * j])
                          : 0.f;
  for (int t0 = g.t_begin; t0 < g.t_end; t0 += kTB) {
    const int n = min(kTB, g.t_end - t0);
    if ((t0 - g.t_begin) % kSub == 0) {
      float* cp = ckpt + (size_t)((t0 - g.t_begin) / kSub) * kS;
#pragma unroll
      for (int i = 0; i < KPW; ++i)
#pragma unroll
        for (int j = 0; j < VPL; ++j) cp[eo(i, j)] = x[i][j];
    }
    __syncthreads();
    stage(t0, n);
    __syncthreads();
    for (int t = 0; t < n; ++t) {
      advance(x, t);
      float dd[VPL], part[KPW];
#pragma unroll
      for (int j = 0; j < VPL; ++j) dd[j] = sm[Lay::DY + t * D + lane + 32 * j];
#pragma unroll
      for (int i = 0; i < KPW; ++i) {
        float p = 0.f;
#pragma unroll
        for (int j = 0; j < VPL; ++j) p = fmaf(x[i][j], dd[j], p);
        part[i] = p;
      }
      const float dq = warp_sum_rows<KPW>(part);
      if (writer) {
        const size_t o = (size_t)(t0 + t) * D + kw;
        dpq[o] = cvt_out<T>(dq);
        dlg[o] = sm[Lay::PQ + t * D + kw] * dq;
      }
    }
  }

  // ---- reverse walk, one sub-range of kSub tokens at a time from the last
#pragma unroll
  for (int i = 0; i < KPW; ++i)
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      x[i][j] = g.gb_init ? __bfloat162float(g.gb_init[(size_t)(k0 + i) * 128 + lane + 32 * j]) : 0.f;
  float rsum = 0.f;  // the range's total of the log-gate term for row kw (writer lanes)
  for (int sb = nsub - 1; sb >= 0; --sb) {
    const int c0 = g.t_begin + sb * kSub, cn = min(kSub, g.t_end - c0);
    // states before each token of the sub-range: subst[u] = h_{c0 + u - 1}
    {
      float h[KPW][VPL];
      const float* cp = ckpt + (size_t)sb * kS;
#pragma unroll
      for (int i = 0; i < KPW; ++i)
#pragma unroll
        for (int j = 0; j < VPL; ++j) h[i][j] = cp[eo(i, j)];
      for (int t0 = c0; t0 < c0 + cn; t0 += kTB) {
        const int n = min(kTB, c0 + cn - t0);
        __syncthreads();
        stage(t0, n);
        __syncthreads();
        for (int t = 0; t < n; ++t) {
          float* st = subst + (size_t)(t0 - c0 + t) * kS;
#pragma unroll
          for (int i = 0; i < KPW; ++i)
#pragma unroll
            for (int j = 0; j < VPL; ++j) st[eo(i, j)] = h[i][j];
          if (t0 - c0 + t + 1 < cn) advance(h, t);
        }
      }
    }
    const int nblk = (cn + kTB - 1) / kTB;
    for (int b = nblk - 1; b >= 0; --b) {
      const int t0 = c0 + b * kTB;
      const int n = min(kTB, c0 + cn - t0);
      __syncthreads();
      stage(t0, n);
      __syncthreads();
      for (int t = n - 1; t >= 0; --t) {
        const float* hp = subst + (size_t)(t0 - c0 + t) * kS;  // h_{t-1}
        float vv[VPL], dd[VPL], part[KPW], pg[KPW], pv[VPL];
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          vv[j] = sm[Lay::VS + t * D + lane + 32 * j];
          dd[j] = sm[Lay::DY + t * D + lane + 32 * j];
          pv[j] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < KPW; i += 4) {
          const float4 q4 = *reinterpret_cast<const float4*>(sm + Lay::PQ + t * D + k0 + i);
          const float4 k4 = *reinterpret_cast<const float4*>(sm + Lay::PK + t * D + k0 + i);
          const float qq[4] = {q4.x, q4.y, q4.z, q4.w}, kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float p = 0.f, q = 0.f;
#pragma unroll
            for (int j = 0; j < VPL; ++j) {
              x[i + u][j] = fmaf(qq[u], dd[j], x[i + u][j]);
              p = fmaf(x[i + u][j], vv[j], p);
              q = fmaf(x[i + u][j], hp[eo(i + u, j)], q);
              pv[j] = fmaf(x[i + u][j], kk[u], pv[j]);
            }
            part[i + u] = p;
            pg[i + u] = q;
          }
        }
#pragma unroll
        for (int j = 0; j < VPL; ++j) sm[Lay::PV + (t * kGWarps + warp) * D + lane + 32 * j] = pv[j];
        const float dk = warp_sum_rows<KPW>(part);
        const float dg = warp_sum_rows<KPW>(pg);
        if (writer) {
          const size_t o = (size_t)(t0 + t) * D + kw;
          dpk[o] = cvt_out<T>(dk);
          rsum += dlg[o] - sm[Lay::PK + t * D + kw] * dk;
          dlg[o] = sm[Lay::GM + t * D + kw] * dg;
        }
        // move the adjoint to the state before token t
#pragma unroll
        for (int i = 0; i < KPW; i += 4) {
          const float4 g4 = *reinterpret_cast<const float4*>(sm + Lay::GM + t * D + k0 + i);
          const float gg[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int j = 0; j < VPL; ++j) x[i + u][j] *= gg[u];
        }
      }
      __syncthreads();
      // the GLA part of dv: the warps' partials summed in a fixed order
      for (int e = tid; e < n * D; e += kGThreads) {
        const int t = e / D, c = e % D;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kGWarps; ++w) s += sm[Lay::PV + (t * kGWarps + w) * D + c];
        dva[(size_t)(t0 + t) * D + c] = s;
      }
    }
  }
  if (g.rtot && writer) g.rtot[kw] = rsum;
  if (g.dh_out) {
#pragma unroll
    for (int i = 0; i < KPW; ++i)
#pragma unroll
      for (int j = 0; j < VPL; ++j) g.dh_out[eo(i, j)] = x[i][j];
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kGThreads) gla_bwd_kernel(BwdArgs a, float* dvacc, float* scratch) {
  extern __shared__ float sm[];
  const int bh = blockIdx.x;
  GlaWalk<T> g{0, a.L, static_cast<const T*>(a.pq), static_cast<const T*>(a.pk),
               a.h0 ? a.h0 + (size_t)bh * D * D : nullptr, nullptr, nullptr,
               a.dh0 ? a.dh0 + (size_t)bh * D * D : nullptr, nullptr,
               scratch + (size_t)bh * walk_scratch_floats(D, a.L)};
  gla_bwd_walks<T, D>(a, sm, bh, g, dvacc);
}

// Wide chunks of the tensor-core backward: one listed chunk per CTA iteration, from the
// chunk-start state and the unscaled end-of-chunk adjoint the scans left.  d log gamma of
// the chunk's tokens is final (the suffix pass skips wide chunks); the chunk's total of
// the log-gate term goes to rtot for the earlier chunks' suffix sums.
__global__ void __launch_bounds__(kGThreads) bwd_wide_kernel(BwdArgs a, WideFix w, float* dvacc) {
  extern __shared__ float sm[];
  pdl_wait();
  const int total = a.B * a.H * w.nc;  // the list's capacity
  const int cnt = (int)min(*w.count, (unsigned)total);
  float* scratch = w.scratch + (size_t)blockIdx.x * walk_scratch_floats(128, kGlaChunk);
  for (int it = blockIdx.x; it < cnt; it += gridDim.x) {
    const int chunk = w.list[it];
    if (chunk < 0 || chunk >= total) continue;
    const int bh = chunk / w.nc, c = chunk % w.nc;
    const int tb = c * kGlaChunk, te = min(a.L, tb + kGlaChunk);
    const size_t so = (size_t)chunk * 128 * 128;
    GlaWalk<bf16> g{tb, te, w.phq_in, w.phk_in, nullptr, w.hs + so, w.gs + so, nullptr,
                    w.rtot + (size_t)chunk * 128, scratch};
    gla_bwd_walks<bf16, 128>(a, sm, bh, g, dvacc);
    __syncthreads();
  }
  pdl_trigger();
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
  } else if (a.L > 0 || a.dh0) {
    const size_t smem = GbLayout<D>::TOTAL * sizeof(float);
    e = cudaFuncSetAttribute(gla_bwd_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    trace_begin("gla_bwd_simt", s);
    gla_bwd_kernel<T, D><<<BH, kGThreads, smem, s>>>(a, w.dvacc, w.walk);
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

int bwd_wide_ctas(int BH, int nc) { return BH * nc < kWideCtas ? BH * nc : kWideCtas; }

size_t bwd_wide_scratch_bytes(int BH, int nc) {
  return (size_t)bwd_wide_ctas(BH, nc) * walk_scratch_floats(128, kGlaChunk) * sizeof(float);
}

size_t bwd_simt_workspace(int B, int H, int L, int dk, int dv, int M) {
  return carve_bytes(B, H, L, dk, dv, M);
}

cudaError_t launch_bwd_wide_fix(const BwdArgs& a, const WideFix& w, float* dvacc, cudaStream_t s,
                                int* launches) {
  const size_t smem = GbLayout<128>::TOTAL * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(bwd_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = bwd_wide_ctas(a.B * a.H, w.nc);
  trace_begin("bwd_wide_fix", s);
  e = launch_pdl(bwd_wide_kernel, dim3(grid), dim3(kGThreads), smem, s, a, w, dvacc);
  trace_end(s);
  ++*launches;
  return e;
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
