// k_decode.cu -- one recurrent decode step for N sequences (memory-bound).
//
// "Lizard" (arXiv 2507.09025), Preliminaries: the recurrent form keeps constant memory
// per sequence; papernotes.org note, 关键设计: GLA recurrence and Anchor Window
// Attention.  Per (sequence n, head) at absolute position p = pos[n]:
//   h <- exp(log_gamma) (.) h + phi_k v^T ;  y_gla = phi_q^T h
//   ring slot (p mod W) <- (k, v)
//   y_win = softmax(scale [q.meta_k ; q.k_t]) [meta_v ; v_t], t in [max(0, p-W+1), p]
//   y = y_gla + alpha y_win ;  pos[n] <- p + 1 (by the last CTA of sequence n)
//
// One CTA per (n, head).  The fp32 state is streamed once: each thread owns 4
// consecutive value columns (one 16-byte load/store) of DK/RG rows, so a warp moves
// 512 contiguous bytes per row and every thread has all of its state loads in flight
// before the first FMA.  The ring is read with 16-byte loads, one warp per key.
#include "lizard_dev.cuh"
#include "lizard_internal.h"

namespace lz {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxW = 1024;
constexpr int kMaxM = 16;

template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThreads) decode_kernel(DecArgs a) {
  constexpr int CG = DV / 4;          // column groups of 4
  constexpr int RG = kThreads / CG;   // row groups
  constexpr int RPT = DK / RG;        // rows per thread
  // 16-byte alignment: s_v and s_red are accessed as float4
  __shared__ __align__(16) float s_pq[DK], s_pk[DK], s_eg[DK], s_q[DK], s_k[DK];
  __shared__ __align__(16) float s_v[DV];
  __shared__ __align__(16) float s_red[RG][DV];
  __shared__ float s_z[kMaxM + kMaxW];
  __shared__ int64_t s_pos;

  const int u = blockIdx.x;  // n * H + head
  const int n = u / a.H, hh = u % a.H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const T* pq = static_cast<const T*>(a.pq) + (size_t)u * DK;
  const T* pk = static_cast<const T*>(a.pk) + (size_t)u * DK;
  const T* qg = static_cast<const T*>(a.q) + (size_t)u * DK;
  const T* kg = static_cast<const T*>(a.k) + (size_t)u * DK;
  const T* vg = static_cast<const T*>(a.v) + (size_t)u * DV;
  const float* lg = a.lg + (size_t)u * DK;
  float* h = a.h + (size_t)u * DK * DV;
  T* kr = static_cast<T*>(a.kr) + (size_t)u * a.W * DK;
  T* vr = static_cast<T*>(a.vr) + (size_t)u * a.W * DV;

  // Issue the state loads first; they are the bulk of the traffic.
  const int cg = tid % CG, rg = tid / CG;
  float4 hv[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
    hv[i] = *reinterpret_cast<const float4*>(h + (size_t)(rg + RG * i) * DV + 4 * cg);

  for (int d = tid; d < DK; d += kThreads) {
    s_pq[d] = ld_f(pq + d);
    s_pk[d] = ld_f(pk + d);
    s_eg[d] = expf(lg[d]);
    s_q[d] = ld_f(qg + d);
    s_k[d] = ld_f(kg + d);
  }
  for (int c = tid; c < DV; c += kThreads) s_v[c] = ld_f(vg + c);
  if (tid == 0) s_pos = a.pos[n];
  __syncthreads();
  const int64_t p = s_pos;
  const float4 v4 = *reinterpret_cast<const float4*>(s_v + 4 * cg);

  // GLA: update the state and form this thread's partial readout.
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = rg + RG * i;
    const float g = s_eg[r], b = s_pk[r], c = s_pq[r];
    float4 x = hv[i];
    x.x = fmaf(g, x.x, b * v4.x);
    x.y = fmaf(g, x.y, b * v4.y);
    x.z = fmaf(g, x.z, b * v4.z);
    x.w = fmaf(g, x.w, b * v4.w);
    *reinterpret_cast<float4*>(h + (size_t)r * DV + 4 * cg) = x;
    acc.x = fmaf(c, x.x, acc.x);
    acc.y = fmaf(c, x.y, acc.y);
    acc.z = fmaf(c, x.z, acc.z);
    acc.w = fmaf(c, x.w, acc.w);
  }
  *reinterpret_cast<float4*>(&s_red[rg][4 * cg]) = acc;

  // Window: write the new token into its slot, then one warp per key for the logits.
  const int slot = (int)(p % a.W);
  for (int d = tid; d < DK; d += kThreads) kr[(size_t)slot * DK + d] = static_cast<T>(kg[d]);
  for (int c = tid; c < DV; c += kThreads) vr[(size_t)slot * DV + c] = static_cast<T>(vg[c]);
  const int64_t t_lo = p - a.W + 1 > 0 ? p - a.W + 1 : 0;
  const int cnt = (int)(p - t_lo + 1);
  const int nkeys = a.M + cnt;
  const T* mk = static_cast<const T*>(a.mk) + (size_t)hh * a.M * DK;
  const T* mv = static_cast<const T*>(a.mv) + (size_t)hh * a.M * DV;
  for (int j = warp; j < nkeys; j += kWarps) {
    float d = 0.f;
    if (j < a.M) {
      for (int e = 4 * lane; e < DK; e += 128) {
        const float4 kv = ld4(mk + (size_t)j * DK + e);
        d += s_q[e] * kv.x + s_q[e + 1] * kv.y + s_q[e + 2] * kv.z + s_q[e + 3] * kv.w;
      }
    } else {
      const int64_t t = t_lo + (j - a.M);
      const int sl = (int)(t % a.W);
      if (sl == slot) {
        for (int e = 4 * lane; e < DK; e += 128)
          d += s_q[e] * s_k[e] + s_q[e + 1] * s_k[e + 1] + s_q[e + 2] * s_k[e + 2] + s_q[e + 3] * s_k[e + 3];
      } else {
        for (int e = 4 * lane; e < DK; e += 128) {
          const float4 kv = ld4(kr + (size_t)sl * DK + e);
          d += s_q[e] * kv.x + s_q[e + 1] * kv.y + s_q[e + 2] * kv.z + s_q[e + 3] * kv.w;
        }
      }
    }
    d = warp_sum(d);
    if (lane == 0) s_z[j] = d * a.scale;
  }
  __syncthreads();
  if (warp == 0) {
    float mx = -INFINITY;
    for (int j = lane; j < nkeys; j += 32) mx = fmaxf(mx, s_z[j]);
    mx = warp_max(mx);
    float sum = 0.f;
    for (int j = lane; j < nkeys; j += 32) {
      const float e = expf(s_z[j] - mx);
      s_z[j] = e;
      sum += e;
    }
    sum = warp_sum(sum);
    const float inv = 1.f / sum;
    for (int j = lane; j < nkeys; j += 32) s_z[j] *= inv;
  }
  __syncthreads();
  // Values: thread takes column c over one half of the keys.
  {
    const int c = tid % DV;
    const int half = tid / DV;  // 0 or 1 when DV = 128; 0..3 when DV = 64
    constexpr int NH = kThreads / DV;
    float yw = 0.f;
    for (int j = half; j < nkeys; j += NH) {
      float val;
      if (j < a.M) {
        val = ld_f(mv + (size_t)j * DV + c);
      } else {
        const int64_t t = t_lo + (j - a.M);
        const int sl = (int)(t % a.W);
        val = (sl == slot) ? s_v[c] : ld_f(vr + (size_t)sl * DV + c);
      }
      yw = fmaf(s_z[j], val, yw);
    }
    // Reduce the NH partial sums through s_red's spare space after the GLA reduce.
    __syncthreads();
    float ygla = 0.f;
    if (tid < DV) {
#pragma unroll
      for (int r = 0; r < RG; ++r) ygla += s_red[r][tid];
    }
    __syncthreads();
    s_red[half][c] = yw;
    __syncthreads();
    if (tid < DV) {
      float ys = 0.f;
#pragma unroll
      for (int r = 0; r < NH; ++r) ys += s_red[r][tid];
      static_cast<T*>(a.y)[(size_t)u * DV + tid] = cvt_out<T>(ygla + a.alpha * ys);
    }
  }

  // The last CTA of sequence n advances its position.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(&a.counters[n], 1u);
    if (prev == (unsigned)a.H - 1) {
      a.pos[n] = p + 1;
      a.counters[n] = 0u;
      __threadfence();
    }
  }
}

// ------------------------------------------------------------------------------------
// Split step for W <= kSplitMaxW: two kernels, each shaped for its own traffic.
//  * decode_gla_kernel streams the fp32 state (128 KiB of the 166 KiB a unit moves):
//    every thread issues its sixteen 16-byte state loads before anything else, three
//    CTAs share an SM, and y_gla goes to y.
//  * decode_win_kernel takes one warp per (sequence, head): the logits over the meta
//    tokens, the ring and the new token, the softmax and y_win in registers and a small
//    per-warp shared row, then adds alpha * y_win into y, writes the new token into its
//    slot and advances pos (last warp of each sequence).  It is launched as a
//    programmatic dependent of decode_gla_kernel, whose outputs it reads only after
//    griddepcontrol.wait, so all of its ring reads overlap the state pass.
// ------------------------------------------------------------------------------------
constexpr int kSplitMaxW = 128;

template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThreads, 3) decode_gla_kernel(DecArgs a) {
  constexpr int CG = DV / 4;
  constexpr int RG = kThreads / CG;
  constexpr int RPT = DK / RG;
  __shared__ __align__(16) float s_pq[DK], s_pk[DK], s_eg[DK];
  __shared__ __align__(16) float s_v[DV];
  __shared__ __align__(16) float s_red[RG][DV];
  const int u = blockIdx.x;
  const int tid = threadIdx.x;
  float* h = a.h + (size_t)u * DK * DV;
  const int cg = tid % CG, rg = tid / CG;
  float4 hv[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
    hv[i] = *reinterpret_cast<const float4*>(h + (size_t)(rg + RG * i) * DV + 4 * cg);
  // the window kernel (launched next) reads nothing this kernel writes before its
  // griddepcontrol.wait: let it start staging its rings during this kernel's tail
  pdl_trigger();
  const T* pq = static_cast<const T*>(a.pq) + (size_t)u * DK;
  const T* pk = static_cast<const T*>(a.pk) + (size_t)u * DK;
  const float* lg = a.lg + (size_t)u * DK;
  for (int d = tid; d < DK; d += kThreads) {
    s_pq[d] = ld_f(pq + d);
    s_pk[d] = ld_f(pk + d);
    s_eg[d] = expf(lg[d]);
  }
  const T* vg = static_cast<const T*>(a.v) + (size_t)u * DV;
  for (int c = tid; c < DV; c += kThreads) s_v[c] = ld_f(vg + c);
  __syncthreads();
  const float4 v4 = *reinterpret_cast<const float4*>(s_v + 4 * cg);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = rg + RG * i;
    const float g = s_eg[r], b = s_pk[r], c = s_pq[r];
    float4 x = hv[i];
    x.x = fmaf(g, x.x, b * v4.x);
    x.y = fmaf(g, x.y, b * v4.y);
    x.z = fmaf(g, x.z, b * v4.z);
    x.w = fmaf(g, x.w, b * v4.w);
    *reinterpret_cast<float4*>(h + (size_t)r * DV + 4 * cg) = x;
    acc.x = fmaf(c, x.x, acc.x);
    acc.y = fmaf(c, x.y, acc.y);
    acc.z = fmaf(c, x.z, acc.z);
    acc.w = fmaf(c, x.w, acc.w);
  }
  *reinterpret_cast<float4*>(&s_red[rg][4 * cg]) = acc;
  __syncthreads();
  if (tid < DV) {
    float yg = 0.f;
#pragma unroll
    for (int r = 0; r < RG; ++r) yg += s_red[r][tid];
    static_cast<T*>(a.y)[(size_t)u * DV + tid] = cvt_out<T>(yg);
  }
}

// One warp per (sequence, head): lane l owns dimensions [l DPL, (l+1) DPL) of every key,
// value, q and y row, so each row is one coalesced load of the warp.  No CTA barrier and
// little register state, so all N*H units are resident at once and the kernel runs at
// the rings' bandwidth; everything before griddepcontrol.wait overlaps the state kernel.
constexpr int kWinUnits = 8;  // warps (units) per CTA
constexpr int kWinRows = kMaxM + kSplitMaxW + 1;

template <typename T, int DPL>
__device__ __forceinline__ void ld_row(const T* p, float (&v)[DPL]) {
  if constexpr (DPL == 4) {
    const float4 f = ld4(p);
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
  } else {
#pragma unroll
    for (int i = 0; i < DPL; ++i) v[i] = ld_f(p + i);
  }
}

// Sum over the lanes of each of 8 values per lane in a fixed butterfly pattern; lane l
// ends with the total of row ((l >> 4) & 1) * 4 + ((l >> 3) & 1) * 2 + ((l >> 2) & 1).
__device__ __forceinline__ float warp_sum8(float (&v)[8]) {
  const int lane = threadIdx.x & 31;
  float w[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) w[m] = v[m];
  int off = 16;
#pragma unroll
  for (int nn = 8; nn > 1; nn >>= 1, off >>= 1) {
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int m = 0; m < nn / 2; ++m) {
      const float send = up ? w[m] : w[m + nn / 2];
      const float keep = up ? w[m + nn / 2] : w[m];
      w[m] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float x = w[0];
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  return x;
}

template <typename T, int D>
__global__ void __launch_bounds__(kWinUnits * 32) decode_win_kernel(DecArgs a) {
  constexpr int DPL = D / 32;
  __shared__ float s_z[kWinUnits][kWinRows];  // logits, then probabilities
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x * kWinUnits + warp;
  if (u >= a.N * a.H) return;
  const int n = u / a.H, hh = u % a.H, W = a.W, M = a.M;
  const int R = M + W + 1;  // rows: the meta tokens, the W ring slots, the new token
  const int d0 = lane * DPL;
  T* kr = static_cast<T*>(a.kr) + (size_t)u * W * D;
  T* vr = static_cast<T*>(a.vr) + (size_t)u * W * D;
  const T* mk = static_cast<const T*>(a.mk) + (size_t)hh * M * D;
  const T* mv = static_cast<const T*>(a.mv) + (size_t)hh * M * D;
  float q[DPL], kn[DPL], vn[DPL];
  ld_row<T, DPL>(static_cast<const T*>(a.q) + (size_t)u * D + d0, q);
  ld_row<T, DPL>(static_cast<const T*>(a.k) + (size_t)u * D + d0, kn);
  ld_row<T, DPL>(static_cast<const T*>(a.v) + (size_t)u * D + d0, vn);
  const int64_t p = a.pos[n];
  // ring slot s holds token t with t mod W = s; the window is [max(0, p-W+1), p], whose
  // token p (the new one) replaces slot p mod W: every other written slot is in it
  const int sp = (int)(p % W);
  auto valid = [&](int r) {
    if (r < M || r == R - 1) return true;
    const int sl = r - M;
    return p >= W ? sl != sp : sl < (int)p;
  };
  auto krow = [&](int r) -> const T* { return r < M ? mk + (size_t)r * D : kr + (size_t)(r - M) * D; };
  auto vrow = [&](int r) -> const T* { return r < M ? mv + (size_t)r * D : vr + (size_t)(r - M) * D; };
  float* z = s_z[warp];

  // logits, sixteen rows (two reductions of eight) at a time
  for (int r0 = 0; r0 < R; r0 += 16) {
    float part[2][8];
    // every load is issued unconditionally (rows past the ring read its last row and are
    // replaced afterwards), so the sixteen loads are in flight together
    float kv[16][DPL];
#pragma unroll
    for (int e = 0; e < 16; ++e) ld_row<T, DPL>(krow(min(r0 + e, R - 2)) + d0, kv[e]);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int r = r0 + e;
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < DPL; ++i) {
        const float k = r < R - 1 ? kv[e][i] : (r == R - 1 ? kn[i] : 0.f);
        acc = fmaf(q[i], k, acc);
      }
      part[e >> 3][e & 7] = acc;
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const float tot = warp_sum8(part[hf]);
      const int r = r0 + 8 * hf + ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
      if ((lane & 3) == 0 && r < R) z[r] = valid(r) ? tot * a.scale : -INFINITY;
    }
  }
  __syncwarp();
  float mx = -INFINITY;
  for (int r = lane; r < R; r += 32) mx = fmaxf(mx, z[r]);
  mx = warp_max(mx);
  float sum = 0.f;
  for (int r = lane; r < R; r += 32) {
    const float e = expf(z[r] - mx);  // 0 for the rows outside the window
    z[r] = e;
    sum += e;
  }
  sum = warp_sum(sum);
  __syncwarp();
  // y_win = sum_r p_r value_r, eight rows at a time
  float yw[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) yw[i] = 0.f;
  for (int r0 = 0; r0 < R; r0 += 16) {
    float vv[16][DPL];
#pragma unroll
    for (int e = 0; e < 16; ++e) ld_row<T, DPL>(vrow(min(r0 + e, R - 2)) + d0, vv[e]);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int r = r0 + e;
      const float pr = r < R ? z[r] : 0.f;
#pragma unroll
      for (int i = 0; i < DPL; ++i) yw[i] = fmaf(pr, r < R - 1 ? vv[e][i] : vn[i], yw[i]);
    }
  }
  // the new token into its slot (this warp read that slot's old content above)
#pragma unroll
  for (int i = 0; i < DPL; ++i) {
    kr[(size_t)sp * D + d0 + i] = static_cast<const T*>(a.k)[(size_t)u * D + d0 + i];
    vr[(size_t)sp * D + d0 + i] = static_cast<const T*>(a.v)[(size_t)u * D + d0 + i];
  }
  // y_gla comes from the state kernel launched just before this one (programmatic
  // dependent launch: everything above overlaps that kernel)
  pdl_wait();
  const float inv = a.alpha / sum;
  T* y = static_cast<T*>(a.y) + (size_t)u * D + d0;
#pragma unroll
  for (int i = 0; i < DPL; ++i) y[i] = cvt_out<T>(ld_f(y + i) + inv * yw[i]);
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(&a.counters[n], 1u);
    if (prev == (unsigned)a.H - 1) {
      a.pos[n] = p + 1;
      a.counters[n] = 0u;
      __threadfence();
    }
  }
}

template <typename T, int D>
cudaError_t launch_typed(const DecArgs& a, cudaStream_t s, int* launches) {
  if (a.W <= kSplitMaxW) {
    // the window kernel reads y_gla written by the GLA kernel on the same stream
    trace_begin("decode_gla", s);
    decode_gla_kernel<T, D, D><<<a.N * a.H, kThreads, 0, s>>>(a);
    trace_end(s);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ++*launches;
    const int units = a.N * a.H;
    trace_begin("decode_win", s);
    e = launch_pdl(decode_win_kernel<T, D>, dim3((units + kWinUnits - 1) / kWinUnits),
                   dim3(kWinUnits * 32), 0, s, a);
    trace_end(s);
    if (e != cudaSuccess) return e;
  } else {
    trace_begin("decode", s);
    decode_kernel<T, D, D><<<a.N * a.H, kThreads, 0, s>>>(a);
    trace_end(s);
  }
  ++*launches;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecArgs& a, lizard_dtype dt, cudaStream_t s, int* launches) {
  if (dt == LIZARD_F32) {
    return a.dk == 64 ? launch_typed<float, 64>(a, s, launches)
                      : launch_typed<float, 128>(a, s, launches);
  }
  return a.dk == 64 ? launch_typed<bf16, 64>(a, s, launches)
                    : launch_typed<bf16, 128>(a, s, launches);
}

}  // namespace lz
