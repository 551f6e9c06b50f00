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
//  * decode_win_kernel stages the two rings in shared memory (keys and values in two
//    copy groups), computes the window softmax (8 lanes per key, lanes interleaved over
//    dimensions so the shared-memory reads are conflict-free), adds alpha * y_win into y,
//    writes the new token into its slot and advances pos (last CTA of each sequence).
//    It is launched as a programmatic dependent of decode_gla_kernel, whose outputs it
//    reads only after griddepcontrol.wait: its ring copies run during the state pass's
//    tail (a 64 x 32 step measured 67 -> 62 us).
// ------------------------------------------------------------------------------------
constexpr int kSplitMaxW = 128;
constexpr int kWinThreads = 256;
constexpr int kWinWarps = kWinThreads / 32;

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

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gsrc)
               : "memory");
}

template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kWinThreads) decode_win_kernel(DecArgs a) {
  extern __shared__ __align__(128) unsigned char wsm[];
  const int W = a.W, M = a.M;
  // keys: W ring rows, M meta rows, then the new token's row; values likewise, so one
  // row index serves both.  The new token has a row of its own, which no ring copy
  // targets, so it needs no ordering against them.
  T* skey = reinterpret_cast<T*>(wsm);            // [W + M + 1][DK]
  T* sval = skey + (size_t)(W + M + 1) * DK;      // [W + M + 1][DV]
  __shared__ __align__(16) float s_q[DK];
  __shared__ float s_z[kMaxM + kSplitMaxW];
  __shared__ int s_row[kMaxM + kSplitMaxW];
  __shared__ float s_part[kWinThreads / DV > 0 ? kWinThreads / DV : 1][DV];
  __shared__ int64_t s_pos;
  const int u = blockIdx.x;
  const int n = u / a.H, hh = u % a.H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  T* kr = static_cast<T*>(a.kr) + (size_t)u * W * DK;
  T* vr = static_cast<T*>(a.vr) + (size_t)u * W * DV;
  const T* kg = static_cast<const T*>(a.k) + (size_t)u * DK;
  const T* vg = static_cast<const T*>(a.v) + (size_t)u * DV;
  if (tid == 0) s_pos = a.pos[n];
  {
    // asynchronous 16-byte copies of both rings and this head's meta rows
    constexpr int KC = DK * sizeof(T) / 16, VC = DV * sizeof(T) / 16;  // 16-B chunks per row
    const T* mkp = static_cast<const T*>(a.mk) + (size_t)hh * M * DK;
    const T* mvp = static_cast<const T*>(a.mv) + (size_t)hh * M * DV;
    for (int e = tid; e < W * KC; e += kWinThreads) cp_async16(skey + e * (16 / sizeof(T)), kr + e * (16 / sizeof(T)));
    for (int e = tid; e < M * KC; e += kWinThreads)
      cp_async16(skey + (size_t)W * DK + e * (16 / sizeof(T)), mkp + e * (16 / sizeof(T)));
    asm volatile("cp.async.commit_group;" ::: "memory");  // keys: the logits need only these
    for (int e = tid; e < W * VC; e += kWinThreads) cp_async16(sval + e * (16 / sizeof(T)), vr + e * (16 / sizeof(T)));
    for (int e = tid; e < M * VC; e += kWinThreads)
      cp_async16(sval + (size_t)W * DV + e * (16 / sizeof(T)), mvp + e * (16 / sizeof(T)));
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  const T* qg = static_cast<const T*>(a.q) + (size_t)u * DK;
  T* y = static_cast<T*>(a.y) + (size_t)u * DV;
  const int nrow = W + M;  // the new token's row
  for (int d = tid; d < DK; d += kWinThreads) {
    s_q[d] = ld_f(qg + d);
    skey[(size_t)nrow * DK + d] = kg[d];
  }
  for (int c = tid; c < DV; c += kWinThreads) sval[(size_t)nrow * DV + c] = vg[c];
  __syncthreads();
  const int64_t p = s_pos;
  const int slot = (int)(p % W);
  // the new token replaces its slot in the global ring (the slot's old token is outside
  // the window, so the copy of it in shared memory is never read)
  for (int d = tid; d < DK; d += kWinThreads) kr[(size_t)slot * DK + d] = kg[d];
  for (int c = tid; c < DV; c += kWinThreads) vr[(size_t)slot * DV + c] = vg[c];
  const int64_t t_lo = p - W + 1 > 0 ? p - W + 1 : 0;
  const int nkeys = M + (int)(p - t_lo + 1);
  // row of key j: meta keys first (rows W..W+M-1), then window token t_lo + i at slot
  // (t_lo + i) mod W, computed as one wrap of s_lo + i; the newest token (p) in its own row
  const int s_lo = (int)(t_lo % W);
  for (int j = tid; j < nkeys; j += kWinThreads) {
    const int i = j - M, r = s_lo + i;
    s_row[j] = j < M ? W + j : (j == nkeys - 1 ? nrow : (r >= W ? r - W : r));
  }
  asm volatile("cp.async.wait_group 1;" ::: "memory");  // this thread's key copies
  __syncthreads();
  {
    // logits: 8 lanes per key, lane l8 takes dimensions {4*l8 + 32*i}
    constexpr int LPK = 8;
    const int sub = lane / LPK, l8 = lane % LPK;
    for (int j0 = warp * 4; j0 < nkeys; j0 += kWinWarps * 4) {
      const int j = j0 + sub;
      float d = 0.f;
      if (j < nkeys) {
        const T* key = skey + (size_t)s_row[j] * DK;
#pragma unroll
        for (int e = 4 * l8; e < DK; e += 32) {
          const float4 q4 = *reinterpret_cast<const float4*>(s_q + e);
          const float4 k4 = ld4(key + e);
          d = fmaf(q4.x, k4.x, d);
          d = fmaf(q4.y, k4.y, d);
          d = fmaf(q4.z, k4.z, d);
          d = fmaf(q4.w, k4.w, d);
        }
      }
#pragma unroll
      for (int o = LPK / 2; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      if (l8 == 0 && j < nkeys) s_z[j] = d * a.scale;
    }
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
  asm volatile("cp.async.wait_group 0;" ::: "memory");  // this thread's value copies
  __syncthreads();
  constexpr int NP = kWinThreads / DV > 0 ? kWinThreads / DV : 1;  // key partitions
  {
    const int c = tid % DV, part = tid / DV;
    if (part < NP) {
      float y0 = 0.f, y1 = 0.f, y2 = 0.f, y3 = 0.f;
      int j = part;
      for (; j + 3 * NP < nkeys; j += 4 * NP) {
        y0 = fmaf(s_z[j], ld_f(sval + (size_t)s_row[j] * DV + c), y0);
        y1 = fmaf(s_z[j + NP], ld_f(sval + (size_t)s_row[j + NP] * DV + c), y1);
        y2 = fmaf(s_z[j + 2 * NP], ld_f(sval + (size_t)s_row[j + 2 * NP] * DV + c), y2);
        y3 = fmaf(s_z[j + 3 * NP], ld_f(sval + (size_t)s_row[j + 3 * NP] * DV + c), y3);
      }
      for (; j < nkeys; j += NP) y0 = fmaf(s_z[j], ld_f(sval + (size_t)s_row[j] * DV + c), y0);
      s_part[part][c] = (y0 + y1) + (y2 + y3);
    }
  }
  __syncthreads();
  // y_gla comes from the GLA kernel launched just before this one (programmatic
  // dependent launch: everything above overlaps that kernel's tail)
  pdl_wait();
  for (int c = tid; c < DV; c += kWinThreads) {
    float ys = 0.f;
#pragma unroll
    for (int r = 0; r < NP; ++r) ys += s_part[r][c];
    y[c] = cvt_out<T>(ld_f(y + c) + a.alpha * ys);
  }
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
    const size_t smem = (size_t)(a.W + a.M + 1) * 2 * D * sizeof(T);
    e = cudaFuncSetAttribute(decode_win_kernel<T, D, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    trace_begin("decode_win", s);
    e = launch_pdl(decode_win_kernel<T, D, D>, dim3(a.N * a.H), dim3(kWinThreads), smem, s, a);
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
