// k_gla_std.cu -- the "standard" gated linear attention forward: the chunkwise (matrix)
// form with every operand and product in fp32 on the CUDA cores.  It is the comparison
// point of the hardware-aware kernel, not part of the Lizard operator.
//
// "Lizard: An Efficient Linearization Framework for LLMs" (arXiv 2507.09025): the matrix
// form of GLA multiplies queries and keys by cumulative products of the gates, which lose
// too much precision in bf16, so standard GLA kernels fall back to fp32 arithmetic without
// tensor cores, 2-3x slower (Preliminaries); its Efficiency section (Table 3) times the
// hardware-aware kernel against such a standard GLA forward.  The same chunkwise form in
// fp32 FFMA, in three passes over 64-token chunks (b = chunk-local inclusive cumulative
// log gate, Gamma_c = b at the chunk's last token):
//   1. state pass, per chunk:  U_c = Khat_c^T V_c,  Khat = phi_k e^{Gamma_c - b}  (<= 1)
//   2. scan, per (batch, head): h_0 = h0,  h_{c+1} = e^{Gamma_c} (.) h_c + U_c; the state
//      entering chunk c is stored over U_c, the last one is h_final
//   3. output pass, per chunk: y = tril(Qt Kt^T) V + Qt h_c,  Qt = phi_q e^{b},
//      Kt = phi_k e^{-b}
// The factorised product e^{b_t} e^{-b_s} needs |b| <= 80 inside a chunk; the output pass
// raises the device-check bit for a chunk beyond that (the standard form has no finite
// answer there, which is what the reparameterised kernel's bounded forms avoid).
// Thread tiles: 256 threads as a 16 x 16 grid; thread (ty, tx) owns rows ty*4 .. ty*4+3
// (plus 64 + ty*4 .. for 128-row outputs) and columns tx*4 .. tx*4+3 (plus 64 + tx*4 ..),
// so that the operands of one k-step are float4 loads a quarter-warp shares.  The output
// pass keeps about 100 KB of shared memory (two CTAs per SM) and streams the chunk's state
// through two 16-row buffers with asynchronous copies.
#include "lizard_dev.cuh"
#include "lizard_internal.h"

namespace lz {
namespace {

constexpr int kC = 64;          // tokens per chunk
constexpr int kThreads = 256;
constexpr float kMaxLog = 80.f;

struct StdArgs {
  int BH, L, nc;
  const void *pq, *pk, *v;
  const float* lg;
  const float* h0;
  float* hf;
  void* y;
  float* U;      // [BH][nc][D][D]: U_c, then the state entering chunk c
  float* G;      // [BH][nc][D]: Gamma_c
  unsigned* status;
};

// Rows (or columns) of a thread: 4 * (D / 64) of them, in groups of 4 at 64 apart.
template <int D>
__device__ __forceinline__ int tile_idx(int t16, int g) { return g * 64 + t16 * 4; }

// pass 1 ---------------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1) gla_std_state_kernel(const StdArgs a) {
  extern __shared__ float smf[];
  float* sb = smf;               // [kC][D] log gamma, then b
  float* sk = sb + kC * D;       // [kC][D] Khat
  float* sv = sk + kC * D;       // [kC][D] V
  __shared__ float s_gam[D];
  const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
  const int t0 = c * kC, n = min(kC, a.L - t0);
  const size_t base = ((size_t)bh * a.L + t0) * D;
  for (int e = tid * 4; e < kC * D; e += kThreads * 4) {
    const int t = e / D;
    const bool in = t < n;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4*>(sb + e) = in ? *reinterpret_cast<const float4*>(a.lg + base + e) : z;
    *reinterpret_cast<float4*>(sk + e) = in ? ld4(static_cast<const T*>(a.pk) + base + e) : z;
    *reinterpret_cast<float4*>(sv + e) = in ? ld4(static_cast<const T*>(a.v) + base + e) : z;
  }
  __syncthreads();
  if (tid < D) {
    float run = 0.f;
    for (int t = 0; t < kC; ++t) {
      run += sb[t * D + tid];
      sb[t * D + tid] = run;
    }
    s_gam[tid] = run;  // padded rows add zero: the last valid token's sum
    a.G[((size_t)bh * a.nc + c) * D + tid] = run;
  }
  __syncthreads();
  for (int e = tid; e < kC * D; e += kThreads) {
    const int d = e % D;
    sk[e] *= expf(s_gam[d] - sb[e]);
  }
  __syncthreads();
  constexpr int NG = D / 64;  // row / column groups of 4 per thread
  const int ty = tid >> 4, tx = tid & 15;
  float acc[4 * NG][4 * NG];
#pragma unroll
  for (int i = 0; i < 4 * NG; ++i)
#pragma unroll
    for (int j = 0; j < 4 * NG; ++j) acc[i][j] = 0.f;
#pragma unroll 4
  for (int t = 0; t < n; ++t) {
    float ar[4 * NG], bc[4 * NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const float4 x = *reinterpret_cast<const float4*>(sk + t * D + tile_idx<D>(ty, g));
      const float4 y = *reinterpret_cast<const float4*>(sv + t * D + tile_idx<D>(tx, g));
      ar[4 * g] = x.x; ar[4 * g + 1] = x.y; ar[4 * g + 2] = x.z; ar[4 * g + 3] = x.w;
      bc[4 * g] = y.x; bc[4 * g + 1] = y.y; bc[4 * g + 2] = y.z; bc[4 * g + 3] = y.w;
    }
#pragma unroll
    for (int i = 0; i < 4 * NG; ++i)
#pragma unroll
      for (int j = 0; j < 4 * NG; ++j) acc[i][j] = fmaf(ar[i], bc[j], acc[i][j]);
  }
  float* U = a.U + ((size_t)bh * a.nc + c) * D * D;
#pragma unroll
  for (int i = 0; i < 4 * NG; ++i) {
    const int d = tile_idx<D>(ty, i / 4) + (i & 3);
#pragma unroll
    for (int g = 0; g < NG; ++g)
      *reinterpret_cast<float4*>(U + d * D + tile_idx<D>(tx, g)) =
          make_float4(acc[i][4 * g], acc[i][4 * g + 1], acc[i][4 * g + 2], acc[i][4 * g + 3]);
  }
}

// pass 2 ---------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreads) gla_std_scan_kernel(const StdArgs a) {
  const int bh = blockIdx.y;
  const int e4 = (blockIdx.x * kThreads + threadIdx.x) * 4;  // first of 4 state entries
  if (e4 >= D * D) return;
  const int d = e4 / D;
  float4 h = a.h0 ? *reinterpret_cast<const float4*>(a.h0 + (size_t)bh * D * D + e4)
                  : make_float4(0.f, 0.f, 0.f, 0.f);
  // eight chunks' U and Gamma loaded before the eight dependent updates
  for (int c0 = 0; c0 < a.nc; c0 += 8) {
    float4 u[8];
    float g[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (c0 + k < a.nc) {
        const size_t sl = (size_t)bh * a.nc + c0 + k;
        u[k] = *reinterpret_cast<const float4*>(a.U + sl * D * D + e4);
        g[k] = expf(a.G[sl * D + d]);
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (c0 + k < a.nc) {
        *reinterpret_cast<float4*>(a.U + ((size_t)bh * a.nc + c0 + k) * D * D + e4) = h;
        h = make_float4(fmaf(g[k], h.x, u[k].x), fmaf(g[k], h.y, u[k].y), fmaf(g[k], h.z, u[k].z),
                        fmaf(g[k], h.w, u[k].w));
      }
    }
  }
  if (a.hf) *reinterpret_cast<float4*>(a.hf + (size_t)bh * D * D + e4) = h;
}

// pass 3 ---------------------------------------------------------------------------------
constexpr int kCP = kC + 4;  // padded row of the transposed [D][kC] tiles
constexpr int kHR = 16;      // rows of the chunk state per staging buffer (two buffers)

// The two state staging buffers sit in the part of the Kt tile that S (transposed) leaves
// free when that part is large enough (D = 128), else after V.
template <int D>
constexpr bool hbuf_in_kt() { return (D - kC) * kCP >= 2 * kHR * D; }

template <int D>
constexpr size_t out_smem_floats() {  // about 100 KB at D = 128: two CTAs per SM
  return 2 * (size_t)D * kCP + (size_t)kC * D + (hbuf_in_kt<D>() ? 0 : 2 * (size_t)kHR * D);
}

__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 2) gla_std_out_kernel(const StdArgs a) {
  extern __shared__ float smf[];
  float* sq = smf;             // [D][kCP] Qt transposed
  float* sk = sq + D * kCP;    // [D][kCP] Kt transposed; then S transposed [kC][kCP]
  float* sv = sk + D * kCP;    // [kC][D]  V
  float* ss = sk;
  float* hb = hbuf_in_kt<D>() ? sk + kC * kCP : sv + kC * D;  // [2][kHR][D] state rows
  const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
  const int t0 = c * kC, n = min(kC, a.L - t0);
  const size_t base = ((size_t)bh * a.L + t0) * D;
  // the state entering the chunk, staged kHR rows at a time for the Qt h product below
  const float* hc = a.U + ((size_t)bh * a.nc + c) * D * D;
  bool wide = false;
  if (tid < D) {
    // thread d walks its key dimension down the chunk: b, then Qt and Kt (transposed)
    const int d = tid;
    const T* pq = static_cast<const T*>(a.pq) + base + d;
    const T* pk = static_cast<const T*>(a.pk) + base + d;
    const float* lg = a.lg + base + d;
    float run = 0.f;
    // 16 tokens' loads in flight before their sequential sums
    for (int t0b = 0; t0b < kC; t0b += 16) {
      float g[16], q[16], k[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int t = t0b + u;
        const bool in = t < n;
        g[u] = in ? lg[(size_t)t * D] : 0.f;
        q[u] = in ? ld_f(pq + (size_t)t * D) : 0.f;
        k[u] = in ? ld_f(pk + (size_t)t * D) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        run += g[u];
        wide |= fabsf(run) > kMaxLog;
        sq[d * kCP + t0b + u] = q[u] * expf(run);
        sk[d * kCP + t0b + u] = k[u] * expf(-run);
      }
    }
  } else {
    for (int e = (tid - D) * 4; e < kC * D; e += (kThreads - D) * 4) {
      const int t = e / D;
      *reinterpret_cast<float4*>(sv + e) =
          t < n ? ld4(static_cast<const T*>(a.v) + base + e) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  if (__syncthreads_or(wide) && tid == 0) raise_status(a.status, kDevCheck);
  const int ty = tid >> 4, tx = tid & 15;
  // S = Qt Kt^T for rows ty*4.., columns tx*4..; tiles wholly above the diagonal are zero
  float s[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
  if (tx <= ty) {
#pragma unroll 4
    for (int d = 0; d < D; ++d) {
      const float4 x = *reinterpret_cast<const float4*>(sq + d * kCP + ty * 4);
      const float4 y = *reinterpret_cast<const float4*>(sk + d * kCP + tx * 4);
      const float xr[4] = {x.x, x.y, x.z, x.w}, yr[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) s[i][j] = fmaf(xr[i], yr[j], s[i][j]);
    }
  }
  __syncthreads();  // Kt is read; S goes over it
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int jj = tx * 4 + j;
    float col[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) col[i] = jj <= ty * 4 + i ? s[i][j] : 0.f;  // causal mask
    *reinterpret_cast<float4*>(ss + jj * kCP + ty * 4) = make_float4(col[0], col[1], col[2], col[3]);
  }
  __syncthreads();
  auto stage_h = [&](int buf, int d0) {
    for (int e = tid * 4; e < kHR * D; e += kThreads * 4) cp_async16(hb + buf * kHR * D + e, hc + d0 * D + e);
    cp_async_commit();
  };
  stage_h(0, 0);  // lands while S V is computed
  // y = S V + Qt h for rows ty*4.., columns tx*4 (+ 64 ..)
  constexpr int NG = D / 64;
  float acc[4][4 * NG];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4 * NG; ++j) acc[i][j] = 0.f;
  const int jmax = min(n, ty * 4 + 4);  // keys after the tile's last row contribute zero
#pragma unroll 2
  for (int j = 0; j < jmax; ++j) {
    const float4 x = *reinterpret_cast<const float4*>(ss + j * kCP + ty * 4);
    const float xr[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const float4 y = *reinterpret_cast<const float4*>(sv + j * D + tile_idx<D>(tx, g));
      const float yr[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][4 * g + e] = fmaf(xr[i], yr[e], acc[i][4 * g + e]);
    }
  }
  for (int d0 = 0; d0 < D; d0 += kHR) {
    const int buf = (d0 / kHR) & 1;
    if (d0 + kHR < D) {
      stage_h(buf ^ 1, d0 + kHR);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // rows d0 .. d0 + kHR - 1 of every thread's copies are in
#pragma unroll 4
    for (int dd = 0; dd < kHR; ++dd) {
      const float4 x = *reinterpret_cast<const float4*>(sq + (d0 + dd) * kCP + ty * 4);
      const float xr[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        const float4 y = *reinterpret_cast<const float4*>(hb + (buf * kHR + dd) * D + tile_idx<D>(tx, g));
        const float yr[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[i][4 * g + e] = fmaf(xr[i], yr[e], acc[i][4 * g + e]);
      }
    }
    __syncthreads();  // the buffer is free for the copy after next
  }
  T* y = static_cast<T*>(a.y) + base;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = ty * 4 + i;
    if (t < n) {
#pragma unroll
      for (int g = 0; g < NG; ++g)
        st4(y + t * D + tile_idx<D>(tx, g),
            make_float4(acc[i][4 * g], acc[i][4 * g + 1], acc[i][4 * g + 2], acc[i][4 * g + 3]));
    }
  }
}

template <typename T, int D>
cudaError_t launch_typed(const StdArgs& a, cudaStream_t s, int* launches) {
  cudaError_t e;
  if (a.L > 0) {
    const size_t smem1 = 3 * (size_t)kC * D * sizeof(float);
    if ((e = cudaFuncSetAttribute(gla_std_state_kernel<T, D>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1)) != cudaSuccess)
      return e;
    trace_begin("gla_std_state", s);
    gla_std_state_kernel<T, D><<<dim3(a.nc, a.BH), kThreads, smem1, s>>>(a);
    trace_end(s);
    ++*launches;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (a.L > 0 || a.hf) {
    trace_begin("gla_std_scan", s);
    gla_std_scan_kernel<D><<<dim3((D * D / 4 + kThreads - 1) / kThreads, a.BH), kThreads, 0, s>>>(a);
    trace_end(s);
    ++*launches;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (a.L > 0) {
    const size_t smem3 = out_smem_floats<D>() * sizeof(float);
    if ((e = cudaFuncSetAttribute(gla_std_out_kernel<T, D>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem3)) != cudaSuccess)
      return e;
    trace_begin("gla_std_out", s);
    gla_std_out_kernel<T, D><<<dim3(a.nc, a.BH), kThreads, smem3, s>>>(a);
    trace_end(s);
    ++*launches;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

size_t gla_std_workspace(int BH, int L, int D) {
  const size_t nc = L > 0 ? (size_t)(L + kC - 1) / kC : 1;
  return align_up((size_t)BH * nc * D * D * sizeof(float), 256) +
         align_up((size_t)BH * nc * D * sizeof(float), 256);
}

cudaError_t launch_gla_std_fwd(int BH, int L, int D, lizard_dtype dt, const void* pq,
                               const void* pk, const void* v, const float* lg, const float* h0,
                               float* hf, void* y, unsigned* status, unsigned char* ws,
                               cudaStream_t s, int* launches) {
  const int nc = L > 0 ? (L + kC - 1) / kC : 1;
  StdArgs a;
  a.BH = BH;
  a.L = L;
  a.nc = nc;
  a.pq = pq;
  a.pk = pk;
  a.v = v;
  a.lg = lg;
  a.h0 = h0;
  a.hf = hf;
  a.y = y;
  a.U = reinterpret_cast<float*>(ws);
  a.G = reinterpret_cast<float*>(ws + align_up((size_t)BH * nc * D * D * sizeof(float), 256));
  a.status = status;
  if (L == 0) {
    // h_final = h0: the scan over one empty chunk (Gamma = 0, U = 0)
    cudaError_t e = cudaMemsetAsync(ws, 0, gla_std_workspace(BH, L, D), s);
    if (e != cudaSuccess) return e;
  }
  if (dt == LIZARD_BF16)
    return D == 128 ? launch_typed<bf16, 128>(a, s, launches) : launch_typed<bf16, 64>(a, s, launches);
  return D == 128 ? launch_typed<float, 128>(a, s, launches) : launch_typed<float, 64>(a, s, launches);
}

}  // namespace lz
