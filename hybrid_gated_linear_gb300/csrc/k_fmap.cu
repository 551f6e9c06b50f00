// k_fmap.cu -- the Hedgehog feature map phi(x) = [exp(x W) (+) exp(-x W)] per head and its
// backward ("Lizard", arXiv 2507.09025, Method: the strictly non-negative Hedgehog feature
// map whose exponential form admits the log-space reparameterisation).
//
//   forward, per (b, h, token):   z = x W  (F columns),  phi = [e^z, e^-z]  (2F features)
//   backward:                     dz = dphi+ e^z - dphi- e^-z   (z recomputed from x)
//                                 dx = dz W^T,   dW[h] = sum over batch and tokens of x^T dz
//
// Tensor-core path (bf16, D = 128 inputs, F = 64): one CTA per 128-token tile for the
// forward (z = x W as one M=128 N=64 K=128 tcgen05 product, the exponentials in the
// epilogue, phi by TMA store); for the backward one CTA per group of kTilesPerCta tiles
// of one (b, h), which recomputes z, forms dz (bf16) in shared memory, and issues
// dx = dz W^T (M=128 N=128 K=64) and dW += x^T dz (M=128 N=64 K=128, accumulated in TMEM
// over the CTA's tiles).  The per-CTA dW partials are then summed in a fixed order.
// CUDA-core path: any D <= 256, F <= 128 with D F <= 16384, fp32 or bf16, exact fp32
// arithmetic, same partial-sum scheme.
#include "lizard_dev.cuh"
#include "lizard_internal.h"
#include "tc_pipe.cuh"

namespace lz {
namespace {

using namespace tc;

constexpr int kT = 128;    // tokens per tile
constexpr int kDin = 128;  // input features (tensor-core path)
constexpr int kDh = 64;    // columns of W (tensor-core path)
constexpr int kThreads = 6 * 32;
constexpr int kTilesPerCta = 4;  // backward tiles per CTA (dW accumulated in TMEM)
// Both backward paths keep one dW partial per kTokPerGroup tokens of each (b, h), so the
// workspace does not depend on the path taken.
constexpr int kTokPerGroup = kTilesPerCta * kT;

struct FmMaps {
  CUtensorMap x, w, out;  // forward: out = phi; backward: out = dx
  CUtensorMap dphi;       // backward only
};

struct FmParams {
  int H, nt, groups;
  float* dw_part;  // backward: [B*H][groups][128][64] fp32
  unsigned* status;
};

// ------------------------------------------------------------------------------------
// forward (tensor cores)
// ------------------------------------------------------------------------------------
enum { FF_LD = 0, FF_Z, FF_DONE, FF_COUNT };
constexpr uint32_t FS_X = 0, FS_W = 32768, FS_BARS = FS_W + 16384;
constexpr size_t kFwdSmem = FS_BARS + 1024 + 1024;

// three CTAs per SM (registers and shared memory), so that one CTA's loads overlap another's
// epilogue
__global__ void __launch_bounds__(kThreads, 3) fmap_fwd_kernel(const __grid_constant__ FmMaps maps,
                                                               const FmParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  using C = Ctl<FF_COUNT>;
  C* ctl = reinterpret_cast<C*>(sm + FS_BARS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x % p.nt, bh = blockIdx.x / p.nt, hh = bh % p.H;
  const int t0 = tile * kT;

  if (threadIdx.x == 0) {
    for (int i = 0; i < FF_COUNT; ++i) mbar_init(&ctl->bar[i], 1u);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&ctl->bar[FF_LD], 32768 + 16384);
      tma_load_3d(sm + FS_X, &maps.x, 0, t0, bh, &ctl->bar[FF_LD]);
      tma_load_3d(sm + FS_X + 16384, &maps.x, 64, t0, bh, &ctl->bar[FF_LD]);
      tma_load_3d(sm + FS_W, &maps.w, 0, 0, hh, &ctl->bar[FF_LD]);
      drain_bar(ctl, FF_LD, 1, globaltimer_ns());
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t sb = smem_u32(sm);
      const bool ok = wait_bar(ctl, FF_LD, 0);
      if (ok) {
        tc_fence_after();
        // z[t][j] = sum_i x[t][i] W[i][j]: A = x (K-major), B = W (K rows, MN-major)
        for (int j = 0; j < kDin / 16; ++j)
          mma_bf16(tmem, desc_k(sb + FS_X, kT, j), desc_mn(sb + FS_W, kDin, j),
                   idesc_bf16(kT, kDh, false, true), j > 0);
        mma_commit(&ctl->bar[FF_Z]);
      }
      mma_commit(&ctl->bar[FF_DONE]);
      drain_bar(ctl, FF_DONE, 1, globaltimer_ns());
    }
  } else {
    const int qw = warp & 3, r = qw * 32 + lane;  // thread = token row of the tile
    const uint32_t tl = tmem + ((uint32_t)(qw * 32) << 16);
    const bool ok = wait_bar(ctl, FF_Z, 0);
    if (ok) {
      tc_fence_after();
      // phi is staged over the x tile, which the (completed) MMA no longer reads
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        uint32_t z[32];
        tmem_ld32(tl + 32 * g, z);
        tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float ep[16], em[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float zz = __uint_as_float(z[16 * h + e]);
            ep[e] = __expf(zz);
            em[e] = __expf(-zz);
          }
          store16_bf16(sm + FS_X, kT, r, 32 * g + 16 * h, ep);
          store16_bf16(sm + FS_X, kT, r, kDh + 32 * g + 16 * h, em);
        }
      }
      fence_proxy_async_smem();
    }
    named_sync(1, 128);
    if (ok && threadIdx.x == 64) {
      tma_store_3d(&maps.out, sm + FS_X, 0, t0, bh);
      tma_store_3d(&maps.out, sm + FS_X + 16384, 64, t0, bh);
      bulk_commit();
      bulk_wait_read();
    }
  }

  pdl_trigger();
  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
  if (threadIdx.x == 0 && ctl->abort) raise_status(p.status, kDevTimeout);
}

// ------------------------------------------------------------------------------------
// backward (tensor cores)
// ------------------------------------------------------------------------------------
// LD: x, dphi (and W with the first tile) landed; Z: z ready; DZ: dz stored (128 arrivals);
// OUT: dx and dW products done; FREE: the dx staging has been read by its TMA store.
enum { FB_LD = 0, FB_Z, FB_DZ, FB_OUT, FB_FREE, FB_DONE, FB_COUNT };
// x 32 KB, W 16 KB, dphi 32 KB (then the dx staging), dz 16 KB
constexpr uint32_t BS_X = 0, BS_W = 32768, BS_DP = BS_W + 16384, BS_DZ = BS_DP + 32768,
                   BS_BARS = BS_DZ + 16384;
constexpr size_t kBwdSmem = BS_BARS + 1024 + 1024;
// TMEM columns: z 0..63, dW 64..127, dx 128..255
constexpr uint32_t TB_Z = 0, TB_DW = 64, TB_DX = 128;

__global__ void __launch_bounds__(kThreads, 1) fmap_bwd_kernel(const __grid_constant__ FmMaps maps,
                                                               const FmParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  using C = Ctl<FB_COUNT>;
  C* ctl = reinterpret_cast<C*>(sm + BS_BARS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = blockIdx.x % p.groups, bh = blockIdx.x / p.groups, hh = bh % p.H;
  const int tile0 = grp * kTilesPerCta;
  const int ntiles = min(kTilesPerCta, p.nt - tile0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < FB_COUNT; ++i) mbar_init(&ctl->bar[i], i == FB_DZ ? 128u : 1u);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      uint32_t armed = 0;
      for (int i = 0; i < ntiles; ++i) {
        // the previous tile's dx staging (over dphi) must have been read out, and its
        // products (which read x) are complete before that
        if (i > 0 && !wait_bar(ctl, FB_FREE, (i - 1) & 1)) break;
        const int t0 = (tile0 + i) * kT;
        mbar_arrive_expect_tx(&ctl->bar[FB_LD], 65536 + (i == 0 ? 16384 : 0));
        ++armed;
        tma_load_3d(sm + BS_X, &maps.x, 0, t0, bh, &ctl->bar[FB_LD]);
        tma_load_3d(sm + BS_X + 16384, &maps.x, 64, t0, bh, &ctl->bar[FB_LD]);
        if (i == 0) tma_load_3d(sm + BS_W, &maps.w, 0, 0, hh, &ctl->bar[FB_LD]);
        tma_load_3d(sm + BS_DP, &maps.dphi, 0, t0, bh, &ctl->bar[FB_LD]);
        tma_load_3d(sm + BS_DP + 16384, &maps.dphi, 64, t0, bh, &ctl->bar[FB_LD]);
      }
      drain_bar(ctl, FB_LD, armed, globaltimer_ns());
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t sb = smem_u32(sm);
      for (int i = 0; i < ntiles; ++i) {
        if (!wait_bar(ctl, FB_LD, i & 1)) break;
        tc_fence_after();
        for (int j = 0; j < kDin / 16; ++j)  // z = x W
          mma_bf16(tmem + TB_Z, desc_k(sb + BS_X, kT, j), desc_mn(sb + BS_W, kDin, j),
                   idesc_bf16(kT, kDh, false, true), j > 0);
        mma_commit(&ctl->bar[FB_Z]);
        if (!wait_bar(ctl, FB_DZ, i & 1)) break;
        tc_fence_after();
        // dx[t][i] = sum_j dz[t][j] W[i][j]: A = dz (K-major), B = W (N rows, K-major)
        for (int j = 0; j < kDh / 16; ++j)
          mma_bf16(tmem + TB_DX, desc_k(sb + BS_DZ, kT, j), desc_k(sb + BS_W, kDin, j),
                   idesc_bf16(kT, kDin, false, false), j > 0);
        // dW[i][j] += sum_t x[t][i] dz[t][j]: A = x^T (MN-major), B = dz (K rows, MN-major)
        for (int j = 0; j < kT / 16; ++j)
          mma_bf16(tmem + TB_DW, desc_mn(sb + BS_X, kT, j), desc_mn(sb + BS_DZ, kT, j),
                   idesc_bf16(kDin, kDh, true, true), i > 0 || j > 0);
        mma_commit(&ctl->bar[FB_OUT]);
      }
      mma_commit(&ctl->bar[FB_DONE]);
      drain_bar(ctl, FB_DONE, 1, globaltimer_ns());
    }
  } else {
    const int qw = warp & 3, r = qw * 32 + lane;  // token row, then input-feature row
    const uint32_t tl = tmem + ((uint32_t)(qw * 32) << 16);
    // every epilogue thread runs all iterations (each holds a named barrier); once a wait
    // fails the remaining ones return at once and only the barriers are kept
    bool ok = true;
    for (int i = 0; i < ntiles; ++i) {
      const int t0 = (tile0 + i) * kT;
      if (ok) ok = wait_bar(ctl, FB_Z, i & 1);
      if (ok) {
        tc_fence_after();
        // dz = dphi+ e^z - dphi- e^-z; rows beyond L hold zero dphi and give dz = 0
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          uint32_t z[32];
          tmem_ld32(tl + TB_Z + 32 * g, z);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int c0 = 32 * g + 16 * h;
            float dz[16];
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              const uint4 a = *reinterpret_cast<const uint4*>(sm + BS_DP + sw128_offset(r, c0 + 8 * m, kT));
              const uint4 b = *reinterpret_cast<const uint4*>(sm + BS_DP + sw128_offset(r, kDh + c0 + 8 * m, kT));
              const uint32_t aa[4] = {a.x, a.y, a.z, a.w}, bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float z0 = __uint_as_float(z[16 * h + 8 * m + 2 * e]);
                const float z1 = __uint_as_float(z[16 * h + 8 * m + 2 * e + 1]);
                dz[8 * m + 2 * e] = __uint_as_float(aa[e] << 16) * __expf(z0) -
                                    __uint_as_float(bb[e] << 16) * __expf(-z0);
                dz[8 * m + 2 * e + 1] = __uint_as_float(aa[e] & 0xffff0000u) * __expf(z1) -
                                        __uint_as_float(bb[e] & 0xffff0000u) * __expf(-z1);
              }
            }
            store16_bf16(sm + BS_DZ, kT, r, c0, dz);
          }
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(&ctl->bar[FB_DZ]);
      if (ok) ok = wait_bar(ctl, FB_OUT, i & 1);
      if (ok) {
        tc_fence_after();
        // dx is staged over this thread's own (already read) row of dphi
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
          uint32_t v[32];
          tmem_ld32(tl + TB_DX + 32 * g, v);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) w[e] = __uint_as_float(v[16 * h + e]);
            store16_bf16(sm + BS_DP, kT, r, 32 * g + 16 * h, w);
          }
        }
        tc_fence_before();
        fence_proxy_async_smem();
      }
      named_sync(1, 128);
      if (threadIdx.x == 64) {
        if (ok) {
          tma_store_3d(&maps.out, sm + BS_DP, 0, t0, bh);
          tma_store_3d(&maps.out, sm + BS_DP + 16384, 64, t0, bh);
          bulk_commit();
          bulk_wait_read();
        }
        mbar_arrive(&ctl->bar[FB_FREE]);
      }
    }
    if (ok) {
      // this CTA's part of dW: lane r is input feature r
      tc_fence_after();
      float4* part = reinterpret_cast<float4*>(
          p.dw_part + (((size_t)bh * p.groups + grp) * kDin + r) * kDh);
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        uint32_t v[32];
        tmem_ld32(tl + TB_DW + 32 * g, v);
        tmem_ld_wait();
#pragma unroll
        for (int m = 0; m < 8; ++m)
          part[8 * g + m] = make_float4(__uint_as_float(v[4 * m]), __uint_as_float(v[4 * m + 1]),
                                        __uint_as_float(v[4 * m + 2]), __uint_as_float(v[4 * m + 3]));
      }
    }
  }

  pdl_trigger();
  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
  if (threadIdx.x == 0 && ctl->abort) raise_status(p.status, kDevTimeout);
}

// ------------------------------------------------------------------------------------
// CUDA-core path (any supported D, F; fp32 or bf16 storage, fp32 arithmetic)
// ------------------------------------------------------------------------------------
constexpr int kSimtTok = 32;  // tokens per CTA (forward) or per sub-tile (backward)
constexpr int kSimtAcc = 16384 / 256;  // dW elements per thread, D F <= 16384

template <typename T>
__global__ void __launch_bounds__(256) fmap_fwd_simt_kernel(int H, int L, int D, int F, const T* x,
                                                            const T* w, T* phi) {
  extern __shared__ float fs[];
  float* ws = fs;               // [D][F]
  float* xs = fs + D * F;       // [kSimtTok][D]
  const int bh = blockIdx.y, hh = bh % H, t0 = blockIdx.x * kSimtTok;
  const int nt = min(kSimtTok, L - t0);
  pdl_wait();
  for (int e = threadIdx.x; e < D * F; e += blockDim.x) ws[e] = ld_f(w + (size_t)hh * D * F + e);
  for (int e = threadIdx.x; e < nt * D; e += blockDim.x)
    xs[e] = ld_f(x + ((size_t)bh * L + t0) * D + e);
  __syncthreads();
  for (int e = threadIdx.x; e < nt * F; e += blockDim.x) {
    const int t = e / F, f = e % F;
    float z = 0.f;
    for (int d = 0; d < D; ++d) z = fmaf(xs[t * D + d], ws[d * F + f], z);
    T* out = phi + ((size_t)bh * L + t0 + t) * 2 * F;
    out[f] = cvt_out<T>(expf(z));
    out[F + f] = cvt_out<T>(expf(-z));
  }
  pdl_trigger();
}

// One CTA per (b, h, group of kTokPerGroup tokens), walked in sub-tiles of kSimtTok;
// the CTA's part of dW is accumulated in registers (thread t holds elements t, t + 256, ...).
template <typename T>
__global__ void __launch_bounds__(256) fmap_bwd_simt_kernel(int H, int L, int D, int F, int groups,
                                                            const T* x, const T* w, const T* dphi,
                                                            T* dx, float* part) {
  extern __shared__ float fs[];
  float* ws = fs;                       // [D][F]
  float* xs = ws + D * F;               // [kSimtTok][D]
  float* dzs = xs + kSimtTok * D;       // [kSimtTok][F]
  const int bh = blockIdx.y, hh = bh % H;
  const int DF = D * F;
  float acc[kSimtAcc];
#pragma unroll
  for (int k = 0; k < kSimtAcc; ++k) acc[k] = 0.f;
  pdl_wait();
  for (int e = threadIdx.x; e < DF; e += blockDim.x) ws[e] = ld_f(w + (size_t)hh * DF + e);
  const int g0 = blockIdx.x * kTokPerGroup, g1 = min(L, g0 + kTokPerGroup);
  for (int t0 = g0; t0 < g1; t0 += kSimtTok) {
    const int nt = min(kSimtTok, g1 - t0);
    __syncthreads();  // the previous sub-tile's xs / dzs are no longer read
    for (int e = threadIdx.x; e < nt * D; e += blockDim.x)
      xs[e] = ld_f(x + ((size_t)bh * L + t0) * D + e);
    __syncthreads();
    for (int e = threadIdx.x; e < nt * F; e += blockDim.x) {
      const int t = e / F, f = e % F;
      float z = 0.f;
      for (int d = 0; d < D; ++d) z = fmaf(xs[t * D + d], ws[d * F + f], z);
      const T* g = dphi + ((size_t)bh * L + t0 + t) * 2 * F;
      dzs[e] = ld_f(g + f) * expf(z) - ld_f(g + F + f) * expf(-z);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < nt * D; e += blockDim.x) {
      const int t = e / D, d = e % D;
      float s = 0.f;
      for (int f = 0; f < F; ++f) s = fmaf(dzs[t * F + f], ws[d * F + f], s);
      dx[((size_t)bh * L + t0 + t) * D + d] = cvt_out<T>(s);
    }
#pragma unroll
    for (int k = 0; k < kSimtAcc; ++k) {
      const int e = threadIdx.x + k * 256;
      if (e < DF) {
        const int d = e / F, f = e % F;
        float s = acc[k];
        for (int t = 0; t < nt; ++t) s = fmaf(xs[t * D + d], dzs[t * F + f], s);
        acc[k] = s;
      }
    }
  }
  float* pp = part + ((size_t)bh * groups + blockIdx.x) * DF;
#pragma unroll
  for (int k = 0; k < kSimtAcc; ++k) {
    const int e = threadIdx.x + k * 256;
    if (e < DF) pp[e] = acc[k];
  }
  pdl_trigger();
}

// dW[h][e] = sum over batch b, then partials p, of part[b][h][p][e]: one thread per (h, e).
__global__ void __launch_bounds__(256) fmap_dw_kernel(int B, int H, int P, int DF, const float* part,
                                                      float* dw) {
  pdl_wait();
  const long n = (long)H * DF;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const int hh = (int)(i / DF), e = (int)(i % DF);
    float s = 0.f;
    for (int b = 0; b < B; ++b) {
      const float* src = part + ((size_t)(b * H + hh) * P) * DF + e;
      for (int q = 0; q < P; ++q) s += src[(size_t)q * DF];
    }
    dw[i] = s;
  }
  pdl_trigger();
}

cudaError_t launch_dw_sum(int B, int H, int P, int DF, const float* part, float* dw,
                          cudaStream_t s, int* launches) {
  const long n = (long)H * DF;
  const int grid = (int)((n + 255) / 256);
  trace_begin("fmap_dw", s);
  const cudaError_t e = launch_pdl(fmap_dw_kernel, dim3(grid), dim3(256), 0, s, B, H, P, DF, part, dw);
  trace_end(s);
  ++*launches;
  return e;
}

int bwd_groups(int L) { return (L + kTokPerGroup - 1) / kTokPerGroup; }
int fwd_simt_ctas(int L) { return (L + kSimtTok - 1) / kSimtTok; }

}  // namespace

bool fmap_tc_supported(int D, int F, lizard_dtype dt) {
  return dt == LIZARD_BF16 && D == kDin && F == kDh && tma_encode_available();
}

bool fmap_simt_supported(int D, int F) {
  return D >= 1 && D <= 256 && F >= 1 && F <= 128 && D * F <= 16384;
}

size_t fmap_bwd_workspace(int B, int H, int L, int D, int F, lizard_dtype dt) {
  (void)dt;
  return align_up((size_t)B * H * bwd_groups(L) * D * F * sizeof(float), 256);
}

cudaError_t launch_fmap_fwd(int B, int H, int L, int D, int F, lizard_dtype dt, const void* x,
                            const void* w, void* phi, unsigned* status, cudaStream_t s,
                            int* launches) {
  if (L == 0) return cudaSuccess;
  if (fmap_tc_supported(D, F, dt)) {
    const int nt = (L + kT - 1) / kT;
    const uint64_t bh = (uint64_t)B * H, Ll = (uint64_t)L;
    FmMaps m;
    const bool ok =
        make_tma_map_bf16(&m.x, x, kDin, Ll, bh, 64, kT, CU_TENSOR_MAP_SWIZZLE_128B) &&
        make_tma_map_bf16(&m.w, w, kDh, kDin, H, kDh, kDin, CU_TENSOR_MAP_SWIZZLE_128B) &&
        make_tma_map_bf16(&m.out, phi, 2 * kDh, Ll, bh, 64, kT, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return cudaErrorInvalidValue;
    m.dphi = m.x;
    const FmParams p{H, nt, 1, nullptr, status};
    cudaError_t e = cudaFuncSetAttribute(fmap_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kFwdSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fmap_fwd_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    trace_begin("fmap_fwd_tc", s);
    e = launch_pdl(fmap_fwd_kernel, dim3(B * H * nt), dim3(kThreads), kFwdSmem, s, m, p);
    trace_end(s);
    ++*launches;
    return e;
  }
  const size_t smem = (size_t)(D * F + kSimtTok * D) * sizeof(float);
  const dim3 grid(fwd_simt_ctas(L), B * H);
  cudaError_t e;
  trace_begin("fmap_fwd_simt", s);
  if (dt == LIZARD_F32) {
    e = cudaFuncSetAttribute(fmap_fwd_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
      e = launch_pdl(fmap_fwd_simt_kernel<float>, grid, dim3(256), smem, s, H, L, D, F,
                     static_cast<const float*>(x), static_cast<const float*>(w), static_cast<float*>(phi));
  } else {
    e = cudaFuncSetAttribute(fmap_fwd_simt_kernel<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
      e = launch_pdl(fmap_fwd_simt_kernel<bf16>, grid, dim3(256), smem, s, H, L, D, F,
                     static_cast<const bf16*>(x), static_cast<const bf16*>(w), static_cast<bf16*>(phi));
  }
  trace_end(s);
  ++*launches;
  return e;
}

cudaError_t launch_fmap_bwd(int B, int H, int L, int D, int F, lizard_dtype dt, const void* x,
                            const void* w, const void* dphi, void* dx, float* dw,
                            unsigned char* ws, unsigned* status, cudaStream_t s, int* launches) {
  float* part = reinterpret_cast<float*>(ws);
  if (L == 0) return cudaMemsetAsync(dw, 0, (size_t)H * D * F * sizeof(float), s);
  if (fmap_tc_supported(D, F, dt)) {
    const int nt = (L + kT - 1) / kT, groups = bwd_groups(L);
    const uint64_t bh = (uint64_t)B * H, Ll = (uint64_t)L;
    FmMaps m;
    const bool ok =
        make_tma_map_bf16(&m.x, x, kDin, Ll, bh, 64, kT, CU_TENSOR_MAP_SWIZZLE_128B) &&
        make_tma_map_bf16(&m.w, w, kDh, kDin, H, kDh, kDin, CU_TENSOR_MAP_SWIZZLE_128B) &&
        make_tma_map_bf16(&m.dphi, dphi, 2 * kDh, Ll, bh, 64, kT, CU_TENSOR_MAP_SWIZZLE_128B) &&
        make_tma_map_bf16(&m.out, dx, kDin, Ll, bh, 64, kT, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return cudaErrorInvalidValue;
    const FmParams p{H, nt, groups, part, status};
    cudaError_t e = cudaFuncSetAttribute(fmap_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kBwdSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fmap_bwd_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    trace_begin("fmap_bwd_tc", s);
    e = launch_pdl(fmap_bwd_kernel, dim3(B * H * groups), dim3(kThreads), kBwdSmem, s, m, p);
    trace_end(s);
    ++*launches;
    if (e != cudaSuccess) return e;
    return launch_dw_sum(B, H, groups, kDin * kDh, part, dw, s, launches);
  }
  const int groups = bwd_groups(L);
  const size_t smem = (size_t)(D * F + kSimtTok * D + kSimtTok * F) * sizeof(float);
  const dim3 grid(groups, B * H);
  cudaError_t e;
  trace_begin("fmap_bwd_simt", s);
  if (dt == LIZARD_F32) {
    e = cudaFuncSetAttribute(fmap_bwd_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
      e = launch_pdl(fmap_bwd_simt_kernel<float>, grid, dim3(256), smem, s, H, L, D, F, groups,
                     static_cast<const float*>(x), static_cast<const float*>(w),
                     static_cast<const float*>(dphi), static_cast<float*>(dx), part);
  } else {
    e = cudaFuncSetAttribute(fmap_bwd_simt_kernel<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
      e = launch_pdl(fmap_bwd_simt_kernel<bf16>, grid, dim3(256), smem, s, H, L, D, F, groups,
                     static_cast<const bf16*>(x), static_cast<const bf16*>(w),
                     static_cast<const bf16*>(dphi), static_cast<bf16*>(dx), part);
  }
  trace_end(s);
  ++*launches;
  if (e != cudaSuccess) return e;
  return launch_dw_sum(B, H, groups, D * F, part, dw, s, launches);
}

}  // namespace lz
