// k_prep_fmap_tc.cu -- the forward's prep pass fused with the Hedgehog feature map, in the
// literal log-space form ("Lizard", arXiv 2507.09025, Method: the gate's cumulative
// products are absorbed into the query and key features; with phi(x) = [exp(xW),
// exp(-xW)] this is exp(+-xW + b) for the queries and exp(+-xW - b) for the keys).
//
// Per (b, h, chunk of 128 tokens), with b the chunk-local inclusive cumulative sum of
// log gamma (one value per key dimension j = 0..127):
//   z_q = x_q W_q, z_k = x_k W_k                       (M=128 N=64 K=128, tcgen05, fp32)
//   Qt[t][j] = exp( z_q[t][j] + b[t][j]),  Qt[t][64+j] = exp(-z_q[t][j] + b[t][64+j])
//   Kt[t][j] = exp( z_k[t][j] - b[t][j]),  Kt[t][64+j] = exp(-z_k[t][j] - b[t][64+j])
//   e^b (bf16), Gamma_c = b at the chunk's last token (fp32)
// which are exactly the context the unfused prep derives from phi_q, phi_k, so the state
// scan, the chunk kernel and a later backward run unchanged.  phi itself is never formed.
// A chunk where some |b| exceeds kMaxLogSum is "wide" (e^{-b} would leave the exponent
// range): its Kt slot gets the bounded exp(+-x W_k + Gamma - b) for the state scan, and
// the chunk is flagged and listed for the exact recomputation, as in the unfused prep.
//
// Warp 0 issues the TMA loads (x_q, x_k, W_q, W_k and the 128x128 fp32 log-gate tile, all
// in flight at once) and warms L2 with the tiles of the CTA one wave later; warp 1 issues
// the two MMAs; warps 2-5 first walk the log-gate tile down its columns (thread = key
// dimension) turning it into b in place, then take one token row each to exponentiate
// and stage Qt, Kt, e^b in the shared memory the MMAs have finished with.
#include "lizard_dev.cuh"
#include "lizard_internal.h"
#include "tc_pipe.cuh"

namespace lz {
namespace {

using namespace tc;

constexpr int kT = 128;   // tokens per chunk (the forward's chunk)
constexpr int kD = 128;   // x features and key dimensions
constexpr int kF = 64;    // columns of each W
constexpr int kThreads = 6 * 32;
constexpr float kMaxLogSum = 80.f;  // |b| beyond which e^{+-b} leaves the fp32/bf16 range

struct PfMaps {
  CUtensorMap xq, xk, wq, wk, lg;  // loads
  CUtensorMap qt, kt, eb;          // stores
};

struct PfParams {
  int H, L, nc;
  int ahead;    // CTAs per wave: the CTA whose tiles this one prefetches into L2
  float* gam;   // [BH][nc][128]
  unsigned* status;
  int *wide, *wlist;  // wide-chunk flags and list [BH][nc]
  unsigned* wcount;
};

enum { P_LD = 0, P_Z, P_DONE, P_COUNT };
// x_q, x_k 32 KB each (then the Qt, Kt staging); W_q, W_k 16 KB each (then the e^b
// staging); the log-gate tile 64 KB fp32 (four 32-column blocks), turned into b in place
constexpr uint32_t PS_XQ = 0, PS_XK = 32768, PS_W = 65536, PS_LG = PS_W + 32768,
                   PS_BARS = PS_LG + 65536;
constexpr size_t kSmem = PS_BARS + 1024 + 1024;
constexpr uint32_t kLoadBytes = 2 * 32768 + 2 * 16384 + 65536;

__global__ void __launch_bounds__(kThreads, 1) prep_fmap_kernel(const __grid_constant__ PfMaps maps,
                                                                const PfParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  using C = Ctl<P_COUNT>;
  C* ctl = reinterpret_cast<C*>(sm + PS_BARS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x % p.nc, bh = blockIdx.x / p.nc, hh = bh % p.H;
  const int t0 = c * kT, n = min(kT, p.L - t0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < P_COUNT; ++i) mbar_init(&ctl->bar[i], 1u);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      uint64_t* bar = &ctl->bar[P_LD];
      mbar_arrive_expect_tx(bar, kLoadBytes);
      tma_load_3d(sm + PS_XQ, &maps.xq, 0, t0, bh, bar);
      tma_load_3d(sm + PS_XQ + 16384, &maps.xq, 64, t0, bh, bar);
      tma_load_3d(sm + PS_XK, &maps.xk, 0, t0, bh, bar);
      tma_load_3d(sm + PS_XK + 16384, &maps.xk, 64, t0, bh, bar);
      tma_load_3d(sm + PS_W, &maps.wq, 0, 0, hh, bar);
      tma_load_3d(sm + PS_W + 16384, &maps.wk, 0, 0, hh, bar);
      for (int x = 0; x < kD; x += 32) tma_load_3d(sm + PS_LG + x * 512, &maps.lg, x, t0, bh, bar);
      // warm L2 with the tiles of the CTA one wave later, once this one's have landed
      const int nb = blockIdx.x + p.ahead;
      if (nb < (int)gridDim.x && wait_bar(ctl, P_LD, 0)) {
        const int nt0 = (nb % p.nc) * kT, nbh = nb / p.nc;
        for (int x = 0; x < kD; x += 64) {
          tma_prefetch_l2_3d(&maps.xq, x, nt0, nbh);
          tma_prefetch_l2_3d(&maps.xk, x, nt0, nbh);
        }
        for (int x = 0; x < kD; x += 32) tma_prefetch_l2_3d(&maps.lg, x, nt0, nbh);
      }
      drain_bar(ctl, P_LD, 1, globaltimer_ns());
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t sb = smem_u32(sm);
      const bool ok = wait_bar(ctl, P_LD, 0);
      if (ok) {
        tc_fence_after();
        // z[t][j] = sum_d x[t][d] W[d][j]: A = x (K-major), B = W (K rows, MN-major)
        for (int j = 0; j < kD / 16; ++j)
          mma_bf16(tmem, desc_k(sb + PS_XQ, kT, j), desc_mn(sb + PS_W, kD, j),
                   idesc_bf16(kT, kF, false, true), j > 0);
        for (int j = 0; j < kD / 16; ++j)
          mma_bf16(tmem + kF, desc_k(sb + PS_XK, kT, j), desc_mn(sb + PS_W + 16384, kD, j),
                   idesc_bf16(kT, kF, false, true), j > 0);
        mma_commit(&ctl->bar[P_Z]);
      }
      mma_commit(&ctl->bar[P_DONE]);
      drain_bar(ctl, P_DONE, 1, globaltimer_ns());
    }
  } else {
    const int et = threadIdx.x - 64;              // 0..127
    const int qw = warp & 3, t = qw * 32 + lane;  // token row of the chunk (TMEM lane)
    const uint32_t tl = tmem + ((uint32_t)(qw * 32) << 16);
    unsigned char* lgs = sm + PS_LG;
    float big = 0.f;
    bool ok = wait_bar(ctl, P_LD, 0);
    if (ok) {
      // b: inclusive sums down the chunk, thread et = key dimension; rows at or beyond L
      // were loaded as zeros and carry b of the last token
      // (eight rows loaded before any is written back, so the loads need not wait for
      // the stores)
      const int j = et;
      float run = 0.f;
#pragma unroll 1
      for (int r0 = 0; r0 < kT; r0 += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          v[u] = *reinterpret_cast<const float*>(lgs + sw128_offset_f32(r0 + u, j, kT));
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          run += v[u];
          v[u] = run;
          if (r0 + u < n) big = fmaxf(big, fabsf(run));
          if (r0 + u == n - 1) p.gam[((size_t)bh * p.nc + c) * kD + j] = run;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<float*>(lgs + sw128_offset_f32(r0 + u, j, kT)) = v[u];
      }
    }
    const bool wide = named_sync_or(1, 128, big > kMaxLogSum);
    if (ok) ok = wait_bar(ctl, P_Z, 0);
    if (ok) {
      tc_fence_after();
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {  // 32 key dimensions at a time
        // dimensions 0..63 take +z, 64..127 take -z of the same column of z
        const uint32_t zc = (uint32_t)((32 * g) & 63);
        uint32_t zq[32], zk[32];
        tmem_ld32(tl + zc, zq);
        tmem_ld32(tl + kF + zc, zk);
        tmem_ld_wait();
        const float sgn = g < 2 ? 1.f : -1.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float bv[16], gv[16], vq[16], vk[16], ve[16];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const float4 v = *reinterpret_cast<const float4*>(
                lgs + sw128_offset_f32(t, 32 * g + 16 * h + 4 * m, kT));
            bv[4 * m] = v.x;
            bv[4 * m + 1] = v.y;
            bv[4 * m + 2] = v.z;
            bv[4 * m + 3] = v.w;
            // a wide chunk's keys are referred to the chunk end: Gamma = b of its last token
            const float4 G = wide ? *reinterpret_cast<const float4*>(
                                        lgs + sw128_offset_f32(n - 1, 32 * g + 16 * h + 4 * m, kT))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            gv[4 * m] = G.x;
            gv[4 * m + 1] = G.y;
            gv[4 * m + 2] = G.z;
            gv[4 * m + 3] = G.w;
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int i = 16 * h + e;
            vq[e] = __expf(fmaf(sgn, __uint_as_float(zq[i]), bv[e]));
            vk[e] = __expf(fmaf(sgn, __uint_as_float(zk[i]), gv[e] - bv[e]));
            ve[e] = __expf(bv[e]);
          }
          // staged over x_q, x_k and the W tiles, which the (completed) MMAs no longer read
          store16_bf16(sm + PS_XQ, kT, t, 32 * g + 16 * h, vq);
          store16_bf16(sm + PS_XK, kT, t, 32 * g + 16 * h, vk);
          store16_bf16(sm + PS_W, kT, t, 32 * g + 16 * h, ve);
        }
      }
    }
    fence_proxy_async_smem();
    named_sync(1, 128);
    if (ok && threadIdx.x == 64) {
      // rows at or beyond L are clipped by the stores
      for (int x = 0; x < kD; x += 64) {
        const uint32_t off = (uint32_t)(x / 64) * 16384u;
        tma_store_3d(&maps.qt, sm + PS_XQ + off, x, t0, bh);
        tma_store_3d(&maps.kt, sm + PS_XK + off, x, t0, bh);
        tma_store_3d(&maps.eb, sm + PS_W + off, x, t0, bh);
      }
      bulk_commit();
      bulk_wait_read();
    }
    if (threadIdx.x == 64) {
      p.wide[(size_t)bh * p.nc + c] = wide ? 1 : 0;
      if (wide) p.wlist[atomicAdd(p.wcount, 1u)] = bh * p.nc + c;
    }
  }

  pdl_trigger();
  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
  if (threadIdx.x == 0 && ctl->abort) raise_status(p.status, kDevTimeout);
}

}  // namespace

cudaError_t launch_gla_prep_fmap(const GlaStatesArgs& a, int H, const void* xq, const void* xk,
                                 const void* wq, const void* wk, cudaStream_t s, int* launches) {
  const int nc = (a.L + kT - 1) / kT;
  const uint64_t bhl = (uint64_t)a.BH, Ll = (uint64_t)a.L;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  PfMaps m;
  const bool ok = make_tma_map_bf16(&m.xq, xq, kD, Ll, bhl, 64, kT, sw) &&
                  make_tma_map_bf16(&m.xk, xk, kD, Ll, bhl, 64, kT, sw) &&
                  make_tma_map_bf16(&m.wq, wq, kF, kD, H, kF, kD, sw) &&
                  make_tma_map_bf16(&m.wk, wk, kF, kD, H, kF, kD, sw) &&
                  make_tma_map_f32(&m.lg, a.lg, kD, Ll, bhl, 32, kT, sw) &&
                  make_tma_map_bf16(&m.qt, a.qt, kD, Ll, bhl, 64, kT, sw) &&
                  make_tma_map_bf16(&m.kt, a.kt, kD, Ll, bhl, 64, kT, sw) &&
                  make_tma_map_bf16(&m.eb, a.eb, kD, Ll, bhl, 64, kT, sw);
  if (!ok) return cudaErrorInvalidValue;
  const PfParams p{H, a.L, nc, ctas_per_wave(1), a.gam, a.status, a.wide, a.wlist, a.wcount};
  cudaError_t e = cudaFuncSetAttribute(prep_fmap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(prep_fmap_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  trace_begin("fwd_prep_fmap", s);
  e = launch_pdl(prep_fmap_kernel, dim3(nc * a.BH), dim3(kThreads), kSmem, s, m, p);
  trace_end(s);
  ++*launches;
  return e;
}

}  // namespace lz
