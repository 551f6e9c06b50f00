// k_gla_states_tc.cu -- the two passes the chunk-parallel GLA kernels (forward and
// backward) start from, for bf16 with dk = dv = 128 and 128-token chunks.
//
//   prep  (CUDA cores)  b = chunk-local inclusive cumsum of log gamma, Gamma = its last
//                       value; Qt = phi_q e^b and Kt = phi_k e^-b in bf16 (and e^b when
//                       asked), Gamma in fp32 ("Lizard", arXiv 2507.09025, Method:
//                       parallel form with cumulative gate products, absorbed in log space
//                       into the features).  e^-b is finite only while |b| stays inside
//                       the exponent range; a chunk where some |b| exceeds kMaxLogSum is
//                       "wide": its Kt slot gets the bounded Kh = phi_k e^{Gamma - b}
//                       instead, and the chunk is flagged and listed for an exact
//                       recomputation (k_fwd_simt.cu, k_bwd_simt.cu).
//   scan  (tcgen05)     the state at every chunk start (direction 0)
//                         h_0 = h0,  h_{c+1} = diag(e^Gamma_c) (h_c + Kt_c^T V_c)
//                                           = diag(e^Gamma_c) h_c + Kh_c^T V_c   (wide c)
//                       and, for the backward, the adjoint of the state at every chunk
//                       end (direction 1)
//                         G_{nc-1} = 0,  G_{c-1} = diag(e^Gamma_c) G_c + Qt_c^T dY_c
//                       stored as bf16 h_c and Gt_c = diag(e^Gamma_c) G_c (G_c itself for a
//                       wide chunk, whose recomputation needs it unscaled); h_nc is h_final
//                       and G_{-1} the adjoint of h0 (fp32).  Every operand is bounded by
//                       the features (b <= 0 for gates in (0, 1]), so the scans stay finite
//                       for every gate.  One CTA per (b, h, 32 dv
//                       columns, direction): warp 0 streams the chunks by TMA through a
//                       ring of 5 (or, two CTAs to an SM, 2) stages, warp 1 issues one
//                       M=128 N=32 K=128 product per chunk into one TMEM tile per stage,
//                       and the scan warps (thread = state row x 32 columns) run the
//                       recurrence in fp32 registers.
#include "lizard_dev.cuh"
#include "lizard_internal.h"
#include "tc_pipe.cuh"

namespace lz {
namespace {

using namespace tc;

constexpr int kC = kGlaChunk;
constexpr int kD = 128;
constexpr float kMaxLogSum = 80.f;  // |chunk-local log-gate sum| beyond which e^{+-b} overflows

// ------------------------------------------------------------------------------------
// prep: one CTA per (chunk, b*h) of 64 threads, each owning two adjacent key dimensions
// (4-byte bf16 pairs, 8-byte log-gate pairs), eight tokens' loads in flight.
// ------------------------------------------------------------------------------------
constexpr int kPrepThreads = kD / 2;

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const GlaStatesArgs p, int nc) {
  const int c = blockIdx.x, bh = blockIdx.y, i2 = threadIdx.x;  // columns 2 i2, 2 i2 + 1
  const int L = p.L, t0 = c * kC, n = min(kC, L - t0);
  const size_t base = ((size_t)bh * L + t0) * (kD / 2) + i2;  // in pairs
  pdl_wait();
  const __nv_bfloat162* pq = reinterpret_cast<const __nv_bfloat162*>(p.pq) + base;
  const __nv_bfloat162* pk = reinterpret_cast<const __nv_bfloat162*>(p.pk) + base;
  const float2* lg = reinterpret_cast<const float2*>(p.lg) + base;
  __nv_bfloat162* qt = reinterpret_cast<__nv_bfloat162*>(p.qt) + base;
  __nv_bfloat162* kt = reinterpret_cast<__nv_bfloat162*>(p.kt) + base;
  __nv_bfloat162* eb = p.eb ? reinterpret_cast<__nv_bfloat162*>(p.eb) + base : nullptr;
  float r0 = 0.f, r1 = 0.f, big = 0.f;
  for (int t8 = 0; t8 < n; t8 += 8) {
    float2 lv[8];
    __nv_bfloat162 qv[8], kv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const bool ok = t8 + u < n;
      const size_t o = (size_t)(t8 + u) * (kD / 2);
      lv[u] = ok ? lg[o] : make_float2(0.f, 0.f);
      qv[u] = ok ? pq[o] : __floats2bfloat162_rn(0.f, 0.f);
      kv[u] = ok ? pk[o] : __floats2bfloat162_rn(0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (t8 + u < n) {
        r0 += lv[u].x;
        r1 += lv[u].y;
        big = fmaxf(big, fmaxf(fabsf(r0), fabsf(r1)));
        const float e0 = __expf(r0), e1 = __expf(r1);
        const float2 q = __bfloat1622float2(qv[u]), k = __bfloat1622float2(kv[u]);
        const size_t o = (size_t)(t8 + u) * (kD / 2);
        qt[o] = __floats2bfloat162_rn(q.x * e0, q.y * e1);
        kt[o] = __floats2bfloat162_rn(k.x * __expf(-r0), k.y * __expf(-r1));
        if (eb) eb[o] = __floats2bfloat162_rn(e0, e1);
      }
    }
  }
  reinterpret_cast<float2*>(p.gam)[((size_t)bh * nc + c) * (kD / 2) + i2] = make_float2(r0, r1);
  // A wide chunk (e^{-b} out of range for some key dimension): the Kt slot gets the
  // bounded Kh = phi_k e^{Gamma - b} for the state scan, recomputing b in the same order.
  const int wide = __syncthreads_or(big > kMaxLogSum);
  if (wide) {
    float s0 = 0.f, s1 = 0.f;
    for (int t = 0; t < n; ++t) {
      const size_t o = (size_t)t * (kD / 2);
      const float2 l = lg[o];
      s0 += l.x;
      s1 += l.y;
      const float2 k = __bfloat1622float2(pk[o]);
      kt[o] = __floats2bfloat162_rn(k.x * expf(r0 - s0), k.y * expf(r1 - s1));
    }
  }
  if (i2 == 0) {
    p.wide[(size_t)bh * nc + c] = wide;
    if (wide) p.wlist[atomicAdd(p.wcount, 1u)] = bh * nc + c;
  }
  pdl_trigger();
}

// ------------------------------------------------------------------------------------
// scan
// ------------------------------------------------------------------------------------
struct ScanMaps {
  CUtensorMap x0, y0, x1, y1;  // direction 0: Kt, V ; direction 1: Qt, dY
};

constexpr uint32_t kScanX = kC * kD * 2;  // 32 KB: Kt or Qt tile
constexpr int kGamAhead = 32;  // chunk decays fetched per refill by each scan row

// SL value columns per CTA (32 or 64) and kStages chunks in flight (TMA ring and TMEM
// buffers).  The Y slice (V or dY) is a 64-byte-swizzled 32-column tile when SL = 32 and a
// 128-byte-swizzled 64-column block when SL = 64.  One scan warp per (TMEM lane quarter,
// 32 columns): every scan thread carries 32 state columns of one row, whatever SL is.
//
// Each tcgen05 instruction the single MMA thread issues costs it on the order of 100 SM
// cycles, whatever the tile's N: a chunk's eight K = 16 MMAs and its commit take ~0.4 us,
// the pace of the chain when the operands are in L2; from DRAM the copies set it.  One
// commit per chunk tells both the producer (stage free) and the scan threads
// (accumulator full).
template <int kStages, int SL>
struct ScanCfg {
  enum { S_FULL = 0, S_DFULL = kStages, S_DFREE = 2 * kStages, S_DONE = 3 * kStages, S_COUNT };
  static constexpr int kScanWarps = 4 * (SL / 32);
  static constexpr int kThreads = (2 + kScanWarps) * 32;
  static constexpr uint32_t kY = kC * SL * 2;
  static constexpr uint32_t kStage = kScanX + kY;  // multiple of 1024
  // each scan warp's rows' next kGamAhead chunk decays, [SL / 32][kGamAhead][128] fp32
  static constexpr uint32_t kGam = kStages * kStage;
  static constexpr uint32_t kBars = kGam + (SL / 32) * kGamAhead * kD * 4;
  static constexpr size_t kSmem = kBars + 1024 + 1024;
  static constexpr uint32_t kTmemCols = kStages * SL <= 32 ? 32 : kStages * SL <= 64 ? 64
                                      : kStages * SL <= 128 ? 128 : kStages * SL <= 256 ? 256 : 512;
  static_assert(SL == 32 || SL == 64, "slice width");
  static_assert(kStages * SL <= 512, "TMEM budget");
  static_assert(kSmem <= 232448, "shared memory per CTA");
};

template <int kStages, int SL>
__global__ void __launch_bounds__(ScanCfg<kStages, SL>::kThreads, 1)
scan_kernel(const __grid_constant__ ScanMaps maps, const GlaStatesArgs p, int nc, int ndir,
            int dir0, int nseg, int cps, float* segf0, float* segf1) {
  using SC = ScanCfg<kStages, SL>;
  enum { S_FULL = SC::S_FULL, S_DFULL = SC::S_DFULL, S_DFREE = SC::S_DFREE,
         S_DONE = SC::S_DONE, S_COUNT = SC::S_COUNT };
  constexpr int kSlicesT = kD / SL;
  constexpr uint32_t kScanBars = SC::kBars, kStageB = SC::kStage;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  using C = Ctl<S_COUNT>;
  C* ctl = reinterpret_cast<C*>(sm + kScanBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int dir = ndir == 2 ? (blockIdx.x & 1) : dir0;
  const int sl = (blockIdx.x / ndir) % kSlicesT;
  const int seg = (blockIdx.x / (ndir * kSlicesT)) % nseg;
  const int bh = blockIdx.x / (ndir * kSlicesT * nseg);
  // this CTA's chunks [cb, ce): the whole sequence, or one segment of a split sequence
  // (each segment scanned from zero; the segments are joined afterwards)
  const int cb = seg * cps, ce = min(nc, cb + cps), nl = ce - cb;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S_COUNT; ++i)
      mbar_init(&ctl->bar[i], (i >= S_DFREE && i < S_DFREE + kStages) ? 32u * SC::kScanWarps : 1u);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem, SC::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      const CUtensorMap* mx = dir ? &maps.x1 : &maps.x0;
      const CUtensorMap* my = dir ? &maps.y1 : &maps.y0;
      uint32_t armed[kStages] = {};
      bool ok = true;
      for (int u = 0; u < nl && ok; ++u) {
        const int c = dir ? ce - 1 - u : cb + u, s = u % kStages, k = u / kStages;
        // the stage is free once the MMAs of its previous chunk have completed
        if (k >= 1 && !(ok = wait_bar(ctl, S_DFULL + s, (k - 1) & 1))) break;
        unsigned char* st = sm + s * kStageB;
        mbar_arrive_expect_tx(&ctl->bar[S_FULL + s], kStageB);
        tma_load_3d(st, mx, 0, c * kC, bh, &ctl->bar[S_FULL + s]);
        tma_load_3d(st + kScanX / 2, mx, 64, c * kC, bh, &ctl->bar[S_FULL + s]);
        if (SL == 32) {
          tma_load_3d(st + kScanX, my, sl * SL, c * kC, bh, &ctl->bar[S_FULL + s]);
        } else {
#pragma unroll
          for (int b64 = 0; b64 < SL / 64; ++b64)
            tma_load_3d(st + kScanX + b64 * (kC * 128), my, sl * SL + 64 * b64, c * kC, bh,
                        &ctl->bar[S_FULL + s]);
        }
#pragma unroll
        for (int r = 0; r < kStages; ++r) armed[r] += r == s ? 1u : 0u;
      }
      if (!ok) ctl->abort = 1;
      const uint64_t t0 = globaltimer_ns();
#pragma unroll
      for (int r = 0; r < kStages; ++r) drain_bar(ctl, S_FULL + r, armed[r], t0);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // D[i][j] = sum_s X[s][i] Y[s][j]: A = X^T (MN-major), B = Y slice (MN-major)
      const uint32_t id = idesc_bf16(kD, SL, true, true);
      const uint32_t sbase = smem_u32(sm);
      // stage 0's operand descriptors; k-step j of a stage adds j * 2048 bytes (16 token rows
      // of 128 B) to A and j * kBStep to B (16 rows of the 64-byte-swizzled 32-column slice,
      // or of the 128-byte-swizzled 64-column block)
      constexpr uint32_t kBStep = SL == 32 ? 1024 : 2048;
      const uint64_t a0 = desc_mn(sbase, kC, 0);
      const uint64_t b0 = SL == 32 ? smem_desc(sbase + kScanX, kC * 64, 512, kSw64)
                                   : desc_mn(sbase + kScanX, kC, 0);
      bool ok = true;
      for (int u = 0; u < nl && ok; ++u) {
        const int s = u % kStages, k = u / kStages;
        if (!(ok = wait_bar(ctl, S_FULL + s, k & 1))) break;
        if (k >= 1 && !(ok = wait_bar(ctl, S_DFREE + s, (k - 1) & 1))) break;
        tc_fence_after();
        // descriptors differ only in the start address (16-byte units, low 14 bits)
        const uint64_t soff = (uint64_t)((s * kStageB) >> 4);
        const uint64_t ad = a0 + soff, bd = b0 + soff;
        const uint32_t dt = tmem + s * SL;
#pragma unroll
        for (int j = 0; j < kC / 16; ++j)
          mma_bf16(dt, ad + (uint64_t)(j * 2048 / 16), bd + (uint64_t)(j * kBStep / 16), id, j > 0);
        mma_commit(&ctl->bar[S_DFULL + s]);
      }
      if (!ok) ctl->abort = 1;
      mma_commit(&ctl->bar[S_DONE]);
      drain_bar(ctl, S_DONE, 1, globaltimer_ns());
    }
  } else {
    // scan warp e: TMEM lane quarter warp % 4 (the quarter a warp may reach), columns
    // 32 * (e / 4) .. + 31 of the slice
    const int qw = warp & 3, cq = (warp - 2) >> 2;
    const int i = qw * 32 + lane;  // state row = TMEM lane
    const int col = sl * SL + 32 * cq;  // first value column of this thread
    const uint32_t tl = tmem + ((uint32_t)(qw * 32) << 16) + 32 * cq;
    float x[32];
    if (dir == 0 && nseg == 1 && p.h0) {  // a split scan joins h0 in afterwards
      const float4* src = reinterpret_cast<const float4*>(p.h0 + ((size_t)bh * kD + i) * kD + col);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float4 v = src[k];
        x[4 * k] = v.x;
        x[4 * k + 1] = v.y;
        x[4 * k + 2] = v.z;
        x[4 * k + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) x[k] = 0.f;
    }
    bf16* outb = dir ? p.gs : p.hs;
    bool ok = true;
    // The chunk decays sit on the scan's chain: each row fetches its next kGamAhead of them
    // with independent loads into its own column of shared memory (read back by the same
    // thread only), so a global load's latency is paid once per kGamAhead chunks.
    float* gsm = reinterpret_cast<float*>(sm + SC::kGam) + cq * kGamAhead * kD;
    uint32_t wbits = 0;  // bit v: chunk u + v of the current batch is wide
    for (int u = 0; u < nl && ok; ++u) {
      const int c = dir ? ce - 1 - u : cb + u, s = u % kStages;
      if (u % kGamAhead == 0) {
        const int cnt = min(kGamAhead, nl - u);
        float gv[kGamAhead];
        int wv[kGamAhead];
#pragma unroll
        for (int v = 0; v < kGamAhead; ++v) {
          const int cv = dir ? ce - 1 - (u + v) : cb + u + v;
          gv[v] = v < cnt ? p.gam[((size_t)bh * nc + cv) * kD + i] : 0.f;
          wv[v] = v < cnt ? p.wide[(size_t)bh * nc + cv] : 0;
        }
        wbits = 0;
#pragma unroll
        for (int v = 0; v < kGamAhead; ++v) {
          gsm[v * kD + i] = gv[v];
          wbits |= (wv[v] != 0 ? 1u : 0u) << v;
        }
      }
      const bool wide = (wbits >> (u % kGamAhead)) & 1u;
      const float g = expf(gsm[(u % kGamAhead) * kD + i]);
      if (!(ok = wait_bar(ctl, S_DFULL + s, (u / kStages) & 1))) break;
      tc_fence_after();
      uint4* dst = reinterpret_cast<uint4*>(outb + (((size_t)bh * nc + c) * kD + i) * kD + col);
      uint32_t d[32];
      tmem_ld32(tl + s * SL, d);
      tmem_ld_wait();
      // a wide chunk keeps its adjoint unscaled (stored before the decay is applied)
      if (dir && !wide) {
#pragma unroll
        for (int k = 0; k < 32; ++k) x[k] *= g;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        dst[k] = make_uint4(pack_bf16x2(x[8 * k], x[8 * k + 1]), pack_bf16x2(x[8 * k + 2], x[8 * k + 3]),
                            pack_bf16x2(x[8 * k + 4], x[8 * k + 5]), pack_bf16x2(x[8 * k + 6], x[8 * k + 7]));
      if (dir) {
        if (wide) {
#pragma unroll
          for (int k = 0; k < 32; ++k) x[k] = fmaf(g, x[k], __uint_as_float(d[k]));
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) x[k] += __uint_as_float(d[k]);
        }
      } else if (wide) {  // Kh^T V is already decayed to the chunk end
#pragma unroll
        for (int k = 0; k < 32; ++k) x[k] = fmaf(g, x[k], __uint_as_float(d[k]));
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) x[k] = g * (x[k] + __uint_as_float(d[k]));
      }
      tc_fence_before();
      mbar_arrive(&ctl->bar[S_DFREE + s]);
    }
    if (!ok) ctl->abort = 1;
    // the final state (h_final / d h0), or this segment's state from zero for the join
    float* fin = nullptr;
    if (nseg > 1)
      fin = (dir ? segf1 : segf0) + (size_t)(bh * nseg + seg) * kD * kD;
    else if (float* f = dir ? p.dh0 : p.hf)
      fin = f + (size_t)bh * kD * kD;
    if (ok && fin) {
      float4* dst = reinterpret_cast<float4*>(fin + (size_t)i * kD + col);
#pragma unroll
      for (int k = 0; k < 8; ++k) dst[k] = make_float4(x[4 * k], x[4 * k + 1], x[4 * k + 2], x[4 * k + 3]);
    }
  }

  pdl_trigger();
  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, SC::kTmemCols);
  }
  if (threadIdx.x == 0 && ctl->abort) raise_status(p.status, kDevTimeout);
}

}  // namespace

cudaError_t launch_gla_prep(const GlaStatesArgs& a, cudaStream_t s, int* launches) {
  const int nc = (a.L + kC - 1) / kC;
  trace_begin(a.dy ? "bwd_prep" : "fwd_prep", s);
  cudaError_t e = launch_pdl(prep_kernel, dim3(nc, a.BH), dim3(kPrepThreads), 0, s, a, nc);
  trace_end(s);
  ++*launches;
  return e;
}

template <int kStages, int SL>
cudaError_t scan_variant(const GlaStatesArgs& a, bool states, bool adjoints, int nc, int nseg,
                         int cps, float* segf0, float* segf1, cudaStream_t s) {
  using SC = ScanCfg<kStages, SL>;
  const uint64_t bhl = (uint64_t)a.BH, Ll = (uint64_t)a.L;
  const uint32_t ybox = SL == 32 ? 32 : 64;
  const CUtensorMapSwizzle ysw = SL == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  ScanMaps m;
  bool ok = true;
  if (states)
    ok = make_tma_map_bf16(&m.x0, a.kt, kD, Ll, bhl, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_tma_map_bf16(&m.y0, a.v, kD, Ll, bhl, ybox, kC, ysw);
  if (adjoints)
    ok = ok && make_tma_map_bf16(&m.x1, a.qt, kD, Ll, bhl, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_tma_map_bf16(&m.y1, a.dy, kD, Ll, bhl, ybox, kC, ysw);
  if (!ok) return cudaErrorInvalidValue;
  if (!states) {
    m.x0 = m.x1;
    m.y0 = m.y1;
  }
  if (!adjoints) {
    m.x1 = m.x0;
    m.y1 = m.y0;
  }
  const int ndir = states && adjoints ? 2 : 1;
  const int dir0 = states ? 0 : 1;
  const int grid = a.BH * (kD / SL) * ndir * nseg;
  auto kern = scan_kernel<kStages, SL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SC::kSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(SC::kThreads), SC::kSmem, s, m, a, nc, ndir, dir0,
                    nseg, cps, segf0, segf1);
}

cudaError_t launch_gla_scan(const GlaStatesArgs& a, GlaScan which, cudaStream_t s, int* launches) {
  const int nc = (a.L + kC - 1) / kC;
  const bool states = which != GlaScan::kAdjoints, adjoints = which != GlaScan::kStates;
  const int ndir = states && adjoints ? 2 : 1;
  // With few (b, h) units the chunks of each are split into segments scanned in parallel
  // and joined afterwards (k_scan_seg.cu).
  const int cap = gla_seg_cap(a.BH, nc);
  int nseg = a.seg ? gla_scan_segments(a.BH, nc, ndir) : 1;
  int cps = nc;
  if (nseg > 1) {
    cps = (nc + nseg - 1) / nseg;
    nseg = (nc + cps - 1) / cps;  // no empty segment
  }
  float* segf0 = nseg > 1 ? a.seg : nullptr;
  float* segf1 = nseg > 1 ? a.seg + (size_t)2 * a.BH * cap * kD * kD : nullptr;
  // 32 value columns per CTA (measured against 64: 26.5 -> 36 us per CTA on B=1, H=32,
  // L=4096, with the MMA phase and the eight scan warps' epilogues both slower); five
  // chunks in flight when the grid fits one wave, else two so that two CTAs share an SM
  trace_begin(adjoints ? "bwd_scan_tc" : "fwd_scan_tc", s);
  cudaError_t e = a.BH * 4 * ndir * nseg <= ctas_per_wave(1)
                      ? scan_variant<5, 32>(a, states, adjoints, nc, nseg, cps, segf0, segf1, s)
                      : scan_variant<2, 32>(a, states, adjoints, nc, nseg, cps, segf0, segf1, s);
  trace_end(s);
  ++*launches;
  if (e != cudaSuccess || nseg == 1) return e;
  for (int dir = 0; dir < 2; ++dir) {
    if ((dir == 0 && !states) || (dir == 1 && !adjoints)) continue;
    e = launch_seg_join(a.BH, nc, nseg, cps, dir, a.gam, a.seg, cap, dir == 0 ? a.h0 : nullptr,
                        dir == 0 ? a.hf : a.dh0, s, launches);
    if (e == cudaSuccess)
      e = launch_seg_fix(a.BH, nc, nseg, cps, dir, a.gam, a.wide, a.seg, cap,
                         dir == 0 ? a.hs : a.gs, dir == 0 && a.h0 != nullptr, s, launches);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace lz
