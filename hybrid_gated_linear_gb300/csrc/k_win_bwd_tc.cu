// k_win_bwd_tc.cu -- backward of the anchor-window branch on tcgen05 tensor cores
// (bf16, d = 128, W <= 65, M <= 16).
//
// Query i attends to the M meta keys and to keys j in [max(0, i-W+1), i] with
// p_ij = softmax_j(scale q_i . k_j) (papernotes.org note on Lizard, 关键设计: Anchor Window
// Attention); its output enters y with weight alpha, so dyw = alpha dy.  The pages give no
// backward; the textbook softmax adjoint is
//   dp_ij = dyw_i . v_j,  D_i = sum_j p_ij dp_ij,  ds_ij = p_ij (dp_ij - D_i)
//   dq_i = scale sum_j ds_ij k_j,  dk_j = scale sum_i ds_ij q_i,  dv_j = sum_i p_ij dyw_i
// and the meta keys/values collect the same sums over every query of the batch.
//
// Both kernels work on 128-token blocks; with W <= 65 a block of queries sees the keys
// of the 192-row band [i0 - 64, i0 + 128), and a block of keys is seen by the queries of
// the band [j0, j0 + 192).
//   query kernel, per (b, h, queries i0 .. i0+127):
//     Z  = Q [Km ; Kband]^T,  dP = dY [Vm ; Vband]^T       M=128 N=16+192 K=128
//     per row: lse, D and ds (bf16, written over the V band in shared memory)
//     dQ = ds [Km ; Kband]                                 M=128 N=128 K=16+192
//     dMk^T = Q^T ds_meta,  dMv^T = dY^T p_meta            M=128 N=16  K=128
//   key kernel, per (b, h, keys j0 .. j0+127):
//     S^T = K Qband^T,  dP^T = V dYband^T                  M=128 N=192 K=128
//     p, ds from S^T, dP^T and the query rows' lse and D
//     dV = p^T dYband,  dK = ds^T Qband                    M=128 N=128 K=192
//   meta kernel: ordered sum of the per-block meta partials over batch and blocks.
// Every wait is bounded as in the other tensor-core kernels.
#include "lizard_dev.cuh"
#include "lizard_internal.h"
#include "tc_pipe.cuh"

namespace lz {
namespace {

using namespace tc;

constexpr int kB = 128;   // block of queries / keys
constexpr int kD = 128;   // dk = dv
constexpr int kBand = 192;
constexpr int kMetaRows = 16;
constexpr float kLog2e = 1.4426950408889634f;
// warp 0 TMA, warp 1 MMA, then kParts warps per TMEM lane quadrant for the row work
constexpr int kParts = 4;
constexpr int kThreads = 64 + kParts * 128;

using Ctl = tc::Ctl<8>;

struct Params {
  int H, L, M, W, nq, nbh;
  int ahead;  // CTAs per wave: the tile whose inputs a CTA prefetches into L2
  float scale, alpha;
  float* lse2;      // [BH][L]  log2-domain log-sum-exp of each query row
  float* Dw;        // [BH][L]
  float* mpart;     // [BH][nq][M][256] meta partials (dk part, then dv part)
  const float* dvacc;  // [BH][L][128] GLA part of dv
  bf16 *dq, *dk, *dv;
  unsigned* status;
  unsigned* tiles;  // query kernel: [0] next block to hand out, [1] CTAs done (both 0
                    // between launches: the last CTA to finish sets them back)
};

// ------------------------------------------------------------------------------------
// query kernel
// ------------------------------------------------------------------------------------
struct QMaps {
  CUtensorMap q, dy, kb, vb, mk, mv;  // loads
  CUtensorMap dqo;                    // store
};

// The query kernel is persistent: one CTA per SM takes query blocks from a counter in
// global memory until none is left (so CTAs that start late, behind the GLA kernels on the
// other stream, simply take fewer).  The loads of the next block start as soon as the MMAs
// of the current one have read their operands, and its logits as soon as the rows have
// read dQ out of TMEM, so copy-in, tensor-core and row phases of consecutive blocks
// overlap; dq leaves through a staging tile of its own.  The TMA thread passes each block
// index (or -1 at the end) to the other roles through a two-slot ring in shared memory,
// published by the arrival on Q_LDK.
enum { Q_LDK = 0, Q_LDV, Q_ZF, Q_DPF, Q_DS, Q_OUT, Q_TMF, Q_DONE };
constexpr uint32_t QS_Q = 0, QS_DY = 32768, QS_KB = 65536, QS_VB = QS_KB + 49152,
                   QS_KM = QS_VB + 49152, QS_VM = QS_KM + 4096, QS_DSM = QS_VM + 4096,
                   QS_PM = QS_DSM + 4096, QS_DQS = QS_PM + 4096, QS_RED = QS_DQS + 32768,
                   QS_BARS = QS_RED + 3 * kParts * 128 * 4;
constexpr size_t kQSmem = QS_BARS + 1024 + 1024;
static_assert(kQSmem <= 232448, "query kernel shared memory");
static_assert(sizeof(Ctl) <= 512, "barrier block below the block-index ring");
// TMEM columns: Z 0..207, dP 208..415, dMk 416, dMv 432; dQ reuses 0..127.
constexpr uint32_t TQ_Z = 0, TQ_DP = 208, TQ_MK = 416, TQ_MV = 432, TQ_DQ = 0;

__global__ void __launch_bounds__(kThreads, 1)
win_q_kernel(const __grid_constant__ QMaps maps, const Params p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(sm + QS_BARS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = p.L, M = p.M, W = p.W;
  const int ntiles = p.nbh * p.nq;
  volatile int* tslot = reinterpret_cast<volatile int*>(sm + QS_BARS + 512);

  if (threadIdx.x == 0) {
    for (int i = 0; i <= Q_DONE; ++i)
      mbar_init(&ctl->bar[i], (i == Q_DS || i == Q_TMF) ? kParts * 128u : 1u);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t meta_bytes = M > 0 ? 2u * kMetaRows * 128u : 0u;
      uint32_t nk = 0, nv = 0;  // phases armed on Q_LDK and Q_LDV
      int t = (int)atomicAdd(p.tiles, 1u);
      while (true) {
        // the previous block's MMAs have read Q, dY, the bands and the ds tiles
        if (nk > 0 && !wait_bar(ctl, Q_OUT, (nk - 1) & 1)) break;
        tslot[nk & 1] = t < ntiles ? t : -1;
        if (t >= ntiles) {
          mbar_arrive(&ctl->bar[Q_LDK]);  // no copy: publishes the end mark
          ++nk;
          break;
        }
        const int bh = t / p.nq, i0 = (t % p.nq) * kB, hh = bh % p.H;
        mbar_arrive_expect_tx(&ctl->bar[Q_LDK], 32768 + 49152 + meta_bytes);
        tma_load_3d(sm + QS_Q, &maps.q, 0, i0, bh, &ctl->bar[Q_LDK]);
        tma_load_3d(sm + QS_Q + 16384, &maps.q, 64, i0, bh, &ctl->bar[Q_LDK]);
        tma_load_3d(sm + QS_KB, &maps.kb, 0, i0 - 64, bh, &ctl->bar[Q_LDK]);
        tma_load_3d(sm + QS_KB + 24576, &maps.kb, 64, i0 - 64, bh, &ctl->bar[Q_LDK]);
        if (M > 0) {
          tma_load_3d(sm + QS_KM, &maps.mk, 0, 0, hh, &ctl->bar[Q_LDK]);
          tma_load_3d(sm + QS_KM + 2048, &maps.mk, 64, 0, hh, &ctl->bar[Q_LDK]);
        }
        ++nk;
        mbar_arrive_expect_tx(&ctl->bar[Q_LDV], 32768 + 49152 + meta_bytes);
        tma_load_3d(sm + QS_DY, &maps.dy, 0, i0, bh, &ctl->bar[Q_LDV]);
        tma_load_3d(sm + QS_DY + 16384, &maps.dy, 64, i0, bh, &ctl->bar[Q_LDV]);
        tma_load_3d(sm + QS_VB, &maps.vb, 0, i0 - 64, bh, &ctl->bar[Q_LDV]);
        tma_load_3d(sm + QS_VB + 24576, &maps.vb, 64, i0 - 64, bh, &ctl->bar[Q_LDV]);
        if (M > 0) {
          tma_load_3d(sm + QS_VM, &maps.mv, 0, 0, hh, &ctl->bar[Q_LDV]);
          tma_load_3d(sm + QS_VM + 2048, &maps.mv, 64, 0, hh, &ctl->bar[Q_LDV]);
        }
        ++nv;
        // take the next block now and warm L2 with its inputs
        t = (int)atomicAdd(p.tiles, 1u);
        if (t < ntiles && wait_bar(ctl, Q_LDV, (nv - 1) & 1)) {
          const int nbh = t / p.nq, ni0 = (t % p.nq) * kB;
          for (int x = 0; x < kD; x += 64) {
            tma_prefetch_l2_3d(&maps.q, x, ni0, nbh);
            tma_prefetch_l2_3d(&maps.kb, x, ni0 - 64, nbh);
            tma_prefetch_l2_3d(&maps.dy, x, ni0, nbh);
            tma_prefetch_l2_3d(&maps.vb, x, ni0 - 64, nbh);
          }
        }
      }
      const uint64_t tw = globaltimer_ns();
      drain_bar(ctl, Q_LDK, nk, tw);
      drain_bar(ctl, Q_LDV, nv, tw);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t sb = smem_u32(sm);
      const uint32_t id16 = idesc_bf16(kB, kMetaRows, false, false);
      const uint32_t id192 = idesc_bf16(kB, kBand, false, false);
      const uint32_t id_dq = idesc_bf16(kB, kD, false, true);
      const uint32_t id_dqm = idesc_bf16(kB, kD, true, true);
      const uint32_t id_meta = idesc_bf16(kD, kMetaRows, true, false);
      bool ok = true;
      for (uint32_t k = 0;; ++k) {
        if (!(ok = wait_bar(ctl, Q_LDK, k & 1))) break;
        if (tslot[k & 1] < 0) break;
        // Z overwrites the columns of the previous block's dQ: wait until the rows have
        // read it
        if (k > 0 && !(ok = wait_bar(ctl, Q_TMF, (k - 1) & 1))) break;
        tc_fence_after();
        if (M > 0)
          for (int j = 0; j < 8; ++j)
            mma_bf16(tmem + TQ_Z, desc_k(sb + QS_Q, kB, j), desc_k(sb + QS_KM, kMetaRows, j), id16, j > 0);
        for (int j = 0; j < 8; ++j)
          mma_bf16(tmem + TQ_Z + 16, desc_k(sb + QS_Q, kB, j), desc_k(sb + QS_KB, kBand, j), id192, j > 0);
        mma_commit(&ctl->bar[Q_ZF]);
        if (!(ok = wait_bar(ctl, Q_LDV, k & 1))) break;
        tc_fence_after();
        if (M > 0)
          for (int j = 0; j < 8; ++j)
            mma_bf16(tmem + TQ_DP, desc_k(sb + QS_DY, kB, j), desc_k(sb + QS_VM, kMetaRows, j), id16, j > 0);
        for (int j = 0; j < 8; ++j)
          mma_bf16(tmem + TQ_DP + 16, desc_k(sb + QS_DY, kB, j), desc_k(sb + QS_VB, kBand, j), id192, j > 0);
        mma_commit(&ctl->bar[Q_DPF]);
        if (!(ok = wait_bar(ctl, Q_DS, k & 1))) break;
        tc_fence_after();
        // dQ = ds_band Kband (+ ds_meta Km); ds_band lives over the V band
        for (int j = 0; j < kBand / 16; ++j)
          mma_bf16(tmem + TQ_DQ, desc_k(sb + QS_VB, kB, j), desc_mn(sb + QS_KB, kBand, j), id_dq, j > 0);
        if (M > 0) {
          mma_bf16(tmem + TQ_DQ, smem_desc(sb + QS_DSM, kMetaRows * 128u, 1024, kSw128),
                   smem_desc(sb + QS_KM, kMetaRows * 128u, 1024, kSw128), id_dqm, true);
          for (int j = 0; j < 8; ++j)
            mma_bf16(tmem + TQ_MK, desc_mn(sb + QS_Q, kB, j), desc_k(sb + QS_DSM, kMetaRows, j), id_meta, j > 0);
          for (int j = 0; j < 8; ++j)
            mma_bf16(tmem + TQ_MV, desc_mn(sb + QS_DY, kB, j), desc_k(sb + QS_PM, kMetaRows, j), id_meta, j > 0);
        }
        mma_commit(&ctl->bar[Q_OUT]);
      }
      if (!ok) ctl->abort = 1;
      mma_commit(&ctl->bar[Q_DONE]);
      drain_bar(ctl, Q_DONE, 1, globaltimer_ns());
    }
  } else {
    // kParts warps share each 32-lane TMEM quadrant: warp 2 + 4u + q reads lanes 32q..32q+31
    // (q = warp mod 4) and takes the column groups g = u, u + kParts, ... of those rows.
    const int qw = warp & 3;
    const int part = (warp - 2) >> 2;
    const int r = qw * 32 + lane;  // query row of the block
    const uint32_t tl = tmem + ((uint32_t)(qw * 32) << 16);
    const float zs = p.scale * kLog2e;
    const int nmeta = M > 0 ? 1 : 0;
    // 16-column band groups any row of this quadrant can see (keys i0 - 64 + b)
    const int g_lo = max(0, 64 + 32 * qw - W + 1) >> 4;
    const int g_hi = (64 + 32 * qw + 31) >> 4;
    const int nband = g_hi - g_lo + 1;  // at most 6 when W <= 65
    // Group slots: band groups 0 .. nband-1, the meta group in slot 7, so that the warps
    // taking slots 3 and 7 (and not those taking 0 and 4) do the meta stores.  Warp `part`
    // takes the slots part and part + kParts.
    constexpr int kMine = 8 / kParts;
    auto slot_used = [&](int s) { return s < nband || (s == 7 && nmeta); };
    auto zcol = [&](int s) { return s == 7 ? 0 : 16 + 16 * (g_lo + s); };
    float* red = reinterpret_cast<float*>(sm + QS_RED);  // [3][kParts][128] partials
    unsigned char* dsb = sm + QS_VB;  // ds band tile, 128 rows x 192 columns
    bool ok = true;
#pragma unroll 1
    for (uint32_t k = 0;; ++k) {
      // every row thread takes the same decision (the named barriers below need all)
      const int t = (ok && (ok = wait_bar(ctl, Q_LDK, k & 1))) ? tslot[k & 1] : -1;
      if (named_sync_or(1, kParts * 128, t < 0)) break;
      const int qb = t % p.nq, bh = t / p.nq;
      const int i0 = qb * kB;
      const int i = i0 + r;
      const bool valid = i < L;
      // band columns b <-> key j = i0 - 64 + b; this row sees b in [blo, bhi]
      const int bhi = 64 + r;
      const int blo = max(64 + r - W + 1, 64 - i0);
      auto vmask = [&](int s) -> uint32_t {
        if (s == 7) return (1u << M) - 1u;  // M <= 16
        const int base = 16 * (g_lo + s);
        const int lo = max(blo - base, 0), hi = min(bhi - base, 15);
        return hi < lo ? 0u : ((0xffffu >> (15 - hi)) >> lo) << lo;
      };
      // the staging tile is free once the previous block's dq store has read it; the
      // named barriers below hold the other rows until then
      if (threadIdx.x == 64) bulk_wait_read();
      uint32_t z[kMine][16], d[kMine][16];
      float mloc = -INFINITY;
      if (ok && (ok = wait_bar(ctl, Q_ZF, k & 1))) {
        tc_fence_after();
#pragma unroll
        for (int u = 0; u < kMine; ++u)
          if (slot_used(part + u * kParts)) tmem_ld16(tl + TQ_Z + zcol(part + u * kParts), z[u]);
        tmem_ld_wait();
        // logits this row does not see become -inf: the maximum needs no test, and
        // 2^-inf = 0 stands for them in the sums below
#pragma unroll
        for (int u = 0; u < kMine; ++u)
          if (slot_used(part + u * kParts)) {
            const uint32_t mk = vmask(part + u * kParts);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              if (!(mk & (1u << e))) z[u][e] = 0xff800000u;
              mloc = fmaxf(mloc, __uint_as_float(z[u][e]));
            }
          }
      }
      red[part * 128 + r] = mloc;
      named_sync(1, kParts * 128);
      float mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < kParts; ++u) mx = fmaxf(mx, red[u * 128 + r]);
      const float mxs = mx * zs;
      // exponentials once: z[u][e] becomes 2^(z scale log2e - max)
      float sum = 0.f, sdp = 0.f;
      if (ok && (ok = wait_bar(ctl, Q_DPF, k & 1))) {
        tc_fence_after();
#pragma unroll
        for (int u = 0; u < kMine; ++u)
          if (slot_used(part + u * kParts)) tmem_ld16(tl + TQ_DP + zcol(part + u * kParts), d[u]);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < kMine; ++u)
          if (slot_used(part + u * kParts)) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float ex = ex2_approx(fmaf(__uint_as_float(z[u][e]), zs, -mxs));
              z[u][e] = __float_as_uint(ex);
              sum += ex;
              sdp = fmaf(ex, __uint_as_float(d[u][e]), sdp);
            }
          }
      }
      red[(kParts + part) * 128 + r] = sum;
      red[(2 * kParts + part) * 128 + r] = sdp;
      named_sync(1, kParts * 128);
      sum = 0.f;
      sdp = 0.f;
#pragma unroll
      for (int u = 0; u < kParts; ++u) {
        sum += red[(kParts + u) * 128 + r];
        sdp += red[(2 * kParts + u) * 128 + r];
      }
      const float lse2 = mxs + __log2f(sum);
      const float Dv = p.alpha * sdp / sum;
      const float pscale = valid ? 1.f / sum : 0.f;
      if (ok) {
#pragma unroll
        for (int u = 0; u < kMine; ++u) {
          const int s = part + u * kParts;
          if (s == 7) {
            // transposed meta tiles: row m, column r
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float pe = __uint_as_float(z[u][e]) * pscale;
              const float de = pe * fmaf(p.alpha, __uint_as_float(d[u][e]), -Dv);
              *reinterpret_cast<bf16*>(sm + QS_DSM + sw128_offset(e, r, kMetaRows)) = __float2bfloat16_rn(de);
              *reinterpret_cast<bf16*>(sm + QS_PM + sw128_offset(e, r, kMetaRows)) = __float2bfloat16_rn(pe);
            }
          } else if (slot_used(s)) {
            // ds in two 8-column halves (one 16-byte store each)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int e0 = 8 * hf + 2 * e;
                const float p0 = __uint_as_float(z[u][e0]) * pscale;
                const float p1 = __uint_as_float(z[u][e0 + 1]) * pscale;
                w[e] = pack_bf16x2(p0 * fmaf(p.alpha, __uint_as_float(d[u][e0]), -Dv),
                                   p1 * fmaf(p.alpha, __uint_as_float(d[u][e0 + 1]), -Dv));
              }
              *reinterpret_cast<uint4*>(dsb + sw128_offset(r, 16 * (g_lo + s) + 8 * hf, kB)) =
                  make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
      // band groups no row of this quadrant sees hold zeros (the tile still holds V)
      for (int g = part; g < kBand / 16; g += kParts)
        if (g < g_lo || g > g_hi) zero16_bf16(dsb, kB, r, 16 * g);
      if (M == 0 && part == kParts - 1) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          *reinterpret_cast<bf16*>(sm + QS_DSM + sw128_offset(e, r, kMetaRows)) = __float2bfloat16_rn(0.f);
          *reinterpret_cast<bf16*>(sm + QS_PM + sw128_offset(e, r, kMetaRows)) = __float2bfloat16_rn(0.f);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(&ctl->bar[Q_DS]);
      if (ok && valid && part == 0) {
        p.lse2[(size_t)bh * L + i] = lse2;
        p.Dw[(size_t)bh * L + i] = Dv;
      }
      // dQ out of TMEM into the staging tile: this warp takes the 16-column slices
      // c = 16 part, 16 (part + kParts), ...; the last warp of the quadrant also the meta
      // products.  Then the next block's Z may overwrite these columns.
      const bool meta_here = M > 0 && part == kParts - 1;
      if (ok && (ok = wait_bar(ctl, Q_OUT, k & 1))) {
        tc_fence_after();
#pragma unroll 1
        for (int c = 16 * part; c < kD; c += 16 * kParts) {
          uint32_t v[16];
          tmem_ld16(tl + TQ_DQ + c, v);
          tmem_ld_wait();
          float w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = p.scale * __uint_as_float(v[e]);
          store16_bf16(sm + QS_DQS, kB, r, c, w);
        }
        fence_proxy_async_smem();
        if (meta_here) {
          // lane r of the meta products = feature dimension r
          float* mp = p.mpart + ((size_t)bh * p.nq + qb) * M * 256 + r;
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            uint32_t mk[16];
            tmem_ld16(tl + (h ? TQ_MV : TQ_MK), mk);
            tmem_ld_wait();
#pragma unroll
            for (int m = 0; m < kMetaRows; ++m)
              if (m < M) mp[m * 256 + 128 * h] = __uint_as_float(mk[m]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&ctl->bar[Q_TMF]);
      named_sync(1, kParts * 128);
      if (ok && threadIdx.x == 64) {
        // rows at or beyond L are clipped by the store
        tma_store_3d(&maps.dqo, sm + QS_DQS, 0, i0, bh);
        tma_store_3d(&maps.dqo, sm + QS_DQS + 16384, 64, i0, bh);
        bulk_commit();
      }
    }
    if (threadIdx.x == 64) bulk_wait_read();
    if (!ok) ctl->abort = 1;
  }

  pdl_trigger();
  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0) {
    if (ctl->abort) raise_status(p.status, kDevTimeout);
    // every CTA has taken its last block index once all have come here
    if (atomicAdd(p.tiles + 1, 1u) == gridDim.x - 1) {
      p.tiles[0] = 0;
      p.tiles[1] = 0;
    }
  }
}

// ------------------------------------------------------------------------------------
// key kernel
// ------------------------------------------------------------------------------------
struct KMaps {
  CUtensorMap k, v, qb, dyb, dva;  // loads (dva: the GLA part of dv, fp32)
  CUtensorMap dvo, dko;            // stores
};

enum { K_LDK = 0, K_LDV, K_SF, K_PDS, K_OUT, K_DVA, K_DONE };
// after the MMAs: dv and dk staged over K and V, the GLA part of dv (fp32) over the bands
constexpr uint32_t KS_DVS = 0, KS_DKS = 32768, KS_DVA = 65536;
constexpr uint32_t KS_K = 0, KS_V = 32768, KS_PT = 0 /* over K and V */, KS_QB = 65536,
                   KS_DYB = KS_QB + 49152, KS_DST = KS_DYB + 49152, KS_ROW = KS_DST + 49152,
                   KS_BARS = KS_ROW + 2048;
constexpr size_t kKSmem = KS_BARS + 1024 + 1024;
constexpr uint32_t TK_S = 0, TK_DP = 192, TK_DV = 0, TK_DK = 192;

__global__ void __launch_bounds__(kThreads, 1)
win_k_kernel(const __grid_constant__ KMaps maps, const Params p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(sm + KS_BARS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb = blockIdx.x % p.nq, bh = blockIdx.x / p.nq;
  const int L = p.L, W = p.W;
  const int j0 = kb * kB;
  float* rl = reinterpret_cast<float*>(sm + KS_ROW);  // lse2 of the band's query rows
  float* rd = rl + kBand;                             // D of the band's query rows

  if (threadIdx.x == 0) {
    for (int i = 0; i <= K_DONE; ++i) mbar_init(&ctl->bar[i], i == K_PDS ? kParts * 128u : 1u);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&ctl->bar[K_LDK], 32768 + 49152);
      tma_load_3d(sm + KS_K, &maps.k, 0, j0, bh, &ctl->bar[K_LDK]);
      tma_load_3d(sm + KS_K + 16384, &maps.k, 64, j0, bh, &ctl->bar[K_LDK]);
      tma_load_3d(sm + KS_QB, &maps.qb, 0, j0, bh, &ctl->bar[K_LDK]);
      tma_load_3d(sm + KS_QB + 24576, &maps.qb, 64, j0, bh, &ctl->bar[K_LDK]);
      mbar_arrive_expect_tx(&ctl->bar[K_LDV], 32768 + 49152);
      tma_load_3d(sm + KS_V, &maps.v, 0, j0, bh, &ctl->bar[K_LDV]);
      tma_load_3d(sm + KS_V + 16384, &maps.v, 64, j0, bh, &ctl->bar[K_LDV]);
      tma_load_3d(sm + KS_DYB, &maps.dyb, 0, j0, bh, &ctl->bar[K_LDV]);
      tma_load_3d(sm + KS_DYB + 24576, &maps.dyb, 64, j0, bh, &ctl->bar[K_LDV]);
      for (int x = 0; x < kD; x += 32) tma_prefetch_l2_3d(&maps.dva, x, j0, bh);
      // warm L2 with the inputs of the tile one wave later
      const int nb = blockIdx.x + p.ahead;
      if (nb < gridDim.x && wait_bar(ctl, K_LDV, 0)) {
        const int nbh = nb / p.nq, nj0 = (nb % p.nq) * kB;
        for (int x = 0; x < kD; x += 64) {
          tma_prefetch_l2_3d(&maps.k, x, nj0, nbh);
          tma_prefetch_l2_3d(&maps.qb, x, nj0, nbh);
          tma_prefetch_l2_3d(&maps.v, x, nj0, nbh);
          tma_prefetch_l2_3d(&maps.dyb, x, nj0, nbh);
        }
      }
      // the GLA part of dv, once the shared memory of the band tiles is free
      uint32_t armed = 0;
      if (wait_bar(ctl, K_OUT, 0)) {
        mbar_arrive_expect_tx(&ctl->bar[K_DVA], kB * kD * 4);
        for (int x = 0; x < kD; x += 32)
          tma_load_3d(sm + KS_DVA + x * 512, &maps.dva, x, j0, bh, &ctl->bar[K_DVA]);
        armed = 1;
      }
      const uint64_t tw = globaltimer_ns();
      drain_bar(ctl, K_LDK, 1, tw);
      drain_bar(ctl, K_LDV, 1, tw);
      drain_bar(ctl, K_DVA, armed, tw);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t sb = smem_u32(sm);
      const uint32_t id_s = idesc_bf16(kB, kBand, false, false);
      const uint32_t id_o = idesc_bf16(kB, kD, false, true);
      bool ok = wait_bar(ctl, K_LDK, 0);
      if (ok) {
        tc_fence_after();
        for (int j = 0; j < 8; ++j)
          mma_bf16(tmem + TK_S, desc_k(sb + KS_K, kB, j), desc_k(sb + KS_QB, kBand, j), id_s, j > 0);
      }
      if (ok && (ok = wait_bar(ctl, K_LDV, 0))) {
        tc_fence_after();
        for (int j = 0; j < 8; ++j)
          mma_bf16(tmem + TK_DP, desc_k(sb + KS_V, kB, j), desc_k(sb + KS_DYB, kBand, j), id_s, j > 0);
        mma_commit(&ctl->bar[K_SF]);
      }
      if (ok && (ok = wait_bar(ctl, K_PDS, 0))) {
        tc_fence_after();
        for (int j = 0; j < kBand / 16; ++j)
          mma_bf16(tmem + TK_DV, desc_k(sb + KS_PT, kB, j), desc_mn(sb + KS_DYB, kBand, j), id_o, j > 0);
        for (int j = 0; j < kBand / 16; ++j)
          mma_bf16(tmem + TK_DK, desc_k(sb + KS_DST, kB, j), desc_mn(sb + KS_QB, kBand, j), id_o, j > 0);
        mma_commit(&ctl->bar[K_OUT]);
      }
      if (!ok) ctl->abort = 1;
      mma_commit(&ctl->bar[K_DONE]);
      drain_bar(ctl, K_DONE, 1, globaltimer_ns());
    }
  } else {
    // kParts warps share each 32-lane TMEM quadrant (as in the query kernel)
    const int qw = warp & 3;
    const int part = (warp - 2) >> 2;
    const int jr = qw * 32 + lane;  // key row of the block
    const int j = j0 + jr;
    const bool valid = j < L;
    const uint32_t tl = tmem + ((uint32_t)(qw * 32) << 16);
    const float zs = p.scale * kLog2e;
    for (int u = threadIdx.x - 64; u < kBand; u += kParts * 128) {
      const int i = j0 + u;
      rl[u] = i < L ? p.lse2[(size_t)bh * L + i] : INFINITY;
      rd[u] = i < L ? p.Dw[(size_t)bh * L + i] : 0.f;
    }
    named_sync(1, kParts * 128);
    // query column u <-> query i = j0 + u; this row is seen by u in [jr, jr + W - 1]
    const int g_lo = (32 * qw) >> 4;
    const int g_hi = min(kBand - 1, 32 * qw + 31 + W - 1) >> 4;
    unsigned char* pt = sm + KS_PT;
    unsigned char* dst = sm + KS_DST;
    bool ok = wait_bar(ctl, K_SF, 0);
    if (ok) {
      tc_fence_after();
      // at most six 16-column groups (W <= 65); this warp takes groups g_lo + part,
      // g_lo + part + kParts, ... and reads them from TMEM with one wait
      constexpr int kMine = (6 + kParts - 1) / kParts;
      const int ng = g_hi - g_lo + 1;
      uint32_t sv[kMine][16], dv[kMine][16];
#pragma unroll
      for (int u = 0; u < kMine; ++u)
        if (part + u * kParts < ng) {
          tmem_ld16(tl + TK_S + 16 * (g_lo + part + u * kParts), sv[u]);
          tmem_ld16(tl + TK_DP + 16 * (g_lo + part + u * kParts), dv[u]);
        }
      tmem_ld_wait();
#pragma unroll
      for (int u = 0; u < kMine; ++u) {
        if (part + u * kParts < ng) {
          const int g = g_lo + part + u * kParts;
          // columns of the group that see this key: bits lo .. hi
          const int lo = max(jr - 16 * g, 0), hi = min(jr + W - 1 - 16 * g, 15);
          const uint32_t mk = (!valid || hi < lo) ? 0u : ((0xffffu >> (15 - hi)) >> lo) << lo;
          float rlv[16], rdv[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 a4 = reinterpret_cast<const float4*>(rl + 16 * g)[q];
            const float4 b4 = reinterpret_cast<const float4*>(rd + 16 * g)[q];
            rlv[4 * q] = a4.x; rlv[4 * q + 1] = a4.y; rlv[4 * q + 2] = a4.z; rlv[4 * q + 3] = a4.w;
            rdv[4 * q] = b4.x; rdv[4 * q + 1] = b4.y; rdv[4 * q + 2] = b4.z; rdv[4 * q + 3] = b4.w;
          }
          float pp[16], ds[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float pe = (mk & (1u << e)) ? ex2_approx(fmaf(__uint_as_float(sv[u][e]), zs, -rlv[e])) : 0.f;
            pp[e] = pe;
            ds[e] = pe * fmaf(p.alpha, __uint_as_float(dv[u][e]), -rdv[e]);
          }
          store16_bf16(pt, kB, jr, 16 * g, pp);
          store16_bf16(dst, kB, jr, 16 * g, ds);
        }
      }
    }
    for (int g = part; g < kBand / 16; g += kParts) {
      if (g < g_lo || g > g_hi) {
        zero16_bf16(pt, kB, jr, 16 * g);
        zero16_bf16(dst, kB, jr, 16 * g);
      }
    }
    tc_fence_before();
    fence_proxy_async_smem();
    mbar_arrive(&ctl->bar[K_PDS]);
    const bool ready = ok && (ok = wait_bar(ctl, K_OUT, 0)) && (ok = wait_bar(ctl, K_DVA, 0));
    if (ready) {
      tc_fence_after();
      // this warp takes the 32-column slices c = 32 part, 32 (part + kParts), ...
#pragma unroll 1
      for (int c = 32 * part; c < kD; c += 32 * kParts) {
        uint32_t v[32], k[32];
        tmem_ld32(tl + TK_DV + c, v);
        tmem_ld32(tl + TK_DK + c, k);
        tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float wv[16], wk[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 g = *reinterpret_cast<const float4*>(
                sm + KS_DVA + sw128_offset_f32(jr, c + 16 * h + 4 * q, kB));
            const float ga[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int k0 = 16 * h + 4 * q + e;
              wv[4 * q + e] = fmaf(p.alpha, __uint_as_float(v[k0]), ga[e]);
              wk[4 * q + e] = p.scale * __uint_as_float(k[k0]);
            }
          }
          store16_bf16(sm + KS_DVS, kB, jr, c + 16 * h, wv);
          store16_bf16(sm + KS_DKS, kB, jr, c + 16 * h, wk);
        }
      }
      fence_proxy_async_smem();
    }
    named_sync(1, kParts * 128);
    if (ready && threadIdx.x == 64) {
      // rows at or beyond L are clipped by the stores
      tma_store_3d(&maps.dvo, sm + KS_DVS, 0, j0, bh);
      tma_store_3d(&maps.dvo, sm + KS_DVS + 16384, 64, j0, bh);
      tma_store_3d(&maps.dko, sm + KS_DKS, 0, j0, bh);
      tma_store_3d(&maps.dko, sm + KS_DKS + 16384, 64, j0, bh);
      bulk_commit();
      bulk_wait_read();
    }
    if (!ok) ctl->abort = 1;
  }

  pdl_trigger();
  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && ctl->abort) raise_status(p.status, kDevTimeout);
}

// ------------------------------------------------------------------------------------
// meta gradients: ordered sum of the per-block partials over (batch, block).
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) win_meta_kernel(int B, int H, int M, int nq, float scale,
                                                       float alpha, const float* mpart, float* dmk,
                                                       float* dmv) {
  const int hh = blockIdx.x, m = blockIdx.y, d = threadIdx.x;
  pdl_wait();
  float s = 0.f;
  for (int b = 0; b < B; ++b) {
    const float* part = mpart + ((size_t)(b * H + hh) * nq) * M * 256 + m * 256 + d;
    // eight loads in flight, added in block order
    int q = 0;
    for (; q + 8 <= nq; q += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = part[(size_t)(q + u) * M * 256];
#pragma unroll
      for (int u = 0; u < 8; ++u) s += v[u];
    }
    for (; q < nq; ++q) s += part[(size_t)q * M * 256];
  }
  if (d < kD) dmk[((size_t)hh * M + m) * kD + d] = scale * s;
  else dmv[((size_t)hh * M + m) * kD + d - kD] = alpha * s;
}

template <typename K, typename Mp>
cudaError_t launch_tc(K kernel, const Mp& maps, const Params& p, int grid, size_t smem,
                      const char* name, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  trace_begin(name, s);
  e = launch_pdl(kernel, dim3(grid), dim3(kThreads), smem, s, maps, p);
  trace_end(s);
  return e;
}

}  // namespace

bool bwd_win_tc_supported(int dk, int dv, int L, int W, int M, lizard_dtype dt) {
  return dt == LIZARD_BF16 && dk == kD && dv == kD && L > 0 && W >= 1 && W <= 65 &&
         M <= kMetaRows && tma_encode_available();
}

size_t bwd_win_tc_meta_floats(int BH, int L, int M) {
  return (size_t)BH * ((L + kB - 1) / kB) * M * 256;
}

// Both halves build the same maps and parameters; `part` selects the query kernel (0) or
// the key kernel (1).
static cudaError_t launch_win_part(int part, const BwdArgs& a, const float* dvacc, float* lse2,
                                   float* Dw, float* mpart, cudaStream_t s, int* launches) {
  const int BH = a.B * a.H, L = a.L;
  const int nq = (L + kB - 1) / kB;
  const uint64_t bhl = (uint64_t)BH, Ll = (uint64_t)L;
  QMaps qm;
  KMaps km;
  bool ok = make_tma_map_bf16(&qm.q, a.q, kD, Ll, bhl, 64, kB, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&qm.dy, a.dy, kD, Ll, bhl, 64, kB, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&qm.kb, a.k, kD, Ll, bhl, 64, kBand, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&qm.vb, a.v, kD, Ll, bhl, 64, kBand, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&km.k, a.k, kD, Ll, bhl, 64, kB, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&km.v, a.v, kD, Ll, bhl, 64, kB, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&km.qb, a.q, kD, Ll, bhl, 64, kBand, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&km.dyb, a.dy, kD, Ll, bhl, 64, kBand, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_f32(&km.dva, dvacc, kD, Ll, bhl, 32, kB, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&km.dvo, a.dvv, kD, Ll, bhl, 64, kB, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&km.dko, a.dk_, kD, Ll, bhl, 64, kB, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&qm.dqo, a.dq, kD, Ll, bhl, 64, kB, CU_TENSOR_MAP_SWIZZLE_128B);
  if (a.M > 0) {
    ok = ok && make_tma_map_bf16(&qm.mk, a.mk, kD, a.M, a.H, 64, kMetaRows, CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_tma_map_bf16(&qm.mv, a.mv, kD, a.M, a.H, 64, kMetaRows, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    qm.mk = qm.q;
    qm.mv = qm.dy;
  }
  if (!ok) return cudaErrorInvalidValue;
  Params p;
  p.H = a.H;
  p.L = L;
  p.M = a.M;
  p.W = a.W;
  p.nq = nq;
  p.nbh = BH;
  p.ahead = ctas_per_wave(1);
  p.tiles = a.status + kWsWinTiles;
  p.scale = a.scale;
  p.alpha = a.alpha;
  p.lse2 = lse2;
  p.Dw = Dw;
  p.mpart = mpart;
  p.dvacc = dvacc;
  p.dq = static_cast<bf16*>(a.dq);
  p.dk = static_cast<bf16*>(a.dk_);
  p.dv = static_cast<bf16*>(a.dvv);
  p.status = a.status;
  const int grid = BH * nq;
  cudaError_t e = part == 1 ? launch_tc(win_k_kernel, km, p, grid, kKSmem, "win_bwd_k_tc", s)
                            : launch_tc(win_q_kernel, qm, p, std::min(grid, ctas_per_wave(1)), kQSmem,
                                        "win_bwd_q_tc", s);
  ++*launches;
  return e;
}

cudaError_t launch_bwd_win_q_tc(const BwdArgs& a, const float* dvacc, float* lse2, float* Dw,
                                float* mpart, cudaStream_t s, int* launches) {
  return launch_win_part(0, a, dvacc, lse2, Dw, mpart, s, launches);
}

cudaError_t launch_bwd_win_k_tc(const BwdArgs& a, const float* dvacc, float* lse2, float* Dw,
                                float* mpart, cudaStream_t s, int* launches) {
  return launch_win_part(1, a, dvacc, lse2, Dw, mpart, s, launches);
}

cudaError_t launch_bwd_win_meta_tc(const BwdArgs& a, const float* mpart, cudaStream_t s,
                                   int* launches) {
  if (a.M == 0) return cudaSuccess;
  const int nq = (a.L + kB - 1) / kB;
  trace_begin("win_bwd_meta", s);
  cudaError_t e = launch_pdl(win_meta_kernel, dim3(a.H, a.M), dim3(256), 0, s, a.B, a.H, a.M, nq,
                             a.scale, a.alpha, mpart, a.dmk, a.dmv);
  trace_end(s);
  ++*launches;
  if (e == cudaSuccess) e = cudaGetLastError();
  return e;
}

}  // namespace lz
