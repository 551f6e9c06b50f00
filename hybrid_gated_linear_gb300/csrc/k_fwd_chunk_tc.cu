// k_fwd_chunk_tc.cu -- chunk-parallel Lizard-attention forward on tcgen05 tensor cores
// (bf16, d = 128, W <= 129, M <= 16).
//
// After the prep and state-scan passes of k_gla_states_tc.cu (Qt = phi_q e^b,
// Kt = phi_k e^-b and the state h_c at every 128-token chunk start), every chunk is
// independent.  One CTA per (b, h, chunk c), tokens t0 .. t0+127:
//   GLA ("Lizard", arXiv 2507.09025, Method: parallel form with cumulative gate products)
//     S  = Qt Kt^T                      M=128 N=128 K=128
//     O  = Qt h_c + mask(S) V           M=128 N=128 K=128 + 128
//   anchor window (papernotes.org note on Lizard, 关键设计: Anchor Window Attention): the
//   queries of the chunk see the M meta keys and the band of keys [t0 - 64 NP, t0 + 128)
//     Z  = q [Km ; Kband]^T             M=128 N=16+128+64NP K=128
//     P  = exp(scale (Z - rowmax)) on the visible keys (bf16), l = row sums of P
//     Ow = P [Vm ; Vband]               M=128 N=128 K=16+128+64NP
//   y = O + alpha Ow / l, rounded to bf16 once and written by a TMA store.
// NP = 1 covers W <= 65 and NP = 2 W <= 129.  Warp 0 issues the TMA loads, warp 1 the
// MMAs (accumulators in TMEM), warps 2-5 (thread = query row) the causal mask, the
// softmax and the epilogue.  The V band is loaded into the GLA operands' shared memory
// once the GLA products are done; with NP = 2 the query tile goes where h_c was.  Every
// wait is bounded; on a timeout the CTA records LIZARD_ERR_TIMEOUT, drains its copies and
// MMAs, frees its tensor memory and returns.
#include "lizard_dev.cuh"
#include "lizard_internal.h"
#include "tc_pipe.cuh"

namespace lz {
namespace {

using namespace tc;

constexpr int kC = kGlaChunk;
constexpr int kD = 128;
constexpr int kMetaRows = 16;
constexpr int kThreads = 6 * 32;
constexpr float kLog2e = 1.4426950408889634f;

template <int NP>
struct FCfg {
  static constexpr int OFF = 64 * NP;          // look-back rows of the key band
  static constexpr int BR = kC + OFF;          // key band rows
  static constexpr bool QOWN = NP == 1;        // query tile in its own buffer
  // shared memory (bytes from a 1024-aligned base); region R holds the GLA operands,
  // then the V band, then the staged output tile
  static constexpr uint32_t QT = 0, KT = 32768, HS = 65536, VT = 98304;
  static constexpr uint32_t VB = 0, VM = VB + BR * 256u, YS = 0;
  static constexpr uint32_t Q = QOWN ? 131072u : HS;
  static constexpr uint32_t KB = QOWN ? 163840u : 131072u;
  static constexpr uint32_t KM = KB + BR * 256u;
  static constexpr uint32_t PMT = KM + 4096;
  static constexpr uint32_t BARS = PMT + 4096;
  static constexpr size_t TOTAL = BARS + 1024 + 1024;
  // TMEM columns: S, then Ow, at 0; Z at TZ (after S has been read when NP = 2); O at 384
  static constexpr uint32_t TS = 0, TOW = 0, TO = 384;
  static constexpr uint32_t TZ = NP == 1 ? 128u : 0u;
  static_assert(TZ + 16 + BR <= TO, "TMEM budget");
  static_assert(VM + 4096 <= 131072, "V band fits in region R");
};

struct FMaps {
  CUtensorMap qt, kt, hs, v, q, kb, mk, vb, mv, y;
};

struct FParams {
  int H, L, M, W, nc;
  int ahead;  // CTAs per wave: the tile whose inputs this CTA prefetches into L2
  float scale, alpha;
  unsigned* status;
};

enum { F_LDG = 0, F_LDW, F_LDQ2, F_LDV2, F_SF, F_ZF, F_SMR, F_GLA, F_PR, F_OWF, F_DONE, F_COUNT };

template <int NP>
__global__ void __launch_bounds__(kThreads, 1)
fwd_chunk_kernel(const __grid_constant__ FMaps maps, const FParams p) {
  using G = FCfg<NP>;
  constexpr int BR = G::BR, OFF = G::OFF;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  using C = Ctl<F_COUNT>;
  C* ctl = reinterpret_cast<C*>(sm + G::BARS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nc = p.nc, M = p.M, W = p.W;
  const int c = blockIdx.x % nc, bh = blockIdx.x / nc;
  const int hh = bh % p.H;
  const int t0 = c * kC;

  if (threadIdx.x == 0) {
    for (int i = 0; i < F_COUNT; ++i) mbar_init(&ctl->bar[i], (i == F_SMR || i == F_PR) ? 128u : 1u);
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
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t meta_bytes = M > 0 ? 2u * kMetaRows * 128u : 0u;
      const uint32_t band_bytes = (uint32_t)BR * 256u;
      uint32_t armed_q2 = 0, armed_v2 = 0;
      mbar_arrive_expect_tx(&ctl->bar[F_LDG], 4 * 32768);
      tma_load_3d(sm + G::QT, &maps.qt, 0, t0, bh, &ctl->bar[F_LDG]);
      tma_load_3d(sm + G::QT + 16384, &maps.qt, 64, t0, bh, &ctl->bar[F_LDG]);
      tma_load_3d(sm + G::KT, &maps.kt, 0, t0, bh, &ctl->bar[F_LDG]);
      tma_load_3d(sm + G::KT + 16384, &maps.kt, 64, t0, bh, &ctl->bar[F_LDG]);
      tma_load_3d(sm + G::HS, &maps.hs, 0, 0, bh * nc + c, &ctl->bar[F_LDG]);
      tma_load_3d(sm + G::HS + 16384, &maps.hs, 64, 0, bh * nc + c, &ctl->bar[F_LDG]);
      tma_load_3d(sm + G::VT, &maps.v, 0, t0, bh, &ctl->bar[F_LDG]);
      tma_load_3d(sm + G::VT + 16384, &maps.v, 64, t0, bh, &ctl->bar[F_LDG]);
      mbar_arrive_expect_tx(&ctl->bar[F_LDW], band_bytes + meta_bytes + (G::QOWN ? 32768u : 0u));
      if (G::QOWN) {
        tma_load_3d(sm + G::Q, &maps.q, 0, t0, bh, &ctl->bar[F_LDW]);
        tma_load_3d(sm + G::Q + 16384, &maps.q, 64, t0, bh, &ctl->bar[F_LDW]);
      }
      tma_load_3d(sm + G::KB, &maps.kb, 0, t0 - OFF, bh, &ctl->bar[F_LDW]);
      tma_load_3d(sm + G::KB + BR * 128, &maps.kb, 64, t0 - OFF, bh, &ctl->bar[F_LDW]);
      if (M > 0) {
        tma_load_3d(sm + G::KM, &maps.mk, 0, 0, hh, &ctl->bar[F_LDW]);
        tma_load_3d(sm + G::KM + 2048, &maps.mk, 64, 0, hh, &ctl->bar[F_LDW]);
      }
      // the V band is loaded only after the GLA products; bring it into L2 now
      tma_prefetch_l2_3d(&maps.vb, 0, t0 - OFF, bh);
      tma_prefetch_l2_3d(&maps.vb, 64, t0 - OFF, bh);
      bool ok = true;
      // warm L2 with the inputs of the tile one wave later once this tile's are in
      const int nb = blockIdx.x + p.ahead;
      if (nb < gridDim.x && (ok = wait_bar(ctl, F_LDW, 0))) {
        const int nbh = nb / nc, nt0 = (nb % nc) * kC;
        for (int x = 0; x < kD; x += 64) {
          tma_prefetch_l2_3d(&maps.qt, x, nt0, nbh);
          tma_prefetch_l2_3d(&maps.kt, x, nt0, nbh);
          tma_prefetch_l2_3d(&maps.hs, x, 0, nb);
          tma_prefetch_l2_3d(&maps.v, x, nt0, nbh);
          tma_prefetch_l2_3d(&maps.q, x, nt0, nbh);
          tma_prefetch_l2_3d(&maps.kb, x, nt0 - OFF, nbh);
        }
      }
      if (ok && !G::QOWN) {
        // the query tile goes where h_c was, once Qt h_c has been computed
        if ((ok = wait_bar(ctl, F_SF, 0))) {
          mbar_arrive_expect_tx(&ctl->bar[F_LDQ2], 32768);
          tma_load_3d(sm + G::Q, &maps.q, 0, t0, bh, &ctl->bar[F_LDQ2]);
          tma_load_3d(sm + G::Q + 16384, &maps.q, 64, t0, bh, &ctl->bar[F_LDQ2]);
          armed_q2 = 1;
        }
      }
      // the V band replaces the GLA operands once every GLA product (and Z) is done
      if (ok && (ok = wait_bar(ctl, F_GLA, 0))) {
        mbar_arrive_expect_tx(&ctl->bar[F_LDV2], band_bytes + meta_bytes);
        tma_load_3d(sm + G::VB, &maps.vb, 0, t0 - OFF, bh, &ctl->bar[F_LDV2]);
        tma_load_3d(sm + G::VB + BR * 128, &maps.vb, 64, t0 - OFF, bh, &ctl->bar[F_LDV2]);
        if (M > 0) {
          tma_load_3d(sm + G::VM, &maps.mv, 0, 0, hh, &ctl->bar[F_LDV2]);
          tma_load_3d(sm + G::VM + 2048, &maps.mv, 64, 0, hh, &ctl->bar[F_LDV2]);
        }
        armed_v2 = 1;
      }
      if (!ok) ctl->abort = 1;
      const uint64_t tw = globaltimer_ns();
      drain_bar(ctl, F_LDG, 1, tw);
      drain_bar(ctl, F_LDW, 1, tw);
      drain_bar(ctl, F_LDQ2, armed_q2, tw);
      drain_bar(ctl, F_LDV2, armed_v2, tw);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sb = smem_u32(sm);
      const uint32_t id_kk = idesc_bf16(kC, kD, false, false);
      const uint32_t id_kn = idesc_bf16(kC, kD, false, true);
      const uint32_t id_nn = idesc_bf16(kC, kD, true, true);
      const uint32_t id_z16 = idesc_bf16(kC, kMetaRows, false, false);
      const uint32_t id_zb = idesc_bf16(kC, BR, false, false);
      auto issue_z = [&]() {
        if (M > 0)
          for (int j = 0; j < 8; ++j)
            mma_bf16(tmem + G::TZ, desc_k(sb + G::Q, kC, j), desc_k(sb + G::KM, kMetaRows, j), id_z16, j > 0);
        for (int j = 0; j < 8; ++j)
          mma_bf16(tmem + G::TZ + 16, desc_k(sb + G::Q, kC, j), desc_k(sb + G::KB, BR, j), id_zb, j > 0);
        mma_commit(&ctl->bar[F_ZF]);
      };
      bool ok = wait_bar(ctl, F_LDG, 0);
      if (ok) {
        tc_fence_after();
        for (int j = 0; j < 8; ++j)  // S = Qt Kt^T
          mma_bf16(tmem + G::TS, desc_k(sb + G::QT, kC, j), desc_k(sb + G::KT, kC, j), id_kk, j > 0);
        for (int j = 0; j < 8; ++j)  // O = Qt h_c   (h_c rows = key dimension = K)
          mma_bf16(tmem + G::TO, desc_k(sb + G::QT, kC, j), desc_mn(sb + G::HS, kD, j), id_kn, j > 0);
        mma_commit(&ctl->bar[F_SF]);
      }
      if (G::QOWN) {
        if (ok && (ok = wait_bar(ctl, F_LDW, 0))) {
          tc_fence_after();
          issue_z();
        }
        if (ok && (ok = wait_bar(ctl, F_SMR, 0))) tc_fence_after();
      } else {
        // Z reuses the columns of S: wait for the causal-mask pass to have read them
        if (ok && (ok = wait_bar(ctl, F_SMR, 0)) && (ok = wait_bar(ctl, F_LDW, 0)) &&
            (ok = wait_bar(ctl, F_LDQ2, 0))) {
          tc_fence_after();
          issue_z();
        }
      }
      if (ok) {
        for (int j = 0; j < 8; ++j)  // O += mask(S) V   (mask(S) written over Kt)
          mma_bf16(tmem + G::TO, desc_k(sb + G::KT, kC, j), desc_mn(sb + G::VT, kC, j), id_kn, true);
        mma_commit(&ctl->bar[F_GLA]);
      }
      if (ok && (ok = wait_bar(ctl, F_PR, 0)) && (ok = wait_bar(ctl, F_LDV2, 0))) {
        tc_fence_after();
        for (int j = 0; j < BR / 16; ++j)  // Ow = P_band V_band   (P written over the key band)
          mma_bf16(tmem + G::TOW, desc_k(sb + G::KB, kC, j), desc_mn(sb + G::VB, BR, j), id_kn, j > 0);
        if (M > 0)  // Ow += P_meta V_meta   (P_meta stored transposed)
          mma_bf16(tmem + G::TOW, smem_desc(sb + G::PMT, kMetaRows * 128u, 1024, kSw128),
                   smem_desc(sb + G::VM, kMetaRows * 128u, 1024, kSw128), id_nn, true);
        mma_commit(&ctl->bar[F_OWF]);
      }
      if (!ok) ctl->abort = 1;
      mma_commit(&ctl->bar[F_DONE]);
      drain_bar(ctl, F_DONE, 1, globaltimer_ns());
    }
  } else {
    // ------------------------------------------------------------------ rows
    const int qw = warp & 3;
    const int r = qw * 32 + lane;  // query row of the chunk
    const uint32_t tl = tmem + ((uint32_t)(qw * 32) << 16);
    bool ok = true;

    // 1. causal mask of S -> bf16 operand over Kt
    if ((ok = wait_bar(ctl, F_SF, 0))) {
      tc_fence_after();
#pragma unroll 1
      for (int g2 = 0; g2 < 4; g2 += 2) {
        uint32_t sv[2][32];
        tmem_ld32(tl + G::TS + 32 * g2, sv[0]);
        tmem_ld32(tl + G::TS + 32 * g2 + 32, sv[1]);
        tmem_ld_wait();
#pragma unroll
        for (int gg = 0; gg < 2; ++gg) {
          float v[16];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int s = 32 * (g2 + gg) + 16 * h + e;
              v[e] = s <= r ? __uint_as_float(sv[gg][16 * h + e]) : 0.f;
            }
            store16_bf16(sm + G::KT, kC, r, 32 * (g2 + gg) + 16 * h, v);
          }
        }
      }
    }
    tc_fence_before();
    fence_proxy_async_smem();
    mbar_arrive(&ctl->bar[F_SMR]);

    // 2. window softmax -> bf16 P over the key band, P_meta transposed
    const float zs = p.scale * kLog2e;
    const int bhi = OFF + r;                       // band column of key i
    const int blo = max(OFF + r - W + 1, OFF - t0);  // first visible band column
    const int g_lo = max(0, OFF + 32 * qw - W + 1) >> 4;
    const int g_hi = (OFF + 32 * qw + 31) >> 4;
    const int nmeta = M > 0 ? 1 : 0;
    const int ng = nmeta + g_hi - g_lo + 1;
    auto zcol = [&](int g) { return g < nmeta ? 0 : 16 + 16 * (g_lo + g - nmeta); };
    // visible columns of group g as a 16-bit mask (bits lo .. hi of the group)
    auto vmask = [&](int g) -> uint32_t {
      if (g < nmeta) return (1u << M) - 1u;  // M <= 16
      const int base = 16 * (g_lo + g - nmeta);
      const int lo = max(blo - base, 0), hi = min(bhi - base, 15);
      return hi < lo ? 0u : ((0xffffu >> (15 - hi)) >> lo) << lo;
    };
    // The window's logits are read from TMEM in batches of GB 16-column groups per wait;
    // with one batch (NP = 1) the exponent pass reuses the registers of the max pass.
    constexpr int GB = NP == 1 ? 8 : 6;
    float sum = 1.f;
    bool zeroed = false;
    if (ok && (ok = wait_bar(ctl, F_ZF, 0))) {
      tc_fence_after();
      // one batch always when NP = 1 (ng <= 7): a constant, so that the loops fold
      const int nbatch = NP == 1 ? 1 : (ng + GB - 1) / GB;
      uint32_t z[GB][16];
      // logits this row does not see are set to -inf once, as they are loaded, so that the
      // max pass is a plain maximum and the exponent pass needs no test (2^-inf = 0)
      auto load_batch = [&](int b) {
#pragma unroll
        for (int k = 0; k < GB; ++k)
          if (b * GB + k < ng) tmem_ld16(tl + G::TZ + zcol(b * GB + k), z[k]);
        if (b == 0 && !zeroed) {
          // band groups no row of this warp sees hold zeros (the tile still holds keys);
          // written while the TMEM loads are in flight (Z, which read the keys, is done)
          for (int g = 0; g < BR / 16; ++g)
            if (g < g_lo || g > g_hi) zero16_bf16(sm + G::KB, kC, r, 16 * g);
          zeroed = true;
        }
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < GB; ++k)
          if (b * GB + k < ng) {
            const uint32_t mk = vmask(b * GB + k);
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (!(mk & (1u << e))) z[k][e] = 0xff800000u;
          }
      };
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      for (int b = 0; b < nbatch; ++b) {
        load_batch(b);
#pragma unroll
        for (int k = 0; k < GB; ++k) {
          if (b * GB + k < ng) {
#pragma unroll
            for (int e = 0; e < 16; ++e) m4[e & 3] = fmaxf(m4[e & 3], __uint_as_float(z[k][e]));
          }
        }
      }
      const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      const float mxs = mx * zs;
      float s2[2] = {0.f, 0.f};
      for (int b = 0; b < nbatch; ++b) {
        if (nbatch > 1) load_batch(b);
#pragma unroll
        for (int k = 0; k < GB; ++k) {
          const int g = b * GB + k;
          if (g < ng) {
            // pairs of probabilities rounded once to bf16: the packed word is what the MMA
            // reads and what the row sum adds up
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float e0 = ex2_approx(fmaf(__uint_as_float(z[k][2 * e]), zs, -mxs));
              const float e1 = ex2_approx(fmaf(__uint_as_float(z[k][2 * e + 1]), zs, -mxs));
              w[e] = pack_bf16x2(e0, e1);
              s2[0] += __uint_as_float(w[e] << 16);
              s2[1] += __uint_as_float(w[e] & 0xffff0000u);
            }
            if (g < nmeta) {
#pragma unroll
              for (int e = 0; e < 16; ++e)
                *reinterpret_cast<uint16_t*>(sm + G::PMT + sw128_offset(e, r, kMetaRows)) =
                    (uint16_t)((e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xffffu));
            } else {
              const int col = 16 * (g_lo + g - nmeta);
              *reinterpret_cast<uint4*>(sm + G::KB + sw128_offset(r, col, kC)) = make_uint4(w[0], w[1], w[2], w[3]);
              *reinterpret_cast<uint4*>(sm + G::KB + sw128_offset(r, col + 8, kC)) = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
        }
      }
      sum = s2[0] + s2[1];
    }
    tc_fence_before();
    fence_proxy_async_smem();
    mbar_arrive(&ctl->bar[F_PR]);

    // 3. y = O + alpha Ow / l -> staged bf16 tile -> TMA store
    if (ok && (ok = wait_bar(ctl, F_OWF, 0))) {
      tc_fence_after();
      const float rinv = p.alpha / sum;
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {
        uint32_t o[32], ow[32];
        tmem_ld32(tl + G::TO + 32 * g, o);
        tmem_ld32(tl + G::TOW + 32 * g, ow);
        tmem_ld_wait();
        float v[16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int e = 0; e < 16; ++e)
            v[e] = fmaf(rinv, __uint_as_float(ow[16 * h + e]), __uint_as_float(o[16 * h + e]));
          store16_bf16(sm + G::YS, kC, r, 32 * g + 16 * h, v);
        }
      }
      fence_proxy_async_smem();
    }
    named_sync(1, 128);
    if (ok && threadIdx.x == 64) {
      // rows at or beyond L are clipped by the store
      tma_store_3d(&maps.y, sm + G::YS, 0, t0, bh);
      tma_store_3d(&maps.y, sm + G::YS + 16384, 64, t0, bh);
      bulk_commit();
      bulk_wait_read();  // shared memory may be released once the stores have read it
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

// The workspace is the context the backward can reuse (GlaCtx).
using FwdWs = GlaCtx;

size_t fwd_ws_layout(int BH, int L, unsigned char* p, FwdWs* w) {
  const size_t nc = (L + kC - 1) / kC;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    unsigned char* r = p ? p + off : nullptr;
    off += align_up(bytes, 256);
    return r;
  };
  FwdWs g;
  g.qt = reinterpret_cast<bf16*>(take((size_t)BH * L * kD * sizeof(bf16)));
  g.kt = reinterpret_cast<bf16*>(take((size_t)BH * L * kD * sizeof(bf16)));
  g.eb = reinterpret_cast<bf16*>(take((size_t)BH * L * kD * sizeof(bf16)));
  g.gam = reinterpret_cast<float*>(take((size_t)BH * nc * kD * sizeof(float)));
  g.hs = reinterpret_cast<bf16*>(take((size_t)BH * nc * kD * kD * sizeof(bf16)));
  g.wide = reinterpret_cast<int*>(take((size_t)BH * nc * sizeof(int)));
  g.wlist = reinterpret_cast<int*>(take((size_t)BH * nc * sizeof(int)));
  const size_t seg = gla_seg_scratch(BH, L);
  g.seg = seg ? reinterpret_cast<float*>(take(seg)) : nullptr;
  if (w) *w = g;
  return off;
}

template <int NP>
cudaError_t launch_np(const FMaps& maps, const FParams& p, int grid, cudaStream_t s) {
  const size_t smem = FCfg<NP>::TOTAL;
  cudaError_t e = cudaFuncSetAttribute(fwd_chunk_kernel<NP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  trace_begin("fwd_chunk_tc", s);
  e = launch_pdl(fwd_chunk_kernel<NP>, dim3(grid), dim3(kThreads), smem, s, maps, p);
  trace_end(s);
  return e;
}

}  // namespace

bool fwd_chunk_tc_supported(int dk, int dv, int L, int W, int M, lizard_dtype dt) {
  return dt == LIZARD_BF16 && dk == kD && dv == kD && L > 0 && W >= 1 && W <= 2 * 64 + 1 &&
         M <= kMetaRows && tma_encode_available();
}

size_t fwd_chunk_tc_workspace(int BH, int L) { return fwd_ws_layout(BH, L, nullptr, nullptr); }

GlaCtx fwd_chunk_tc_ctx(int BH, int L, unsigned char* ws) {
  GlaCtx c;
  fwd_ws_layout(BH, L, ws, &c);
  return c;
}

cudaError_t launch_fwd_chunk_tc(const FwdArgs& a, unsigned char* ws, cudaStream_t s, int* launches) {
  const int BH = a.B * a.H, L = a.L;
  const int nc = (L + kC - 1) / kC;
  FwdWs w;
  fwd_ws_layout(BH, L, ws, &w);
  cudaError_t e;
  GlaStatesArgs ga{BH, L, a.pq, a.pk, a.lg, a.v, nullptr, a.h0, a.hf, nullptr,
                   w.qt, w.kt, w.eb, w.gam, w.hs, nullptr, a.status, w.seg,
                   w.wide, w.wlist, a.wcount ? a.wcount : a.status + kWsWideCount};
  e = a.xq ? launch_gla_prep_fmap(ga, a.H, a.xq, a.xk, a.wq, a.wk, s, launches)
           : launch_gla_prep(ga, s, launches);
  if (e != cudaSuccess) return e;
  if ((e = launch_gla_scan(ga, GlaScan::kStates, s, launches)) != cudaSuccess) return e;

  const int np = a.W <= 65 ? 1 : 2;
  const uint32_t br = (uint32_t)(kC + 64 * np);
  const uint64_t bhl = (uint64_t)BH, Ll = (uint64_t)L, zs = (uint64_t)BH * nc;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  FMaps m;
  bool ok = make_tma_map_bf16(&m.qt, w.qt, kD, Ll, bhl, 64, kC, sw) &&
            make_tma_map_bf16(&m.kt, w.kt, kD, Ll, bhl, 64, kC, sw) &&
            make_tma_map_bf16(&m.hs, w.hs, kD, kD, zs, 64, kC, sw) &&
            make_tma_map_bf16(&m.v, a.v, kD, Ll, bhl, 64, kC, sw) &&
            make_tma_map_bf16(&m.q, a.q, kD, Ll, bhl, 64, kC, sw) &&
            make_tma_map_bf16(&m.kb, a.k, kD, Ll, bhl, 64, br, sw) &&
            make_tma_map_bf16(&m.vb, a.v, kD, Ll, bhl, 64, br, sw) &&
            make_tma_map_bf16(&m.y, a.y, kD, Ll, bhl, 64, kC, sw);
  if (a.M > 0) {
    ok = ok && make_tma_map_bf16(&m.mk, a.mk, kD, a.M, a.H, 64, kMetaRows, sw) &&
         make_tma_map_bf16(&m.mv, a.mv, kD, a.M, a.H, 64, kMetaRows, sw);
  } else {
    m.mk = m.q;
    m.mv = m.v;
  }
  if (!ok) return cudaErrorInvalidValue;
  FParams p{a.H, L, a.M, a.W, nc, ctas_per_wave(1), a.scale, a.alpha, a.status};
  e = np == 1 ? launch_np<1>(m, p, BH * nc, s) : launch_np<2>(m, p, BH * nc, s);
  ++*launches;
  if (e != cudaSuccess) return e;
  // Chunks whose gate range the factorisation cannot hold are recomputed exactly; the
  // recomputation also leaves their phi_q, phi_k in the context's e^b and Kt sections.
  WideFix wf{ga.wcount, w.wlist, nc, w.hs};
  wf.phq = w.eb;
  wf.phk = w.kt;
  return launch_fwd_wide_fix(a, wf, s, launches);
}

}  // namespace lz
