// k_bwd_tc.cu -- backward of the GLA branch on tcgen05 tensor cores (bf16, d = 128).
//
// The pages give no backward formulas; this is the exact adjoint of the chunkwise forward
// ("Lizard", arXiv 2507.09025, Method: parallel form with cumulative gate products), laid
// out so that every chunk is independent once two linear scans over the chunk states are
// done.  Chunks hold C = 128 tokens; b is the chunk-local inclusive cumsum of log gamma,
// Gamma its last value, Qt = phi_q e^b, Kt = phi_k e^-b, h_c the state at the start of
// chunk c and G_c the adjoint of the state at its end.
//
//   1. prep   (k_gla_states_tc.cu)  Qt, Kt and e^b in bf16, Gamma in fp32.
//   2. scan   (k_gla_states_tc.cu)  h_{c+1} = diag(e^Gamma_c) (h_c + Kt_c^T V_c), h_0 = h0
//                                   G_{c-1} = diag(e^Gamma_c) G_c + Qt_c^T dY_c, G_{nc-1} = 0
//                                   stored as bf16 h_c and Gt_c = diag(e^Gamma_c) G_c;
//                                   G_{-1} is the adjoint of h0.
//   3. chunk  (tcgen05)     per (b, h, chunk), every product M = N = K = 128:
//                             A = dY V^T,  P = Qt Kt^T        (masked to s <= t, bf16)
//                             dQt = dY h^T + A Kt,   dKt = V Gt^T + A^T Qt
//                             dV  = Kt Gt + P^T dY
//                           then d phi_q = dQt e^b, d phi_k = dKt e^-b, and the per-token
//                           log-gate term r = phi_q d phi_q - phi_k d phi_k = Qt dQt - Kt dKt
//                           summed from the chunk's end (and its chunk total); outputs are
//                           staged in shared memory and written by TMA stores.
//   4. suffix (CUDA cores)  d log gamma_t = sum_{t' >= t} r_t': adds the totals of the later
//                           chunks.
//
// Every wait is bounded; on a timeout the CTA records LIZARD_ERR_TIMEOUT in the status
// word, drains its copies and MMAs, frees its tensor memory and returns.
#include "lizard_dev.cuh"
#include "lizard_internal.h"
#include "tc_pipe.cuh"

namespace lz {
namespace {

using namespace tc;

constexpr int kC = kGlaChunk;  // chunk
constexpr int kD = 128;        // dk = dv

struct GlaWs {
  bf16 *qt, *kt, *eb;  // [BH][L][128]
  float* gam;          // [BH][nc][128]
  bf16 *hs, *gs;       // [BH][nc][128][128]
  float* rtot;         // [BH][nc][128]
  float* seg;          // scratch of a split scan, or null
  int *wide, *wlist;   // wide-chunk flags and list [BH][nc]
  float* wfix;         // walk scratch of the wide-chunk recomputation
};

size_t gla_ws_layout(int BH, int L, unsigned char* p, GlaWs* w) {
  const size_t nc = (L + kC - 1) / kC;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    unsigned char* r = p ? p + off : nullptr;
    off += align_up(bytes, 256);
    return r;
  };
  const size_t tok = (size_t)BH * L * kD * sizeof(bf16);
  const size_t st = (size_t)BH * nc * kD * kD * sizeof(bf16);
  const size_t vec = (size_t)BH * nc * kD * sizeof(float);
  GlaWs g;
  g.qt = reinterpret_cast<bf16*>(take(tok));
  g.kt = reinterpret_cast<bf16*>(take(tok));
  g.eb = reinterpret_cast<bf16*>(take(tok));
  g.gam = reinterpret_cast<float*>(take(vec));
  g.hs = reinterpret_cast<bf16*>(take(st));
  g.gs = reinterpret_cast<bf16*>(take(st));
  g.rtot = reinterpret_cast<float*>(take(vec));
  g.wide = reinterpret_cast<int*>(take((size_t)BH * nc * sizeof(int)));
  g.wlist = reinterpret_cast<int*>(take((size_t)BH * nc * sizeof(int)));
  g.wfix = reinterpret_cast<float*>(take(bwd_wide_scratch_bytes(BH, (int)nc)));
  const size_t seg = gla_seg_scratch(BH, L);
  g.seg = seg ? reinterpret_cast<float*>(take(seg)) : nullptr;
  if (w) *w = g;
  return off;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ------------------------------------------------------------------------------------
// 3. chunk: one CTA per (b*h, chunk); warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
//    (thread = tile row, half of the columns).
// ------------------------------------------------------------------------------------
struct ChunkMaps {
  CUtensorMap dy, v, qt, kt, hs, gs, eb;  // loads
  CUtensorMap dpq, dpk, dlg, dvo;        // stores
};

struct ChunkP {
  int L, nc;
  int ahead;  // CTAs per wave: the tile whose inputs this CTA prefetches into L2
  float* rtot;
  unsigned* status;
};

enum {
  M_LD0 = 0, M_LD1, M_LD2, M_LD3, M_A, M_P, M_AS, M_PS, M_DV, M_EB, M_DONE, M_COUNT
};
constexpr uint32_t kTile = kC * kD * 2;  // 32 KB
// seven 32 KB tiles (e^b has its own, so it loads with the others), the [8][32] partial
// sums of r, the barriers: the 227 KB a CTA may have
constexpr uint32_t C_DY = 0, C_V = kTile, C_QT = 2 * kTile, C_KT = 3 * kTile, C_HS = 4 * kTile,
                   C_GS = 5 * kTile, C_EB = 6 * kTile, C_RED = 7 * kTile, C_BARS = C_RED + 1024;
constexpr size_t kChunkSmem = C_BARS + 1024 + 1024;
static_assert(kChunkSmem <= 232448, "shared memory per CTA");
constexpr int kChunkThreads = 10 * 32;
constexpr int kEpiThreads = 8 * 32;
// TMEM columns
constexpr uint32_t T_A = 0, T_P = 128, T_DQ = 256, T_DK = 384;

__global__ void __launch_bounds__(kChunkThreads, 1)
chunk_kernel(const __grid_constant__ ChunkMaps maps, const ChunkP p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  using Ctl = tc::Ctl<M_COUNT>;
  Ctl* ctl = reinterpret_cast<Ctl*>(sm + C_BARS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nc = p.nc, L = p.L;
  const int c = blockIdx.x % nc, bh = blockIdx.x / nc;
  const int t0 = c * kC, n = min(kC, L - t0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < M_COUNT; ++i)
      mbar_init(&ctl->bar[i], (i == M_AS || i == M_PS) ? (uint32_t)kEpiThreads : 1u);
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
      const int zs = bh * nc + c;
      mbar_arrive_expect_tx(&ctl->bar[M_LD0], 2 * kTile);
      tma_load_3d(sm + C_DY, &maps.dy, 0, t0, bh, &ctl->bar[M_LD0]);
      tma_load_3d(sm + C_DY + kTile / 2, &maps.dy, 64, t0, bh, &ctl->bar[M_LD0]);
      tma_load_3d(sm + C_HS, &maps.hs, 0, 0, zs, &ctl->bar[M_LD0]);
      tma_load_3d(sm + C_HS + kTile / 2, &maps.hs, 64, 0, zs, &ctl->bar[M_LD0]);
      mbar_arrive_expect_tx(&ctl->bar[M_LD1], kTile);
      tma_load_3d(sm + C_V, &maps.v, 0, t0, bh, &ctl->bar[M_LD1]);
      tma_load_3d(sm + C_V + kTile / 2, &maps.v, 64, t0, bh, &ctl->bar[M_LD1]);
      mbar_arrive_expect_tx(&ctl->bar[M_LD2], kTile);
      tma_load_3d(sm + C_GS, &maps.gs, 0, 0, zs, &ctl->bar[M_LD2]);
      tma_load_3d(sm + C_GS + kTile / 2, &maps.gs, 64, 0, zs, &ctl->bar[M_LD2]);
      mbar_arrive_expect_tx(&ctl->bar[M_LD3], 2 * kTile);
      tma_load_3d(sm + C_QT, &maps.qt, 0, t0, bh, &ctl->bar[M_LD3]);
      tma_load_3d(sm + C_QT + kTile / 2, &maps.qt, 64, t0, bh, &ctl->bar[M_LD3]);
      tma_load_3d(sm + C_KT, &maps.kt, 0, t0, bh, &ctl->bar[M_LD3]);
      tma_load_3d(sm + C_KT + kTile / 2, &maps.kt, 64, t0, bh, &ctl->bar[M_LD3]);
      mbar_arrive_expect_tx(&ctl->bar[M_EB], kTile);
      tma_load_3d(sm + C_EB, &maps.eb, 0, t0, bh, &ctl->bar[M_EB]);
      tma_load_3d(sm + C_EB + kTile / 2, &maps.eb, 64, t0, bh, &ctl->bar[M_EB]);
      // Once this tile's inputs are in, warm L2 with those of the tile one wave later, so
      // that its loads overlap this tile's tensor-core and epilogue phases.
      const int nb = blockIdx.x + p.ahead;
      if (nb < gridDim.x && wait_bar(ctl, M_LD3, 0)) {
        const int nbh = nb / nc, nt0 = (nb % nc) * kC, nzs = nb;
        for (int x = 0; x < kD; x += 64) {
          tma_prefetch_l2_3d(&maps.dy, x, nt0, nbh);
          tma_prefetch_l2_3d(&maps.hs, x, 0, nzs);
          tma_prefetch_l2_3d(&maps.v, x, nt0, nbh);
          tma_prefetch_l2_3d(&maps.gs, x, 0, nzs);
          tma_prefetch_l2_3d(&maps.qt, x, nt0, nbh);
          tma_prefetch_l2_3d(&maps.kt, x, nt0, nbh);
          tma_prefetch_l2_3d(&maps.eb, x, nt0, nbh);
        }
      }
      const uint64_t tw = globaltimer_ns();
      for (int b = M_LD0; b <= M_LD3; ++b) drain_bar(ctl, b, 1, tw);
      drain_bar(ctl, M_EB, 1, tw);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_kk = idesc_bf16(kC, kD, false, false);
      const uint32_t id_kn = idesc_bf16(kC, kD, false, true);
      const uint32_t id_nn = idesc_bf16(kC, kD, true, true);
      const uint32_t sb = smem_u32(sm);
      auto mma_kk = [&](uint32_t d, uint32_t a, uint32_t b, bool acc) {
        for (int j = 0; j < 8; ++j) mma_bf16(tmem + d, desc_k(a, kC, j), desc_k(b, kC, j), id_kk, acc || j > 0);
      };
      auto mma_kn = [&](uint32_t d, uint32_t a, uint32_t b, bool acc) {
        for (int j = 0; j < 8; ++j) mma_bf16(tmem + d, desc_k(a, kC, j), desc_mn(b, kC, j), id_kn, acc || j > 0);
      };
      auto mma_nn = [&](uint32_t d, uint32_t a, uint32_t b, bool acc) {
        for (int j = 0; j < 8; ++j) mma_bf16(tmem + d, desc_mn(a, kC, j), desc_mn(b, kC, j), id_nn, acc || j > 0);
      };
      bool ok = wait_bar(ctl, M_LD0, 0);
      if (ok) {
        tc_fence_after();
        mma_kk(T_DQ, sb + C_DY, sb + C_HS, false);  // dQt  = dY h^T
      }
      if (ok && (ok = wait_bar(ctl, M_LD1, 0))) {
        tc_fence_after();
        mma_kk(T_A, sb + C_DY, sb + C_V, false);    // A    = dY V^T
        mma_commit(&ctl->bar[M_A]);                 // (h tile free)
      }
      if (ok && (ok = wait_bar(ctl, M_LD2, 0))) {
        tc_fence_after();
        mma_kk(T_DK, sb + C_V, sb + C_GS, false);   // dKt  = V Gt^T
      }
      if (ok && (ok = wait_bar(ctl, M_LD3, 0))) {
        tc_fence_after();
        mma_kk(T_P, sb + C_QT, sb + C_KT, false);   // P    = Qt Kt^T
        mma_commit(&ctl->bar[M_P]);                 // (V tile free)
      }
      if (ok && (ok = wait_bar(ctl, M_AS, 0))) {
        tc_fence_after();
        mma_kn(T_DQ, sb + C_HS, sb + C_KT, true);   // dQt += A Kt
        mma_nn(T_DK, sb + C_HS, sb + C_QT, true);   // dKt += A^T Qt
        mma_kn(T_A, sb + C_KT, sb + C_GS, false);   // dV   = Kt Gt
      }
      if (ok && (ok = wait_bar(ctl, M_PS, 0))) {
        tc_fence_after();
        mma_nn(T_A, sb + C_V, sb + C_DY, true);     // dV  += P^T dY
        mma_commit(&ctl->bar[M_DV]);
      }
      if (!ok) ctl->abort = 1;
      mma_commit(&ctl->bar[M_DONE]);
      drain_bar(ctl, M_DONE, 1, globaltimer_ns());
    }
  } else {
    const int ew = warp - 2;      // 0..7
    const int qw = warp & 3;      // TMEM lane quarter
    const int hf = ew >> 2;       // column half
    const int t = qw * 32 + lane; // tile row
    const bool valid = t < n;
    const uint32_t tl = tmem + ((uint32_t)(qw * 32) << 16);
    float* red = reinterpret_cast<float*>(sm + C_RED);  // [8 segments][32] partial sums of r
    bool ok = true;

    // Masked (s <= t) bf16 copy of this thread's 64 columns of an M = N = 128 product,
    // K-major rows t.
    auto mask_store = [&](uint32_t tcol, unsigned char* dst) {
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        uint32_t r[32];
        tmem_ld32(tl + tcol + 64 * hf + 32 * g, r);
        tmem_ld_wait();
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int s0 = 64 * hf + 32 * g + 8 * m;
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s = s0 + 2 * e;
            w[e] = pack_bf16x2(s <= t ? __uint_as_float(r[8 * m + 2 * e]) : 0.f,
                               s + 1 <= t ? __uint_as_float(r[8 * m + 2 * e + 1]) : 0.f);
          }
          *reinterpret_cast<uint4*>(dst + sw128_offset(t, s0, kC)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    };

    if ((ok = wait_bar(ctl, M_A, 0))) {
      tc_fence_after();
      mask_store(T_A, sm + C_HS);
    }
    tc_fence_before();
    fence_proxy_async_smem();
    mbar_arrive(&ctl->bar[M_AS]);
    if (ok && (ok = wait_bar(ctl, M_P, 0))) {
      tc_fence_after();
      mask_store(T_P, sm + C_V);
    }
    tc_fence_before();
    fence_proxy_async_smem();
    mbar_arrive(&ctl->bar[M_PS]);

    // d phi_q, d phi_k, the log-gate term r summed from the chunk's end, and the GLA part
    // of dv, in four rounds of 32 columns (16 per thread).  Each round is staged in one of
    // two buffers carved from the operand tiles the MMAs no longer need and written by TMA
    // stores, which drain while the next round is computed.  e^b arrives by TMA with the
    // other inputs, in a tile of its own.
    const bool ready = ok && (ok = wait_bar(ctl, M_DV, 0)) && (ok = wait_bar(ctl, M_EB, 0));
    if (ready) tc_fence_after();
    const int et = threadIdx.x - 64;           // 0..255
    const int scol = et & 31, seg = et >> 5;   // suffix pass: column of the round, 16-row segment
    // lane 0 of the first four epilogue warps each issue one of the round's four stores (a
    // TMA issue costs its thread tens of nanoseconds; four warps issue side by side)
    const int sidx = scol == 0 && seg < 4 ? seg : -1;
    const CUtensorMap* smap = sidx == 0 ? &maps.dpq : sidx == 1 ? &maps.dpk : sidx == 2 ? &maps.dlg : &maps.dvo;
#pragma unroll 1
    for (int R = 0; R < 4; ++R) {
      // buffer 0: dY tile + first half of V; buffer 1: second half of V + Gt tile
      unsigned char* sdq = sm + ((R & 1) ? C_V + 16384 : C_DY);
      unsigned char* sdk = sdq + 8192;
      unsigned char* srr = sm + ((R & 1) ? C_GS : C_DY + 16384);
      unsigned char* sdv = srr + 16384;
      const int cl = 16 * hf;       // columns within the round
      const int i0 = 32 * R + cl;   // columns of the tile
      if (ready) {
        uint32_t dq[16], dk[16], dv[16];
        tmem_ld16(tl + T_DQ + i0, dq);
        tmem_ld16(tl + T_DK + i0, dk);
        tmem_ld16(tl + T_A + i0, dv);
        tmem_ld_wait();
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint32_t off = sw128_offset(t, i0 + 8 * m, kC);
          const uint4 qv = *reinterpret_cast<const uint4*>(sm + C_QT + off);
          const uint4 kv = *reinterpret_cast<const uint4*>(sm + C_KT + off);
          const uint4 ev = *reinterpret_cast<const uint4*>(sm + C_EB + off);
          const uint32_t qa[4] = {qv.x, qv.y, qv.z, qv.w};
          const uint32_t ka[4] = {kv.x, kv.y, kv.z, kv.w};
          const uint32_t ea[4] = {ev.x, ev.y, ev.z, ev.w};
          uint32_t wq[4], wk[4];
          float rr[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k0 = 8 * m + 2 * e;
            const float q0 = __uint_as_float(dq[k0]), q1 = __uint_as_float(dq[k0 + 1]);
            const float d0 = __uint_as_float(dk[k0]), d1 = __uint_as_float(dk[k0 + 1]);
            const float e0 = bf_lo(ea[e]), e1 = bf_hi(ea[e]);
            wq[e] = pack_bf16x2(q0 * e0, q1 * e1);
            wk[e] = pack_bf16x2(valid ? __fdividef(d0, e0) : 0.f, valid ? __fdividef(d1, e1) : 0.f);
            rr[2 * e] = valid ? bf_lo(qa[e]) * q0 - bf_lo(ka[e]) * d0 : 0.f;
            rr[2 * e + 1] = valid ? bf_hi(qa[e]) * q1 - bf_hi(ka[e]) * d1 : 0.f;
          }
          *reinterpret_cast<uint4*>(sdq + sw64_offset(t, cl + 8 * m)) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
          *reinterpret_cast<uint4*>(sdk + sw64_offset(t, cl + 8 * m)) = make_uint4(wk[0], wk[1], wk[2], wk[3]);
          *reinterpret_cast<float4*>(srr + sw128_offset_f32(t, cl + 8 * m, kC)) =
              make_float4(rr[0], rr[1], rr[2], rr[3]);
          *reinterpret_cast<float4*>(srr + sw128_offset_f32(t, cl + 8 * m + 4, kC)) =
              make_float4(rr[4], rr[5], rr[6], rr[7]);
        }
#pragma unroll
        for (int m = 0; m < 4; ++m)
          *reinterpret_cast<float4*>(sdv + sw128_offset_f32(t, cl + 4 * m, kC)) =
              make_float4(__uint_as_float(dv[4 * m]), __uint_as_float(dv[4 * m + 1]),
                          __uint_as_float(dv[4 * m + 2]), __uint_as_float(dv[4 * m + 3]));
      }
      named_sync(1, kEpiThreads);
      // suffix sums of r down the chunk: 8 segments of 16 rows per column; the thread keeps
      // its segment's 16 values in registers between the two passes
      float rv[16];
      if (ready) {
        float part = 0.f;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          rv[u] = *reinterpret_cast<const float*>(srr + sw128_offset_f32(16 * seg + u, scol, kC));
          part += rv[u];
        }
        red[seg * 32 + scol] = part;
      }
      named_sync(1, kEpiThreads);
      if (ready) {
        float run = 0.f;
#pragma unroll
        for (int s2 = 7; s2 > 0; --s2)
          if (s2 > seg) run += red[s2 * 32 + scol];
#pragma unroll
        for (int u = 15; u >= 0; --u) {
          run += rv[u];
          *reinterpret_cast<float*>(srr + sw128_offset_f32(16 * seg + u, scol, kC)) = run;
        }
        if (seg == 0) p.rtot[((size_t)bh * nc + c) * kD + 32 * R + scol] = run;
      }
      fence_proxy_async_smem();
      named_sync(1, kEpiThreads);
      if (ready && sidx >= 0) {
        // rows at or beyond L are clipped by the stores
        tma_store_3d(smap, sidx == 0 ? sdq : sidx == 1 ? sdk : sidx == 2 ? srr : sdv, 32 * R, t0, bh);
        bulk_commit();
        bulk_wait_read_prev();  // this thread's store of round R-1 (the other buffer) has been read
      }
      named_sync(1, kEpiThreads);
    }
    if (ready && sidx >= 0) bulk_wait_read();
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
// 4. suffix: one CTA per (chunk, b*h), thread = key dimension; adds the sums of the later
//    chunks to the in-chunk suffix sums.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kD) suffix_kernel(int L, int nc, float* dlg, const float* rtot,
                                                   const int* wide) {
  const int c = blockIdx.x, bh = blockIdx.y, i = threadIdx.x;
  pdl_wait();
  // the last chunk has nothing to add; a wide chunk's values are final already
  if (c == nc - 1 || wide[(size_t)bh * nc + c]) {
    pdl_trigger();
    return;
  }
  // the later chunks' totals, in four independent sums so that their loads overlap
  float cs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int c2 = c + 1; c2 < nc; ++c2) cs[(c2 - c - 1) & 3] += rtot[((size_t)bh * nc + c2) * kD + i];
  const float carry = (cs[0] + cs[1]) + (cs[2] + cs[3]);
  const int t0 = c * kC, n = min(kC, L - t0);
  float* r = dlg + ((size_t)bh * L + t0) * kD + i;
#pragma unroll 8
  for (int t = 0; t < n; ++t) r[(size_t)t * kD] += carry;
  pdl_trigger();
}

template <typename K, typename M, typename P>
cudaError_t launch_tc(K kernel, const M& maps, const P& p, int grid, int threads, size_t smem,
                      const char* name, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  trace_begin(name, s);
  e = launch_pdl(kernel, dim3(grid), dim3(threads), smem, s, maps, p);
  trace_end(s);
  return e;
}

}  // namespace

bool fwd_ctx_usable(int dk, int dv, int L, int W, int M, lizard_dtype dt) {
  return fwd_chunk_tc_supported(dk, dv, L, W, M, dt);
}

bool bwd_gla_tc_supported(int dk, int dv, int L, lizard_dtype dt) {
  return dt == LIZARD_BF16 && dk == kD && dv == kD && L > 0 && tma_encode_available();
}

size_t bwd_gla_tc_workspace(int BH, int L) { return gla_ws_layout(BH, L, nullptr, nullptr); }

cudaError_t launch_bwd_gla_tc(const BwdArgs& a, float* dvacc, unsigned char* ws, cudaStream_t s,
                              int* launches) {
  const int BH = a.B * a.H, L = a.L;
  const int nc = (L + kC - 1) / kC;
  GlaWs w;
  gla_ws_layout(BH, L, ws, &w);
  cudaError_t e;

  // With the forward's context, its Qt, Kt, e^b, Gamma and chunk states are reused and
  // only the adjoint scan runs.
  const bool ctx = a.fwd_ws != nullptr && fwd_ctx_usable(a.dk, a.dv, a.L, a.W, a.M, LIZARD_BF16);
  // Wide chunks: listed by this call's prep, or by the forward's (count in its header).
  // From the forward's context their phi_q, phi_k are read where its recomputation left
  // them (the e^b and Kt sections), otherwise from the inputs.
  unsigned* wcount = a.status + kWsWideCount;
  const bf16* phq_in = static_cast<const bf16*>(a.pq);
  const bf16* phk_in = static_cast<const bf16*>(a.pk);
  if (ctx) {
    const GlaCtx fc = fwd_chunk_tc_ctx(BH, L, a.fwd_ws);
    w.qt = fc.qt;
    w.kt = fc.kt;
    w.eb = fc.eb;
    w.gam = fc.gam;
    w.hs = fc.hs;
    w.wide = fc.wide;
    w.wlist = fc.wlist;
    wcount = reinterpret_cast<unsigned*>(a.fwd_ws - kWsHeader) + kWsWideCount;
    phq_in = fc.eb;
    phk_in = fc.kt;
  }
  GlaStatesArgs ga{BH, L, a.pq, a.pk, a.lg, a.v, a.dy, a.h0, nullptr, a.dh0,
                   w.qt, w.kt, w.eb, w.gam, w.hs, w.gs, a.status, w.seg,
                   w.wide, w.wlist, wcount};
  if (!ctx && (e = launch_gla_prep(ga, s, launches)) != cudaSuccess) return e;
  if ((e = launch_gla_scan(ga, ctx ? GlaScan::kAdjoints : GlaScan::kBoth, s, launches)) != cudaSuccess)
    return e;

  const uint64_t bhl = (uint64_t)BH, Ll = (uint64_t)L, zs = (uint64_t)BH * nc;
  ChunkMaps cm;
  bool ok = make_tma_map_bf16(&cm.dy, a.dy, kD, Ll, bhl, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&cm.v, a.v, kD, Ll, bhl, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&cm.qt, w.qt, kD, Ll, bhl, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&cm.kt, w.kt, kD, Ll, bhl, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&cm.hs, w.hs, kD, kD, zs, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&cm.gs, w.gs, kD, kD, zs, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&cm.eb, w.eb, kD, Ll, bhl, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&cm.dpq, a.dpq, kD, Ll, bhl, 32, kC, CU_TENSOR_MAP_SWIZZLE_64B) &&
            make_tma_map_bf16(&cm.dpk, a.dpk, kD, Ll, bhl, 32, kC, CU_TENSOR_MAP_SWIZZLE_64B) &&
            make_tma_map_f32(&cm.dlg, a.dlg, kD, Ll, bhl, 32, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_f32(&cm.dvo, dvacc, kD, Ll, bhl, 32, kC, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;

  ChunkP cp{L, nc, ctas_per_wave(1), w.rtot, a.status};
  e = launch_tc(chunk_kernel, cm, cp, BH * nc, kChunkThreads, kChunkSmem, "bwd_chunk_tc", s);
  ++*launches;
  if (e != cudaSuccess) return e;

  // Wide chunks recomputed exactly (their in-chunk sums and totals of the log-gate term
  // included) before the suffix pass adds the later chunks' totals.
  WideFix wf{wcount, w.wlist, nc, w.hs, w.gs};
  wf.phq_in = phq_in;
  wf.phk_in = phk_in;
  wf.rtot = w.rtot;
  wf.scratch = w.wfix;
  if ((e = launch_bwd_wide_fix(a, wf, dvacc, s, launches)) != cudaSuccess) return e;

  trace_begin("bwd_suffix", s);
  e = launch_pdl(suffix_kernel, dim3(nc, BH), dim3(kD), 0, s, L, nc, a.dlg,
                 static_cast<const float*>(w.rtot), static_cast<const int*>(w.wide));
  trace_end(s);
  ++*launches;
  return e;
}

}  // namespace lz
