// k_fwd_tc.cu -- fused Lizard-attention forward on tcgen05 tensor cores (bf16, d = 128).
//
// One CTA per (batch, head, 32-column slice of dv): the four CTAs of a head walk the
// 64-token chunks in order, each keeping its 128 x 32 fp32 slice of the GLA state in
// tensor memory.  Per chunk c (tokens t0 .. t0+63), with b the chunk-local inclusive
// cumsum of log gamma and Gamma its last value ("Lizard", arXiv 2507.09025, Method:
// parallel form with cumulative gate products, absorbed into the features):
//   Qt = phi_q * e^b, Kt = phi_k * e^-b                         (CUDA cores, in place)
//   S  = Qt Kt^T                       M=64  N=64  K=128        (tcgen05)
//   O  = Qt h_bf16 + mask(S)_bf16 V    M=64  N=32  K=128 / 64   (tcgen05)
//   h  = diag(e^Gamma) (h + Kt^T V)    M=128 N=32  K=64         (tcgen05 + CUDA cores)
// and the anchor window (papernotes.org note on Lizard, 关键设计: Anchor Window
// Attention) on the same chunk:
//   Z  = q [meta_k ; k_{chunk-NP..chunk}]^T   M=64 N=16+64(NP+1) K=128 (tcgen05)
//   P  = exp(scale (Z - rowmax)) on the visible keys, 0 elsewhere  (CUDA cores)
//   Ow = P [meta_v ; v]                        M=64 N=32              (tcgen05)
//   y  = O + alpha * Ow / rowsum(P), rounded to bf16 once.
// NP is how many earlier chunks the window reaches: 1 for W <= 65, 2 for W <= 129.
// With NP = 1 the window logits and probabilities are double-buffered, so the MMA
// issuer starts chunk c+1's logits before it waits for chunk c's softmax.
//
// All operands arrive by TMA (3D maps over [B*H, L, d]; rows outside [0, L) read as
// zeros), accumulate in fp32 in TMEM, and every wait is bounded: on a timeout the CTA
// records LIZARD_ERR_TIMEOUT in the status word, drains its copies and MMAs, frees its
// tensor memory and returns.
//
// Warp roles (18 warps): 0 TMA producer; 1 MMA issuer + TMEM owner; 2-9 feature
// transform (thread = key dimension x token half); 10-13 window softmax and epilogue on
// the M=64 tiles (rows 16w..16w+15 sit in lanes 0-15 of warp w%4's TMEM quarter);
// 14-17 causal mask of S and the state rescale (thread = key dimension, all 128 lanes).
#include <mutex>

#include "lizard_dev.cuh"
#include "lizard_internal.h"
#include "tc_sm100.cuh"

namespace lz {
namespace {

using namespace tc;

constexpr int kC = 64;   // chunk
constexpr int kD = 128;  // dk = dv
constexpr int kNV = 32;  // dv columns per CTA
constexpr int kSlices = kD / kNV;
constexpr int kThreads = 18 * 32;
constexpr uint64_t kWaitNs = 1000000000ull;      // 1 s for the exit drains
constexpr long long kWaitCycles = 2000000000ll;  // ~1 s of SM clock per wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaxLogSum = 80.f;  // |chunk-local log-gate sum| beyond which e^{+-b} overflows

template <int NP>
struct Cfg {
  static constexpr int NR = NP + 2;                 // k/v ring slots
  static constexpr int NZ = NP == 1 ? 2 : 1;        // Z / P buffers
  static constexpr int ZC = 16 + kC * (NP + 1);     // Z columns
  static constexpr int PATOMS = NP + 2;             // 64-column atoms of a P tile
  // TMEM columns
  static constexpr uint32_t TS = 0;      // S, 64
  static constexpr uint32_t TO = 64;     // O, 2 x 32
  static constexpr uint32_t TOW = 128;   // Ow, 2 x 32
  static constexpr uint32_t TH = 192;    // h, 32
  static constexpr uint32_t TZ = 224;    // Z, NZ x ZC
  static_assert(TZ + NZ * ZC <= 512, "TMEM budget");
  // shared memory (byte offsets from a 1024-aligned base)
  static constexpr uint32_t STAGE = 32768;                  // phi_q, phi_k tiles
  static constexpr uint32_t Q = 2 * STAGE;                  // q tile
  static constexpr uint32_t KRING = Q + 16384;              // NR x 16 KB
  static constexpr uint32_t VRING = KRING + NR * 16384;     // NR x 4 KB
  static constexpr uint32_t METAK = VRING + NR * 4096;      // 4 KB
  static constexpr uint32_t METAV = METAK + 4096;           // 1 KB
  static constexpr uint32_t SBF = METAV + 1024;             // 8 KB
  static constexpr uint32_t PBUF = SBF + 8192;              // NZ x PATOMS x 8 KB
  static constexpr uint32_t HBF = PBUF + NZ * PATOMS * 8192;
  static constexpr uint32_t EG = HBF + 8192;                // eg[2][128], qsum[2][4][128]
  static constexpr uint32_t BARS = EG + 8192;
  static constexpr uint32_t TOTAL = BARS + 1024 + 1024;     // + alignment slack
};

struct Params {
  int H, L, M, W;
  float scale, alpha;
  const float* lg;
  bf16* y;
  const float* h0;
  float* hf;
  unsigned* status;
};

struct Maps {
  CUtensorMap phq, phk, q, k, v, mk, mv;
};

// Barrier indices; [2] entries are indexed by chunk parity (or buffer).
enum {
  B_FULL = 0, B_EMPTY = 2, B_OPND = 4, B_EGFULL = 6, B_EGFREE = 8, B_QX = 10,
  B_SPARE = 12, B_OFULL = 14, B_OFREE = 16, B_SWFULL = 18, B_SWFREE = 20, B_PREADY = 22,
  B_PFREE = 24, B_KFULL = 26, B_KEMPTY = 30, B_VFULL = 34, B_VEMPTY = 38, B_SFULL = 42,
  B_SFREE, B_QFULL, B_QEMPTY, B_META, B_SBFREADY, B_SBFFREE, B_HACC, B_HREADY, B_MMADONE,
  B_COUNT
};

__host__ __device__ constexpr uint32_t bar_count(int i) {
  return (i == B_OPND || i == B_OPND + 1 || i == B_QX || i == B_QX + 1) ? 256u
         : (i == B_EGFULL || i == B_EGFULL + 1) ? 64u
         : (i == B_EGFREE || i == B_EGFREE + 1 || i == B_OFREE || i == B_OFREE + 1 ||
            i == B_SWFREE || i == B_SWFREE + 1 || i == B_PREADY || i == B_PREADY + 1 ||
            i == B_SFREE || i == B_SBFREADY || i == B_HREADY)
             ? 128u
             : 1u;
}

struct Ctl {
  uint64_t bar[B_COUNT];
  uint32_t tmem;
  int abort;
};

// Bounded wait: gives up (and raises the CTA's abort flag) after kWaitCycles SM clock
// cycles -- about one second at the top clock -- or as soon as another role aborted.
__device__ __forceinline__ bool wait_bar(Ctl* ctl, int i, uint32_t parity) {
  uint64_t* b = &ctl->bar[i];
  if (mbar_try_wait(b, parity)) return true;
  const long long t0 = clock64();
  while (true) {
#pragma unroll 1
    for (int k = 0; k < 32; ++k)
      if (mbar_try_wait(b, parity)) return true;
    if (*(volatile int*)&ctl->abort) return false;
    if (clock64() - t0 > kWaitCycles) {
      *(volatile int*)&ctl->abort = 1;
      return false;
    }
  }
}

// Waits, without time-out bookkeeping of its own, for the last armed phase of a
// barrier; used only while leaving.
__device__ __forceinline__ void drain_bar(Ctl* ctl, int i, uint32_t armed, uint64_t t0) {
  if (armed == 0) return;
  while (!mbar_try_wait(&ctl->bar[i], (armed - 1) & 1))
    if (globaltimer_ns() - t0 > kWaitNs) break;
}

// K-major SW128 operand descriptor for k-step j (16 elements) of a tile with `rows` rows.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int rows, int j) {
  return smem_desc(base + (uint32_t)((j * 16) >> 6) * rows * 128u + (uint32_t)((j * 16) & 63) * 2u,
                   16, 1024, kSw128);
}

template <int NP>
__global__ void __launch_bounds__(kThreads, 1)
fwd_tc_kernel(const __grid_constant__ Maps maps, const Params p) {
  using G = Cfg<NP>;
  constexpr int NR = G::NR, NZ = G::NZ, ZC = G::ZC;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(sm + G::BARS);
  float* eg = reinterpret_cast<float*>(sm + G::EG);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x / kSlices;
  const int c0 = (blockIdx.x % kSlices) * kNV;
  const int hh = bh % p.H;
  const int L = p.L;
  const int nc = (L + kC - 1) / kC;

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) mbar_init(&ctl->bar[i], bar_count(i));
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&maps.phq);
      tma_prefetch_desc(&maps.k);
      uint32_t armed_full0 = 0, armed_full1 = 0, armed_q = 0;
      uint32_t armed_k[NR], armed_v[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r) armed_k[r] = armed_v[r] = 0;
      bool ok = true;
      if (p.M > 0) {
        mbar_arrive_expect_tx(&ctl->bar[B_META], 4096 + 1024);
        tma_load_3d(sm + G::METAK, &maps.mk, 0, 0, hh, &ctl->bar[B_META]);
        tma_load_3d(sm + G::METAK + 2048, &maps.mk, 64, 0, hh, &ctl->bar[B_META]);
        tma_load_3d(sm + G::METAV, &maps.mv, c0, 0, hh, &ctl->bar[B_META]);
      } else {
        mbar_arrive(&ctl->bar[B_META]);
      }
      // k and v tiles of chunk j (j may be negative: rows before 0 read as zeros).  Keys
      // are released after the logits MMA, values after the P.V MMA.
      auto load_k = [&](int j) -> bool {
        const int u = j + NP, r = u % NR;
        if (u >= NR && !wait_bar(ctl, B_KEMPTY + r, ((u / NR) - 1) & 1)) return false;
        mbar_arrive_expect_tx(&ctl->bar[B_KFULL + r], 16384);
        unsigned char* kd = sm + G::KRING + r * 16384;
        tma_load_3d(kd, &maps.k, 0, j * kC, bh, &ctl->bar[B_KFULL + r]);
        tma_load_3d(kd + 8192, &maps.k, 64, j * kC, bh, &ctl->bar[B_KFULL + r]);
#pragma unroll
        for (int rr = 0; rr < NR; ++rr) armed_k[rr] += rr == r ? 1u : 0u;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int u = j + NP, r = u % NR;
        if (u >= NR && !wait_bar(ctl, B_VEMPTY + r, ((u / NR) - 1) & 1)) return false;
        mbar_arrive_expect_tx(&ctl->bar[B_VFULL + r], 4096);
        tma_load_3d(sm + G::VRING + r * 4096, &maps.v, c0, j * kC, bh, &ctl->bar[B_VFULL + r]);
#pragma unroll
        for (int rr = 0; rr < NR; ++rr) armed_v[rr] += rr == r ? 1u : 0u;
        return true;
      };
      for (int j = -NP; j < 0 && ok; ++j) ok = load_k(j) && load_v(j);
      for (int c = 0; c < nc && ok; ++c) {
        const int s = c & 1, u = c >> 1;
        if (u >= 1 && !(ok = wait_bar(ctl, B_EMPTY + s, (u - 1) & 1))) break;
        mbar_arrive_expect_tx(&ctl->bar[B_FULL + s], 32768);
        unsigned char* st = sm + s * G::STAGE;
        tma_load_3d(st, &maps.phq, 0, c * kC, bh, &ctl->bar[B_FULL + s]);
        tma_load_3d(st + 8192, &maps.phq, 64, c * kC, bh, &ctl->bar[B_FULL + s]);
        tma_load_3d(st + 16384, &maps.phk, 0, c * kC, bh, &ctl->bar[B_FULL + s]);
        tma_load_3d(st + 24576, &maps.phk, 64, c * kC, bh, &ctl->bar[B_FULL + s]);
        if (s) ++armed_full1;
        else ++armed_full0;
        if (!(ok = load_k(c))) break;
        if (c >= 1 && !(ok = wait_bar(ctl, B_QEMPTY, (c - 1) & 1))) break;
        mbar_arrive_expect_tx(&ctl->bar[B_QFULL], 16384);
        tma_load_3d(sm + G::Q, &maps.q, 0, c * kC, bh, &ctl->bar[B_QFULL]);
        tma_load_3d(sm + G::Q + 8192, &maps.q, 64, c * kC, bh, &ctl->bar[B_QFULL]);
        ++armed_q;
        if (!(ok = load_v(c))) break;
      }
      if (!ok) ctl->abort = 1;
      // Never leave with copies in flight.
      const uint64_t t0 = globaltimer_ns();
      drain_bar(ctl, B_FULL, armed_full0, t0);
      drain_bar(ctl, B_FULL + 1, armed_full1, t0);
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        drain_bar(ctl, B_KFULL + r, armed_k[r], t0);
        drain_bar(ctl, B_VFULL + r, armed_v[r], t0);
      }
      drain_bar(ctl, B_QFULL, armed_q, t0);
      drain_bar(ctl, B_META, p.M > 0 ? 1u : 0u, t0);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(64, 64, false, false);
      const uint32_t id_o = idesc_bf16(64, kNV, false, true);
      const uint32_t id_h = idesc_bf16(128, kNV, true, true);
      const uint32_t id_z16 = idesc_bf16(64, 16, false, false);
      const uint32_t id_z64 = idesc_bf16(64, 64, false, false);
      const uint32_t sbase = smem_u32(sm);
      bool ok = wait_bar(ctl, B_META, 0);

      auto issue_S = [&](int c) -> bool {
        const int s = c & 1;
        if (!wait_bar(ctl, B_OPND + s, (c >> 1) & 1)) return false;
        if (c >= 1 && !wait_bar(ctl, B_SFREE, (c - 1) & 1)) return false;
        tc_fence_after();
        const uint32_t phq = sbase + s * G::STAGE, phk = phq + 16384;
        for (int j = 0; j < 8; ++j)
          mma_bf16(tmem + G::TS, desc_kmajor(phq, 64, j), desc_kmajor(phk, 64, j), id_s, j > 0);
        mma_commit(&ctl->bar[B_SFULL]);
        return true;
      };
      auto issue_Z = [&](int c) -> bool {
        const int zb = c % NZ, zu = c / NZ;
        if (!wait_bar(ctl, B_QFULL, c & 1)) return false;
        if (!wait_bar(ctl, B_KFULL + (c + NP) % NR, ((c + NP) / NR) & 1)) return false;
        if (c == 0)
          for (int jn = -NP; jn < 0; ++jn)
            if (!wait_bar(ctl, B_KFULL + (jn + NP) % NR, 0)) return false;
        if (zu >= 1 && !wait_bar(ctl, B_SWFREE + zb, (zu - 1) & 1)) return false;
        tc_fence_after();
        const uint32_t qb = sbase + G::Q;
        const uint32_t tz = tmem + G::TZ + zb * ZC;
        if (p.M > 0) {
          for (int j = 0; j < 8; ++j)
            mma_bf16(tz, desc_kmajor(qb, 64, j), desc_kmajor(sbase + G::METAK, 16, j), id_z16, j > 0);
        }
        for (int b = 0; b <= NP; ++b) {
          const uint32_t kb = sbase + G::KRING + ((c + b) % NR) * 16384;
          for (int j = 0; j < 8; ++j)
            mma_bf16(tz + 16 + 64 * b, desc_kmajor(qb, 64, j), desc_kmajor(kb, 64, j), id_z64, j > 0);
        }
        mma_commit(&ctl->bar[B_SWFULL + zb]);
        mma_commit(&ctl->bar[B_QEMPTY]);
        mma_commit(&ctl->bar[B_KEMPTY + c % NR]);  // chunk c - NP's keys are done
        return true;
      };
      auto issue_OH = [&](int c) -> bool {
        const int s = c & 1, u = c >> 1;
        if (!wait_bar(ctl, B_HREADY, c & 1)) return false;
        if (u >= 1 && !wait_bar(ctl, B_OFREE + s, (u - 1) & 1)) return false;
        if (!wait_bar(ctl, B_VFULL + (c + NP) % NR, ((c + NP) / NR) & 1)) return false;
        if (c == 0)
          for (int jn = -NP; jn < 0; ++jn)
            if (!wait_bar(ctl, B_VFULL + (jn + NP) % NR, 0)) return false;
        tc_fence_after();
        const uint32_t phq = sbase + s * G::STAGE, phk = phq + 16384;
        const uint32_t hb = sbase + G::HBF;
        for (int j = 0; j < 8; ++j)
          mma_bf16(tmem + G::TO + s * 32, desc_kmajor(phq, 64, j),
                   smem_desc(hb + j * 1024, 8192, 512, kSw64), id_o, j > 0);
        const uint32_t vb = sbase + G::VRING + ((c + NP) % NR) * 4096;
        for (int j = 0; j < 4; ++j)
          mma_bf16(tmem + G::TH, smem_desc(phk + j * 2048, 8192, 1024, kSw128),
                   smem_desc(vb + j * 1024, 4096, 512, kSw64), id_h, true);
        mma_commit(&ctl->bar[B_HACC]);
        return true;
      };
      auto issue_SV = [&](int c) -> bool {
        const int s = c & 1;
        if (!wait_bar(ctl, B_SBFREADY, c & 1)) return false;
        tc_fence_after();
        const uint32_t vb = sbase + G::VRING + ((c + NP) % NR) * 4096;
        for (int j = 0; j < 4; ++j)
          mma_bf16(tmem + G::TO + s * 32, desc_kmajor(sbase + G::SBF, 64, j),
                   smem_desc(vb + j * 1024, 4096, 512, kSw64), id_o, true);
        mma_commit(&ctl->bar[B_SBFFREE]);
        mma_commit(&ctl->bar[B_EMPTY + s]);
        return true;
      };
      auto issue_PV = [&](int c) -> bool {
        const int s = c & 1, pb = c % NZ;
        if (!wait_bar(ctl, B_PREADY + pb, (c / NZ) & 1)) return false;
        tc_fence_after();
        const uint32_t pt = sbase + G::PBUF + pb * (G::PATOMS * 8192);
        const uint32_t tow = tmem + G::TOW + s * 32;
        if (p.M > 0)
          mma_bf16(tow, desc_kmajor(pt, 64, 0), smem_desc(sbase + G::METAV, 1024, 512, kSw64), id_o,
                   false);
        for (int b = 0; b <= NP; ++b) {
          const uint32_t vv = sbase + G::VRING + ((c + b) % NR) * 4096;
          for (int j = 0; j < 4; ++j)
            mma_bf16(tow, desc_kmajor(pt, 64, 1 + b * 4 + j),
                     smem_desc(vv + j * 1024, 4096, 512, kSw64), id_o, p.M > 0 || b > 0 || j > 0);
        }
        mma_commit(&ctl->bar[B_PFREE + pb]);
        mma_commit(&ctl->bar[B_OFULL + s]);
        mma_commit(&ctl->bar[B_VEMPTY + c % NR]);  // chunk c - NP's values are done
        return true;
      };

      if (ok && nc > 0) ok = issue_S(0) && issue_Z(0);
      for (int c = 0; c < nc && ok; ++c) {
        ok = issue_OH(c) && issue_SV(c);
        if (ok && c + 1 < nc) ok = issue_S(c + 1);
        if (ok && NZ == 2 && c + 1 < nc) ok = issue_Z(c + 1);
        if (ok) ok = issue_PV(c);
        if (ok && NZ == 1 && c + 1 < nc) ok = issue_Z(c + 1);
      }
      if (!ok) ctl->abort = 1;
      mma_commit(&ctl->bar[B_MMADONE]);
      drain_bar(ctl, B_MMADONE, 1, globaltimer_ns());
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------------ transform
    // 256 threads: column pair cp (key dimensions 2cp, 2cp+1) x token quarter qt (tokens
    // 16qt .. 16qt+15).  The quarters exchange their partial sums through shared memory;
    // the raw log gate of the next chunk is prefetched into registers.
    const int tt = threadIdx.x - 64;
    const int cp = tt & 63, qt = tt >> 6;
    const float2* lgp = reinterpret_cast<const float2*>(p.lg + (size_t)bh * L * kD) + cp;
    float* qsum = eg + 256;  // [2][4][128]
    float2 lgv[16];
    auto fetch = [&](int c) {
      const int tb = c * kC + 16 * qt;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        lgv[i] = (tb + i < L) ? lgp[(size_t)(tb + i) * (kD / 2)] : make_float2(0.f, 0.f);
    };
    fetch(0);
    bool ok = true;
    // byte offset of columns (2cp, 2cp+1) in row t of a 64-row 128-byte-swizzled tile
    const uint32_t colb = (uint32_t)(cp >> 5) * 8192u + (uint32_t)(cp & 3) * 4u;
    const uint32_t chk = (uint32_t)((cp & 31) >> 2);
    for (int c = 0; c < nc && ok; ++c) {
      const int s = c & 1, u = c >> 1;
      float2 part = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        part.x += lgv[i].x;
        part.y += lgv[i].y;
      }
      *reinterpret_cast<float2*>(qsum + (s * 4 + qt) * 128 + 2 * cp) = part;
      mbar_arrive(&ctl->bar[B_QX + s]);
      if (!(ok = wait_bar(ctl, B_QX + s, u & 1))) break;
      float r0 = 0.f, r1 = 0.f;
      for (int q2 = 0; q2 < qt; ++q2) {
        const float2 v2 = *reinterpret_cast<const float2*>(qsum + (s * 4 + q2) * 128 + 2 * cp);
        r0 += v2.x;
        r1 += v2.y;
      }
      r0 *= kLog2e;
      r1 *= kLog2e;
      if (!(ok = wait_bar(ctl, B_FULL + s, u & 1))) break;
      unsigned char* phq = sm + s * G::STAGE;
      unsigned char* phk = phq + 16384;
      float big = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int t = 16 * qt + i;
        r0 = fmaf(lgv[i].x, kLog2e, r0);  // log2 of the cumulative gate, column 2cp
        r1 = fmaf(lgv[i].y, kLog2e, r1);  // column 2cp+1
        big = fmaxf(big, fmaxf(fabsf(r0), fabsf(r1)));
        const uint32_t off = colb + (uint32_t)t * 128u + ((chk ^ (uint32_t)(i & 7)) << 4);
        uint32_t* qp = reinterpret_cast<uint32_t*>(phq + off);
        uint32_t* kp = reinterpret_cast<uint32_t*>(phk + off);
        const uint32_t qv = *qp, kv = *kp;
        *qp = pack_bf16x2(__uint_as_float(qv << 16) * ex2_approx(r0),
                          __uint_as_float(qv & 0xffff0000u) * ex2_approx(r1));
        *kp = pack_bf16x2(__uint_as_float(kv << 16) * ex2_approx(-r0),
                          __uint_as_float(kv & 0xffff0000u) * ex2_approx(-r1));
      }
      if (c + 1 < nc) fetch(c + 1);
      // e^{+-b} must stay inside the fp32/bf16 range for the factorised form.
      if (big > kMaxLogSum * kLog2e) raise_status(p.status, kDevCheck);
      if (qt == 3) {
        if (u >= 1 && !(ok = wait_bar(ctl, B_EGFREE + s, (u - 1) & 1))) break;
        *reinterpret_cast<float2*>(eg + s * 128 + 2 * cp) = make_float2(ex2_approx(r0), ex2_approx(r1));
        mbar_arrive(&ctl->bar[B_EGFULL + s]);
      }
      fence_proxy_async_smem();
      mbar_arrive(&ctl->bar[B_OPND + s]);
    }
    if (!ok) ctl->abort = 1;
  } else if (warp < 14) {
    // ------------------------------------------------------------------ window softmax + epilogue
    const int qw = warp & 3;                 // TMEM lane quarter
    const int row = qw * 16 + lane;          // tile row (valid when lane < 16)
    const bool has_row = lane < 16;
    const uint32_t tq = tmem + ((uint32_t)(qw * 32) << 16);
    float rinv0 = 0.f, rinv1 = 0.f;          // alpha / row sum of P, by chunk parity
    bool ok = true;
    auto epilogue = [&](int c) -> bool {
      const int s = c & 1, u = c >> 1;
      if (!wait_bar(ctl, B_OFULL + s, u & 1)) return false;
      tc_fence_after();
      const int t = c * kC + row;
      const float r = s ? rinv1 : rinv0;
      uint4* dst = reinterpret_cast<uint4*>(p.y + ((size_t)bh * L + t) * kD + c0);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t o[16], ow[16];
        tmem_ld16(tq + G::TO + s * 32 + 16 * half, o);
        tmem_ld16(tq + G::TOW + s * 32 + 16 * half, ow);
        tmem_ld_wait();
        if (has_row && t < L) {
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            pk[i] = pack_bf16x2(fmaf(r, __uint_as_float(ow[2 * i]), __uint_as_float(o[2 * i])),
                                fmaf(r, __uint_as_float(ow[2 * i + 1]), __uint_as_float(o[2 * i + 1])));
          dst[2 * half] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          dst[2 * half + 1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
      tc_fence_before();
      mbar_arrive(&ctl->bar[B_OFREE + s]);
      return true;
    };
    // Z columns this warp's 16 rows can see: the meta block (columns 0..15) when M > 0,
    // then the 16-column groups [cb_lo, cb_hi] covering the window band.
    const int band_lo = max(16, 16 + kC * NP + 16 * qw - p.W + 1);
    const int band_hi = min(ZC - 1, 16 + kC * NP + 16 * qw + 15);
    const int cb_lo = band_lo & ~15, cb_hi = band_hi & ~15;
    const int nmeta = p.M > 0 ? 1 : 0;
    const int ngrp = nmeta + (cb_hi - cb_lo) / 16 + 1;  // 16-column groups to read
    const float zs = p.scale * kLog2e;
    for (int c = 0; c < nc && ok; ++c) {
      const int zb = c % NZ;
      const int t0 = c * kC;
      if (!(ok = wait_bar(ctl, B_SWFULL + zb, (c / NZ) & 1))) break;
      tc_fence_after();
      const uint32_t tz = tq + G::TZ + zb * ZC;
      // Visible columns of this row: [cmin, cmax] plus meta columns < M.
      const int i_abs = t0 + row;
      const int kbase = t0 - kC * NP;
      const int cmin = 16 + max(0, i_abs - p.W + 1) - kbase;
      const unsigned span = (unsigned)(i_abs - max(0, i_abs - p.W + 1));
      auto col_of = [&](int g) { return g < nmeta ? 0 : cb_lo + 16 * (g - nmeta); };
      auto visible = [&](int col, int i) {
        return col == 0 ? i < p.M : (unsigned)(col + i - cmin) <= span;
      };
      // pass 1: row max over the visible logits, two 16-column groups per TMEM wait
      float mx = -INFINITY;
      for (int g = 0; g < ngrp; g += 2) {
        uint32_t z0[16], z1[16];
        tmem_ld16(tz + col_of(g), z0);
        if (g + 1 < ngrp) tmem_ld16(tz + col_of(g + 1), z1);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (visible(col_of(g), i)) mx = fmaxf(mx, __uint_as_float(z0[i]));
          if (g + 1 < ngrp && visible(col_of(g + 1), i)) mx = fmaxf(mx, __uint_as_float(z1[i]));
        }
      }
      const float mxs = mx * zs;
      if (c >= NZ && !(ok = wait_bar(ctl, B_PFREE + zb, ((c / NZ) - 1) & 1))) break;
      unsigned char* pt = sm + G::PBUF + zb * (G::PATOMS * 8192);
      // columns outside the band and the meta block hold zero probability
      if (has_row) {
        for (int cb = 0; cb < ZC; cb += 16) {
          if ((cb == 0 && nmeta) || (cb >= cb_lo && cb <= cb_hi)) continue;
          *reinterpret_cast<uint4*>(pt + sw128_offset(row, cb, 64)) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(pt + sw128_offset(row, cb + 8, 64)) = make_uint4(0, 0, 0, 0);
        }
      }
      // pass 2: exponentials of the visible logits, written as the bf16 A operand
      float sum = 0.f;
      for (int g = 0; g < ngrp; g += 2) {
        uint32_t z[2][16];
        tmem_ld16(tz + col_of(g), z[0]);
        if (g + 1 < ngrp) tmem_ld16(tz + col_of(g + 1), z[1]);
        tmem_ld_wait();
#pragma unroll
        for (int gg = 0; gg < 2; ++gg) {
          if (g + gg >= ngrp) break;
          const int cb = col_of(g + gg);
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float e0 = visible(cb, 2 * i) ? ex2_approx(fmaf(__uint_as_float(z[gg][2 * i]), zs, -mxs)) : 0.f;
            const float e1 = visible(cb, 2 * i + 1) ? ex2_approx(fmaf(__uint_as_float(z[gg][2 * i + 1]), zs, -mxs)) : 0.f;
            w[i] = pack_bf16x2(e0, e1);
            sum += __uint_as_float(w[i] << 16) + __uint_as_float(w[i] & 0xffff0000u);
          }
          if (has_row) {
            *reinterpret_cast<uint4*>(pt + sw128_offset(row, cb, 64)) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(pt + sw128_offset(row, cb + 8, 64)) = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&ctl->bar[B_SWFREE + zb]);
      if (c & 1) rinv1 = p.alpha / sum;
      else rinv0 = p.alpha / sum;
      fence_proxy_async_smem();
      mbar_arrive(&ctl->bar[B_PREADY + zb]);
      if (c >= 1 && !(ok = epilogue(c - 1))) break;
    }
    if (ok && nc >= 1) ok = epilogue(nc - 1);
    if (!ok) ctl->abort = 1;
  } else {
    // ------------------------------------------------------------------ causal mask + state rescale
    const int qw = warp & 3;
    const int kk = qw * 32 + lane;  // TMEM lane = key dimension (state)
    const int row = qw * 16 + lane;  // tile row of S (valid when lane < 16)
    const bool has_row = lane < 16;
    const uint32_t tq = tmem + ((uint32_t)(qw * 32) << 16);
    const uint32_t th = tq + G::TH;
    unsigned char* hb = sm + G::HBF;
    unsigned char* sb = sm + G::SBF;
    auto store_h = [&](const uint32_t (&h)[32]) {
      // bf16 copy, MN-major 64-byte swizzle: row kk holds this slice's 32 columns.
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          w[i] = pack_bf16x2(__uint_as_float(h[ch * 8 + 2 * i]), __uint_as_float(h[ch * 8 + 2 * i + 1]));
        *reinterpret_cast<uint4*>(hb + sw64_offset(kk, ch * 8)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    };
    {
      uint32_t h[32];
#pragma unroll
      for (int i = 0; i < 32; ++i)
        h[i] = __float_as_uint(p.h0 ? p.h0[((size_t)bh * kD + kk) * kD + c0 + i] : 0.f);
      tmem_st32(th, h);
      tmem_st_wait();
      store_h(h);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&ctl->bar[B_HREADY]);
    }
    bool ok = true;
    for (int c = 0; c < nc && ok; ++c) {
      const int s = c & 1, u = c >> 1;
      // causal mask of S -> bf16 operand
      if (!(ok = wait_bar(ctl, B_SFULL, c & 1))) break;
      if (c >= 1 && !(ok = wait_bar(ctl, B_SBFFREE, (c - 1) & 1))) break;
      tc_fence_after();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t sv[32];
        tmem_ld32(tq + G::TS + 32 * half, sv);
        tmem_ld_wait();
        if (has_row) {
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int c1 = 32 * half + ch * 8 + 2 * i;
              w[i] = pack_bf16x2(c1 <= row ? __uint_as_float(sv[ch * 8 + 2 * i]) : 0.f,
                                 c1 + 1 <= row ? __uint_as_float(sv[ch * 8 + 2 * i + 1]) : 0.f);
            }
            *reinterpret_cast<uint4*>(sb + sw128_offset(row, 32 * half + ch * 8, 64)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&ctl->bar[B_SFREE]);
      fence_proxy_async_smem();
      mbar_arrive(&ctl->bar[B_SBFREADY]);
      // state rescale h <- diag(e^Gamma) h and its bf16 copy
      if (!(ok = wait_bar(ctl, B_HACC, c & 1))) break;
      if (!(ok = wait_bar(ctl, B_EGFULL + s, u & 1))) break;
      tc_fence_after();
      uint32_t h[32];
      tmem_ld32(th, h);
      tmem_ld_wait();
      const float g = eg[s * 128 + kk];
      mbar_arrive(&ctl->bar[B_EGFREE + s]);
#pragma unroll
      for (int i = 0; i < 32; ++i) h[i] = __float_as_uint(__uint_as_float(h[i]) * g);
      tmem_st32(th, h);
      tmem_st_wait();
      store_h(h);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&ctl->bar[B_HREADY]);
      if (c == nc - 1 && p.hf) {
#pragma unroll
        for (int i = 0; i < 32; ++i) p.hf[((size_t)bh * kD + kk) * kD + c0 + i] = __uint_as_float(h[i]);
      }
    }
    if (!ok) ctl->abort = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && ctl->abort) raise_status(p.status, kDevTimeout);
}

}  // namespace

// ------------------------------------------------------------------------------------
// host side: TMA descriptors
// ------------------------------------------------------------------------------------
namespace {
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled get_encode() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(ptr);
  });
  return fn;
}
}  // namespace

bool tma_encode_available() { return get_encode() != nullptr; }

bool make_tma_map_bf16(CUtensorMap* m, const void* base, uint64_t dim0, uint64_t dim1,
                       uint64_t dim2, uint32_t box0, uint32_t box1, CUtensorMapSwizzle sw) {
  EncodeTiled enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {dim0, dim1, dim2};
  cuuint64_t strides[2] = {dim0 * 2, dim0 * dim1 * 2};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
template <int NP>
cudaError_t launch_np(const Maps& maps, const Params& p, int grid, cudaStream_t s) {
  const size_t smem = Cfg<NP>::TOTAL;
  cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  trace_begin("fwd_tc", s);
  fwd_tc_kernel<NP><<<grid, kThreads, smem, s>>>(maps, p);
  trace_end(s);
  return cudaGetLastError();
}

}  // namespace

bool fwd_tc_supported(const FwdArgs& a, lizard_dtype dt) {
  return dt == LIZARD_BF16 && a.dk == kD && a.dv == kD && a.L > 0 && a.W <= 2 * kC + 1 &&
         a.M <= 16 && tma_encode_available();
}

cudaError_t launch_fwd_tc(const FwdArgs& a, cudaStream_t s, int* launches) {
  Maps maps;
  const uint64_t BH = (uint64_t)a.B * a.H, L = (uint64_t)a.L;
  bool ok = make_tma_map_bf16(&maps.phq, a.pq, kD, L, BH, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&maps.phk, a.pk, kD, L, BH, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&maps.q, a.q, kD, L, BH, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&maps.k, a.k, kD, L, BH, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tma_map_bf16(&maps.v, a.v, kD, L, BH, kNV, kC, CU_TENSOR_MAP_SWIZZLE_64B);
  if (a.M > 0) {
    ok = ok && make_tma_map_bf16(&maps.mk, a.mk, kD, a.M, a.H, 64, 16, CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_tma_map_bf16(&maps.mv, a.mv, kD, a.M, a.H, kNV, 16, CU_TENSOR_MAP_SWIZZLE_64B);
  } else {
    maps.mk = maps.phq;
    maps.mv = maps.v;
  }
  if (!ok) return cudaErrorInvalidValue;
  Params p;
  p.H = a.H;
  p.L = a.L;
  p.M = a.M;
  p.W = a.W;
  p.scale = a.scale;
  p.alpha = a.alpha;
  p.lg = a.lg;
  p.y = static_cast<bf16*>(a.y);
  p.h0 = a.h0;
  p.hf = a.hf;
  p.status = a.status;
  const int grid = (int)(BH * kSlices);
  cudaError_t e = a.W <= kC + 1 ? launch_np<1>(maps, p, grid, s) : launch_np<2>(maps, p, grid, s);
  ++*launches;
  return e;
}

}  // namespace lz
