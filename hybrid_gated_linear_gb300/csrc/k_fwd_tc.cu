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
//   Z  = q [meta_k ; k_{chunk-Np..chunk}]^T   M=64 N=16+64(Np+1) K=128 (tcgen05)
//   P  = exp(scale (Z - rowmax)) on the visible keys, 0 elsewhere  (CUDA cores)
//   Ow = P [meta_v ; v]                        M=64 N=32              (tcgen05)
//   y  = O + alpha * Ow / rowsum(P), rounded to bf16 once.
// All operands arrive by TMA (3D maps over [B*H, L, d]; rows outside [0, L) read as
// zeros), accumulate in fp32 in TMEM, and every wait is bounded in time: on a timeout
// the CTA records LIZARD_ERR_TIMEOUT in the status word and returns cleanly.
//
// Warp roles (14 warps): 0 TMA producer; 1 MMA issuer + TMEM owner; 2-5 feature
// transform (thread = key dimension); 6-9 row work on the M=64 tiles (mask, window
// softmax, epilogue; rows 16w..16w+15 sit in lanes 0-15 of warp w%4's TMEM quarter);
// 10-13 state rescale (thread = key dimension, all 128 TMEM lanes).
#include <mutex>

#include "lizard_dev.cuh"
#include "lizard_internal.h"
#include "tc_sm100.cuh"

namespace lz {
namespace {

using namespace tc;

constexpr int kC = 64;          // chunk
constexpr int kD = 128;         // dk = dv
constexpr int kNV = 32;         // dv columns per CTA
constexpr int kSlices = kD / kNV;
constexpr int kThreads = 14 * 32;
constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s per wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaxLogSum = 80.f;  // |chunk-local log-gate sum| beyond which e^{+-b} overflows

// TMEM columns.
constexpr uint32_t kTS = 0;      // S, 2 x 64
constexpr uint32_t kTO = 128;    // O, 2 x 32
constexpr uint32_t kTOW = 192;   // Ow, 2 x 32
constexpr uint32_t kTH = 256;    // h, 32
constexpr uint32_t kTZ = 288;    // Z, up to 16 + 64*3 = 208
constexpr uint32_t kTmemCols = 512;

struct Params {
  int BH, H, L, M, W;
  int np;      // previous chunks the window reaches (1 or 2)
  int nr;      // k/v ring slots = np + 2
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

// Shared-memory plan (byte offsets from a 1024-aligned base).
struct Smem {
  static constexpr uint32_t kStage = 2 * 16384;            // phi_q, phi_k tiles
  static constexpr uint32_t kStages = 0;                    // 2 stages
  static constexpr uint32_t kQ = kStages + 2 * kStage;      // q tile 16 KB
  static constexpr uint32_t kKring = kQ + 16384;            // nr x 16 KB
  __host__ __device__ static uint32_t vring(int nr) { return kKring + nr * 16384u; }
  __host__ __device__ static uint32_t metak(int nr) { return vring(nr) + nr * 4096u; }
  __host__ __device__ static uint32_t metav(int nr) { return metak(nr) + 4096u; }
  __host__ __device__ static uint32_t sbf(int nr) { return metav(nr) + 1024u; }
  __host__ __device__ static uint32_t pbuf(int nr) { return sbf(nr) + 8192u; }
  __host__ __device__ static uint32_t hbf(int nr) { return pbuf(nr) + (uint32_t)nr * 8192u; }
  __host__ __device__ static uint32_t eg(int nr) { return hbf(nr) + 8192u; }
  __host__ __device__ static uint32_t rinv(int nr) { return eg(nr) + 2 * 512u; }
  __host__ __device__ static uint32_t bars(int nr) { return rinv(nr) + 2 * 256u; }
  __host__ __device__ static uint32_t total(int nr) { return bars(nr) + 1024u + 1024u; }
};

// Barrier indices.
enum {
  B_FULL = 0, B_EMPTY = 2, B_OPND = 4, B_SFULL = 6, B_SFREE = 8, B_OFULL = 10, B_OFREE = 12,
  B_EGFULL = 14, B_EGFREE = 16, B_QFULL = 18, B_QEMPTY, B_META, B_SWFULL, B_SWFREE, B_SBFREADY,
  B_SBFFREE, B_PREADY, B_PFREE, B_HACC, B_HREADY, B_MMADONE, B_KVFULL /* 4 */,
  B_KVEMPTY = B_KVFULL + 4, B_COUNT = B_KVEMPTY + 4
};

struct Ctl {
  uint64_t bar[B_COUNT];
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ bool wait_bar(Ctl* ctl, int i, uint32_t parity) {
  uint64_t* b = &ctl->bar[i];
  if (mbar_try_wait(b, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(b, parity)) return true;
    if (*(volatile int*)&ctl->abort) return false;
    if (globaltimer_ns() - t0 > kWaitNs) {
      *(volatile int*)&ctl->abort = 1;
      return false;
    }
  }
}

// K-major SW128 operand descriptor for k-step j (16 elements) of a tile with `rows` rows.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int rows, int j) {
  return smem_desc(base + (uint32_t)((j * 16) >> 6) * rows * 128u + (uint32_t)((j * 16) & 63) * 2u,
                   16, 1024, kSw128);
}

__global__ void __launch_bounds__(kThreads, 1)
fwd_tc_kernel(const __grid_constant__ Maps maps, const Params p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int nr = p.nr, np = p.np;
  Ctl* ctl = reinterpret_cast<Ctl*>(sm + Smem::bars(nr));
  float* eg = reinterpret_cast<float*>(sm + Smem::eg(nr));
  float* rinv_s = reinterpret_cast<float*>(sm + Smem::rinv(nr));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x / kSlices;
  const int slice = blockIdx.x % kSlices;
  const int c0 = slice * kNV;
  const int hh = bh % p.H;
  const int L = p.L;
  const int nc = (L + kC - 1) / kC;
  const int nkeys_cols = 16 + kC * (np + 1);  // columns of Z

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      uint32_t cnt = 1;
      if (i == B_OPND || i == B_OPND + 1 || i == B_SFREE || i == B_SFREE + 1 || i == B_OFREE ||
          i == B_OFREE + 1 || i == B_EGFULL || i == B_EGFULL + 1 || i == B_EGFREE ||
          i == B_EGFREE + 1 || i == B_SWFREE || i == B_SBFREADY || i == B_PREADY ||
          i == B_HREADY)
        cnt = 128;
      mbar_init(&ctl->bar[i], cnt);
    }
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&maps.phq);
      tma_prefetch_desc(&maps.k);
      uint32_t armed_full[2] = {0, 0}, armed_kv[4] = {0, 0, 0, 0}, armed_q = 0;
      bool ok = true;
      if (p.M > 0) {
        mbar_arrive_expect_tx(&ctl->bar[B_META], 4096 + 1024);
        tma_load_3d(sm + Smem::metak(nr), &maps.mk, 0, 0, hh, &ctl->bar[B_META]);
        tma_load_3d(sm + Smem::metak(nr) + 2048, &maps.mk, 64, 0, hh, &ctl->bar[B_META]);
        tma_load_3d(sm + Smem::metav(nr), &maps.mv, c0, 0, hh, &ctl->bar[B_META]);
      } else {
        mbar_arrive(&ctl->bar[B_META]);
      }
      auto load_kv = [&](int j) -> bool {
        const int u = j + np, r = u % nr;
        if (u >= nr && !wait_bar(ctl, B_KVEMPTY + r, ((u / nr) - 1) & 1)) return false;
        mbar_arrive_expect_tx(&ctl->bar[B_KVFULL + r], 16384 + 4096);
        unsigned char* kd = sm + Smem::kKring + r * 16384;
        tma_load_3d(kd, &maps.k, 0, j * kC, bh, &ctl->bar[B_KVFULL + r]);
        tma_load_3d(kd + 8192, &maps.k, 64, j * kC, bh, &ctl->bar[B_KVFULL + r]);
        tma_load_3d(sm + Smem::vring(nr) + r * 4096, &maps.v, c0, j * kC, bh,
                    &ctl->bar[B_KVFULL + r]);
        ++armed_kv[r];
        return true;
      };
      for (int j = -np; j < 0 && ok; ++j) ok = load_kv(j);
      for (int c = 0; c < nc && ok; ++c) {
        ok = load_kv(c);
        if (!ok) break;
        const int s = c & 1, u = c >> 1;
        if (u >= 1 && !(ok = wait_bar(ctl, B_EMPTY + s, (u - 1) & 1))) break;
        mbar_arrive_expect_tx(&ctl->bar[B_FULL + s], 32768);
        unsigned char* st = sm + Smem::kStages + s * Smem::kStage;
        tma_load_3d(st, &maps.phq, 0, c * kC, bh, &ctl->bar[B_FULL + s]);
        tma_load_3d(st + 8192, &maps.phq, 64, c * kC, bh, &ctl->bar[B_FULL + s]);
        tma_load_3d(st + 16384, &maps.phk, 0, c * kC, bh, &ctl->bar[B_FULL + s]);
        tma_load_3d(st + 24576, &maps.phk, 64, c * kC, bh, &ctl->bar[B_FULL + s]);
        ++armed_full[s];
        if (c >= 1 && !(ok = wait_bar(ctl, B_QEMPTY, (c - 1) & 1))) break;
        mbar_arrive_expect_tx(&ctl->bar[B_QFULL], 16384);
        tma_load_3d(sm + Smem::kQ, &maps.q, 0, c * kC, bh, &ctl->bar[B_QFULL]);
        tma_load_3d(sm + Smem::kQ + 8192, &maps.q, 64, c * kC, bh, &ctl->bar[B_QFULL]);
        ++armed_q;
      }
      // Never leave with copies in flight: wait for the last armed phase of each barrier.
      ctl->abort |= ok ? 0 : 1;
      const uint64_t t0 = globaltimer_ns();
      auto drain = [&](int i, uint32_t armed) {
        if (armed == 0) return;
        while (!mbar_try_wait(&ctl->bar[i], (armed - 1) & 1))
          if (globaltimer_ns() - t0 > kWaitNs) break;
      };
      for (int s = 0; s < 2; ++s) drain(B_FULL + s, armed_full[s]);
      for (int r = 0; r < nr; ++r) drain(B_KVFULL + r, armed_kv[r]);
      drain(B_QFULL, armed_q);
      drain(B_META, p.M > 0 ? 1 : 0);
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
      for (int c = 0; c < nc && ok; ++c) {
        const int s = c & 1, u = c >> 1;
        const int slot = (c + np) % nr;
        const uint32_t phq = sbase + Smem::kStages + s * Smem::kStage;
        const uint32_t phk = phq + 16384;
        const uint32_t ts = tmem + kTS + s * 64, to = tmem + kTO + s * 32,
                       tow = tmem + kTOW + s * 32;
        if (!(ok = wait_bar(ctl, B_OPND + s, u & 1))) break;
        if (!(ok = wait_bar(ctl, B_KVFULL + slot, ((c + np) / nr) & 1))) break;
        if (u >= 1 && !(ok = wait_bar(ctl, B_SFREE + s, (u - 1) & 1))) break;
        tc_fence_after();
        // S = Qt Kt^T
        for (int j = 0; j < 8; ++j)
          mma_bf16(ts, desc_kmajor(phq, 64, j), desc_kmajor(phk, 64, j), id_s, j > 0);
        mma_commit(&ctl->bar[B_SFULL + s]);
        // Z = q [meta_k ; k_prev.. ; k_cur]^T
        if (!(ok = wait_bar(ctl, B_QFULL, c & 1))) break;
        if (c >= 1 && !(ok = wait_bar(ctl, B_SWFREE, (c - 1) & 1))) break;
        tc_fence_after();
        if (c == 0) {
          for (int jn = -np; jn < 0 && ok; ++jn) ok = wait_bar(ctl, B_KVFULL + (jn + np) % nr, 0);
          if (!ok) break;
          tc_fence_after();
        }
        const uint32_t qb = sbase + Smem::kQ;
        if (p.M > 0) {
          for (int j = 0; j < 8; ++j)
            mma_bf16(tmem + kTZ, desc_kmajor(qb, 64, j),
                     desc_kmajor(sbase + Smem::metak(nr), 16, j), id_z16, j > 0);
        }
        for (int b = 0; b <= np; ++b) {
          const int r = (c - np + b + np) % nr;
          const uint32_t kb = sbase + Smem::kKring + r * 16384;
          for (int j = 0; j < 8; ++j)
            mma_bf16(tmem + kTZ + 16 + 64 * b, desc_kmajor(qb, 64, j), desc_kmajor(kb, 64, j),
                     id_z64, j > 0);
        }
        mma_commit(&ctl->bar[B_SWFULL]);
        mma_commit(&ctl->bar[B_QEMPTY]);
        // O = Qt h ; h += Kt^T V
        if (!(ok = wait_bar(ctl, B_HREADY, c & 1))) break;
        if (u >= 1 && !(ok = wait_bar(ctl, B_OFREE + s, (u - 1) & 1))) break;
        tc_fence_after();
        const uint32_t hb = sbase + Smem::hbf(nr);
        for (int j = 0; j < 8; ++j)
          mma_bf16(to, desc_kmajor(phq, 64, j), smem_desc(hb + j * 1024, 8192, 512, kSw64), id_o,
                   j > 0);
        const uint32_t vb = sbase + Smem::vring(nr) + slot * 4096;
        for (int j = 0; j < 4; ++j)
          mma_bf16(tmem + kTH, smem_desc(phk + j * 2048, 8192, 1024, kSw128),
                   smem_desc(vb + j * 1024, 4096, 512, kSw64), id_h, true);
        mma_commit(&ctl->bar[B_HACC]);
        // O += mask(S) V
        if (!(ok = wait_bar(ctl, B_SBFREADY, c & 1))) break;
        tc_fence_after();
        const uint32_t sbf = sbase + Smem::sbf(nr);
        for (int j = 0; j < 4; ++j)
          mma_bf16(to, desc_kmajor(sbf, 64, j), smem_desc(vb + j * 1024, 4096, 512, kSw64), id_o,
                   true);
        mma_commit(&ctl->bar[B_SBFFREE]);
        mma_commit(&ctl->bar[B_EMPTY + s]);
        // Ow = P [meta_v ; v_prev.. ; v_cur]
        if (!(ok = wait_bar(ctl, B_PREADY, c & 1))) break;
        tc_fence_after();
        const uint32_t pb = sbase + Smem::pbuf(nr);
        // meta block: P columns 0..15 (k-step 0 of atom 0), V rows = meta_v tile
        if (p.M > 0)
          mma_bf16(tow, desc_kmajor(pb, 64, 0),
                   smem_desc(sbase + Smem::metav(nr), 1024, 512, kSw64), id_o, false);
        for (int b = 0; b <= np; ++b) {
          const int r = (c - np + b + np) % nr;
          const uint32_t vv = sbase + Smem::vring(nr) + r * 4096;
          for (int j = 0; j < 4; ++j)
            mma_bf16(tow, desc_kmajor(pb, 64, 1 + b * 4 + j),
                     smem_desc(vv + j * 1024, 4096, 512, kSw64), id_o, p.M > 0 || b > 0 || j > 0);
        }
        mma_commit(&ctl->bar[B_PFREE]);
        mma_commit(&ctl->bar[B_OFULL + s]);
        mma_commit(&ctl->bar[B_KVEMPTY + (c + np - np) % nr]);
      }
      if (!ok) ctl->abort = 1;
      mma_commit(&ctl->bar[B_MMADONE]);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&ctl->bar[B_MMADONE], 0))
        if (globaltimer_ns() - t0 > kWaitNs) break;
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------------ transform
    const int kk = threadIdx.x - 64;  // key dimension 0..127
    const float* lg = p.lg + (size_t)bh * L * kD + kk;
    bool ok = true;
    for (int c = 0; c < nc && ok; ++c) {
      const int s = c & 1, u = c >> 1;
      const int t0 = c * kC, n = min(kC, L - t0);
      if (!(ok = wait_bar(ctl, B_FULL + s, u & 1))) break;
      if (u >= 1 && !(ok = wait_bar(ctl, B_EGFREE + s, (u - 1) & 1))) break;
      unsigned char* phq = sm + Smem::kStages + s * Smem::kStage;
      unsigned char* phk = phq + 16384;
      float run = 0.f, big = 0.f;
      float lgv[8];
      for (int t8 = 0; t8 < kC; t8 += 8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) lgv[i] = (t8 + i < n) ? lg[(size_t)(t0 + t8 + i) * kD] : 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int t = t8 + i;
          run += lgv[i];
          big = fmaxf(big, fabsf(run));
          const float e = exp2f(run * kLog2e);
          const float ei = exp2f(-run * kLog2e);
          const uint32_t off = sw128_offset(t, kk, 64);
          bf16* q = reinterpret_cast<bf16*>(phq + off);
          bf16* k = reinterpret_cast<bf16*>(phk + off);
          *q = __float2bfloat16_rn(__bfloat162float(*q) * e);
          *k = __float2bfloat16_rn(__bfloat162float(*k) * ei);
        }
      }
      eg[s * 128 + kk] = exp2f(run * kLog2e);
      // e^{+-b} must stay inside the fp32/bf16 range for the factorised form.
      if (big > kMaxLogSum) raise_status(p.status, kDevCheck);
      fence_proxy_async_smem();
      mbar_arrive(&ctl->bar[B_OPND + s]);
      mbar_arrive(&ctl->bar[B_EGFULL + s]);
    }
    if (!ok) ctl->abort = 1;
  } else if (warp < 10) {
    // ------------------------------------------------------------------ row work (M = 64)
    const int qw = warp & 3;                      // TMEM lane quarter
    const int row = qw * 16 + lane;               // tile row (valid when lane < 16)
    const bool has_row = lane < 16;
    const uint32_t tq = tmem + ((uint32_t)(qw * 32) << 16);
    bool ok = true;
    auto epilogue = [&](int c) -> bool {
      const int s = c & 1, u = c >> 1;
      if (!wait_bar(ctl, B_OFULL + s, u & 1)) return false;
      tc_fence_after();
      uint32_t o[32], ow[32];
      tmem_ld32(tq + kTO + s * 32, o);
      tmem_ld32(tq + kTOW + s * 32, ow);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&ctl->bar[B_OFREE + s]);
      const int t = c * kC + row;
      if (has_row && t < L) {
        const float r = rinv_s[s * 64 + row];
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) + r * __uint_as_float(ow[2 * i]),
                              __uint_as_float(o[2 * i + 1]) + r * __uint_as_float(ow[2 * i + 1]));
        uint4* dst = reinterpret_cast<uint4*>(p.y + ((size_t)bh * L + t) * kD + c0);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
      return true;
    };
    for (int c = 0; c < nc && ok; ++c) {
      const int s = c & 1, u = c >> 1;
      const int t0 = c * kC;
      // (a) causal mask of S -> bf16 operand
      if (!(ok = wait_bar(ctl, B_SFULL + s, u & 1))) break;
      tc_fence_after();
      if (c >= 1 && !(ok = wait_bar(ctl, B_SBFFREE, (c - 1) & 1))) break;
      {
        unsigned char* sb = sm + Smem::sbf(nr);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t sv[32];
          tmem_ld32(tq + kTS + s * 64 + 32 * half, sv);
          tmem_ld_wait();
          if (has_row) {
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
              uint32_t w[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int c1 = 32 * half + ch * 8 + 2 * i, c2 = c1 + 1;
                const float x1 = c1 <= row ? __uint_as_float(sv[ch * 8 + 2 * i]) : 0.f;
                const float x2 = c2 <= row ? __uint_as_float(sv[ch * 8 + 2 * i + 1]) : 0.f;
                w[i] = pack_bf16x2(x1, x2);
              }
              *reinterpret_cast<uint4*>(sb + sw128_offset(row, 32 * half + ch * 8, 64)) =
                  make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&ctl->bar[B_SFREE + s]);
      fence_proxy_async_smem();
      mbar_arrive(&ctl->bar[B_SBFREADY]);
      // epilogue of the previous chunk overlaps the next MMAs
      if (c >= 1 && !(ok = epilogue(c - 1))) break;
      // (b) window softmax: P = exp(scale (z - max)) on visible keys
      if (!(ok = wait_bar(ctl, B_SWFULL, c & 1))) break;
      tc_fence_after();
      const int i_abs = t0 + row;
      const int jlo = max(0, i_abs - p.W + 1);
      const int kbase = t0 - kC * np;  // key index of Z column 16
      const float zs = p.scale * kLog2e;
      float mx = -INFINITY;
      for (int cb = 0; cb < nkeys_cols; cb += 16) {
        uint32_t z[32];
        tmem_ld32(tq + kTZ + cb, z);  // reads 32 columns; only 16 are used per step
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int col = cb + i;
          const int j = kbase + col - 16;
          const bool vis = col < 16 ? col < p.M : (j >= jlo && j <= i_abs);
          if (vis) mx = fmaxf(mx, __uint_as_float(z[i]));
        }
      }
      if (c >= 1 && !(ok = wait_bar(ctl, B_PFREE, (c - 1) & 1))) break;
      float sum = 0.f;
      unsigned char* pb = sm + Smem::pbuf(nr);
      for (int cb = 0; cb < nkeys_cols; cb += 16) {
        uint32_t z[32];
        tmem_ld32(tq + kTZ + cb, z);
        tmem_ld_wait();
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float e2[2];
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int col = cb + 2 * i + h2;
            const int j = kbase + col - 16;
            const bool vis = col < 16 ? col < p.M : (j >= jlo && j <= i_abs);
            e2[h2] = vis ? exp2f((__uint_as_float(z[2 * i + h2]) - mx) * zs) : 0.f;
          }
          w[i] = pack_bf16x2(e2[0], e2[1]);
          sum += __uint_as_float(w[i] << 16) + __uint_as_float(w[i] & 0xffff0000u);
        }
        if (has_row) {
          *reinterpret_cast<uint4*>(pb + sw128_offset(row, cb, 64)) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(pb + sw128_offset(row, cb + 8, 64)) = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
      tc_fence_before();
      mbar_arrive(&ctl->bar[B_SWFREE]);
      if (has_row) rinv_s[s * 64 + row] = p.alpha / sum;
      fence_proxy_async_smem();
      mbar_arrive(&ctl->bar[B_PREADY]);
    }
    if (ok && nc >= 1) ok = epilogue(nc - 1);
    if (!ok) ctl->abort = 1;
  } else {
    // ------------------------------------------------------------------ state rescale
    const int qw = warp & 3;
    const int kk = qw * 32 + lane;  // TMEM lane = key dimension
    const uint32_t th = tmem + ((uint32_t)(qw * 32) << 16) + kTH;
    unsigned char* hb = sm + Smem::hbf(nr);
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
    if (nc == 0 && p.hf) {
      for (int i = 0; i < 32; ++i)
        p.hf[((size_t)bh * kD + kk) * kD + c0 + i] = p.h0 ? p.h0[((size_t)bh * kD + kk) * kD + c0 + i] : 0.f;
    }
    if (!ok) ctl->abort = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && ctl->abort) raise_status(p.status, kDevTimeout);
}

// ------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------
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

// 3D bf16 map over [dim2][dim1][dim0] (dim0 contiguous) with a box {box0, box1, 1}.
bool make_map(CUtensorMap* m, const void* base, uint64_t dim0, uint64_t dim1, uint64_t dim2,
              uint32_t box0, uint32_t box1, CUtensorMapSwizzle sw) {
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

}  // namespace

bool fwd_tc_supported(const FwdArgs& a, lizard_dtype dt) {
  return dt == LIZARD_BF16 && a.dk == kD && a.dv == kD && a.L > 0 && a.W <= 2 * kC + 1 &&
         a.M <= 16 && get_encode() != nullptr;
}

cudaError_t launch_fwd_tc(const FwdArgs& a, cudaStream_t s, int* launches) {
  Maps maps;
  const uint64_t BH = (uint64_t)a.B * a.H, L = (uint64_t)a.L;
  bool ok = make_map(&maps.phq, a.pq, kD, L, BH, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&maps.phk, a.pk, kD, L, BH, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&maps.q, a.q, kD, L, BH, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&maps.k, a.k, kD, L, BH, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&maps.v, a.v, kD, L, BH, kNV, kC, CU_TENSOR_MAP_SWIZZLE_64B);
  if (a.M > 0) {
    ok = ok && make_map(&maps.mk, a.mk, kD, a.M, a.H, 64, 16, CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map(&maps.mv, a.mv, kD, a.M, a.H, kNV, 16, CU_TENSOR_MAP_SWIZZLE_64B);
  } else {
    maps.mk = maps.phq;
    maps.mv = maps.v;
  }
  if (!ok) return cudaErrorInvalidValue;
  Params p;
  p.BH = (int)BH;
  p.H = a.H;
  p.L = a.L;
  p.M = a.M;
  p.W = a.W;
  p.np = a.W <= kC + 1 ? 1 : 2;
  p.nr = p.np + 2;
  p.scale = a.scale;
  p.alpha = a.alpha;
  p.lg = a.lg;
  p.y = static_cast<bf16*>(a.y);
  p.h0 = a.h0;
  p.hf = a.hf;
  p.status = a.status;
  const size_t smem = Smem::total(p.nr);
  cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  trace_begin("fwd_tc", s);
  fwd_tc_kernel<<<(unsigned)(BH * kSlices), kThreads, smem, s>>>(maps, p);
  trace_end(s);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace lz
