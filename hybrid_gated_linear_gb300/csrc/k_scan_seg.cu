// k_scan_seg.cu -- joining the segments of a split state scan.
//
// When the (b, h) units are too few to fill the GPU, the state scan of k_gla_states_tc.cu
// cuts each unit's chunks into segments and scans them in parallel, each from zero.  The
// segments are then joined with the associative combine of the recurrence ("Lizard", arXiv 2507.09025, Preliminaries:
// recurrent form): a segment with summed log gate G and state F from a zero start maps an
// incoming state H to diag(e^G) H + F.
//   states (forward):    H_0 = h0 (or 0), H_{s+1} = diag(e^{G_s}) H_s + F_s, h_final = H_nseg
//   adjoints (reverse):  R_last = 0, R_{s-1} = diag(e^{G_s}) R_s + F_s,   d h0 = R_{-1}
// and every chunk's stored state gets the incoming state carried to it:
//   h_c  += diag(e^{sum of Gamma over the segment's chunks before c}) H_s
//   Gt_c += diag(e^{sum of Gamma over chunks c .. segment end}) R_s
// (Gt_c = diag(e^{Gamma_c}) G_c is what the adjoint scan stores; for a chunk flagged wide it
// stores G_c itself, and the sum starts at chunk c + 1).  All sums run in chunk
// order, so the result does not depend on scheduling.
#include "lizard_dev.cuh"
#include "lizard_internal.h"

namespace lz {
namespace {

constexpr int kD = 128;
constexpr int kS = kD * kD;

// One thread per (unit, row k, four columns): the 32 threads of a row form one warp.  The
// segments are walked in order, in batches of kJB: a batch's gate sums and partial states
// do not depend on the running state, so all of their loads are issued before the walk
// uses any of them.  The gate sum of segment s over its chunks [c0, c1) is split over
// the 32 lanes (lane j adds c0 + j, c0 + j + 32, ... in that order) and reduced in a
// fixed butterfly order.
constexpr int kJB = 8;

__global__ void __launch_bounds__(256) seg_join_kernel(int nc, int nseg, int cps, int dir,
                                                       const float* __restrict__ gam,
                                                       const float* __restrict__ segf,
                                                       float* __restrict__ segh,
                                                       const float* __restrict__ h0,
                                                       float* __restrict__ fin) {
  const int bh = blockIdx.y, e = blockIdx.x * blockDim.x + threadIdx.x;
  const int k = e >> 5, v = (e & 31) * 4, lane = threadIdx.x & 31;
  pdl_wait();
  const size_t un = (size_t)bh * nseg, off = (size_t)k * kD + v;
  const float* gk = gam + (size_t)bh * nc * kD + k;  // gam of chunk c, row k: gk[c * kD]
  float4 H = make_float4(0.f, 0.f, 0.f, 0.f);
  if (dir == 0 && h0) H = *reinterpret_cast<const float4*>(h0 + (size_t)bh * kS + off);
  for (int t0 = 0; t0 < nseg; t0 += kJB) {
    float G[kJB];
    float4 F[kJB];
#pragma unroll
    for (int b = 0; b < kJB; ++b) {
      const int t = t0 + b;
      const int s = dir ? nseg - 1 - t : t;
      const int c0 = s * cps, c1 = min(nc, c0 + cps);
      const bool live = t < nseg;
      // the first two chunks of each lane as straight-line loads, the rest in a loop
      const int ca = c0 + lane, cb = ca + 32;
      const float va = live && ca < c1 ? gk[(size_t)ca * kD] : 0.f;
      const float vb = live && cb < c1 ? gk[(size_t)cb * kD] : 0.f;
      F[b] = live ? *reinterpret_cast<const float4*>(segf + (un + s) * kS + off)
                  : make_float4(0.f, 0.f, 0.f, 0.f);
      float acc = va + vb;
      if (live)
        for (int c = cb + 32; c < c1; c += 32) acc += gk[(size_t)c * kD];
      G[b] = acc;
    }
#pragma unroll
    for (int b = 0; b < kJB; ++b) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) G[b] += __shfl_xor_sync(0xffffffffu, G[b], o);
    }
#pragma unroll
    for (int b = 0; b < kJB; ++b) {
      const int t = t0 + b;
      if (t < nseg) {
        const int s = dir ? nseg - 1 - t : t;
        *reinterpret_cast<float4*>(segh + (un + s) * kS + off) = H;
        const float f = expf(G[b]);
        H = make_float4(fmaf(f, H.x, F[b].x), fmaf(f, H.y, F[b].y), fmaf(f, H.z, F[b].z),
                        fmaf(f, H.w, F[b].w));
      }
    }
  }
  if (fin) *reinterpret_cast<float4*>(fin + (size_t)bh * kS + off) = H;
  pdl_trigger();
}

// One CTA per (chunk, unit): the decay from the segment boundary to the chunk for every
// row, then the stored bf16 state updated eight elements per thread and step.
__global__ void __launch_bounds__(256) seg_fix_kernel(int nc, int nseg, int cps, int dir,
                                                      int with_h0, const float* __restrict__ gam,
                                                      const int* __restrict__ wide,
                                                      const float* __restrict__ segh,
                                                      bf16* __restrict__ st) {
  const int c = blockIdx.x, bh = blockIdx.y, s = c / cps;
  __shared__ float f[kD];
  pdl_wait();
  if ((dir == 0 && s == 0 && !with_h0) || (dir == 1 && s == nseg - 1)) {
    pdl_trigger();
    return;  // the incoming state is zero
  }
  if (threadIdx.x < kD) {
    // one row per thread: with a CTA per chunk, the many CTAs on an SM hide these sums'
    // load latency (the pass is bound by reading and writing the states)
    const int k = threadIdx.x;
    const int c0 = dir == 0 ? s * cps : c + (wide[(size_t)bh * nc + c] ? 1 : 0);
    const int c1 = dir == 0 ? c : min(nc, (s + 1) * cps);
    float B = 0.f;
    for (int c2 = c0; c2 < c1; ++c2) B += gam[((size_t)bh * nc + c2) * kD + k];
    f[k] = expf(B);
  }
  __syncthreads();
  const float* H = segh + ((size_t)bh * nseg + s) * kS;
  bf16* dst = st + ((size_t)bh * nc + c) * kS;
  for (int e8 = threadIdx.x; e8 < kS / 8; e8 += blockDim.x) {
    const int k = e8 >> 4, v = (e8 & 15) * 8;
    const size_t off = (size_t)k * kD + v;
    uint4 raw = *reinterpret_cast<const uint4*>(dst + off);
    const float4 h_lo = *reinterpret_cast<const float4*>(H + off);
    const float4 h_hi = *reinterpret_cast<const float4*>(H + off + 4);
    const float hv[8] = {h_lo.x, h_lo.y, h_lo.z, h_lo.w, h_hi.x, h_hi.y, h_hi.z, h_hi.w};
    uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    const float fk = f[k];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float a = __uint_as_float(w[q] << 16), b = __uint_as_float(w[q] & 0xffff0000u);
      const __nv_bfloat162 o = __floats2bfloat162_rn(fmaf(fk, hv[2 * q], a), fmaf(fk, hv[2 * q + 1], b));
      w[q] = *reinterpret_cast<const uint32_t*>(&o);
    }
    *reinterpret_cast<uint4*>(dst + off) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  pdl_trigger();
}

}  // namespace

int gla_seg_cap(int BH, int nc) {
  const int cap = min(nc / kSegMinChunks, kSegMaxCtas / max(1, BH * (kD / 32)));
  return cap >= 2 ? cap : 1;
}

size_t gla_seg_scratch(int BH, int L) {
  const int nc = (L + kGlaChunk - 1) / kGlaChunk;
  const int cap = gla_seg_cap(BH, nc);
  if (cap < 2) return 0;
  return (size_t)2 * 2 * BH * cap * kS * sizeof(float);  // (F, H) for each direction
}

int gla_scan_segments(int BH, int nc, int ndir) {
  const int cap = gla_seg_cap(BH, nc);
  const int fit = ctas_per_wave(1) / max(1, BH * (kD / 32) * ndir);
  const int n = min(cap, fit);
  return n >= 2 ? n : 1;
}

cudaError_t launch_seg_join(int BH, int nc, int nseg, int cps, int dir, const float* gam,
                            float* seg, int cap, const float* h0, float* fin, cudaStream_t s,
                            int* launches) {
  float* segf = seg + (size_t)dir * 2 * BH * cap * kS;
  float* segh = segf + (size_t)BH * cap * kS;
  trace_begin("scan_join", s);
  cudaError_t e = launch_pdl(seg_join_kernel, dim3(kS / 4 / 256, BH), dim3(256), 0, s, nc, nseg,
                             cps, dir, gam, static_cast<const float*>(segf), segh, h0, fin);
  trace_end(s);
  ++*launches;
  return e;
}

cudaError_t launch_seg_fix(int BH, int nc, int nseg, int cps, int dir, const float* gam,
                           const int* wide, float* seg, int cap, bf16* st, bool with_h0,
                           cudaStream_t s, int* launches) {
  const float* segh = seg + (size_t)dir * 2 * BH * cap * kS + (size_t)BH * cap * kS;
  trace_begin("scan_fix", s);
  cudaError_t e = launch_pdl(seg_fix_kernel, dim3(nc, BH), dim3(256), 0, s, nc, nseg, cps, dir,
                             with_h0 ? 1 : 0, gam, wide, segh, st);
  trace_end(s);
  ++*launches;
  return e;
}

}  // namespace lz
