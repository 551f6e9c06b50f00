// lizard_internal.h -- shared declarations of the CUDA library (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>

#include "lizard.h"

namespace lz {

using bf16 = __nv_bfloat16;

// Device status word bits (first word of every workspace).
enum : unsigned { kDevTimeout = 1u, kDevCheck = 2u };

// Every workspace starts with this many bytes: the status word, then zero padding.
constexpr size_t kWsHeader = 256;
// Word of the header that counts the tensor-core path's wide chunks (zeroed per call).
constexpr int kWsWideCount = 4;
// Words of the header that hand out the window-backward query blocks: the block counter
// and the count of CTAs done; zero at every call (the header is cleared) and left at zero
// by every launch that completes.
constexpr int kWsWinTiles = 8;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Arguments of one forward call after validation (device pointers).
struct FwdArgs {
  int B, H, L, dk, dv, M, W;
  float scale, alpha;
  const void *pq, *pk, *v;
  const float* lg;
  const void *q, *k, *mk, *mv;
  void* y;
  const float* h0;
  float* hf;
  unsigned* status;
  unsigned char* ws;  // workspace after the header
  // Set instead of pq/pk when the forward starts from the raw projections and the
  // Hedgehog feature map (x [B,H,L,128] bf16, one W [128,64] bf16 per head).
  const void *xq = nullptr, *xk = nullptr, *wq = nullptr, *wk = nullptr;
  // Counter of the tensor-core path's wide chunks, zero before the call (null: word
  // kWsWideCount of the status header).  A backward that reuses this forward's context
  // reads it at word kWsWideCount of the header in front of the forward's scratch.
  unsigned* wcount = nullptr;
};

struct BwdArgs {
  int B, H, L, dk, dv, M, W;
  float scale, alpha;
  const void *pq, *pk, *v;
  const float* lg;
  const void *q, *k, *mk, *mv;
  const float* h0;
  const void* dy;
  void *dpq, *dpk, *dvv;
  float* dlg;
  void *dq, *dk_;
  float *dmk, *dmv, *dh0;
  unsigned* status;
  unsigned char* ws;  // workspace after the header
  size_t ws_bytes;
  unsigned char* fwd_ws;  // forward workspace after its header (reused context) or null
};

struct DecArgs {
  int N, H, dk, dv, M, W;
  float scale, alpha;
  const void *pq, *pk, *v;
  const float* lg;
  const void *q, *k, *mk, *mv;
  float* h;
  void *kr, *vr;
  int64_t* pos;
  void* y;
  unsigned* counters;  // N zero-initialised words
  unsigned* status;
};

// The value lizard_last_launch_count returns on this host thread (set by every entry point).
void set_last_launches(int n);

// Optional per-kernel event tracing (no-ops unless enabled on this host thread).
void trace_begin(const char* name, cudaStream_t s);
void trace_end(cudaStream_t s);

// TMA descriptors (driver entry point resolved once per process).
bool tma_encode_available();
// 3D bf16 tensor map over [dim2][dim1][dim0] (dim0 contiguous), box {box0, box1, 1}; rows
// outside the tensor read as zeros.
bool make_tma_map_bf16(CUtensorMap* m, const void* base, uint64_t dim0, uint64_t dim1,
                       uint64_t dim2, uint32_t box0, uint32_t box1, CUtensorMapSwizzle sw);
// Same for fp32 elements.
bool make_tma_map_f32(CUtensorMap* m, const void* base, uint64_t dim0, uint64_t dim1,
                      uint64_t dim2, uint32_t box0, uint32_t box1, CUtensorMapSwizzle sw);

// Launches `kernel` on `s` with programmatic stream serialisation, so that its CTAs may
// start (and run up to pdl_wait) while the previous kernel on the stream drains.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Number of SMs of the current device times `per_sm` (cached per device).
int ctas_per_wave(int per_sm);

// Launchers: return the first CUDA error and add the number of kernels they enqueued
// to *launches.
cudaError_t launch_chunk_cumsum(int units, int L, int dk, int chunk, const float* lg, float* b,
                                float* gamma_chunk, cudaStream_t s, int* launches);
cudaError_t launch_fwd_simt(const FwdArgs& a, lizard_dtype dt, cudaStream_t s, int* launches);
// Chunk-parallel tensor-core forward (bf16, dk = dv = 128, L > 0, 1 <= W <= 129,
// M <= 16); scratch of fwd_chunk_tc_workspace(B*H, L) bytes at a.ws.
bool fwd_chunk_tc_supported(int dk, int dv, int L, int W, int M, lizard_dtype dt);
size_t fwd_chunk_tc_workspace(int BH, int L);
cudaError_t launch_fwd_chunk_tc(const FwdArgs& a, unsigned char* ws, cudaStream_t s, int* launches);
// Chunk length of the chunk-parallel tensor-core GLA kernels.
constexpr int kGlaChunk = 128;

// Inputs and outputs of the two passes the chunk-parallel GLA kernels start from
// (k_gla_states_tc.cu); bf16, dk = dv = 128.  qt, kt, eb [BH][L][128] bf16 (eb may be
// null), gam [BH][nc][128] fp32, hs / gs [BH][nc][128][128] bf16 with nc = ceil(L/128);
// h0 may be null (zeros); hf (h_final) and dh0 may be null.
struct GlaStatesArgs {
  int BH, L;
  const void *pq, *pk;
  const float* lg;
  const void *v, *dy;
  const float* h0;
  float *hf, *dh0;
  bf16 *qt, *kt, *eb;
  float* gam;
  bf16 *hs, *gs;
  unsigned* status;
  // gla_seg_scratch bytes for a split scan (null: never split)
  float* seg = nullptr;
  // Wide chunks (the gate factorisation e^{+b} e^{-b} out of range): flags [BH][nc]
  // (1 = wide), the list of their indices bh * nc + c, and its length.
  int* wide = nullptr;
  int* wlist = nullptr;
  unsigned* wcount = nullptr;
};

// The exact recomputation of the wide chunks after the tensor-core kernels: the listed
// chunks, their chunk-start states hs (and, backward, the unscaled end-of-chunk adjoints
// gs) [BH][nc][128][128] bf16.  The forward writes the listed chunks' phi_q, phi_k into
// phq, phk ([BH][L][128] bf16: the context's e^b and Kt sections, which the chunk
// kernels no longer need for those chunks); a backward from that context reads them
// back there (phq_in, phk_in), otherwise from its phi_q, phi_k inputs.
struct WideFix {
  const unsigned* count;
  const int* list;
  int nc;
  const bf16* hs;
  const bf16* gs = nullptr;
  bf16 *phq = nullptr, *phk = nullptr;
  const bf16 *phq_in = nullptr, *phk_in = nullptr;
  float* rtot = nullptr;  // backward: per-chunk totals of the log-gate term [BH][nc][128]
  float* scratch = nullptr;  // backward: bwd_wide_scratch_bytes of walk scratch
};
// CTAs of the backward's wide-chunk recomputation (each with its own walk scratch), and
// the scratch they need.
constexpr int kWideCtas = 32;
int bwd_wide_ctas(int BH, int nc);
size_t bwd_wide_scratch_bytes(int BH, int nc);
cudaError_t launch_fwd_wide_fix(const FwdArgs& a, const WideFix& w, cudaStream_t s, int* launches);
cudaError_t launch_bwd_wide_fix(const BwdArgs& a, const WideFix& w, float* dvacc, cudaStream_t s,
                                int* launches);
cudaError_t launch_gla_prep(const GlaStatesArgs& a, cudaStream_t s, int* launches);
// The prep pass fused with the Hedgehog feature map (k_prep_fmap_tc.cu): the same Qt, Kt,
// e^b and Gamma from x_q, x_k [BH][L][128] and per-head W_q, W_k [H][128][64] (bf16), as
// exp(+-x W_q + b) and exp(+-x W_k - b); needs a.qt, a.kt, a.eb, a.gam, a.lg.
cudaError_t launch_gla_prep_fmap(const GlaStatesArgs& a, int H, const void* xq, const void* xk,
                                 const void* wq, const void* wk, cudaStream_t s, int* launches);
// Sequence split of the scans (k_scan_seg.cu): when the B*H units leave most SMs idle,
// each unit's chunks are cut into segments scanned in parallel from zero and then joined.
constexpr int kSegMinChunks = 8;  // chunks per segment at least
constexpr int kSegMaxCtas = 256;  // bound on the CTAs of one scan wave, for sizing scratch
int gla_seg_cap(int BH, int nc);                // segments the scratch is sized for (1: none)
size_t gla_seg_scratch(int BH, int L);          // bytes, 0 when never split
int gla_scan_segments(int BH, int nc, int ndir);  // segments to use on this device (1: none)
cudaError_t launch_seg_join(int BH, int nc, int nseg, int cps, int dir, const float* gam,
                            float* seg, int cap, const float* h0, float* fin, cudaStream_t s,
                            int* launches);
cudaError_t launch_seg_fix(int BH, int nc, int nseg, int cps, int dir, const float* gam,
                           const int* wide, float* seg, int cap, bf16* st, bool with_h0,
                           cudaStream_t s, int* launches);
// Which scans: the chunk-start states h_c, the scaled adjoints Gt_c, or both.
enum class GlaScan { kStates, kAdjoints, kBoth };
cudaError_t launch_gla_scan(const GlaStatesArgs& a, GlaScan which, cudaStream_t s, int* launches);

// What the chunk-parallel forward leaves in its workspace for the backward: Qt, Kt, e^b,
// Gamma and the chunk-start states h_c (see GlaStatesArgs for the layouts).
struct GlaCtx {
  bf16 *qt, *kt, *eb;
  float* gam;
  bf16* hs;
  float* seg = nullptr;  // scratch of a split scan (not part of the reused context)
  int* wide = nullptr;   // wide-chunk flags [BH][nc] and list [BH][nc]
  int* wlist = nullptr;
};
// The context inside a forward workspace (after its header) of B*H units of L tokens.
GlaCtx fwd_chunk_tc_ctx(int BH, int L, unsigned char* ws);

// Tensor-core backward of the GLA branch (bf16, dk = dv = 128, L > 0): writes d_phi_q,
// d_phi_k, d_log_gamma, d_h0 and the GLA part of dv (fp32 [B*H][L][128]) to dvacc, using
// bwd_gla_tc_workspace(B*H, L) bytes of scratch at ws (256-byte aligned).
bool bwd_gla_tc_supported(int dk, int dv, int L, lizard_dtype dt);
size_t bwd_gla_tc_workspace(int BH, int L);
cudaError_t launch_bwd_gla_tc(const BwdArgs& a, float* dvacc, unsigned char* ws, cudaStream_t s,
                              int* launches);
// True when the forward of these dims used the chunk-parallel tensor-core path, so that its
// workspace holds a GlaCtx the tensor-core GLA backward can reuse.
bool fwd_ctx_usable(int dk, int dv, int L, int W, int M, lizard_dtype dt);
// Tensor-core backward of the window branch (bf16, dk = dv = 128, 1 <= W <= 65, M <= 16,
// L > 0): writes d_q, d_k, d_v (adding the GLA part from dvacc), d_meta_k, d_meta_v; uses
// lse2/Dw ([B*H][L] fp32) and mpart (bwd_win_tc_meta_floats) as scratch.
bool bwd_win_tc_supported(int dk, int dv, int L, int W, int M, lizard_dtype dt);
size_t bwd_win_tc_meta_floats(int BH, int L, int M);
// The query half (dq, row statistics, meta partials), the ordered sum of the meta partials
// into d_meta_k / d_meta_v, and the key half (dk, dv with the GLA part from dvacc); the
// meta sum and the key half need the query half's outputs.
cudaError_t launch_bwd_win_q_tc(const BwdArgs& a, const float* dvacc, float* lse2, float* Dw,
                                float* mpart, cudaStream_t s, int* launches);
cudaError_t launch_bwd_win_k_tc(const BwdArgs& a, const float* dvacc, float* lse2, float* Dw,
                                float* mpart, cudaStream_t s, int* launches);
cudaError_t launch_bwd_win_meta_tc(const BwdArgs& a, const float* mpart, cudaStream_t s,
                                   int* launches);

// A second stream of the current device with a fork and a join event, for work that may
// run beside the caller's stream inside one call; enqueue under side_stream_lock().
struct SideStream {
  cudaStream_t stream;
  cudaEvent_t fork, join, done;
};
SideStream* side_stream();
std::mutex& side_stream_lock();
size_t bwd_simt_workspace(int B, int H, int L, int dk, int dv, int M);
cudaError_t launch_bwd_simt(const BwdArgs& a, lizard_dtype dt, cudaStream_t s, int* launches);
cudaError_t launch_decode(const DecArgs& a, lizard_dtype dt, cudaStream_t s, int* launches);
// Segment-state combine and the prefill -> decode ring fill (k_state.cu).
// Hedgehog feature map (k_fmap.cu).
bool fmap_tc_supported(int D, int F, lizard_dtype dt);
bool fmap_simt_supported(int D, int F);
size_t fmap_bwd_workspace(int B, int H, int L, int D, int F, lizard_dtype dt);
cudaError_t launch_fmap_fwd(int B, int H, int L, int D, int F, lizard_dtype dt, const void* x,
                            const void* w, void* phi, unsigned* status, cudaStream_t s,
                            int* launches);
cudaError_t launch_fmap_bwd(int B, int H, int L, int D, int F, lizard_dtype dt, const void* x,
                            const void* w, const void* dphi, void* dx, float* dw,
                            unsigned char* ws, unsigned* status, cudaStream_t s, int* launches);

// Gate projection log gamma = logsigmoid(x W) / tau and its backward (k_gate.cu).
size_t gate_bwd_workspace(int B, int H, int L, int D, int dk);
// The standard (fp32, CUDA-core) chunkwise GLA forward used as the comparison point
// (k_gla_std.cu).
size_t gla_std_workspace(int BH, int L, int D);
cudaError_t launch_gla_std_fwd(int BH, int L, int D, lizard_dtype dt, const void* pq,
                               const void* pk, const void* v, const float* lg, const float* h0,
                               float* hf, void* y, unsigned* status, unsigned char* ws,
                               cudaStream_t s, int* launches);

cudaError_t launch_gate_fwd(int B, int H, int L, int D, int dk, lizard_dtype dt, float tau,
                            const void* x, const void* w, float* lg, cudaStream_t s, int* launches);
cudaError_t launch_gate_bwd(int B, int H, int L, int D, int dk, lizard_dtype dt, float tau,
                            const void* x, const void* w, const float* dlg, void* dx, float* dw,
                            unsigned char* ws, cudaStream_t s, int* launches);

cudaError_t launch_state_combine(int units, int dk, int dv, const float* ga, const float* ha,
                                 const float* gb, const float* hb, float* go, float* ho,
                                 cudaStream_t s, int* launches);
cudaError_t launch_ring_fill(int N, int H, int L, int W, int dk, int dv, lizard_dtype dt,
                             const void* k, const void* v, void* kr, void* vr, int64_t* pos,
                             cudaStream_t s, int* launches);

}  // namespace lz
