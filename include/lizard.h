/*
 * lizard.h -- C ABI of the GB300 (sm_103a) Lizard-attention library.
 *
 * The operator (sources cited per call below):
 *   GLA branch     h_i = gamma_i (.) h_{i-1} + phi_k_i v_i^T,   y_gla_i = phi_q_i^T h_i
 *                  with gamma_i = exp(log_gamma_i) per key dimension, scaling the rows of
 *                  h (the key dimension).  ["Lizard: An Efficient Linearization Framework
 *                  for Large Language Models", papernotes.org note, 方法详解/关键设计:
 *                  GLA replacing RoPE; arXiv 2507.09025, Method: parallel GLA form]
 *   Window branch  y_win_i = softmax(scale * [q_i.meta_k ; q_i.k_j]) [meta_v ; v_j] over the
 *                  M meta tokens and the W tokens j in [max(0, i-W+1), i].
 *                  [papernotes.org note, 关键设计: Anchor Window Attention]
 *   Merge          y = y_gla + alpha * y_win.  [papernotes.org note, 整体框架]
 *
 * Conventions shared by every call:
 *   - Device pointers only (unless stated), caller-owned; the library never allocates,
 *     frees or keeps a pointer after the call returns.  Buffers must stay alive until the
 *     work queued on `stream` has finished.
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy default stream.
 *     Every call is asynchronous: it validates arguments on the host, enqueues kernels
 *     and returns; only lizard_check_device_errors synchronises.
 *   - Per-token tensors are contiguous row-major [B,H,L,d] ("BHLD"); meta tensors are
 *     [H,M,d] (one set per head, shared by every batch entry); states are [B,H,dk,dv]
 *     fp32 with dk the row (gated) dimension.
 *   - "T" tensors (phi_q, phi_k, v, q, k, meta_k, meta_v, y, dy, d_phi_q, d_phi_k, d_v,
 *     d_q, d_k) have the element type `dtype` (fp32 or bf16); log_gamma, states and
 *     d_log_gamma, d_meta_* are always fp32.  Accumulation is fp32 throughout.
 *   - The raw q/k of the window branch have dimension dk (same as phi_q/phi_k).
 *   - Every pointer must be 16-byte aligned.  Outputs must not alias inputs (the decode
 *     state h, rings and pos are in-out by design).
 *   - Errors: invalid arguments return a status before anything is enqueued; a failed
 *     launch returns LIZARD_ERR_CUDA; conditions found on the device (a bounded wait that
 *     ran out, a range guard) set a word in the workspace that
 *     lizard_check_device_errors reads.  Nothing throws across this boundary.
 */
#ifndef LIZARD_H
#define LIZARD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LIZARD_ABI_VERSION 2

typedef enum lizard_status {
    LIZARD_OK = 0,
    LIZARD_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, aliasing */
    LIZARD_ERR_UNSUPPORTED = 2,   /* valid but not built (e.g. head dim not 64/128) */
    LIZARD_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    LIZARD_ERR_TIMEOUT = 4,       /* a device-side bounded wait ran out (device word) */
    LIZARD_ERR_DEVICE_CHECK = 5,  /* a device-side guard fired (device word) */
    LIZARD_ERR_WORKSPACE = 6      /* workspace missing or smaller than required */
} lizard_status;

typedef enum lizard_dtype { LIZARD_F32 = 0, LIZARD_BF16 = 1 } lizard_dtype;

/* Shape of a forward/backward call. */
typedef struct lizard_dims {
    int32_t B;            /* batch, >= 1 */
    int32_t H;            /* heads, >= 1 */
    int32_t L;            /* tokens, >= 0 (0 is a no-op apart from h_final) */
    int32_t dk;           /* key/query dim: 64 or 128 */
    int32_t dv;           /* value dim: equal to dk */
    int32_t M;            /* meta tokens per head, 0..16 */
    lizard_dtype dtype;   /* element type of the "T" tensors */
    float scale;          /* window softmax scale; <= 0 selects 1/sqrt(dk) */
} lizard_dims;

/* Shape of one decode step: N sequences, one new token each. */
typedef struct lizard_decode_dims {
    int32_t N, H, dk, dv, M;
    lizard_dtype dtype;
    float scale;
} lizard_decode_dims;

/* Device-workspace bytes each call needs (0 means workspace may be NULL). */
size_t lizard_fwd_workspace_bytes(const lizard_dims* dims, int32_t W);
size_t lizard_bwd_workspace_bytes(const lizard_dims* dims, int32_t W);
size_t lizard_decode_workspace_bytes(const lizard_decode_dims* dims);

/*
 * Forward pass: y = y_gla + alpha * y_win.
 *   phi_q, phi_k, q, k [B,H,L,dk] T;  v [B,H,L,dv] T;  log_gamma [B,H,L,dk] fp32 (<= 0
 *   expected; any finite value is accepted);  meta_k [H,M,dk], meta_v [H,M,dv] T (NULL
 *   when M = 0);  W >= 1 window length (keys including self; the backward needs
 *   min(W, L) <= 4096, else LIZARD_ERR_UNSUPPORTED);  alpha any finite value.
 *   y [B,H,L,dv] T output.  h0 [B,H,dk,dv] fp32 initial state or NULL (zeros).
 *   h_final [B,H,dk,dv] fp32 final state or NULL.
 * The GLA branch is computed chunkwise with the decay products absorbed in log space
 * into the query/key features ("Lizard", arXiv 2507.09025, Method: hardware-aware
 * reparameterisation); the result equals the recurrence up to rounding.  Every finite
 * log_gamma <= 0 gives a finite result: a 128-token chunk whose cumulative log gate
 * leaves [-80, 80] (where e^{-b} would overflow) is recomputed exactly by the recurrence
 * on CUDA cores, so strong gates cost time, not accuracy.
 */
lizard_status lizard_attn_fwd(const lizard_dims* dims, const void* phi_q, const void* phi_k,
                              const void* v, const float* log_gamma, const void* q,
                              const void* k, const void* meta_k, const void* meta_v,
                              int32_t W, float alpha, void* y, const float* h0,
                              float* h_final, void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * Forward pass started from the raw projections, with the Hedgehog feature map fused into
 * the log-space absorption of the gate ("Lizard", arXiv 2507.09025, Method: phi(x) =
 * [exp(xW) (+) exp(-xW)], the cumulative gate absorbed into the query and key features):
 * the query and key features of the chunkwise form are computed directly as
 * exp(+-x_q W_q + b) and exp(+-x_k W_k - b) (b the chunk-local cumulative log gate), so
 * phi is never written.  The result is lizard_attn_fwd with
 *   phi_q = [exp(x_q W_q), exp(-x_q W_q)],  phi_k = [exp(x_k W_k), exp(-x_k W_k)]
 * (the map of lizard_feature_map_fwd) up to rounding.
 *   x_q, x_k [B,H,L,128] bf16; w_q, w_k [H,128,64] bf16 (W[h][d][f]); every other argument
 *   as in lizard_attn_fwd.  Only bf16 with dk = dv = 128, W <= 129 and M <= 16 (the
 *   tensor-core forward); other shapes return LIZARD_ERR_UNSUPPORTED -- call
 *   lizard_feature_map_fwd and lizard_attn_fwd instead.  The workspace is
 *   lizard_fwd_workspace_bytes(dims, W); it holds the same saved context as
 *   lizard_attn_fwd's, so lizard_attn_bwd(..., phi_q = NULL, phi_k = NULL, ...,
 *   fwd_workspace = this workspace) returns d_phi_q, d_phi_k, from which
 *   lizard_feature_map_bwd gives the gradients of x_q, x_k, W_q, W_k.  Chunks whose
 *   log-gate range is too wide for the factorised form are recomputed exactly, as in
 *   lizard_attn_fwd (their phi is formed there in fp32 from x and W).
 */
lizard_status lizard_attn_fwd_fmap(const lizard_dims* dims, const void* x_q, const void* x_k,
                                   const void* w_q, const void* w_k, const void* v,
                                   const float* log_gamma, const void* q, const void* k,
                                   const void* meta_k, const void* meta_v, int32_t W,
                                   float alpha, void* y, const float* h0, float* h_final,
                                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward pass of lizard_attn_fwd for the loss sum(y * dy).
 *   Inputs as in lizard_attn_fwd plus dy [B,H,L,dv] T.
 *   Outputs: d_phi_q, d_phi_k, d_q, d_k [B,H,L,dk] T; d_v [B,H,L,dv] T (GLA + window);
 *   d_log_gamma [B,H,L,dk] fp32; d_meta_k [H,M,dk], d_meta_v [H,M,dv] fp32, summed over
 *   batch and tokens (NULL when M = 0); d_h0 [B,H,dk,dv] fp32 or NULL.
 * fwd_workspace: NULL, or the workspace of the lizard_attn_fwd call this backward belongs
 *   to (same dims and W, same phi_q, phi_k, v, log_gamma and h0, unchanged since).  The
 *   forward's workspace then holds the chunk features and chunk-start states, which the
 *   backward reuses instead of recomputing them; a forward that did not leave them (other
 *   shapes or dtypes) is detected from dims and W and the pointer is then ignored.
 *   Passing a workspace that does not match these conditions gives wrong gradients.
 *   When that context is used (bf16, dk = dv = 128, a forward on the tensor-core path:
 *   W <= 129 and M <= 16), phi_q and phi_k are not read and may be NULL -- the case of a
 *   forward started from lizard_attn_fwd_fmap, which never forms phi.  Otherwise NULL
 *   phi_q / phi_k with L > 0 is LIZARD_ERR_INVALID_ARG.
 * The pages give no backward formulas; this is the exact adjoint of the forward.  The
 * log-gate gradient uses d log_gamma_t = sum_{t'>=t} (phi_q (.) d_phi_q - phi_k (.) d_phi_k)_{t'}
 * (exact because the gate enters only through its cumulative sums).  Deterministic:
 * no floating-point atomics.
 */
lizard_status lizard_attn_bwd(const lizard_dims* dims, const void* phi_q, const void* phi_k,
                              const void* v, const float* log_gamma, const void* q,
                              const void* k, const void* meta_k, const void* meta_v,
                              int32_t W, float alpha, const float* h0, const void* dy,
                              void* d_phi_q, void* d_phi_k, void* d_v, float* d_log_gamma,
                              void* d_q, void* d_k, float* d_meta_k, float* d_meta_v,
                              float* d_h0, const void* fwd_workspace, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * Forward and backward of one training step with every tensor in HOST memory.
 *   Arguments as lizard_attn_fwd followed by lizard_attn_bwd (same shapes, types and
 *   optional pointers), except that phi_q ... dy, y, h_final and all gradients are host
 *   pointers.  Page-locked (pinned) host memory lets the copies run concurrently with the
 *   kernels; pageable memory works, with serialised copies.  `workspace` is DEVICE memory
 *   of lizard_fwd_bwd_host_workspace_bytes(dims, W) bytes.
 * The heads are processed in slices of up to ceil(H/8) (the first and the last narrower, to
 * shorten the pipeline's fill and drain): while slice s is computed on `stream`,
 * the inputs of slice s+1 are copied in and the results of slice s-1 copied out on two
 * streams of the library's own (created once per device), ordered after the work already
 * queued on `stream`; before returning, the call makes `stream` wait for the last copy,
 * so synchronising `stream` covers the whole step.  Host buffers must stay valid and
 * unchanged until then.  Results are identical to the two device calls.  Device
 * conditions are reported through lizard_check_device_errors(workspace, stream).
 */
size_t lizard_fwd_bwd_host_workspace_bytes(const lizard_dims* dims, int32_t W);
lizard_status lizard_attn_fwd_bwd_host(const lizard_dims* dims, const void* phi_q,
                                       const void* phi_k, const void* v, const float* log_gamma,
                                       const void* q, const void* k, const void* meta_k,
                                       const void* meta_v, int32_t W, float alpha,
                                       const float* h0, const void* dy, void* y, float* h_final,
                                       void* d_phi_q, void* d_phi_k, void* d_v,
                                       float* d_log_gamma, void* d_q, void* d_k, float* d_meta_k,
                                       float* d_meta_v, float* d_h0, void* workspace,
                                       size_t workspace_bytes, void* stream);

/*
 * One recurrent decode step for N sequences (constant memory per sequence: the state
 * and a W-slot ring; "Lizard", arXiv 2507.09025, Preliminaries: recurrent form).
 *   Token inputs phi_q, phi_k, q, k [N,H,dk] T; v [N,H,dv] T; log_gamma [N,H,dk] fp32.
 *   meta_k [H,M,dk], meta_v [H,M,dv] T.  W >= 1 ring length (= window length).
 *   In-out: h [N,H,dk,dv] fp32; k_ring [N,H,W,dk] T; v_ring [N,H,W,dv] T; pos [N] int64
 *   (device) = absolute position of the new token, >= 0.
 *   Per sequence n at position p = pos[n]: h <- gamma (.) h + phi_k v^T; y_gla = phi_q^T h;
 *   ring slot p mod W <- (k, v); y_win = softmax over the M meta tokens and the
 *   min(p+1, W) tokens [max(0, p-W+1), p]; y = y_gla + alpha * y_win; pos[n] <- p + 1.
 *   y [N,H,dv] T output.
 * Workspace: lizard_decode_workspace_bytes(dims) bytes that must be zero-filled before
 * the first step (lizard_workspace_init does that); each step leaves it zeroed again.
 * A workspace must not be shared by steps that run concurrently.
 */
lizard_status lizard_decode_step(const lizard_decode_dims* dims, const void* phi_q,
                                 const void* phi_k, const void* v, const float* log_gamma,
                                 const void* q, const void* k, const void* meta_k,
                                 const void* meta_v, int32_t W, float alpha, float* h,
                                 void* k_ring, void* v_ring, int64_t* pos, void* y,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Allocation-free decode step (the paper has no counterpart; this is a library service).
 * For callers that cannot allocate device memory: a host program or language binding
 * that embeds this library without a device allocator of its own, or a serving runtime
 * whose memory pool owns all device memory and may not call cudaMalloc on the per-token
 * path.  Same arguments and results as lizard_decode_step, without the workspace: the
 * per-sequence counters live in a fixed device array inside the library (a little over
 * 64 KiB, held on every GPU that uses it until the process exits), so N is limited to
 * LIZARD_NOALLOC_MAX_SEQUENCES; a larger N returns LIZARD_ERR_UNSUPPORTED before anything
 * is enqueued.  The first call on each device looks up the array's address on the
 * current device; make that first call before any stream capture begins.  Each call
 * clears the counters on `stream` before its kernel.  Every call in the process shares
 * the one array, so calls whose work overlaps on the GPU (other streams, other threads)
 * race on it: order them.  These calls report no device status word; their kernels are
 * counted by lizard_last_launch_count like every other call's.  Nothing is allocated or
 * freed.
 */
#define LIZARD_NOALLOC_MAX_SEQUENCES 16384
lizard_status lizard_decode_step_noalloc(const lizard_decode_dims* dims, const void* phi_q,
                                         const void* phi_k, const void* v,
                                         const float* log_gamma, const void* q, const void* k,
                                         const void* meta_k, const void* meta_v, int32_t W,
                                         float alpha, float* h, void* k_ring, void* v_ring,
                                         int64_t* pos, void* y, void* stream);

/*
 * Prefill -> decode handoff: fills the decode rings after a prefill of L tokens.
 *   k [N,H,L,dk], v [N,H,L,dv] T: the raw window keys and values of the prefill (device;
 *   NULL allowed when L = 0).  Out: k_ring [N,H,W,dk], v_ring [N,H,W,dv] T with slot
 *   t mod W holding token t for t in [max(0, L-W), L) and zeros elsewhere; pos [N] int64
 *   set to L.  With the state h = h_final of lizard_attn_fwd over the same prefill (its
 *   [B,H,dk,dv] layout is the decode state's [N,H,dk,dv] with N = B), the next
 *   lizard_decode_step continues the sequence exactly where the prefill stopped.
 *   ("Lizard", arXiv 2507.09025, Preliminaries: recurrent form; papernotes.org note,
 *   关键设计: Anchor Window Attention.)
 */
lizard_status lizard_decode_ring_fill(const lizard_decode_dims* dims, int32_t L, int32_t W,
                                      const void* k, const void* v, void* k_ring, void* v_ring,
                                      int64_t* pos, void* stream);

/*
 * Associative combine of segment states for a sequence split ("Lizard", arXiv 2507.09025,
 * Preliminaries: recurrent form).  A segment with log-gate sum Gamma [dk] and final state
 * h [dk,dv] from a zero start maps an initial state h0 to diag(e^Gamma) h0 + h, so
 *   (Gamma_a, h_a) o (Gamma_b, h_b) = (Gamma_a + Gamma_b, diag(e^Gamma_b) h_a + h_b)
 * for segment a followed by segment b.  units independent pairs; gamma_* [units,dk] fp32,
 * h_* [units,dk,dv] fp32 (device); dv a multiple of 4; gamma_out may be NULL.  h_out may
 * be h_a or h_b (in place); gamma_out must not overlap gamma_a or gamma_b.  Segment sums
 * come from lizard_chunk_cumsum (chunk = segment length) and segment states from
 * lizard_attn_fwd (h0 = NULL, h_final); the combined state is the h0 of the next segment.
 */
lizard_status lizard_state_combine(int32_t units, int32_t dk, int32_t dv, const float* gamma_a,
                                   const float* h_a, const float* gamma_b, const float* h_b,
                                   float* gamma_out, float* h_out, void* stream);

/*
 * Hedgehog feature map of one projection and its backward ("Lizard", arXiv 2507.09025,
 * Method: the strictly non-negative map phi(x) = [exp(x W) (+) exp(-x W)] whose
 * exponential form admits the log-space reparameterisation).  Per (b, h, token):
 *   z = x W[h]  (F values),   phi = [exp(z_0..z_{F-1}), exp(-z_0..-z_{F-1})]  (2F values).
 * x [B,H,L,D] T, W [H,D,F] T (one matrix per head, row-major: W[h][d][f]),
 * phi [B,H,L,2F] T.  The outputs phi are what lizard_attn_fwd takes as phi_q / phi_k
 * (2F = dk).  D in 1..256, F in 1..128, D*F <= 16384; bf16 with D = 128, F = 64 runs on
 * tensor cores (fp32 accumulation, bf16 phi), everything else on CUDA cores in fp32.
 * L = 0 is a no-op (the backward then zero-fills d_w).
 * Backward, with dphi+ / dphi- the first / last F features of d_phi [B,H,L,2F] T:
 *   dz = dphi+ exp(z) - dphi- exp(-z),  d_x = dz W^T  [B,H,L,D] T,
 *   d_w[h] = sum over b and tokens of x^T dz  [H,D,F] fp32, summed in a fixed order
 *   (run-to-run identical).
 * Workspace: lizard_feature_map_workspace_bytes (is_bwd 0 or 1); its first word is the
 * device status word read by lizard_check_device_errors.  Outputs must not overlap
 * inputs or the workspace.
 */
typedef struct lizard_fmap_dims {
    int32_t B, H, L;      /* batch, heads, tokens (L >= 0) */
    int32_t D;            /* input features per head */
    int32_t F;            /* columns of W; phi has 2F features */
    lizard_dtype dtype;   /* element type of x, W, phi, d_phi, d_x */
} lizard_fmap_dims;

size_t lizard_feature_map_workspace_bytes(const lizard_fmap_dims* dims, int32_t is_bwd);
lizard_status lizard_feature_map_fwd(const lizard_fmap_dims* dims, const void* x, const void* w,
                                     void* phi, void* workspace, size_t workspace_bytes,
                                     void* stream);
lizard_status lizard_feature_map_bwd(const lizard_fmap_dims* dims, const void* x, const void* w,
                                     const void* d_phi, void* d_x, float* d_w, void* workspace,
                                     size_t workspace_bytes, void* stream);

/*
 * Chunk-local inclusive cumulative sum of log gamma (the reference point of the
 * log-space reparameterisation; "Lizard", arXiv 2507.09025, Method: cumulative gate
 * products c_t).  log_gamma [units,L,dk] fp32 -> b [units,L,dk] fp32 with
 * b_t = sum_{s = chunk start..t} log_gamma_s, chunks [c*chunk, min((c+1)*chunk, L));
 * gamma_chunk [units, ceil(L/chunk), dk] fp32 = b at each chunk's last token (nullable).
 * dk in 1..1024, chunk in 1..1024.
 */
lizard_status lizard_chunk_cumsum(int32_t units, int32_t L, int32_t dk, int32_t chunk,
                                  const float* log_gamma, float* b, float* gamma_chunk,
                                  void* stream);

/* Zero-fills a workspace on `stream` (asynchronous). */
lizard_status lizard_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Synchronises `stream`, then reads and clears the device status word in `workspace`.
 * Returns LIZARD_OK, LIZARD_ERR_TIMEOUT or LIZARD_ERR_DEVICE_CHECK (or LIZARD_ERR_CUDA if
 * the stream itself reports an error).
 */
lizard_status lizard_check_device_errors(void* workspace, void* stream);

/*
 * Gate projection in front of the operator ("Lizard", arXiv 2507.09025, Method: the gate
 * projection W_gamma is trained; papernotes.org note, 关键设计: gamma_i is computed by
 * W_gamma).  The pages fix neither the projection's input nor its nonlinearity; this
 * library takes the form of the workloads' gates:
 *   log_gamma[b,h,t,k] = logsigmoid( sum_d x[b,h,t,d] W[h,d,k] ) / tau
 * so every gamma lies in (0, 1); tau > 0 is a temperature (tau <= 0 selects 16).
 *   x [B,H,L,D] T (D in 1..256); w [H,D,dk] T (dk = 64 or 128); log_gamma [B,H,L,dk]
 *   fp32 output, the operator's log_gamma input.
 * The backward takes d_log_gamma [B,H,L,dk] fp32 (from lizard_attn_bwd) and returns
 *   d_x [B,H,L,D] T and d_w [H,D,dk] fp32, the latter summed over batch and tokens in a
 *   fixed order (run-to-run identical); its workspace is lizard_gate_workspace_bytes
 *   (caller-owned, 16-byte aligned; the forward needs none and may pass NULL, 0).
 * CUDA cores, fp32 arithmetic.
 */
typedef struct lizard_gate_dims {
    int32_t B, H, L;      /* batch, heads, tokens (L >= 0) */
    int32_t D;            /* input features, 1..256 */
    int32_t dk;           /* key dimension: 64 or 128 */
    lizard_dtype dtype;   /* element type of x, w, d_x */
    float tau;            /* temperature; <= 0 selects 16 */
} lizard_gate_dims;
size_t lizard_gate_workspace_bytes(const lizard_gate_dims* dims);
lizard_status lizard_gate_fwd(const lizard_gate_dims* dims, const void* x, const void* w,
                              float* log_gamma, void* stream);
lizard_status lizard_gate_bwd(const lizard_gate_dims* dims, const void* x, const void* w,
                              const float* d_log_gamma, void* d_x, float* d_w, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * The "standard" chunkwise GLA forward, the comparison point of the hardware-aware kernel
 * (not part of the Lizard operator).  "Lizard" (arXiv 2507.09025), Preliminaries: the
 * matrix form of GLA needs the cumulative gate products in full precision, so standard
 * GLA kernels fall back to fp32 arithmetic without tensor cores; Efficiency, Table 3:
 * forward latency of the Lizard kernel against such a standard GLA.  This call computes
 * the GLA branch alone,
 *   y_i = phi_q_i^T h_i,  h_i = gamma_i (.) h_{i-1} + phi_k_i v_i^T  (h_{-1} = h0),
 * chunkwise over 64-token chunks with every operand and product in fp32 on CUDA cores
 * (FFMA): chunk states K^T V, a scan over chunks, then tril(Qt Kt^T) V + Qt h per chunk
 * with Qt = phi_q e^{b}, Kt = phi_k e^{-b} (b the chunk-local cumulative log gate).
 *   dims: B, H, L, dk = dv in {64, 128}, dtype (M and scale are ignored); B * H <= 65535.
 *   phi_q, phi_k [B,H,L,dk] T;  v [B,H,L,dv] T;  log_gamma [B,H,L,dk] fp32;  y [B,H,L,dv] T
 *   output;  h0, h_final [B,H,dk,dv] fp32 or NULL.
 *   workspace: lizard_gla_std_workspace_bytes(dims) bytes (every chunk's state in fp32),
 *   caller-owned, 16-byte aligned.
 * The factorised form has no finite value when the cumulative log gate inside a chunk
 * leaves [-80, 80]; such a chunk sets LIZARD_ERR_DEVICE_CHECK in the workspace status word
 * (lizard_attn_fwd has no such limit).
 */
size_t lizard_gla_std_workspace_bytes(const lizard_dims* dims);
lizard_status lizard_gla_std_fwd(const lizard_dims* dims, const void* phi_q, const void* phi_k,
                                 const void* v, const float* log_gamma, void* y, const float* h0,
                                 float* h_final, void* workspace, size_t workspace_bytes,
                                 void* stream);

/*
 * Self-test of the device-side failure detection (a library service; the pages have no
 * counterpart).  Every wait of the tile kernels on an mbarrier is bounded: when it runs
 * out the CTA stops its other roles, drains what it has in flight, frees its tensor
 * memory, returns, and the call's workspace status word reads LIZARD_ERR_TIMEOUT.  No
 * valid input makes a wait run out, so this call makes one run out on purpose: a single
 * CTA arms a barrier for bytes that no copy will deliver (nothing is in flight, so
 * nothing can fault) and waits wait_cycles SM clock cycles (1 .. about 2e9; 2e5 is about
 * 100 us).  Afterwards lizard_check_device_errors(workspace) returns LIZARD_ERR_TIMEOUT
 * and clears the word, and the context stays usable.  workspace: at least 256 bytes,
 * 16-byte aligned; its status word is zeroed first on `stream`.
 */
lizard_status lizard_selftest_wait_timeout(void* workspace, size_t workspace_bytes,
                                           int64_t wait_cycles, void* stream);

/* Static description of a status code. */
const char* lizard_status_string(lizard_status status);

/* LIZARD_ABI_VERSION of the library that was loaded. */
int32_t lizard_abi_version(void);

/* Number of kernels the most recent call of this thread enqueued (for launch counts). */
int32_t lizard_last_launch_count(void);

/*
 * Per-kernel device timing.  While enabled (per host thread), every kernel the library
 * enqueues is bracketed by two CUDA events on its stream.  lizard_trace_read waits for
 * the recorded events, writes up to max_records NUL-terminated kernel names (name_len
 * bytes each) and durations in milliseconds, returns the count and clears the log.
 */
lizard_status lizard_trace_enable(int32_t enable);
int32_t lizard_trace_read(char* names, int32_t name_len, float* ms, int32_t max_records);

#ifdef __cplusplus
}
#endif

#endif /* LIZARD_H */
