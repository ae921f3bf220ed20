/*
 * ssm.h -- C ABI of the B300 selective state-space (S6) library, libssm.so.
 *
 * Five operations, each on the caller's CUDA stream:
 *   ssm_causal_conv1d_fwd       depthwise causal conv1d (+ SiLU), the block's short conv
 *   ssm_selective_scan_fwd      selective scan forward (optionally with the conv fused in
 *                               front), returning y and the final state h_L
 *   ssm_selective_state_update  one recurrent (decode) step for a batch of sequences
 *   ssm_selective_scan_bwd      the scan's backward pass (training)
 *   ssm_causal_conv1d_bwd       the conv prologue's backward pass (training)
 *
 * Sources (page title, section):
 *   "Mamba" (ai360xpert.com, core ML), "The selection mechanism":
 *       Delta_t = softplus(W x_t + b), Abar_t = exp(Delta_t A), Bbar_t ~ Delta_t B.
 *   "Mamba (Selective State-Space Model)" (gunjandhanuka.github.io), "Key math":
 *       B_t, C_t, Delta_t computed from the input; A learned; hardware-aware parallel scan.
 *   "Mamba" (ozercemkelahmet.com/tools/mamba), "How it works" steps 1-5,
 *       "A minimal selective scan in PyTorch", "Deployment notes" (state passed between
 *       prompt chunks; constant-size state at inference).
 *   "Overview of Mamba (SSM) Model" (bembew.net), "How the Mamba Block Works":
 *       depthwise conv + SiLU before the SSM, SiLU(z) gate, Mamba(d_model, d_state, d_conv, expand).
 *
 * Conventions shared by every call
 *   - Device pointers only (cudaMalloc'd or equivalent), contiguous, row-major, in the
 *     layouts stated per argument. The caller owns every buffer, including the scan's
 *     workspace; the library allocates nothing and keeps no state between calls.
 *   - Per-token tensors use the I/O dtype `io` (SSM_F32 = float, SSM_BF16 = bfloat16).
 *     Parameters (A, D, delta_bias, conv weight/bias) and states (h0, h_last, the decode
 *     state) are always float32. Arithmetic is float32 throughout; bf16 results are
 *     rounded to nearest-even once, on store.
 *   - Pointers must be aligned to their element size. Per-token base pointers that are
 *     16-byte aligned, with rows whose byte length is a multiple of 16, take the
 *     vectorised path; anything else takes a slower element-wise path with the same
 *     results.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Every call is
 *     asynchronous with respect to the host and does not synchronise.
 *   - Errors: argument checks happen on the host before any launch and return
 *     SSM_ERR_INVALID_ARG or SSM_ERR_UNSUPPORTED without touching device memory. A
 *     failed launch returns SSM_ERR_CUDA. No call aborts, prints or throws.
 *   - Empty work (batch == 0 or dim == 0) returns SSM_OK without a launch.
 *   - dstate (N) is 1..32 for the forward scan and the decode step (compiled for N <= 16
 *     and N <= 32), 1..16 for the backward pass. d_conv (K) is 1..4 when a conv weight is
 *     given.
 *   - Tensors named as inputs are only read; outputs must not alias inputs, except the
 *     decode state and window, which are updated in place.
 */
#ifndef SSM_H_
#define SSM_H_

#include <stddef.h>

#if defined(__GNUC__) || defined(__clang__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SSM_OK = 0,
  SSM_ERR_INVALID_ARG = 1, /* a required pointer is NULL, a size is negative, a buffer is too small */
  SSM_ERR_UNSUPPORTED = 2, /* a valid request outside the compiled limits (dstate > 32, or > 16 for
                              the backward pass; d_conv > 4, misaligned pointer, unknown dtype) */
  SSM_ERR_CUDA = 3         /* a CUDA runtime call or kernel launch failed */
} ssm_status;

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype;

/* Option bits of the flags argument. SSM_SCAN_REVERSE: the scan entry points only.
 * SSM_SCAN_S4D_REAL: ssm_selective_scan_fwd (and its no-allocation form) only. */
#define SSM_SCAN_REVERSE 1u
#define SSM_SCAN_ZOH 2u
#define SSM_SCAN_S4D_REAL 4u

/* Library version (major * 10000 + minor * 100 + patch). */
SSM_API int ssm_version(void);

/* Static, human-readable name of a status code. */
SSM_API const char* ssm_status_string(int status);

/*
 * Causal depthwise conv1d of every channel, optionally followed by SiLU:
 *   out[b,d,t] = act( sum_{k=0}^{K-1} w[d,k] * x[b,d,t-(K-1)+k] + bias[d] ),
 * where x[b,d,s] for s < 0 is conv_init[b,d,(K-1)+s] (or 0 when conv_init is NULL).
 * ("Overview of Mamba (SSM) Model", block: depthwise convolution and SiLU before the SSM;
 *  "Mamba" ozercemkelahmet.com, glossary: a causal conv only sees current and past positions.)
 *
 *   x          [batch, dim, seqlen] io        input
 *   w          [dim, d_conv] float32          filter taps; w[d, K-1] multiplies the current input
 *   bias       [dim] float32 or NULL (= 0)
 *   conv_init  [batch, dim, d_conv-1] io or NULL: raw inputs preceding t = 0, oldest first
 *   out        [batch, dim, seqlen] io        output (must not alias x)
 *   apply_silu 0 or 1
 */
SSM_API ssm_status ssm_causal_conv1d_fwd(const void* x, const float* w, const float* bias, const void* conv_init,
                                 void* out, int batch, int dim, int seqlen, int d_conv, int apply_silu,
                                 ssm_dtype io, void* stream);

/*
 * Chunk length the scan uses when asked for chunk_len = 0, for this problem on the
 * current device (a multiple of 64, or seqlen rounded up to 64 when no chunking pays).
 */
SSM_API int ssm_scan_default_chunk_len(int batch, int dim, int seqlen, int dstate, ssm_dtype io);

/*
 * Workspace bytes ssm_selective_scan_fwd needs for this problem and chunk length
 * (chunk_len = 0 means ssm_scan_default_chunk_len). 0 when the scan runs as one chunk.
 */
SSM_API size_t ssm_scan_workspace_bytes(int batch, int dim, int seqlen, int dstate, int chunk_len, ssm_dtype io);

/*
 * Selective scan forward, for every batch element b and channel d:
 *   u_t     = x_t, or silu(causal conv of x)_t when conv_w != NULL (as ssm_causal_conv1d_fwd)
 *   Delta_t = softplus(delta_t + delta_bias[d])      (delta_t + delta_bias[d] if delta_softplus == 0)
 *   h_t[n]  = exp(Delta_t A[d,n]) h_{t-1}[n] + Delta_t B[b,n,t] u_t,    h_{-1} = h0 (or 0)
 *   y_t     = sum_n C[b,n,t] h_t[n] + D[d] u_t
 *   out_t   = y_t * silu(z_t)                        (y_t when z == NULL)
 * ("Mamba" ai360xpert.com, selection mechanism; "Mamba" ozercemkelahmet.com, steps 1-4 and the
 *  PyTorch slow reference; "Overview of Mamba (SSM) Model", the SiLU gate.)
 * The per-step state never leaves the chip. Time is cut into chunks of chunk_len steps; when
 * there is more than one chunk, a first kernel writes each chunk's carry (the sum of Delta
 * and the chunk's end state from zero) to the workspace, and the main kernel starts every
 * chunk from the composition of its predecessors' carries,
 *   (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2),  a = exp(A * sum Delta),
 * the associative operator of the parallel scan ("Mamba" ai360xpert.com, "Why this breaks
 * the parallel form"; "Mamba" ozercemkelahmet.com, step 4).
 *
 *   x           [batch, dim, seqlen] io   the scan input u, or the conv input when conv_w != NULL
 *   delta       [batch, dim, seqlen] io   step-size pre-activation
 *   A           [dim, dstate] float32     (negative for a stable decay)
 *   B, C        [batch, dstate, seqlen] io  per-token input / output maps, shared by all channels
 *   D           [dim] float32 or NULL (no skip term)
 *   z           [batch, dim, seqlen] io or NULL (no gate)
 *   delta_bias  [dim] float32 or NULL (= 0)
 *   delta_softplus  0 or 1
 *   conv_w      [dim, d_conv] float32 or NULL (no conv prologue); conv_b [dim] float32 or NULL
 *   conv_init   [batch, dim, d_conv-1] io or NULL: raw inputs before t = 0 (a previous chunk's tail)
 *   h0          [batch, dim, dstate] float32 or NULL (zero initial state)
 *   out         [batch, dim, seqlen] io   output
 *   h_last      [batch, dim, dstate] float32 or NULL: the state after the last step (h0 if seqlen == 0)
 *   conv_state_out [batch, dim, d_conv-1] io or NULL: the last d_conv-1 raw inputs of the stream
 *               conv_init ++ x, ready to be passed as the decode window or the next conv_init
 *   chunk_len   0 = library default; otherwise >= 1, rounded up to a multiple of 64
 *   workspace   device buffer of at least ssm_scan_workspace_bytes(...) bytes, 256-byte aligned,
 *               or NULL/0 bytes. With chunk_len = 0 the library lowers the chunk count until the
 *               given workspace suffices (one chunk needs none); with an explicit chunk_len a
 *               too-small workspace is SSM_ERR_INVALID_ARG. Its contents need no initialisation.
 *   flags       0, or any of SSM_SCAN_REVERSE, SSM_SCAN_ZOH, SSM_SCAN_S4D_REAL; any other bit is
 *               SSM_ERR_INVALID_ARG.
 *
 * SSM_SCAN_S4D_REAL: an opt-in fast path for the S4D-real structure of A, A[d,n] = (n+1) A[d,0]
 * (the pages' initialisation A = -(1..N): "Mamba", ozercemkelahmet.com, "A minimal selective scan
 * in PyTorch"). There Abar_n = exp(Delta A[d,n]) = Abar_0^(n+1), so each group of 4 states takes one
 * exp2, the anchor Abar_0^(4g+1), and multiplies by Abar_0, Abar_0^2, Abar_0^3: 4 exp2 per 16
 * states in place of 16. Every CTA checks the structure on the A it loads (an exact float
 * comparison with (n+1) A[d,0], over all its channels) and takes the generic path when any
 * channel fails it, so the flag never changes what is computed, only its rounding: no Abar_n
 * carries more than about 4 times the relative error of one exp2. It applies to
 * whole-channel passes of the Euler rule (N <= 16, one lane per channel, the plan of long
 * sequences); with SSM_SCAN_ZOH, N > 16 or the two-lane plan the flag is ignored. Trained A
 * drifts from its initialisation, so the generic path is the one the library is measured on.
 *
 * SSM_SCAN_ZOH: zero-order-hold discretisation of the input term,
 *   h_t[n] = exp(Delta_t A[d,n]) h_{t-1}[n] + expm1(Delta_t A[d,n]) / A[d,n] * B[b,n,t] u_t
 * ("Mamba", ai360xpert.com, "Show Me the Code": B_bar = (1 - A_bar)/(-A) B; "Mamba",
 * inferensys.com: the continuous system is discretized by a zero-order hold), instead of the
 * default Euler term Delta_t B u_t. Where A[d,n] = 0 the factor is its limit Delta_t; near it
 * the factor is taken from its series, so it stays accurate as Delta A -> 0.
 *
 * SSM_SCAN_REVERSE: the backward scan of a bidirectional layer ("Mamba", ozercemkelahmet.com,
 * "Bidirectional and multi-directional scans": one scan forward, one backward, results merged
 * by the caller). It is the same operation applied to the time-reversed stream:
 *   out = flip(scan(flip(x), flip(delta), flip(B), flip(C), flip(z))),  flip: t -> L-1-t,
 * so the recurrence runs from t = L-1 down to t = 0 and the conv looks at t .. t+K-1.
 * h0 is the state before t = L-1, h_last the state after t = 0; conv_init holds the K-1 raw
 * inputs that follow the sequence, in reversed order (conv_init[j] is x at L+K-2-j), and
 * conv_state_out returns x at K-2, ..., 0, which is the conv_init of a backward call over the
 * part of the sequence before this one.
 */
SSM_API ssm_status ssm_selective_scan_fwd(const void* x, const void* delta, const float* A, const void* B, const void* C,
                                  const float* D, const void* z, const float* delta_bias, int delta_softplus,
                                  const float* conv_w, const float* conv_b, int d_conv, const void* conv_init,
                                  const float* h0, void* out, float* h_last, void* conv_state_out, int batch,
                                  int dim, int seqlen, int dstate, ssm_dtype io, int chunk_len, void* workspace,
                                  size_t workspace_bytes, unsigned int flags, void* stream);

/*
 * Workspace bytes ssm_selective_scan_bwd needs: about 8.5 bytes per (b, d, t) for the state
 * checkpoints (16 fp32 states and a sum every 8 steps), 4 bytes per (b, 32-channel tile, t, n)
 * for the partial sums of dB and dC, and the per-chunk aggregates and partial dA, dD, dbias.
 */
SSM_API size_t ssm_scan_bwd_workspace_bytes(int batch, int dim, int seqlen, int dstate, ssm_dtype io);

/*
 * Backward pass of ssm_selective_scan_fwd (training) for the forward-time Euler scan with the
 * scan input u given directly (conv_w = NULL in the forward call): the gradients of a scalar
 * loss L from dout = dL/dout and dh_last = dL/dh_last, through the adjoint recurrence
 *   g_t[n] = dL/dh_t[n] = exp(Delta_{t+1} A[d,n]) g_{t+1}[n] + C[b,n,t] dy_t,   g_{L-1} starts at dh_last
 *   dy_t  = dout_t silu(z_t)          dz_t = dout_t y_t silu'(z_t)
 *   du_t  = D[d] dy_t + sum_n g_t[n] Delta_t B[b,n,t]
 *   ddelta_t = sigmoid(delta_t + bias) sum_n g_t[n] (A[d,n] Abar_t[n] h_{t-1}[n] + B[b,n,t] u_t)
 *   dA[d,n] = sum_{b,t} g_t[n] Delta_t Abar_t[n] h_{t-1}[n]      dB[b,n,t] = sum_d g_t[n] Delta_t u_t
 *   dC[b,n,t] = sum_d dy_t h_t[n]     dD[d] = sum_{b,t} dy_t u_t     ddelta_bias[d] = sum_{b,t} ddelta_t
 *   dh0[b,d,n] = Abar_0[n] g_0[n]
 * (the chain rule on the forward definition; "Mamba (Selective State-Space Model)",
 * gunjandhanuka.github.io, "Cost of selectivity": training runs through the parallel scan). Without
 * softplus the sigmoid factor is 1.
 *
 * Inputs as for the forward call (u in place of x); dout [batch, dim, seqlen] io; dh_last
 * [batch, dim, dstate] float32 or NULL (= 0).
 * Outputs (all written, none accumulated into):
 *   du, ddelta [batch, dim, seqlen] io;  dz [batch, dim, seqlen] io, required when z != NULL;
 *   dA [dim, dstate], dB, dC [batch, dstate, seqlen], dD [dim], ddelta_bias [dim],
 *   dh0 [batch, dim, dstate], all float32; dD, ddelta_bias and dh0 may be NULL (not computed).
 * The call makes two passes over the data: a forward pass writes a state checkpoint every 8
 * steps to the workspace (ssm_scan_bwd_workspace_bytes, 256-byte aligned, no initialisation
 * needed), then a reverse pass recomputes each 4 steps' states from them and walks the
 * adjoint back. Channel and sequence sums are formed in a fixed order, so the results are
 * deterministic.
 *   flags  must be 0: SSM_SCAN_REVERSE and SSM_SCAN_ZOH have no backward pass here
 *          (SSM_ERR_UNSUPPORTED); unknown bits are SSM_ERR_INVALID_ARG.
 */
SSM_API ssm_status ssm_selective_scan_bwd(const void* u, const void* delta, const float* A, const void* B,
                                          const void* C, const float* D, const void* z, const float* delta_bias,
                                          int delta_softplus, const float* h0, const void* dout,
                                          const float* dh_last, void* du, void* ddelta, void* dz, float* dA,
                                          float* dB, float* dC, float* dD, float* ddelta_bias, float* dh0,
                                          int batch, int dim, int seqlen, int dstate, ssm_dtype io,
                                          void* workspace, size_t workspace_bytes, unsigned int flags,
                                          void* stream);

/*
 * Workspace bytes ssm_causal_conv1d_bwd needs (20 bytes per 1024 steps of every row).
 */
SSM_API size_t ssm_conv_bwd_workspace_bytes(int batch, int dim, int seqlen, int d_conv, ssm_dtype io);

/*
 * Backward of ssm_causal_conv1d_fwd (training): with acc_t = sum_k w[d,k] xs(t-(K-1)+k) + bias[d]
 * and out_t = silu(acc_t) (apply_silu) or acc_t, where xs(s) is x for s >= 0 and conv_init for
 * s < 0, the chain rule gives from dout = dL/dout
 *   dacc_t = dout_t silu'(acc_t)        dx[s] = sum_k w[d,k] dacc_{s+(K-1)-k}
 *   dconv_init: the same sum at the window positions s = -(K-1) .. -1
 *   dw[d,k] = sum_{b,t} dacc_t xs(t-(K-1)+k)      dbias[d] = sum_{b,t} dacc_t
 * ("Overview of Mamba (SSM) Model", "How the Mamba Block Works": the conv and SiLU in front of
 * the SSM; with ssm_selective_scan_bwd, whose du is this call's dout, it completes the
 * gradient of the fused block.)
 *   x, dout, dx  [batch, dim, seqlen] io;  conv_init, dconv_init [batch, dim, d_conv-1] io or NULL
 *   w [dim, d_conv], bias [dim] or NULL: float32;  dw [dim, d_conv], dbias [dim] or NULL: float32
 *   workspace    ssm_conv_bwd_workspace_bytes(...) bytes, 16-byte aligned, no initialisation
 * All outputs are written, not accumulated into; sums are formed in a fixed order.
 */
SSM_API ssm_status ssm_causal_conv1d_bwd(const void* x, const float* w, const float* bias, const void* conv_init,
                                         const void* dout, int apply_silu, void* dx, float* dw, float* dbias,
                                         void* dconv_init, int batch, int dim, int seqlen, int d_conv, ssm_dtype io,
                                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * One recurrent (decode) step for every sequence b and channel d, state updated in place:
 *   window   = [conv_state[b,d,0 .. K-2], x[b,d]]          (oldest first)
 *   u        = silu(sum_k conv_w[d,k] window[k] + conv_b[d]);   conv_state <- window[1 .. K-1]
 *              (u = x[b,d] when conv_w == NULL; conv_state is then unused and may be NULL)
 *   Delta    = softplus(delta[b,d] + delta_bias[d])
 *   state[n] = exp(Delta A[d,n]) state[n] + Delta B[b,n] u
 *              (with SSM_SCAN_ZOH: + expm1(Delta A[d,n]) / A[d,n] B[b,n] u, as for the scan)
 *   y[b,d]   = (sum_n C[b,n] state[n] + D[d] u) * silu(z[b,d])
 * ("Mamba" ozercemkelahmet.com, step 5 and deployment notes: a fixed-size state per sequence
 *  updated once per token; "Mamba (Selective State-Space Model)", constant inference state.)
 *
 *   state       [batch, dim, dstate] float32, in/out
 *   conv_state  [batch, dim, d_conv-1] io, in/out (the raw-input window)
 *   x, delta    [batch, dim] io;   z [batch, dim] io or NULL
 *   A           [dim, dstate] float32;   B, C [batch, dstate] io
 *   D, delta_bias, conv_w, conv_b as for the scan
 *   y           [batch, dim] io output
 *   flags       0 or SSM_SCAN_ZOH; any other bit is SSM_ERR_INVALID_ARG
 */
SSM_API ssm_status ssm_selective_state_update(float* state, void* conv_state, const void* x, const void* delta,
                                      const float* A, const void* B, const void* C, const float* D, const void* z,
                                      const float* delta_bias, int delta_softplus, const float* conv_w,
                                      const float* conv_b, int d_conv, void* y, int batch, int dim, int dstate,
                                      ssm_dtype io, unsigned int flags, void* stream);

/*
 * Segment aggregate of the selective scan, for scans split across sequence segments (a long
 * prompt processed in parts on several GPUs, or in parts on one). "Mamba" (ozercemkelahmet.com),
 * "Deployment notes": long prompts are processed in chunks that pass the state on; the
 * associative operator that makes the segments independent is the composition of the affine
 * maps h -> a h + b of "Mamba" (inferensys.com glossary), the parallel-scan paragraph.
 *
 * For one segment of a sequence (the tokens t0 .. t0+seqlen-1 of each (batch, channel)),
 * with the arguments and layouts of ssm_selective_scan_fwd (x, delta, B, conv prologue,
 * delta_bias / softplus, flags SSM_SCAN_REVERSE and SSM_SCAN_ZOH):
 *   S_out [batch, dim] float32          = sum over the segment of Delta_t (natural units), so
 *                                         that exp(A[d,n] S) is the segment's decay of state n;
 *   h_out [batch, dim, dstate] float32  = the state at the segment's end when it starts at zero.
 * The state after the segment from an initial state h is exp(A S) h + h_out (elementwise per
 * state), so segments can be aggregated independently and composed in order afterwards
 * (ssm_scan_compose). conv_init is the conv window before the segment: the last d_conv-1 raw
 * inputs of the previous segment (or of the stream before the sequence).
 * The workspace holds per-chunk partial aggregates: ssm_scan_aggregate_workspace_bytes bytes,
 * 256-byte aligned; a smaller one returns SSM_ERR_INVALID_ARG. seqlen == 0 writes zeros.
 */
SSM_API size_t ssm_scan_aggregate_workspace_bytes(int batch, int dim, int seqlen, int dstate, ssm_dtype io);
SSM_API ssm_status ssm_selective_scan_aggregate(const void* x, const void* delta, const float* A, const void* B,
                                                const float* delta_bias, int delta_softplus, const float* conv_w,
                                                const float* conv_b, int d_conv, const void* conv_init, float* S_out,
                                                float* h_out, int batch, int dim, int seqlen, int dstate,
                                                ssm_dtype io, void* workspace, size_t workspace_bytes,
                                                unsigned int flags, void* stream);

/*
 * Composition of segment aggregates: h_out = the state after nseg segments that start from
 * h0, i.e. h = exp(A S_j) h + b_j for j = 0 .. nseg-1 with h = h0 (zeros when h0 is NULL).
 *   S  [nseg, batch, dim] float32, b [nseg, batch, dim, dstate] float32 (from
 *   ssm_selective_scan_aggregate, segment after segment); A [dim, dstate]; h0 and h_out
 *   [batch, dim, dstate] float32 (h_out may alias h0). nseg == 0 copies h0 (or writes zeros).
 */
SSM_API ssm_status ssm_scan_compose(const float* S, const float* b, const float* A, const float* h0, float* h_out,
                                    int nseg, int batch, int dim, int dstate, void* stream);

/*
 * Size in bytes of the fixed device array that ssm_selective_scan_fwd_noalloc uses as its
 * chunk-carry scratch. Every GPU that loads the library holds this much memory until exit.
 */
#define SSM_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

/*
 * ssm_selective_scan_fwd for callers that cannot allocate device memory: callers that own
 * only their inputs and outputs (for example a host framework's plugin interface that hands
 * over tensor pointers but no workspace) or a serving loop that must not call cudaMalloc,
 * which can block on device-wide synchronisation. The pages have no counterpart to this
 * call; it is a deployment convenience of this library.
 *
 * Arguments, layouts and results are those of ssm_selective_scan_fwd without the workspace:
 * the chunk carries go to a file-scope device array of SSM_NOALLOC_SCRATCH_BYTES bytes
 * instead. The call allocates nothing (no cudaMalloc, no cudaFree, no allocating library
 * routine).
 *   - Every call looks up that array's device address in the current device's context
 *     (cudaGetSymbolAddress, which allocates nothing). The first call on a device also loads
 *     the library's device code there: make that first call before any stream capture.
 *   - With chunk_len = 0 the scan uses as many chunks as fit the array (one chunk needs
 *     none). An explicit chunk_len whose carries need more than SSM_NOALLOC_SCRATCH_BYTES
 *     (see ssm_scan_workspace_bytes) returns SSM_ERR_UNSUPPORTED before anything runs.
 *   - Every call shares the one array and it keeps the last call's contents. Nothing in it
 *     needs clearing: each call's carry kernel writes every entry its main kernel reads.
 *     Calls that overlap on the GPU (different streams, or different host threads without
 *     ordering) race on the array and give wrong results; serialise them.
 */
SSM_API ssm_status ssm_selective_scan_fwd_noalloc(const void* x, const void* delta, const float* A, const void* B,
                                                  const void* C, const float* D, const void* z,
                                                  const float* delta_bias, int delta_softplus, const float* conv_w,
                                                  const float* conv_b, int d_conv, const void* conv_init,
                                                  const float* h0, void* out, float* h_last, void* conv_state_out,
                                                  int batch, int dim, int seqlen, int dstate, ssm_dtype io,
                                                  int chunk_len, unsigned int flags, void* stream);

/*
 * Multi-head selective SSM with one decay per head: the layer of the structured state-space
 * duality ("Mamba" (ai360xpert.com / inferensys.com pages), "Mamba-2 introduces the Structured
 * State Space Duality": multi-head SSM with selective parameters per head, the state dimension
 * used like a head dimension, the computation mapped to structured matrix products that run on
 * tensor cores; "Mamba" (ozercemkelahmet.com), "Mamba-2 and the dual view": the layer as a
 * masked matrix product with a decaying mask). For every batch element b and head h, with a
 * state H of headdim x dstate:
 *   Delta_t   = softplus(dt[b,t,h] + dt_bias[h])        (the raw sum when dt_softplus == 0)
 *   H_t[p][n] = exp(Delta_t A[h]) H_{t-1}[p][n] + Delta_t x[b,t,h,p] B[b,t,n],   H_{-1} = h0 or 0
 *   y[b,t,h,p] = sum_n C[b,t,n] H_t[p][n] + D[h] x[b,t,h,p]
 * B and C are shared by all heads. The GPU evaluates the chunked dual form in one kernel: one
 * CTA per (batch, head) walks chunks of 128 steps with the running state on the chip, and per
 * chunk computes the masked product (C B^T masked and decayed) X, C H_in and the chunk's state
 * increment (decayed B)^T X on the tensor cores (tcgen05, bf16 operands, fp32 accumulation).
 * The three operands the kernel computes (the masked product, H_in and the decayed B) enter as
 * pairs of bf16 terms, hi = bf16(v) and lo = bf16(v - hi), so the result keeps the bf16-I/O
 * bound, |y - exact| <= 1e-2 + 2e-2 |exact|.
 *
 *   x       [batch, seqlen, nheads, headdim] bf16      y [batch, seqlen, nheads, headdim] bf16
 *   dt      [batch, seqlen, nheads] bf16               B, C [batch, seqlen, dstate] bf16
 *   A, D, dt_bias [nheads] float32 (D, dt_bias may be NULL)
 *   h0, h_last [batch, nheads, headdim, dstate] float32 or NULL (h_last = h0 or 0 when seqlen == 0)
 *   io      SSM_BF16 only (SSM_F32 returns SSM_ERR_UNSUPPORTED); headdim must be 64 and dstate
 *           128, else SSM_ERR_UNSUPPORTED
 *   workspace  device buffer of ssm_ssd_workspace_bytes(...) bytes (256), 256-byte aligned;
 *           its contents need no initialisation. After the call (once the stream reaches it)
 *           its first 4 bytes hold a status word: 0 on success; 1 if a wait on the tensor cores
 *           or on a tensor-map copy ran out; 2 if the kernel's shared memory was not 1024-byte
 *           aligned (not expected: the kernel checks rather than assumes it). On a nonzero word
 *           y and h_last are undefined; the context stays usable.
 * x, B, C and y must be 16-byte aligned; dt 2-byte aligned. The call allocates nothing and
 * runs one kernel (after clearing the status word) on `stream`.
 */
SSM_API size_t ssm_ssd_workspace_bytes(int batch, int seqlen, int nheads, int headdim, int dstate, ssm_dtype io);

/*
 * Test hooks, process-wide, for tests only (0 = none, the default).
 *   SSM_TEST_SSD_SKIP_MMA: ssm_ssd_fwd issues no tensor-core GEMMs, so its first wait for them
 *   runs out (after a shortened bound, well under a second). The kernel then records status 1
 *   in the workspace word, frees its tensor memory and returns; the results are undefined.
 *   This exercises the bounded-wait path without faulting or hanging the GPU.
 */
#define SSM_TEST_SSD_SKIP_MMA 1u
SSM_API void ssm_set_test_hooks(unsigned int flags);
SSM_API ssm_status ssm_ssd_fwd(const void* x, const void* dt, const float* A, const void* B, const void* C,
                               const float* D, const float* dt_bias, int dt_softplus, const float* h0, void* y,
                               float* h_last, int batch, int seqlen, int nheads, int headdim, int dstate,
                               ssm_dtype io, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Range checks of the debug build.
 *
 * libssm_debug.so is this library compiled with SSM_DEBUG_BOUNDS: before each global-memory
 * access of the scan (main, carry, segment aggregate and composition), decode, conv (forward
 * and backward), scan backward and state-space-duality kernels, the element range it touches
 * is tested against the size of its tensor, as the call's arguments give them (the duality
 * kernel's bulk tensor copies are clipped by their tensor maps instead). An access outside its
 * tensor is skipped (a load reads zero) and sets a bit of a device error word; nothing traps.
 * Bits: 1 scan, 2 decode, 4 conv, 8 segment aggregate / composition, 16 scan backward,
 * 32 state-space duality.
 *
 * ssm_debug_bounds_status synchronises the device (a blocking copy from the word), stores the
 * word's bits in *flags_out and, when clear is 1, resets them to zero. It returns
 * SSM_ERR_UNSUPPORTED from the release library (libssm.so), which has no checks compiled in,
 * SSM_ERR_INVALID_ARG for a NULL flags_out or a clear other than 0 or 1, and SSM_ERR_CUDA if
 * the copy fails. A zero word after a call means that every checked access of it lay inside
 * its tensor.
 */
SSM_API ssm_status ssm_debug_bounds_status(unsigned int* flags_out, int clear);

#ifdef __cplusplus
}
#endif

#endif /* SSM_H_ */
