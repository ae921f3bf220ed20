// ssm_internal.h -- host-side launch interface between the C ABI (ssm_api.cu) and the
// kernels. Plain structs of pointers and sizes; no torch types.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace ssm {

// Largest state size the decode and backward kernels hold in registers.
constexpr int kMaxDstate = 16;
// Largest state size of the forward scan (two compile-time geometries: N <= 16 and N <= 32).
constexpr int kMaxDstateScan = 32;
// Largest conv width; narrower filters are zero-padded on the old side to this width.
constexpr int kMaxConv = 4;
// Chunk lengths are multiples of the scan's time tile.
constexpr int kChunkQuantum = 64;

struct ScanArgs {
  const void* x;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* delta_bias;
  int delta_softplus;
  const float* conv_w;   // NULL: no conv prologue
  const float* conv_b;
  int d_conv;
  const void* conv_init;
  const float* h0;
  void* out;
  float* h_last;
  void* conv_state_out;
  int batch, dim, seqlen, dstate;
  int bf16;              // io dtype: 0 = fp32, 1 = bf16
  int vec;               // 1: 16-byte vector path is legal for every per-token tensor
  int chunk_len;         // multiple of kChunkQuantum, >= 1 chunk
  int nchunks;
  int lanes;             // lanes per channel of the main pass: 1 (N <= 16), 2 (N <= 16) or 4 (N <= 32)
  int reverse;           // 1: the scan runs from t = L-1 down to t = 0
  int zoh;               // 1: zero-order-hold input term expm1(Delta A)/A B u
  int s4d;               // 1: take Abar_n = Abar_0^(n+1) where every channel of a CTA has A[d,n] = (n+1) A[d,0]
  int ws_chunks;         // carry entries the workspace holds (nchunks-1; nchunks for a segment aggregate)
  float* ws_S;           // [ws_chunks][batch*dim] sum of Delta per chunk
  float* ws_h;           // [ws_chunks][batch*dim][scan_state_stride(dstate)] chunk end state from zero
};

struct ConvArgs {
  const void* x;
  const float* w;
  const float* bias;
  const void* conv_init;
  void* out;
  int batch, dim, seqlen, d_conv, apply_silu;
  int bf16;
  int vec;
};

// Multi-head SSM with one decay per head (state-space-duality layer), bf16 I/O, head dim 64,
// state dim 128, chunks of 128 steps.
struct SsdArgs {
  const void* x;         // [batch, seqlen, nheads, 64] bf16
  const void* dt;        // [batch, seqlen, nheads] bf16
  const float* A;        // [nheads]
  const void* B;         // [batch, seqlen, 128] bf16
  const void* C;
  const float* D;        // [nheads] or NULL
  const float* dt_bias;  // [nheads] or NULL
  int dt_softplus;
  const float* h0;       // [batch, nheads, 64, 128] or NULL
  void* y;               // [batch, seqlen, nheads, 64] bf16
  float* h_last;         // [batch, nheads, 64, 128] or NULL
  int batch, seqlen, nheads, nchunks;
  int* ws_status;        // nonzero after the call: a tensor-core wait ran out
};

struct ConvBwdArgs {
  const void* x;
  const float* w;
  const float* bias;
  const void* conv_init;
  const void* dout;
  void* dx;
  float* dw;
  float* dbias;          // NULL: not computed
  void* dconv_init;      // NULL: not computed
  int batch, dim, seqlen, d_conv, apply_silu;
  int bf16;
  float* ws_part;        // [batch*dim][segments][5] per-block dw (padded taps) and dbias sums
};

struct DecodeArgs {
  float* state;
  void* conv_state;
  const void* x;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* delta_bias;
  int delta_softplus;
  const float* conv_w;
  const float* conv_b;
  int d_conv;
  void* y;
  int batch, dim, dstate;
  int bf16;
  int zoh;               // 1: zero-order-hold input term expm1(Delta A)/A B u
};

struct ScanBwdArgs {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* delta_bias;
  int delta_softplus;
  const float* h0;
  const void* dout;
  const float* dh_last;
  void* du;
  void* ddelta;
  void* dz;
  float* dA;
  float* dB;
  float* dC;
  float* dD;
  float* ddelta_bias;
  float* dh0;
  int batch, dim, seqlen, dstate;
  int bf16;
  int vec;               // 16-byte staging: row bytes a multiple of 16, bases 16-byte aligned
  int chunk_len;         // multiple of the 8-step tile; the sequence is cut into nchunks chunks
  int nchunks;
  float* ws_ck;          // [batch][channel tiles][tiles] checkpoints: states from zero at the chunk
                         //   start and sums of Delta', before every 8-step tile
  float* fS;             // [nchunks][batch*dim]: sum of Delta' of the chunk
  float* fh;             // [nchunks][batch*dim][16]: chunk end state from a zero start
  float* bh;             // [nchunks][batch*dim][16]: adjoint leaving the chunk start, zero at its end
  float* ws_dBC;         // [batch][channel tiles][seqlen][32]: per-tile channel sums (dB at n, dC at 16+n)
  float* ws_dA;          // [nchunks][batch][dim][16]
  float* ws_dD;          // [nchunks][batch][dim]
  float* ws_dbias;       // [nchunks][batch][dim]
};

// Channels one main-pass CTA covers with `lanes` lanes per channel (1, 2 or 4).
int scan_channels_per_cta(int lanes);
// CTAs of that main-pass kernel resident per SM (occupancy query; the shared-memory limit
// without a device)
int scan_resident_ctas_per_sm(bool bf16, int lanes);
// Per-channel stride of the chunk end states in the scan workspace: 16 for N <= 16, else 32.
int scan_state_stride(int dstate);

// Workspace layout of the chunked scan.
size_t scan_workspace_bytes(long long channels, int nchunks, int dstate);
void scan_workspace_split(void* ws, long long channels, int nchunks, float** S, float** h);

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t stream);

// Segment aggregates (sequence-parallel scans): the carry kernel over all of the segment's
// chunks, then a fold into S_out [batch*dim] (sum of Delta) and h_out [batch*dim, dstate] (end
// state from zero). The workspace holds a.nchunks carries (scan_workspace_bytes(channels,
// a.nchunks + 1, dstate) bytes, split with scan_workspace_split the same way).
cudaError_t launch_scan_aggregate(const ScanArgs& a, float* S_out, float* h_out, cudaStream_t stream);
cudaError_t launch_scan_compose(const float* S, const float* b, const float* A, const float* h0, float* h_out,
                                int nseg, int batch, int dim, int dstate, cudaStream_t stream);
int scan_carry_resident_ctas_per_sm(bool bf16, int dstate);
int scan_carry_channels_per_cta(int dstate);

// State-space-duality layer: chunk length, workspace layout and launch.
int ssd_chunk_len();
size_t ssd_workspace_bytes(int batch, int nheads, int nchunks);
void ssd_workspace_split(void* ws, int batch, int nheads, int nchunks, SsdArgs& a);
cudaError_t launch_ssd(const SsdArgs& a, cudaStream_t stream);
// the forward chunk carries only (ws_S, ws_h for chunks 0 .. nchunks-2; no conv, forward time)
cudaError_t launch_scan_carry(const ScanArgs& a, cudaStream_t stream);
size_t scan_bwd_workspace_bytes(int batch, int dim, int seqlen, int nchunks);
void scan_bwd_workspace_split(void* ws, int batch, int dim, int seqlen, int nchunks, ScanBwdArgs& a);
int scan_bwd_resident_ctas_per_sm(bool bf16);
int scan_bwd_tile_steps();
int scan_bwd_channels_per_cta();
cudaError_t launch_scan_bwd(const ScanBwdArgs& a, cudaStream_t stream);
cudaError_t launch_conv(const ConvArgs& a, cudaStream_t stream);
size_t conv_bwd_workspace_bytes(int batch, int dim, int seqlen);
cudaError_t launch_conv_bwd(const ConvBwdArgs& a, cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

// Bounds-check error words of the debug build (ssm_bounds.cuh), one per translation unit;
// cudaErrorNotSupported without SSM_DEBUG_BOUNDS.
cudaError_t scan_bounds_flags(unsigned* out, bool clear);
cudaError_t decode_bounds_flags(unsigned* out, bool clear);
cudaError_t conv_bounds_flags(unsigned* out, bool clear);
cudaError_t scan_bwd_bounds_flags(unsigned* out, bool clear);
cudaError_t conv_bwd_bounds_flags(unsigned* out, bool clear);
cudaError_t ssd_bounds_flags(unsigned* out, bool clear);

}  // namespace ssm
