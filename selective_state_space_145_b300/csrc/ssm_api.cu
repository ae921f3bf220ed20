// ssm_api.cu -- the C ABI (include/ssm.h): host-side argument checks, the chunking policy
// and dispatch to the kernels. No device memory is allocated here and nothing is cached
// between calls except which kernels have had their shared-memory limit raised.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ssm.h"
#include "ssm_internal.h"

namespace {

using ssm::kChunkQuantum;
using ssm::kMaxConv;
using ssm::kMaxDstate;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int io_bytes(ssm_dtype io) { return io == SSM_BF16 ? 2 : 4; }

bool io_ok(ssm_dtype io) { return io == SSM_F32 || io == SSM_BF16; }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 148;
  }
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 148;
  }
  return n;
}

long long round_up(long long v, long long m) { return (v + m - 1) / m * m; }

// The default policy: how the main pass maps a channel onto lanes, and the chunk length.
// The scan is sequential in t within a CTA, so a problem with few channels leaves most SMs idle
// unless the sequence is split into chunks, and every chunk but the last costs a carry pass.
//  * N > 16: four lanes of 8 states per channel; chunks by the one-wave rule below.
//  * N <= 16 with enough channels that the main pass, at two lanes of 8 states per channel,
//    fills more than half a wave of resident CTAs: two lanes per channel, one chunk.
//  * otherwise the sequence is split, and the main pass takes one lane per channel with all 16
//    states, which keeps every per-channel value in registers: the one-wave rule splits only as
//    far as q chunks of CTAs still fit one wave (q times the CTAs, each walking 1/q of the
//    sequence; a second wave would cost as much as it saves).
// Once a sequence is split, chunks longer than kLongChunk are cut further: the extra waves of
// short chunks balance better than one wave of very long ones.
constexpr long long kLongChunk = 3072;  // a multiple of kChunkQuantum

struct ScanPlan {
  int lanes;
  int chunk_len;
};

long long scan_ctas(int batch, int dim, int lanes) {
  const int cpc = ssm::scan_channels_per_cta(lanes);
  return ((dim + cpc - 1) / cpc) * (long long)batch;
}

ScanPlan default_plan(int batch, int dim, int seqlen, int dstate, bool bf16) {
  const long long whole = round_up(seqlen > 0 ? seqlen : 1, kChunkQuantum);
  int lanes = dstate > 16 ? 4 : 2;
  long long ctas = scan_ctas(batch, dim, lanes);
  long long resident = (long long)sm_count() * ssm::scan_resident_ctas_per_sm(bf16, lanes);
  if (ctas <= 0 || 2 * ctas > resident) return {lanes, (int)whole};
  if (lanes == 2) {
    lanes = 1;
    ctas = scan_ctas(batch, dim, lanes);
    resident = (long long)sm_count() * ssm::scan_resident_ctas_per_sm(bf16, lanes);
  }
  long long q = resident / ctas;
  const long long qmax = (seqlen + kChunkQuantum - 1) / kChunkQuantum;
  if (q > qmax) q = qmax;
  if (q <= 1) return {lanes, (int)whole};
  const long long cl = round_up((seqlen + q - 1) / q, kChunkQuantum);
  return {lanes, (int)(cl > kLongChunk ? kLongChunk : cl)};
}

// Lanes per channel for a given chunking (N <= 16): whole channels per lane when the chunks'
// whole-channel CTAs are at least one per SM (chunked problems and problems with many
// channels), two lanes per channel otherwise: a tiny problem (say 64 channels, 256 steps) is
// bound by the serial work per lane, which two lanes of 8 states halve (20 against 30 us).
int lanes_for(int batch, int dim, int nchunks, int dstate) {
  if (dstate > 16) return 4;
  const long long w1 = scan_ctas(batch, dim, 1) * nchunks;
  if ((nchunks > 1 && w1 >= sm_count()) || w1 >= 4LL * sm_count()) return 1;
  return 2;
}

int default_chunk_len_impl(int batch, int dim, int seqlen, int dstate, bool bf16) {
  return default_plan(batch, dim, seqlen, dstate, bf16).chunk_len;
}

// Chunk length of the backward pass: as many chunks as fill one wave of the reverse kernel
// (its occupancy), in whole tiles of scan_bwd_tile_steps() steps and at least kBwdMinChunk steps.
constexpr int kBwdMinChunk = 32;
int bwd_chunk_len(int batch, int dim, int seqlen, bool bf16) {
  const int quantum = ssm::scan_bwd_tile_steps();
  const long long ctas = (long long)((dim + ssm::scan_bwd_channels_per_cta() - 1) / ssm::scan_bwd_channels_per_cta()) *
                         batch;
  const long long resident = (long long)sm_count() * ssm::scan_bwd_resident_ctas_per_sm(bf16);
  const long long whole = round_up(seqlen > 0 ? seqlen : 1, quantum);
  if (ctas <= 0 || 2 * ctas > resident) return (int)whole;
  long long q = resident / ctas;
  const long long qmax = (seqlen + kBwdMinChunk - 1) / kBwdMinChunk;
  if (q > qmax) q = qmax;
  if (q <= 1) return (int)whole;
  return (int)round_up((seqlen + q - 1) / q, quantum);
}

int nchunks_for(int seqlen, int chunk_len) {
  if (seqlen <= 0) return 1;
  return (int)((seqlen + (long long)chunk_len - 1) / chunk_len);
}

bool dims_ok(int batch, int dim, int seqlen, int dstate) {
  return batch >= 0 && dim >= 0 && seqlen >= 0 && dstate >= 1 && batch <= 65535;
}

}  // namespace

extern "C" {

int ssm_version(void) { return 200; }  // 0.2.0: reverse and ZOH flags, backward passes

const char* ssm_status_string(int status) {
  switch (status) {
    case SSM_OK: return "SSM_OK";
    case SSM_ERR_INVALID_ARG: return "SSM_ERR_INVALID_ARG";
    case SSM_ERR_UNSUPPORTED: return "SSM_ERR_UNSUPPORTED";
    case SSM_ERR_CUDA: return "SSM_ERR_CUDA";
    default: return "SSM_UNKNOWN_STATUS";
  }
}

int ssm_scan_default_chunk_len(int batch, int dim, int seqlen, int dstate, ssm_dtype io) {
  if (batch <= 0 || dim <= 0 || seqlen < 0) return kChunkQuantum;
  return default_chunk_len_impl(batch, dim, seqlen, dstate, io == SSM_BF16);
}

size_t ssm_scan_workspace_bytes(int batch, int dim, int seqlen, int dstate, int chunk_len, ssm_dtype io) {
  if (batch <= 0 || dim <= 0 || seqlen <= 0 || chunk_len < 0) return 0;
  int cl = chunk_len == 0 ? ssm_scan_default_chunk_len(batch, dim, seqlen, dstate, io)
                          : (int)round_up(chunk_len, kChunkQuantum);
  return ssm::scan_workspace_bytes((long long)batch * dim, nchunks_for(seqlen, cl), dstate);
}

ssm_status ssm_causal_conv1d_fwd(const void* x, const float* w, const float* bias, const void* conv_init, void* out,
                                 int batch, int dim, int seqlen, int d_conv, int apply_silu, ssm_dtype io,
                                 void* stream) {
  if (!io_ok(io)) return SSM_ERR_UNSUPPORTED;
  if (batch < 0 || dim < 0 || seqlen < 0) return SSM_ERR_INVALID_ARG;
  if (d_conv < 1) return SSM_ERR_INVALID_ARG;
  if (d_conv > kMaxConv) return SSM_ERR_UNSUPPORTED;
  if (apply_silu != 0 && apply_silu != 1) return SSM_ERR_INVALID_ARG;
  if ((long long)batch * dim == 0 || seqlen == 0) return SSM_OK;
  if (!x || !w || !out) return SSM_ERR_INVALID_ARG;
  const size_t es = io_bytes(io);
  if (!aligned(x, es) || !aligned(out, es) || !aligned(w, 4) || (bias && !aligned(bias, 4)) ||
      (conv_init && !aligned(conv_init, es)))
    return SSM_ERR_UNSUPPORTED;
  ssm::ConvArgs a;
  a.x = x; a.w = w; a.bias = bias; a.conv_init = conv_init; a.out = out;
  a.batch = batch; a.dim = dim; a.seqlen = seqlen; a.d_conv = d_conv; a.apply_silu = apply_silu;
  a.bf16 = io == SSM_BF16;
  a.vec = (seqlen % 4 == 0) && aligned(x, 16) && aligned(out, 16);
  return ssm::launch_conv(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status ssm_selective_scan_fwd(const void* x, const void* delta, const float* A, const void* B, const void* C,
                                  const float* D, const void* z, const float* delta_bias, int delta_softplus,
                                  const float* conv_w, const float* conv_b, int d_conv, const void* conv_init,
                                  const float* h0, void* out, float* h_last, void* conv_state_out, int batch,
                                  int dim, int seqlen, int dstate, ssm_dtype io, int chunk_len, void* workspace,
                                  size_t workspace_bytes, unsigned int flags, void* stream) {
  if (!io_ok(io)) return SSM_ERR_UNSUPPORTED;
  if (flags & ~(SSM_SCAN_REVERSE | SSM_SCAN_ZOH | SSM_SCAN_S4D_REAL)) return SSM_ERR_INVALID_ARG;
  if (!dims_ok(batch, dim, seqlen, dstate)) return SSM_ERR_INVALID_ARG;
  if (dstate > ssm::kMaxDstateScan) return SSM_ERR_UNSUPPORTED;
  if (delta_softplus != 0 && delta_softplus != 1) return SSM_ERR_INVALID_ARG;
  if (chunk_len < 0) return SSM_ERR_INVALID_ARG;
  const bool conv = conv_w != nullptr;
  if (conv || conv_init || conv_state_out) {
    if (d_conv < 1) return SSM_ERR_INVALID_ARG;
    if (d_conv > kMaxConv) return SSM_ERR_UNSUPPORTED;
  }
  if (!conv && (conv_b || conv_init)) return SSM_ERR_INVALID_ARG;
  if ((long long)batch * dim == 0) return SSM_OK;
  // per-token tensors may be NULL only when there are no tokens
  if (!A || (seqlen > 0 && (!x || !delta || !B || !C || !out))) return SSM_ERR_INVALID_ARG;
  const size_t es = io_bytes(io);
  const void* io_ptrs[] = {x, delta, B, C, z, out, conv_init, conv_state_out};
  for (const void* p : io_ptrs)
    if (p && !aligned(p, es)) return SSM_ERR_UNSUPPORTED;
  const void* f_ptrs[] = {A, D, delta_bias, conv_w, conv_b, h0, h_last};
  for (const void* p : f_ptrs)
    if (p && !aligned(p, 4)) return SSM_ERR_UNSUPPORTED;

  // chunking
  int cl;
  if (chunk_len == 0) {
    cl = default_chunk_len_impl(batch, dim, seqlen, dstate, io == SSM_BF16);
    // lower the chunk count until the given workspace suffices
    while (nchunks_for(seqlen, cl) > 1 &&
           ssm::scan_workspace_bytes((long long)batch * dim, nchunks_for(seqlen, cl), dstate) >
               (workspace ? workspace_bytes : 0)) {
      const int q = nchunks_for(seqlen, cl) - 1;
      cl = (int)round_up((seqlen + q - 1) / q, kChunkQuantum);
    }
  } else {
    if (chunk_len > (1 << 30)) chunk_len = 1 << 30;
    cl = (int)round_up(chunk_len, kChunkQuantum);
  }
  const int nchunks = nchunks_for(seqlen, cl);
  if (nchunks > 65535) return SSM_ERR_INVALID_ARG;
  // the zero-order-hold series roughly doubles an update's register and FMA work: two lanes of 8
  // states per channel run it faster than whole channels per lane (block fp32: 68 against 97 us;
  // level on the long scan)
  const int lanes = (flags & SSM_SCAN_ZOH) && dstate <= 16 ? 2 : lanes_for(batch, dim, nchunks, dstate);
  const size_t need = ssm::scan_workspace_bytes((long long)batch * dim, nchunks, dstate);
  if (need > 0) {
    if (!workspace || workspace_bytes < need) return SSM_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return SSM_ERR_UNSUPPORTED;
  }

  ssm::ScanArgs a;
  a.x = x; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.delta_bias = delta_bias;
  a.delta_softplus = delta_softplus; a.conv_w = conv_w; a.conv_b = conv_b; a.d_conv = d_conv;
  a.conv_init = conv_init; a.h0 = h0; a.out = out; a.h_last = h_last; a.conv_state_out = conv_state_out;
  a.batch = batch; a.dim = dim; a.seqlen = seqlen; a.dstate = dstate;
  a.bf16 = io == SSM_BF16;
  const bool rows16 = ((long long)seqlen * (long long)es) % 16 == 0;
  a.vec = rows16 && aligned(x, 16) && aligned(delta, 16) && aligned(B, 16) && aligned(C, 16) &&
          aligned(out, 16) && (!z || aligned(z, 16));
  a.chunk_len = cl;
  a.nchunks = nchunks;
  a.ws_chunks = nchunks - 1;
  a.lanes = lanes;
  a.reverse = (flags & SSM_SCAN_REVERSE) ? 1 : 0;
  a.zoh = (flags & SSM_SCAN_ZOH) ? 1 : 0;
  a.s4d = (flags & SSM_SCAN_S4D_REAL) && !(flags & SSM_SCAN_ZOH) ? 1 : 0;
  ssm::scan_workspace_split(workspace, (long long)batch * dim, nchunks, &a.ws_S, &a.ws_h);
  return ssm::launch_scan(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

// Chunking of a segment aggregate: as many chunks as one wave of carry CTAs holds, in
// multiples of kChunkQuantum, at most kLongChunk steps each.
int aggregate_chunk_len(int batch, int dim, int seqlen, int dstate, bool bf16) {
  const int cpc = ssm::scan_carry_channels_per_cta(dstate);
  const long long ctas = ((dim + cpc - 1) / cpc) * (long long)batch;
  const long long resident = (long long)sm_count() * ssm::scan_carry_resident_ctas_per_sm(bf16, dstate);
  long long q = ctas > 0 ? resident / ctas : 1;
  const long long qmax = (seqlen + kChunkQuantum - 1) / kChunkQuantum;
  if (q > qmax) q = qmax;
  if (q < 1) q = 1;
  const long long cl = round_up((seqlen + q - 1) / q, kChunkQuantum);
  return (int)(cl > kLongChunk ? kLongChunk : cl);
}

size_t ssm_scan_aggregate_workspace_bytes(int batch, int dim, int seqlen, int dstate, ssm_dtype io) {
  if (batch <= 0 || dim <= 0 || seqlen <= 0 || dstate < 1) return 0;
  const int cl = aggregate_chunk_len(batch, dim, seqlen, dstate, io == SSM_BF16);
  return ssm::scan_workspace_bytes((long long)batch * dim, nchunks_for(seqlen, cl) + 1, dstate);
}

ssm_status ssm_selective_scan_aggregate(const void* x, const void* delta, const float* A, const void* B,
                                        const float* delta_bias, int delta_softplus, const float* conv_w,
                                        const float* conv_b, int d_conv, const void* conv_init, float* S_out,
                                        float* h_out, int batch, int dim, int seqlen, int dstate, ssm_dtype io,
                                        void* workspace, size_t workspace_bytes, unsigned int flags, void* stream) {
  if (!io_ok(io)) return SSM_ERR_UNSUPPORTED;
  if (flags & ~(SSM_SCAN_REVERSE | SSM_SCAN_ZOH)) return SSM_ERR_INVALID_ARG;
  if (!dims_ok(batch, dim, seqlen, dstate)) return SSM_ERR_INVALID_ARG;
  if (dstate > ssm::kMaxDstateScan) return SSM_ERR_UNSUPPORTED;
  if (delta_softplus != 0 && delta_softplus != 1) return SSM_ERR_INVALID_ARG;
  const bool conv = conv_w != nullptr;
  if (conv || conv_init) {
    if (d_conv < 1) return SSM_ERR_INVALID_ARG;
    if (d_conv > kMaxConv) return SSM_ERR_UNSUPPORTED;
  }
  if (!conv && (conv_b || conv_init)) return SSM_ERR_INVALID_ARG;
  if ((long long)batch * dim == 0) return SSM_OK;
  if (!A || !S_out || !h_out || (seqlen > 0 && (!x || !delta || !B))) return SSM_ERR_INVALID_ARG;
  const size_t es = io_bytes(io);
  const void* io_ptrs[] = {x, delta, B, conv_init};
  for (const void* p : io_ptrs)
    if (p && !aligned(p, es)) return SSM_ERR_UNSUPPORTED;
  const void* f_ptrs[] = {A, delta_bias, conv_w, conv_b, S_out, h_out};
  for (const void* p : f_ptrs)
    if (p && !aligned(p, 4)) return SSM_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long BD = (long long)batch * dim;
  if (seqlen == 0) {  // no tokens: nothing decays and nothing enters
    if (cudaMemsetAsync(S_out, 0, BD * sizeof(float), st) != cudaSuccess ||
        cudaMemsetAsync(h_out, 0, BD * dstate * sizeof(float), st) != cudaSuccess)
      return SSM_ERR_CUDA;
    return SSM_OK;
  }
  const int cl = aggregate_chunk_len(batch, dim, seqlen, dstate, io == SSM_BF16);
  const int nchunks = nchunks_for(seqlen, cl);
  if (nchunks > 65535) return SSM_ERR_INVALID_ARG;
  const size_t need = ssm::scan_workspace_bytes(BD, nchunks + 1, dstate);
  if (!workspace || workspace_bytes < need) return SSM_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return SSM_ERR_UNSUPPORTED;
  ssm::ScanArgs a{};
  a.x = x; a.delta = delta; a.A = A; a.B = B; a.C = nullptr; a.D = nullptr; a.z = nullptr;
  a.delta_bias = delta_bias; a.delta_softplus = delta_softplus; a.conv_w = conv_w; a.conv_b = conv_b;
  a.d_conv = d_conv; a.conv_init = conv_init; a.h0 = nullptr; a.out = nullptr; a.h_last = nullptr;
  a.conv_state_out = nullptr;
  a.batch = batch; a.dim = dim; a.seqlen = seqlen; a.dstate = dstate; a.bf16 = io == SSM_BF16;
  const bool rows16 = ((long long)seqlen * (long long)es) % 16 == 0;
  a.vec = rows16 && aligned(x, 16) && aligned(delta, 16) && aligned(B, 16);
  a.chunk_len = cl;
  a.nchunks = nchunks;
  a.ws_chunks = nchunks;
  a.lanes = 1;
  a.reverse = (flags & SSM_SCAN_REVERSE) ? 1 : 0;
  a.zoh = (flags & SSM_SCAN_ZOH) ? 1 : 0;
  ssm::scan_workspace_split(workspace, BD, nchunks + 1, &a.ws_S, &a.ws_h);
  return ssm::launch_scan_aggregate(a, S_out, h_out, st) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status ssm_scan_compose(const float* S, const float* b, const float* A, const float* h0, float* h_out, int nseg,
                            int batch, int dim, int dstate, void* stream) {
  if (nseg < 0 || batch < 0 || dim < 0 || dstate < 1) return SSM_ERR_INVALID_ARG;
  if (dstate > ssm::kMaxDstateScan) return SSM_ERR_UNSUPPORTED;
  if ((long long)batch * dim == 0) return SSM_OK;
  if (!A || !h_out || (nseg > 0 && (!S || !b))) return SSM_ERR_INVALID_ARG;
  const void* f_ptrs[] = {S, b, A, h0, h_out};
  for (const void* p : f_ptrs)
    if (p && !aligned(p, 4)) return SSM_ERR_UNSUPPORTED;
  return ssm::launch_scan_compose(S, b, A, h0, h_out, nseg, batch, dim, dstate, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? SSM_OK
             : SSM_ERR_CUDA;
}

ssm_status ssm_selective_state_update(float* state, void* conv_state, const void* x, const void* delta,
                                      const float* A, const void* B, const void* C, const float* D, const void* z,
                                      const float* delta_bias, int delta_softplus, const float* conv_w,
                                      const float* conv_b, int d_conv, void* y, int batch, int dim, int dstate,
                                      ssm_dtype io, unsigned int flags, void* stream) {
  if (!io_ok(io)) return SSM_ERR_UNSUPPORTED;
  if (flags & ~SSM_SCAN_ZOH) return SSM_ERR_INVALID_ARG;
  if (batch < 0 || dim < 0 || dstate < 1) return SSM_ERR_INVALID_ARG;
  if (dstate > ssm::kMaxDstateScan) return SSM_ERR_UNSUPPORTED;
  if (delta_softplus != 0 && delta_softplus != 1) return SSM_ERR_INVALID_ARG;
  const bool conv = conv_w != nullptr;
  if (conv) {
    if (d_conv < 1) return SSM_ERR_INVALID_ARG;
    if (d_conv > kMaxConv) return SSM_ERR_UNSUPPORTED;
    if (d_conv > 1 && !conv_state) return SSM_ERR_INVALID_ARG;
  } else if (conv_b) {
    return SSM_ERR_INVALID_ARG;
  }
  if ((long long)batch * dim == 0) return SSM_OK;
  if (!state || !x || !delta || !A || !B || !C || !y) return SSM_ERR_INVALID_ARG;
  const size_t es = io_bytes(io);
  const void* io_ptrs[] = {x, delta, B, C, z, y, conv ? conv_state : nullptr};
  for (const void* p : io_ptrs)
    if (p && !aligned(p, es)) return SSM_ERR_UNSUPPORTED;
  const void* f_ptrs[] = {state, A, D, delta_bias, conv_w, conv_b};
  for (const void* p : f_ptrs)
    if (p && !aligned(p, 4)) return SSM_ERR_UNSUPPORTED;
  ssm::DecodeArgs a;
  a.state = state; a.conv_state = conv ? conv_state : nullptr; a.x = x; a.delta = delta; a.A = A; a.B = B;
  a.C = C; a.D = D; a.z = z; a.delta_bias = delta_bias; a.delta_softplus = delta_softplus;
  a.conv_w = conv_w; a.conv_b = conv_b; a.d_conv = conv ? d_conv : 0; a.y = y;
  a.batch = batch; a.dim = dim; a.dstate = dstate; a.bf16 = io == SSM_BF16;
  a.zoh = (flags & SSM_SCAN_ZOH) ? 1 : 0;
  return ssm::launch_decode(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

size_t ssm_scan_bwd_workspace_bytes(int batch, int dim, int seqlen, int dstate, ssm_dtype io) {
  (void)dstate;
  if (batch <= 0 || dim <= 0 || seqlen < 0) return 0;
  const int cl = bwd_chunk_len(batch, dim, seqlen, io == SSM_BF16);
  return ssm::scan_bwd_workspace_bytes(batch, dim, seqlen, nchunks_for(seqlen, cl));
}

ssm_status ssm_selective_scan_bwd(const void* u, const void* delta, const float* A, const void* B, const void* C,
                                  const float* D, const void* z, const float* delta_bias, int delta_softplus,
                                  const float* h0, const void* dout, const float* dh_last, void* du, void* ddelta,
                                  void* dz, float* dA, float* dB, float* dC, float* dD, float* ddelta_bias,
                                  float* dh0, int batch, int dim, int seqlen, int dstate, ssm_dtype io,
                                  void* workspace, size_t workspace_bytes, unsigned int flags, void* stream) {
  if (!io_ok(io)) return SSM_ERR_UNSUPPORTED;
  if (flags & ~(SSM_SCAN_REVERSE | SSM_SCAN_ZOH)) return SSM_ERR_INVALID_ARG;
  if (flags) return SSM_ERR_UNSUPPORTED;  // the backward pass covers the forward-time Euler scan
  if (!dims_ok(batch, dim, seqlen, dstate)) return SSM_ERR_INVALID_ARG;
  if (dstate > kMaxDstate) return SSM_ERR_UNSUPPORTED;
  if (delta_softplus != 0 && delta_softplus != 1) return SSM_ERR_INVALID_ARG;
  if ((long long)batch * dim == 0) return SSM_OK;
  if (!A || !dA) return SSM_ERR_INVALID_ARG;
  if (seqlen > 0 && (!u || !delta || !B || !C || !dout || !du || !ddelta || !dB || !dC))
    return SSM_ERR_INVALID_ARG;
  if (z && seqlen > 0 && !dz) return SSM_ERR_INVALID_ARG;
  const size_t es = io_bytes(io);
  const void* io_ptrs[] = {u, delta, B, C, z, dout, du, ddelta, dz};
  for (const void* p : io_ptrs)
    if (p && !aligned(p, es)) return SSM_ERR_UNSUPPORTED;
  const void* f_ptrs[] = {A, D, delta_bias, h0, dh_last, dA, dB, dC, dD, ddelta_bias, dh0};
  for (const void* p : f_ptrs)
    if (p && !aligned(p, 4)) return SSM_ERR_UNSUPPORTED;
  // time is cut into chunks when the channels alone leave SMs idle (as in the forward pass)
  const int cl = bwd_chunk_len(batch, dim, seqlen, io == SSM_BF16);
  const int nchunks = nchunks_for(seqlen, cl);
  if (nchunks > 65535) return SSM_ERR_INVALID_ARG;
  const size_t need = ssm::scan_bwd_workspace_bytes(batch, dim, seqlen, nchunks);
  if (!workspace || workspace_bytes < need) return SSM_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return SSM_ERR_UNSUPPORTED;
  ssm::ScanBwdArgs a;
  a.u = u; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.delta_bias = delta_bias;
  a.delta_softplus = delta_softplus; a.h0 = h0; a.dout = dout; a.dh_last = dh_last;
  a.du = du; a.ddelta = ddelta; a.dz = dz; a.dA = dA; a.dB = dB; a.dC = dC; a.dD = dD;
  a.ddelta_bias = ddelta_bias; a.dh0 = dh0;
  a.batch = batch; a.dim = dim; a.seqlen = seqlen; a.dstate = dstate; a.bf16 = io == SSM_BF16;
  bool vec = ((long long)seqlen * (long long)es) % 16 == 0;
  const void* vec_ptrs[] = {u, delta, B, C, z, dout, du, ddelta, dz};
  for (const void* p : vec_ptrs)
    if (p && !aligned(p, 16)) vec = false;
  a.vec = vec;
  a.chunk_len = cl;
  a.nchunks = nchunks;
  ssm::scan_bwd_workspace_split(workspace, batch, dim, seqlen, nchunks, a);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return ssm::launch_scan_bwd(a, st) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

size_t ssm_conv_bwd_workspace_bytes(int batch, int dim, int seqlen, int d_conv, ssm_dtype io) {
  (void)d_conv;
  (void)io;
  if (batch <= 0 || dim <= 0 || seqlen < 0) return 0;
  return ssm::conv_bwd_workspace_bytes(batch, dim, seqlen);
}

ssm_status ssm_causal_conv1d_bwd(const void* x, const float* w, const float* bias, const void* conv_init,
                                 const void* dout, int apply_silu, void* dx, float* dw, float* dbias,
                                 void* dconv_init, int batch, int dim, int seqlen, int d_conv, ssm_dtype io,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  if (!io_ok(io)) return SSM_ERR_UNSUPPORTED;
  if (batch < 0 || dim < 0 || seqlen < 0) return SSM_ERR_INVALID_ARG;
  if (d_conv < 1) return SSM_ERR_INVALID_ARG;
  if (d_conv > kMaxConv) return SSM_ERR_UNSUPPORTED;
  if (apply_silu != 0 && apply_silu != 1) return SSM_ERR_INVALID_ARG;
  if ((long long)batch * dim == 0) return SSM_OK;
  if (!w || !dw) return SSM_ERR_INVALID_ARG;
  if (seqlen > 0 && (!x || !dout || !dx)) return SSM_ERR_INVALID_ARG;
  const size_t es = io_bytes(io);
  const void* io_ptrs[] = {x, conv_init, dout, dx, dconv_init};
  for (const void* p : io_ptrs)
    if (p && !aligned(p, es)) return SSM_ERR_UNSUPPORTED;
  const void* f_ptrs[] = {w, bias, dw, dbias};
  for (const void* p : f_ptrs)
    if (p && !aligned(p, 4)) return SSM_ERR_UNSUPPORTED;
  const size_t need = ssm::conv_bwd_workspace_bytes(batch, dim, seqlen);
  if (!workspace || workspace_bytes < need) return SSM_ERR_INVALID_ARG;
  if (!aligned(workspace, 16)) return SSM_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (seqlen == 0 && dconv_init && d_conv > 1) {
    // no step reaches the window: its gradient is zero
    if (cudaMemsetAsync(dconv_init, 0, (size_t)batch * dim * (d_conv - 1) * es, st) != cudaSuccess)
      return SSM_ERR_CUDA;
  }
  ssm::ConvBwdArgs a;
  a.x = x; a.w = w; a.bias = bias; a.conv_init = conv_init; a.dout = dout; a.dx = dx; a.dw = dw; a.dbias = dbias;
  a.dconv_init = d_conv > 1 ? dconv_init : nullptr;
  a.batch = batch; a.dim = dim; a.seqlen = seqlen; a.d_conv = d_conv; a.apply_silu = apply_silu;
  a.bf16 = io == SSM_BF16;
  a.ws_part = static_cast<float*>(workspace);
  return ssm::launch_conv_bwd(a, st) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

size_t ssm_ssd_workspace_bytes(int batch, int seqlen, int nheads, int headdim, int dstate, ssm_dtype io) {
  if (batch <= 0 || seqlen <= 0 || nheads <= 0 || headdim != 64 || dstate != 128 || io != SSM_BF16) return 0;
  const int q = ssm::ssd_chunk_len();
  return ssm::ssd_workspace_bytes(batch, nheads, (int)(((long long)seqlen + q - 1) / q));
}

ssm_status ssm_ssd_fwd(const void* x, const void* dt, const float* A, const void* B, const void* C, const float* D,
                       const float* dt_bias, int dt_softplus, const float* h0, void* y, float* h_last, int batch,
                       int seqlen, int nheads, int headdim, int dstate, ssm_dtype io, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (!io_ok(io)) return SSM_ERR_UNSUPPORTED;
  if (batch < 0 || seqlen < 0 || nheads < 0 || headdim < 1 || dstate < 1) return SSM_ERR_INVALID_ARG;
  if (dt_softplus != 0 && dt_softplus != 1) return SSM_ERR_INVALID_ARG;
  if (io != SSM_BF16 || headdim != 64 || dstate != 128) return SSM_ERR_UNSUPPORTED;
  if (batch > 65535 || nheads > 65535) return SSM_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((long long)batch * nheads == 0) return SSM_OK;
  const size_t state_bytes = (size_t)batch * nheads * headdim * dstate * sizeof(float);
  if (seqlen == 0) {  // no tokens: the final state is the initial one
    if (!h_last) return SSM_OK;
    const cudaError_t e = h0 ? cudaMemcpyAsync(h_last, h0, state_bytes, cudaMemcpyDeviceToDevice, st)
                             : cudaMemsetAsync(h_last, 0, state_bytes, st);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
  }
  if (!x || !dt || !A || !B || !C || !y) return SSM_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(y, 16) || !aligned(dt, 2) ||
      !aligned(A, 4) || (D && !aligned(D, 4)) || (dt_bias && !aligned(dt_bias, 4)) || (h0 && !aligned(h0, 4)) ||
      (h_last && !aligned(h_last, 4)))
    return SSM_ERR_UNSUPPORTED;
  const int q = ssm::ssd_chunk_len();
  const long long nchunks = ((long long)seqlen + q - 1) / q;
  if (nchunks > (1LL << 30)) return SSM_ERR_INVALID_ARG;
  const size_t need = ssm::ssd_workspace_bytes(batch, nheads, (int)nchunks);
  if (!workspace || workspace_bytes < need) return SSM_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return SSM_ERR_UNSUPPORTED;
  ssm::SsdArgs a;
  a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.dt_bias = dt_bias; a.dt_softplus = dt_softplus;
  a.h0 = h0; a.y = y; a.h_last = h_last;
  a.batch = batch; a.seqlen = seqlen; a.nheads = nheads; a.nchunks = (int)nchunks;
  ssm::ssd_workspace_split(workspace, batch, nheads, (int)nchunks, a);
  return ssm::launch_ssd(a, st) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status ssm_debug_bounds_status(unsigned int* flags_out, int clear) {
  if (!flags_out || (clear != 0 && clear != 1)) return SSM_ERR_INVALID_ARG;
  unsigned scan = 0, decode = 0, conv = 0, bwd = 0, cbwd = 0, ssd = 0;
  cudaError_t e = ssm::scan_bounds_flags(&scan, clear != 0);
  if (e == cudaErrorNotSupported) return SSM_ERR_UNSUPPORTED;  // a release build: no checks compiled in
  if (e == cudaSuccess) e = ssm::decode_bounds_flags(&decode, clear != 0);
  if (e == cudaSuccess) e = ssm::conv_bounds_flags(&conv, clear != 0);
  if (e == cudaSuccess) e = ssm::scan_bwd_bounds_flags(&bwd, clear != 0);
  if (e == cudaSuccess) e = ssm::conv_bwd_bounds_flags(&cbwd, clear != 0);
  if (e == cudaSuccess) e = ssm::ssd_bounds_flags(&ssd, clear != 0);
  if (e != cudaSuccess) return SSM_ERR_CUDA;
  *flags_out = scan | decode | conv | bwd | cbwd | ssd;
  return SSM_OK;
}

}  // extern "C"
