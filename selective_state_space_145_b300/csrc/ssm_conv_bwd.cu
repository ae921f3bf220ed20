// ssm_conv_bwd.cu -- backward of the causal depthwise conv1d (+ SiLU) prologue (training).
//
// Forward ("Overview of Mamba (SSM) Model", "How the Mamba Block Works": a depthwise
// convolution and SiLU in front of the SSM):
//   acc_t = sum_{k<K} w[d,k] xs(t-(K-1)+k) + bias[d],  out_t = silu(acc_t) (or acc_t),
//   xs(s) = x[s] for s >= 0, the window (conv_init) for s < 0.
// The chain rule gives, from dout = dL/dout,
//   dacc_t = dout_t silu'(acc_t),  silu'(a) = s(a) (1 + a (1 - s(a)))  (or dout_t)
//   dx[s] = sum_k w[k] dacc_{s+(K-1)-k};  dwindow likewise for s < 0
//   dw[d,k] = sum_{b,t} dacc_t xs(t-(K-1)+k);  dbias[d] = sum_{b,t} dacc_t.
//
// Design. A block takes 1024 consecutive steps of one row; one thread owns 16 bytes of each
// input row: 8 steps (bf16, 128 threads) or 4 (fp32, 256 threads). The block stages x at its
// steps (plus a 4-step halo on each side) and then dacc at its steps (plus the 3 that follow)
// in shared memory, so every activation is computed once: each thread computes acc and dacc at
// its own steps, and one thread adds the 3 steps past the block. dx at a step takes the 4 dacc
// values that reach it from the staged row. Rows whose length is a multiple of the thread's
// steps at 16-byte aligned addresses move them with one 16-byte load or store. Each thread
// adds the dw / dbias terms of its own steps; the block reduces them and writes one partial,
// and a second kernel sums the partials over sequences and segments in a fixed order. The conv
// taps are zero-padded to 4 (w[4-K+k] holds tap k).
#include "ssm_bounds.cuh"
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kCBSeg = 1024;             // steps per block
constexpr int kCBMaxThreads = 256;
constexpr int kCBPart = kMaxConv + 1;    // partial: dw taps (padded) + dbias
static_assert(kMaxConv == 4, "the staged halos hold 4 steps");

template <typename T>
struct CBGeo {
  static constexpr int kSpt = 16 / (int)sizeof(T);   // steps per thread: one 16-byte piece
  static constexpr int kThreads = kCBSeg / kSpt;
};

// VEC: the row length is a multiple of the thread's steps and x, dout, dx are 16-byte aligned.
template <typename T, bool VEC>
__global__ void __launch_bounds__(kCBMaxThreads) conv_bwd_kernel(const ConvBwdArgs a, int nseg) {
  constexpr int kCBSpt = CBGeo<T>::kSpt;
  constexpr int kCBThreads = CBGeo<T>::kThreads;
  __shared__ float red[kCBThreads / 32][kCBPart];
  __shared__ __align__(16) float sx[kCBSeg + 8];   // x at steps base-4 .. base+kCBSeg+3
  __shared__ __align__(16) float sda[kCBSeg + 4];  // dacc at steps base .. base+kCBSeg+3
  const int L = a.seqlen, K = a.d_conv;
  const long long c = blockIdx.x / nseg;          // channel row b * dim + d
  const int seg = blockIdx.x % nseg;
  const int d = (int)(c % a.dim);
  const int tid = threadIdx.x;
  const int base = seg * kCBSeg;
  const int s0 = base + tid * kCBSpt;             // this thread's steps
  const T* __restrict__ x = static_cast<const T*>(a.x) + c * L;
  const T* __restrict__ dout = static_cast<const T*>(a.dout) + c * L;
  const T* win = a.conv_init ? static_cast<const T*>(a.conv_init) + c * (K - 1) : nullptr;
  // debug build: the block's row, window row, taps and partial slot lie inside their tensors
  // (the test is uniform over the block, so a skipped block skips its barriers as a whole)
  {
    const long long rows = (long long)a.batch * a.dim;
    if (!in_bounds(c * L, L, rows * L, kBoundsConv) || !in_bounds((long long)d * K, K, (long long)a.dim * K, kBoundsConv) ||
        !in_bounds(c * (K - 1), K - 1, rows * (K - 1), kBoundsConv) ||
        !in_bounds(((long long)c * nseg + seg) * kCBPart, kCBPart, rows * nseg * kCBPart, kBoundsConv))
      return;
  }

  float wp[kMaxConv];
#pragma unroll
  for (int i = 0; i < kMaxConv; ++i) {
    const int k = i - (kMaxConv - K);  // tap k sits at padded slot i
    wp[i] = k >= 0 ? a.w[(long long)d * K + k] : 0.f;
  }
  const float cb = a.bias ? a.bias[d] : 0.f;
  auto xs = [&](int s) -> float {
    if (s >= L) return 0.f;
    if (s >= 0) return to_f32(x[s]);
    return (win && s >= -(K - 1)) ? to_f32(win[(K - 1) + s]) : 0.f;
  };
  // dacc at step t from the staged x at t-3 .. t (xw) and dout_t (zero past L)
  auto dacc = [&](int t, const float* xw, float g) -> float {
    if (t >= L) return 0.f;
    float acc = cb;
#pragma unroll
    for (int i = 0; i < kMaxConv; ++i) acc = fmaf(wp[i], xw[i], acc);
    if (a.apply_silu) {
      const float sg = rcp_approx(1.0f + ex2_approx(-acc * kLog2e));
      g *= sg * fmaf(acc, 1.0f - sg, 1.0f);
    }
    return g;
  };

  // ---- stage x; own steps from registers, the halos from one warp
  float xo[kCBSpt], go[kCBSpt];
  if (VEC && s0 < L) {
    if constexpr (kCBSpt == 8) {
      load8(x + s0, xo);
      load8(dout + s0, go);
    } else {
      load4(x + s0, xo);
      load4(dout + s0, go);
    }
  } else {
#pragma unroll
    for (int j = 0; j < kCBSpt; ++j) {
      const bool in = s0 + j < L;
      xo[j] = in ? to_f32(x[s0 + j]) : 0.f;
      go[j] = in ? to_f32(dout[s0 + j]) : 0.f;
    }
  }
#pragma unroll
  for (int j = 0; j < kCBSpt; j += 4)
    *reinterpret_cast<float4*>(&sx[4 + kCBSpt * tid + j]) = make_float4(xo[j], xo[j + 1], xo[j + 2], xo[j + 3]);
  if (tid < 4) sx[tid] = xs(base - 4 + tid);
  else if (tid < 8) sx[kCBSeg + tid] = xs(base + kCBSeg + tid - 4);
  __syncthreads();

  // ---- dacc at the own steps; x at s0-4 .. s0-1 is sx[kCBSpt tid .. kCBSpt tid + 3]
  float xv[kCBSpt + 4];
  {
    const float4 p = *reinterpret_cast<const float4*>(&sx[kCBSpt * tid]);
    xv[0] = p.x; xv[1] = p.y; xv[2] = p.z; xv[3] = p.w;
#pragma unroll
    for (int j = 0; j < kCBSpt; ++j) xv[4 + j] = xo[j];
  }
  float da[kCBSpt];
#pragma unroll
  for (int j = 0; j < kCBSpt; ++j) da[j] = dacc(s0 + j, xv + j + 1, go[j]);
#pragma unroll
  for (int j = 0; j < kCBSpt; j += 4)
    *reinterpret_cast<float4*>(&sda[kCBSpt * tid + j]) = make_float4(da[j], da[j + 1], da[j + 2], da[j + 3]);
  if (tid == kCBThreads - 1) {
    // the 3 steps past the block reach its last dx values
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int t = base + kCBSeg + j;
      sda[kCBSeg + j] = dacc(t, &sx[kCBSeg + 1 + j], t < L ? to_f32(dout[t]) : 0.f);
    }
    sda[kCBSeg + 3] = 0.f;
  }
  __syncthreads();

  // ---- dx at the own steps: dx[s] = sum_i wp[i] dacc_{s+3-i}; dacc at s0 .. s0+kCBSpt+2
  float dn[kCBSpt + 4];
  {
    const float4 q = *reinterpret_cast<const float4*>(&sda[kCBSpt * tid + kCBSpt]);
#pragma unroll
    for (int j = 0; j < kCBSpt; ++j) dn[j] = da[j];
    dn[kCBSpt] = q.x; dn[kCBSpt + 1] = q.y; dn[kCBSpt + 2] = q.z; dn[kCBSpt + 3] = q.w;
  }
  float dxv[kCBSpt];
#pragma unroll
  for (int j = 0; j < kCBSpt; ++j) {
    float v = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxConv; ++i) v = fmaf(wp[i], dn[j + 3 - i], v);
    dxv[j] = v;
  }
  T* dx = static_cast<T*>(a.dx) + c * L;
  if (VEC && s0 < L) {
    if constexpr (kCBSpt == 8) {
      store8(dx + s0, dxv);
    } else {
      store4(dx + s0, dxv);
    }
  } else {
#pragma unroll
    for (int j = 0; j < kCBSpt; ++j)
      if (s0 + j < L) dx[s0 + j] = from_f32<T>(dxv[j]);
  }
  // window gradient: positions -(K-1) .. -1, reached by dacc_0 .. dacc_{K-2}
  if (s0 == 0 && a.dconv_init && K > 1) {
    T* dw_out = static_cast<T*>(a.dconv_init) + c * (K - 1);
    for (int j = 0; j < K - 1; ++j) {
      const int s = j - (K - 1);
      float v = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxConv; ++i) {
        const int t = s + 3 - i;
        if (t >= 0 && t < L) v = fmaf(wp[i], dn[t], v);
      }
      dw_out[j] = from_f32<T>(v);
    }
  }
  // this thread's dw / dbias terms (its own 8 steps only)
  float part[kCBPart];
#pragma unroll
  for (int i = 0; i < kCBPart; ++i) part[i] = 0.f;
#pragma unroll
  for (int j = 0; j < kCBSpt; ++j) {
#pragma unroll
    for (int i = 0; i < kMaxConv; ++i) part[i] = fmaf(da[j], xv[j + 1 + i], part[i]);
    part[kMaxConv] += da[j];
  }
  // block reduction (fixed order): warp shuffles, then warp 0 over the warps
#pragma unroll
  for (int i = 0; i < kCBPart; ++i)
    for (int o = 16; o > 0; o >>= 1) part[i] += __shfl_xor_sync(0xffffffffu, part[i], o);
  const int lane = tid % 32, warp = tid / 32;
  if (lane == 0)
#pragma unroll
    for (int i = 0; i < kCBPart; ++i) red[warp][i] = part[i];
  __syncthreads();
  if (tid < kCBPart) {
    float sum = 0.f;
    for (int w = 0; w < kCBThreads / 32; ++w) sum += red[w][tid];
    a.ws_part[((long long)c * nseg + seg) * kCBPart + tid] = sum;
  }
}

// dw[d, k] and dbias[d]: sums of the partials of every sequence and segment of channel d
__global__ void conv_bwd_reduce_kernel(const ConvBwdArgs a, int nseg) {
  const int K = a.d_conv;
  const int total = a.dim * (K + 1);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int d = i / (K + 1), k = i % (K + 1);
    const int slot = k < K ? kMaxConv - K + k : kMaxConv;  // padded tap, or dbias
    float s = 0.f;
    const long long nparts = (long long)a.batch * a.dim * nseg * kCBPart;
    for (int b = 0; b < a.batch; ++b)
      for (int g = 0; g < nseg; ++g) {
        const long long j = (((long long)b * a.dim + d) * nseg + g) * kCBPart + slot;
        if (in_bounds(j, 1, nparts, kBoundsConv)) s += a.ws_part[j];
      }
    if (k < K) a.dw[(long long)d * K + k] = s;
    else if (a.dbias) a.dbias[d] = s;
  }
}

template <typename T>
cudaError_t launch_conv_bwd_t(const ConvBwdArgs& a, cudaStream_t stream) {
  const int nseg = (a.seqlen + kCBSeg - 1) / kCBSeg;
  const long long blocks = (long long)a.batch * a.dim * nseg;
  if (blocks > 0) {
    const uintptr_t vb = 16;
    const bool vec = a.seqlen % CBGeo<T>::kSpt == 0 && reinterpret_cast<uintptr_t>(a.x) % vb == 0 &&
                     reinterpret_cast<uintptr_t>(a.dout) % vb == 0 && reinterpret_cast<uintptr_t>(a.dx) % vb == 0;
    if (vec)
      conv_bwd_kernel<T, true><<<(unsigned)blocks, CBGeo<T>::kThreads, 0, stream>>>(a, nseg);
    else
      conv_bwd_kernel<T, false><<<(unsigned)blocks, CBGeo<T>::kThreads, 0, stream>>>(a, nseg);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  const int total = a.dim * (a.d_conv + 1);
  conv_bwd_reduce_kernel<<<(total + 255) / 256, 256, 0, stream>>>(a, nseg);
  return cudaGetLastError();
}

}  // namespace

size_t conv_bwd_workspace_bytes(int batch, int dim, int seqlen) {
  const long long nseg = (seqlen + kCBSeg - 1) / kCBSeg;
  return (size_t)((long long)batch * dim * (nseg > 0 ? nseg : 1) * kCBPart * sizeof(float));
}

cudaError_t launch_conv_bwd(const ConvBwdArgs& a, cudaStream_t stream) {
  if (a.bf16) return launch_conv_bwd_t<__nv_bfloat16>(a, stream);
  return launch_conv_bwd_t<float>(a, stream);
}

cudaError_t conv_bwd_bounds_flags(unsigned* out, bool clear) {
#ifdef SSM_DEBUG_BOUNDS
  return bounds_flags_read(out, clear);
#else
  (void)out;
  (void)clear;
  return cudaErrorNotSupported;
#endif
}

}  // namespace ssm
