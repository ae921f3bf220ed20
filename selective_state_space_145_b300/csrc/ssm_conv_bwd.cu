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
// Design. One thread owns 4 consecutive positions s of one row: it recomputes acc and dacc at
// the K+3 steps that reach them, writes dx for its 4 positions, and adds the dw / dbias terms
// of its own 4 steps. A block (1024 steps of one row) reduces those terms and writes one
// partial; a second kernel sums the partials over sequences and segments in a fixed order.
// The conv taps are zero-padded to 4 (w[4-K+k] holds tap k).
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kCBThreads = 256;
constexpr int kCBSeg = kCBThreads * 4;   // steps per block
constexpr int kCBPart = kMaxConv + 1;    // partial: dw taps (padded) + dbias

template <typename T>
__global__ void __launch_bounds__(kCBThreads) conv_bwd_kernel(const ConvBwdArgs a, int nseg) {
  __shared__ float red[kCBThreads / 32][kCBPart];
  const int L = a.seqlen, K = a.d_conv;
  const long long c = blockIdx.x / nseg;          // channel row b * dim + d
  const int seg = blockIdx.x % nseg;
  const int d = (int)(c % a.dim);
  const int s0 = seg * kCBSeg + threadIdx.x * 4;  // this thread's 4 positions
  const T* __restrict__ x = static_cast<const T*>(a.x) + c * L;
  const T* __restrict__ dout = static_cast<const T*>(a.dout) + c * L;
  const T* win = a.conv_init ? static_cast<const T*>(a.conv_init) + c * (K - 1) : nullptr;

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

  // x at s0-3 .. s0+6, dacc at s0 .. s0+6 (zero past L)
  float xv[10];
#pragma unroll
  for (int j = 0; j < 10; ++j) xv[j] = xs(s0 - 3 + j);
  float da[7];
#pragma unroll
  for (int j = 0; j < 7; ++j) {
    const int t = s0 + j;
    float g = 0.f;
    if (t < L) {
      float acc = cb;
#pragma unroll
      for (int i = 0; i < kMaxConv; ++i) acc = fmaf(wp[i], xv[j + i], acc);
      g = to_f32(dout[t]);
      if (a.apply_silu) {
        const float sg = rcp_approx(1.0f + ex2_approx(-acc * kLog2e));
        g *= sg * fmaf(acc, 1.0f - sg, 1.0f);
      }
    }
    da[j] = g;
  }
  // dx at s0 .. s0+3: dx[s] = sum_i wp[i] dacc_{s+3-i}
  T* dx = static_cast<T*>(a.dx) + c * L;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (s0 + j < L) {
      float v = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxConv; ++i) v = fmaf(wp[i], da[j + 3 - i], v);
      dx[s0 + j] = from_f32<T>(v);
    }
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
        if (t >= 0 && t < 7 && t < L) v = fmaf(wp[i], da[t], v);
      }
      dw_out[j] = from_f32<T>(v);
    }
  }
  // this thread's dw / dbias terms (its own 4 steps only)
  float part[kCBPart];
#pragma unroll
  for (int i = 0; i < kCBPart; ++i) part[i] = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int i = 0; i < kMaxConv; ++i) part[i] = fmaf(da[j], xv[j + i], part[i]);
    part[kMaxConv] += da[j];
  }
  // block reduction (fixed order): warp shuffles, then warp 0 over the warps
#pragma unroll
  for (int i = 0; i < kCBPart; ++i)
    for (int o = 16; o > 0; o >>= 1) part[i] += __shfl_xor_sync(0xffffffffu, part[i], o);
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  if (lane == 0)
#pragma unroll
    for (int i = 0; i < kCBPart; ++i) red[warp][i] = part[i];
  __syncthreads();
  if (threadIdx.x < kCBPart) {
    float s = 0.f;
    for (int w = 0; w < kCBThreads / 32; ++w) s += red[w][threadIdx.x];
    a.ws_part[((long long)c * nseg + seg) * kCBPart + threadIdx.x] = s;
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
    for (int b = 0; b < a.batch; ++b)
      for (int g = 0; g < nseg; ++g) s += a.ws_part[(((long long)b * a.dim + d) * nseg + g) * kCBPart + slot];
    if (k < K) a.dw[(long long)d * K + k] = s;
    else if (a.dbias) a.dbias[d] = s;
  }
}

template <typename T>
cudaError_t launch_conv_bwd_t(const ConvBwdArgs& a, cudaStream_t stream) {
  const int nseg = (a.seqlen + kCBSeg - 1) / kCBSeg;
  const long long blocks = (long long)a.batch * a.dim * nseg;
  if (blocks > 0) {
    conv_bwd_kernel<T><<<(unsigned)blocks, kCBThreads, 0, stream>>>(a, nseg);
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

}  // namespace ssm
