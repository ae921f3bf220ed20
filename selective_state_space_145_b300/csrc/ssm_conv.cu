// ssm_conv.cu -- standalone causal depthwise conv1d (+ SiLU), the Mamba block's short conv
// ("Overview of Mamba (SSM) Model", "How the Mamba Block Works": a depthwise convolution and
// SiLU before the selective SSM; "Mamba", ozercemkelahmet.com, glossary: a causal conv only
// sees current and past positions).
//
//   out[b,d,t] = act( sum_{k<K} w[d,k] x[b,d,t-(K-1)+k] + bias[d] ),  x[b,d,s<0] = conv_init
//
// Memory-bound: one thread produces 4 consecutive outputs of one row from one 4-element
// vector load plus the previous vector (an L1/L2 hit) for the K-1 halo, so every input
// element comes from HBM once and every output is written once.
#include "ssm_bounds.cuh"
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kConvThreads = 256;

template <typename T, bool VEC>
__global__ void __launch_bounds__(kConvThreads) conv_kernel(const ConvArgs a) {
  const int L = a.seqlen, K = a.d_conv;
  const long long nseg = (L + 3) / 4;
  const long long total = (long long)a.batch * a.dim * nseg;
  const T* __restrict__ x = static_cast<const T*>(a.x);
  T* __restrict__ out = static_cast<T*>(a.out);
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long c = idx / nseg;
    const int t0 = (int)(idx % nseg) * 4;
    const int d = (int)(c % a.dim);
    // debug build: the row, its taps and its window must lie inside their tensors
    const long long tok = total / nseg * L;
    if (!in_bounds(c * L + t0, min(4, L - t0), tok, kBoundsConv) ||
        !in_bounds((long long)d * K, K, (long long)a.dim * K, kBoundsConv) ||
        !in_bounds(c * (K - 1), K - 1, total / nseg * (K - 1), kBoundsConv))
      continue;
    float w[kMaxConv] = {0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < K; ++k) w[kMaxConv - K + k] = a.w[(long long)d * K + k];
    const float cb = a.bias ? a.bias[d] : 0.f;
    const T* row = x + c * L;
    float win[7];  // x[t0-3 .. t0+3]
    if (VEC && in_bounds(c * L + t0, 4, tok, kBoundsConv)) {
      float cur[4];
      load4(row + t0, cur);
#pragma unroll
      for (int j = 0; j < 4; ++j) win[3 + j] = cur[j];
      if (t0 >= 4) {
        float prev[4];
        load4(row + t0 - 4, prev);
        win[0] = prev[1];
        win[1] = prev[2];
        win[2] = prev[3];
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) win[3 + j] = (t0 + j < L) ? to_f32(row[t0 + j]) : 0.f;
      if (t0 >= 4) {
#pragma unroll
        for (int j = 0; j < 3; ++j) win[j] = to_f32(row[t0 - 3 + j]);
      }
    }
    if (t0 < 4) {
      // t0 == 0: the K-1 inputs before the row come from conv_init (oldest first) or are zero
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const int s = j - 3;  // position relative to t = 0
        float v = 0.f;
        if (a.conv_init && s >= -(K - 1)) v = to_f32(static_cast<const T*>(a.conv_init)[c * (K - 1) + (K - 1) + s]);
        win[j] = v;
      }
    }
    float o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float acc = fmaf(w[0], win[j], cb);
      acc = fmaf(w[1], win[j + 1], acc);
      acc = fmaf(w[2], win[j + 2], acc);
      acc = fmaf(w[3], win[j + 3], acc);
      o[j] = a.apply_silu ? silu_f(acc) : acc;
    }
    if (VEC && in_bounds(c * L + t0, 4, tok, kBoundsConv)) {
      store4(out + c * L + t0, o);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (t0 + j < L) out[c * L + t0 + j] = from_f32<T>(o[j]);
    }
  }
}

template <typename T, bool VEC>
cudaError_t launch_t(const ConvArgs& a, cudaStream_t stream) {
  const long long total = (long long)a.batch * a.dim * ((a.seqlen + 3) / 4);
  long long blocks = (total + kConvThreads - 1) / kConvThreads;
  if (blocks > (1LL << 20)) blocks = 1LL << 20;  // grid-stride beyond this
  if (blocks < 1) blocks = 1;
  conv_kernel<T, VEC><<<(unsigned)blocks, kConvThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv(const ConvArgs& a, cudaStream_t stream) {
  if (a.bf16) return a.vec ? launch_t<__nv_bfloat16, true>(a, stream) : launch_t<__nv_bfloat16, false>(a, stream);
  return a.vec ? launch_t<float, true>(a, stream) : launch_t<float, false>(a, stream);
}

cudaError_t conv_bounds_flags(unsigned* out, bool clear) {
#ifdef SSM_DEBUG_BOUNDS
  return bounds_flags_read(out, clear);
#else
  (void)out;
  (void)clear;
  return cudaErrorNotSupported;
#endif
}

}  // namespace ssm
