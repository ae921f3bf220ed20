// ssm_decode.cu -- batched single-token selective state update (recurrent / decode mode).
//
// "Mamba", ozercemkelahmet.com, "Step 5: training versus inference" and "Deployment notes":
// at inference the model keeps only a fixed-size state per sequence and updates it once per
// token; "Mamba (Selective State-Space Model)", "Key math": the inference state is O(N d)
// per layer and constant in the sequence length.
//
// Per (b, d): shift the raw-input conv window, u = silu(conv), Delta = softplus(delta + bias),
// state[n] = exp(Delta A[d,n]) state[n] + Delta B[b,n] u, y = (C.state + D u) silu(z).
//
// HBM-bound (the fp32 state is read and written once: 128 of the ~150 bytes a channel moves).
// Four adjacent threads own one channel, four states each, so a warp moves 8 channels x 64 B
// of state per access with 16-byte loads and stores; C.state is reduced over the four
// threads with two shuffles.
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kDecThreads = 256;

template <typename T, bool VEC>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(const DecodeArgs a) {
  constexpr bool PRECISE = IoTraits<T>::kPrecise;
  const long long gt = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long c = gt >> 2;  // channel index b*dim + d
  const int g = (int)(gt & 3);  // states 4g .. 4g+3
  const long long BD = (long long)a.batch * a.dim;
  const bool valid = c < BD;    // the four threads of a channel agree
  const int N = a.dstate;
  const int d = valid ? (int)(c % a.dim) : 0;
  const long long b = valid ? c / a.dim : 0;

  float u = 0.f, Delta = 0.f, zv = 0.f;
  T old[kMaxConv - 1];
  const int K = a.d_conv;
  if (valid) {
    const float xv = to_f32(static_cast<const T*>(a.x)[c]);
    if (a.conv_w) {
      const T* cs = static_cast<const T*>(a.conv_state) + c * (K - 1);
      float acc = a.conv_b ? a.conv_b[d] : 0.f;
      for (int k = 0; k < K - 1; ++k) {
        old[k] = cs[k];
        acc = fmaf(a.conv_w[(long long)d * K + k], to_f32(old[k]), acc);
      }
      acc = fmaf(a.conv_w[(long long)d * K + K - 1], xv, acc);
      u = silu_f(acc);
    } else {
      u = xv;
    }
    const float v = to_f32(static_cast<const T*>(a.delta)[c]) + (a.delta_bias ? a.delta_bias[d] : 0.f);
    Delta = a.delta_softplus ? softplus_f<PRECISE>(v) : v;
    if (a.z) zv = to_f32(static_cast<const T*>(a.z)[c]);
  }

  // every lane of the warp gets here: the four threads of a channel have read the old
  // window before any of them overwrites a slot
  __syncwarp();
  if (valid && a.conv_w && g < K - 1) {
    // thread g rewrites window slot g (the window shifts one place towards the old end)
    T* cs = static_cast<T*>(a.conv_state) + c * (K - 1);
    cs[g] = (g + 1 < K - 1) ? old[g + 1] : static_cast<const T*>(a.x)[c];
  }

  float h[4] = {0.f, 0.f, 0.f, 0.f};
  float part = 0.f;
  if (valid) {
    float* st = a.state + c * N + 4 * g;
    const float* Ad = a.A + (long long)d * N + 4 * g;
    const T* Bb = static_cast<const T*>(a.B) + b * N + 4 * g;
    const T* Cb = static_cast<const T*>(a.C) + b * N + 4 * g;
    const float du = Delta * u;
    if (VEC) {
      const float4 hv = *reinterpret_cast<const float4*>(st);
      const float4 av = *reinterpret_cast<const float4*>(Ad);
      float bv[4], cv[4];
      load4(Bb, bv);
      load4(Cb, cv);
      h[0] = hv.x; h[1] = hv.y; h[2] = hv.z; h[3] = hv.w;
      const float aa[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        h[j] = fmaf(ex2_approx(Delta * (aa[j] * kLog2e)), h[j], du * bv[j]);
        part = fmaf(cv[j], h[j], part);
      }
      *reinterpret_cast<float4*>(st) = make_float4(h[0], h[1], h[2], h[3]);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (4 * g + j < N) {
          const float hj = st[j];
          const float nh = fmaf(ex2_approx(Delta * (Ad[j] * kLog2e)), hj, du * to_f32(Bb[j]));
          st[j] = nh;
          part = fmaf(to_f32(Cb[j]), nh, part);
        }
      }
    }
  }
  part += __shfl_xor_sync(0xffffffffu, part, 1);
  part += __shfl_xor_sync(0xffffffffu, part, 2);
  if (valid && g == 0) {
    float y = fmaf(a.D ? a.D[d] : 0.f, u, part);
    if (a.z) y *= silu_f(zv);
    static_cast<T*>(a.y)[c] = from_f32<T>(y);
  }
}

template <typename T, bool VEC>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t stream) {
  const long long threads = (long long)a.batch * a.dim * 4;
  const long long blocks = (threads + kDecThreads - 1) / kDecThreads;
  decode_kernel<T, VEC><<<(unsigned)blocks, kDecThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  const bool vec = a.dstate == kMaxDstate && (reinterpret_cast<uintptr_t>(a.state) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(a.A) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(a.B) % (a.bf16 ? 8 : 16) == 0) &&
                   (reinterpret_cast<uintptr_t>(a.C) % (a.bf16 ? 8 : 16) == 0);
  if (a.bf16) return vec ? launch_t<__nv_bfloat16, true>(a, stream) : launch_t<__nv_bfloat16, false>(a, stream);
  return vec ? launch_t<float, true>(a, stream) : launch_t<float, false>(a, stream);
}

}  // namespace ssm
