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
// threads with two shuffles. Each group of four threads serves two channels and issues all
// of their loads before any arithmetic, to keep enough bytes in flight for HBM.
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kDecThreads = 256;
constexpr int kChanPerGroup = 2;  // channels per 4-thread group: two independent loads in flight

template <typename T, bool VEC>
__global__ void __launch_bounds__(kDecThreads, 4) decode_kernel(const DecodeArgs a) {
  constexpr bool PRECISE = IoTraits<T>::kPrecise;
  const long long gt = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long grp = gt >> 2;   // 4-thread group
  const int g = (int)(gt & 3);     // states 4g .. 4g+3
  const long long BD = (long long)a.batch * a.dim;
  const long long ngroups = (BD + kChanPerGroup - 1) / kChanPerGroup;
  const int N = a.dstate;
  const int K = a.d_conv;

  // group grp owns channels grp and grp + ngroups (each half of the grid is contiguous)
  long long ch[kChanPerGroup];
  bool valid[kChanPerGroup];
  int dd[kChanPerGroup];
  long long bb[kChanPerGroup];
  float xv[kChanPerGroup], dv[kChanPerGroup], zv[kChanPerGroup];
  T old[kChanPerGroup][kMaxConv - 1];
  float hs[kChanPerGroup][4], av[kChanPerGroup][4], bv[kChanPerGroup][4], cv[kChanPerGroup][4];

  // ---- issue every load first
#pragma unroll
  for (int i = 0; i < kChanPerGroup; ++i) {
    ch[i] = grp + i * ngroups;
    valid[i] = grp < ngroups && ch[i] < BD;
    const long long c = valid[i] ? ch[i] : 0;
    dd[i] = (int)(c % a.dim);
    bb[i] = c / a.dim;
    xv[i] = dv[i] = zv[i] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) hs[i][k] = av[i][k] = bv[i][k] = cv[i][k] = 0.f;
    if (!valid[i]) continue;
    xv[i] = to_f32(static_cast<const T*>(a.x)[c]);
    dv[i] = to_f32(static_cast<const T*>(a.delta)[c]);
    if (a.z) zv[i] = to_f32(static_cast<const T*>(a.z)[c]);
    if (a.conv_w) {
      const T* cs = static_cast<const T*>(a.conv_state) + c * (K - 1);
#pragma unroll
      for (int k = 0; k < kMaxConv - 1; ++k)
        if (k < K - 1) old[i][k] = cs[k];
    }
    const float* st = a.state + c * N + 4 * g;
    const float* Ad = a.A + (long long)dd[i] * N + 4 * g;
    const T* Bb = static_cast<const T*>(a.B) + bb[i] * N + 4 * g;
    const T* Cb = static_cast<const T*>(a.C) + bb[i] * N + 4 * g;
    if (VEC) {
      const float4 h4 = *reinterpret_cast<const float4*>(st);
      const float4 a4 = *reinterpret_cast<const float4*>(Ad);
      hs[i][0] = h4.x; hs[i][1] = h4.y; hs[i][2] = h4.z; hs[i][3] = h4.w;
      av[i][0] = a4.x; av[i][1] = a4.y; av[i][2] = a4.z; av[i][3] = a4.w;
      load4(Bb, bv[i]);
      load4(Cb, cv[i]);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (4 * g + k < N) {
          hs[i][k] = st[k];
          av[i][k] = Ad[k];
          bv[i][k] = to_f32(Bb[k]);
          cv[i][k] = to_f32(Cb[k]);
        }
      }
    }
  }

  // every lane of the warp gets here: the four threads of a channel have read the old
  // window before any of them overwrites a slot
  __syncwarp();

  float part[kChanPerGroup], u[kChanPerGroup];
#pragma unroll
  for (int i = 0; i < kChanPerGroup; ++i) {
    part[i] = 0.f;
    u[i] = 0.f;
    if (!valid[i]) continue;
    const long long c = ch[i];
    const int d = dd[i];
    if (a.conv_w) {
      const float* w = a.conv_w + (long long)d * K;
      float acc = a.conv_b ? a.conv_b[d] : 0.f;
#pragma unroll
      for (int k = 0; k < kMaxConv - 1; ++k)
        if (k < K - 1) acc = fmaf(w[k], to_f32(old[i][k]), acc);
      acc = fmaf(w[K - 1], xv[i], acc);
      u[i] = silu_f(acc);
      if (g < K - 1) {
        // thread g rewrites window slot g (the window shifts one place towards the old end)
        T* cs = static_cast<T*>(a.conv_state) + c * (K - 1);
        T nv = static_cast<const T*>(a.x)[c];
#pragma unroll
        for (int k = 0; k < kMaxConv - 2; ++k)
          if (k == g && k + 1 < K - 1) nv = old[i][k + 1];
        cs[g] = nv;
      }
    } else {
      u[i] = xv[i];
    }
    const float v = dv[i] + (a.delta_bias ? a.delta_bias[d] : 0.f);
    const float Delta = a.delta_softplus ? softplus_f<PRECISE>(v) : v;
    const float du = Delta * u[i];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      hs[i][k] = fmaf(ex2_approx(Delta * (av[i][k] * kLog2e)), hs[i][k], du * bv[i][k]);
      part[i] = fmaf(cv[i][k], hs[i][k], part[i]);
    }
    float* st = a.state + c * N + 4 * g;
    if (VEC) {
      *reinterpret_cast<float4*>(st) = make_float4(hs[i][0], hs[i][1], hs[i][2], hs[i][3]);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (4 * g + k < N) st[k] = hs[i][k];
    }
  }
#pragma unroll
  for (int i = 0; i < kChanPerGroup; ++i) {
    part[i] += __shfl_xor_sync(0xffffffffu, part[i], 1);
    part[i] += __shfl_xor_sync(0xffffffffu, part[i], 2);
    if (valid[i] && g == 0) {
      const int d = dd[i];
      float y = fmaf(a.D ? a.D[d] : 0.f, u[i], part[i]);
      if (a.z) y *= silu_f(zv[i]);
      static_cast<T*>(a.y)[ch[i]] = from_f32<T>(y);
    }
  }
}

template <typename T, bool VEC>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t stream) {
  const long long BD = (long long)a.batch * a.dim;
  const long long threads = (BD + kChanPerGroup - 1) / kChanPerGroup * 4;
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
