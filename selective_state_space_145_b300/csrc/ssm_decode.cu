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
// HBM-bound: the fp32 state is read and written once (128 of the ~150 bytes a channel moves).
// Four adjacent threads own one channel, four states each, so a warp moves 8 channels x 64 B
// of state per access with 16-byte loads and stores; C.state is reduced over the four
// threads with two shuffles. Tiles of 64 channels never cross a sequence, so no index needs
// a division, and the conv width is a compile-time constant.
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

// ---------------------------------------------------------------- one channel's step
// For the four threads that own a channel (this thread holds states 4g .. 4g+3).
// KC = d_conv (0: no conv); the window holds K1 = KC - 1 raw inputs. Returns this thread's
// part of C.h.
template <typename T, int KC>
__device__ __forceinline__ float channel_step(const DecodeArgs& a, int d, float xv, float dv, const T* win,
                                              float (&h)[4], const float (&av)[4], const float (&bv)[4],
                                              const float (&cv)[4], float& u) {
  constexpr bool PRECISE = IoTraits<T>::kPrecise;
  constexpr int K1 = KC > 0 ? KC - 1 : 0;
  u = xv;
  if (KC > 0) {
    const float* w = a.conv_w + (long long)d * KC;
    float acc = a.conv_b ? a.conv_b[d] : 0.f;
#pragma unroll
    for (int k = 0; k < K1; ++k) acc = fmaf(w[k], to_f32(win[k]), acc);
    acc = fmaf(w[K1], xv, acc);
    u = silu_f(acc);
  }
  const float v = dv + (a.delta_bias ? a.delta_bias[d] : 0.f);
  const float Delta = a.delta_softplus ? softplus_f<PRECISE>(v) : v;
  const float du = Delta * u;
  const float dl2 = Delta * kLog2e;  // exp(Delta A) = 2^(Delta log2(e) A)
  float part = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    h[j] = fmaf(ex2_approx(dl2 * av[j]), h[j], du * bv[j]);
    part = fmaf(cv[j], h[j], part);
  }
  return part;
}

// ---------------------------------------------------------------- general kernel
// Any N <= 16 and any alignment. Grid (ceil(dim / 64), batch): one CTA covers 64 channels of
// one sequence, four threads per channel.
constexpr int kDecThreads = 256;
constexpr int kDecCh = kDecThreads / 4;

template <typename T, int KC>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(const DecodeArgs a) {
  constexpr int K1 = KC > 0 ? KC - 1 : 0;
  const int c = threadIdx.x / 4, g = threadIdx.x % 4;
  const int d = blockIdx.x * kDecCh + c;
  const long long b = blockIdx.y;
  const bool valid = d < a.dim;
  const int N = a.dstate;
  const long long cc = b * a.dim + d;
  float h[4] = {0.f, 0.f, 0.f, 0.f}, av[4] = {0.f, 0.f, 0.f, 0.f}, bv[4] = {0.f, 0.f, 0.f, 0.f},
        cv[4] = {0.f, 0.f, 0.f, 0.f};
  T win[K1 > 0 ? K1 : 1];
  float xv = 0.f, dv = 0.f, zv = 0.f;
  if (valid) {
    const T* Bb = static_cast<const T*>(a.B) + b * N;
    const T* Cb = static_cast<const T*>(a.C) + b * N;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = 4 * g + j;
      if (n < N) {
        h[j] = a.state[cc * N + n];
        av[j] = a.A[(long long)d * N + n];
        bv[j] = to_f32(Bb[n]);
        cv[j] = to_f32(Cb[n]);
      }
    }
    xv = to_f32(static_cast<const T*>(a.x)[cc]);
    dv = to_f32(static_cast<const T*>(a.delta)[cc]);
    if (a.z) zv = to_f32(static_cast<const T*>(a.z)[cc]);
#pragma unroll
    for (int k = 0; k < K1; ++k) win[k] = static_cast<const T*>(a.conv_state)[cc * K1 + k];
  }
  // every lane of the warp gets here: the four threads of a channel have read the old
  // window before any of them overwrites a slot
  __syncwarp();
  float u = 0.f;
  float part = valid ? channel_step<T, KC>(a, d, xv, dv, win, h, av, bv, cv, u) : 0.f;
  part += __shfl_xor_sync(0xffffffffu, part, 1);
  part += __shfl_xor_sync(0xffffffffu, part, 2);
  if (!valid) return;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (4 * g + j < N) a.state[cc * N + 4 * g + j] = h[j];
  if (g == 0) {
    float y = fmaf(a.D ? a.D[d] : 0.f, u, part);
    if (a.z) y *= silu_f(zv);
    static_cast<T*>(a.y)[cc] = from_f32<T>(y);
  }
  if (g < K1) {
    // the window shifts one place towards the old end; the newest slot takes x
    T nv = static_cast<const T*>(a.x)[cc];
#pragma unroll
    for (int k = 0; k + 1 < K1; ++k)
      if (k == g) nv = win[k + 1];
    static_cast<T*>(a.conv_state)[cc * K1 + g] = nv;
  }
}

// ---------------------------------------------------------------- streaming kernel (N = 16)
//
// Persistent CTAs walk tiles of 64 channels of one sequence. A 4-stage cp.async ring stages
// each tile's fp32 state (4 KB) and its x, delta, z and conv-window bytes in shared memory,
// so a CTA keeps three tiles on their way from HBM without holding registers for them; the
// new state goes back with coalesced 16-byte stores. Needs dim * element size a multiple of
// 16 bytes (every tile then starts 16-byte aligned) and 16-byte aligned pointers.
constexpr int kStrThreads = 256;
constexpr int kStrCh = kStrThreads / 4;
constexpr int kStrStages = 4;

template <typename T>
struct __align__(16) StrSmem {
  float st[kStrStages][kStrCh * kMaxDstate];
  T x[kStrStages][kStrCh];
  T dl[kStrStages][kStrCh];
  T z[kStrStages][kStrCh];
  T win[kStrStages][kStrCh * (kMaxConv - 1)];
};

template <typename T, int KC>
__global__ void __launch_bounds__(kStrThreads) decode_stream_kernel(const DecodeArgs a) {
  constexpr int K1 = KC > 0 ? KC - 1 : 0;
  constexpr int ES = (int)sizeof(T);
  constexpr int EPC = 16 / ES;             // I/O elements per 16-byte chunk
  constexpr int kCpa = kStrCh / EPC;       // chunks of one per-channel I/O array per tile
  __shared__ StrSmem<T> S;
  const int tid = threadIdx.x;
  const int c = tid / 4, g = tid % 4;
  const int dim = a.dim;
  const int tiles_per_row = (dim + kStrCh - 1) / kStrCh;
  const T* gx = static_cast<const T*>(a.x);
  const T* gd = static_cast<const T*>(a.delta);
  const T* gz = static_cast<const T*>(a.z);
  const T* gw = static_cast<const T*>(a.conv_state);

  // Tiles are visited as tile = blockIdx.x + i * gridDim.x; (sequence, tile-in-row) pairs are
  // advanced incrementally so that no index needs a division inside the loop.
  struct Pos {
    int b, t;  // sequence, tile within the sequence
  };
  const int step_b = (int)(gridDim.x / (unsigned)tiles_per_row);
  const int step_t = (int)(gridDim.x % (unsigned)tiles_per_row);
  auto advance = [&](Pos p) {
    p.b += step_b;
    p.t += step_t;
    if (p.t >= tiles_per_row) {
      p.t -= tiles_per_row;
      ++p.b;
    }
    return p;
  };
  auto issue_tile = [&](Pos p, int slot) {
    const int b = p.b;
    const int d0 = p.t * kStrCh;
    const long long c0 = (long long)b * dim + d0;
    const int nvalid = min(kStrCh, dim - d0);  // channels of this tile inside the sequence
    {  // state: one 16-byte chunk (4 states) per thread
      const bool ok = c < nvalid;
      cp_async16(&S.st[slot][tid * 4], ok ? (const void*)(a.state + c0 * kMaxDstate + tid * 4) : (const void*)a.state,
                 ok ? 16u : 0u);
    }
    for (int e = tid; e < (3 + K1) * kCpa; e += kStrThreads) {
      const int arr = e / kCpa, ch = e % kCpa;
      if (arr < 3) {
        const T* base = arr == 0 ? gx : (arr == 1 ? gd : gz);
        T* dst = arr == 0 ? S.x[slot] : (arr == 1 ? S.dl[slot] : S.z[slot]);
        const int first = ch * EPC;
        const int n = nvalid - first;
        const unsigned bytes = (base == nullptr || n <= 0) ? 0u : (n >= EPC ? 16u : (unsigned)(n * ES));
        cp_async16(dst + first, bytes ? (const void*)(base + c0 + first) : (const void*)a.state, bytes);
      } else {
        const int first = (e - 3 * kCpa) * EPC;  // element within this tile's window block
        const int n = nvalid * K1 - first;
        const unsigned bytes = n <= 0 ? 0u : (n >= EPC ? 16u : (unsigned)(n * ES));
        cp_async16(S.win[slot] + first, bytes ? (const void*)(gw + c0 * K1 + first) : (const void*)a.state, bytes);
      }
    }
  };

  Pos cur{(int)(blockIdx.x / (unsigned)tiles_per_row), (int)(blockIdx.x % (unsigned)tiles_per_row)};
  Pos ahead = cur;  // the tile kStrStages-1 visits ahead of `cur`
#pragma unroll 1
  for (int st = 0; st < kStrStages - 1; ++st) {
    if (ahead.b < a.batch) issue_tile(ahead, st);
    cp_async_commit();
    ahead = advance(ahead);
  }

#pragma unroll 1
  for (int i = 0; cur.b < a.batch; ++i, cur = advance(cur)) {
    const int slot = i % kStrStages;
    cp_async_wait<kStrStages - 2>();
    __syncthreads();  // tile i visible; every thread is done with tile i-1, whose slot is refilled next
    if (ahead.b < a.batch) issue_tile(ahead, (i + kStrStages - 1) % kStrStages);
    cp_async_commit();
    ahead = advance(ahead);
    const int b = cur.b;
    const int d = cur.t * kStrCh + c;
    const bool valid = d < dim;
    const long long cc = (long long)b * dim + d;
    float av[4] = {0.f, 0.f, 0.f, 0.f}, bv[4], cv[4];
    if (valid) {
      const float4 a4 = *reinterpret_cast<const float4*>(a.A + (long long)d * kMaxDstate + 4 * g);
      av[0] = a4.x; av[1] = a4.y; av[2] = a4.z; av[3] = a4.w;
    }
    load4(static_cast<const T*>(a.B) + (long long)b * kMaxDstate + 4 * g, bv);
    load4(static_cast<const T*>(a.C) + (long long)b * kMaxDstate + 4 * g, cv);
    const float4 h4 = *reinterpret_cast<const float4*>(&S.st[slot][c * kMaxDstate + 4 * g]);
    float h[4] = {h4.x, h4.y, h4.z, h4.w};
    float u = 0.f;
    const T* win = &S.win[slot][c * K1];
    float part = channel_step<T, KC>(a, valid ? d : 0, to_f32(S.x[slot][c]), to_f32(S.dl[slot][c]), win, h, av,
                                     bv, cv, u);
    part += __shfl_xor_sync(0xffffffffu, part, 1);
    part += __shfl_xor_sync(0xffffffffu, part, 2);
    if (valid) {
      *reinterpret_cast<float4*>(a.state + cc * kMaxDstate + 4 * g) = make_float4(h[0], h[1], h[2], h[3]);
      if (g == 0) {
        float y = fmaf(a.D ? a.D[d] : 0.f, u, part);
        if (gz) y *= silu_f(to_f32(S.z[slot][c]));
        static_cast<T*>(a.y)[cc] = from_f32<T>(y);
      }
      if (g < K1) {
        // the window shifts one place towards the old end; the newest slot takes x
        static_cast<T*>(a.conv_state)[cc * K1 + g] = (g + 1 < K1) ? win[g + 1] : S.x[slot][c];
      }
    }
  }
}

template <typename T, int KC>
cudaError_t launch_general(const DecodeArgs& a, cudaStream_t stream) {
  dim3 grid((a.dim + kDecCh - 1) / kDecCh, a.batch);
  decode_kernel<T, KC><<<grid, kDecThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <typename T, int KC>
cudaError_t launch_stream(const DecodeArgs& a, cudaStream_t stream) {
  // persistent grid: exactly the CTAs that are resident at once, so no CTA waits for a slot
  static int resident[64] = {0};
  int dev = 0, sms = 148;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int per_sm = (dev >= 0 && dev < 64) ? resident[dev] : 0;
  if (per_sm == 0) {
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_stream_kernel<T, KC>, kStrThreads, 0);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
    if (dev >= 0 && dev < 64) resident[dev] = per_sm;
  }
  const long long ntiles = (long long)a.batch * ((a.dim + kStrCh - 1) / kStrCh);
  long long grid = (long long)sms * per_sm;
  if (grid > ntiles) grid = ntiles;
  decode_stream_kernel<T, KC><<<(unsigned)grid, kStrThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_k(const DecodeArgs& a, bool stream_ok, cudaStream_t s) {
  const int KC = a.conv_w ? a.d_conv : 0;
  if (stream_ok) {
    switch (KC) {
      case 0: return launch_stream<T, 0>(a, s);
      case 1: return launch_stream<T, 1>(a, s);
      case 2: return launch_stream<T, 2>(a, s);
      case 3: return launch_stream<T, 3>(a, s);
      default: return launch_stream<T, 4>(a, s);
    }
  }
  switch (KC) {
    case 0: return launch_general<T, 0>(a, s);
    case 1: return launch_general<T, 1>(a, s);
    case 2: return launch_general<T, 2>(a, s);
    case 3: return launch_general<T, 3>(a, s);
    default: return launch_general<T, 4>(a, s);
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  auto al = [](const void* p, uintptr_t n) { return p == nullptr || reinterpret_cast<uintptr_t>(p) % n == 0; };
  const int es = a.bf16 ? 2 : 4;
  const bool stream_ok = a.dstate == kMaxDstate && (a.dim * es) % 16 == 0 && al(a.state, 16) && al(a.A, 16) &&
                         al(a.B, 16) && al(a.C, 16) && al(a.x, 16) && al(a.delta, 16) && al(a.z, 16) &&
                         (a.conv_w == nullptr || al(a.conv_state, 16));
  return a.bf16 ? dispatch_k<__nv_bfloat16>(a, stream_ok, stream) : dispatch_k<float>(a, stream_ok, stream);
}

}  // namespace ssm
