// ssm_scan.cu -- selective scan forward (S6) with the fused causal-conv + SiLU prologue
// and the cross-chunk carry.
//
// What it computes ("Mamba", ai360xpert.com, "The selection mechanism"; "Mamba",
// ozercemkelahmet.com, "How it works" steps 1-4; "Overview of Mamba (SSM) Model",
// "How the Mamba Block Works"): for every (b, d)
//   u_t = silu(conv(x)_t) or x_t,  Delta_t = softplus(delta_t + bias_d),
//   h_t[n] = exp(Delta_t A[d,n]) h_{t-1}[n] + Delta_t B[b,n,t] u_t,
//   out_t = (sum_n C[b,n,t] h_t[n] + D_d u_t) * silu(z_t).
//
// Design (one CTA = DT channels of one batch element x one time chunk):
//  * per time tile of kTT steps, the raw x / delta / z rows and the shared B / C rows are
//    copied global->shared with 16-byte cp.async, double-buffered so tile i+1 lands
//    while tile i is computed;
//  * an element-wise phase turns each (t, d) into Delta, Delta*u and u once (conv, SiLU,
//    softplus), in fp32 shared memory, so no per-(t, d) work is repeated per state;
//  * the scan phase gives each channel TPC = 16 / NPT threads holding NPT states each in
//    registers; a thread walks the tile sequentially, one exp2 per state update, and
//    leaves its partial C.h per step in shared memory;
//  * an epilogue sums the partials, adds D*u, applies the gate and stores coalesced rows.
//  The per-step state never leaves registers. With more than one chunk, a carry kernel
//  (same code, CARRY = true) first writes every chunk's sum of Delta and its end state
//  from zero; the main kernel starts chunk q from h0 composed with the carries of chunks
//  0..q-1 through (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2), a = exp(A sum Delta).
#include <algorithm>
#include <cstdio>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kThreads = 128;   // threads per CTA
constexpr int kTT = 32;         // time steps per tile
constexpr int kTP = kTT + 4;    // padded row stride of the fp32 tile arrays (keeps float4 alignment)

template <int NPT>
struct Cfg {
  static constexpr int TPC = kMaxDstate / NPT;  // threads per channel
  static constexpr int DT = kThreads / TPC;     // channels per CTA
};

template <typename T, int NPT>
struct __align__(16) Smem {
  static constexpr int DT = Cfg<NPT>::DT;
  static constexpr int TPC = Cfg<NPT>::TPC;
  // raw staging in the I/O dtype, double-buffered
  T raw_x[2][DT][kTT];
  T raw_d[2][DT][kTT];
  T raw_z[2][DT][kTT];
  T raw_B[2][kMaxDstate][kTT];
  T raw_C[2][kMaxDstate][kTT];
  // fp32 tile arrays
  float s_delta[DT][kTP];
  float s_du[DT][kTP];
  float s_u[DT][kTP];
  float s_y[TPC][DT][kTP];
  float s_B[kTT][kMaxDstate];
  float s_C[kTT][kMaxDstate];
  float s_halo[2][DT][4];   // the 3 raw inputs before the tile (ping-pong by tile parity)
  float s_par[DT][8];       // delta_bias, D, conv taps w0..w3 (zero-padded on the old side), conv bias
};

template <typename T, int NPT, bool CONV, bool VEC, bool CARRY>
__global__ void __launch_bounds__(kThreads) scan_kernel(const ScanArgs a) {
  using Cf = Cfg<NPT>;
  constexpr int TPC = Cf::TPC;
  constexpr int DT = Cf::DT;
  constexpr bool PRECISE = IoTraits<T>::kPrecise;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem<T, NPT>& S = *reinterpret_cast<Smem<T, NPT>*>(smem_raw);

  const int tid = threadIdx.x;
  const int d0 = blockIdx.x * DT;
  const int q = blockIdx.y;
  const int b = blockIdx.z;
  const int L = a.seqlen, N = a.dstate, dim = a.dim;
  const long long BD = (long long)a.batch * dim;
  const int t_begin = q * a.chunk_len;
  const int t_end = min(L, t_begin + a.chunk_len);
  const int ntiles = t_end > t_begin ? (t_end - t_begin + kTT - 1) / kTT : 0;

  const T* __restrict__ gx = static_cast<const T*>(a.x);
  const T* __restrict__ gd = static_cast<const T*>(a.delta);
  const T* __restrict__ gz = static_cast<const T*>(a.z);
  const T* __restrict__ gB = static_cast<const T*>(a.B);
  const T* __restrict__ gC = static_cast<const T*>(a.C);
  const bool has_z = (gz != nullptr) && !CARRY;

  // ---- per-channel parameters and the conv halo before the chunk
  for (int i = tid; i < DT; i += kThreads) {
    const int d = d0 + i;
    float par[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float hv[3] = {0.f, 0.f, 0.f};
    if (d < dim) {
      par[0] = a.delta_bias ? a.delta_bias[d] : 0.f;
      par[1] = a.D ? a.D[d] : 0.f;
      if (CONV) {
        const int K = a.d_conv;
        for (int k = 0; k < K; ++k) par[2 + (kMaxConv - K) + k] = a.conv_w[(long long)d * K + k];
        par[6] = a.conv_b ? a.conv_b[d] : 0.f;
        const long long c = (long long)b * dim + d;
        if (q == 0) {
          if (a.conv_init) {
            const T* ci = static_cast<const T*>(a.conv_init) + c * (K - 1);
            for (int j = 0; j < K - 1; ++j) hv[3 - (K - 1) + j] = to_f32(ci[j]);
          }
        } else {
          for (int j = 0; j < 3; ++j) hv[j] = to_f32(gx[c * L + (t_begin - 3 + j)]);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) S.s_par[i][k] = par[k];
#pragma unroll
    for (int j = 0; j < 3; ++j) S.s_halo[0][i][j] = hv[j];
    S.s_halo[0][i][3] = 0.f;
  }

  // ---- scan role of this thread: channel c_loc, states g*NPT .. g*NPT+NPT-1
  const int c_loc = tid / TPC;
  const int g = tid % TPC;
  const int d_me = d0 + c_loc;
  const bool valid = d_me < dim;
  const long long c_me = (long long)b * dim + d_me;
  float h[NPT], a2[NPT];
#pragma unroll
  for (int k = 0; k < NPT; ++k) {
    const int n = g * NPT + k;
    a2[k] = (valid && n < N) ? a.A[(long long)d_me * N + n] * kLog2e : 0.f;
    h[k] = 0.f;
  }
  if (!CARRY && valid) {
    if (a.h0) {
#pragma unroll
      for (int k = 0; k < NPT; ++k) {
        const int n = g * NPT + k;
        if (n < N) h[k] = a.h0[c_me * N + n];
      }
    }
    // carry-in: compose the aggregates of chunks 0 .. q-1 onto h0
    for (int j = 0; j < q; ++j) {
      const float Sj = a.ws_S[(long long)j * BD + c_me];
      const float* hj = a.ws_h + ((long long)j * BD + c_me) * kMaxDstate + g * NPT;
#pragma unroll
      for (int k = 0; k < NPT; ++k) h[k] = fmaf(ex2_approx(Sj * a2[k]), h[k], hj[k]);
    }
  }
  float dsum = 0.f;  // CARRY: sum of Delta over the chunk

  // ---- raw tile loaders
  constexpr int kRowsMain = 3 * DT + 2 * kMaxDstate;
  constexpr int kRowsCarry = 2 * DT + kMaxDstate;
  constexpr int kRows = CARRY ? kRowsCarry : kRowsMain;
  // map a staging row to (global row pointer, shared row pointer); returns false for padding rows
  auto row_ptrs = [&](int r, int bf, const T*& src, T*& dst) -> bool {
    if (r < DT) {
      dst = S.raw_x[bf][r];
      const int d = d0 + r;
      src = gx + ((long long)b * dim + d) * L;
      return d < dim;
    }
    r -= DT;
    if (r < DT) {
      dst = S.raw_d[bf][r];
      const int d = d0 + r;
      src = gd + ((long long)b * dim + d) * L;
      return d < dim;
    }
    r -= DT;
    if (!CARRY) {
      if (r < DT) {
        dst = S.raw_z[bf][r];
        const int d = d0 + r;
        src = has_z ? gz + ((long long)b * dim + d) * L : gx;
        return has_z && d < dim;
      }
      r -= DT;
    }
    if (r < kMaxDstate) {
      dst = S.raw_B[bf][r];
      src = gB + ((long long)b * N + r) * L;
      return r < N;
    }
    r -= kMaxDstate;
    dst = S.raw_C[bf][r];
    src = gC + ((long long)b * N + r) * L;
    return r < N;
  };

  auto issue_tile_async = [&](int it, int bf) {
    constexpr int EPC = 16 / (int)sizeof(T);  // elements per 16-byte chunk
    constexpr int CPR = kTT / EPC;            // chunks per row
    const int t0 = t_begin + it * kTT;
    const int tl = min(kTT, t_end - t0);
    for (int e = tid; e < kRows * CPR; e += kThreads) {
      const int r = e / CPR, tt = (e % CPR) * EPC;
      const T* src;
      T* dst;
      const bool ok = row_ptrs(r, bf, src, dst) && tt < tl;
      cp_async16(dst + tt, ok ? (const void*)(src + t0 + tt) : (const void*)gx, ok ? 16u : 0u);
    }
  };

  auto load_tile_sync = [&](int it, int bf) {
    const int t0 = t_begin + it * kTT;
    const int tl = min(kTT, t_end - t0);
    for (int e = tid; e < kRows * kTT; e += kThreads) {
      const int r = e / kTT, tt = e % kTT;
      const T* src;
      T* dst;
      const bool ok = row_ptrs(r, bf, src, dst) && tt < tl;
      dst[tt] = ok ? src[t0 + tt] : from_f32<T>(0.f);
    }
  };

  if (VEC && ntiles > 0) {
    issue_tile_async(0, 0);
    cp_async_commit();
  }

  for (int it = 0; it < ntiles; ++it) {
    const int bf = it & 1;
    const int t0 = t_begin + it * kTT;
    const int tl = min(kTT, t_end - t0);
    if (VEC) {
      cp_async_wait<0>();
    } else {
      load_tile_sync(it, bf);
    }
    __syncthreads();  // (A) tile `it` visible; every thread is past iteration it-1
    if (VEC && it + 1 < ntiles) {
      issue_tile_async(it + 1, bf ^ 1);
      cp_async_commit();
    }

    // ---- element-wise phase: B, C -> fp32 t-major; x, delta -> u, Delta, Delta*u
    for (int e = tid; e < kMaxDstate * kTT; e += kThreads) {
      const int n = e / kTT, t = e % kTT;
      const bool ok = n < N && t < tl;
      S.s_B[t][n] = ok ? to_f32(S.raw_B[bf][n][t]) : 0.f;
      if (!CARRY) S.s_C[t][n] = ok ? to_f32(S.raw_C[bf][n][t]) : 0.f;
    }
    for (int e = tid; e < DT * (kTT / 4); e += kThreads) {
      const int i = e / (kTT / 4), tt = (e % (kTT / 4)) * 4;
      float xv[4], dv[4], u[4];
      load4(&S.raw_x[bf][i][tt], xv);
      load4(&S.raw_d[bf][i][tt], dv);
      const float bias = S.s_par[i][0];
      if (CONV) {
        float win[7];
        if (tt == 0) {
          win[0] = S.s_halo[bf][i][0];
          win[1] = S.s_halo[bf][i][1];
          win[2] = S.s_halo[bf][i][2];
        } else {
          float pv[4];
          load4(&S.raw_x[bf][i][tt - 4], pv);
          win[0] = pv[1];
          win[1] = pv[2];
          win[2] = pv[3];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) win[3 + j] = xv[j];
        const float w0 = S.s_par[i][2], w1 = S.s_par[i][3], w2 = S.s_par[i][4], w3 = S.s_par[i][5];
        const float cb = S.s_par[i][6];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float acc = fmaf(w0, win[j], cb);
          acc = fmaf(w1, win[j + 1], acc);
          acc = fmaf(w2, win[j + 2], acc);
          acc = fmaf(w3, win[j + 3], acc);
          u[j] = silu_f(acc);
        }
        if (tt == kTT - 4) {
          S.s_halo[bf ^ 1][i][0] = xv[1];
          S.s_halo[bf ^ 1][i][1] = xv[2];
          S.s_halo[bf ^ 1][i][2] = xv[3];
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) u[j] = xv[j];
      }
      float dl[4], du[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float v = dv[j] + bias;
        float D_ = a.delta_softplus ? softplus_f<PRECISE>(v) : v;
        const bool tin = tt + j < tl;
        D_ = tin ? D_ : 0.f;
        u[j] = tin ? u[j] : 0.f;
        dl[j] = D_;
        du[j] = D_ * u[j];
      }
      store4(&S.s_delta[i][tt], dl);
      store4(&S.s_du[i][tt], du);
      if (!CARRY) store4(&S.s_u[i][tt], u);
    }
    __syncthreads();  // (B)

    // ---- scan phase: sequential in t, NPT states per thread in registers
    {
      const int tl4 = (tl + 3) & ~3;  // steps past tl have Delta = 0, Delta*u = 0: identity updates
      for (int t = 0; t < tl4; t += 4) {
        const float4 dl4 = *reinterpret_cast<const float4*>(&S.s_delta[c_loc][t]);
        const float4 du4 = *reinterpret_cast<const float4*>(&S.s_du[c_loc][t]);
        const float dl[4] = {dl4.x, dl4.y, dl4.z, dl4.w};
        const float du[4] = {du4.x, du4.y, du4.z, du4.w};
        float yv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float bq[NPT], cq[NPT];
          if (NPT % 4 == 0) {
#pragma unroll
            for (int k = 0; k < NPT; k += 4) {
              const float4 bb = *reinterpret_cast<const float4*>(&S.s_B[t + j][g * NPT + k]);
              bq[k] = bb.x; bq[k + 1] = bb.y; bq[k + 2] = bb.z; bq[k + 3] = bb.w;
              if (!CARRY) {
                const float4 cc = *reinterpret_cast<const float4*>(&S.s_C[t + j][g * NPT + k]);
                cq[k] = cc.x; cq[k + 1] = cc.y; cq[k + 2] = cc.z; cq[k + 3] = cc.w;
              }
            }
          } else {
#pragma unroll
            for (int k = 0; k < NPT; ++k) {
              bq[k] = S.s_B[t + j][g * NPT + k];
              if (!CARRY) cq[k] = S.s_C[t + j][g * NPT + k];
            }
          }
          float acc = 0.f;
#pragma unroll
          for (int k = 0; k < NPT; ++k) {
            const float ab = ex2_approx(dl[j] * a2[k]);
            h[k] = fmaf(ab, h[k], du[j] * bq[k]);
            if (!CARRY) acc = fmaf(cq[k], h[k], acc);
          }
          if (CARRY) dsum += dl[j];
          yv[j] = acc;
        }
        if (!CARRY) store4(&S.s_y[g][c_loc][t], yv);
      }
    }

    if (!CARRY) {
      __syncthreads();  // (C)
      // ---- epilogue: y = sum of partials + D u, gate, store
      for (int e = tid; e < DT * (kTT / 4); e += kThreads) {
        const int i = e / (kTT / 4), tt = (e % (kTT / 4)) * 4;
        const int d = d0 + i;
        if (d >= dim || tt >= tl) continue;
        float y[4], uu[4];
        load4(&S.s_y[0][i][tt], y);
#pragma unroll
        for (int gg = 1; gg < TPC; ++gg) {
          float p[4];
          load4(&S.s_y[gg][i][tt], p);
#pragma unroll
          for (int j = 0; j < 4; ++j) y[j] += p[j];
        }
        load4(&S.s_u[i][tt], uu);
        const float Dd = S.s_par[i][1];
        float o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = fmaf(Dd, uu[j], y[j]);
        if (has_z) {
          float zz[4];
          load4(&S.raw_z[bf][i][tt], zz);
#pragma unroll
          for (int j = 0; j < 4; ++j) o[j] *= silu_f(zz[j]);
        }
        T* dst = static_cast<T*>(a.out) + ((long long)b * dim + d) * L + t0 + tt;
        if (VEC) {
          store4(dst, o);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (tt + j < tl) dst[j] = from_f32<T>(o[j]);
        }
      }
    }
  }

  // ---- chunk results
  if (valid) {
    if (CARRY) {
      float* hw = a.ws_h + ((long long)q * BD + c_me) * kMaxDstate + g * NPT;
#pragma unroll
      for (int k = 0; k < NPT; ++k) hw[k] = h[k];
      if (g == 0) a.ws_S[(long long)q * BD + c_me] = dsum;
    } else if (q == a.nchunks - 1 && a.h_last) {
#pragma unroll
      for (int k = 0; k < NPT; ++k) {
        const int n = g * NPT + k;
        if (n < N) a.h_last[c_me * N + n] = h[k];
      }
    }
  }
  if (!CARRY && q == a.nchunks - 1 && a.conv_state_out && a.d_conv > 1) {
    // the last K-1 raw inputs of the stream conv_init ++ x (copied bit for bit)
    const int K1 = a.d_conv - 1;
    for (int e = tid; e < DT * K1; e += kThreads) {
      const int i = e / K1, j = e % K1;
      const int d = d0 + i;
      if (d >= dim) continue;
      const long long c = (long long)b * dim + d;
      const int s = L - K1 + j;
      T v;
      if (s >= 0) v = gx[c * L + s];
      else v = a.conv_init ? static_cast<const T*>(a.conv_init)[c * K1 + (K1 + s)] : from_f32<T>(0.f);
      static_cast<T*>(a.conv_state_out)[c * K1 + j] = v;
    }
  }
}

template <typename T, int NPT, bool CONV, bool VEC, bool CARRY>
cudaError_t launch_one(const ScanArgs& a, int nchunks_grid, cudaStream_t stream) {
  constexpr int DT = Cfg<NPT>::DT;
  const size_t smem = sizeof(Smem<T, NPT>);
  auto kern = scan_kernel<T, NPT, CONV, VEC, CARRY>;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) configured[dev] = 1;
  }
  dim3 grid((a.dim + DT - 1) / DT, nchunks_grid, a.batch);
  kern<<<grid, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

template <typename T, int NPT, bool CONV, bool VEC>
cudaError_t launch_pair(const ScanArgs& a, cudaStream_t stream) {
  if (a.nchunks > 1) {
    cudaError_t err = launch_one<T, NPT, CONV, VEC, true>(a, a.nchunks - 1, stream);
    if (err != cudaSuccess) return err;
  }
  return launch_one<T, NPT, CONV, VEC, false>(a, a.nchunks, stream);
}

template <typename T, int NPT>
cudaError_t dispatch_conv_vec(const ScanArgs& a, cudaStream_t s) {
  const bool conv = a.conv_w != nullptr;
  if (conv) return a.vec ? launch_pair<T, NPT, true, true>(a, s) : launch_pair<T, NPT, true, false>(a, s);
  return a.vec ? launch_pair<T, NPT, false, true>(a, s) : launch_pair<T, NPT, false, false>(a, s);
}

template <typename T>
cudaError_t dispatch_npt(const ScanArgs& a, cudaStream_t s) {
  if (a.npt == 1) return dispatch_conv_vec<T, 1>(a, s);
  return dispatch_conv_vec<T, 4>(a, s);
}

}  // namespace

size_t scan_workspace_bytes(long long channels, int nchunks) {
  if (nchunks <= 1) return 0;
  const long long m = (long long)(nchunks - 1) * channels;
  const size_t s_bytes = ((size_t)m * sizeof(float) + 255) & ~(size_t)255;
  return s_bytes + (size_t)m * kMaxDstate * sizeof(float);
}

void scan_workspace_split(void* ws, long long channels, int nchunks, float** S, float** h) {
  if (nchunks <= 1 || ws == nullptr) {
    *S = nullptr;
    *h = nullptr;
    return;
  }
  const long long m = (long long)(nchunks - 1) * channels;
  const size_t s_bytes = ((size_t)m * sizeof(float) + 255) & ~(size_t)255;
  *S = static_cast<float*>(ws);
  *h = reinterpret_cast<float*>(static_cast<char*>(ws) + s_bytes);
}

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t stream) {
  if (a.bf16) return dispatch_npt<__nv_bfloat16>(a, stream);
  return dispatch_npt<float>(a, stream);
}

}  // namespace ssm
