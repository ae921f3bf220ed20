// ssm_ssd.cu -- multi-head selective SSM with one decay per head (the layer of the structured
// state-space duality) on the 5th-generation tensor cores.
//
// What it computes ("Mamba" (ai360xpert.com / inferensys.com pages), "Mamba-2 introduces the
// Structured State Space Duality": multi-head SSM, the state dimension used like a head
// dimension, the computation mapped to structured matrix products; "Mamba" (ozercemkelahmet.com),
// "Mamba-2 and the dual view": the layer as a masked matrix product with a decaying mask). Per
// batch element b and head h, state H [P x N]:
//   Delta_t = softplus(dt[b,t,h] + dt_bias[h]),  a_t = exp(Delta_t A[h])
//   H_t = a_t H_{t-1} + Delta_t x_t B_t^T,  y_t = H_t C_t + D[h] x_t
// Chunked form (chunk of Q = 128 steps, c_t = sum of Delta A over the chunk up to t):
//   intra-chunk:  y_t += sum_{s<=t} (C_t . B_s) exp(c_t - c_s) Delta_s x_s     (masked G = C B^T)
//   chunk state:  S = sum_s exp(c_end - c_s) Delta_s B_s x_s^T                  ([N x P], from zero)
//   carry-in:     H_in(chunk q+1) = exp(c_end(q)) H_in(q) + S(q)                 (sequential, cheap)
//   inter-chunk:  y_t += exp(c_t) C_t . H_in
// Three launches: chunk states (one tcgen05 GEMM per chunk), the carry pass (CUDA cores), chunk
// outputs (tcgen05 GEMMs per chunk: G = C B^T, G' X, C H_in). Every GEMM is bf16 x bf16 into fp32
// tensor memory; operands are staged into shared memory with 16-byte cp.async copies in the
// no-swizzle core-matrix layout; the masked decay of G is applied in registers between GEMMs.
// Operands the kernels compute (G' and H_in) are carried as two bf16 terms, hi = bf16(v) and
// lo = bf16(v - hi), multiplied in two GEMMs into one accumulator: a single bf16 rounding of them
// costs up to 2^-9 of each summand, which for sums of 128 products of O(1) terms that cancel
// exceeds the bf16-I/O tolerance on a fraction of a percent of the outputs.
#include <cuda_bf16.h>

#include "ssm_device.cuh"
#include "ssm_internal.h"
#include "ssm_umma.cuh"

namespace ssm {
namespace {

constexpr int kQ = 128;  // chunk length; one thread (and one TMEM lane) per step
constexpr int kP = 64;   // head dim
constexpr int kN = 128;  // state dim
constexpr int kThreads = 128;
static_assert(kQ == kN, "the masked G' [Q x Q] reuses the B tile [Q x N]");
static_assert(kQ == kThreads, "one thread per step");

using bf16 = __nv_bfloat16;

// Shared-memory layout of the chunk-state kernel (byte offsets).
struct StateSmem {
  static constexpr int B = 0;                    // B^T [N x Q], MN-major: A operand (M = n, K = s)
  static constexpr int X = B + kQ * kN * 2;      // X [Q x P] scaled rows, MN-major: B operand (N = p, K = s)
  static constexpr int bytes = X + kQ * kP * 2;  // 48 KB
};

// Shared-memory layout of the chunk-output kernel.
struct ScanSmem {
  static constexpr int C = 0;                    // C [Q x N], K-major: A operand (M = t, K = n); then
                                                 // G'_lo [Q x Q], K-major
  static constexpr int BG = C + kQ * kN * 2;     // B [Q x N], K-major: B operand (N = s, K = n); then
                                                 // G'_hi [Q x Q], K-major: A operand (M = t, K = s)
  static constexpr int X = BG + kQ * kN * 2;     // X [Q x P], MN-major: B operand (N = p, K = s)
  static constexpr int S = X + kQ * kP * 2;      // H_in hi [N x P], MN-major: B operand (N = p, K = n);
                                                 // then c_t and Delta_t of the chunk (1 KB)
  static constexpr int SL = S + kN * kP * 2;     // H_in lo [N x P]
  static constexpr int bytes = SL + kN * kP * 2; // 112 KB: two CTAs per SM, 2 x 256 TMEM columns
};

// TMEM columns of the chunk-output kernel: G [128 x 128], C H_in [128 x 64], G' X [128 x 64].
constexpr uint32_t kColG = 0, kColOff = 128, kColDiag = 192, kScanCols = 256;
constexpr uint32_t kStateCols = 64;

// Delta_t of this thread's step and the inclusive prefix over the chunk of Delta A log2(e).
__device__ __forceinline__ void chunk_decay(const SsdArgs& a, int b, int h, int t0, int len, float* s_wsum,
                                            float& Delta, float& cs) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  Delta = 0.f;
  if (t < len) {
    const float v = to_f32(static_cast<const bf16*>(a.dt)[((long long)b * a.seqlen + t0 + t) * a.nheads + h]) +
                    (a.dt_bias ? a.dt_bias[h] : 0.f);
    Delta = a.dt_softplus ? softplus_f<true>(v) : v;
  }
  float v = Delta * a.A[h] * kLog2e;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) s_wsum[warp] = v;
  __syncthreads();
  float off = 0.f;
  for (int w = 0; w < warp; ++w) off += s_wsum[w];
  cs = v + off;
}

// 8 bf16 of a 16-byte shared-memory chunk to fp32
__device__ __forceinline__ void unpack8(const unsigned char* p, float (&f)[8]) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 x = __bfloat1622float2(e[k]);
    f[2 * k] = x.x;
    f[2 * k + 1] = x.y;
  }
}
__device__ __forceinline__ uint4 pack8(const float* f) {
  uint4 v;
  __nv_bfloat162* e = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int k = 0; k < 4; ++k) e[k] = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);
  return v;
}

// ---- launch 1: S(q) = sum_s exp(c_end - c_s) Delta_s B_s x_s^T for every chunk q, as
// D[n][p] = sum_s B[s][n] * (w_s x[s][p]); one CTA per (chunk, head, batch).
__global__ void __launch_bounds__(kThreads) ssd_chunk_state_kernel(const SsdArgs a) {
  extern __shared__ __align__(128) unsigned char sm[];
  __shared__ uint64_t mbar;
  __shared__ uint32_t tslot;
  __shared__ float s_wsum[4];
  __shared__ float s_cs_end;
  const int t = threadIdx.x, warp = t >> 5;
  const int q = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int L = a.seqlen, H = a.nheads;
  const int t0 = q * kQ, len = min(kQ, L - t0);
  const bf16* gB = static_cast<const bf16*>(a.B);
  const bf16* gx = static_cast<const bf16*>(a.x);
  unsigned char* sB = sm + StateSmem::B;
  unsigned char* sX = sm + StateSmem::X;

  // stage: a 16-byte chunk of row s holds 8 consecutive n (or p) at step s; rows past the
  // sequence end are zero-filled
  for (int i = t; i < kQ * kN / 8; i += kThreads) {
    const int s = i / (kN / 8), n0 = (i % (kN / 8)) * 8;
    const bool ok = s < len;
    cp_async16(sB + umma::mnmajor_off(n0, s, kN), ok ? (const void*)(gB + ((long long)b * L + t0 + s) * kN + n0)
                                                     : (const void*)gB, ok ? 16u : 0u);
  }
  for (int i = t; i < kQ * kP / 8; i += kThreads) {
    const int s = i / (kP / 8), p0 = (i % (kP / 8)) * 8;
    const bool ok = s < len;
    cp_async16(sX + umma::mnmajor_off(p0, s, kP),
               ok ? (const void*)(gx + (((long long)b * L + t0 + s) * H + h) * kP + p0) : (const void*)gx,
               ok ? 16u : 0u);
  }
  cp_async_commit();
  float Delta, cs;
  chunk_decay(a, b, h, t0, len, s_wsum, Delta, cs);
  if (t == kQ - 1) s_cs_end = cs;  // steps past the end add nothing, so the last prefix is the total
  cp_async_wait<0>();
  __syncthreads();
  const float cs_end = s_cs_end;
  // row t of X times Delta_t exp(c_end - c_t), rounded back to bf16 in place
  const float w = Delta * ex2_approx(cs_end - cs);
#pragma unroll
  for (int j = 0; j < kP / 8; ++j) {
    unsigned char* p = sX + umma::mnmajor_off(j * 8, t, kP);
    float f[8];
    unpack8(p, f);
#pragma unroll
    for (int k = 0; k < 8; ++k) f[k] *= w;
    *reinterpret_cast<uint4*>(p) = pack8(f);
  }
  umma::fence_proxy_async();
  if (warp == 0) umma::tmem_alloc(&tslot, kStateCols);
  if (t == 0) umma::mbar_init(&mbar, 1);
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tbase = tslot;
  if (t == 0) {
    constexpr uint32_t idesc = umma::idesc_bf16(kN, kP, true, true);
#pragma unroll 1
    for (int kk = 0; kk < kQ / 16; ++kk)
      umma::mma_bf16(tbase, umma::desc_mnmajor(smem_addr(sB), kk, kN), umma::desc_mnmajor(smem_addr(sX), kk, kP),
                     idesc, kk > 0);
    umma::mma_commit(&mbar);
  }
  const bool ok = __all_sync(0xffffffffu, umma::mbar_wait(&mbar, 0));
  umma::fence_after_sync();
  const long long bhq = ((long long)b * H + h) * a.nchunks + q;
  if (ok) {
    float* dst = a.ws_S + (bhq * kN + t) * kP;  // row n = t of S
#pragma unroll
    for (int c0 = 0; c0 < kP; c0 += 16) {
      float v[16];
      umma::tmem_ld16(tbase + ((uint32_t)(warp * 32) << 16) + c0, v);
#pragma unroll
      for (int j = 0; j < 16; j += 4)
        *reinterpret_cast<float4*>(dst + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
    }
  } else if ((t & 31) == 0) {
    atomicExch(a.ws_status, 1);
  }
  if (t == 0) a.ws_cs[bhq] = cs_end;
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 0) umma::tmem_dealloc(tbase, kStateCols);
}

// ---- launch 2: the state entering each chunk, H_in(q+1) = exp(c_end(q)) H_in(q) + S(q), kept in
// fp32 and written as two bf16 terms [N x P] for the output GEMMs; the final state goes to
// h_last [P x N].
constexpr int kPassThreads = 256;
__global__ void __launch_bounds__(kPassThreads) ssd_state_pass_kernel(const SsdArgs a) {
  constexpr int kE = kN * kP;
  constexpr int kPer = kE / 4 / kPassThreads;  // float4 groups per thread
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const long long bh = (long long)b * a.nheads + h;
  float4 S[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int e = (k * kPassThreads + tid) * 4, n = e / kP, p = e % kP;
    if (a.h0) {
      const float* h0 = a.h0 + bh * kE;  // [P][N]
      S[k] = make_float4(h0[p * kN + n], h0[(p + 1) * kN + n], h0[(p + 2) * kN + n], h0[(p + 3) * kN + n]);
    } else {
      S[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  bf16* sin = static_cast<bf16*>(a.ws_Sin);
  bf16* sin_lo = static_cast<bf16*>(a.ws_Sin_lo);
  for (int q = 0; q < a.nchunks; ++q) {
    const long long base = (bh * a.nchunks + q) * kE;
    const float dec = ex2_approx(a.ws_cs[bh * a.nchunks + q]);
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int e = (k * kPassThreads + tid) * 4;
      const __nv_bfloat162 h01 = __floats2bfloat162_rn(S[k].x, S[k].y), h23 = __floats2bfloat162_rn(S[k].z, S[k].w);
      const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
      const __nv_bfloat162 l01 = __floats2bfloat162_rn(S[k].x - f01.x, S[k].y - f01.y);
      const __nv_bfloat162 l23 = __floats2bfloat162_rn(S[k].z - f23.x, S[k].w - f23.y);
      uint2 u;
      u.x = *reinterpret_cast<const uint32_t*>(&h01);
      u.y = *reinterpret_cast<const uint32_t*>(&h23);
      *reinterpret_cast<uint2*>(sin + base + e) = u;
      u.x = *reinterpret_cast<const uint32_t*>(&l01);
      u.y = *reinterpret_cast<const uint32_t*>(&l23);
      *reinterpret_cast<uint2*>(sin_lo + base + e) = u;
      const float4 d = *reinterpret_cast<const float4*>(a.ws_S + base + e);
      S[k] = make_float4(fmaf(dec, S[k].x, d.x), fmaf(dec, S[k].y, d.y), fmaf(dec, S[k].z, d.z),
                         fmaf(dec, S[k].w, d.w));
    }
  }
  if (a.h_last) {
    float* hl = a.h_last + bh * kE;  // [P][N]
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int e = (k * kPassThreads + tid) * 4, n = e / kP, p = e % kP;
      hl[p * kN + n] = S[k].x;
      hl[(p + 1) * kN + n] = S[k].y;
      hl[(p + 2) * kN + n] = S[k].z;
      hl[(p + 3) * kN + n] = S[k].w;
    }
  }
}

// ---- launch 3: y_t = sum_{s<=t} G[t][s] exp(c_t - c_s) Delta_s x_s + exp(c_t) C_t . H_in + D x_t.
__global__ void __launch_bounds__(kThreads) ssd_chunk_scan_kernel(const SsdArgs a) {
  extern __shared__ __align__(128) unsigned char sm[];
  __shared__ uint64_t mbar;
  __shared__ uint32_t tslot;
  __shared__ float s_wsum[4];
  const int t = threadIdx.x, warp = t >> 5;
  const int q = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int L = a.seqlen, H = a.nheads;
  const int t0 = q * kQ, len = min(kQ, L - t0);
  const bf16* gB = static_cast<const bf16*>(a.B);
  const bf16* gC = static_cast<const bf16*>(a.C);
  const bf16* gx = static_cast<const bf16*>(a.x);
  const long long bhq = ((long long)b * H + h) * a.nchunks + q;
  const bf16* gS = static_cast<const bf16*>(a.ws_Sin) + bhq * kN * kP;
  const bf16* gSl = static_cast<const bf16*>(a.ws_Sin_lo) + bhq * kN * kP;
  unsigned char* sC = sm + ScanSmem::C;
  unsigned char* sBG = sm + ScanSmem::BG;
  unsigned char* sX = sm + ScanSmem::X;
  unsigned char* sS = sm + ScanSmem::S;
  unsigned char* sSl = sm + ScanSmem::SL;
  float* s_cs = reinterpret_cast<float*>(sS);  // after the first GEMMs: c_t and Delta_t
  float* s_dl = s_cs + kQ;

  for (int i = t; i < kQ * kN / 8; i += kThreads) {
    const int s = i / (kN / 8), n0 = (i % (kN / 8)) * 8;
    const bool ok = s < len;
    const long long g = ((long long)b * L + t0 + s) * kN + n0;
    cp_async16(sC + umma::kmajor_off(s, n0, kN), ok ? (const void*)(gC + g) : (const void*)gC, ok ? 16u : 0u);
    cp_async16(sBG + umma::kmajor_off(s, n0, kN), ok ? (const void*)(gB + g) : (const void*)gB, ok ? 16u : 0u);
  }
  for (int i = t; i < kQ * kP / 8; i += kThreads) {
    const int s = i / (kP / 8), p0 = (i % (kP / 8)) * 8;
    const bool ok = s < len;
    cp_async16(sX + umma::mnmajor_off(p0, s, kP),
               ok ? (const void*)(gx + (((long long)b * L + t0 + s) * H + h) * kP + p0) : (const void*)gx,
               ok ? 16u : 0u);
  }
  for (int i = t; i < kN * kP / 8; i += kThreads) {
    const int n = i / (kP / 8), p0 = (i % (kP / 8)) * 8;
    cp_async16(sS + umma::mnmajor_off(p0, n, kP), gS + n * kP + p0, 16u);
    cp_async16(sSl + umma::mnmajor_off(p0, n, kP), gSl + n * kP + p0, 16u);
  }
  cp_async_commit();
  float Delta, cs;
  chunk_decay(a, b, h, t0, len, s_wsum, Delta, cs);
  cp_async_wait<0>();
  umma::fence_proxy_async();
  if (warp == 0) umma::tmem_alloc(&tslot, kScanCols);
  if (t == 0) umma::mbar_init(&mbar, 1);
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tbase = tslot;
  const uint32_t trow = tbase + ((uint32_t)(warp * 32) << 16);
  if (t == 0) {
    constexpr uint32_t idG = umma::idesc_bf16(kQ, kQ, false, false);
    constexpr uint32_t idOff = umma::idesc_bf16(kQ, kP, false, true);
#pragma unroll 1
    for (int kk = 0; kk < kN / 16; ++kk)
      umma::mma_bf16(tbase + kColG, umma::desc_kmajor(smem_addr(sC), kk, kN),
                     umma::desc_kmajor(smem_addr(sBG), kk, kN), idG, kk > 0);
#pragma unroll 1
    for (int kk = 0; kk < kN / 16; ++kk)
      umma::mma_bf16(tbase + kColOff, umma::desc_kmajor(smem_addr(sC), kk, kN),
                     umma::desc_mnmajor(smem_addr(sS), kk, kP), idOff, kk > 0);
#pragma unroll 1
    for (int kk = 0; kk < kN / 16; ++kk)
      umma::mma_bf16(tbase + kColOff, umma::desc_kmajor(smem_addr(sC), kk, kN),
                     umma::desc_mnmajor(smem_addr(sSl), kk, kP), idOff, true);
    umma::mma_commit(&mbar);
  }
  bool ok = __all_sync(0xffffffffu, umma::mbar_wait(&mbar, 0));
  umma::fence_after_sync();
  // the GEMMs that read C, B and H_in have completed: their tiles take c_t, Delta_t and G'
  s_cs[t] = cs;
  s_dl[t] = Delta;
  __syncthreads();
  // G' = G masked to s <= t, times exp(c_t - c_s) Delta_s, as hi + lo bf16 terms in the places of
  // the B and C tiles
#pragma unroll 1
  for (int s0 = 0; s0 < kQ; s0 += 16) {
    float g[16];
    if (ok) umma::tmem_ld16(trow + kColG + s0, g);
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int s = s0 + j;
      const float e = ex2_approx(cs - s_cs[s]) * s_dl[s];
      v[j] = (ok && s <= t) ? g[j] * e : 0.f;
    }
    float hi[16], lo[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      hi[j] = __bfloat162float(__float2bfloat16_rn(v[j]));
      lo[j] = v[j] - hi[j];
    }
    *reinterpret_cast<uint4*>(sBG + umma::kmajor_off(t, s0, kQ)) = pack8(hi);
    *reinterpret_cast<uint4*>(sBG + umma::kmajor_off(t, s0 + 8, kQ)) = pack8(hi + 8);
    *reinterpret_cast<uint4*>(sC + umma::kmajor_off(t, s0, kQ)) = pack8(lo);
    *reinterpret_cast<uint4*>(sC + umma::kmajor_off(t, s0 + 8, kQ)) = pack8(lo + 8);
  }
  umma::fence_proxy_async();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  if (t == 0) {
    constexpr uint32_t idDiag = umma::idesc_bf16(kQ, kP, false, true);
#pragma unroll 1
    for (int kk = 0; kk < kQ / 16; ++kk)
      umma::mma_bf16(tbase + kColDiag, umma::desc_kmajor(smem_addr(sBG), kk, kQ),
                     umma::desc_mnmajor(smem_addr(sX), kk, kP), idDiag, kk > 0);
#pragma unroll 1
    for (int kk = 0; kk < kQ / 16; ++kk)
      umma::mma_bf16(tbase + kColDiag, umma::desc_kmajor(smem_addr(sC), kk, kQ),
                     umma::desc_mnmajor(smem_addr(sX), kk, kP), idDiag, true);
    umma::mma_commit(&mbar);
  }
  ok = __all_sync(0xffffffffu, umma::mbar_wait(&mbar, 1)) && ok;
  umma::fence_after_sync();
  if (!ok && (t & 31) == 0) atomicExch(a.ws_status, 1);
  // epilogue: row t
  const float et = ex2_approx(cs);
  const float Dh = a.D ? a.D[h] : 0.f;
  bf16* yrow = static_cast<bf16*>(a.y) + (((long long)b * L + t0 + t) * H + h) * kP;
#pragma unroll 1
  for (int p0 = 0; p0 < kP; p0 += 16) {
    float yd[16], yo[16];
    if (ok) {
      umma::tmem_ld16(trow + kColDiag + p0, yd);
      umma::tmem_ld16(trow + kColOff + p0, yo);
    }
    float xv[16];
    unpack8(sX + umma::mnmajor_off(p0, t, kP), *reinterpret_cast<float(*)[8]>(xv));
    unpack8(sX + umma::mnmajor_off(p0 + 8, t, kP), *reinterpret_cast<float(*)[8]>(xv + 8));
    float o[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j] = ok ? fmaf(et, yo[j], yd[j]) + Dh * xv[j] : 0.f;
    if (t < len) {
      *reinterpret_cast<uint4*>(yrow + p0) = pack8(o);
      *reinterpret_cast<uint4*>(yrow + p0 + 8) = pack8(o + 8);
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 0) umma::tmem_dealloc(tbase, kScanCols);
}

}  // namespace

int ssd_chunk_len() { return kQ; }

size_t ssd_workspace_bytes(int batch, int nheads, int nchunks) {
  const size_t pairs = (size_t)batch * nheads * nchunks;
  const size_t cs = (pairs * sizeof(float) + 255) & ~(size_t)255;
  return 256 + cs + pairs * kN * kP * (sizeof(float) + 2 * sizeof(bf16));
}

void ssd_workspace_split(void* ws, int batch, int nheads, int nchunks, SsdArgs& a) {
  const size_t pairs = (size_t)batch * nheads * nchunks;
  const size_t cs = (pairs * sizeof(float) + 255) & ~(size_t)255;
  char* p = static_cast<char*>(ws);
  a.ws_status = reinterpret_cast<int*>(p);
  a.ws_cs = reinterpret_cast<float*>(p + 256);
  a.ws_S = reinterpret_cast<float*>(p + 256 + cs);
  a.ws_Sin = p + 256 + cs + pairs * kN * kP * sizeof(float);
  a.ws_Sin_lo = p + 256 + cs + pairs * kN * kP * (sizeof(float) + sizeof(bf16));
}

cudaError_t launch_ssd(const SsdArgs& a, cudaStream_t stream) {
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    err = cudaFuncSetAttribute(ssd_chunk_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, StateSmem::bytes);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(ssd_chunk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ScanSmem::bytes);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) configured[dev] = 1;
  }
  err = cudaMemsetAsync(a.ws_status, 0, sizeof(int), stream);
  if (err != cudaSuccess) return err;
  const dim3 grid(a.nchunks, a.nheads, a.batch);
  ssd_chunk_state_kernel<<<grid, kThreads, StateSmem::bytes, stream>>>(a);
  ssd_state_pass_kernel<<<dim3(a.nheads, a.batch), kPassThreads, 0, stream>>>(a);
  ssd_chunk_scan_kernel<<<grid, kThreads, ScanSmem::bytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ssm
