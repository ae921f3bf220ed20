// ssm_ssd.cu -- multi-head selective SSM with one decay per head (the layer of the structured
// state-space duality) on the 5th-generation tensor cores.
//
// What it computes ("Mamba" (ai360xpert.com / inferensys.com pages), "Mamba-2 introduces the
// Structured State Space Duality": multi-head SSM, the state dimension used like a head
// dimension, the computation mapped to structured matrix products; "Mamba" (ozercemkelahmet.com),
// "Mamba-2 and the dual view": the layer as a masked matrix product with a decaying mask). Per
// batch element b and head h, state H [N x P] (stored transposed to the public [P x N]):
//   Delta_t = softplus(dt[b,t,h] + dt_bias[h]),  a_t = exp(Delta_t A[h])
//   H_t = a_t H_{t-1} + Delta_t B_t x_t^T,  y_t = H_t^T C_t + D[h] x_t
// Chunked form (chunks of Q = 128 steps; c_t = sum of Delta A over the chunk up to t):
//   y_t   = sum_{s<=t} (C_t . B_s) exp(c_t - c_s) Delta_s x_s  +  exp(c_t) C_t . H_in  +  D x_t
//   H_out = exp(c_end) H_in + sum_s exp(c_end - c_s) Delta_s B_s x_s^T
//
// Design. One CTA of 256 threads per (batch, head) walks the chunks in order and keeps the
// running state on the chip: fp32 in registers (row n of H is held by threads n and n + 128,
// 32 columns each), and as the bf16 operand of the next chunk's GEMM in shared memory. Rows of
// the tensor-memory accumulators map to threads; the two warps that share a row split its
// columns. Per chunk, two rounds of tcgen05 GEMMs
// (bf16 operands, fp32 accumulators in tensor memory, issued by one thread, completion through an
// mbarrier):
//   round A:  G = C B^T [Q x Q] and Y_off = C H_in [Q x P];
//   (threads) G' = G masked to s <= t and scaled by exp(c_t - c_s) Delta_s; B~ = B scaled per row
//             by Delta_s exp(c_end - c_s);
//   round B:  Y_diag = G' X [Q x P] and S = B~^T X [N x P];
//   (threads) y = Y_diag + exp(c_t) Y_off + D x; H <- exp(c_end) H + S.
// The next chunk's C, B and X are copied in while the epilogue and the state update of the current
// one run: when the sequence length is a multiple of the chunk, by three TMA bulk-tensor copies
// issued by one thread, whose 4-D / 5-D boxes (8 elements, 8 rows, column groups, row groups)
// land directly in the no-swizzle core-matrix layout; otherwise by 16-byte cp.async copies with
// zero fill past the end. The B tile serves as
// the K-major B operand of G and, scaled, as the MN-major A operand of S: the two layouts are the
// same bytes. Operands the kernel computes (G' and H_in) are carried as two bf16 terms,
// hi = bf16(v) and lo = bf16(v - hi), multiplied in two GEMMs into one accumulator: a single bf16
// rounding of them costs up to 2^-9 of each summand, which for sums of 128 products of O(1)
// terms that cancel exceeds the bf16-I/O tolerance on a fraction of a percent of the outputs.
#include <cstring>

#include <cuda.h>  // CUtensorMap and its encoder's signature (resolved at run time, not linked)
#include <cuda_bf16.h>

#include "ssm_device.cuh"
#include "ssm_internal.h"
#include "ssm_umma.cuh"

namespace ssm {
namespace {

constexpr int kQ = 128;  // chunk length; one TMEM lane per step
constexpr int kP = 64;   // head dim
constexpr int kN = 128;  // state dim
constexpr int kThreads = 256;  // two threads per row (step or state row), each with half the columns
constexpr int kHalfP = kP / 2;
static_assert(kQ == kN && 2 * kQ == kThreads, "two threads per step and per state row");

using bf16 = __nv_bfloat16;

// Shared-memory layout (byte offsets); 112 KB, so two CTAs fit an SM.
struct Smem {
  static constexpr int C = 0;                    // C [Q x N], K-major: A operand of G and Y_off (M = t,
                                                 // K = n); after round A, G'_hi [Q x Q], K-major
  static constexpr int B = C + kQ * kN * 2;      // B [Q x N]: K-major B operand of G (N = s, K = n); scaled,
                                                 // the MN-major A operand of S (M = n, K = s)
  static constexpr int X = B + kQ * kN * 2;      // X [Q x P], MN-major: B operand of Y_diag and S (N = p, K = s)
  static constexpr int H = X + kQ * kP * 2;      // H_in hi, lo [N x P] each, MN-major: B operand of Y_off
                                                 // (N = p, K = n); after round A, G'_lo [Q x Q], K-major
  static constexpr int HL = H + kN * kP * 2;
  static constexpr int bytes = HL + kN * kP * 2;
};

// TMEM columns: G [128 x 128] (Y_diag [128 x 64] after it), Y_off [128 x 64], S [128 x 64].
constexpr uint32_t kColG = 0, kColDiag = 0, kColOff = 128, kColS = 192, kCols = 256;

__device__ __forceinline__ void unpack8(const unsigned char* p, float* f) {
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
// v = hi + lo with hi = bf16(v), lo = bf16(v - hi), 8 values
__device__ __forceinline__ void split8(const float* v, uint4& hi, uint4& lo) {
  float h[8], l[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    h[k] = __bfloat162float(__float2bfloat16_rn(v[k]));
    l[k] = v[k] - h[k];
  }
  hi = pack8(h);
  lo = pack8(l);
}

// TMA: the tiles come from three tensor maps (C and B: 4-D, X: 5-D, described at launch_ssd).
template <bool TMA>
__global__ void __launch_bounds__(kThreads, 2)
    ssd_fused_kernel(const SsdArgs a, const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmX) {
  extern __shared__ __align__(128) unsigned char sm[];
  __shared__ uint64_t mbar;
  __shared__ uint64_t tbar;  // TMA completion
  __shared__ uint32_t tslot;
  __shared__ float s_wsum[8];
  __shared__ float s_z[kQ];  // lg2(Delta_s) - c_s: exp(c_t - c_s) Delta_s = 2^(c_t + z_s) in log2 units
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = tid & (kQ - 1);  // the row (step t, or state row n) of this thread
  const int half = tid >> 7;     // which half of the row's columns
  const int wq = warp & 3;       // TMEM lane quarter of this warp
  const int h = blockIdx.x, b = blockIdx.y;
  const int L = a.seqlen, H = a.nheads, nc = a.nchunks;
  const long long bh = (long long)b * H + h;
  const bf16* gB = static_cast<const bf16*>(a.B);
  const bf16* gC = static_cast<const bf16*>(a.C);
  const bf16* gx = static_cast<const bf16*>(a.x);
  const bf16* gdt = static_cast<const bf16*>(a.dt);
  unsigned char* sC = sm + Smem::C;
  unsigned char* sB = sm + Smem::B;
  unsigned char* sX = sm + Smem::X;
  unsigned char* sH = sm + Smem::H;
  unsigned char* sHL = sm + Smem::HL;
  const float A2 = a.A[h] * kLog2e;
  const float bias = a.dt_bias ? a.dt_bias[h] : 0.f;
  const float Dh = a.D ? a.D[h] : 0.f;

  // C, B, X of chunk q into their tiles; rows past the sequence end are zero-filled. Copy k of
  // thread tid: C / B row s = tid/16 + 16k, columns 8 (tid%16) ..; X row s = tid/8 + 32k, columns
  // 8 (tid%8) .. (the core-matrix offsets of those rows and columns, written out)
  const uint32_t cb_soff = (uint32_t)((tid / 128) * 2048 + (tid % 16) * 128 + ((tid / 16) % 8) * 16);  // + 4096 k
  const uint32_t x_soff = (uint32_t)((tid / 64) * 1024 + (tid % 8) * 128 + ((tid / 8) % 8) * 16);     // + 4096 k
  auto stage = [&](int q) {
    const int t0 = q * kQ, len = min(kQ, L - t0);
    if (TMA) {  // whole chunks only: no row of another sequence, none past the end
      if (tid == 0) {
        umma::fence_proxy_async();
        umma::mbar_expect_tx(&tbar, (uint32_t)(2 * kQ * kN * 2 + kQ * kP * 2));
        const int r8 = (int)(((long long)b * L + t0) / 8);
        umma::tma_load_4d(sC, &tmC, 0, 0, 0, r8, &tbar);
        umma::tma_load_4d(sB, &tmB, 0, 0, 0, r8, &tbar);
        umma::tma_load_5d(sX, &tmX, 0, 0, 0, r8, h, &tbar);
      }
      return;
    }
    const long long cbg = ((long long)b * L + t0 + tid / 16) * kN + (tid % 16) * 8;
#pragma unroll
    for (int k = 0; k < kQ * kN / 8 / kThreads; ++k) {
      const bool ok = tid / 16 + 16 * k < len;
      const long long g = cbg + (long long)k * 16 * kN;
      cp_async16(sC + cb_soff + 4096u * k, ok ? (const void*)(gC + g) : (const void*)gC, ok ? 16u : 0u);
      cp_async16(sB + cb_soff + 4096u * k, ok ? (const void*)(gB + g) : (const void*)gB, ok ? 16u : 0u);
    }
    const long long xg = (((long long)b * L + t0 + tid / 8) * H + h) * kP + (tid % 8) * 8;
#pragma unroll
    for (int k = 0; k < kQ * kP / 8 / kThreads; ++k) {
      const bool ok = tid / 8 + 32 * k < len;
      const long long g = xg + (long long)k * 32 * H * kP;
      cp_async16(sX + x_soff + 4096u * k, ok ? (const void*)(gx + g) : (const void*)gx, ok ? 16u : 0u);
    }
    cp_async_commit();
  };
  auto load_dt = [&](int q) -> float {
    const int s = q * kQ + t;
    return s < L ? to_f32(gdt[((long long)b * L + s) * H + h]) : 0.f;
  };

  // running state: row n = t of H [N x P], columns pb .. pb + 31, fp32
  const int pb = half * kHalfP;
  float Hs[kHalfP];
#pragma unroll
  for (int p = 0; p < kHalfP; ++p) Hs[p] = a.h0 ? a.h0[(bh * kP + pb + p) * kN + t] : 0.f;
  // its bf16 hi / lo operand tiles (element (p, n) of the B operand of Y_off)
  auto write_state = [&]() {
#pragma unroll
    for (int p0 = 0; p0 < kHalfP; p0 += 8) {
      uint4 hi, lo;
      split8(Hs + p0, hi, lo);
      *reinterpret_cast<uint4*>(sH + umma::mnmajor_off(pb + p0, t, kP)) = hi;
      *reinterpret_cast<uint4*>(sHL + umma::mnmajor_off(pb + p0, t, kP)) = lo;
    }
  };
  write_state();
  float dtv = load_dt(0);
  if (warp == 0) umma::tmem_alloc(&tslot, kCols);
  if (tid == 0) {
    umma::mbar_init(&mbar, 1);
    umma::mbar_init(&tbar, 1);
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  stage(0);
  uint32_t tparity = 0;
  const uint32_t tbase = tslot;
  const uint32_t trow = tbase + ((uint32_t)(wq * 32) << 16);
  uint32_t parity = 0;
  bool ok = true;

#pragma unroll 1
  for (int q = 0; q < nc; ++q) {
    const int t0 = q * kQ, len = min(kQ, L - t0);
    // ---- Delta_t and the prefix c_t (log2 units) of this chunk; the next chunk's dt in flight
    float Delta = 0.f;
    if (t < len) Delta = a.dt_softplus ? softplus_f<true>(dtv + bias) : dtv + bias;
    if (q + 1 < nc) dtv = load_dt(q + 1);
    float v = Delta * A2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float n = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += n;
    }
    if (lane == 31) s_wsum[warp] = v;
    __syncthreads();
    // both halves scan all 128 steps; each reads its own half's warp totals
    const float* ws = s_wsum + 4 * half;
    float off = 0.f, c_end = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      if (w < wq) off += ws[w];
      if (w < 3) c_end += ws[w];
    }
    c_end += ws[3];
    const float cs = v + off;
    if (half == 0) s_z[t] = lg2_approx(Delta) - cs;  // -inf past the end (Delta = 0): those columns vanish
    if (TMA) {
      ok = __syncthreads_and(umma::mbar_wait(&tbar, tparity)) && ok;
      tparity ^= 1;
      if (!ok) break;
    } else {
      cp_async_wait<0>();
    }
    umma::fence_proxy_async();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();

    // ---- round A: G = C B^T, Y_off = C H_in (hi + lo)
    if (tid == 0) {
      constexpr uint32_t idG = umma::idesc_bf16(kQ, kQ, false, false);
      constexpr uint32_t idOff = umma::idesc_bf16(kQ, kP, false, true);
#pragma unroll 1
      for (int kk = 0; kk < kN / 16; ++kk)
        umma::mma_bf16(tbase + kColG, umma::desc_kmajor(smem_addr(sC), kk, kN),
                       umma::desc_kmajor(smem_addr(sB), kk, kN), idG, kk > 0);
#pragma unroll 1
      for (int kk = 0; kk < kN / 16; ++kk)
        umma::mma_bf16(tbase + kColOff, umma::desc_kmajor(smem_addr(sC), kk, kN),
                       umma::desc_mnmajor(smem_addr(sH), kk, kP), idOff, kk > 0);
#pragma unroll 1
      for (int kk = 0; kk < kN / 16; ++kk)
        umma::mma_bf16(tbase + kColOff, umma::desc_kmajor(smem_addr(sC), kk, kN),
                       umma::desc_mnmajor(smem_addr(sHL), kk, kP), idOff, true);
      umma::mma_commit(&mbar);
    }
    ok = __syncthreads_and(umma::mbar_wait(&mbar, parity)) && ok;
    parity ^= 1;
    umma::fence_after_sync();
    if (!ok) break;

    // ---- G' (hi into the C tile, lo into the H tiles) and B~ = Delta_s exp(c_end - c_s) B_s
#pragma unroll 1
    for (int j2 = 0; j2 < 2; ++j2) {
      const int s0 = 32 * (2 * j2 + half);
      uint4 hi[4], lo[4];
      if (s0 < 32 * (wq + 1)) {  // some row of this warp reaches column s0
        float g[32];
        umma::tmem_ld32(trow + kColG + s0, g);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int s = s0 + j;
          g[j] = s <= t ? g[j] * ex2_approx(cs + s_z[s]) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) split8(g + 8 * k, hi[k], lo[k]);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) hi[k] = lo[k] = make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        *reinterpret_cast<uint4*>(sC + umma::kmajor_off(t, s0 + 8 * k, kQ)) = hi[k];
        *reinterpret_cast<uint4*>(sH + umma::kmajor_off(t, s0 + 8 * k, kQ)) = lo[k];
      }
    }
    {
      const float w = Delta * ex2_approx(c_end - cs);
#pragma unroll 4
      for (int n0 = half * (kN / 2); n0 < (half + 1) * (kN / 2); n0 += 8) {
        unsigned char* p = sB + umma::kmajor_off(t, n0, kN);
        float f[8];
        unpack8(p, f);
#pragma unroll
        for (int k = 0; k < 8; ++k) f[k] *= w;
        *reinterpret_cast<uint4*>(p) = pack8(f);
      }
    }
    umma::fence_proxy_async();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();

    // ---- round B: Y_diag = G' X (hi + lo), S = B~^T X
    if (tid == 0) {
      constexpr uint32_t idDiag = umma::idesc_bf16(kQ, kP, false, true);
      constexpr uint32_t idS = umma::idesc_bf16(kN, kP, true, true);
#pragma unroll 1
      for (int kk = 0; kk < kQ / 16; ++kk)
        umma::mma_bf16(tbase + kColDiag, umma::desc_kmajor(smem_addr(sC), kk, kQ),
                       umma::desc_mnmajor(smem_addr(sX), kk, kP), idDiag, kk > 0);
#pragma unroll 1
      for (int kk = 0; kk < kQ / 16; ++kk)
        umma::mma_bf16(tbase + kColDiag, umma::desc_kmajor(smem_addr(sH), kk, kQ),
                       umma::desc_mnmajor(smem_addr(sX), kk, kP), idDiag, true);
#pragma unroll 1
      for (int kk = 0; kk < kQ / 16; ++kk)
        umma::mma_bf16(tbase + kColS, umma::desc_mnmajor(smem_addr(sB), kk, kN),
                       umma::desc_mnmajor(smem_addr(sX), kk, kP), idS, kk > 0);
      umma::mma_commit(&mbar);
    }
    // this step's x, for the skip term, before the tile is refilled
    uint4 xr[kHalfP / 8];
#pragma unroll
    for (int j = 0; j < kHalfP / 8; ++j)
      xr[j] = *reinterpret_cast<const uint4*>(sX + umma::mnmajor_off(pb + 8 * j, t, kP));
    ok = __syncthreads_and(umma::mbar_wait(&mbar, parity)) && ok;
    parity ^= 1;
    umma::fence_after_sync();
    if (!ok) break;
    // every operand tile is free: bring in the next chunk while this one finishes
    if (q + 1 < nc) stage(q + 1);

    // ---- epilogue (row t) and state update (row n = t)
    const float et = ex2_approx(cs), dec = ex2_approx(c_end);
    bf16* yrow = static_cast<bf16*>(a.y) + (((long long)b * L + t0 + t) * H + h) * kP;
#pragma unroll
    for (int p0 = 0; p0 < kHalfP; p0 += 16) {
      float yd[16], yo[16], sv[16];
      umma::tmem_ld16x3(trow + kColDiag + pb + p0, trow + kColOff + pb + p0, trow + kColS + pb + p0, yd, yo, sv);
      float xv[16];
      unpack8(reinterpret_cast<const unsigned char*>(&xr[p0 / 8]), xv);
      unpack8(reinterpret_cast<const unsigned char*>(&xr[p0 / 8 + 1]), xv + 8);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        yd[j] = fmaf(et, yo[j], yd[j]) + Dh * xv[j];
        Hs[p0 + j] = fmaf(dec, Hs[p0 + j], sv[j]);
      }
      if (t < len) {
        *reinterpret_cast<uint4*>(yrow + pb + p0) = pack8(yd);
        *reinterpret_cast<uint4*>(yrow + pb + p0 + 8) = pack8(yd + 8);
      }
    }
    write_state();
    umma::fence_before_sync();
  }

  if (!ok) {
    if (tid == 0) atomicExch(a.ws_status, 1);
  } else if (a.h_last) {
#pragma unroll
    for (int p = 0; p < kHalfP; ++p) a.h_last[(bh * kP + pb + p) * kN + t] = Hs[p];
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 0) umma::tmem_dealloc(tbase, kCols);
}

// cuTensorMapEncodeTiled, looked up once through the runtime (the library does not link the
// driver library itself)
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiled encoder() {
  static EncodeTiled fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
    cudaGetLastError();
  }
  return fn;
}

// The tensor maps of the TMA path. Rows are flat (batch * seqlen + t). C, B [rows, 128]: dims
// (n%8, row%8, n/8, row/8); X [rows, heads, 64]: dims (p%8, row%8, p/8, row/8, head). A box
// (8, 8, all column groups, 16 row groups) is one 128-row chunk in core-matrix order.
bool make_maps(const SsdArgs& a, CUtensorMap* mC, CUtensorMap* mB, CUtensorMap* mX) {
  EncodeTiled enc = encoder();
  if (!enc) return false;
  const cuuint64_t rows = (cuuint64_t)a.batch * a.seqlen;
  const cuuint64_t dCB[4] = {8, 8, kN / 8, rows / 8};
  const cuuint64_t sCB[3] = {kN * 2, 16, 8 * kN * 2};
  const cuuint32_t bCB[4] = {8, 8, kN / 8, kQ / 8};
  const cuuint32_t e4[4] = {1, 1, 1, 1};
  const cuuint64_t H = (cuuint64_t)a.nheads;
  const cuuint64_t dX[5] = {8, 8, kP / 8, rows / 8, H};
  const cuuint64_t sX[4] = {H * kP * 2, 16, 8 * H * kP * 2, kP * 2};
  const cuuint32_t bX[5] = {8, 8, kP / 8, kQ / 8, 1};
  const cuuint32_t e5[5] = {1, 1, 1, 1, 1};
  auto go = [&](CUtensorMap* m, const void* base, cuuint32_t rank, const cuuint64_t* d, const cuuint64_t* st,
                const cuuint32_t* bx, const cuuint32_t* el) {
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), d, st, bx, el,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  return go(mC, a.C, 4, dCB, sCB, bCB, e4) && go(mB, a.B, 4, dCB, sCB, bCB, e4) && go(mX, a.x, 5, dX, sX, bX, e5);
}

}  // namespace

int ssd_chunk_len() { return kQ; }

size_t ssd_workspace_bytes(int batch, int nheads, int nchunks) {
  (void)batch;
  (void)nheads;
  (void)nchunks;
  return 256;  // the status word
}

void ssd_workspace_split(void* ws, int batch, int nheads, int nchunks, SsdArgs& a) {
  (void)batch;
  (void)nheads;
  (void)nchunks;
  a.ws_status = static_cast<int*>(ws);
}

cudaError_t launch_ssd(const SsdArgs& a, cudaStream_t stream) {
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    err = cudaFuncSetAttribute(ssd_fused_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem::bytes);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(ssd_fused_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem::bytes);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) configured[dev] = 1;
  }
  err = cudaMemsetAsync(a.ws_status, 0, sizeof(int), stream);
  if (err != cudaSuccess) return err;
  CUtensorMap mC, mB, mX;
  const dim3 grid(a.nheads, a.batch);
  if (a.seqlen % kQ == 0 && make_maps(a, &mC, &mB, &mX)) {
    ssd_fused_kernel<true><<<grid, kThreads, Smem::bytes, stream>>>(a, mC, mB, mX);
  } else {
    memset(&mC, 0, sizeof(mC));
    ssd_fused_kernel<false><<<grid, kThreads, Smem::bytes, stream>>>(a, mC, mC, mC);
  }
  return cudaGetLastError();
}

}  // namespace ssm
