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
// columns. Per chunk, two rounds of tcgen05 GEMMs (bf16 operands, fp32 accumulators in tensor
// memory, issued by one thread, completion through an mbarrier):
//   round A:  G = C B^T [Q x Q] and Y_off = C H_in [Q x P];
//   (threads) G' = G masked to s <= t and scaled by exp(c_t - c_s) Delta_s, into tensor memory as
//             the A operand of Y_diag; exp(c_t) Y_off into Y_diag's accumulator; B~ = B scaled
//             per row by Delta_s exp(c_end - c_s);
//   round B:  Y_diag += G' X [Q x P] and S = B~^T X [N x P];
//   (threads) y = Y_diag + D x; H <- exp(c_end) H + S.
// Every shared-memory tile is stored in the 128-byte swizzled layout (rows of 128 bytes in
// 1024-byte atoms). The next chunk's C, B and X are copied in while the epilogue and the state
// update of the current one run: when the sequence length is a multiple of the chunk, by five TMA
// bulk-tensor copies of 128-byte rows issued by one thread (C and B as two slabs of 64 columns, X
// as one box), which apply the swizzle themselves; otherwise by 16-byte cp.async copies with zero
// fill past the end. The next chunk's decay prefix is computed while round B runs.
//
// Precision. The three operands the kernel computes (G', H_in and B~) are carried as two bf16
// terms, hi = bf16(v) and lo = bf16(v - hi), each multiplied by the same bf16 input: a single bf16
// rounding costs up to 2^-9 of each summand, which for sums of 128 products of O(1) terms that
// cancel exceeds the bf16-I/O tolerance. For G' and H_in that happened on a fraction of a percent
// of the outputs; for B~, whose error the state carries from chunk to chunk, on 2 of the 33.5
// million outputs of the 8 x 2048 x 32-head workload. G' hi and lo are two GEMMs into one
// accumulator. The H_in hi and lo tiles are adjacent 64-column spans of one MN-major operand, so
// C H_in is one GEMM of N = 128 whose halves are added when exp(c_t) Y_off is formed. B~ hi
// replaces B in its tile (B serves as the K-major B operand of G and, scaled, as the MN-major A
// operand of S: the same bytes); B~ lo goes to the C tile, free after round A since G' lives in
// tensor memory.
//
// Each tcgen05.mma costs its issuing thread tens of cycles whatever its size, so the MMA loops are
// unrolled (constant descriptor offsets). Two CTAs share an SM and its shared-memory bandwidth.
#include <cstring>
#include <type_traits>

#include <cuda.h>  // CUtensorMap and its encoder's signature (resolved at run time, not linked)
#include <cuda_bf16.h>

#include "../../include/ssm.h"
#include "ssm_bounds.cuh"
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

// Shared-memory layout (byte offsets, all 1024-aligned); 112 KB plus the small variables, so two
// CTAs fit an SM. Every tile is 128-byte swizzled; 128 x 128 tiles are two slabs of 64 columns.
struct Smem {
  static constexpr int C = 0;                    // C [Q x N], K-major: A operand of G and Y_off (M = t,
                                                 // K = n); after round A, G'_hi [Q x Q], K-major
  static constexpr int B = C + kQ * kN * 2;      // B [Q x N]: K-major B operand of G (N = s, K = n); scaled,
                                                 // the MN-major A operand of S (M = n, K = s)
  static constexpr int X = B + kQ * kN * 2;      // X [Q x P], MN-major: B operand of Y_diag and S (N = p, K = s)
  static constexpr int H = X + kQ * kP * 2;      // H_in hi, lo [N x P] each, MN-major: B operand of Y_off
                                                 // (N = p, K = n); after round A, G'_lo [Q x Q], K-major
  static constexpr int HL = H + kN * kP * 2;
  static constexpr int MBAR = HL + kN * kP * 2;  // GEMM and TMA mbarriers, the TMEM address, warp
                                                 // sums of the decay scan, lg2 Delta - c
  static constexpr int TSLOT = MBAR + 16;
  static constexpr int WSUM = TSLOT + 16;
  static constexpr int Z = WSUM + 32;
  static constexpr int bytes = Z + kQ * 4;
};
constexpr uint32_t kSlab = kQ * 128;  // bytes of a 64-column slab of a 128-row tile

// TMEM columns. Round A: G [128 x 128] at 0, C [H_in hi | H_in lo] [128 x 128] at 128. The G'
// pass writes G' in G's place as the A operand of Y_diag (bf16 pairs, hi and lo of column block b
// at 32 b and 32 b + 16), and 2^(c_t) Y_off into columns 192..255, where round B's Y_diag
// GEMMs accumulate onto it; S [128 x 64] takes columns 128..191.
constexpr uint32_t kColG = 0, kColOff = 128, kColOffLo = 192, kColDiag = 192, kColS = 128, kCols = 256;

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
// v = hi + lo with hi = bf16(v), lo = bf16(v - hi), 8 values, converted in pairs
__device__ __forceinline__ void split8(const float* v, uint4& hi, uint4& lo) {
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&hi);
  __nv_bfloat162* l = reinterpret_cast<__nv_bfloat162*>(&lo);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    h[k] = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
    const float2 hf = __bfloat1622float2(h[k]);
    l[k] = __floats2bfloat162_rn(v[2 * k] - hf.x, v[2 * k + 1] - hf.y);
  }
}

// The pair v = hi + lo as bf16x2 terms (the first element in the low half): hi = bf16(v),
// lo = bf16(v - hi).
__device__ __forceinline__ void split2(float2 v, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(v.x - hf.x, v.y - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// TMA: the tiles come from three tensor maps (C and B: 2-D [rows, 128], X: 3-D [rows, heads,
// 64]; 128-byte swizzle; described at launch_ssd).
template <bool TMA>
__global__ void __launch_bounds__(kThreads, 2)
    ssd_fused_kernel(const SsdArgs a, const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmX, const int test_skip_mma) {
  extern __shared__ __align__(1024) unsigned char sm[];
  uint64_t& mbar = *reinterpret_cast<uint64_t*>(sm + Smem::MBAR);
  uint64_t& tbar = *reinterpret_cast<uint64_t*>(sm + Smem::MBAR + 8);  // TMA completion
  uint32_t& tslot = *reinterpret_cast<uint32_t*>(sm + Smem::TSLOT);
  float* s_wsum = reinterpret_cast<float*>(sm + Smem::WSUM);
  float* s_z = reinterpret_cast<float*>(sm + Smem::Z);  // lg2(Delta_s) - c_s: exp(c_t - c_s) Delta_s = 2^(c_t + z_s)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the swizzle atoms need a 1024-aligned tile base; the dynamic window starts at the CTA's
  // shared-memory base, so this holds, but it is checked rather than assumed
  if (smem_addr(sm) & 1023u) {
    if (tid == 0) atomicExch(a.ws_status, 2);
    return;
  }
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
  // element counts for the range checks of the debug build (the TMA copies are clipped by their
  // tensor maps instead)
  const long long nCB = (long long)a.batch * L * kN, nX = (long long)a.batch * L * H * kP;
  const long long nDt = (long long)a.batch * L * H, nSt = (long long)a.batch * H * kP * kN;
  const float A2 = a.A[h] * kLog2e;
  const float bias = a.dt_bias ? a.dt_bias[h] : 0.f;
  const float Dh = a.D ? a.D[h] : 0.f;

  // C, B, X of chunk q into their tiles; rows past the sequence end are zero-filled. Copy k of
  // thread tid (cp.async path): C / B row s = tid/16 + 16k, 16-byte chunk tid%16 (slab chunk/8);
  // X row s = tid/8 + 32k, chunk tid%8
  auto stage = [&](int q) {
    const int t0 = q * kQ, len = min(kQ, L - t0);
    if (TMA) {  // whole chunks only: no row of another sequence, none past the end
      if (tid == 0) {
        umma::fence_proxy_async();
        umma::mbar_expect_tx(&tbar, (uint32_t)(2 * kQ * kN * 2 + kQ * kP * 2));
        const int r0 = (int)((long long)b * L + t0);
        umma::tma_load_2d(sC, &tmC, 0, r0, &tbar);
        umma::tma_load_2d(sC + kSlab, &tmC, 64, r0, &tbar);
        umma::tma_load_2d(sB, &tmB, 0, r0, &tbar);
        umma::tma_load_2d(sB + kSlab, &tmB, 64, r0, &tbar);
        umma::tma_load_3d(sX, &tmX, 0, h, r0, &tbar);
      }
      return;
    }
    const int cch = tid % 16;
    const long long cbg = ((long long)b * L + t0 + tid / 16) * kN + cch * 8;
#pragma unroll
    for (int k = 0; k < kQ * kN / 8 / kThreads; ++k) {
      const int srow = tid / 16 + 16 * k;
      const long long g = cbg + (long long)k * 16 * kN;
      const bool ok = srow < len && in_bounds(g, 8, nCB, kBoundsSsd);
      const uint32_t off = (uint32_t)(cch >> 3) * kSlab + umma::sw128_off(srow, cch & 7);
      cp_async16(sC + off, ok ? (const void*)(gC + g) : (const void*)gC, ok ? 16u : 0u);
      cp_async16(sB + off, ok ? (const void*)(gB + g) : (const void*)gB, ok ? 16u : 0u);
    }
    const long long xg = (((long long)b * L + t0 + tid / 8) * H + h) * kP + (tid % 8) * 8;
#pragma unroll
    for (int k = 0; k < kQ * kP / 8 / kThreads; ++k) {
      const int srow = tid / 8 + 32 * k;
      const long long g = xg + (long long)k * 32 * H * kP;
      const bool ok = srow < len && in_bounds(g, 8, nX, kBoundsSsd);
      cp_async16(sX + umma::sw128_off(srow, tid % 8), ok ? (const void*)(gx + g) : (const void*)gx, ok ? 16u : 0u);
    }
    cp_async_commit();
  };
  auto load_dt = [&](int q) -> bf16 {
    const int s = q * kQ + t;
    const long long i = ((long long)b * L + s) * H + h;
    return (s < L && in_bounds(i, 1, nDt, kBoundsSsd)) ? gdt[i] : __float2bfloat16_rn(0.f);
  };

  // running state: row n = t of H [N x P], columns pb .. pb + 31, fp32
  const int pb = half * kHalfP;
  float Hs[kHalfP];
  // this thread's state elements: (bh, p, t) for p = pb .. pb + 31, stride kN
  const bool st_ok = in_bounds((bh * kP + pb) * kN + t, (long long)(kHalfP - 1) * kN + 1, nSt, kBoundsSsd);
#pragma unroll
  for (int p = 0; p < kHalfP; ++p) Hs[p] = (a.h0 && st_ok) ? a.h0[(bh * kP + pb + p) * kN + t] : 0.f;
  // its bf16 hi / lo operand tiles (element (p, n) of the B operand of Y_off)
  auto write_state = [&]() {
#pragma unroll
    for (int p0 = 0; p0 < kHalfP; p0 += 8) {
      uint4 hi, lo;
      split8(Hs + p0, hi, lo);
      const uint32_t off = umma::sw128_off(t, (pb + p0) >> 3);  // row n = t, chunk p / 8
      *reinterpret_cast<uint4*>(sH + off) = hi;
      *reinterpret_cast<uint4*>(sHL + off) = lo;
    }
  };
  write_state();
  bf16 dtv = load_dt(0);
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
  // the test hook's waits give up sooner: nothing will complete them
  const uint32_t wait_limit = test_skip_mma ? (1u << 12) : umma::kWaitLimit;
  const uint32_t tbase = tslot;
  const uint32_t trow = tbase + ((uint32_t)(wq * 32) << 16);
  uint32_t parity = 0;
  bool ok = true;

  // Delta_t of chunk q (dt already loaded), the prefix c_t (log2 units) and its total, and the
  // shared lg2(Delta_s) - c_s; one barrier, so every thread calls it
  auto decay = [&](int q, float dtq, float& Delta, float& cs, float& c_end) {
    const int len = min(kQ, L - q * kQ);
    Delta = 0.f;
    if (t < len) Delta = a.dt_softplus ? softplus_f<true>(dtq + bias) : dtq + bias;
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
    float off = 0.f;
    c_end = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      if (w < wq) off += ws[w];
      if (w < 3) c_end += ws[w];
    }
    c_end += ws[3];
    cs = v + off;
    if (half == 0) s_z[t] = lg2_approx(Delta) - cs;  // -inf past the end (Delta = 0): those columns vanish
  };
  float Delta, cs, c_end;
  decay(0, to_f32(dtv), Delta, cs, c_end);
  if (nc > 1) dtv = load_dt(1);

#pragma unroll 1
  for (int q = 0; q < nc; ++q) {
    const int t0 = q * kQ, len = min(kQ, L - t0);
    if (TMA) {
      ok = __syncthreads_and(umma::mbar_wait(&tbar, tparity) && ok);
      tparity ^= 1;
      if (!ok) break;
    } else {
      cp_async_wait<0>();
    }
    umma::fence_proxy_async();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();

    // ---- round A: G = C B^T, Y_off = C [H_in hi | H_in lo] (one N = 128 GEMM)
    if (tid == 0 && !test_skip_mma) {
      constexpr uint32_t idG = umma::idesc_bf16(kQ, kQ, false, false);
      constexpr uint32_t idOff = umma::idesc_bf16(kQ, 2 * kP, false, true);
#pragma unroll
      for (int kk = 0; kk < kN / 16; ++kk)
        umma::mma_bf16(tbase + kColG, umma::desc_sw128_kmajor(smem_addr(sC), kk, kSlab),
                       umma::desc_sw128_kmajor(smem_addr(sB), kk, kSlab), idG, kk > 0);
#pragma unroll
      for (int kk = 0; kk < kN / 16; ++kk)
        umma::mma_bf16(tbase + kColOff, umma::desc_sw128_kmajor(smem_addr(sC), kk, kSlab),
                       umma::desc_sw128_mnmajor(smem_addr(sH), kk, kSlab), idOff, kk > 0);
      umma::mma_commit(&mbar);
    }
    ok = __syncthreads_and(umma::mbar_wait(&mbar, parity, wait_limit) && ok);
    parity ^= 1;
    umma::fence_after_sync();
    if (!ok) break;

    // ---- G' into TMEM, 2^(c_t) Y_off into Y_diag's accumulator, B~ = Delta_s 2^(c_end - c_s) B_s
    // Column block b = 2 j2 + half (steps s0 = 32 b ..) of row t: G'[t, s] = G[t, s]
    // 2^(c_t + lg2 Delta_s - c_s) for s <= t, written as bf16 pairs (hi to columns 32 b ..,
    // lo to 32 b + 16 ..) in the columns of G this thread has just read. The warp's rows are
    // 32 wq .. 32 wq + 31: a block left of its diagonal needs no mask, one right of it is zero.
#pragma unroll 1
    for (int j2 = 0; j2 < 2; ++j2) {
      const int s0 = 32 * (2 * j2 + half);
      uint32_t hi[16], lo[16];
      if (s0 <= 32 * wq) {
        float g[32];
        umma::tmem_ld32(trow + kColG + s0, g);
        const float4* zq = reinterpret_cast<const float4*>(s_z + s0);
        const bool diag = s0 == 32 * wq;
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 z = zq[j4];
          const float2 a0 = fadd2(f2(cs), make_float2(z.x, z.y)), a1 = fadd2(f2(cs), make_float2(z.z, z.w));
          float2 v0 = fmul2(make_float2(g[4 * j4], g[4 * j4 + 1]), make_float2(ex2_approx(a0.x), ex2_approx(a0.y)));
          float2 v1 = fmul2(make_float2(g[4 * j4 + 2], g[4 * j4 + 3]), make_float2(ex2_approx(a1.x), ex2_approx(a1.y)));
          if (diag) {  // exp2 of a masked entry may overflow; the select drops it
            const int s = s0 + 4 * j4;
            v0 = make_float2(s <= t ? v0.x : 0.f, s + 1 <= t ? v0.y : 0.f);
            v1 = make_float2(s + 2 <= t ? v1.x : 0.f, s + 3 <= t ? v1.y : 0.f);
          }
          split2(v0, hi[2 * j4], lo[2 * j4]);
          split2(v1, hi[2 * j4 + 1], lo[2 * j4 + 1]);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) hi[k] = lo[k] = 0u;
      }
      umma::tmem_st16(trow + kColG + s0, hi);
      umma::tmem_st16(trow + kColG + s0 + 16, lo);
    }
    {
      // Y_diag's accumulator starts as 2^(c_t) (C H_in hi + C H_in lo): this thread's columns of
      // row t, read and rewritten by this thread alone
      const float et = ex2_approx(cs);
#pragma unroll
      for (int c0 = 0; c0 < kHalfP; c0 += 16) {
        float oh[16], ol[16];
        umma::tmem_ld16x2(trow + kColOff + pb + c0, trow + kColOffLo + pb + c0, oh, ol);
        uint32_t v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(et * (oh[j] + ol[j]));
        umma::tmem_st16(trow + kColDiag + pb + c0, v);
      }
    }
    {
      // B~ row r = w_r B_r as hi = bf16(v) in place in the B tile and lo = bf16(v - hi) at the
      // same position of the spent C tile: the MN-major A operands of S's two GEMMs. NC 16-byte
      // chunks of row r from chunk c0 on; every load is issued before the first store (the
      // stores could alias the loads as far as the compiler knows). Chunk c of row r sits at
      // position c ^ (r % 8) of the swizzled row.
      auto scale = [&](auto nc_tag, int r, int slab, int c0, float w) {
        constexpr int NC = decltype(nc_tag)::value;
        const uint32_t rowo = (uint32_t)slab * kSlab + (uint32_t)((r >> 3) * 1024 + (r & 7) * 128);
        uint4 v[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) v[c] = *reinterpret_cast<const uint4*>(sB + rowo + 16 * ((c0 + c) ^ (r & 7)));
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          uint32_t* e = reinterpret_cast<uint32_t*>(&v[c]);
          uint4 l;
          uint32_t* le = reinterpret_cast<uint32_t*>(&l);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 x = fmul2(__bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&e[k])), f2(w));
            split2(x, e[k], le[k]);
          }
          *reinterpret_cast<uint4*>(sC + rowo + 16 * ((c0 + c) ^ (r & 7))) = l;
        }
#pragma unroll
        for (int c = 0; c < NC; ++c) *reinterpret_cast<uint4*>(sB + rowo + 16 * ((c0 + c) ^ (r & 7))) = v[c];
      };
      // The G' pass above is uneven: rows are bound to warps by their TMEM lane quarter; warps 2,
      // 3 and 7 mask two column blocks, warps 0, 1, 5 and 6 one, warp 4 none. The B rows are
      // dealt out against that (in 16-byte chunks, about as costly as a sixth of a block):
      // warp w's own rows are row t of slab `half`, 8 chunks; warps 2, 3 and 7 keep chunks
      // 0..3 of theirs, warp 4 takes chunks 4..7 of warps 2 and 3, and chunks 4..7 of warp 7's
      // rows go one each to warps 0, 1, 5 and 6.
      using C8 = std::integral_constant<int, 8>;
      using C4 = std::integral_constant<int, 4>;
      using C1 = std::integral_constant<int, 1>;
      const float w_own = Delta * ex2_approx(c_end - cs);
      if (warp == 2 || warp == 3 || warp == 7) {
        scale(C4{}, t, half, 0, w_own);
      } else {
        scale(C8{}, t, half, 0, w_own);
        if (warp == 4) {  // chunks 4..7 of rows 64..127 of slab 0 (warps 2 and 3)
          scale(C4{}, 64 + lane, 0, 4, ex2_approx(s_z[64 + lane] + c_end));
          scale(C4{}, 96 + lane, 0, 4, ex2_approx(s_z[96 + lane] + c_end));
        } else {  // one of chunks 4..7 of rows 96..127 of slab 1 (warp 7)
          const int c0 = warp == 0 ? 4 : warp == 1 ? 5 : warp == 5 ? 6 : 7;
          scale(C1{}, 96 + lane, 1, c0, ex2_approx(s_z[96 + lane] + c_end));
        }
      }
    }
    umma::tmem_wait_st();
    umma::fence_proxy_async();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();

    // ---- round B: Y_diag += G' X (A from TMEM, hi + lo), S = B~^T X (hi + lo)
    if (tid == 0) {
      constexpr uint32_t idDiag = umma::idesc_bf16(kQ, kP, false, true);
      constexpr uint32_t idS = umma::idesc_bf16(kN, kP, true, true);
#pragma unroll
      for (int kk = 0; kk < kQ / 16; ++kk) {  // K slice kk: steps 16 kk .., block kk / 2
        const uint32_t a = tbase + kColG + 32u * (kk >> 1) + 8u * (kk & 1);
        const uint64_t bx = umma::desc_sw128_mnmajor(smem_addr(sX), kk, kSlab);
        umma::mma_bf16_ta(tbase + kColDiag, a, bx, idDiag, true);
        umma::mma_bf16_ta(tbase + kColDiag, a + 16u, bx, idDiag, true);
      }
#pragma unroll
      for (int kk = 0; kk < kQ / 16; ++kk)
        umma::mma_bf16(tbase + kColS, umma::desc_sw128_mnmajor(smem_addr(sB), kk, kSlab),
                       umma::desc_sw128_mnmajor(smem_addr(sX), kk, kSlab), idS, kk > 0);
#pragma unroll
      for (int kk = 0; kk < kQ / 16; ++kk)
        umma::mma_bf16(tbase + kColS, umma::desc_sw128_mnmajor(smem_addr(sC), kk, kSlab),
                       umma::desc_sw128_mnmajor(smem_addr(sX), kk, kSlab), idS, true);
      umma::mma_commit(&mbar);
    }
    // this step's x, for the skip term, before the tile is refilled
    uint4 xr[kHalfP / 8];
#pragma unroll
    for (int j = 0; j < kHalfP / 8; ++j)
      xr[j] = *reinterpret_cast<const uint4*>(sX + umma::sw128_off(t, (pb >> 3) + j));
    // the next chunk's decays while round B runs (every reader of this chunk's lg2 Delta - c has
    // passed the barrier before round B)
    float Delta_n = 0.f, cs_n = 0.f, c_end_n = 0.f;
    if (q + 1 < nc) {
      decay(q + 1, to_f32(dtv), Delta_n, cs_n, c_end_n);
      if (q + 2 < nc) dtv = load_dt(q + 2);
    }
    ok = __syncthreads_and(umma::mbar_wait(&mbar, parity) && ok);
    parity ^= 1;
    umma::fence_after_sync();
    if (!ok) break;
    // every operand tile is free: bring in the next chunk while this one finishes
    if (q + 1 < nc) stage(q + 1);

    // ---- epilogue (row t) and state update (row n = t)
    const float dec = ex2_approx(c_end);
    bf16* yrow = static_cast<bf16*>(a.y) + (((long long)b * L + t0 + t) * H + h) * kP;
#pragma unroll
    for (int p0 = 0; p0 < kHalfP; p0 += 8) {
      float yd[8], sv[8];
      umma::tmem_ld8x2(trow + kColDiag + pb + p0, trow + kColS + pb + p0, yd, sv);
      float xv[8];
      unpack8(reinterpret_cast<const unsigned char*>(&xr[p0 / 8]), xv);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        yd[j] = fmaf(Dh, xv[j], yd[j]);
        Hs[p0 + j] = fmaf(dec, Hs[p0 + j], sv[j]);
      }
      if (t < len && in_bounds((((long long)b * L + t0 + t) * H + h) * kP + pb + p0, 8, nX, kBoundsSsd))
        *reinterpret_cast<uint4*>(yrow + pb + p0) = pack8(yd);
    }
    write_state();
    umma::fence_before_sync();
    Delta = Delta_n;
    cs = cs_n;
    c_end = c_end_n;
  }

  if (!ok) {
    if (tid == 0) atomicExch(a.ws_status, 1);
  } else if (a.h_last && st_ok) {
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

// The tensor maps of the TMA path, 128-byte swizzle. Rows are flat (batch * seqlen + t). C, B
// [rows, 128]: a box of 64 columns x 128 rows is one slab; X [rows, heads, 64]: a box of
// 64 x 1 x 128 is the whole tile of one head.
bool make_maps(const SsdArgs& a, CUtensorMap* mC, CUtensorMap* mB, CUtensorMap* mX) {
  EncodeTiled enc = encoder();
  if (!enc) return false;
  const cuuint64_t rows = (cuuint64_t)a.batch * a.seqlen;
  const cuuint64_t dCB[2] = {kN, rows};
  const cuuint64_t sCB[1] = {kN * 2};
  const cuuint32_t bCB[2] = {64, kQ};
  const cuuint32_t e2[2] = {1, 1};
  const cuuint64_t H = (cuuint64_t)a.nheads;
  const cuuint64_t dX[3] = {kP, H, rows};
  const cuuint64_t sX[2] = {kP * 2, H * kP * 2};
  const cuuint32_t bX[3] = {kP, 1, kQ};
  const cuuint32_t e3[3] = {1, 1, 1};
  auto go = [&](CUtensorMap* m, const void* base, cuuint32_t rank, const cuuint64_t* d, const cuuint64_t* st,
                const cuuint32_t* bx, const cuuint32_t* el) {
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), d, st, bx, el,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  return go(mC, a.C, 2, dCB, sCB, bCB, e2) && go(mB, a.B, 2, dCB, sCB, bCB, e2) && go(mX, a.x, 3, dX, sX, bX, e3);
}

}  // namespace

namespace {
unsigned int g_test_hooks = 0;  // SSM_TEST_* flags (ssm_set_test_hooks)
}

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
  const int skip_mma = (g_test_hooks & 1u) ? 1 : 0;
  err = cudaMemsetAsync(a.ws_status, 0, sizeof(int), stream);
  if (err != cudaSuccess) return err;
  CUtensorMap mC, mB, mX;
  const dim3 grid(a.nheads, a.batch);
  // TMA row coordinates are 32-bit: the flat row index batch * seqlen must stay below 2^31
  const bool tma_rows_fit = (long long)a.batch * a.seqlen < (1LL << 31);
  if (a.seqlen % kQ == 0 && tma_rows_fit && make_maps(a, &mC, &mB, &mX)) {
    ssd_fused_kernel<true><<<grid, kThreads, Smem::bytes, stream>>>(a, mC, mB, mX, skip_mma);
  } else {
    memset(&mC, 0, sizeof(mC));
    ssd_fused_kernel<false><<<grid, kThreads, Smem::bytes, stream>>>(a, mC, mC, mC, skip_mma);
  }
  return cudaGetLastError();
}

cudaError_t ssd_bounds_flags(unsigned* out, bool clear) {
#ifdef SSM_DEBUG_BOUNDS
  return bounds_flags_read(out, clear);
#else
  (void)out;
  (void)clear;
  return cudaErrorNotSupported;
#endif
}

}  // namespace ssm

// Test hooks of the C ABI (include/ssm.h): they only affect the state-space-duality launches.
extern "C" SSM_API void ssm_set_test_hooks(unsigned int flags) { ssm::g_test_hooks = flags; }
