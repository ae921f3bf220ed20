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
// Design. Every CTA is a single warp that owns a group of channels of one sequence over one
// time chunk from staging to store, so nothing but __syncwarp orders its phases. One state
// update costs one exp2 on the special-function pipe and four fp32 operations on the FMA pipe
// (Delta A, Delta u B, the recurrence, the readout); both pipes take 4 cycles per 32 updates
// per SMSP on this part, and ex2 overlaps with packed f32x2 FMA work, so the kernels keep the
// FMA-pipe work packed and every lane's states independent. B and C reach the lanes as
// broadcast shared-memory loads, which contend with the exp2 and FMA work (one 16-byte
// broadcast per 4 values; with 8 of them beside 16 exp2 and 32 packed FMAs a step costs 118
// cycles instead of 68), and every per-channel value passed between lanes costs a shared
// store and load; the geometries below trade these costs against the lanes each problem needs.
//
// Main pass, three geometries (the host picks one per problem):
//  * whole channels (N <= 16, time-chunked problems or problems with enough channels): lane l
//    holds all 16 states of channels l and l + 32, and does their element-wise work (conv,
//    SiLU, softplus, gate), scan, readout and store in one loop over 8 steps; nothing per
//    (t, d) passes through shared memory, and each B / C load serves two channels. 16-step tiles.
//  * two lanes per channel (N <= 16, unchunked problems with few channels per SM): 8 states per
//    lane, 16 channels per warp; the owner of each 8-step block computes its element-wise values
//    into shared memory, both lanes scan, and the owner sums the two partial readouts. 32-step
//    tiles.
//  * four lanes per channel (N <= 32): the same with 8 states per lane and 8 channels per warp.
// In all of them the raw rows of x, delta, z and B, C are copied global -> shared with
// 16-byte cp.async into a two-slot ring one tile ahead, and B, C are converted to fp32 in
// step-major order (ln 2 folded into B) before the scan.
// Carry pass (only when time is chunked): one lane per channel with all 16 states (two lanes
// of 16 states for N <= 32) walks each chunk but the last from a zero state and writes the
// chunk's sum of Delta' and its end state; element-wise work and the scan run in one loop,
// four steps at a time. The main pass starts chunk q from h0 composed with the carries of
// chunks 0..q-1 through (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2),
// a = 2^(A sum Delta') = exp(A sum Delta); it follows the carry kernel in stream order.
// Options (template parameters): REV walks time backward (the backward scan of a
// bidirectional layer); ZOH uses the zero-order-hold input term expm1(Delta A)/A B u.
// The per-step state never leaves registers.
#include <algorithm>

#include <type_traits>

#include "ssm_bounds.cuh"
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kT = 32;           // time steps per tile of the two- and four-lane main pass
constexpr int kT1 = 16;          // time steps per tile of the one-lane main pass and the carry pass
constexpr int kBlk = 8;          // steps per element-wise / epilogue block
constexpr int kNB = kT / kBlk;   // blocks per tile
constexpr int kTP = kT + 4;      // row stride of the per-channel fp32 arrays (float4 aligned)

// Raw rows of a TT-step tile are padded (bf16: 80 / 48 bytes, fp32: 144 / 80 bytes for 32 / 16
// steps) so that the lanes of a quarter-warp, each reading its own channel's row with a
// 16-byte load, hit distinct banks.
template <typename T, int TT>
__host__ __device__ constexpr int row_stride() { return sizeof(T) == 2 ? TT + 8 : TT + 4; }

constexpr size_t align16(size_t v) { return (v + 15) & ~(size_t)15; }

// Element counts of the tensors a scan call touches (for the debug build's range checks).
struct Extents {
  long long tok, bc, st, dn, win, wsS, wsH;
};
__device__ __forceinline__ Extents extents_of(const ScanArgs& a) {
  const long long BD = (long long)a.batch * a.dim;
  Extents e;
  e.tok = BD * a.seqlen;
  e.bc = (long long)a.batch * a.dstate * a.seqlen;
  e.st = BD * a.dstate;
  e.dn = (long long)a.dim * a.dstate;
  e.win = BD * (a.d_conv > 1 ? a.d_conv - 1 : 0);
  e.wsS = (long long)a.ws_chunks * BD;
  e.wsH = e.wsS * (a.dstate <= 16 ? 16 : 32);
  return e;
}

// Main-pass geometry: G lanes per channel, 8 states per lane.
template <int G>
struct MainGeo {
  static constexpr int kS = 8;
  static constexpr int kCPW = 32 / G;        // channels per warp
  static constexpr int kN = kS * G;          // states the warp holds per channel (16 or 32)
  static constexpr int kBCS = kN + 4;        // row stride of the step-major fp32 B / C arrays
};

// Carry-pass geometry: G lanes per channel, 16 states per lane, K channels per lane (the
// lane's channels c, c + 32/G, ...: every B row it loads serves K channels).
template <int G, int K>
struct CarryGeo {
  static constexpr int kS = 16;
  static constexpr int kCPW = K * 32 / G;
  static constexpr int kN = kS * G;
  static constexpr int kBCS = kN + 4;
};

// Shared-memory layout of the main pass (byte offsets):
//   ring  [2][R][RS]     raw rows: x, delta, z (kCPW each), B, C (kN each)
//   Bt,Ct [kT][kBCS]     B (times ln 2 for Euler), C as fp32, step-major
//   dl    [kCPW][kTP]    Delta'
//   du    [kCPW][kTP]    scan input (Delta' u, or u for ZOH)
//   sk    [kCPW][kTP]    D u
//   y     [G][kCPW][kTP] partial readouts, one per lane of the channel
//   halo  [2][kCPW][4]   the 3 raw inputs before the tile (ping-pong by tile parity)
template <typename T, int G>
struct MainLayout {
  using Geo = MainGeo<G>;
  static constexpr int RS = row_stride<T, kT>();
  static constexpr int R = 3 * Geo::kCPW + 2 * Geo::kN;
  static constexpr size_t slot_bytes = sizeof(T) * (size_t)R * RS;
  static constexpr size_t ring = 0;
  static constexpr size_t Bt = align16(ring + 2 * slot_bytes);
  static constexpr size_t Ct = Bt + sizeof(float) * kT * Geo::kBCS;
  static constexpr size_t dl = Ct + sizeof(float) * kT * Geo::kBCS;
  static constexpr size_t du = dl + sizeof(float) * Geo::kCPW * kTP;
  static constexpr size_t sk = du + sizeof(float) * Geo::kCPW * kTP;
  static constexpr size_t y = sk + sizeof(float) * Geo::kCPW * kTP;
  static constexpr size_t halo = y + sizeof(float) * G * Geo::kCPW * kTP;
  static constexpr size_t bytes = halo + sizeof(float) * 2 * Geo::kCPW * 4;
  static_assert(slot_bytes % 16 == 0, "ring slots stay 16-byte aligned");
};

// Shared-memory layout of the carry pass (16-step tiles): ring [2][R][RS] (x, delta, B) and
// B as fp32, step-major.
template <typename T, int G, int K>
struct CarryLayout {
  using Geo = CarryGeo<G, K>;
  static constexpr int RS = row_stride<T, kT1>();
  static constexpr int R = 2 * Geo::kCPW + Geo::kN;
  static constexpr size_t slot_bytes = sizeof(T) * (size_t)R * RS;
  static constexpr size_t ring = 0;
  static constexpr size_t Bt = align16(ring + 2 * slot_bytes);
  static constexpr size_t bytes = Bt + sizeof(float) * kT1 * Geo::kBCS;
  static_assert(slot_bytes % 16 == 0, "ring slots stay 16-byte aligned");
};

// ---------------------------------------------------------------- staging

// Copies the raw rows of one tile into a ring slot. Row r of the slot belongs to array
// arr_of(r) (0 = x, 1 = delta, 2 = z, 3 = B, 4 = C) and to channel / state r - first row of
// that array. Every lane copies a fixed 16-byte column; rows past dim or N, z rows without a
// gate and steps outside the chunk are zero-filled. A staged row holds the tile's TT steps in
// real order: forward, column p is virtual step t0 + p; backward, it is virtual step
// t0 + TT-1-p, and the row starts at real position L - t0 - TT.
template <typename T, int TT, int CPW, int NR, bool HAS_Z, bool HAS_C>
struct Stager {
  static constexpr int kEPC = 16 / (int)sizeof(T);     // elements per 16-byte chunk
  static constexpr int kCPR = TT / kEPC;               // chunks per row
  static constexpr int kRPC = 32 / kCPR;               // rows per copy step of the warp
  static constexpr int kRows = (HAS_Z ? 3 : 2) * CPW + (HAS_C ? 2 : 1) * NR;
  static constexpr int kCopies = kRows / kRPC;
  static_assert(kRows % kRPC == 0 && CPW % kRPC == 0 && NR % kRPC == 0, "copy steps stay inside one array");

  long long off_c;   // element offset of this lane's first channel row at t = 0, plus its column
  long long off_n;   // the same for its first state row of B / C
  int lrow;          // row of this lane within a copy step
  int col;           // its column (elements)

  __device__ void init(const ScanArgs& a, int b, int d0, int lane) {
    lrow = lane / kCPR;
    col = (lane % kCPR) * kEPC;
    off_c = ((long long)b * a.dim + d0 + lrow) * a.seqlen + col;
    off_n = ((long long)b * a.dstate + lrow) * a.seqlen + col;
  }

  template <bool REV>
  __device__ void issue(const ScanArgs& a, T (*slot)[row_stride<T, TT>()], int d0, int t0, int t_end,
                        bool has_z) const {
    const int L = a.seqlen;
    const int seg = REV ? L - t0 - TT : t0;
    // rows are a whole number of 16-byte chunks long, so a chunk is all in or all out
    const bool tin = REV ? col >= TT - (t_end - t0) : col < t_end - t0;
#pragma unroll
    for (int k = 0; k < kCopies; ++k) {
      const int r = k * kRPC + lrow;
      const int r0 = k * kRPC;           // first row of the step: fixes the array at compile time
      const T* src = nullptr;
      bool ok = tin;
      long long idx = 0, ext = 0;  // element offset of the chunk in its tensor, and the tensor's size
      if (r0 < CPW) {
        ok = ok && d0 + (r0 % CPW) + lrow < a.dim;
        idx = off_c + (long long)(r0 % CPW) * L;
        src = static_cast<const T*>(a.x) + idx;
      } else if (r0 < 2 * CPW) {
        ok = ok && d0 + (r0 % CPW) + lrow < a.dim;
        idx = off_c + (long long)(r0 % CPW) * L;
        src = static_cast<const T*>(a.delta) + idx;
      } else if (HAS_Z && r0 < 3 * CPW) {
        ok = ok && has_z && d0 + (r0 % CPW) + lrow < a.dim;
        idx = off_c + (long long)(r0 % CPW) * L;
        src = static_cast<const T*>(a.z) + idx;
      } else {
        const int rb = r0 - (HAS_Z ? 3 : 2) * CPW;
        const int n0 = rb % NR;
        ok = ok && n0 + lrow < a.dstate;
        idx = off_n + (long long)n0 * L;
        src = static_cast<const T*>(rb < NR ? a.B : a.C) + idx;
      }
      if (ok) {
        const Extents ex = extents_of(a);
        ext = (r0 < (HAS_Z ? 3 : 2) * CPW) ? ex.tok : ex.bc;
        ok = in_bounds(idx + seg, kEPC, ext, kBoundsScan);
      }
      cp_async16(&slot[r][col], ok ? (const void*)(src + seg) : a.x, ok ? 16u : 0u);
    }
  }

  // The same rows, element by element (rows not 16-byte aligned).
  template <bool REV>
  __device__ void load_sync(const ScanArgs& a, T (*slot)[row_stride<T, TT>()], int d0, int t0, int t_end,
                            bool has_z) const {
    const int L = a.seqlen;
    const int tl = min(TT, t_end - t0);
    const int seg = REV ? L - t0 - TT : t0;
#pragma unroll 1
    for (int k = 0; k < kCopies; ++k) {
      const int r = k * kRPC + lrow;
      const int r0 = k * kRPC;
      const T* src = nullptr;
      bool ok = true;
      long long idx = 0;
      if (r0 < CPW) {
        ok = d0 + (r0 % CPW) + lrow < a.dim;
        idx = off_c + (long long)(r0 % CPW) * L;
        src = static_cast<const T*>(a.x) + idx;
      } else if (r0 < 2 * CPW) {
        ok = d0 + (r0 % CPW) + lrow < a.dim;
        idx = off_c + (long long)(r0 % CPW) * L;
        src = static_cast<const T*>(a.delta) + idx;
      } else if (HAS_Z && r0 < 3 * CPW) {
        ok = has_z && d0 + (r0 % CPW) + lrow < a.dim;
        idx = off_c + (long long)(r0 % CPW) * L;
        src = static_cast<const T*>(a.z) + idx;
      } else {
        const int rb = r0 - (HAS_Z ? 3 : 2) * CPW;
        const int n0 = rb % NR;
        ok = n0 + lrow < a.dstate;
        idx = off_n + (long long)n0 * L;
        src = static_cast<const T*>(rb < NR ? a.B : a.C) + idx;
      }
      const Extents ex = extents_of(a);
      const long long ext = (r0 < (HAS_Z ? 3 : 2) * CPW) ? ex.tok : ex.bc;
#pragma unroll
      for (int e = 0; e < kEPC; ++e) {
        const bool in = REV ? col + e >= TT - tl : col + e < tl;
        slot[r][col + e] =
            (ok && in && in_bounds(idx + seg + e, 1, ext, kBoundsScan)) ? src[seg + e] : from_f32<T>(0.f);
      }
    }
  }
};

// B (and C) rows of a slot -> fp32 step-major [TT][BCS]; lane i converts 4x4 blocks.
// Euler's B carries the ln 2 that turns Delta' (log2 units) back into Delta in Delta' u B.
template <typename T, int TT, int NR, int BCS, bool REV>
__device__ __forceinline__ void transpose_rows(const T (*src)[row_stride<T, TT>()], float (*dst)[BCS], float scale,
                                               int lane) {
  constexpr int kBlocks = (NR / 4) * (TT / 4);
#pragma unroll
  for (int blk = lane; blk < kBlocks; blk += 32) {
    const int n0 = (blk % (NR / 4)) * 4, s0 = (blk / (NR / 4)) * 4;
    float v[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (REV) {  // virtual steps s0 .. s0+3 are columns TT-1-s0 down to TT-4-s0
        float r[4];
        load4(&src[n0 + i][TT - 4 - s0], r);
        v[i][0] = r[3]; v[i][1] = r[2]; v[i][2] = r[1]; v[i][3] = r[0];
      } else {
        load4(&src[n0 + i][s0], v[i]);
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<float4*>(&dst[s0 + j][n0]) =
          make_float4(v[0][j] * scale, v[1][j] * scale, v[2][j] * scale, v[3][j] * scale);
  }
}

// Loads 8 virtual steps tt .. tt+7 of a staged row of a TT-step tile (backward: columns
// TT-1-tt down to TT-8-tt).
template <typename T, int TT, bool REV>
__device__ __forceinline__ void load_seg8(const T* row, int tt, float (&v)[8]) {
  if (REV) {
    float r[8];
    load8(row + (TT - 8 - tt), r);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = r[7 - j];
  } else {
    load8(row + tt, v);
  }
}

// Loads 4 virtual steps tt .. tt+3 of a staged row of a TT-step tile.
template <typename T, int TT, bool REV>
__device__ __forceinline__ void load_seg4(const T* row, int tt, float (&v)[4]) {
  if (REV) {
    float r[4];
    load4(row + (TT - 4 - tt), r);
    v[0] = r[3]; v[1] = r[2]; v[2] = r[1]; v[3] = r[0];
  } else {
    load4(row + tt, v);
  }
}

// The conv taps w0..w3 (w3 on the current input) on the window x[t-3 .. t]; scalar FMAs.
__device__ __forceinline__ float conv4(const float* win, float w0, float w1, float w2, float w3, float cb) {
  float c = fmaf(w0, win[0], cb);
  c = fmaf(w1, win[1], c);
  c = fmaf(w2, win[2], c);
  return fmaf(w3, win[3], c);
}

// Per-channel parameters of channel d: delta bias, skip weight, conv taps (zero-padded to 4).
struct ChannelParams {
  float bias, bias_l2, Dd, w0, w1, w2, w3, cb;
};

template <bool CONV>
__device__ __forceinline__ ChannelParams channel_params(const ScanArgs& a, int d, bool valid) {
  ChannelParams p{0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (valid && in_bounds(d, 1, a.dim, kBoundsScan)) {
    p.bias = a.delta_bias ? a.delta_bias[d] : 0.f;
    p.Dd = a.D ? a.D[d] : 0.f;
    if (CONV && in_bounds((long long)d * a.d_conv, a.d_conv, (long long)a.dim * a.d_conv, kBoundsScan)) {
      const int K = a.d_conv;
      const float* wp = a.conv_w + (long long)d * K;
      p.w3 = wp[K - 1];
      if (K >= 2) p.w2 = wp[K - 2];
      if (K >= 3) p.w1 = wp[K - 3];
      if (K >= 4) p.w0 = wp[K - 4];
      p.cb = a.conv_b ? a.conv_b[d] : 0.f;
    }
  }
  p.bias_l2 = p.bias * kLog2e;
  return p;
}

// The 3 raw inputs before virtual step t_begin of channel (b, d): conv_init (or zeros) for the
// first chunk, else x itself.
template <typename T, bool REV>
__device__ __forceinline__ void halo_at(const ScanArgs& a, long long cc, int t_begin, int q, bool valid,
                                        float (&hv)[3]) {
  hv[0] = hv[1] = hv[2] = 0.f;
  if (!valid) return;
  const int K = a.d_conv, L = a.seqlen;
  const T* gx = static_cast<const T*>(a.x);
  const Extents ex = extents_of(a);
  if (q == 0) {
    if (a.conv_init && in_bounds(cc * (K - 1), K - 1, ex.win, kBoundsScan)) {
      const T* ci = static_cast<const T*>(a.conv_init) + cc * (K - 1);
      if (K >= 2) hv[2] = to_f32(ci[K - 2]);
      if (K >= 3) hv[1] = to_f32(ci[K - 3]);
      if (K >= 4) hv[0] = to_f32(ci[K - 4]);
    }
  } else {
    auto real_t = [&](int tau) { return REV ? L - 1 - tau : tau; };
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const long long i = cc * L + real_t(t_begin - 3 + j);
      if (in_bounds(i, 1, ex.tok, kBoundsScan)) hv[j] = to_f32(gx[i]);
    }
  }
}

// ---------------------------------------------------------------- main pass

template <typename T, int G, bool CONV, bool VEC, bool REV, bool ZOH>
__global__ void __launch_bounds__(32) scan_main_kernel(const ScanArgs a) {
  const Extents ex = extents_of(a);  // tensor sizes for the range checks of the debug build
  constexpr bool PRECISE = IoTraits<T>::kPrecise;
  using Geo = MainGeo<G>;
  using Lay = MainLayout<T, G>;
  constexpr int CPW = Geo::kCPW;
  constexpr int BCS = Geo::kBCS;
  constexpr int RS = Lay::RS;
  constexpr int NB_OWN = kNB / G;   // 8-step blocks each lane owns per tile
  using St = Stager<T, kT, CPW, Geo::kN, true, true>;
  static_assert(St::kRows == Lay::R, "staged rows");
  static_assert(kNB % G == 0, "blocks divide among a channel's lanes");

  extern __shared__ __align__(16) unsigned char smem_raw[];
  T (*const ring)[Lay::R][RS] = reinterpret_cast<T (*)[Lay::R][RS]>(smem_raw + Lay::ring);
  float (*const s_B)[BCS] = reinterpret_cast<float (*)[BCS]>(smem_raw + Lay::Bt);
  float (*const s_C)[BCS] = reinterpret_cast<float (*)[BCS]>(smem_raw + Lay::Ct);
  float (*const s_dl)[kTP] = reinterpret_cast<float (*)[kTP]>(smem_raw + Lay::dl);
  float (*const s_du)[kTP] = reinterpret_cast<float (*)[kTP]>(smem_raw + Lay::du);
  float (*const s_sk)[kTP] = reinterpret_cast<float (*)[kTP]>(smem_raw + Lay::sk);
  float (*const s_y)[CPW][kTP] = reinterpret_cast<float (*)[CPW][kTP]>(smem_raw + Lay::y);
  float (*const s_halo)[CPW][4] = reinterpret_cast<float (*)[CPW][4]>(smem_raw + Lay::halo);

  const int lane = threadIdx.x;
  const int c = lane / G;            // channel within the warp
  const int g = lane % G;            // state group: states 8g .. 8g+7
  const int d0 = blockIdx.x * CPW;
  const int b = blockIdx.y;
  const int q = blockIdx.z;          // chunk slowest: the chunk-0 CTAs, which need no carry, start first
  const int L = a.seqlen, N = a.dstate, dim = a.dim;
  const long long BD = (long long)a.batch * dim;
  const int t_begin = q * a.chunk_len;
  const int t_end = min(L, t_begin + a.chunk_len);
  const int ntiles = t_end > t_begin ? (t_end - t_begin + kT - 1) / kT : 0;
  const int d = d0 + c;
  const bool valid = d < dim;
  const long long cc = (long long)b * dim + d;
  const bool has_z = a.z != nullptr;
  const int NS = N <= 16 ? 16 : 32;  // per-channel state stride of the carry workspace

  St st;
  st.init(a, b, d0, lane);
  if (VEC && ntiles > 0) {
    st.template issue<REV>(a, ring[0], d0, t_begin, t_end, has_z);
    cp_async_commit();
  }

  const ChannelParams cp = channel_params<CONV>(a, d, valid);
  if (CONV && g == 0) {
    float hv[3];
    halo_at<T, REV>(a, cc, t_begin, q, valid, hv);
    s_halo[0][c][0] = hv[0];
    s_halo[0][c][1] = hv[1];
    s_halo[0][c][2] = hv[2];
  }

  // ---- states n = 8g .. 8g+7 and A (Delta is kept in log2 units, so 2^(Delta' A) = exp(Delta A))
  float2 h[4], av[4], ia[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int n0 = 8 * g + 2 * k;
    const bool arow = valid && in_bounds((long long)d * N, N, ex.dn, kBoundsScan);
    av[k] = make_float2((arow && n0 < N) ? a.A[(long long)d * N + n0] : 0.f,
                        (arow && n0 + 1 < N) ? a.A[(long long)d * N + n0 + 1] : 0.f);
    h[k] = make_float2(0.f, 0.f);
    ia[k] = make_float2(0.f, 0.f);
    if (ZOH) {
      auto inv = [](float v) { return v != 0.f ? 1.0f / v : 0.f; };
      ia[k] = make_float2(inv(av[k].x), inv(av[k].y));
    }
  }
  if (valid) {
    if (a.h0 && in_bounds(cc * N, N, ex.st, kBoundsScan)) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int n0 = 8 * g + 2 * k;
        h[k] = make_float2(n0 < N ? a.h0[cc * N + n0] : 0.f, n0 + 1 < N ? a.h0[cc * N + n0 + 1] : 0.f);
      }
    }
    // carry-in (the carry kernel ran before this one in stream order): compose the aggregates
    // of chunks 0 .. q-1 onto h0, two chunks' loads at a time
    for (int j0 = 0; j0 < q; j0 += 2) {
      float Sj[2];
      float4 hb[2][2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const long long e = (long long)(j0 + k < q ? j0 + k : 0) * BD + cc;
        const bool in = j0 + k < q && in_bounds(e, 1, ex.wsS, kBoundsScan) &&
                        in_bounds(e * NS + 8 * g, 8, ex.wsH, kBoundsScan);
        Sj[k] = in ? a.ws_S[e] : 0.f;
        const float4* hp = reinterpret_cast<const float4*>(a.ws_h + e * NS + 8 * g);
        hb[k][0] = in ? hp[0] : make_float4(0.f, 0.f, 0.f, 0.f);
        hb[k][1] = in ? hp[1] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (j0 + k < q) {
          const float2 hv[4] = {make_float2(hb[k][0].x, hb[k][0].y), make_float2(hb[k][0].z, hb[k][0].w),
                                make_float2(hb[k][1].x, hb[k][1].y), make_float2(hb[k][1].z, hb[k][1].w)};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 x = fmul2(f2(Sj[k]), av[i]);
            h[i] = ffma2(make_float2(ex2_approx(x.x), ex2_approx(x.y)), h[i], hv[i]);
          }
        }
      }
    }
  }

  for (int it = 0; it < ntiles; ++it) {
    const int bf = it & 1;      // ring slot and halo ping-pong of tile `it`
    const int t0 = t_begin + it * kT;
    const int tl = min(kT, t_end - t0);
    if (VEC) {
      cp_async_wait<0>();
    } else {
      st.template load_sync<REV>(a, ring[bf], d0, t0, t_end, has_z);
    }
    __syncwarp();  // (A) tile `it` visible to the warp; every lane is past tile it-1, so its slot can be refilled
    if (VEC && it + 1 < ntiles) {
      st.template issue<REV>(a, ring[bf ^ 1], d0, t0 + kT, t_end, has_z);
      cp_async_commit();
    }
    const T (*raw)[RS] = ring[bf];

    // ---- B, C -> fp32 step-major (rows past N / steps past the end are zero)
    transpose_rows<T, kT, Geo::kN, BCS, REV>(raw + 3 * CPW, s_B, ZOH ? 1.0f : kLn2, lane);
    transpose_rows<T, kT, Geo::kN, BCS, REV>(raw + 3 * CPW + Geo::kN, s_C, 1.0f, lane);

    // ---- element-wise phase: lane (c, g) owns the 8-step blocks g, g + G, ...
#pragma unroll
    for (int ob = 0; ob < NB_OWN; ++ob) {
      const int blk = g + ob * G;
      const int tt = blk * kBlk;
      float xv[kBlk], dv[kBlk];
      load_seg8<T, kT, REV>(raw[c], tt, xv);
      load_seg8<T, kT, REV>(raw[CPW + c], tt, dv);
      float win[kBlk + 3];
      if (CONV) {
        if (blk == 0) {
          win[0] = s_halo[bf][c][0];
          win[1] = s_halo[bf][c][1];
          win[2] = s_halo[bf][c][2];
        } else {
          float pv[4];
          if (REV) {  // virtual tt-1, tt-2, tt-3 are columns kT-tt, +1, +2
            load4(&raw[c][kT - tt], pv);
            win[0] = pv[2]; win[1] = pv[1]; win[2] = pv[0];
          } else {
            load4(&raw[c][tt - 4], pv);
            win[0] = pv[1]; win[1] = pv[2]; win[2] = pv[3];
          }
        }
        if (blk == kNB - 1) {
          s_halo[bf ^ 1][c][0] = xv[kBlk - 3];
          s_halo[bf ^ 1][c][1] = xv[kBlk - 2];
          s_halo[bf ^ 1][c][2] = xv[kBlk - 1];
        }
#pragma unroll
        for (int j = 0; j < kBlk; ++j) win[3 + j] = xv[j];
      }
      float dl[kBlk], du[kBlk], sk[kBlk];
      const bool full = tt + kBlk <= tl;
#pragma unroll
      for (int j = 0; j < kBlk; j += 2) {
        float2 u;
        if (CONV) {
          u = silu2_tier<PRECISE>(make_float2(conv4(&win[j], cp.w0, cp.w1, cp.w2, cp.w3, cp.cb),
                                              conv4(&win[j + 1], cp.w0, cp.w1, cp.w2, cp.w3, cp.cb)));
        } else {
          u = make_float2(xv[j], xv[j + 1]);
        }
        float2 D2 = delta_log2<PRECISE>(make_float2(dv[j], dv[j + 1]), cp.bias, cp.bias_l2, a.delta_softplus);
        if (!full) {  // steps past the tile end are identity updates: Delta = 0, u = 0
          const bool i0 = tt + j < tl, i1 = tt + j + 1 < tl;
          D2 = make_float2(i0 ? D2.x : 0.f, i1 ? D2.y : 0.f);
          u = make_float2(i0 ? u.x : 0.f, i1 ? u.y : 0.f);
        }
        // the scan's per-step input: Delta' u (Euler) or u (ZOH, whose factor is per state)
        const float2 du2 = ZOH ? u : fmul2(D2, u);
        const float2 sk2 = fmul2(f2(cp.Dd), u);
        dl[j] = D2.x; dl[j + 1] = D2.y;
        du[j] = du2.x; du[j + 1] = du2.y;
        sk[j] = sk2.x; sk[j + 1] = sk2.y;
      }
      store8(&s_dl[c][tt], dl);
      store8(&s_du[c][tt], du);
      store8(&s_sk[c][tt], sk);
    }
    __syncwarp();  // (B)

    // ---- scan phase: sequential in t; steps past tl have Delta = 0 and Delta u = 0 (identity)
    {
      const int tlu = (tl + 3) & ~3;
#pragma unroll 1
      for (int t = 0; t < tlu; t += 4) {
        const float4 dl4 = *reinterpret_cast<const float4*>(&s_dl[c][t]);
        const float4 du4 = *reinterpret_cast<const float4*>(&s_du[c][t]);
        const float dls[4] = {dl4.x, dl4.y, dl4.z, dl4.w};
        const float dus[4] = {du4.x, du4.y, du4.z, du4.w};
        float yv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 b0 = *reinterpret_cast<const float4*>(&s_B[t + j][8 * g]);
          const float4 b1 = *reinterpret_cast<const float4*>(&s_B[t + j][8 * g + 4]);
          const float2 bv[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                                make_float2(b1.z, b1.w)};
          const float2 dd = f2(dls[j]);
          const float2 uu = f2(dus[j]);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 x = fmul2(dd, av[k]);
            const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            float2 in = fmul2(uu, bv[k]);
            if (ZOH) in = fmul2(in, zoh_factor2(x, e, dd, ia[k]));
            h[k] = ffma2(e, h[k], in);
          }
          const float4 c0 = *reinterpret_cast<const float4*>(&s_C[t + j][8 * g]);
          const float4 c1 = *reinterpret_cast<const float4*>(&s_C[t + j][8 * g + 4]);
          float2 p = fmul2(h[0], make_float2(c0.x, c0.y));
          p = ffma2(h[1], make_float2(c0.z, c0.w), p);
          p = ffma2(h[2], make_float2(c1.x, c1.y), p);
          p = ffma2(h[3], make_float2(c1.z, c1.w), p);
          yv[j] = p.x + p.y;
        }
        *reinterpret_cast<float4*>(&s_y[g][c][t]) = make_float4(yv[0], yv[1], yv[2], yv[3]);
      }
    }
    __syncwarp();  // (C) the G partials of channel c come from the G lanes of the channel

    // ---- epilogue: out = (sum of the partials + D u) * silu(z) for the owned blocks
    if (valid) {
      T* orow = static_cast<T*>(a.out) + cc * L;
#pragma unroll
      for (int ob = 0; ob < NB_OWN; ++ob) {
        const int blk = g + ob * G;
        const int tt = blk * kBlk;
        if (tt >= tl) continue;
        float ys[kBlk], tmp[kBlk];
        load8(&s_sk[c][tt], ys);
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          load8(&s_y[gg][c][tt], tmp);
#pragma unroll
          for (int j = 0; j < kBlk; j += 2) {
            const float2 s = fadd2(make_float2(ys[j], ys[j + 1]), make_float2(tmp[j], tmp[j + 1]));
            ys[j] = s.x; ys[j + 1] = s.y;
          }
        }
        float o[kBlk];
        if (has_z) {
          float zv[kBlk];
          load_seg8<T, kT, REV>(raw[2 * CPW + c], tt, zv);
#pragma unroll
          for (int j = 0; j < kBlk; j += 2) {
            const float2 gt = silu2_tier<PRECISE>(make_float2(zv[j], zv[j + 1]));
            const float2 y = fmul2(make_float2(ys[j], ys[j + 1]), gt);
            o[j] = y.x; o[j + 1] = y.y;
          }
        } else {
#pragma unroll
          for (int j = 0; j < kBlk; ++j) o[j] = ys[j];
        }
        if (REV) {
          // virtual tt+j is real L-1-(t0+tt+j): the block is stored reversed
          if (VEC && tt + kBlk <= tl) {
            float r[kBlk];
#pragma unroll
            for (int j = 0; j < kBlk; ++j) r[j] = o[kBlk - 1 - j];
            if (ptr_in(static_cast<T*>(a.out), orow + (L - t0 - tt - kBlk), kBlk, ex.tok, kBoundsScan))
              store8(orow + (L - t0 - tt - kBlk), r);
          } else if (VEC && tt + 4 <= tl) {  // fp32 rows can end on a 4-step boundary
            const float r4[4] = {o[3], o[2], o[1], o[0]};
            if (ptr_in(static_cast<T*>(a.out), orow + (L - t0 - tt - 4), 4, ex.tok, kBoundsScan))
              store4(orow + (L - t0 - tt - 4), r4);
          } else {
#pragma unroll
            for (int j = 0; j < kBlk; ++j)
              if (tt + j < tl && ptr_in(static_cast<T*>(a.out), orow + (L - 1 - (t0 + tt + j)), 1, ex.tok, kBoundsScan))
                orow[L - 1 - (t0 + tt + j)] = from_f32<T>(o[j]);
          }
        } else {
          T* dst = orow + t0 + tt;
          if (VEC && tt + kBlk <= tl) {
            if (ptr_in(static_cast<T*>(a.out), dst, kBlk, ex.tok, kBoundsScan)) store8(dst, o);
          } else if (VEC && tt + 4 <= tl) {  // fp32 rows can end on a 4-step boundary
            const float o4[4] = {o[0], o[1], o[2], o[3]};
            if (ptr_in(static_cast<T*>(a.out), dst, 4, ex.tok, kBoundsScan)) store4(dst, o4);
          } else {
#pragma unroll
            for (int j = 0; j < kBlk; ++j)
              if (tt + j < tl && ptr_in(static_cast<T*>(a.out), dst + j, 1, ex.tok, kBoundsScan)) dst[j] = from_f32<T>(o[j]);
          }
        }
      }
    }
  }

  // ---- chunk results
  if (valid && q == a.nchunks - 1) {
    if (a.h_last && in_bounds(cc * N, N, ex.st, kBoundsScan)) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int n0 = 8 * g + 2 * k;
        if (n0 < N) a.h_last[cc * N + n0] = h[k].x;
        if (n0 + 1 < N) a.h_last[cc * N + n0 + 1] = h[k].y;
      }
    }
    if (a.conv_state_out && a.d_conv > 1) {
      // the last K-1 raw inputs of the stream conv_init ++ x, copied bit for bit
      const T* gx = static_cast<const T*>(a.x);
      const int K1 = a.d_conv - 1;
      for (int j = g; j < K1; j += G) {
        const int s = L - K1 + j;
        T v = from_f32<T>(0.f);
        if (s >= 0) {
          const long long i = cc * L + (REV ? L - 1 - s : s);
          if (in_bounds(i, 1, ex.tok, kBoundsScan)) v = gx[i];
        } else if (a.conv_init && in_bounds(cc * K1 + (K1 + s), 1, ex.win, kBoundsScan)) {
          v = static_cast<const T*>(a.conv_init)[cc * K1 + (K1 + s)];
        }
        if (in_bounds(cc * K1 + j, 1, ex.win, kBoundsScan)) static_cast<T*>(a.conv_state_out)[cc * K1 + j] = v;
      }
    }
  }
}

// ---------------------------------------------------------------- main pass, whole channels per lane

// Shared-memory layout of the main pass with whole channels per lane (16-step tiles):
// ring [2][R][RS] (x, delta, z: 32 K rows each; B, C: 16 rows each) and B, C as fp32,
// step-major.
template <typename T, int K>
struct Main1Layout {
  static constexpr int kCPW = 32 * K;
  static constexpr int kN = 16;
  static constexpr int kBCS = kN + 4;
  static constexpr int RS = row_stride<T, kT1>();
  static constexpr int R = 3 * kCPW + 2 * kN;
  static constexpr size_t slot_bytes = sizeof(T) * (size_t)R * RS;
  static constexpr size_t ring = 0;
  static constexpr size_t Bt = align16(ring + 2 * slot_bytes);
  static constexpr size_t Ct = Bt + sizeof(float) * kT1 * kBCS;
  static constexpr size_t bytes = Ct + sizeof(float) * kT1 * kBCS;
  static_assert(slot_bytes % 16 == 0, "ring slots stay 16-byte aligned");
};

// Main pass for N <= 16 with whole channels per lane: lane l holds all 16 states of the K
// channels l, l + 32, ... of its CTA and does their element-wise work, scan, readout, skip,
// gate and store in one loop, 8 steps at a time, so nothing per (t, d) passes through shared
// memory. Its shared reads are its own raw rows and the broadcast B / C rows, and every B / C
// load serves K channels: with K = 2 the loads per state update are half those of one channel
// per lane, which matters because broadcast shared loads contend with the exp2 and FMA work.
template <typename T, int K, bool CONV, bool VEC, bool REV, bool ZOH, bool S4D = false>
__global__ void __launch_bounds__(32, 8) scan_main1_kernel(const ScanArgs a) {
  static_assert(!(S4D && ZOH), "the S4D-real powers serve the Euler rule only");
  const Extents ex = extents_of(a);  // tensor sizes for the range checks of the debug build
  constexpr bool PRECISE = IoTraits<T>::kPrecise;
  using Lay = Main1Layout<T, K>;
  constexpr int CPW = Lay::kCPW;
  constexpr int BCS = Lay::kBCS;
  constexpr int RS = Lay::RS;
  using St = Stager<T, kT1, CPW, Lay::kN, true, true>;
  static_assert(St::kRows == Lay::R, "staged rows");

  extern __shared__ __align__(16) unsigned char smem_raw[];
  T (*const ring)[Lay::R][RS] = reinterpret_cast<T (*)[Lay::R][RS]>(smem_raw + Lay::ring);
  float (*const s_B)[BCS] = reinterpret_cast<float (*)[BCS]>(smem_raw + Lay::Bt);
  float (*const s_C)[BCS] = reinterpret_cast<float (*)[BCS]>(smem_raw + Lay::Ct);

  const int lane = threadIdx.x;
  const int d0 = blockIdx.x * CPW;
  const int b = blockIdx.y;
  const int q = blockIdx.z;          // chunk slowest: the chunk-0 CTAs, which need no carry, start first
  const int L = a.seqlen, N = a.dstate, dim = a.dim;
  const long long BD = (long long)a.batch * dim;
  const int t_begin = q * a.chunk_len;
  const int t_end = min(L, t_begin + a.chunk_len);
  const int ntiles = t_end > t_begin ? (t_end - t_begin + kT1 - 1) / kT1 : 0;
  const bool has_z = a.z != nullptr;

  St st;
  st.init(a, b, d0, lane);
  if (VEC && ntiles > 0) {
    st.template issue<REV>(a, ring[0], d0, t_begin, t_end, has_z);
    cp_async_commit();
  }
  bool valid[K];
  long long cc[K];
  ChannelParams cp[K];
  float w3[K][3];       // the last 3 raw inputs before the current step (conv window)
  float2 h[K][8], av[K][8], ia[K][8];
#pragma unroll
  for (int kc = 0; kc < K; ++kc) {
    const int d = d0 + lane + 32 * kc;
    valid[kc] = d < dim;
    cc[kc] = (long long)b * dim + d;
    cp[kc] = channel_params<CONV>(a, d, valid[kc]);
    w3[kc][0] = w3[kc][1] = w3[kc][2] = 0.f;
    if (CONV) halo_at<T, REV>(a, cc[kc], t_begin, q, valid[kc], w3[kc]);
    // the 16 states and A (Delta is kept in log2 units, so 2^(Delta' A) = exp(Delta A))
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int n0 = 2 * k;
      const bool arow = valid[kc] && in_bounds((long long)d * N, N, ex.dn, kBoundsScan);
      av[kc][k] = make_float2((arow && n0 < N) ? a.A[(long long)d * N + n0] : 0.f,
                              (arow && n0 + 1 < N) ? a.A[(long long)d * N + n0 + 1] : 0.f);
      h[kc][k] = make_float2(0.f, 0.f);
      ia[kc][k] = make_float2(0.f, 0.f);
      if (ZOH) {
        auto inv = [](float v) { return v != 0.f ? 1.0f / v : 0.f; };
        ia[kc][k] = make_float2(inv(av[kc][k].x), inv(av[kc][k].y));
      }
    }
    if (valid[kc] && a.h0 && in_bounds(cc[kc] * N, N, ex.st, kBoundsScan)) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int n0 = 2 * k;
        h[kc][k] = make_float2(n0 < N ? a.h0[cc[kc] * N + n0] : 0.f, n0 + 1 < N ? a.h0[cc[kc] * N + n0 + 1] : 0.f);
      }
    }
  }
  // S4D-real: when A[d, n] = (n+1) A[d, 0] holds exactly for every channel of the CTA (one warp
  // vote), Abar_n = Abar_0^(n+1) comes from one exp2 per 4 states and multiplies; otherwise the
  // generic exp2 per state
  float A0[K];
  bool s4_lane = true;
#pragma unroll
  for (int kc = 0; kc < K; ++kc) {
    A0[kc] = av[kc][0].x;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (2 * k < N) s4_lane = s4_lane && av[kc][k].x == (float)(2 * k + 1) * A0[kc];
      if (2 * k + 1 < N) s4_lane = s4_lane && av[kc][k].y == (float)(2 * k + 2) * A0[kc];
    }
  }
  const bool s4d_ok = S4D && __all_sync(0xffffffffu, s4_lane);
  if (q > 0) {
    // carry-in (the carry kernel ran before this one in stream order): compose the aggregates
    // of chunks 0 .. q-1 onto h0
#pragma unroll
    for (int kc = 0; kc < K; ++kc) {
      if (!valid[kc]) continue;
      for (int j = 0; j < q; ++j) {
        const long long e = (long long)j * BD + cc[kc];
        if (!in_bounds(e, 1, ex.wsS, kBoundsScan) || !in_bounds(e * 16, 16, ex.wsH, kBoundsScan)) continue;
        const float Sj = a.ws_S[e];
        const float4* hp = reinterpret_cast<const float4*>(a.ws_h + e * 16);
        float4 hb[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) hb[k] = hp[k];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 x0 = fmul2(f2(Sj), av[kc][2 * k]), x1 = fmul2(f2(Sj), av[kc][2 * k + 1]);
          h[kc][2 * k] = ffma2(make_float2(ex2_approx(x0.x), ex2_approx(x0.y)), h[kc][2 * k],
                               make_float2(hb[k].x, hb[k].y));
          h[kc][2 * k + 1] = ffma2(make_float2(ex2_approx(x1.x), ex2_approx(x1.y)), h[kc][2 * k + 1],
                                   make_float2(hb[k].z, hb[k].w));
        }
      }
    }
  }

  // the walk over the chunk's tiles; POW: Abar_n = Abar_0^(n+1) by multiplies (S4D-real)
  auto walk = [&](auto pow_tag) {
    constexpr bool POW = decltype(pow_tag)::value;
    for (int it = 0; it < ntiles; ++it) {
      const int bf = it & 1;
      const int t0 = t_begin + it * kT1;
      const int tl = min(kT1, t_end - t0);
      if (VEC) {
        cp_async_wait<0>();
      } else {
        st.template load_sync<REV>(a, ring[bf], d0, t0, t_end, has_z);
      }
      __syncwarp();  // tile `it` visible to the warp; every lane is past tile it-1, so its slot can be refilled
      if (VEC && it + 1 < ntiles) {
        st.template issue<REV>(a, ring[bf ^ 1], d0, t0 + kT1, t_end, has_z);
        cp_async_commit();
      }
      const T (*raw)[RS] = ring[bf];
      // B and C -> fp32 step-major: lanes 0-15 convert B, lanes 16-31 C (16 blocks of 4x4 each)
      if (lane < 16) transpose_rows<T, kT1, Lay::kN, BCS, REV>(raw + 3 * CPW, s_B, ZOH ? 1.0f : kLn2, lane);
      else transpose_rows<T, kT1, Lay::kN, BCS, REV>(raw + 3 * CPW + Lay::kN, s_C, 1.0f, lane - 16);
      __syncwarp();

#pragma unroll 1
      for (int tt = 0; tt < tl; tt += kBlk) {
        const bool full = tt + kBlk <= tl;
        // ---- element-wise work of steps tt .. tt+7: u, Delta', the scan input, D u
        float dl[K][kBlk], du[K][kBlk], sk[K][kBlk];
#pragma unroll
        for (int kc = 0; kc < K; ++kc) {
          float xv[kBlk], dv[kBlk];
          load_seg8<T, kT1, REV>(raw[lane + 32 * kc], tt, xv);
          load_seg8<T, kT1, REV>(raw[CPW + lane + 32 * kc], tt, dv);
#pragma unroll
          for (int j = 0; j < kBlk; j += 2) {
            float2 u;
            if (CONV) {
              const float win0[4] = {w3[kc][0], w3[kc][1], w3[kc][2], xv[j]};
              const float win1[4] = {w3[kc][1], w3[kc][2], xv[j], xv[j + 1]};
              const float c0 = conv4(win0, cp[kc].w0, cp[kc].w1, cp[kc].w2, cp[kc].w3, cp[kc].cb);
              const float c1 = conv4(win1, cp[kc].w0, cp[kc].w1, cp[kc].w2, cp[kc].w3, cp[kc].cb);
              w3[kc][0] = w3[kc][2]; w3[kc][1] = xv[j]; w3[kc][2] = xv[j + 1];
              u = silu2_tier<PRECISE>(make_float2(c0, c1));
            } else {
              u = make_float2(xv[j], xv[j + 1]);
            }
            float2 D2 = delta_log2<PRECISE>(make_float2(dv[j], dv[j + 1]), cp[kc].bias, cp[kc].bias_l2,
                                            a.delta_softplus);
            if (!full) {  // steps past the tile end are identity updates: Delta = 0, u = 0
              const bool i0 = tt + j < tl, i1 = tt + j + 1 < tl;
              D2 = make_float2(i0 ? D2.x : 0.f, i1 ? D2.y : 0.f);
              u = make_float2(i0 ? u.x : 0.f, i1 ? u.y : 0.f);
            }
            const float2 du2 = ZOH ? u : fmul2(D2, u);
            const float2 sk2 = fmul2(f2(cp[kc].Dd), u);
            dl[kc][j] = D2.x; dl[kc][j + 1] = D2.y;
            du[kc][j] = du2.x; du[kc][j + 1] = du2.y;
            sk[kc][j] = sk2.x; sk[kc][j + 1] = sk2.y;
          }
        }
        // ---- scan of the 8 steps: 16 states per channel, one exp2 per state update; each
        // B / C row loaded serves the K channels
        float yv[K][kBlk];
#pragma unroll
        for (int j = 0; j < kBlk; ++j) {
          float2 p0[K], p1[K];
#pragma unroll
          for (int kc = 0; kc < K; ++kc) p0[kc] = p1[kc] = f2(0.f);
          // POW: states 4g .. 4g+3 take the anchor Abar_0^(4g+1) (one exp2) times (1, Abar_0,
          // Abar_0^2, Abar_0^3), so no Abar_n carries more than 4 times the rounding of one exp2
          float2 v01[K], v23[K];
          float x0[K];
          if constexpr (POW) {
#pragma unroll
            for (int kc = 0; kc < K; ++kc) {
              x0[kc] = dl[kc][j] * A0[kc];
              const float e0 = ex2_approx(x0[kc]);
              const float e2 = e0 * e0;
              v01[kc] = make_float2(1.f, e0);
              v23[kc] = make_float2(e2, e2 * e0);
            }
          }
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const float4 bq = *reinterpret_cast<const float4*>(&s_B[tt + j][4 * k4]);
            const float4 cq = *reinterpret_cast<const float4*>(&s_C[tt + j][4 * k4]);
            const float2 bv[2] = {make_float2(bq.x, bq.y), make_float2(bq.z, bq.w)};
#pragma unroll
            for (int kc = 0; kc < K; ++kc) {
              const float2 dd = f2(dl[kc][j]);
              const float2 uu = f2(du[kc][j]);
              float anchor = 0.f;  // POW: Abar_0^(4 k4 + 1), the exp2 of states 4 k4 .. 4 k4 + 3
              if constexpr (POW) anchor = ex2_approx((float)(4 * k4 + 1) * x0[kc]);
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                const int k = 2 * k4 + i;
                float2 x, e;
                if constexpr (POW) {
                  e = fmul2(f2(anchor), i == 0 ? v01[kc] : v23[kc]);
                  x = e;  // unused: POW serves the Euler rule only
                } else {
                  x = fmul2(dd, av[kc][k]);
                  e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                }
                float2 in = fmul2(uu, bv[i]);
                if (ZOH) in = fmul2(in, zoh_factor2(x, e, dd, ia[kc][k]));
                h[kc][k] = ffma2(e, h[kc][k], in);
              }
              p0[kc] = ffma2(h[kc][2 * k4], make_float2(cq.x, cq.y), p0[kc]);
              p1[kc] = ffma2(h[kc][2 * k4 + 1], make_float2(cq.z, cq.w), p1[kc]);
            }
          }
#pragma unroll
          for (int kc = 0; kc < K; ++kc) {
            const float2 p = fadd2(p0[kc], p1[kc]);
            yv[kc][j] = p.x + p.y + sk[kc][j];
          }
        }
        // ---- gate and store
#pragma unroll
        for (int kc = 0; kc < K; ++kc) {
          if (!valid[kc]) continue;
          T* const orow = static_cast<T*>(a.out) + cc[kc] * L;
          float o[kBlk];
          if (has_z) {
            float zv[kBlk];
            load_seg8<T, kT1, REV>(raw[2 * CPW + lane + 32 * kc], tt, zv);
#pragma unroll
            for (int j = 0; j < kBlk; j += 2) {
              const float2 gt = silu2_tier<PRECISE>(make_float2(zv[j], zv[j + 1]));
              const float2 y = fmul2(make_float2(yv[kc][j], yv[kc][j + 1]), gt);
              o[j] = y.x; o[j + 1] = y.y;
            }
          } else {
#pragma unroll
            for (int j = 0; j < kBlk; ++j) o[j] = yv[kc][j];
          }
          if (REV) {
            if (VEC && full) {
              float r[kBlk];
#pragma unroll
              for (int j = 0; j < kBlk; ++j) r[j] = o[kBlk - 1 - j];
              if (ptr_in(static_cast<T*>(a.out), orow + (L - t0 - tt - kBlk), kBlk, ex.tok, kBoundsScan))
                store8(orow + (L - t0 - tt - kBlk), r);
            } else if (VEC && tt + 4 <= tl) {  // fp32 rows can end on a 4-step boundary
              const float r4[4] = {o[3], o[2], o[1], o[0]};
              if (ptr_in(static_cast<T*>(a.out), orow + (L - t0 - tt - 4), 4, ex.tok, kBoundsScan))
                store4(orow + (L - t0 - tt - 4), r4);
            } else {
#pragma unroll
              for (int j = 0; j < kBlk; ++j)
                if (tt + j < tl && ptr_in(static_cast<T*>(a.out), orow + (L - 1 - (t0 + tt + j)), 1, ex.tok, kBoundsScan))
                  orow[L - 1 - (t0 + tt + j)] = from_f32<T>(o[j]);
            }
          } else {
            T* dst = orow + t0 + tt;
            if (VEC && full) {
              if (ptr_in(static_cast<T*>(a.out), dst, kBlk, ex.tok, kBoundsScan)) store8(dst, o);
            } else if (VEC && tt + 4 <= tl) {
              const float o4[4] = {o[0], o[1], o[2], o[3]};
              if (ptr_in(static_cast<T*>(a.out), dst, 4, ex.tok, kBoundsScan)) store4(dst, o4);
            } else {
#pragma unroll
              for (int j = 0; j < kBlk; ++j)
                if (tt + j < tl && ptr_in(static_cast<T*>(a.out), dst + j, 1, ex.tok, kBoundsScan)) dst[j] = from_f32<T>(o[j]);
            }
          }
        }
      }
    }

  };
  if constexpr (S4D) {
    if (s4d_ok) walk(std::true_type{});
    else walk(std::false_type{});
  } else {
    walk(std::false_type{});
  }

  // ---- chunk results
  if (q == a.nchunks - 1) {
#pragma unroll
    for (int kc = 0; kc < K; ++kc) {
      if (!valid[kc]) continue;
      if (a.h_last && in_bounds(cc[kc] * N, N, ex.st, kBoundsScan)) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int n0 = 2 * k;
          if (n0 < N) a.h_last[cc[kc] * N + n0] = h[kc][k].x;
          if (n0 + 1 < N) a.h_last[cc[kc] * N + n0 + 1] = h[kc][k].y;
        }
      }
      if (a.conv_state_out && a.d_conv > 1) {
        // the last K-1 raw inputs of the stream conv_init ++ x, copied bit for bit
        const T* gx = static_cast<const T*>(a.x);
        const int K1 = a.d_conv - 1;
        for (int j = 0; j < K1; ++j) {
          const int s = L - K1 + j;
          T v = from_f32<T>(0.f);
          if (s >= 0) {
            const long long i = cc[kc] * L + (REV ? L - 1 - s : s);
            if (in_bounds(i, 1, ex.tok, kBoundsScan)) v = gx[i];
          } else if (a.conv_init && in_bounds(cc[kc] * K1 + (K1 + s), 1, ex.win, kBoundsScan)) {
            v = static_cast<const T*>(a.conv_init)[cc[kc] * K1 + (K1 + s)];
          }
          if (in_bounds(cc[kc] * K1 + j, 1, ex.win, kBoundsScan)) static_cast<T*>(a.conv_state_out)[cc[kc] * K1 + j] = v;
        }
      }
    }
  }
}

// ---------------------------------------------------------------- carry pass

template <typename T, int G, int K, bool CONV, bool VEC, bool REV, bool ZOH, bool S4D = false>
__global__ void __launch_bounds__(32, 16) scan_carry_kernel(const ScanArgs a) {
  static_assert(!S4D || (G == 1 && !ZOH), "the S4D-real powers: whole channels, Euler rule");
  const Extents ex = extents_of(a);  // tensor sizes for the range checks of the debug build
  constexpr bool PRECISE = IoTraits<T>::kPrecise;
  using Geo = CarryGeo<G, K>;
  using Lay = CarryLayout<T, G, K>;
  constexpr int CPW = Geo::kCPW;
  constexpr int CPL = 32 / G;       // distance between a lane's channels
  constexpr int BCS = Geo::kBCS;
  constexpr int RS = Lay::RS;
  using St = Stager<T, kT1, CPW, Geo::kN, false, false>;
  static_assert(St::kRows == Lay::R, "staged rows");

  extern __shared__ __align__(16) unsigned char smem_raw[];
  T (*const ring)[Lay::R][RS] = reinterpret_cast<T (*)[Lay::R][RS]>(smem_raw + Lay::ring);
  float (*const s_B)[BCS] = reinterpret_cast<float (*)[BCS]>(smem_raw + Lay::Bt);

  const int lane = threadIdx.x;
  const int c = lane / G;            // the lane's first channel within the CTA
  const int g = lane % G;            // states 16g .. 16g+15
  const int d0 = blockIdx.x * CPW;
  const int b = blockIdx.y;
  const int q = blockIdx.z;
  const int L = a.seqlen, N = a.dstate, dim = a.dim;
  const long long BD = (long long)a.batch * dim;
  const int t_begin = q * a.chunk_len;
  const int t_end = min(L, t_begin + a.chunk_len);
  const int ntiles = t_end > t_begin ? (t_end - t_begin + kT1 - 1) / kT1 : 0;
  const int NS = N <= 16 ? 16 : 32;

  St st;
  st.init(a, b, d0, lane);
  if (VEC && ntiles > 0) {
    st.template issue<REV>(a, ring[0], d0, t_begin, t_end, false);
    cp_async_commit();
  }
  bool valid[K];
  long long cc[K];
  ChannelParams cp[K];
  float w3[K][3];       // the last 3 raw inputs before the current step (conv window)
  float2 h[K][8], av[K][8], ia[K][8];
  float dsum[K];        // sum of Delta' over the chunk
#pragma unroll
  for (int kc = 0; kc < K; ++kc) {
    const int d = d0 + c + kc * CPL;
    valid[kc] = d < dim;
    cc[kc] = (long long)b * dim + d;
    cp[kc] = channel_params<CONV>(a, d, valid[kc]);
    w3[kc][0] = w3[kc][1] = w3[kc][2] = 0.f;
    if (CONV) halo_at<T, REV>(a, cc[kc], t_begin, q, valid[kc], w3[kc]);
    dsum[kc] = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int n0 = 16 * g + 2 * k;
      const bool arow = valid[kc] && in_bounds((long long)d * N, N, ex.dn, kBoundsScan);
      av[kc][k] = make_float2((arow && n0 < N) ? a.A[(long long)d * N + n0] : 0.f,
                              (arow && n0 + 1 < N) ? a.A[(long long)d * N + n0 + 1] : 0.f);
      h[kc][k] = make_float2(0.f, 0.f);
      ia[kc][k] = make_float2(0.f, 0.f);
      if (ZOH) {
        auto inv = [](float v) { return v != 0.f ? 1.0f / v : 0.f; };
        ia[kc][k] = make_float2(inv(av[kc][k].x), inv(av[kc][k].y));
      }
    }
  }

  // S4D-real check and powers as in the whole-channel main pass
  float A0[K];
  bool s4_lane = true;
#pragma unroll
  for (int kc = 0; kc < K; ++kc) {
    A0[kc] = av[kc][0].x;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (2 * k < N) s4_lane = s4_lane && av[kc][k].x == (float)(2 * k + 1) * A0[kc];
      if (2 * k + 1 < N) s4_lane = s4_lane && av[kc][k].y == (float)(2 * k + 2) * A0[kc];
    }
  }
  const bool s4d_ok = S4D && __all_sync(0xffffffffu, s4_lane);

  auto walk = [&](auto pow_tag) {
    constexpr bool POW = decltype(pow_tag)::value;
    for (int it = 0; it < ntiles; ++it) {
      const int bf = it & 1;
      const int t0 = t_begin + it * kT1;
      const int tl = min(kT1, t_end - t0);
      if (VEC) {
        cp_async_wait<0>();
      } else {
        st.template load_sync<REV>(a, ring[bf], d0, t0, t_end, false);
      }
      __syncwarp();
      if (VEC && it + 1 < ntiles) {
        st.template issue<REV>(a, ring[bf ^ 1], d0, t0 + kT1, t_end, false);
        cp_async_commit();
      }
      const T (*raw)[RS] = ring[bf];
      transpose_rows<T, kT1, Geo::kN, BCS, REV>(raw + 2 * CPW, s_B, ZOH ? 1.0f : kLn2, lane);
      __syncwarp();

      // ---- element-wise work and scan, four steps at a time
      const int tlu = (tl + 3) & ~3;
#pragma unroll 1
      for (int t = 0; t < tlu; t += 4) {
        float dl[K][4], du[K][4];
#pragma unroll
        for (int kc = 0; kc < K; ++kc) {
          float xv[4], dv[4];
          load_seg4<T, kT1, REV>(raw[c + kc * CPL], t, xv);
          load_seg4<T, kT1, REV>(raw[CPW + c + kc * CPL], t, dv);
#pragma unroll
          for (int j = 0; j < 4; j += 2) {
            float2 u;
            if (CONV) {
              const float win0[4] = {w3[kc][0], w3[kc][1], w3[kc][2], xv[j]};
              const float c0 = conv4(win0, cp[kc].w0, cp[kc].w1, cp[kc].w2, cp[kc].w3, cp[kc].cb);
              const float win1[4] = {w3[kc][1], w3[kc][2], xv[j], xv[j + 1]};
              const float c1 = conv4(win1, cp[kc].w0, cp[kc].w1, cp[kc].w2, cp[kc].w3, cp[kc].cb);
              w3[kc][0] = w3[kc][2]; w3[kc][1] = xv[j]; w3[kc][2] = xv[j + 1];
              u = silu2_tier<PRECISE>(make_float2(c0, c1));
            } else {
              u = make_float2(xv[j], xv[j + 1]);
            }
            float2 D2 = delta_log2<PRECISE>(make_float2(dv[j], dv[j + 1]), cp[kc].bias, cp[kc].bias_l2,
                                            a.delta_softplus);
            if (t + 4 > tl) {  // steps past the tile end are identity updates: Delta = 0, u = 0
              const bool i0 = t + j < tl, i1 = t + j + 1 < tl;
              D2 = make_float2(i0 ? D2.x : 0.f, i1 ? D2.y : 0.f);
              u = make_float2(i0 ? u.x : 0.f, i1 ? u.y : 0.f);
            }
            const float2 du2 = ZOH ? u : fmul2(D2, u);
            dl[kc][j] = D2.x; dl[kc][j + 1] = D2.y;
            du[kc][j] = du2.x; du[kc][j + 1] = du2.y;
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int kc = 0; kc < K; ++kc) dsum[kc] += dl[kc][j];
          float2 v01[K], v23[K];
          float x0[K];
          if constexpr (POW) {
#pragma unroll
            for (int kc = 0; kc < K; ++kc) {
              x0[kc] = dl[kc][j] * A0[kc];
              const float e0 = ex2_approx(x0[kc]);
              const float e2 = e0 * e0;
              v01[kc] = make_float2(1.f, e0);
              v23[kc] = make_float2(e2, e2 * e0);
            }
          }
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const float4 bq = *reinterpret_cast<const float4*>(&s_B[t + j][16 * g + 4 * k4]);
            const float2 bv[2] = {make_float2(bq.x, bq.y), make_float2(bq.z, bq.w)};
#pragma unroll
            for (int kc = 0; kc < K; ++kc) {
              const float2 dd = f2(dl[kc][j]);
              const float2 uu = f2(du[kc][j]);
              float anchor = 0.f;  // POW: Abar_0^(4 k4 + 1), the exp2 of states 4 k4 .. 4 k4 + 3
              if constexpr (POW) anchor = ex2_approx((float)(4 * k4 + 1) * x0[kc]);
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                const int k = 2 * k4 + i;
                float2 x, e;
                if constexpr (POW) {
                  e = fmul2(f2(anchor), i == 0 ? v01[kc] : v23[kc]);
                  x = e;  // unused: POW serves the Euler rule only
                } else {
                  x = fmul2(dd, av[kc][k]);
                  e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                }
                float2 in = fmul2(uu, bv[i]);
                if (ZOH) in = fmul2(in, zoh_factor2(x, e, dd, ia[kc][k]));
                h[kc][k] = ffma2(e, h[kc][k], in);
              }
            }
          }
        }
      }
    }
  };
  if constexpr (S4D) {
    if (s4d_ok) walk(std::true_type{});
    else walk(std::false_type{});
  } else {
    walk(std::false_type{});
  }

#pragma unroll
  for (int kc = 0; kc < K; ++kc) {
    const long long e = (long long)q * BD + cc[kc];
    if (valid[kc] && in_bounds(e * NS + 16 * g, 16, ex.wsH, kBoundsScan) && in_bounds(e, 1, ex.wsS, kBoundsScan)) {
      // lane g's 16 states lie at 16g .. 16g+15 of the channel's stride (16 for G = 1, 32 for G = 2)
      float4* hp = reinterpret_cast<float4*>(a.ws_h + e * NS + 16 * g);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        hp[k] = make_float4(h[kc][2 * k].x, h[kc][2 * k].y, h[kc][2 * k + 1].x, h[kc][2 * k + 1].y);
      if (g == 0) a.ws_S[e] = dsum[kc];
    }
  }
}

// ---------------------------------------------------------------- launch

// Opts a kernel into its dynamic shared memory once per device.
template <typename K>
cudaError_t prepare(K kernel, size_t smem, int (&configured)[64]) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 0 && dev < 64 && configured[dev]) return cudaSuccess;
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err == cudaSuccess && dev >= 0 && dev < 64) configured[dev] = 1;
  return err;
}

template <typename T, int G, bool CONV, bool VEC, bool REV, bool ZOH>
cudaError_t prepare_main() {
  static int configured[64] = {0};
  return prepare(scan_main_kernel<T, G, CONV, VEC, REV, ZOH>, MainLayout<T, G>::bytes, configured);
}

template <typename T, int G, int K, bool CONV, bool VEC, bool REV, bool ZOH, bool S4D = false>
cudaError_t prepare_carry() {
  static int configured[64] = {0};
  return prepare(scan_carry_kernel<T, G, K, CONV, VEC, REV, ZOH, S4D>, CarryLayout<T, G, K>::bytes, configured);
}

template <typename T, int G, bool CONV, bool VEC, bool REV, bool ZOH>
cudaError_t launch_main(const ScanArgs& a, cudaStream_t stream) {
  cudaError_t err = prepare_main<T, G, CONV, VEC, REV, ZOH>();
  if (err != cudaSuccess) return err;
  const dim3 grid((a.dim + MainGeo<G>::kCPW - 1) / MainGeo<G>::kCPW, a.batch, a.nchunks);
  scan_main_kernel<T, G, CONV, VEC, REV, ZOH><<<grid, 32, MainLayout<T, G>::bytes, stream>>>(a);
  return cudaGetLastError();
}

template <typename T, int G, int K, bool CONV, bool VEC, bool REV, bool ZOH, bool S4D = false>
cudaError_t launch_carry(const ScanArgs& a, cudaStream_t stream, int ncarry) {
  cudaError_t err = prepare_carry<T, G, K, CONV, VEC, REV, ZOH, S4D>();
  if (err != cudaSuccess) return err;
  constexpr int cpw = CarryGeo<G, K>::kCPW;
  const dim3 grid((a.dim + cpw - 1) / cpw, a.batch, ncarry);
  scan_carry_kernel<T, G, K, CONV, VEC, REV, ZOH, S4D><<<grid, 32, CarryLayout<T, G, K>::bytes, stream>>>(a);
  return cudaGetLastError();
}

constexpr int kMain1K = 2;  // channels per lane of the whole-channel main pass

template <typename T, bool CONV, bool VEC, bool REV, bool ZOH, bool S4D = false>
cudaError_t prepare_main1() {
  static int configured[64] = {0};
  return prepare(scan_main1_kernel<T, kMain1K, CONV, VEC, REV, ZOH, S4D>, Main1Layout<T, kMain1K>::bytes,
                 configured);
}

template <typename T, bool CONV, bool VEC, bool REV, bool ZOH, bool S4D = false>
cudaError_t launch_main1(const ScanArgs& a, cudaStream_t stream) {
  cudaError_t err = prepare_main1<T, CONV, VEC, REV, ZOH, S4D>();
  if (err != cudaSuccess) return err;
  using Lay = Main1Layout<T, kMain1K>;
  const dim3 grid((a.dim + Lay::kCPW - 1) / Lay::kCPW, a.batch, a.nchunks);
  scan_main1_kernel<T, kMain1K, CONV, VEC, REV, ZOH, S4D><<<grid, 32, Lay::bytes, stream>>>(a);
  return cudaGetLastError();
}

// S4D: the S4D-real powers, for whole-channel passes (N <= 16, one lane per channel) only; the
// caller routes every other plan to S4D = false.
template <typename T, bool CONV, bool VEC, bool REV, bool ZOH, bool S4D = false>
cudaError_t launch_pair(const ScanArgs& a, cudaStream_t stream) {
  const bool big = a.dstate > 16;
  if constexpr (S4D) {
    if (a.nchunks > 1) {
      const cudaError_t err = launch_carry<T, 1, 1, CONV, VEC, REV, ZOH, true>(a, stream, a.nchunks - 1);
      if (err != cudaSuccess) return err;
    }
    return launch_main1<T, CONV, VEC, REV, ZOH, true>(a, stream);
  }
  if (a.nchunks > 1) {
    cudaError_t err = big ? launch_carry<T, 2, 1, CONV, VEC, REV, ZOH>(a, stream, a.nchunks - 1)
                          : launch_carry<T, 1, 1, CONV, VEC, REV, ZOH>(a, stream, a.nchunks - 1);
    if (err != cudaSuccess) return err;
  }
  // The main pass follows the carry pass in stream order. Launched as its programmatic
  // dependent instead, the main CTAs of later chunks took SM slots as carry CTAs finished and
  // waited there, which placed them unevenly across the SMSPs (long scan: 2-5% slower).
  if (big) return launch_main<T, 4, CONV, VEC, REV, ZOH>(a, stream);
  if (a.lanes == 1) return launch_main1<T, CONV, VEC, REV, ZOH>(a, stream);
  return launch_main<T, 2, CONV, VEC, REV, ZOH>(a, stream);
}

template <typename T, bool REV, bool ZOH, bool S4D = false>
cudaError_t dispatch_opts(const ScanArgs& a, cudaStream_t s) {
  const bool conv = a.conv_w != nullptr;
  if (conv)
    return a.vec ? launch_pair<T, true, true, REV, ZOH, S4D>(a, s) : launch_pair<T, true, false, REV, ZOH, S4D>(a, s);
  return a.vec ? launch_pair<T, false, true, REV, ZOH, S4D>(a, s) : launch_pair<T, false, false, REV, ZOH, S4D>(a, s);
}

template <typename T>
cudaError_t dispatch(const ScanArgs& a, cudaStream_t s) {
  if (a.zoh) return a.reverse ? dispatch_opts<T, true, true>(a, s) : dispatch_opts<T, false, true>(a, s);
  if (a.s4d && a.lanes == 1 && a.dstate <= 16)
    return a.reverse ? dispatch_opts<T, true, false, true>(a, s) : dispatch_opts<T, false, false, true>(a, s);
  return a.reverse ? dispatch_opts<T, true, false>(a, s) : dispatch_opts<T, false, false>(a, s);
}

template <typename T, int G>
int resident_main_ctas() {
  int n = 0;
  if (prepare_main<T, G, true, true, false, false>() != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, scan_main_kernel<T, G, true, true, false, false>, 32,
                                                    MainLayout<T, G>::bytes) != cudaSuccess ||
      n <= 0) {
    cudaGetLastError();
    // no device to ask: the shared-memory limit the kernel is built for
    return (int)(227 * 1024 / (MainLayout<T, G>::bytes + 1024));
  }
  return n;
}

template <typename T>
int resident_main1_ctas() {
  using Lay = Main1Layout<T, kMain1K>;
  int n = 0;
  if (prepare_main1<T, true, true, false, false>() != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, scan_main1_kernel<T, kMain1K, true, true, false, false>, 32,
                                                    Lay::bytes) != cudaSuccess ||
      n <= 0) {
    cudaGetLastError();
    return (int)(227 * 1024 / (Lay::bytes + 1024));
  }
  return n;
}

// ---------------------------------------------------------------- segment aggregates

// Folds the carries of a segment's q chunks into the segment's aggregate: S = sum_j S_j (log2
// units in, natural units out) and h = 2^(A S_j) h + h_j over j = 0 .. q-1 from h = 0, the
// segment's end state from a zero state. One thread per (channel, state).
__global__ void aggregate_fold_kernel(const float* __restrict__ S, const float* __restrict__ hs,
                                      const float* __restrict__ A, float* __restrict__ S_out,
                                      float* __restrict__ h_out, long long BD, int dim, int N, int NS, int nq) {
  const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (i >= BD * N) return;
  const long long cc = i / N;
  const int n = (int)(i % N);
  const int d = (int)(cc % dim);
  if (!in_bounds((long long)d * N + n, 1, (long long)dim * N, kBoundsSegment)) return;
  const float a = A[(long long)d * N + n];
  float sum = 0.f, h = 0.f;
  for (int j = 0; j < nq; ++j) {
    const long long e = (long long)j * BD + cc;
    if (!in_bounds(e, 1, nq * BD, kBoundsSegment) || !in_bounds(e * NS + n, 1, nq * BD * NS, kBoundsSegment))
      continue;
    const float sj = S[e];
    h = fmaf(ex2_approx(a * sj), h, hs[e * NS + n]);
    sum += sj;
  }
  h_out[cc * N + n] = h;
  if (n == 0) S_out[cc] = sum * kLn2;
}

// Composition of segment aggregates onto an initial state: h = exp(A S_j) h + b_j for
// j = 0 .. nseg-1 (S in natural units). One thread per (channel, state).
__global__ void compose_kernel(const float* __restrict__ S, const float* __restrict__ b, const float* __restrict__ A,
                               const float* __restrict__ h0, float* __restrict__ h_out, long long BD, int dim, int N,
                               int nseg) {
  const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (i >= BD * N) return;
  const long long cc = i / N;
  const int n = (int)(i % N);
  const int d = (int)(cc % dim);
  if (!in_bounds((long long)d * N + n, 1, (long long)dim * N, kBoundsSegment)) return;
  const float a = A[(long long)d * N + n] * kLog2e;
  float h = h0 ? h0[cc * N + n] : 0.f;
  for (int j = 0; j < nseg; ++j) {
    const long long e = (long long)j * BD + cc;
    if (!in_bounds(e, 1, nseg * BD, kBoundsSegment) || !in_bounds(e * N + n, 1, nseg * BD * N, kBoundsSegment))
      continue;
    h = fmaf(ex2_approx(a * S[e]), h, b[e * N + n]);
  }
  h_out[cc * N + n] = h;
}

template <typename T, bool CONV, bool VEC, bool REV, bool ZOH>
cudaError_t launch_aggregate_t(const ScanArgs& a, float* S_out, float* h_out, cudaStream_t stream) {
  // every chunk of the segment, the last one included, goes through the carry kernel
  const bool big = a.dstate > 16;
  cudaError_t err = big ? launch_carry<T, 2, 1, CONV, VEC, REV, ZOH>(a, stream, a.nchunks)
                        : launch_carry<T, 1, 1, CONV, VEC, REV, ZOH>(a, stream, a.nchunks);
  if (err != cudaSuccess) return err;
  const long long BD = (long long)a.batch * a.dim;
  const long long n = BD * a.dstate;
  const int threads = 256;
  aggregate_fold_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, stream>>>(
      a.ws_S, a.ws_h, a.A, S_out, h_out, BD, a.dim, a.dstate, scan_state_stride(a.dstate), a.nchunks);
  return cudaGetLastError();
}

template <typename T, bool REV, bool ZOH>
cudaError_t aggregate_opts(const ScanArgs& a, float* S_out, float* h_out, cudaStream_t s) {
  const bool conv = a.conv_w != nullptr;
  if (conv)
    return a.vec ? launch_aggregate_t<T, true, true, REV, ZOH>(a, S_out, h_out, s)
                 : launch_aggregate_t<T, true, false, REV, ZOH>(a, S_out, h_out, s);
  return a.vec ? launch_aggregate_t<T, false, true, REV, ZOH>(a, S_out, h_out, s)
               : launch_aggregate_t<T, false, false, REV, ZOH>(a, S_out, h_out, s);
}

template <typename T>
cudaError_t aggregate_dispatch(const ScanArgs& a, float* S_out, float* h_out, cudaStream_t s) {
  if (a.zoh)
    return a.reverse ? aggregate_opts<T, true, true>(a, S_out, h_out, s) : aggregate_opts<T, false, true>(a, S_out, h_out, s);
  return a.reverse ? aggregate_opts<T, true, false>(a, S_out, h_out, s) : aggregate_opts<T, false, false>(a, S_out, h_out, s);
}

}  // namespace

int scan_carry_resident_ctas_per_sm(bool bf16, int dstate) {
  int n = 0;
  cudaError_t e;
  if (dstate > 16)
    e = bf16 ? (prepare_carry<__nv_bfloat16, 2, 1, false, true, false, false>(),
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, scan_carry_kernel<__nv_bfloat16, 2, 1, false, true, false, false>,
                                                              32, CarryLayout<__nv_bfloat16, 2, 1>::bytes))
             : (prepare_carry<float, 2, 1, false, true, false, false>(),
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, scan_carry_kernel<float, 2, 1, false, true, false, false>, 32,
                                                              CarryLayout<float, 2, 1>::bytes));
  else
    e = bf16 ? (prepare_carry<__nv_bfloat16, 1, 1, false, true, false, false>(),
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, scan_carry_kernel<__nv_bfloat16, 1, 1, false, true, false, false>,
                                                              32, CarryLayout<__nv_bfloat16, 1, 1>::bytes))
             : (prepare_carry<float, 1, 1, false, true, false, false>(),
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, scan_carry_kernel<float, 1, 1, false, true, false, false>, 32,
                                                              CarryLayout<float, 1, 1>::bytes));
  if (e != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 16;  // no device to ask: the register limit the kernel is built for
  }
  return n;
}

int scan_carry_channels_per_cta(int dstate) { return dstate > 16 ? CarryGeo<2, 1>::kCPW : CarryGeo<1, 1>::kCPW; }

cudaError_t launch_scan_aggregate(const ScanArgs& a, float* S_out, float* h_out, cudaStream_t stream) {
  if (a.bf16) return aggregate_dispatch<__nv_bfloat16>(a, S_out, h_out, stream);
  return aggregate_dispatch<float>(a, S_out, h_out, stream);
}

cudaError_t launch_scan_compose(const float* S, const float* b, const float* A, const float* h0, float* h_out,
                                int nseg, int batch, int dim, int dstate, cudaStream_t stream) {
  const long long BD = (long long)batch * dim;
  const long long n = BD * dstate;
  const int threads = 256;
  compose_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, stream>>>(S, b, A, h0, h_out, BD, dim, dstate,
                                                                                   nseg);
  return cudaGetLastError();
}

int scan_channels_per_cta(int lanes) {
  return lanes == 1 ? Main1Layout<float, kMain1K>::kCPW : (lanes == 2 ? MainGeo<2>::kCPW : MainGeo<4>::kCPW);
}

int scan_resident_ctas_per_sm(bool bf16, int lanes) {
  if (lanes == 1) return bf16 ? resident_main1_ctas<__nv_bfloat16>() : resident_main1_ctas<float>();
  if (lanes == 4) return bf16 ? resident_main_ctas<__nv_bfloat16, 4>() : resident_main_ctas<float, 4>();
  return bf16 ? resident_main_ctas<__nv_bfloat16, 2>() : resident_main_ctas<float, 2>();
}

int scan_state_stride(int dstate) { return dstate <= 16 ? 16 : 32; }

size_t scan_workspace_bytes(long long channels, int nchunks, int dstate) {
  if (nchunks <= 1) return 0;
  const long long m = (long long)(nchunks - 1) * channels;
  const size_t s_bytes = ((size_t)m * sizeof(float) + 255) & ~(size_t)255;
  return s_bytes + (size_t)m * scan_state_stride(dstate) * sizeof(float);
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

cudaError_t launch_scan_carry(const ScanArgs& a, cudaStream_t stream) {
  // the forward carries alone (chunks 0 .. nchunks-2), forward time, Euler, no conv, N <= 16
  if (a.nchunks <= 1) return cudaSuccess;
  if (a.bf16)
    return a.vec ? launch_carry<__nv_bfloat16, 1, 1, false, true, false, false>(a, stream, a.nchunks - 1)
                 : launch_carry<__nv_bfloat16, 1, 1, false, false, false, false>(a, stream, a.nchunks - 1);
  return a.vec ? launch_carry<float, 1, 1, false, true, false, false>(a, stream, a.nchunks - 1)
               : launch_carry<float, 1, 1, false, false, false, false>(a, stream, a.nchunks - 1);
}

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t stream) {
  if (a.bf16) return dispatch<__nv_bfloat16>(a, stream);
  return dispatch<float>(a, stream);
}

cudaError_t scan_bounds_flags(unsigned* out, bool clear) {
#ifdef SSM_DEBUG_BOUNDS
  return bounds_flags_read(out, clear);
#else
  (void)out;
  (void)clear;
  return cudaErrorNotSupported;
#endif
}

}  // namespace ssm
