// ssm_scan_bwd.cu -- backward pass of the selective scan (training), Euler rule, forward time,
// scan input u given directly (no fused conv).
//
// What it computes: the gradients of a scalar loss through
//   Delta_t = softplus(delta_t + bias_d),  h_t[n] = exp(Delta_t A[d,n]) h_{t-1}[n] + Delta_t B[b,n,t] u_t,
//   y_t = sum_n C[b,n,t] h_t[n] + D_d u_t,  out_t = y_t silu(z_t)
// from dout = dL/dout and dh_last = dL/dh_{L-1}. The adjoint g_t[n] = dL/dh_t[n] obeys the
// same recurrence run backward, g_t = exp(Delta_{t+1} A) g_{t+1} + C_t dy_t ("Mamba (Selective
// State-Space Model)", gunjandhanuka.github.io, "Cost of selectivity": training runs through
// the parallel scan), and
//   dy_t = dout_t silu(z_t),  dz_t = dout_t y_t silu'(z_t),  du_t = D dy_t + sum_n g_t Delta_t B_t,
//   dDelta_t = sum_n g_t (A Abar_t h_{t-1} + B_t u_t),  ddelta_t = dDelta_t sigmoid(delta_t + bias),
//   dA += g_t Delta_t Abar_t h_{t-1},  dB_t += g_t Delta_t u_t,  dC_t += dy_t h_t,  dD += dy_t u_t,
//   dh0 = Abar_0 g_0.
// Abar_t h_{t-1} is taken as h_t - Delta_t B_t u_t, so the adjoint needs the states h_t alone.
//
// Design: two passes over the data, then a reduction. Every CTA is one warp; lane c owns
// channel d0 + c of one sequence with its 16 states in registers; time is cut into chunks
// (a multiple of the 8-step tile) when the channels alone leave SMs idle.
//  * Checkpoint pass (scan_bwd_ckpt_kernel), per chunk, forward in time from a zero state.
//    At the start of every 8-step tile it writes the state so far and the sum of Delta' so
//    far (Delta' = Delta log2 e); at the chunk's end the chunk's aggregate (sum of Delta', end
//    state). With several chunks, every chunk after the first also folds its adjoint aggregate
//    on the way: the adjoint that leaves the chunk's start when its end receives zero,
//    sum_t P_t C_t dy_t with P_t = Abar_start ... Abar_t, a running product of the Abar the
//    state update computes anyway.
//  * Reverse pass (scan_bwd_kernel), per chunk, tiles from the chunk's end to its start.
//    The chunk's start state h_in is h0 composed with the aggregates of the chunks before it;
//    the adjoint entering its end is dh_last composed with the adjoint aggregates of the
//    chunks after it. A tile's start state is 2^(A S) h_in + (its checkpoint). A tile is two
//    4-step sub-tiles: a sub-tile's forward states are recomputed into registers, then the
//    adjoint walks back over them. The tile's per-(step, channel) inputs are staged once by
//    cp.async and transposed to fp32 [step][lane] (conflict-free per-step reads); B and C to
//    fp32 [step][32] (broadcast reads). dB_t and dC_t (sums over the CTA's 32 channels) go
//    through a shared-memory transpose: each lane writes its 32 products as a row, then sums
//    one column. Outputs du, ddelta, dz leave as one 16-byte row segment per lane and tile.
//  * Reduction (scan_bwd_reduce_kernel): dB, dC over the channel tiles; dA, dD, dbias over the
//    chunks and sequences; in a fixed order, so results are deterministic.
#include "ssm_bounds.cuh"
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kW = 32;            // channels per CTA: one warp, one channel per lane
constexpr int kTB = 8;            // steps per tile (the checkpoint spacing)
constexpr int kSub = 4;           // steps per sub-tile (forward states kept in registers)
constexpr int kNS = kMaxDstate;   // states per lane
static_assert(kTB == 2 * kSub, "a tile is two sub-tiles");
static_assert(kNS == 16, "16 states per lane");

// Checkpoint of one (CTA, tile): the 32 channels' states at the tile start, from a zero state at
// the chunk start (states 4k .. 4k+3 of lane c at h[k][c]), and the sums of Delta' from the
// chunk start to the tile start.
struct Ckpt {
  float4 h[4][kW];
  float S[kW];
};
static_assert(sizeof(Ckpt) % 16 == 0, "checkpoints move in 16-byte pieces");

// Raw rows of one tile in shared memory: kCh per-channel arrays (32 rows each), then kSt
// per-state arrays (16 rows each); kTB elements per row at a stride of RS elements (16 bytes
// for bf16; 48 for fp32, so that lane c's two 16-byte reads of row c are conflict-free).
template <typename T, int kCh, int kSt>
struct Rows {
  static constexpr int kEPC = 16 / (int)sizeof(T);  // elements per 16-byte piece
  static constexpr int kCPR = kTB / kEPC;           // pieces per row
  static constexpr int RS = sizeof(T) == 2 ? kTB : kTB + 4;
  static constexpr int kRows = kCh * kW + kSt * kNS;
  static constexpr int kBytes = kRows * RS * (int)sizeof(T);
};

// One row of a tile: steps [t0, t0 + kTB) of row `rowbase` of `arr` (zeros past L or when !ok).
template <typename T, int RS, bool VEC>
__device__ __forceinline__ void copy_row(T* dst, const T* arr, long long rowbase, bool ok, long long ext, int t0,
                                         int L, const void* fallback) {
  constexpr int kEPC = 16 / (int)sizeof(T);
  if (VEC) {
#pragma unroll
    for (int j = 0; j < kTB / kEPC; ++j) {
      const int t = t0 + j * kEPC;
      const bool v = ok && t < L && in_bounds(rowbase + t, kEPC, ext, kBoundsBackward);
      cp_async16(dst + j * kEPC, v ? (const void*)(arr + rowbase + t) : fallback, v ? 16u : 0u);
    }
  } else {
#pragma unroll
    for (int s = 0; s < kTB; ++s) {
      const int t = t0 + s;
      dst[s] = (ok && t < L && in_bounds(rowbase + t, 1, ext, kBoundsBackward)) ? arr[rowbase + t] : from_f32<T>(0.f);
    }
  }
}

// Stages steps [t0, t0 + kTB) of channel arrays c0..c3 (lane c copies its own channel d0 + c of
// sequence b in each) and state arrays s0, s1 (lanes 0..15 rows n of s0, lanes 16..31 of s1)
// into `ring`; zeros past L, dim, N or for a NULL array. VEC: 16-byte cp.async pieces (the
// caller commits the group); else plain loads.
template <typename T, int kCh, int kSt, bool VEC>
__device__ __forceinline__ void stage_tile(T* ring, const ScanBwdArgs& a, const T* c0, const T* c1, const T* c2,
                                           const T* c3, const T* s0, const T* s1, int b, int d0, int t0, int lane) {
  using R = Rows<T, kCh, kSt>;
  const int L = a.seqlen, N = a.dstate, dim = a.dim;
  const long long tok = (long long)a.batch * dim * L, bcx = (long long)a.batch * N * L;
  const long long crow = ((long long)b * dim + d0 + lane) * L;
  const bool cvalid = d0 + lane < dim;
#pragma unroll
  for (int m = 0; m < kCh; ++m) {
    const T* arr = m == 0 ? c0 : (m == 1 ? c1 : (m == 2 ? c2 : c3));  // m is known once unrolled
    copy_row<T, R::RS, VEC>(ring + (m * kW + lane) * R::RS, arr, crow, cvalid && arr != nullptr, tok, t0, L, c0);
  }
  if (lane < kSt * kNS) {
    const int n = lane % kNS;
    const T* sarr = lane < kNS ? s0 : s1;
    copy_row<T, R::RS, VEC>(ring + (kCh * kW + lane) * R::RS, sarr, ((long long)b * N + n) * L,
                            n < N && sarr != nullptr, bcx, t0, L, c0);
  }
}

// The checkpoint record of tile `it`: 136 16-byte pieces.
__device__ __forceinline__ void stage_ckpt(Ckpt* dst, const Ckpt* src, long long rec, long long nrec, int lane) {
  if (!in_bounds(rec, 1, nrec, kBoundsBackward)) return;
  const char* s = reinterpret_cast<const char*>(src + rec);
  char* d = reinterpret_cast<char*>(dst);
#pragma unroll 1
  for (int i = lane; i < (int)(sizeof(Ckpt) / 16); i += kW) cp_async16(d + 16 * i, s + 16 * i, 16u);
}

__device__ __forceinline__ float2 ex2x2(float2 x) { return make_float2(ex2_approx(x.x), ex2_approx(x.y)); }

// ---------------------------------------------------------------- checkpoint pass
// ADJ: also the chunk's adjoint aggregate (needs dout, z and C).
template <typename T, bool VEC, bool ADJ>
__global__ void __launch_bounds__(kW, 16) scan_bwd_ckpt_kernel(const ScanBwdArgs a) {
  constexpr bool PRECISE = IoTraits<T>::kPrecise;
  constexpr int kCh = ADJ ? 4 : 2, kSt = ADJ ? 2 : 1;
  using R = Rows<T, kCh, kSt>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  auto ring = [&](int slot) { return reinterpret_cast<T*>(smem_raw + slot * R::kBytes); };
  float (*const BC)[kW] = reinterpret_cast<float (*)[kW]>(smem_raw + 2 * R::kBytes);

  const int lane = threadIdx.x;
  const int dtile = blockIdx.x, b = blockIdx.y, q = blockIdx.z;
  const int ndt = gridDim.x;
  const int d0 = dtile * kW, d = d0 + lane;
  const int L = a.seqlen, N = a.dstate, dim = a.dim;
  const bool valid = d < dim;
  const long long BD = (long long)a.batch * dim, cc = (long long)b * dim + d;
  const int ntiles = (L + kTB - 1) / kTB;
  const int it_begin = q * (a.chunk_len / kTB);
  const int it_end = min(ntiles, it_begin + a.chunk_len / kTB);
  const T* gu = static_cast<const T*>(a.u);
  const T* gdl = static_cast<const T*>(a.delta);
  const T* gdo = static_cast<const T*>(a.dout);
  const T* gz = static_cast<const T*>(a.z);
  const T* gB = static_cast<const T*>(a.B);
  const T* gC = static_cast<const T*>(a.C);
  Ckpt* const ck = reinterpret_cast<Ckpt*>(a.ws_ck);
  const long long nrec = (long long)a.batch * ndt * ntiles;
  const long long rec0 = ((long long)b * ndt + dtile) * ntiles;

  const bool arow = valid && in_bounds((long long)d * N, N, (long long)dim * N, kBoundsBackward);
  float2 An[kNS / 2];
#pragma unroll
  for (int k = 0; k < kNS / 2; ++k)
    An[k] = make_float2(arow && 2 * k < N ? a.A[(long long)d * N + 2 * k] : 0.f,
                        arow && 2 * k + 1 < N ? a.A[(long long)d * N + 2 * k + 1] : 0.f);
  const float bias = (valid && a.delta_bias) ? a.delta_bias[d] : 0.f;

  // the first chunk's adjoint aggregate is never composed: skip its inputs and arithmetic
  const bool adj = ADJ && q > 0;
  const T* const gdo_s = adj ? gdo : nullptr;
  const T* const gz_s = adj ? gz : nullptr;
  const T* const gC_s = adj ? gC : nullptr;
  float2 h[kNS / 2], g[kNS / 2], P[kNS / 2];
#pragma unroll
  for (int k = 0; k < kNS / 2; ++k) {
    h[k] = g[k] = make_float2(0.f, 0.f);
    P[k] = make_float2(1.f, 1.f);
  }
  float S = 0.f;

  if (it_begin < it_end) {
    stage_tile<T, kCh, kSt, VEC>(ring(0), a, gu, gdl, gdo_s, gz_s, gB, gC_s, b, d0, it_begin * kTB, lane);
    cp_async_commit();
  }
#pragma unroll 1
  for (int it = it_begin; it < it_end; ++it) {
    const int t0 = it * kTB, tl = min(kTB, L - t0);
    // the checkpoint of this tile: the state and the sum of Delta' before it
    if (in_bounds(rec0 + it, 1, nrec, kBoundsBackward)) {
      Ckpt& c = ck[rec0 + it];
#pragma unroll
      for (int k = 0; k < 4; ++k) c.h[k][lane] = make_float4(h[2 * k].x, h[2 * k].y, h[2 * k + 1].x, h[2 * k + 1].y);
      c.S[lane] = S;
    }
    if (it + 1 < it_end)
      stage_tile<T, kCh, kSt, VEC>(ring((it + 1 - it_begin) & 1), a, gu, gdl, gdo_s, gz_s, gB, gC_s, b, d0, t0 + kTB,
                                   lane);
    cp_async_commit();
    cp_async_wait<1>();
    __syncwarp();  // (A) this tile's rows have landed for every lane; every lane is done with BC
    const T* rg = ring((it - it_begin) & 1);
    float x[kTB], du[kTB], dy[kTB];
    {
      float uv[kTB], dv[kTB];
      load8(rg + (0 * kW + lane) * R::RS, uv);
      load8(rg + (1 * kW + lane) * R::RS, dv);
      float dov[kTB], zv[kTB];
      if (ADJ) {
        load8(rg + (2 * kW + lane) * R::RS, dov);
        load8(rg + (3 * kW + lane) * R::RS, zv);
      }
#pragma unroll
      for (int s = 0; s < kTB; ++s) {
        const bool in = valid && s < tl;
        const float v = dv[s] + bias;
        const float Dl = a.delta_softplus ? softplus_f<PRECISE>(v) : v;
        x[s] = in ? Dl * kLog2e : 0.f;
        du[s] = in ? Dl * uv[s] : 0.f;
        if (ADJ) dy[s] = (in && adj) ? (gz ? dov[s] * silu_f(zv[s]) : dov[s]) : 0.f;
      }
      // B (and C) rows, transposed to [step][state] (C at 16 + n)
      if (lane < kSt * kNS) {
        float bv[kTB];
        load8(rg + (kCh * kW + lane) * R::RS, bv);
#pragma unroll
        for (int s = 0; s < kTB; ++s) BC[s][lane] = bv[s];
      }
    }
    __syncwarp();  // (B) BC visible
#pragma unroll
    for (int s = 0; s < kTB; ++s) {
      S += x[s];
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const float4 B4 = *reinterpret_cast<const float4*>(&BC[s][4 * k4]);
        const float2 Bv[2] = {make_float2(B4.x, B4.y), make_float2(B4.z, B4.w)};
        float2 Cv[2];
        if (ADJ) {
          const float4 C4 = *reinterpret_cast<const float4*>(&BC[s][kNS + 4 * k4]);
          Cv[0] = make_float2(C4.x, C4.y);
          Cv[1] = make_float2(C4.z, C4.w);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int k = 2 * k4 + i;
          const float2 e = ex2x2(fmul2(f2(x[s]), An[k]));
          h[k] = ffma2(e, h[k], fmul2(f2(du[s]), Bv[i]));
          if (ADJ) {
            P[k] = fmul2(P[k], e);
            g[k] = ffma2(P[k], fmul2(Cv[i], f2(dy[s])), g[k]);
          }
        }
      }
    }
  }
  cp_async_wait<0>();
  // the chunk's aggregates: [nchunks][batch * dim] sums, [nchunks][batch * dim][16] states
  const long long e = (long long)q * BD + cc;
  if (valid && in_bounds(e, 1, (long long)a.nchunks * BD, kBoundsBackward)) {
    a.fS[e] = S;
    float4* fh = reinterpret_cast<float4*>(a.fh + e * kNS);
    float4* bh = reinterpret_cast<float4*>(a.bh + e * kNS);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      fh[k] = make_float4(h[2 * k].x, h[2 * k].y, h[2 * k + 1].x, h[2 * k + 1].y);
      if (ADJ) bh[k] = make_float4(g[2 * k].x, g[2 * k].y, g[2 * k + 1].x, g[2 * k + 1].y);
    }
  }
}

// ---------------------------------------------------------------- reverse pass

template <typename T>
struct RevSmem {
  using R = Rows<T, 4, 2>;                 // u, delta, dout, z; B, C
  static constexpr int ring = 0;
  static constexpr int ck = ring + R::kBytes;
  static constexpr int arr = ck + (int)sizeof(Ckpt);  // x, u, dy, gz, sg: [5][kTB][kW] fp32
  static constexpr int bc = arr + 5 * kTB * kW * 4;   // [kTB][kW]: B at n, C at 16 + n
  static constexpr int hst = bc + kTB * kW * 4;       // float4 [4][kW]: the tile's start state
  static constexpr int hin = hst + 4 * kW * 16;       // float4 [4][kW]: the chunk's start state
  static constexpr int red = hin + 4 * kW * 16;       // [kW][kRed]: dB / dC products, one row per lane
  static constexpr int kRed = 2 * kNS + 4;
  static constexpr int bytes = red + kW * kRed * 4;
};

template <typename T, bool VEC>
__global__ void __launch_bounds__(kW, 12) scan_bwd_kernel(const ScanBwdArgs a) {
  constexpr bool PRECISE = IoTraits<T>::kPrecise;
  using Lay = RevSmem<T>;
  using R = typename Lay::R;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  T* const ring = reinterpret_cast<T*>(smem_raw + Lay::ring);
  Ckpt& cks = *reinterpret_cast<Ckpt*>(smem_raw + Lay::ck);
  float (*const X)[kW] = reinterpret_cast<float (*)[kW]>(smem_raw + Lay::arr);      // Delta'
  float (*const U)[kW] = X + kTB;      // u; after the adjoint step: du
  float (*const DY)[kW] = X + 2 * kTB; // dL/dy
  float (*const GZ)[kW] = X + 3 * kTB; // dout silu'(z); after the forward step: dz
  float (*const SG)[kW] = X + 4 * kTB; // sigmoid(delta + bias); after the adjoint step: ddelta
  float (*const BC)[kW] = reinterpret_cast<float (*)[kW]>(smem_raw + Lay::bc);
  float4 (*const hst)[kW] = reinterpret_cast<float4 (*)[kW]>(smem_raw + Lay::hst);
  float4 (*const hin)[kW] = reinterpret_cast<float4 (*)[kW]>(smem_raw + Lay::hin);
  float (*const red)[Lay::kRed] = reinterpret_cast<float (*)[Lay::kRed]>(smem_raw + Lay::red);

  const int lane = threadIdx.x;
  const int dtile = blockIdx.x, b = blockIdx.y, q = blockIdx.z;
  const int ndt = gridDim.x, Q = a.nchunks;
  const int d0 = dtile * kW, d = d0 + lane;
  const int L = a.seqlen, N = a.dstate, dim = a.dim;
  const bool valid = d < dim;
  const long long BD = (long long)a.batch * dim, cc = (long long)b * dim + d;
  const int ntiles = (L + kTB - 1) / kTB;
  const int it_begin = q * (a.chunk_len / kTB);
  const int it_end = min(ntiles, it_begin + a.chunk_len / kTB);
  const bool has_z = a.z != nullptr;
  const T* gu = static_cast<const T*>(a.u);
  const T* gdl = static_cast<const T*>(a.delta);
  const T* gdo = static_cast<const T*>(a.dout);
  const T* gz = static_cast<const T*>(a.z);
  const T* gB = static_cast<const T*>(a.B);
  const T* gC = static_cast<const T*>(a.C);
  const Ckpt* const ck = reinterpret_cast<const Ckpt*>(a.ws_ck);
  const long long nrec = (long long)a.batch * ndt * ntiles;
  const long long rec0 = ((long long)b * ndt + dtile) * ntiles;
  const long long tok = BD * L;
  const long long nagg = (long long)Q * BD;

  // prefetch the last tile of the chunk while the carries are composed
  if (it_begin < it_end) {
    stage_tile<T, 4, 2, VEC>(ring, a, gu, gdl, gdo, gz, gB, gC, b, d0, (it_end - 1) * kTB, lane);
    stage_ckpt(&cks, ck, rec0 + it_end - 1, nrec, lane);
  }
  cp_async_commit();

  const bool arow = valid && in_bounds((long long)d * N, N, (long long)dim * N, kBoundsBackward);
  const bool srow = valid && in_bounds(cc * N, N, BD * N, kBoundsBackward);
  float2 An[kNS / 2];
#pragma unroll
  for (int k = 0; k < kNS / 2; ++k)
    An[k] = make_float2(arow && 2 * k < N ? a.A[(long long)d * N + 2 * k] : 0.f,
                        arow && 2 * k + 1 < N ? a.A[(long long)d * N + 2 * k + 1] : 0.f);
  const float bias = (valid && a.delta_bias) ? a.delta_bias[d] : 0.f;
  const float Dd = (valid && a.D) ? a.D[d] : 0.f;

  // ---- the chunk's start state: h0 composed with the aggregates of chunks 0 .. q-1
  const bool need_hin = q > 0 || a.h0 != nullptr;
  if (need_hin) {
    float2 h[kNS / 2];
#pragma unroll
    for (int k = 0; k < kNS / 2; ++k)
      h[k] = make_float2(srow && a.h0 && 2 * k < N ? a.h0[cc * N + 2 * k] : 0.f,
                         srow && a.h0 && 2 * k + 1 < N ? a.h0[cc * N + 2 * k + 1] : 0.f);
#pragma unroll 1
    for (int j = 0; j < q; ++j) {
      const long long e = (long long)j * BD + cc;
      if (!valid || !in_bounds(e, 1, nagg, kBoundsBackward)) break;
      const float Sj = a.fS[e];
      const float4* hp = reinterpret_cast<const float4*>(a.fh + e * kNS);
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const float4 v = hp[k4];
        h[2 * k4] = ffma2(ex2x2(fmul2(f2(Sj), An[2 * k4])), h[2 * k4], make_float2(v.x, v.y));
        h[2 * k4 + 1] = ffma2(ex2x2(fmul2(f2(Sj), An[2 * k4 + 1])), h[2 * k4 + 1], make_float2(v.z, v.w));
      }
    }
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4)
      hin[k4][lane] = make_float4(h[2 * k4].x, h[2 * k4].y, h[2 * k4 + 1].x, h[2 * k4 + 1].y);
  }
  // ---- the adjoint entering the chunk's end: dh_last composed with chunks nchunks-1 .. q+1
  float2 gad[kNS / 2];
#pragma unroll
  for (int k = 0; k < kNS / 2; ++k)
    gad[k] = make_float2(srow && a.dh_last && 2 * k < N ? a.dh_last[cc * N + 2 * k] : 0.f,
                         srow && a.dh_last && 2 * k + 1 < N ? a.dh_last[cc * N + 2 * k + 1] : 0.f);
#pragma unroll 1
  for (int j = Q - 1; j > q; --j) {
    const long long e = (long long)j * BD + cc;
    if (!valid || !in_bounds(e, 1, nagg, kBoundsBackward)) break;
    const float Sj = a.fS[e];
    const float4* gp = reinterpret_cast<const float4*>(a.bh + e * kNS);
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
      const float4 v = gp[k4];
      gad[2 * k4] = ffma2(ex2x2(fmul2(f2(Sj), An[2 * k4])), gad[2 * k4], make_float2(v.x, v.y));
      gad[2 * k4 + 1] = ffma2(ex2x2(fmul2(f2(Sj), An[2 * k4 + 1])), gad[2 * k4 + 1], make_float2(v.z, v.w));
    }
  }

  float2 dA[kNS / 2];
#pragma unroll
  for (int k = 0; k < kNS / 2; ++k) dA[k] = make_float2(0.f, 0.f);
  float dD_acc = 0.f, dbias_acc = 0.f;
  float* const dbc = a.ws_dBC + ((long long)b * ndt + dtile) * (long long)L * (2 * kNS);

  // one forward step of the recomputation: h <- 2^(Delta' A) h + Delta u B; with Y, also
  // y_t = C.h_t + D u_t and dz_t = y_t dout_t silu'(z_t) (into GZ)
  auto fwd_step = [&](int s, float2 (&h)[kNS / 2], bool Y) {
    const float xv = X[s][lane], uv = U[s][lane];
    const float duv = xv * kLn2 * uv;
    float2 y2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
      const float4 B4 = *reinterpret_cast<const float4*>(&BC[s][4 * k4]);
      const float2 Bv[2] = {make_float2(B4.x, B4.y), make_float2(B4.z, B4.w)};
      float2 Cv[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      if (Y) {
        const float4 C4 = *reinterpret_cast<const float4*>(&BC[s][kNS + 4 * k4]);
        Cv[0] = make_float2(C4.x, C4.y);
        Cv[1] = make_float2(C4.z, C4.w);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int k = 2 * k4 + i;
        h[k] = ffma2(ex2x2(fmul2(f2(xv), An[k])), h[k], fmul2(f2(duv), Bv[i]));
        if (Y) y2 = ffma2(Cv[i], h[k], y2);
      }
    }
    if (Y && has_z) GZ[s][lane] = fmaf(Dd, uv, y2.x + y2.y) * GZ[s][lane];
  };

  // one adjoint step over the state hs = h_t: gradients of step t, then the adjoint moves to t-1
  auto adj_step = [&](int s, int t, const float2 (&hs)[kNS / 2]) {
    const float xv = X[s][lane], uv = U[s][lane], dyv = DY[s][lane], sgv = SG[s][lane];
    const float Dl = xv * kLn2, duv = Dl * uv;
    float2 sgb = make_float2(0.f, 0.f), sat = make_float2(0.f, 0.f);
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
      const float4 B4 = *reinterpret_cast<const float4*>(&BC[s][4 * k4]);
      const float4 C4 = *reinterpret_cast<const float4*>(&BC[s][kNS + 4 * k4]);
      const float2 Bv[2] = {make_float2(B4.x, B4.y), make_float2(B4.z, B4.w)};
      const float2 Cv[2] = {make_float2(C4.x, C4.y), make_float2(C4.z, C4.w)};
      float2 pb[2], pc[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int k = 2 * k4 + i;
        const float2 gt = ffma2(Cv[i], f2(dyv), gad[k]);          // g_t = g + C_t dy_t
        const float2 m = ffma2(f2(-duv), Bv[i], hs[k]);            // Abar_t h_{t-1} = h_t - Delta u B
        const float2 tm = fmul2(gt, m);
        sat = ffma2(An[k], tm, sat);
        dA[k] = ffma2(f2(Dl), tm, dA[k]);
        sgb = ffma2(gt, Bv[i], sgb);
        pb[i] = fmul2(gt, f2(duv));                               // dB_t term g_t Delta u
        pc[i] = fmul2(hs[k], f2(dyv));                            // dC_t term dy h_t
        gad[k] = fmul2(ex2x2(fmul2(f2(xv), An[k])), gt);          // g <- Abar_t g_t
      }
      *reinterpret_cast<float4*>(&red[lane][4 * k4]) = make_float4(pb[0].x, pb[0].y, pb[1].x, pb[1].y);
      *reinterpret_cast<float4*>(&red[lane][kNS + 4 * k4]) = make_float4(pc[0].x, pc[0].y, pc[1].x, pc[1].y);
    }
    const float sgbs = sgb.x + sgb.y;
    const float ddv = fmaf(uv, sgbs, sat.x + sat.y) * sgv;
    U[s][lane] = fmaf(Dd, dyv, Dl * sgbs);  // du
    SG[s][lane] = ddv;                      // ddelta
    dD_acc = fmaf(dyv, uv, dD_acc);
    dbias_acc += ddv;
    __syncwarp();  // (R1) every lane's products are in its row
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
    for (int c = 0; c < kW; c += 4) {
      s0 += red[c][lane];
      s1 += red[c + 1][lane];
      s2 += red[c + 2][lane];
      s3 += red[c + 3][lane];
    }
    if (t < L && in_bounds((long long)t * (2 * kNS) + lane, 1, (long long)L * (2 * kNS), kBoundsBackward))
      dbc[(long long)t * (2 * kNS) + lane] = (s0 + s1) + (s2 + s3);
    __syncwarp();  // (R2) every column is read before the next step's rows
  };

#pragma unroll 1
  for (int it = it_end - 1; it >= it_begin; --it) {
    const int t0 = it * kTB, tl = min(kTB, L - t0);
    cp_async_wait<0>();
    __syncwarp();  // (A) this tile's rows and checkpoint have landed; every lane is done with BC
    // ---- per-(step, channel) values of lane's channel, [step][lane] in fp32
    {
      float uv[kTB], dv[kTB], dov[kTB], zv[kTB];
      load8(ring + (0 * kW + lane) * R::RS, uv);
      load8(ring + (1 * kW + lane) * R::RS, dv);
      load8(ring + (2 * kW + lane) * R::RS, dov);
      load8(ring + (3 * kW + lane) * R::RS, zv);
#pragma unroll
      for (int s = 0; s < kTB; ++s) {
        const bool in = valid && s < tl;
        const float v = dv[s] + bias;
        float Dl = v, sg = 1.f;
        if (a.delta_softplus) {
          Dl = softplus_f<PRECISE>(v);
          sg = rcp_approx(1.0f + ex2_approx(-v * kLog2e));
        }
        float dy = dov[s], gzv = 0.f;
        if (has_z) {
          const float sz = rcp_approx(1.0f + ex2_approx(-zv[s] * kLog2e));
          dy = dov[s] * zv[s] * sz;
          gzv = dov[s] * sz * (1.0f + zv[s] * (1.0f - sz));
        }
        X[s][lane] = in ? Dl * kLog2e : 0.f;
        U[s][lane] = in ? uv[s] : 0.f;
        DY[s][lane] = in ? dy : 0.f;
        GZ[s][lane] = in ? gzv : 0.f;
        SG[s][lane] = in ? sg : 0.f;
      }
      float bv[kTB];
      load8(ring + (4 * kW + lane) * R::RS, bv);
#pragma unroll
      for (int s = 0; s < kTB; ++s) BC[s][lane] = bv[s];
      // the tile's start state: 2^(A S) h_in + the checkpoint from zero
      const float Sck = cks.S[lane];
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        float4 v = cks.h[k4][lane];
        if (need_hin) {
          const float4 hi = hin[k4][lane];
          const float2 e0 = ex2x2(fmul2(f2(Sck), An[2 * k4])), e1 = ex2x2(fmul2(f2(Sck), An[2 * k4 + 1]));
          v = make_float4(fmaf(e0.x, hi.x, v.x), fmaf(e0.y, hi.y, v.y), fmaf(e1.x, hi.z, v.z), fmaf(e1.y, hi.w, v.w));
        }
        hst[k4][lane] = v;
      }
    }
    __syncwarp();  // (B) BC visible; the ring and the checkpoint slot are free
    if (it > it_begin) {
      stage_tile<T, 4, 2, VEC>(ring, a, gu, gdl, gdo, gz, gB, gC, b, d0, t0 - kTB, lane);
      stage_ckpt(&cks, ck, rec0 + it - 1, nrec, lane);
    }
    cp_async_commit();

    // ---- sub-tile 1 (steps 4..7) from the state after step 3, then sub-tile 0 from the tile start
#pragma unroll 1
    for (int half = 1; half >= 0; --half) {
      const int s0 = half * kSub;
      float2 hist[kSub][kNS / 2];
      float2 h[kNS / 2];
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const float4 v = hst[k4][lane];
        h[2 * k4] = make_float2(v.x, v.y);
        h[2 * k4 + 1] = make_float2(v.z, v.w);
      }
      if (half == 1) {
#pragma unroll
        for (int s = 0; s < kSub; ++s) fwd_step(s, h, false);
      }
#pragma unroll
      for (int j = 0; j < kSub; ++j) {
        fwd_step(s0 + j, h, true);
#pragma unroll
        for (int k = 0; k < kNS / 2; ++k) hist[j][k] = h[k];
      }
#pragma unroll
      for (int j = kSub - 1; j >= 0; --j) adj_step(s0 + j, t0 + s0 + j, hist[j]);
    }

    // ---- du, ddelta, dz of the tile: one row segment per lane
    if (valid) {
      float o[3][kTB];
#pragma unroll
      for (int s = 0; s < kTB; ++s) {
        o[0][s] = U[s][lane];
        o[1][s] = SG[s][lane];
        o[2][s] = GZ[s][lane];
      }
      T* const dst[3] = {static_cast<T*>(a.du), static_cast<T*>(a.ddelta), static_cast<T*>(a.dz)};
      const long long base = cc * L + t0;
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        if (k == 2 && !has_z) continue;
        if (VEC && tl == kTB) {
          if (in_bounds(base, kTB, tok, kBoundsBackward)) store8(dst[k] + base, o[k]);
        } else if (VEC && tl == 4) {
          const float o4[4] = {o[k][0], o[k][1], o[k][2], o[k][3]};
          if (in_bounds(base, 4, tok, kBoundsBackward)) store4(dst[k] + base, o4);
        } else {
#pragma unroll
          for (int s = 0; s < kTB; ++s)
            if (s < tl && in_bounds(base + s, 1, tok, kBoundsBackward)) dst[k][base + s] = from_f32<T>(o[k][s]);
        }
      }
    }
  }
  cp_async_wait<0>();

  // ---- per-channel results of the chunk
  if (valid) {
    if (q == 0 && a.dh0 && srow) {
#pragma unroll
      for (int k = 0; k < kNS / 2; ++k) {
        if (2 * k < N) a.dh0[cc * N + 2 * k] = gad[k].x;
        if (2 * k + 1 < N) a.dh0[cc * N + 2 * k + 1] = gad[k].y;
      }
    }
    const long long e = (long long)q * BD + cc;
    if (in_bounds(e, 1, nagg, kBoundsBackward)) {
      float4* dap = reinterpret_cast<float4*>(a.ws_dA + e * kNS);
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4)
        dap[k4] = make_float4(dA[2 * k4].x, dA[2 * k4].y, dA[2 * k4 + 1].x, dA[2 * k4 + 1].y);
      a.ws_dD[e] = dD_acc;
      a.ws_dbias[e] = dbias_acc;
    }
  }
}

// ---------------------------------------------------------------- reduction
// Blocks [0, nbc): dB, dC [b, n, t] for 8 steps of one sequence (one warp per step, lane v for
// sum v of the step's 32), summed over the channel tiles in order, 8 tiles' loads in flight at
// a time; written through shared memory as 8-step row pieces. The other blocks: dA [d, n],
// dD [d], ddelta_bias [d], summed over chunks and sequences in order, one thread per output.
constexpr int kRedThreads = 256;
constexpr int kRedSteps = kRedThreads / 32;

__device__ __forceinline__ float sum_strided(const float* src, long long stride, int n) {
  float acc = 0.f;
  int i = 0;
  for (; i + 8 <= n; i += 8) {
    float r[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) r[j] = src[(i + j) * stride];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc += r[j];
  }
  for (; i < n; ++i) acc += src[i * stride];
  return acc;
}

__global__ void __launch_bounds__(kRedThreads) scan_bwd_reduce_kernel(const ScanBwdArgs a, int ndt, int nbc) {
  __shared__ float tile[kRedSteps][33];
  const int L = a.seqlen, N = a.dstate;
  if ((int)blockIdx.x < nbc) {
    const int tblocks = (L + kRedSteps - 1) / kRedSteps;
    const int b = blockIdx.x / tblocks, tb = blockIdx.x % tblocks;
    const int w = threadIdx.x / 32, v = threadIdx.x % 32;
    const int t = tb * kRedSteps + w;
    const long long stride = (long long)L * (2 * kNS);
    const long long first = ((long long)b * ndt * L + t) * (2 * kNS) + v;
    const long long nws = (long long)a.batch * ndt * stride;
    float acc = 0.f;
    if (t < L && in_bounds(first, 1, nws, kBoundsBackward) &&
        in_bounds(first + (ndt - 1) * stride, 1, nws, kBoundsBackward))
      acc = sum_strided(a.ws_dBC + first, stride, ndt);
    tile[w][v] = acc;
    __syncthreads();
    {
      const int vv = threadIdx.x / kRedSteps, tt = threadIdx.x % kRedSteps, t2 = tb * kRedSteps + tt;
      const int n = vv % kNS;
      if (t2 < L && n < N) (vv < kNS ? a.dB : a.dC)[((long long)b * N + n) * L + t2] = tile[tt][vv];
    }
    return;
  }
  const long long nA = (long long)a.dim * N;
  const long long total = nA + 2LL * a.dim;
  const int QB = a.nchunks * a.batch;
  for (long long i = (blockIdx.x - nbc) * (long long)kRedThreads + threadIdx.x; i < total;
       i += (long long)(gridDim.x - nbc) * kRedThreads) {
    if (i < nA) {
      const long long dd = i / N, n = i % N;
      a.dA[i] = sum_strided(a.ws_dA + dd * kNS + n, (long long)a.dim * kNS, QB);
    } else {
      const long long j = i - nA;
      const bool isBias = j >= a.dim;
      const long long dd = isBias ? j - a.dim : j;
      float* dst = isBias ? a.ddelta_bias : a.dD;
      if (dst) dst[dd] = sum_strided((isBias ? a.ws_dbias : a.ws_dD) + dd, a.dim, QB);
    }
  }
}

// ---------------------------------------------------------------- launch

template <typename K>
cudaError_t set_smem(K kernel, int bytes, int (&configured)[64]) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 0 && dev < 64 && configured[dev]) return cudaSuccess;
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err == cudaSuccess && dev >= 0 && dev < 64) configured[dev] = 1;
  return err;
}

template <typename T, bool VEC, bool ADJ>
cudaError_t launch_ckpt(const ScanBwdArgs& a, dim3 grid, cudaStream_t stream) {
  static int configured[64] = {0};
  using R = Rows<T, ADJ ? 4 : 2, ADJ ? 2 : 1>;
  const int smem = 2 * R::kBytes + kTB * kW * 4;
  cudaError_t err = set_smem(scan_bwd_ckpt_kernel<T, VEC, ADJ>, smem, configured);
  if (err != cudaSuccess) return err;
  scan_bwd_ckpt_kernel<T, VEC, ADJ><<<grid, kW, smem, stream>>>(a);
  return cudaGetLastError();
}

template <typename T, bool VEC>
cudaError_t prepare_rev() {
  static int configured[64] = {0};
  return set_smem(scan_bwd_kernel<T, VEC>, RevSmem<T>::bytes, configured);
}

template <typename T, bool VEC>
cudaError_t launch_bwd_t(const ScanBwdArgs& a, cudaStream_t stream) {
  const int ndt = (a.dim + kW - 1) / kW;
  const dim3 grid(ndt, a.batch, a.nchunks);
  cudaError_t err = a.nchunks > 1 ? launch_ckpt<T, VEC, true>(a, grid, stream) : launch_ckpt<T, VEC, false>(a, grid, stream);
  if (err != cudaSuccess) return err;
  err = prepare_rev<T, VEC>();
  if (err != cudaSuccess) return err;
  scan_bwd_kernel<T, VEC><<<grid, kW, RevSmem<T>::bytes, stream>>>(a);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const long long nbc = (long long)a.batch * ((a.seqlen + kRedSteps - 1) / kRedSteps);
  long long np = ((long long)a.dim * (a.dstate + 2) + kRedThreads - 1) / kRedThreads;
  if (np > 148 * 4) np = 148 * 4;
  if (np < 1) np = 1;
  scan_bwd_reduce_kernel<<<(unsigned)(nbc + np), kRedThreads, 0, stream>>>(a, ndt, (int)nbc);
  return cudaGetLastError();
}

template <typename T>
int rev_resident() {
  int n = 0;
  if (prepare_rev<T, true>() != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, scan_bwd_kernel<T, true>, kW, RevSmem<T>::bytes) !=
          cudaSuccess ||
      n <= 0) {
    cudaGetLastError();
    return sizeof(T) == 2 ? 11 : 9;  // no device to ask: what registers and shared memory allow
  }
  return n;
}

size_t up256(long long v) { return (size_t)((v + 255) & ~255LL); }

}  // namespace

int scan_bwd_resident_ctas_per_sm(bool bf16) { return bf16 ? rev_resident<__nv_bfloat16>() : rev_resident<float>(); }

int scan_bwd_channels_per_cta() { return kW; }

int scan_bwd_tile_steps() { return kTB; }

size_t scan_bwd_workspace_bytes(int batch, int dim, int seqlen, int nchunks) {
  const long long ndt = (dim + kW - 1) / kW;
  const long long ntiles = (seqlen + kTB - 1) / kTB;
  const long long BD = (long long)batch * dim;
  const long long Q = nchunks < 1 ? 1 : nchunks;
  size_t s = up256(batch * ndt * ntiles * (long long)sizeof(Ckpt));  // checkpoints
  s += up256(Q * BD * 4LL) + 2 * up256(Q * BD * kNS * 4LL);         // chunk aggregates fS, fh, bh
  s += up256(batch * ndt * (long long)seqlen * 2 * kNS * 4LL);      // dB, dC per channel tile
  s += up256(Q * BD * kNS * 4LL) + 2 * up256(Q * BD * 4LL);         // dA, dD, dbias per chunk
  return s;
}

void scan_bwd_workspace_split(void* ws, int batch, int dim, int seqlen, int nchunks, ScanBwdArgs& a) {
  const long long ndt = (dim + kW - 1) / kW;
  const long long ntiles = (seqlen + kTB - 1) / kTB;
  const long long BD = (long long)batch * dim;
  const long long Q = nchunks < 1 ? 1 : nchunks;
  char* p = static_cast<char*>(ws);
  auto take = [&](size_t bytes) { char* r = p; p += bytes; return reinterpret_cast<float*>(r); };
  a.ws_ck = take(up256(batch * ndt * ntiles * (long long)sizeof(Ckpt)));
  a.fS = take(up256(Q * BD * 4LL));
  a.fh = take(up256(Q * BD * kNS * 4LL));
  a.bh = take(up256(Q * BD * kNS * 4LL));
  a.ws_dBC = take(up256(batch * ndt * (long long)seqlen * 2 * kNS * 4LL));
  a.ws_dA = take(up256(Q * BD * kNS * 4LL));
  a.ws_dD = take(up256(Q * BD * 4LL));
  a.ws_dbias = take(up256(Q * BD * 4LL));
}

cudaError_t launch_scan_bwd(const ScanBwdArgs& a, cudaStream_t stream) {
  if (a.bf16) return a.vec ? launch_bwd_t<__nv_bfloat16, true>(a, stream) : launch_bwd_t<__nv_bfloat16, false>(a, stream);
  return a.vec ? launch_bwd_t<float, true>(a, stream) : launch_bwd_t<float, false>(a, stream);
}

cudaError_t scan_bwd_bounds_flags(unsigned* out, bool clear) {
#ifdef SSM_DEBUG_BOUNDS
  return bounds_flags_read(out, clear);
#else
  (void)out;
  (void)clear;
  return cudaErrorNotSupported;
#endif
}

}  // namespace ssm
