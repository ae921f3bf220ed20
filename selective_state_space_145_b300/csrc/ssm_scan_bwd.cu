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
//
// Design. One CTA = 32 channels of one sequence, the whole sequence, 128 threads; thread
// (c, g) holds states 4g .. 4g+3 of channel c, as in the forward kernel.
//  * Checkpoint pass: the forward recurrence (no readout) over the sequence, writing the state
//    before every 16-step tile to the workspace. Each tile's global loads are issued into
//    registers one tile ahead, so they complete while the previous tile computes.
//  * Reverse pass, tile by tile from the end: stage the tile's u, delta, z, dout rows and B, C;
//    recompute h_t of the tile's steps from its checkpoint into shared memory, with the
//    readout partials that give y_t; then dy, dz; the channel sums of dC_t over the CTA's 32
//    channels; the adjoint walk (backward over the tile, four states per thread in registers),
//    which leaves g_t in the slot of h_t; the channel sums of dB_t; and du, ddelta.
//  * dA, dD and dbias accumulate per channel in registers. dB, dC, dA, dD, dbias are written as
//    per-CTA partials and summed over channel tiles / sequences by a second kernel in a fixed
//    order (deterministic, no atomics).
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kBThreads = 128;
constexpr int kBDT = 32;        // channels per CTA
constexpr int kBT = 16;         // steps per tile
constexpr int kBTP = kBT + 1;   // padded row of the per-(channel, step) arrays
static_assert(kBThreads == kBDT * 4, "four threads per channel");
constexpr int kOut = kBT * kMaxDstate / kBThreads;  // (step, state) channel sums per thread
static_assert(kOut == 2, "channel sums: two states (one 8-byte load) per thread");

struct BwdSmem {
  float4 hist[kBT][kBThreads];        // h_t of the tile, then the adjoint g_t
  float Bt[kBT][kMaxDstate];          // B, C of the tile, fp32, t-major
  float Ct[kBT][kMaxDstate];
  float dl[kBDT][kBTP];               // Delta' = Delta log2(e)
  float Dl[kBDT][kBTP];               // Delta
  float uu[kBDT][kBTP];               // u
  float du[kBDT][kBTP];               // Delta u
  float sg[kBDT][kBTP];               // dDelta / d(delta)
  float dy[kBDT][kBTP];               // dL/dy
  float dout[kBDT][kBTP];
  float zz[kBDT][kBTP];
  float p0[4][kBDT][kBTP];            // per-state-group partials: readout, then du
  float p1[4][kBDT][kBTP];            // per-state-group partials of dDelta
};

// ADJ: the adjoint carry of one chunk (chunks 1 .. nchunks-1): the adjoint walked backward over
// the chunk from zero with its own dy_t C_t inputs, and the chunk's sum of Delta', so that every
// chunk can start from the composed adjoint of the chunks after it.
template <typename T, bool ADJ>
__global__ void __launch_bounds__(kBThreads, 3) scan_bwd_kernel(const ScanBwdArgs a) {
  constexpr bool PRECISE = IoTraits<T>::kPrecise;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  BwdSmem& S = *reinterpret_cast<BwdSmem*>(smem_raw);
  const int tid = threadIdx.x;
  const int c = tid % kBDT, g = tid / kBDT;
  const int dtile = blockIdx.x, b = blockIdx.y;
  const int d0 = dtile * kBDT, d = d0 + c;
  const int L = a.seqlen, N = a.dstate, dim = a.dim;
  const bool valid = d < dim;
  const long long cc = (long long)b * dim + d;
  const int ntiles = (L + kBT - 1) / kBT;
  const int Q = a.nchunks;
  const int q = ADJ ? blockIdx.z + 1 : blockIdx.z;   // chunk; chunk boundaries are tile boundaries
  const int it_begin = q * (a.chunk_len / kBT);
  const int it_end = min(ntiles, it_begin + a.chunk_len / kBT);
  const long long BD = (long long)a.batch * dim;
  const long long cta = (long long)b * gridDim.x + dtile;
  float4* ckpt = reinterpret_cast<float4*>(a.ws_ckpt) + cta * (long long)ntiles * kBThreads;

  const T* gu = static_cast<const T*>(a.u);
  const T* gdel = static_cast<const T*>(a.delta);
  const T* gz = static_cast<const T*>(a.z);
  const T* gdo = static_cast<const T*>(a.dout);
  const T* gB = static_cast<const T*>(a.B);
  const T* gC = static_cast<const T*>(a.C);

  const float Dd = (valid && a.D) ? a.D[d] : 0.f;
  float An[4];  // A of this thread's states (Delta is staged in log2 units)
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int n = 4 * g + k;
    An[k] = (valid && n < N) ? a.A[(long long)d * N + n] : 0.f;
  }

  // ---- staging of tile `it`, in two halves: fetch() issues the global loads into registers
  // (so the next tile's loads are in flight while this tile computes); put() derives Delta,
  // its softplus derivative and Delta u and stores everything to shared memory (zeros past
  // L / dim / N: identity steps with Delta = 0 and u = 0).
  constexpr int kPE = kBDT * kBT / kBThreads;           // per-(channel, step) elements per thread
  constexpr int kPB = kBT * kMaxDstate / kBThreads;     // B / C elements per thread
  struct Fetched {
    float u[kPE], dv[kPE], z[kPE], dout[kPE], B[kPB], C[kPB];
  };
  auto fetch = [&](int it, bool need_all, Fetched& f) {
    const int t0 = it * kBT;
#pragma unroll
    for (int k = 0; k < kPE; ++k) {
      const int e = tid + k * kBThreads;
      const int ch = e / kBT, s = e % kBT, t = t0 + s;
      const bool in = d0 + ch < dim && t < L;
      const long long idx = ((long long)b * dim + d0 + ch) * L + t;
      f.u[k] = in ? to_f32(gu[idx]) : 0.f;
      f.dv[k] = in ? to_f32(gdel[idx]) : 0.f;
      f.z[k] = (in && need_all && gz) ? to_f32(gz[idx]) : 0.f;
      f.dout[k] = (in && need_all) ? to_f32(gdo[idx]) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kPB; ++k) {
      const int e = tid + k * kBThreads;
      const int n = e / kBT, s = e % kBT, t = t0 + s;
      const bool in = n < N && t < L;
      const long long idx = ((long long)b * N + n) * L + t;
      f.B[k] = in ? to_f32(gB[idx]) : 0.f;
      f.C[k] = (in && need_all) ? to_f32(gC[idx]) : 0.f;
    }
  };
  auto put = [&](int it, const Fetched& f) {
    const int t0 = it * kBT;
#pragma unroll
    for (int k = 0; k < kPE; ++k) {
      const int e = tid + k * kBThreads;
      const int ch = e / kBT, s = e % kBT, t = t0 + s;
      const bool in = d0 + ch < dim && t < L;
      float D = 0.f, sgv = 0.f;
      if (in) {
        const float v = f.dv[k] + ((a.delta_bias) ? a.delta_bias[d0 + ch] : 0.f);
        if (a.delta_softplus) {
          D = softplus_f<PRECISE>(v);
          sgv = rcp_approx(1.0f + ex2_approx(-v * kLog2e));
        } else {
          D = v;
          sgv = 1.0f;
        }
      }
      S.Dl[ch][s] = D;
      S.dl[ch][s] = D * kLog2e;
      S.uu[ch][s] = f.u[k];
      S.du[ch][s] = D * f.u[k];
      S.sg[ch][s] = sgv;
      S.zz[ch][s] = f.z[k];
      S.dout[ch][s] = f.dout[k];
    }
#pragma unroll
    for (int k = 0; k < kPB; ++k) {
      const int e = tid + k * kBThreads;
      const int n = e / kBT, s = e % kBT;
      S.Bt[s][n] = f.B[k];
      S.Ct[s][n] = f.C[k];
    }
  };
  Fetched fb;

  // ---- checkpoint pass: the state before every tile of the chunk, from the chunk's start
  // state h0 o carry_0 o ... o carry_{q-1} (forward carries: a = 2^(A sum Delta'), b = end state)
  float h[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) h[k] = (valid && a.h0 && 4 * g + k < N) ? a.h0[cc * N + 4 * g + k] : 0.f;
  if (!ADJ && valid) {
    for (int j = 0; j < q; ++j) {
      const float Sj = a.fS[(long long)j * BD + cc];
      const float4 hb = *reinterpret_cast<const float4*>(a.fh + ((long long)j * BD + cc) * kMaxDstate + 4 * g);
      const float hbv[4] = {hb.x, hb.y, hb.z, hb.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) h[k] = fmaf(ex2_approx(Sj * An[k]), h[k], hbv[k]);
    }
  }
  if (!ADJ && it_begin < it_end) fetch(it_begin, false, fb);
  for (int it = it_begin; it < (ADJ ? it_begin : it_end); ++it) {
    ckpt[(long long)it * kBThreads + tid] = make_float4(h[0], h[1], h[2], h[3]);
    __syncthreads();  // previous tile's smem reads are done
    put(it, fb);
    if (it + 1 < it_end) fetch(it + 1, false, fb);
    __syncthreads();
    for (int s = 0; s < kBT; ++s) {
      const float x = S.dl[c][s], w = S.du[c][s];
      const float4 B4 = *reinterpret_cast<const float4*>(&S.Bt[s][4 * g]);
      const float Bv[4] = {B4.x, B4.y, B4.z, B4.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) h[k] = fmaf(ex2_approx(x * An[k]), h[k], w * Bv[k]);
    }
  }

  // ---- reverse pass. The adjoint entering the chunk's end: dh_last composed with the adjoint
  // carries of chunks nchunks-1 .. q+1 (ADJ: zero)
  float gad[4] = {0.f, 0.f, 0.f, 0.f};
  if (!ADJ) {
#pragma unroll
    for (int k = 0; k < 4; ++k) gad[k] = (valid && a.dh_last && 4 * g + k < N) ? a.dh_last[cc * N + 4 * g + k] : 0.f;
    if (valid) {
      for (int j = Q - 1; j > q; --j) {
        const float Sj = a.bS[(long long)j * BD + cc];
        const float4 gb = *reinterpret_cast<const float4*>(a.bh + ((long long)j * BD + cc) * kMaxDstate + 4 * g);
        const float gbv[4] = {gb.x, gb.y, gb.z, gb.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) gad[k] = fmaf(ex2_approx(Sj * An[k]), gad[k], gbv[k]);
      }
    }
  }
  float dsum = 0.f;  // ADJ: the chunk's sum of Delta (log2 units)
  float dA_acc[4] = {0.f, 0.f, 0.f, 0.f};
  float dD_acc = 0.f, dbias_acc = 0.f;
  // channel sums: thread -> step tid / (16 / kOut), states n0 .. n0 + kOut - 1 of one group
  const int rs = tid / (kMaxDstate / kOut), rn0 = kOut * (tid % (kMaxDstate / kOut));
  const int rg = rn0 / 4, rk = rn0 % 4;
  if (it_begin < it_end) fetch(it_end - 1, true, fb);
  for (int it = it_end - 1; it >= it_begin; --it) {
    const int t0 = it * kBT;
    const int tl = min(kBT, L - t0);
    __syncthreads();  // the previous tile is done with shared memory
    put(it, fb);
    const float4 hs = ADJ ? make_float4(0.f, 0.f, 0.f, 0.f) : ckpt[(long long)it * kBThreads + tid];
    if (it > it_begin) fetch(it - 1, true, fb);
    __syncthreads();
    if (ADJ) {
      // dy only (no y needed), then the adjoint from zero over the tile
      constexpr int kSPT0 = kBT / 4;
      for (int s = kSPT0 * g; s < kSPT0 * g + kSPT0; ++s) {
        const float dov = S.dout[c][s];
        float dyv = dov;
        if (gz) {
          const float zv = S.zz[c][s];
          dyv = dov * zv * rcp_approx(1.0f + ex2_approx(-zv * kLog2e));
        }
        S.dy[c][s] = dyv;
      }
      __syncthreads();
      for (int s = kBT - 1; s >= 0; --s) {
        const float dyv = S.dy[c][s], x = S.dl[c][s];
#pragma unroll
        for (int k = 0; k < 4; ++k) gad[k] = ex2_approx(x * An[k]) * fmaf(S.Ct[s][4 * g + k], dyv, gad[k]);
        dsum += x;
      }
      continue;
    }
    // recompute h_t of the tile, with this group's readout partial
    {
      float hh[4] = {hs.x, hs.y, hs.z, hs.w};
      for (int s = 0; s < kBT; ++s) {
        const float x = S.dl[c][s], w = S.du[c][s];
        const float4 B4 = *reinterpret_cast<const float4*>(&S.Bt[s][4 * g]);
        const float4 C4 = *reinterpret_cast<const float4*>(&S.Ct[s][4 * g]);
        const float Bv[4] = {B4.x, B4.y, B4.z, B4.w}, Cv[4] = {C4.x, C4.y, C4.z, C4.w};
        float p = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          hh[k] = fmaf(ex2_approx(x * An[k]), hh[k], w * Bv[k]);
          p = fmaf(Cv[k], hh[k], p);
        }
        S.hist[s][tid] = make_float4(hh[0], hh[1], hh[2], hh[3]);
        S.p0[g][c][s] = p;
      }
    }
    __syncthreads();
    // y, dy, dz for this thread's steps of channel c
    constexpr int kSPT = kBT / 4;  // steps per thread
    for (int s = kSPT * g; s < kSPT * g + kSPT; ++s) {
      const float y = S.p0[0][c][s] + S.p0[1][c][s] + S.p0[2][c][s] + S.p0[3][c][s] + Dd * S.uu[c][s];
      const float dov = S.dout[c][s];
      float dyv = dov;
      if (gz) {
        const float zv = S.zz[c][s];
        const float sz = rcp_approx(1.0f + ex2_approx(-zv * kLog2e));
        dyv = dov * zv * sz;
        if (valid && s < tl)
          static_cast<T*>(a.dz)[cc * L + t0 + s] = from_f32<T>(dov * y * sz * (1.0f + zv * (1.0f - sz)));
      }
      S.dy[c][s] = dyv;
      dD_acc = fmaf(dyv, S.uu[c][s], dD_acc);
    }
    __syncthreads();
    // dC_t[n] over the CTA's channels (this thread: step rs, states rn0, rn0 + 1)
    {
      float acc0 = 0.f, acc1 = 0.f;
      for (int j = 0; j < kBDT; ++j) {
        const int ch = (j + tid) % kBDT;
        const float2 hv = reinterpret_cast<const float2*>(&S.hist[rs][rg * kBDT + ch])[rk / 2];
        const float dyv = S.dy[ch][rs];
        acc0 = fmaf(dyv, hv.x, acc0);
        acc1 = fmaf(dyv, hv.y, acc1);
      }
      if (rs < tl) {
        float* out = a.ws_dC + (((long long)b * gridDim.x + dtile) * kMaxDstate) * L;
        if (rn0 < N) out[(long long)rn0 * L + t0 + rs] = acc0;
        if (rn0 + 1 < N) out[(long long)(rn0 + 1) * L + t0 + rs] = acc1;
      }
    }
    __syncthreads();  // dC has read every h_t; the adjoint walk overwrites them
    // adjoint walk: steps kBT-1 .. 0 of the tile
    // per state: g_t = g + C dy; with gB = g_t B and t1 = g_t Abar h_{t-1},
    //   du part = Delta sum gB,  dDelta part = sum A t1 + u sum gB,  dA += Delta t1,  g <- Abar g_t
    for (int s = kBT - 1; s >= 0; --s) {
      const float dyv = S.dy[c][s], x = S.dl[c][s], Dl = S.Dl[c][s], uv = S.uu[c][s];
      const float4 hp4 = s > 0 ? S.hist[s - 1][tid] : hs;
      const float4 B4 = *reinterpret_cast<const float4*>(&S.Bt[s][4 * g]);
      const float4 C4 = *reinterpret_cast<const float4*>(&S.Ct[s][4 * g]);
      const float hp[4] = {hp4.x, hp4.y, hp4.z, hp4.w};
      const float Bv[4] = {B4.x, B4.y, B4.z, B4.w}, Cv[4] = {C4.x, C4.y, C4.z, C4.w};
      float sgb = 0.f, sat = 0.f, gt[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float e = ex2_approx(x * An[k]);
        gt[k] = fmaf(Cv[k], dyv, gad[k]);
        sgb = fmaf(gt[k], Bv[k], sgb);
        const float t1 = gt[k] * (e * hp[k]);
        sat = fmaf(An[k], t1, sat);
        dA_acc[k] = fmaf(Dl, t1, dA_acc[k]);
        gad[k] = e * gt[k];
      }
      S.hist[s][tid] = make_float4(gt[0], gt[1], gt[2], gt[3]);
      S.p0[g][c][s] = Dl * sgb;
      S.p1[g][c][s] = fmaf(uv, sgb, sat);
    }
    __syncthreads();
    // dB_t[n] over the CTA's channels from g_t and Delta u
    {
      float acc0 = 0.f, acc1 = 0.f;
      for (int j = 0; j < kBDT; ++j) {
        const int ch = (j + tid) % kBDT;
        const float2 gv = reinterpret_cast<const float2*>(&S.hist[rs][rg * kBDT + ch])[rk / 2];
        const float w = S.du[ch][rs];
        acc0 = fmaf(w, gv.x, acc0);
        acc1 = fmaf(w, gv.y, acc1);
      }
      if (rs < tl) {
        float* out = a.ws_dB + (((long long)b * gridDim.x + dtile) * kMaxDstate) * L;
        if (rn0 < N) out[(long long)rn0 * L + t0 + rs] = acc0;
        if (rn0 + 1 < N) out[(long long)(rn0 + 1) * L + t0 + rs] = acc1;
      }
    }
    // du, ddelta for this thread's steps of channel c
    for (int s = kSPT * g; s < kSPT * g + kSPT; ++s) {
      if (!valid || s >= tl) continue;
      const float duv = Dd * S.dy[c][s] + S.p0[0][c][s] + S.p0[1][c][s] + S.p0[2][c][s] + S.p0[3][c][s];
      const float dD = (S.p1[0][c][s] + S.p1[1][c][s] + S.p1[2][c][s] + S.p1[3][c][s]) * S.sg[c][s];
      static_cast<T*>(a.du)[cc * L + t0 + s] = from_f32<T>(duv);
      static_cast<T*>(a.ddelta)[cc * L + t0 + s] = from_f32<T>(dD);
      dbias_acc += dD;
    }
  }

  // ---- per-channel results
  if (ADJ) {
    if (valid) {
      *reinterpret_cast<float4*>(a.bh + ((long long)q * BD + cc) * kMaxDstate + 4 * g) =
          make_float4(gad[0], gad[1], gad[2], gad[3]);
      if (g == 0) a.bS[(long long)q * BD + cc] = dsum;
    }
    return;
  }
  if (valid) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int n = 4 * g + k;
      if (n < N) {
        if (a.dh0 && q == 0) a.dh0[cc * N + n] = gad[k];
        a.ws_dA[((long long)q * BD + cc) * N + n] = dA_acc[k];
      }
    }
  }
  // dD and dbias: the four threads of a channel each hold a quarter of every tile's steps
  __syncthreads();
  S.p0[g][c][0] = dD_acc;
  S.p1[g][c][0] = dbias_acc;
  __syncthreads();
  if (g == 0 && valid) {
    a.ws_dD[(long long)q * BD + cc] = S.p0[0][c][0] + S.p0[1][c][0] + S.p0[2][c][0] + S.p0[3][c][0];
    a.ws_dbias[(long long)q * BD + cc] = S.p1[0][c][0] + S.p1[1][c][0] + S.p1[2][c][0] + S.p1[3][c][0];
  }
}

// Sums of the per-CTA partials, in a fixed order:
//   dB, dC [b, n, t] over the channel tiles of sequence b; dA [d, n], dD, dbias [d] over b.
__global__ void scan_bwd_reduce_kernel(const ScanBwdArgs a, int ndt) {
  const long long L = a.seqlen, N = a.dstate;
  const long long nBC = (long long)a.batch * N * L;
  const long long nA = (long long)a.dim * N;
  const long long total = 2 * nBC + nA + 2LL * a.dim;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    if (i < 2 * nBC) {
      const bool isC = i >= nBC;
      const long long j = isC ? i - nBC : i;
      const long long b = j / (N * L), r = j % (N * L);
      const float* src = isC ? a.ws_dC : a.ws_dB;
      float s = 0.f;
      for (int dt = 0; dt < ndt; ++dt) s += src[((b * ndt + dt) * kMaxDstate) * L + r];
      (isC ? a.dC : a.dB)[j] = s;
    } else if (i < 2 * nBC + nA) {
      const long long j = i - 2 * nBC;  // d * N + n
      float s = 0.f;
      for (int qb = 0; qb < a.nchunks * a.batch; ++qb) s += a.ws_dA[(long long)qb * nA + j];
      a.dA[j] = s;
    } else {
      const long long j = i - 2 * nBC - nA;
      const bool isBias = j >= a.dim;
      const long long dd = isBias ? j - a.dim : j;
      const float* src = isBias ? a.ws_dbias : a.ws_dD;
      float s = 0.f;
      for (int qb = 0; qb < a.nchunks * a.batch; ++qb) s += src[(long long)qb * a.dim + dd];
      float* dst = isBias ? a.ddelta_bias : a.dD;
      if (dst) dst[dd] = s;
    }
  }
}

template <typename T, bool ADJ>
cudaError_t prepare_bwd() {
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 0 && dev < 64 && configured[dev]) return cudaSuccess;
  err = cudaFuncSetAttribute(scan_bwd_kernel<T, ADJ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(BwdSmem));
  if (err == cudaSuccess && dev >= 0 && dev < 64) configured[dev] = 1;
  return err;
}

template <typename T>
cudaError_t launch_bwd_t(const ScanBwdArgs& a, cudaStream_t stream) {
  const size_t smem = sizeof(BwdSmem);
  cudaError_t err = prepare_bwd<T, false>();
  if (err != cudaSuccess) return err;
  const int ndt = (a.dim + kBDT - 1) / kBDT;
  if (a.nchunks > 1) {
    // adjoint carries of chunks 1 .. nchunks-1 (the forward carries are already on the stream)
    err = prepare_bwd<T, true>();
    if (err != cudaSuccess) return err;
    scan_bwd_kernel<T, true><<<dim3(ndt, a.batch, a.nchunks - 1), kBThreads, smem, stream>>>(a);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  scan_bwd_kernel<T, false><<<dim3(ndt, a.batch, a.nchunks), kBThreads, smem, stream>>>(a);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const long long total = 2LL * a.batch * a.dstate * a.seqlen + (long long)a.dim * a.dstate + 2LL * a.dim;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 148 * 16) blocks = 148 * 16;
  if (blocks < 1) blocks = 1;
  scan_bwd_reduce_kernel<<<(unsigned)blocks, threads, 0, stream>>>(a, ndt);
  return cudaGetLastError();
}

template <typename T>
int bwd_resident() {
  int n = 0;
  if (prepare_bwd<T, false>() != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, scan_bwd_kernel<T, false>, kBThreads, sizeof(BwdSmem)) !=
          cudaSuccess ||
      n <= 0) {
    cudaGetLastError();
    return 3;  // no device to ask: the figure the kernel is built for
  }
  return n;
}

auto up256 = [](long long v) { return (size_t)((v + 255) & ~255LL); };

}  // namespace

int scan_bwd_resident_ctas_per_sm(bool bf16) { return bf16 ? bwd_resident<__nv_bfloat16>() : bwd_resident<float>(); }

int scan_bwd_channels_per_cta() { return kBDT; }

size_t scan_bwd_workspace_bytes(int batch, int dim, int seqlen, int nchunks) {
  const long long ndt = (dim + kBDT - 1) / kBDT;
  const long long ntiles = (seqlen + kBT - 1) / kBT;
  const long long BD = (long long)batch * dim;
  const long long Q = nchunks < 1 ? 1 : nchunks;
  size_t s = up256(batch * ndt * ntiles * kBThreads * 16LL);             // checkpoints
  s += 2 * up256(batch * ndt * (long long)kMaxDstate * seqlen * 4LL);     // dB, dC partials
  s += up256(Q * BD * kMaxDstate * 4LL);                                  // dA partials
  s += 2 * up256(Q * BD * 4LL);                                           // dD, dbias partials
  s += up256((Q - 1) * BD * 4LL) + up256((Q - 1) * BD * kMaxDstate * 4LL); // forward carries
  s += up256(Q * BD * 4LL) + up256(Q * BD * kMaxDstate * 4LL);             // adjoint carries
  return s;
}

void scan_bwd_workspace_split(void* ws, int batch, int dim, int seqlen, int nchunks, ScanBwdArgs& a) {
  const long long ndt = (dim + kBDT - 1) / kBDT;
  const long long ntiles = (seqlen + kBT - 1) / kBT;
  const long long BD = (long long)batch * dim;
  const long long Q = nchunks < 1 ? 1 : nchunks;
  char* p = static_cast<char*>(ws);
  auto take = [&](size_t bytes) { char* r = p; p += bytes; return reinterpret_cast<float*>(r); };
  a.ws_ckpt = take(up256(batch * ndt * ntiles * kBThreads * 16LL));
  a.ws_dB = take(up256(batch * ndt * (long long)kMaxDstate * seqlen * 4LL));
  a.ws_dC = take(up256(batch * ndt * (long long)kMaxDstate * seqlen * 4LL));
  a.ws_dA = take(up256(Q * BD * kMaxDstate * 4LL));
  a.ws_dD = take(up256(Q * BD * 4LL));
  a.ws_dbias = take(up256(Q * BD * 4LL));
  float* fS = take(up256((Q - 1) * BD * 4LL));
  float* fh = take(up256((Q - 1) * BD * kMaxDstate * 4LL));
  a.fS = fS;
  a.fh = fh;
  a.bS = take(up256(Q * BD * 4LL));
  a.bh = take(up256(Q * BD * kMaxDstate * 4LL));
}

cudaError_t launch_scan_bwd(const ScanBwdArgs& a, cudaStream_t stream) {
  if (a.bf16) return launch_bwd_t<__nv_bfloat16>(a, stream);
  return launch_bwd_t<float>(a, stream);
}

}  // namespace ssm
