// ssm_device.cuh -- device-side helpers shared by the scan, conv and decode kernels:
// I/O dtype conversion, vector moves, and the transcendental building blocks
// (exp2, sigmoid/SiLU, softplus) in the two precision tiers the library uses.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- MUFU primitives (PTX)

// 2^x on the special-function unit; flushes subnormal results to zero.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// tanh on the SFU; relative error about 2^-11 (used only by the bf16 tier).
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- packed fp32 pairs (sm_100+ f32x2)
// One instruction computes two fp32 lanes; the FMA pipe throughput per element is unchanged,
// the issue slots are halved.

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

// ---------------------------------------------------------------- activations

// silu(x) = x * sigmoid(x) = x / (1 + e^-x). For x -> -inf, e^-x -> inf and the
// reciprocal gives 0; for x -> +inf it gives x.
__device__ __forceinline__ float silu_f(float x) {
  return x * rcp_approx(1.0f + ex2_approx(-x * kLog2e));
}

// log(1 + e) for e in [0, 1]: log(1 + e) = 2 atanh(s) with s = e / (2 + e) in [0, 1/3], summed
// as s (1 + s^2/3 + s^4/5 + ... + s^12/13); the first omitted term is below 2e-8 relative, so
// the result is good to a few ulp, including for tiny e where 1 + e rounds.
__device__ __forceinline__ float log1p_unit(float e) {
  const float s = e * rcp_approx(2.0f + e);
  const float s2 = s * s;
  float p = fmaf(s2, 1.0f / 13.0f, 1.0f / 11.0f);
  p = fmaf(s2, p, 1.0f / 9.0f);
  p = fmaf(s2, p, 1.0f / 7.0f);
  p = fmaf(s2, p, 1.0f / 5.0f);
  p = fmaf(s2, p, 1.0f / 3.0f);
  p = fmaf(s2, p, 1.0f);
  return 2.0f * s * p;
}

// softplus(v) = log(1 + e^v).
// PRECISE: max(v, 0) + log(1 + e^-|v|), exact in form for every v, accurate to ~1e-6 relative.
// Fast tier: lg2(1 + 2^(v log2 e)) ln 2, v itself above 20 (the remainder is below e^-20
// relative); its relative error near Delta ~ 1e-3 is ~2e-4, inside the bf16 output tolerance.
template <bool PRECISE>
__device__ __forceinline__ float softplus_f(float v) {
  if (PRECISE) return fmaxf(v, 0.0f) + log1p_unit(ex2_approx(-fabsf(v) * kLog2e));
  if (v > 20.0f) return v;
  return lg2_approx(1.0f + ex2_approx(v * kLog2e)) * kLn2;
}

// Pairwise forms: the FMA-pipe work packed two lanes per instruction, the SFU work per element.

// silu, accurate tier: x / (1 + 2^(-x log2 e)).
__device__ __forceinline__ float2 silu2(float2 x) {
  const float2 t = fmul2(x, f2(-kLog2e));
  const float2 den = fadd2(make_float2(ex2_approx(t.x), ex2_approx(t.y)), f2(1.0f));
  return fmul2(x, make_float2(rcp_approx(den.x), rcp_approx(den.y)));
}

// silu, fast tier: with h = x/2, silu(x) = h + h tanh(h); one SFU op per element.
__device__ __forceinline__ float2 silu2_tanh(float2 x) {
  const float2 h = fmul2(x, f2(0.5f));
  return ffma2(h, make_float2(tanh_approx(h.x), tanh_approx(h.y)), h);
}

template <bool PRECISE>
__device__ __forceinline__ float2 silu2_tier(float2 x) {
  if (PRECISE) return silu2(x);
  return silu2_tanh(x);
}

// Delta log2(e) from the raw delta: Delta = softplus(delta + bias) (or delta + bias when
// softplus is off). The scan keeps Delta in these log2 units, so exp(Delta A) = 2^(Delta' A)
// needs no scaling of A; bias_l2 = bias log2(e).
template <bool PRECISE>
__device__ __forceinline__ float2 delta_log2(float2 dv, float bias, float bias_l2, bool softplus) {
  if (PRECISE) {
    float2 v = fadd2(dv, f2(bias));
    if (softplus) v = make_float2(softplus_f<true>(v.x), softplus_f<true>(v.y));
    return fmul2(v, f2(kLog2e));
  }
  const float2 t = ffma2(dv, f2(kLog2e), f2(bias_l2));
  if (!softplus) return t;
  // softplus(v) log2(e) = lg2(1 + 2^t), t = v log2(e); t itself above 20 log2(e)
  const float2 s = fadd2(make_float2(ex2_approx(t.x), ex2_approx(t.y)), f2(1.0f));
  const float kT = 20.0f * kLog2e;
  return make_float2(t.x > kT ? t.x : lg2_approx(s.x), t.y > kT ? t.y : lg2_approx(s.y));
}

// Zero-order-hold input factor expm1(Delta A) / A (so that Bbar = factor * B), from
// x = Delta' A (Delta' = Delta log2 e, so Delta A = x ln 2), e = 2^x, Delta' and 1/A (0 for A = 0):
//   |Delta A| < 1/16: Delta expm1(y)/y = Delta' (ln2 + x ln2^2/2 + x^2 ln2^3/6 + x^3 ln2^4/24
//                     + x^4 ln2^5/120), the series truncated after y^4 (next term below 2e-9
//                     relative); this also covers A = 0, where the factor is Delta;
//   otherwise:        (e - 1) / A, where e's 2^-22 error is at most 3e-6 of e - 1.
constexpr float kZohC1 = 0.6931471805599453f;   // ln2
constexpr float kZohC2 = 0.2402265069591007f;   // ln2^2 / 2
constexpr float kZohC3 = 0.0555041086648216f;   // ln2^3 / 6
constexpr float kZohC4 = 0.0096181291076285f;   // ln2^4 / 24
constexpr float kZohC5 = 0.0013333558146428f;   // ln2^5 / 120
constexpr float kZohSmall = 0.0901684400555602f;  // 1 / (16 ln2): |x| below it means |Delta A| < 1/16

__device__ __forceinline__ float zoh_factor(float x, float e, float dlog2, float invA) {
  float p = fmaf(x, kZohC5, kZohC4);
  p = fmaf(x, p, kZohC3);
  p = fmaf(x, p, kZohC2);
  p = fmaf(x, p, kZohC1);
  return fabsf(x) < kZohSmall ? dlog2 * p : (e - 1.0f) * invA;
}

__device__ __forceinline__ float2 zoh_factor2(float2 x, float2 e, float2 dlog2, float2 invA) {
  float2 p = ffma2(x, f2(kZohC5), f2(kZohC4));
  p = ffma2(x, p, f2(kZohC3));
  p = ffma2(x, p, f2(kZohC2));
  p = ffma2(x, p, f2(kZohC1));
  const float2 small = fmul2(dlog2, p);
  const float2 large = fmul2(fadd2(e, f2(-1.0f)), invA);
  return make_float2(fabsf(x.x) < kZohSmall ? small.x : large.x, fabsf(x.y) < kZohSmall ? small.y : large.y);
}

// ---------------------------------------------------------------- I/O dtype

template <typename T> struct IoTraits;
template <> struct IoTraits<float> {
  static constexpr int kBytes = 4;
  static constexpr bool kPrecise = true;   // fp32 I/O: accurate softplus
};
template <> struct IoTraits<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  static constexpr bool kPrecise = false;  // bf16 I/O: fast transcendental tier
};

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Load 4 consecutive elements (t .. t+3) as floats. The pointer must be 4-element aligned
// in the vector path (16 B for fp32, 8 B for bf16).
__device__ __forceinline__ void load4(const float* p, float (&v)[4]) {
  float4 q = *reinterpret_cast<const float4*>(p);
  v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&v)[4]) {
  uint2 q = *reinterpret_cast<const uint2*>(p);
  v[0] = __uint_as_float(q.x << 16);
  v[1] = __uint_as_float(q.x & 0xffff0000u);
  v[2] = __uint_as_float(q.y << 16);
  v[3] = __uint_as_float(q.y & 0xffff0000u);
}

__device__ __forceinline__ void store4(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, const float (&v)[4]) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
  __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
  uint2 q;
  q.x = *reinterpret_cast<uint32_t*>(&a);
  q.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = q;
}

// 8 consecutive elements; 16-byte aligned pointer (bf16: one 16-byte access, fp32: two).
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 q = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------- async copies (sm_80+ cp.async)

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared copy; src_bytes = 0 zero-fills the destination without reading.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_addr(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

}  // namespace ssm
