// Device-side building blocks shared by the softmax kernels (sm_103a).
//
// Arithmetic conventions, following "Softmax numerics architecture - max
// subtract, fp32 accumulate, fusion, online":
//   - the running maximum and the sum are fp32 whatever the storage type
//     ("Why the accumulator is fp32 even when the inputs are not");
//   - exp(z) is evaluated as 2^(z log2 e) on the hardware exp2 unit ("On CPU,
//     and the pitfalls worth naming": fold log2 e into one constant);
//   - the maximum is taken lane-wise with one horizontal reduction at the end
//     (same section, first pitfall).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace smx {

// log2(e) = 1 / ln 2 split as a sum of two floats: L2E_HI = fp32(log2 e) and
// L2E_LO = fp32(log2 e - L2E_HI).  LN2 = fp32(ln 2).
constexpr float L2E_HI = 1.44269502162933349609375f;  // 0x3FB8AA3B
constexpr float L2E_LO = 1.925963033500011079e-08f;   // 0x32A57060
constexpr float LN2 = 0.693147182464599609375f;       // 0x3F317218
constexpr float L2E_LO_LN2 = 1.3349759e-08f;          // fp32(L2E_LO * ln 2)

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }
__device__ __forceinline__ float pos_inf() { return __int_as_float(0x7f800000); }
__device__ __forceinline__ float qnan() { return __int_as_float(0x7fffffff); }

// Hardware 2^u (MUFU).  The .ftz form flushes subnormal results to zero; the
// plain form keeps them (needed only when a bf16 output can be subnormal).
__device__ __forceinline__ float ex2_ftz(float u) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(u));
  return r;
}
__device__ __forceinline__ float ex2_full(float u) {
  float r;
  asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(u));
  return r;
}

// 1/D for the normaliser: hardware reciprocal estimate refined by one
// Newton-Raphson step r' = r + r (1 - D r), carried out with FMAs.  D lies in
// [1, cols] on every row this is used for (the argmax term alone contributes 1),
// so no range handling is needed; the result is within about 1 ulp of 1/D.
__device__ __forceinline__ float recip_refined(float D) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(D));
  const float e = __fmaf_rn(-D, r, 1.0f);
  return __fmaf_rn(r, e, r);
}

// max that propagates NaN (IEEE maximum, not maxNum): a NaN anywhere in the
// row must reach the row's statistics.
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
// The same over three operands in one instruction (sm_100 family).
__device__ __forceinline__ float fmax3_nan(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// e^(x - m), fast form: one rounding of x - m, one of the product by log2 e.
// Relative error about (|x - m| + 1) * 2^-23 plus that of the exp2 unit; used
// where the result is rounded to a 16-bit type or only enters a sum.
template <bool SUBNORMAL>
__device__ __forceinline__ float exp_shift_fast(float x, float m) {
  const float u = __fmul_rn(__fsub_rn(x, m), L2E_HI);
  return SUBNORMAL ? ex2_full(u) : ex2_ftz(u);
}

// e^(x - m), compensated form for fp32 results.  With |x - m| up to ~100 a
// plain fp32 argument carries an absolute error up to ~2^-18, which is a
// relative error of the same size in the result.  Here the difference is kept
// as t + t_lo (Knuth's TwoSum: t_lo is the exact rounding error of x - m) and
// the product by log2 e as u + u_lo (u_lo from the exact FMA residual of
// t * L2E_HI, plus the t * L2E_LO and t_lo * log2 e terms).  Then
// 2^(u + u_lo) = 2^u (1 + u_lo ln 2 + O(u_lo^2)), with |u_lo| < 2^-16, so the
// result's error is essentially that of the exp2 unit.  A difference below
// -110 (including one that overflowed to -inf, or x = -inf) gives +0 directly:
// e^-110 is below the smallest fp32 subnormal, and the TwoSum of infinities
// would otherwise produce NaN.  A NaN operand still yields NaN.
__device__ __forceinline__ float exp_shift_accurate(float x, float m) {
  const float t = __fsub_rn(x, m);
  const float z = __fsub_rn(t, x);
  const float t_lo = __fadd_rn(__fsub_rn(x, __fsub_rn(t, z)), __fsub_rn(-m, z));
  const float u = __fmul_rn(t, L2E_HI);
  // ln 2 * (u_exact - u): the exact product residual, the t * L2E_LO term and
  // t_lo * log2 e, each scaled by ln 2 (ln 2 * log2 e = 1 up to 2^-25, which is
  // far below these terms' own size)
  const float r = __fmaf_rn(t, L2E_HI, -u);
  const float corr = __fmaf_rn(r, LN2, __fmaf_rn(t, L2E_LO_LN2, t_lo));
  const float e = ex2_ftz(u);
  // selected, not branched: the TwoSum of an infinite t is NaN
  return t < -110.0f ? 0.0f : __fmaf_rn(e, corr, e);
}

// ---------------------------------------------------------------------------
// (m, d) block summaries.  The merge rescales both sums to the larger maximum
// ("Online stable softmax", "Derive the update for two blocks"); the empty
// block (-inf, 0) is selected around, never evaluated, so -inf - (-inf) never
// occurs.  Written so that merge(a, b) and merge(b, a) give identical bits
// (explicit round-to-nearest operations, no contraction), which keeps every
// lane of a butterfly reduction in agreement.
// ---------------------------------------------------------------------------
struct MD {
  float m, d;
};

__device__ __forceinline__ float rescale_factor(float m_old, float m_new) {
  // e^(m_old - m_new) for finite m_new >= m_old; exactly 1 when equal, 0 for
  // the empty block.
  if (m_old == m_new) return 1.0f;
  if (m_old == neg_inf()) return 0.0f;
  return exp_shift_accurate(m_old, m_new);
}

// The policy for special maxima matches the fp64 reference exactly: a NaN
// maximum poisons both fields, the empty block is the identity (and two empty
// blocks give (-inf, 0)), a +inf maximum gives (+inf, NaN).
__device__ __forceinline__ MD md_merge(MD a, MD b) {
  if (a.m != a.m || b.m != b.m) return MD{qnan(), qnan()};
  if (a.m == neg_inf()) return b.m == neg_inf() ? MD{neg_inf(), 0.0f} : b;
  if (b.m == neg_inf()) return a;
  const float m = fmaxf(a.m, b.m);
  if (m == pos_inf()) return MD{pos_inf(), qnan()};
  const float fa = rescale_factor(a.m, m);
  const float fb = rescale_factor(b.m, m);
  return MD{m, __fadd_rn(__fmul_rn(a.d, fa), __fmul_rn(b.d, fb))};
}

// ---------------------------------------------------------------------------
// Warp reductions (butterfly over all 32 lanes, every lane gets the result).
// ---------------------------------------------------------------------------
// One instruction on sm_100-family GPUs: the warp's NaN-propagating maximum
// delivered to every lane.
__device__ __forceinline__ float warp_max_nan(float v) {
  float r;
  asm volatile("redux.sync.max.NaN.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// The warp's minimum (NaN operands do not reach it: callers use it only when
// the warp's NaN-propagating maximum is finite).
__device__ __forceinline__ float warp_min(float v) {
  float r;
  asm volatile("redux.sync.min.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ MD warp_merge(MD v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    MD o{__shfl_xor_sync(0xffffffffu, v.m, off), __shfl_xor_sync(0xffffffffu, v.d, off)};
    v = md_merge(v, o);
  }
  // identical in every lane by construction; broadcast lane 0 all the same
  v.m = __shfl_sync(0xffffffffu, v.m, 0);
  v.d = __shfl_sync(0xffffffffu, v.d, 0);
  return v;
}

// ---------------------------------------------------------------------------
// Packed fp32 pairs (one f32x2 instruction for two lanes' worth of arithmetic;
// each half is rounded exactly as the scalar operation would be).
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long pk(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float pk_lo(unsigned long long v) { return __uint_as_float((unsigned)v); }
__device__ __forceinline__ float pk_hi(unsigned long long v) {
  return __uint_as_float((unsigned)(v >> 32));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// exp_shift_accurate for two lanes at once in f32x2 arithmetic.  Every step is
// the scalar step with each half rounded the same way (a - b as fma(b, -1, a),
// -u as t * (-L2E_HI): both exact rewrites), so the results are bit-identical
// to two scalar calls, in about half the instructions.
__device__ __forceinline__ void exp_shift_accurate2(float x0, float x1, float m, float& e0, float& e1) {
  const unsigned long long X = pk(x0, x1), NM = pk(-m, -m), N1 = pk(-1.0f, -1.0f);
  const unsigned long long T = add2(X, NM);          // t = x - m
  const unsigned long long Z = fma2(X, N1, T);       // z = t - x
  const unsigned long long TZ = fma2(Z, N1, T);      // t - z
  const unsigned long long TLO = add2(fma2(TZ, N1, X), fma2(Z, N1, NM));  // (x - (t - z)) + (-m - z)
  const unsigned long long UN = mul2(T, pk(-L2E_HI, -L2E_HI));           // -u
  const unsigned long long R = fma2(T, pk(L2E_HI, L2E_HI), UN);          // t L2E_HI - u, exact
  const unsigned long long C =
      fma2(R, pk(LN2, LN2), fma2(T, pk(L2E_LO_LN2, L2E_LO_LN2), TLO));
  const unsigned long long E = pk(ex2_ftz(-pk_lo(UN)), ex2_ftz(-pk_hi(UN)));
  const unsigned long long RES = fma2(E, C, E);
  e0 = pk_lo(T) < -110.0f ? 0.0f : pk_lo(RES);
  e1 = pk_hi(T) < -110.0f ? 0.0f : pk_hi(RES);
}

// ---------------------------------------------------------------------------
// Storage types.  A 16-byte vector holds V = 16 / sizeof(T) elements.
// ---------------------------------------------------------------------------
template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int V = 4;
  __device__ static __forceinline__ float to_f32(float v) { return v; }
  __device__ static __forceinline__ float from_f32(float v) { return v; }
};
template <>
struct Elem<__half> {
  static constexpr int V = 8;
  __device__ static __forceinline__ float to_f32(__half v) { return __half2float(v); }
  __device__ static __forceinline__ __half from_f32(float v) { return __float2half_rn(v); }
};
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int V = 8;
  __device__ static __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ static __forceinline__ __nv_bfloat16 from_f32(float v) { return __float2bfloat16_rn(v); }
};

// 16-byte read-only streaming load (no L1 allocation) and unpack to fp32.
template <typename T>
__device__ __forceinline__ void load_vec16(const T* p, float (&f)[Elem<T>::V]) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  const T* e = reinterpret_cast<const T*>(&r);
#pragma unroll
  for (int i = 0; i < Elem<T>::V; ++i) f[i] = Elem<T>::to_f32(e[i]);
}

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& r, float (&f)[Elem<T>::V]) {
  const T* e = reinterpret_cast<const T*>(&r);
#pragma unroll
  for (int i = 0; i < Elem<T>::V; ++i) f[i] = Elem<T>::to_f32(e[i]);
}

// Store N fp32 values converted to T at p (N * sizeof(T) bytes, aligned to that
// size, N * sizeof(T) in {8, 16, 32}).
template <typename T, int N>
__device__ __forceinline__ void store_vec(T* p, const float (&f)[N]) {
  constexpr int BYTES = N * (int)sizeof(T);
  static_assert(BYTES == 8 || BYTES == 16 || BYTES == 32, "vector store size");
  union {
    T e[N];
    uint2 u2[BYTES / 8];
    uint4 u4[(BYTES + 15) / 16];
  } u;
#pragma unroll
  for (int i = 0; i < N; ++i) u.e[i] = Elem<T>::from_f32(f[i]);
  if constexpr (BYTES == 8) {
    __stcs(reinterpret_cast<uint2*>(p), u.u2[0]);
  } else {
#pragma unroll
    for (int i = 0; i < BYTES / 16; ++i) __stcs(reinterpret_cast<uint4*>(p) + i, u.u4[i]);
  }
}

// Device status word (one per device, allocated by the host library).
enum : int { DEV_OK = 0, DEV_TIMEOUT = 5 };

}  // namespace smx
