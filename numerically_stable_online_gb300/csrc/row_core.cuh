// Per-row work shared by the register-resident and the streamed kernels: a
// row is held by a group of G threads, VPT 16-byte vectors per thread, widened
// to fp32; thread g's vector j starts at element (j*G + g)*V.
//
// The exponent argument.  "Softmax numerics architecture...", section "On CPU,
// and the pitfalls worth naming", folds log2 e into one constant so that the
// kernel calls exp2; here the whole shift is folded too:
//     u_j = fma(x_j, L2E_HI, c),  c = RN(-M * L2E_HI) (+ s),
// one FFMA per element, exact product and one rounding of a result near the
// row's own range.  The rounding of c is an offset common to every element, so
// it cancels in p_j = e_j / sum_k e_k ("The max-subtraction identity, and why
// it is exact": any common shift cancels); the statistics path, which reports
// d itself, multiplies the sum once by 2^(c_lo) with c_lo the exact residual of
// c.  For bf16 outputs s = 8 scales every e_j by 2^8 (cancelled by the same
// argument) so that the flush-to-zero exp2 never flushes a value that would
// round to a nonzero bf16 subnormal (those need e_j >= 2^-134).  fp32 outputs
// use the compensated exponential of smx_device.cuh instead.
#pragma once

#include <type_traits>

#include "smx_device.cuh"

namespace smx {

enum : int { MODE_SOFTMAX = 0, MODE_STATS = 1 };

template <typename OutT, int MODE>
struct ExpPolicy {
  static constexpr bool ACCURATE = (MODE == MODE_SOFTMAX) && std::is_same<OutT, float>::value;
  static constexpr float SCALE_LOG2 =
      (MODE == MODE_SOFTMAX && std::is_same<OutT, __nv_bfloat16>::value) ? 8.0f : 0.0f;
};

// e^(x - M) one element at a time (cluster and generic kernels): compensated
// for fp32 outputs, the plain form otherwise (bf16 outputs keep subnormals).
template <typename OutT, int MODE>
__device__ __forceinline__ float exp_for(float x, float M) {
  if constexpr (ExpPolicy<OutT, MODE>::ACCURATE) {
    return exp_shift_accurate(x, M);
  } else {
    return exp_shift_fast<(MODE == MODE_SOFTMAX && std::is_same<OutT, __nv_bfloat16>::value)>(x, M);
  }
}

// Masked load of one vector: lanes at or past L become -inf (the exclusion
// value).  SMEM selects a shared-memory source.
template <typename InT, bool SMEM>
__device__ __forceinline__ void load_masked(const InT* p, int e0, int L, float (&f)[Elem<InT>::V]) {
  constexpr int V = Elem<InT>::V;
  if (e0 + V <= L) {
    if constexpr (SMEM) unpack16<InT>(*reinterpret_cast<const uint4*>(p), f);
    else load_vec16<InT>(p, f);
  } else if (e0 < L) {
    if constexpr (SMEM) unpack16<InT>(*reinterpret_cast<const uint4*>(p), f);
    else load_vec16<InT>(p, f);
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (e0 + i >= L) f[i] = neg_inf();
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) f[i] = neg_inf();
  }
}

template <int VPT, int V>
__device__ __forceinline__ float local_max(const float (&v)[VPT][V]) {
  float m = neg_inf();
#pragma unroll
  for (int j = 0; j < VPT; ++j)
#pragma unroll
    for (int i = 0; i < V; i += 2) m = fmax3_nan(m, v[j][i], v[j][i + 1]);
  return m;
}

// Replace v by the exponentials against the row maximum M and return this
// thread's share of their sum (pairwise within each vector).  Requires M != -inf.
template <typename OutT, int MODE, int VPT, int V>
__device__ __forceinline__ float exp_and_sum(float (&v)[VPT][V], float M) {
  using P = ExpPolicy<OutT, MODE>;
  if constexpr (P::ACCURATE) {
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      float sk[V];
#pragma unroll
      for (int i = 0; i < V; i += 2) {
        exp_shift_accurate2(v[j][i], v[j][i + 1], M, v[j][i], v[j][i + 1]);
        sk[i] = v[j][i];
        sk[i + 1] = v[j][i + 1];
      }
#pragma unroll
      for (int w = V / 2; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) sk[i] = __fadd_rn(sk[i], sk[i + w]);
      s = __fadd_rn(s, sk[0]);
    }
    return s;
  } else {
    // u = x * L2E_HI + c two lanes at a time (f32x2), then exp2 per lane; with
    // |M| near the top of the fp32 range -M * log2 e would overflow, so there
    // x - M is taken first (a difference that overflows is -inf and gives 0)
    const bool huge = !(fabsf(M) < 1e38f);
    const float c = huge ? P::SCALE_LOG2 : __fmaf_rn(-M, L2E_HI, P::SCALE_LOG2);
    const float msub = huge ? M : 0.0f;
    const unsigned long long k2 = pk(L2E_HI, L2E_HI), c2 = pk(c, c);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      if (huge) {
#pragma unroll
        for (int i = 0; i < V; ++i) v[j][i] = __fsub_rn(v[j][i], msub);
      }
#pragma unroll
      for (int i = 0; i < V; i += 2) {
        const unsigned long long u = fma2(pk(v[j][i], v[j][i + 1]), k2, c2);
        v[j][i] = ex2_ftz(pk_lo(u));
        v[j][i + 1] = ex2_ftz(pk_hi(u));
      }
    }
    // pairwise sums, two partial sums at a time
    unsigned long long acc = pk(0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      unsigned long long q[V / 2];
#pragma unroll
      for (int i = 0; i < V / 2; ++i) q[i] = pk(v[j][2 * i], v[j][2 * i + 1]);
#pragma unroll
      for (int w = V / 4; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) q[i] = add2(q[i], q[i + w]);
      acc = add2(acc, q[0]);
    }
    return __fadd_rn(pk_lo(acc), pk_hi(acc));
  }
}

// This thread's share of sum_j e^(x_j - M) as the statistics path forms it
// (to be corrected by stats_correct), leaving v unchanged.  Requires M != -inf.
template <int VPT, int V>
__device__ __forceinline__ float sum_exp(const float (&v)[VPT][V], float M) {
  unsigned long long acc = pk(0.0f, 0.0f);
  const unsigned long long k2 = pk(L2E_HI, L2E_HI);
  if (fabsf(M) < 1e38f) {
    const float c = __fmul_rn(-M, L2E_HI);
    const unsigned long long c2 = pk(c, c);
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
      for (int i = 0; i < V; i += 2) {
        const unsigned long long u = fma2(pk(v[j][i], v[j][i + 1]), k2, c2);
        acc = add2(acc, pk(ex2_ftz(pk_lo(u)), ex2_ftz(pk_hi(u))));
      }
  } else {  // |M| near the top of the range: x - M first (see exp_and_sum)
    const unsigned long long nm = pk(-M, -M);
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
      for (int i = 0; i < V; i += 2) {
        const unsigned long long u = mul2(add2(pk(v[j][i], v[j][i + 1]), nm), k2);
        acc = add2(acc, pk(ex2_ftz(pk_lo(u)), ex2_ftz(pk_hi(u))));
      }
  }
  return __fadd_rn(pk_lo(acc), pk_hi(acc));
}

// One element's exponential exactly as exp_and_sum<OutT, MODE_SOFTMAX> forms
// it (same operations, same rounding): the compensated exponential for fp32
// outputs, else 2^(fma(x, L2E_HI, c)) with its row constant c.
template <typename OutT>
__device__ __forceinline__ float exp_like_softmax(float x, float M) {
  using P = ExpPolicy<OutT, MODE_SOFTMAX>;
  if constexpr (P::ACCURATE) {
    return exp_shift_accurate(x, M);
  } else {
    if (!(fabsf(M) < 1e38f)) return ex2_ftz(__fmaf_rn(__fsub_rn(x, M), L2E_HI, P::SCALE_LOG2));
    return ex2_ftz(__fmaf_rn(x, L2E_HI, __fmaf_rn(-M, L2E_HI, P::SCALE_LOG2)));
  }
}

// The exponent offset, in log2 units, of the sum exp_and_sum<OutT,
// MODE_SOFTMAX> forms: its terms are 2^(x L2E_HI + c) = 2^((x - M) L2E_HI) *
// 2^delta with delta = c + M L2E_HI exactly, c = RN(-M L2E_HI + s).  With
// a = RN(-M L2E_HI) and e1 its exact residual, delta = (c - a) - e1, where
// c - a is exact (Sterbenz) unless |M| is small, when its rounding is far
// below the error of the sum.  So log d = log(sum) - delta ln 2.  The
// compensated exponential (fp32 outputs) has no offset.
template <typename OutT>
__device__ __forceinline__ float softmax_sum_offset_log2(float M) {
  using P = ExpPolicy<OutT, MODE_SOFTMAX>;
  if constexpr (P::ACCURATE) {
    return 0.0f;
  } else {
    if (!(fabsf(M) < 1e38f)) return P::SCALE_LOG2;
    const float a = __fmul_rn(-M, L2E_HI);
    const float e1 = __fmaf_rn(-M, L2E_HI, -a);
    const float c = __fmaf_rn(-M, L2E_HI, P::SCALE_LOG2);
    return __fsub_rn(__fsub_rn(c, a), e1);
  }
}

// Store log_softmax of the row held in v (inputs x): (x - M) - ld with
// ld = log D, two subtractions so that the result does not carry the rounding
// of a large M + log D; -inf in masked lanes (x = -inf there already) and on
// zero rows; NaN in the valid lanes of NaN rows.
template <typename OutT, int VPT, int V>
__device__ __forceinline__ void store_log(OutT* yr, int G, int g, int ncols, int L, const float (&v)[VPT][V],
                                          bool zero_row, bool nan_row, float M, float ld) {
  const unsigned long long nm = pk(-M, -M), nl = pk(-ld, -ld);
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int e0 = (j * G + g) * V;
    if (e0 < ncols) {
      float q[V];
      if (!zero_row && !nan_row) {
#pragma unroll
        for (int i = 0; i < V; i += 2) {
          const unsigned long long t = add2(add2(pk(v[j][i], v[j][i + 1]), nm), nl);
          q[i] = pk_lo(t);
          q[i + 1] = pk_hi(t);
        }
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) q[i] = (nan_row && e0 + i < L) ? qnan() : neg_inf();
      }
      store_vec<OutT, V>(yr + e0, q);
    }
  }
}

// The statistics path's d: the sum of exp2(fma(x, L2E_HI, c_hi)) times
// 2^(c_lo), c_lo the exact rounding residual of c_hi = RN(-M * L2E_HI).
__device__ __forceinline__ float stats_correct(float sum, float M) {
  if (!(fabsf(M) < 1e38f)) return sum;  // the subtract-first branch has no offset
  const float c_hi = __fmul_rn(-M, L2E_HI);
  const float c_lo = __fmaf_rn(-M, L2E_HI, -c_hi);
  return __fmaf_rn(sum, __fmul_rn(c_lo, LN2), sum);
}

// Normalise and store the row held in v (exponentials), or the policy's zero /
// NaN row.  Uniform branches per row; one multiply per element on normal rows.
template <typename OutT, int VPT, int V>
__device__ __forceinline__ void store_row(OutT* yr, int G, int g, int ncols, int L, const float (&v)[VPT][V],
                                          bool zero_row, bool nan_row, float rD) {
  if (!zero_row && !nan_row) {
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int e0 = (j * G + g) * V;
      if (e0 < ncols) {
        float p[V];
        const unsigned long long r2 = pk(rD, rD);
#pragma unroll
        for (int i = 0; i < V; i += 2) {
          const unsigned long long q = mul2(pk(v[j][i], v[j][i + 1]), r2);
          p[i] = pk_lo(q);
          p[i + 1] = pk_hi(q);
        }
        store_vec<OutT, V>(yr + e0, p);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int e0 = (j * G + g) * V;
      if (e0 < ncols) {
        float p[V];
#pragma unroll
        for (int i = 0; i < V; ++i) p[i] = (nan_row && e0 + i < L) ? qnan() : 0.0f;
        store_vec<OutT, V>(yr + e0, p);
      }
    }
  }
}

// e^(x - M) / D for one element (pass 2, and the cluster kernel's normalise
// pass): compensated for fp32 outputs; otherwise one FFMA with the per-row
// constant c2 = RN(-M log2 e + s) and rD2 = 2^(-s + c2_err) / D, c2_err the
// exact rounding residual of c2 (s = 8 for bf16 keeps its subnormals, as in
// row_core.cuh).  The summaries come from other CTAs, so the rounding of c2
// does not cancel against the sum and is carried explicitly.  With |M| near
// the top of the fp32 range (huge) the difference is taken first instead.
struct OutConst {
  float M, c2, rD, rD2;
  bool huge;
};

template <typename OutT>
__device__ __forceinline__ OutConst make_out_const(float M, float D) {
  constexpr float SC = ExpPolicy<OutT, MODE_SOFTMAX>::SCALE_LOG2;
  OutConst k;
  k.M = M;
  k.huge = !(fabsf(M) < 1e38f);
  k.rD = recip_refined(D);
  k.c2 = SC;
  float c2_err = 0.0f;
  if (!k.huge) {
    const float a = __fmul_rn(-M, L2E_HI);
    const float e1 = __fmaf_rn(-M, L2E_HI, -a);  // exact residual of the product
    k.c2 = __fadd_rn(a, SC);
    const float bb = __fsub_rn(k.c2, a);         // TwoSum(a, SC) residual
    const float e2 = __fadd_rn(__fsub_rn(a, __fsub_rn(k.c2, bb)), __fsub_rn(SC, bb));
    c2_err = __fadd_rn(e1, e2);
  }
  k.rD2 = __fmul_rn(__fmul_rn(k.rD, SC == 0.0f ? 1.0f : 0.00390625f), __fmaf_rn(c2_err, LN2, 1.0f));
  return k;
}

template <typename OutT>
__device__ __forceinline__ float out_value(float x, const OutConst& k) {
  if constexpr (ExpPolicy<OutT, MODE_SOFTMAX>::ACCURATE) {
    return __fmul_rn(exp_shift_accurate(x, k.M), k.rD);
  } else {
    const float u = k.huge ? __fmaf_rn(__fsub_rn(x, k.M), L2E_HI, k.c2) : __fmaf_rn(x, L2E_HI, k.c2);
    return __fmul_rn(ex2_ftz(u), k.rD2);
  }
}

// out_value of a vector's lanes, two at a time where the arithmetic packs
// (identical results to the scalar form).
template <typename OutT, int V>
__device__ __forceinline__ void out_values(const float (&x)[V], const OutConst& k, float (&q)[V]) {
  if constexpr (ExpPolicy<OutT, MODE_SOFTMAX>::ACCURATE) {
#pragma unroll
    for (int i = 0; i < V; i += 2) {
      float e0, e1;
      exp_shift_accurate2(x[i], x[i + 1], k.M, e0, e1);
      const unsigned long long r = mul2(pk(e0, e1), pk(k.rD, k.rD));
      q[i] = pk_lo(r);
      q[i + 1] = pk_hi(r);
    }
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) q[i] = out_value<OutT>(x[i], k);
  }
}

}  // namespace smx
