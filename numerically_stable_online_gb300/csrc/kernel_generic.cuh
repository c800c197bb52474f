// Generic row softmax for any alignment and any cols, and the element-wise
// merge of block summaries.
//
// The generic kernel is the two-pass online softmax of "Kernel visualization:
// online softmax" ("Online softmax: two passes"): pass 1 folds every element
// into a running (m, d) with the per-element recurrence m_i = max(m_{i-1},
// x_i), d_i = d_{i-1} e^(m_{i-1} - m_i) + e^(x_i - m_i), from (m_0, d_0) =
// (-inf, 0) ("Online softmax", "Derivation"), one running state per thread;
// the threads' states merge as block summaries; pass 2 re-reads the row and
// writes exp(x - M) / D.  It reads the row twice (2 reads + 1 write), so it
// serves only shapes the vectorised kernels cannot take: unaligned pointers or
// cols * sizeof(type) not a multiple of 16.
//
// The same kernel takes the other modes of the streamed kernel on such shapes:
// row statistics (LSE when d_out is null), log_softmax (MODE_LOG), normalising
// with given per-row (m_in, d_in) (MODE_APPLY, no first pass), and
// cross-entropy (MODE_CE: loss, and the gradient when y is given).
#pragma once

#include "kernel_stream.cuh"

namespace smx {

constexpr int GENERIC_THREADS = 256;

template <typename InT, typename OutT, int MODE>
__global__ void __launch_bounds__(GENERIC_THREADS)
    k_rows_generic(const InT* __restrict__ x, OutT* __restrict__ y, float* __restrict__ m_out,
                   float* __restrict__ d_out, const float* __restrict__ m_in,
                   const float* __restrict__ d_in, int64_t rows, int64_t cols,
                   const int32_t* __restrict__ valid_len, int64_t row0,
                   const int64_t* __restrict__ target, float* __restrict__ loss) {
  __shared__ float s_m[GENERIC_THREADS / 32], s_d[GENERIC_THREADS / 32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t row = row0 + blockIdx.x;
  int64_t L = cols;
  if (valid_len != nullptr) {
    const int64_t v = __ldg(valid_len + row);
    L = v < 0 ? 0 : (v > cols ? cols : v);
  }
  const InT* xr = x + row * cols;

  float M, D;
  if constexpr (MODE == MODE_APPLY) {
    M = __ldg(m_in + row);
    D = __ldg(d_in + row);
  } else {
    // Pass 1: per-element recurrence over finite values; NaN and +inf are noted
    // and settled by the policy after the merge.
    float m = neg_inf(), d = 0.0f;
    int flags = 0;  // 1: NaN seen, 2: +inf seen
    for (int64_t j = t; j < L; j += GENERIC_THREADS) {
      const float v = Elem<InT>::to_f32(xr[j]);
      if (v != v) {
        flags |= 1;
      } else if (v == pos_inf()) {
        flags |= 2;
      } else if (v != neg_inf()) {
        if (v > m) {
          d = __fadd_rn(__fmul_rn(d, rescale_factor(m, v)), 1.0f);  // e^(v - v) = 1
          m = v;
        } else {
          d = __fadd_rn(d, exp_shift_fast<false>(v, m));
        }
      }
    }
    MD md = warp_merge(MD{m, d});
    if (lane == 0) {
      s_m[warp] = md.m;
      s_d[warp] = md.d;
    }
    // __syncthreads_or returns a predicate (non-zero if any thread's is), so
    // each flag gets its own vote
    const int any_nan = __syncthreads_or(flags & 1);
    const int any_pinf = __syncthreads_or(flags & 2);
    md = warp_merge(lane < GENERIC_THREADS / 32 ? MD{s_m[lane], s_d[lane]} : MD{neg_inf(), 0.0f});
    M = md.m;
    D = md.d;
    if (any_nan) {
      M = qnan();
      D = qnan();
    } else if (any_pinf) {
      M = pos_inf();
      D = qnan();
    }
  }

  if constexpr (MODE == MODE_STATS) {
    if (t == 0) {
      if (d_out != nullptr) {
        m_out[row] = M;
        d_out[row] = D;
      } else {  // LSE = m + log d
        m_out[row] = M == neg_inf() ? neg_inf() : __fadd_rn(M, logf(D));
      }
    }
  } else if constexpr (MODE == MODE_CE) {
    const int64_t tg = __ldg(target + row);
    const bool ignored = tg < 0 || tg >= L;
    const bool bad = M == neg_inf() || M != M || D != D;
    if (t == 0) {
      float out = 0.0f;
      if (!ignored)
        out = bad ? qnan() : __fadd_rn(__fsub_rn(M, Elem<InT>::to_f32(xr[tg])), logf(D));
      loss[row] = out;
    }
    if (y != nullptr) {
      OutT* yr = y + row * cols;
      const float rD = recip_refined(D);
      for (int64_t j = t; j < cols; j += GENERIC_THREADS) {
        float q = 0.0f;
        if (!ignored && j < L) {
          if (bad) q = qnan();
          else q = __fmul_rn(exp_for<OutT, MODE_SOFTMAX>(Elem<InT>::to_f32(xr[j]), M), rD);
          if (j == tg) q = __fsub_rn(q, 1.0f);
        }
        yr[j] = Elem<OutT>::from_f32(q);
      }
    }
  } else if constexpr (MODE == MODE_LOG) {
    OutT* yr = y + row * cols;
    const bool zero_row = (M == neg_inf());
    const bool nan_row = !zero_row && (D != D);
    const float ld = zero_row ? 0.0f : logf(D);
    for (int64_t j = t; j < cols; j += GENERIC_THREADS) {
      float q = neg_inf();
      if (j < L && !zero_row)
        q = nan_row ? qnan() : __fsub_rn(__fsub_rn(Elem<InT>::to_f32(xr[j]), M), ld);
      yr[j] = Elem<OutT>::from_f32(q);
    }
  } else {
    OutT* yr = y + row * cols;
    const bool zero_row = (M == neg_inf());
    const bool nan_row = !zero_row && (D != D || M != M || M == pos_inf());
    const float rD = recip_refined(D);
    for (int64_t j = t; j < cols; j += GENERIC_THREADS) {
      float p = 0.0f;
      if (j < L && !zero_row) {
        if (nan_row) p = qnan();
        else p = __fmul_rn(exp_for<OutT, MODE_SOFTMAX>(Elem<InT>::to_f32(xr[j]), M), rD);
      }
      yr[j] = Elem<OutT>::from_f32(p);
    }
  }
}

}  // namespace smx
