// Register-resident row softmax: one HBM read and one HBM write per element.
//
// A row is owned by a group of G threads (a warp, or a whole CTA); each thread
// holds VPT 16-byte vectors of the row in registers, widened to fp32.  The row
// never leaves the chip between its load and its store, so the traffic is the
// 1-read + 1-write minimum of "Softmax numerics architecture...", section
// "Fusion and the memory-traffic account" ("Stable softmax...", fifth
// paragraph, for the caveat that this holds only while the row fits).
//
// Steps, with all values in fp32:
//   1. load the valid prefix (lanes >= L become -inf, the exclusion value of
//      "Online stable softmax", "Masks, empty rows, and precision"; vectors
//      wholly past L are never loaded);
//   2. lane-wise maximum, then one butterfly over the warp and one pass over
//      the per-warp maxima (first pitfall of "On CPU, and the pitfalls worth
//      naming");
//   3. e_j = exp(x_j - M) kept in the registers that held x_j, and the row sum
//      D = sum e_j reduced the same way (pairwise inside a thread, then a tree:
//      "Why the accumulator is fp32...");
//   4. y_j = e_j * (1/D), converted to the output type, stored.
// Because the maximum is exact before any exponential is taken, no rescale is
// needed on this path; the (m, d) merge is used where a row is split across
// CTAs (kernel_cluster.cuh).
#pragma once

#include <type_traits>

#include "smx_device.cuh"

namespace smx {

enum : int { MODE_SOFTMAX = 0, MODE_STATS = 1 };

template <typename OutT>
struct OutPolicy {
  // fp32 outputs need the compensated exponential; 16-bit outputs are rounded
  // far above its error.  bf16 shares fp32's exponent range, so its outputs
  // can be subnormal and the exp2 must not flush them.
  static constexpr bool ACCURATE = std::is_same<OutT, float>::value;
  static constexpr bool SUBNORMAL = std::is_same<OutT, __nv_bfloat16>::value;
};

template <typename OutT, int MODE>
__device__ __forceinline__ float exp_for(float x, float M) {
  if constexpr (MODE == MODE_SOFTMAX && OutPolicy<OutT>::ACCURATE) {
    return x == neg_inf() ? 0.0f : exp_shift_accurate(x, M);
  } else {
    return exp_shift_fast<(MODE == MODE_SOFTMAX && OutPolicy<OutT>::SUBNORMAL)>(x, M);
  }
}

// Store V consecutive outputs starting at element e0 of the row.
template <typename OutT, int V>
__device__ __forceinline__ void store_out(OutT* yr, int e0, const float (&p)[V]) {
  store_vec<OutT, V>(yr + e0, p);
}

template <typename InT, typename OutT, int VPT, bool WARP_ROW, int MODE>
__global__ void __launch_bounds__(1024)
    k_rows_regs(const InT* __restrict__ x, OutT* __restrict__ y, float* __restrict__ m_out,
                float* __restrict__ d_out, int64_t rows, int64_t cols,
                const int32_t* __restrict__ valid_len, int64_t row0) {
  constexpr int V = Elem<InT>::V;
  __shared__ float s_max[32];
  __shared__ float s_sum[32];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int G = WARP_ROW ? 32 : (int)blockDim.x;
  const int g = WARP_ROW ? lane : (int)threadIdx.x;
  const int64_t row = row0 + (WARP_ROW ? (int64_t)blockIdx.x * (blockDim.x >> 5) + warp
                                       : (int64_t)blockIdx.x);
  if (WARP_ROW && row >= rows) return;  // whole warp leaves; no block barrier below

  // In-row offsets fit in 32 bits on this path (the host sends rows of at most
  // 32768 elements here).
  const int ncols = (int)cols;
  int L = ncols;
  if (valid_len != nullptr) {
    const int v = __ldg(valid_len + row);
    L = v < 0 ? 0 : (v > ncols ? ncols : v);
  }
  const InT* xr = x + row * cols;

  // 1. load (vector k of thread g starts at element (k*G + g)*V)
  float v[VPT][V];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int e0 = (k * G + g) * V;
    if (e0 < L) {
      load_vec16<InT>(xr + e0, v[k]);
#pragma unroll
      for (int i = 0; i < V; ++i)
        if (e0 + i >= L) v[k][i] = neg_inf();
    } else {
#pragma unroll
      for (int i = 0; i < V; ++i) v[k][i] = neg_inf();
    }
  }

  // 2. row maximum (NaN-propagating)
  float mx = neg_inf();
#pragma unroll
  for (int k = 0; k < VPT; ++k)
#pragma unroll
    for (int i = 0; i < V; ++i) mx = fmax_nan(mx, v[k][i]);
  mx = warp_max_nan(mx);
  if (!WARP_ROW) {
    const int nw = G >> 5;
    if (lane == 0) s_max[warp] = mx;
    __syncthreads();
    mx = warp_max_nan(lane < nw ? s_max[lane] : neg_inf());
  }
  const float M = mx;

  // 3. exponentials against the row maximum, and their sum
  float D = 0.0f;
  if (M != neg_inf()) {
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
#pragma unroll
      for (int i = 0; i < V; ++i) v[k][i] = exp_for<OutT, MODE>(v[k][i], M);
      float sk[V];
#pragma unroll
      for (int i = 0; i < V; ++i) sk[i] = v[k][i];
#pragma unroll
      for (int w = V / 2; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) sk[i] = __fadd_rn(sk[i], sk[i + w]);
      s = __fadd_rn(s, sk[0]);
    }
    s = warp_sum(s);
    if (!WARP_ROW) {
      const int nw = G >> 5;
      if (lane == 0) s_sum[warp] = s;
      __syncthreads();
      s = warp_sum(lane < nw ? s_sum[lane] : 0.0f);
    }
    D = s;
  }

  if constexpr (MODE == MODE_STATS) {
    if (g == 0) {
      m_out[row] = M;
      d_out[row] = D;  // (-inf, 0) for empty rows; NaN rows carry NaN in D
    }
    return;
  } else {
    OutT* yr = y + row * cols;
    // Row classes of the declared policy: empty / all -inf -> zeros; NaN or
    // +inf present (D is NaN) -> NaN in valid lanes; otherwise normal.
    const bool zero_row = (M == neg_inf());
    const bool nan_row = !zero_row && (D != D);
    const float rD = recip_refined(D);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int e0 = (k * G + g) * V;
      if (e0 < ncols) {
        float p[V];
#pragma unroll
        for (int i = 0; i < V; ++i) {
          if (zero_row) p[i] = 0.0f;
          else if (nan_row) p[i] = (e0 + i < L) ? qnan() : 0.0f;
          else p[i] = __fmul_rn(v[k][i], rD);
        }
        store_out<OutT, V>(yr, e0, p);
      }
    }
  }
}

}  // namespace smx
