// Register-resident row softmax: one HBM read and one HBM write per element.
//
// A row is owned by a group of G threads (a warp, or a whole CTA); each thread
// holds VPT 16-byte vectors of the row in registers, widened to fp32.  The row
// never leaves the chip between its load and its store, so the traffic is the
// 1-read + 1-write minimum of "Softmax numerics architecture...", section
// "Fusion and the memory-traffic account" ("Stable softmax...", fifth
// paragraph, for the caveat that this holds only while the row fits).
//
// Steps, with all values in fp32 (row_core.cuh):
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

#include "row_core.cuh"

namespace smx {

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

  // In-row offsets fit in 32 bits (the host sends rows of at most 32768
  // elements here).
  const int ncols = (int)cols;
  int L = ncols;
  if (valid_len != nullptr) {
    const int v = __ldg(valid_len + row);
    L = v < 0 ? 0 : (v > ncols ? ncols : v);
  }
  const InT* xr = x + row * cols;

  float v[VPT][V];
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int e0 = (j * G + g) * V;
    load_masked<InT, false>(xr + e0, e0, L, v[j]);
  }

  float mx = warp_max_nan(local_max(v));
  if (!WARP_ROW) {
    if (lane == 0) s_max[warp] = mx;
    __syncthreads();
    mx = warp_max_nan(lane < (G >> 5) ? s_max[lane] : neg_inf());
  }
  const float M = mx;

  float D = 0.0f;
  if (M != neg_inf()) {
    float s = warp_sum(exp_and_sum<OutT, MODE>(v, M));
    if (!WARP_ROW) {
      if (lane == 0) s_sum[warp] = s;
      __syncthreads();
      s = warp_sum(lane < (G >> 5) ? s_sum[lane] : 0.0f);
    }
    D = s;
  }

  if constexpr (MODE == MODE_STATS) {
    if (g == 0) {
      m_out[row] = M;
      d_out[row] = M == neg_inf() ? 0.0f : stats_correct(D, M);
    }
  } else {
    const bool zero_row = (M == neg_inf());
    const bool nan_row = !zero_row && (D != D);
    store_row<OutT, VPT, V>(y + row * cols, G, g, ncols, L, v, zero_row, nan_row, recip_refined(D));
  }
}

}  // namespace smx
