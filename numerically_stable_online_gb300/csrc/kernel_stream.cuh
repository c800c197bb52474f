// Persistent row softmax that keeps the next rows' reads in flight while it
// reduces the current one; rows of up to 32 KiB.
//
// Same arithmetic as the register-resident kernel (kernel_regs.cuh, via
// row_core.cuh): exact row maximum, exponentials against it with their fp32
// sum, one normalising multiply; one HBM read and one HBM write per element.
// The register kernel's CTA holds no reads in flight while it reduces its row;
// here a persistent CTA of G threads walks the rows blockIdx.x,
// blockIdx.x + gridDim.x, ... and every thread prefetches its own 16-byte
// vectors of the next DEPTH rows into its own shared-memory words with
// cp.async (one commit group per row).  Each thread reads back only what it
// copied itself, so the prefetch needs no barrier; a row's group is awaited
// with cp.async.wait_group just before the row is used.
#pragma once

#include "row_core.cuh"

namespace smx {

__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_dst), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// SMX_STREAM_MAXNREG (a build-time tuning knob) caps the registers per thread,
// trading spills for resident CTAs.
#ifdef SMX_STREAM_MAXNREG
#define SMX_STREAM_REGS __maxnreg__(SMX_STREAM_MAXNREG)
#else
#define SMX_STREAM_REGS __launch_bounds__(1024)
#endif

template <typename InT, typename OutT, int VPT, int MODE, int DEPTH>
__global__ void SMX_STREAM_REGS
    k_rows_stream(const InT* __restrict__ x, OutT* __restrict__ y, float* __restrict__ m_out,
                  float* __restrict__ d_out, int64_t rows, int64_t cols,
                  const int32_t* __restrict__ valid_len) {
  constexpr int V = Elem<InT>::V;
  extern __shared__ __align__(16) uint4 sbuf[];  // [DEPTH][VPT][G]: thread g owns column g
  // s_max alternates between rows: a row with no valid lane skips the sum's
  // barrier, so only the next row's max barrier separates reads from rewrites
  __shared__ float s_max[2][32], s_sum[32];

  const int G = blockDim.x, g = threadIdx.x, lane = g & 31, warp = g >> 5, nw = G >> 5;
  const int ncols = (int)cols;
  const uint32_t my_slot = static_cast<uint32_t>(__cvta_generic_to_shared(sbuf + g));
  const uint32_t slot_stride = (uint32_t)(VPT * G * 16);  // bytes between ring slots

  auto length_of = [&](int64_t row) {
    if (valid_len == nullptr) return ncols;
    const int v = __ldg(valid_len + row);
    return v < 0 ? 0 : (v > ncols ? ncols : v);
  };
  // copy this thread's vectors of `row` into ring slot d; always one group
  auto prefetch = [&](int64_t row, int d) {
    int L = 0;
    if (row < rows) {
      L = length_of(row);
      const InT* xr = x + row * cols;
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
        const int e0 = (j * G + g) * V;
        if (e0 < L) cp_async16(my_slot + d * slot_stride + j * G * 16, xr + e0);
      }
    }
    cp_async_commit();
    return L;
  };

  int64_t row = blockIdx.x;
  int Ls[DEPTH];
#pragma unroll
  for (int d = 0; d < DEPTH; ++d) Ls[d] = prefetch(row + (int64_t)d * gridDim.x, d);

  for (int d = 0, par = 0; row < rows; row += gridDim.x, par ^= 1) {
    cp_async_wait<DEPTH - 1>();  // this thread's copies of `row` have landed
    const int L = Ls[0];
    float v[VPT][V];
    const InT* sx = reinterpret_cast<const InT*>(sbuf + (size_t)d * VPT * G);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int e0 = (j * G + g) * V;
      load_masked<InT, true>(sx + e0, e0, L, v[j]);
    }
    float mx = warp_max_nan(local_max(v));
    // the slot's words are in registers now: refill it with the row DEPTH ahead
#pragma unroll
    for (int i = 0; i + 1 < DEPTH; ++i) Ls[i] = Ls[i + 1];
    Ls[DEPTH - 1] = prefetch(row + (int64_t)DEPTH * gridDim.x, d);
    d = d + 1 == DEPTH ? 0 : d + 1;

    if (lane == 0) s_max[par][warp] = mx;
    __syncthreads();
    mx = warp_max_nan(lane < nw ? s_max[par][lane] : neg_inf());
    const float M = mx;
    float Dsum = 0.0f;
    if (M != neg_inf()) {
      float sum = warp_sum(exp_and_sum<OutT, MODE>(v, M));
      if (lane == 0) s_sum[warp] = sum;
      __syncthreads();
      Dsum = warp_sum(lane < nw ? s_sum[lane] : 0.0f);
    }
    if constexpr (MODE == MODE_STATS) {
      if (g == 0) {
        m_out[row] = M;
        d_out[row] = M == neg_inf() ? 0.0f : stats_correct(Dsum, M);
      }
    } else {
      const bool zero_row = (M == neg_inf());
      const bool nan_row = !zero_row && (Dsum != Dsum);
      store_row<OutT, VPT, V>(y + row * cols, G, g, ncols, L, v, zero_row, nan_row,
                              recip_refined(Dsum));
    }
  }
  cp_async_wait<0>();  // no copy may still target this CTA's shared memory at exit
}

}  // namespace smx
