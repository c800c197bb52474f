// Persistent, TMA-pipelined row softmax for rows of up to 32 KiB.
//
// Same arithmetic as the register-resident kernel (kernel_regs.cuh): exact row
// maximum, then exponentials against it and their fp32 sum, then one
// normalising multiply; one HBM read and one HBM write per element.  What
// changes is how the reads are kept in flight.  Each CTA is persistent and
// walks the rows blockIdx.x, blockIdx.x + gridDim.x, ...:
//
//   - warp 0 is the producer: one lane copies whole rows (their valid prefix
//     only) into a ring of S shared-memory slots with bulk asynchronous copies
//     (cp.async.bulk), signalling a "full" mbarrier per slot;
//   - the other warps form NG consumer groups of WG warps; group g takes the
//     CTA's rows g, g + NG, ...: it waits for the slot's full barrier, moves
//     the row into registers, releases the slot on its "empty" barrier (so the
//     producer can refill it while the row is still being reduced), and then
//     reduces and writes the row straight from registers.
//
// Up to S rows per CTA are in flight at once, independent of how long the
// reductions take.  All waits are bounded (SMX_ERR_TIMEOUT in the status word
// when a bound runs out).
#pragma once

#include "kernel_cluster.cuh"
#include "kernel_regs.cuh"

namespace smx {

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

struct PipeShape {
  int stages;            // slots in the ring
  int groups;            // consumer groups
  int warps_per_group;   // warps per row
  int slot_bytes;        // bytes per slot (multiple of 128)
};

template <typename InT, typename OutT, int VPT, int MODE>
__global__ void __launch_bounds__(1024, 1)
    k_rows_pipe(const InT* __restrict__ x, OutT* __restrict__ y, float* __restrict__ m_out,
                float* __restrict__ d_out, int64_t rows, int64_t cols,
                const int32_t* __restrict__ valid_len, PipeShape sh, int64_t max_polls,
                int* __restrict__ status) {
  constexpr int V = Elem<InT>::V;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int S = sh.stages, NG = sh.groups, WG = sh.warps_per_group;
  const int G = WG * 32;  // threads per row
  uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + (size_t)S * sh.slot_bytes);
  uint64_t* empty = full + S;
  float* s_red = reinterpret_cast<float*>(empty + S);  // [NG][2][WG]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ncols = (int)cols;
  const int64_t n_k = rows > blockIdx.x ? (rows - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), WG);
    }
    mbar_fence_init();
  }
  __syncthreads();

  bool timed_out = false;
  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      for (int64_t k = 0; k < n_k; ++k) {
        const int s = (int)(k % S);
        const int64_t use = k / S;
        if (use > 0 &&
            !mbar_wait_bounded(smem_addr(&empty[s]), (uint32_t)((use - 1) & 1), timed_out ? 1 : max_polls))
          timed_out = true;
        const int64_t row = blockIdx.x + k * gridDim.x;
        int L = ncols;
        if (valid_len != nullptr) {
          const int v = __ldg(valid_len + row);
          L = v < 0 ? 0 : (v > ncols ? ncols : v);
        }
        const uint32_t bytes = (uint32_t)(((L + V - 1) / V) * 16);
        if (bytes > 0) {
          mbar_arrive_expect_tx(smem_addr(&full[s]), bytes);
          bulk_load_g2s(smem_addr(smem_raw + (size_t)s * sh.slot_bytes), x + row * cols, bytes,
                        smem_addr(&full[s]));
        } else {
          mbar_arrive(smem_addr(&full[s]));
        }
      }
      // before the CTA may exit, every slot's last fill must have landed
      for (int64_t k = n_k > S ? n_k - S : 0; k < n_k; ++k) {
        const int s = (int)(k % S);
        if (!mbar_wait_bounded(smem_addr(&full[s]), (uint32_t)((k / S) & 1), max_polls)) timed_out = true;
      }
    }
  } else {
    // ---------------- consumers ----------------
    const int cw = warp - 1;
    const int g = cw / WG;            // group
    const int wg = cw % WG;           // warp within the group
    const int tg = wg * 32 + lane;    // thread within the group
    const int bar_id = 1 + g;
    float* red_max = s_red + (size_t)g * 2 * WG;
    float* red_sum = red_max + WG;
    if (g < NG) {
      for (int64_t k = g; k < n_k; k += NG) {
        const int s = (int)(k % S);
        if (!mbar_wait_bounded(smem_addr(&full[s]), (uint32_t)((k / S) & 1), timed_out ? 1 : max_polls))
          timed_out = true;
        const int64_t row = blockIdx.x + k * gridDim.x;
        int L = ncols;
        if (valid_len != nullptr) {
          const int v = __ldg(valid_len + row);
          L = v < 0 ? 0 : (v > ncols ? ncols : v);
        }
        const InT* sx = reinterpret_cast<const InT*>(smem_raw + (size_t)s * sh.slot_bytes);
        float v[VPT][V];
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
          const int e0 = (j * G + tg) * V;
          if (e0 < L) {
            unpack16<InT>(*reinterpret_cast<const uint4*>(sx + e0), v[j]);
#pragma unroll
            for (int i = 0; i < V; ++i)
              if (e0 + i >= L) v[j][i] = neg_inf();
          } else {
#pragma unroll
            for (int i = 0; i < V; ++i) v[j][i] = neg_inf();
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[s]));  // slot may be refilled

        // row maximum
        float mx = neg_inf();
#pragma unroll
        for (int j = 0; j < VPT; ++j)
#pragma unroll
          for (int i = 0; i < V; ++i) mx = fmax_nan(mx, v[j][i]);
        mx = warp_max_nan(mx);
        if (WG > 1) {
          if (lane == 0) red_max[wg] = mx;
          named_barrier(bar_id, G);
          mx = warp_max_nan(lane < WG ? red_max[lane] : neg_inf());
        }
        const float M = mx;
        // exponentials and their sum
        float D = 0.0f;
        if (M != neg_inf()) {
          float sum = 0.0f;
#pragma unroll
          for (int j = 0; j < VPT; ++j) {
#pragma unroll
            for (int i = 0; i < V; ++i) v[j][i] = exp_for<OutT, MODE>(v[j][i], M);
            float sk[V];
#pragma unroll
            for (int i = 0; i < V; ++i) sk[i] = v[j][i];
#pragma unroll
            for (int w = V / 2; w > 0; w >>= 1)
#pragma unroll
              for (int i = 0; i < w; ++i) sk[i] = __fadd_rn(sk[i], sk[i + w]);
            sum = __fadd_rn(sum, sk[0]);
          }
          sum = warp_sum(sum);
          if (WG > 1) {
            if (lane == 0) red_sum[wg] = sum;
            named_barrier(bar_id, G);
            sum = warp_sum(lane < WG ? red_sum[lane] : 0.0f);
          }
          D = sum;
        }
        if constexpr (MODE == MODE_STATS) {
          if (tg == 0) {
            m_out[row] = M;
            d_out[row] = D;
          }
        } else {
          OutT* yr = y + row * cols;
          const bool zero_row = (M == neg_inf());
          const bool nan_row = !zero_row && (D != D);
          const float rD = recip_refined(D);
#pragma unroll
          for (int j = 0; j < VPT; ++j) {
            const int e0 = (j * G + tg) * V;
            if (e0 < ncols) {
              float p[V];
#pragma unroll
              for (int i = 0; i < V; ++i) {
                if (zero_row) p[i] = 0.0f;
                else if (nan_row) p[i] = (e0 + i < L) ? qnan() : 0.0f;
                else p[i] = __fmul_rn(v[j][i], rD);
              }
              store_vec<OutT, V>(yr + e0, p);
            }
          }
        }
      }
    }
  }
  if (timed_out) atomicOr(status, DEV_TIMEOUT);
}

}  // namespace smx
