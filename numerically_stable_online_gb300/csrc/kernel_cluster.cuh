// Long-row softmax: one row split across the CTAs of a thread-block cluster.
//
// The pages' answer to a row that does not fit on chip is the block summary:
// process the row in blocks, keep (m, d) per block, merge the summaries by
// rescaling both sums to the larger maximum ("Stable softmax: keep the
// normalizer consistent as tiles arrive", third paragraph; "Online stable
// softmax", "Derive the update for two blocks"; "Softmax numerics
// architecture...", "Online softmax: one recurrence, one fewer pass").  Here
// the blocks are the C chunks of a row held by the C CTAs of one cluster:
//
//   - CTA c owns elements [c*chunk, (c+1)*chunk) of the row.  The first part of
//     the chunk is staged in shared memory by bulk asynchronous copies (TMA,
//     cp.async.bulk, one mbarrier per piece so work starts as pieces land), the
//     next part is held in registers (RV 16-byte vectors per thread), and any
//     remainder is streamed from global memory twice (counted as re-read
//     traffic; none for rows that fit the cluster).
//   - Each thread folds its vectors into a running (m, d) with the tiled online
//     update ("Kernel visualization: online softmax", "Tiled version"); the
//     threads' summaries merge through a warp butterfly and shared memory into
//     the CTA summary.
//   - The C CTA summaries are exchanged through distributed shared memory after
//     one cluster barrier; every CTA merges all C of them in rank order, so all
//     get identical (M, D).
//   - Each CTA writes its chunk: y = exp(x - M) / D from the on-chip copy.
//
// No multicast is used: each CTA fetches only its own chunk.  Every wait on an
// mbarrier is bounded; when a bound runs out the kernel records
// SMX_ERR_TIMEOUT in the device status word and still takes every cluster
// barrier, so no CTA of the cluster is left waiting.
#pragma once

#include "row_core.cuh"
#include "smx_async.cuh"
#include "smx_launch.h"

namespace smx {

constexpr int CLUSTER_PIECES = 8;

// Fold one vector of V elements into a thread's running (m, d): the tiled
// online update with the tile = this vector.  Masked lanes hold -inf.
template <int V>
__device__ __forceinline__ void online_fold(float& m, float& d, const float (&f)[V]) {
  float vmax = f[0];
#pragma unroll
  for (int i = 1; i < V; ++i) vmax = fmax_nan(vmax, f[i]);
  const float m_new = fmax_nan(m, vmax);
  if (m_new == neg_inf()) return;  // nothing valid seen yet
  if (m_new != m) {
    // correct the running sum to the new maximum (d is 0 while m is -inf);
    // a NaN maximum poisons d, a +inf maximum is settled by the terms below
    d = (m_new != m_new) ? qnan() : __fmul_rn(d, rescale_factor(m, m_new));
    m = m_new;
  }
  float s[V];
#pragma unroll
  for (int i = 0; i < V; ++i) s[i] = exp_shift_fast<false>(f[i], m);
#pragma unroll
  for (int w = V / 2; w > 0; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) s[i] = __fadd_rn(s[i], s[i + w]);
  d = __fadd_rn(d, s[0]);
}

template <int V>
__device__ __forceinline__ void mask_tail(float (&f)[V], int64_t e0, int64_t L) {
#pragma unroll
  for (int i = 0; i < V; ++i)
    if (e0 + i >= L) f[i] = neg_inf();
}

// One element's output on the normalise pass: e^(x - M) / D.  fp32 outputs use
// the compensated exponential; 16-bit outputs one FFMA with the per-row
// constant c2 = RN(-M log2 e + s) and rD2 = 2^(-s + c2_err) / D, where c2_err is
// the exact rounding residual of c2 (s = 8 for bf16 keeps its subnormals, as in
// row_core.cuh).  Here D comes from other CTAs' sums, so the rounding of c2
// does not cancel and must be carried explicitly.
template <typename OutT>
__device__ __forceinline__ float cluster_out(float x, float M, float c2, float rD, float rD2) {
  if constexpr (ExpPolicy<OutT, MODE_SOFTMAX>::ACCURATE) {
    return __fmul_rn(exp_shift_accurate(x, M), rD);
  } else {
    return __fmul_rn(ex2_ftz(__fmaf_rn(x, L2E_HI, c2)), rD2);
  }
}

template <typename InT, typename OutT, int RV, int MODE>
__global__ void __launch_bounds__(CLUSTER_THREADS, 1)
    k_rows_cluster(const InT* __restrict__ x, OutT* __restrict__ y, float* __restrict__ m_out,
                   float* __restrict__ d_out, int64_t rows, int64_t cols,
                   const int32_t* __restrict__ valid_len, int64_t row0, int64_t chunk,
                   int64_t smem_elems, int64_t max_polls, int* __restrict__ status) {
  constexpr int V = Elem<InT>::V;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const InT* sx = reinterpret_cast<const InT*>(smem_raw);
  __shared__ __align__(8) uint64_t bars[CLUSTER_PIECES];
  __shared__ float s_m[32], s_d[32];
  __shared__ float s_cta[2];  // this CTA's (m, d), read by the peers

  const int T = CLUSTER_THREADS;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t crank = cluster_ctarank();
  const uint32_t csize = cluster_nctarank();
  const int64_t row = row0 + blockIdx.y;

  int64_t L = cols;
  if (valid_len != nullptr) {
    const int64_t v = __ldg(valid_len + row);
    L = v < 0 ? 0 : (v > cols ? cols : v);
  }
  const InT* xr = x + row * cols;

  // Chunk geometry in vectors (all element offsets are multiples of V).
  const int64_t c0 = (int64_t)crank * chunk;
  const int64_t c1 = c0 + chunk < cols ? c0 + chunk : cols;
  const int64_t c_nv = c1 > c0 ? (c1 - c0) / V : 0;
  int64_t vend = ((L + V - 1) / V) * V;  // valid data rounded up to a vector
  if (vend > c1) vend = c1;
  const int64_t v_nv = vend > c0 ? (vend - c0) / V : 0;               // valid vectors
  const int64_t a_nv = smem_elems / V < c_nv ? smem_elems / V : c_nv;  // staged region
  const int64_t s_nv = a_nv < v_nv ? a_nv : v_nv;                     // staged and valid
  const int64_t b_nv = a_nv + (int64_t)T * RV < c_nv ? a_nv + (int64_t)T * RV : c_nv;

  // Issue the staged region's copies, one mbarrier per piece.
  const int64_t piece_nv = (s_nv + CLUSTER_PIECES - 1) / CLUSTER_PIECES;
  if (t == 0) {
    for (int p = 0; p < CLUSTER_PIECES; ++p) mbar_init(smem_addr(&bars[p]), 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (t == 0) {
    for (int p = 0; p < CLUSTER_PIECES; ++p) {
      const int64_t p0 = (int64_t)p * piece_nv;
      const int64_t p1 = p0 + piece_nv < s_nv ? p0 + piece_nv : s_nv;
      if (p1 > p0) {
        const uint32_t bytes = (uint32_t)((p1 - p0) * 16);
        mbar_arrive_expect_tx(smem_addr(&bars[p]), bytes);
        bulk_load_g2s(smem_addr(smem_raw + p0 * 16), xr + c0 + p0 * V, bytes, smem_addr(&bars[p]));
      }
    }
  }

  // Register part: vector a_nv + k*T + t of the chunk.
  float r[RV][V];
#pragma unroll
  for (int k = 0; k < RV; ++k) {
    const int64_t vi = a_nv + (int64_t)k * T + t;
    if (vi < b_nv && vi < v_nv) {
      load_vec16<InT>(xr + c0 + vi * V, r[k]);
      mask_tail<V>(r[k], c0 + vi * V, L);
    } else {
#pragma unroll
      for (int i = 0; i < V; ++i) r[k][i] = neg_inf();
    }
  }

  // Pass 1a: exact maximum of the on-chip part (pieces processed as they land).
  float mx = neg_inf();
  bool timed_out = false;
  for (int p = 0; p < CLUSTER_PIECES; ++p) {
    const int64_t p0 = (int64_t)p * piece_nv;
    const int64_t p1 = p0 + piece_nv < s_nv ? p0 + piece_nv : s_nv;
    if (p1 <= p0) break;
    // after one wait has run out, later pieces get a single poll each
    if (!mbar_wait_bounded(smem_addr(&bars[p]), 0, timed_out ? 1 : max_polls)) timed_out = true;
    for (int64_t vi = p0 + t; vi < p1; vi += T) {
      float f[V];
      unpack16<InT>(*reinterpret_cast<const uint4*>(sx + vi * V), f);
      mask_tail<V>(f, c0 + vi * V, L);
#pragma unroll
      for (int i = 0; i < V; ++i) mx = fmax_nan(mx, f[i]);
    }
  }
#pragma unroll
  for (int k = 0; k < RV; ++k)
#pragma unroll
    for (int i = 0; i < V; ++i) mx = fmax_nan(mx, r[k][i]);
  mx = warp_max_nan(mx);
  if (lane == 0) s_m[warp] = mx;
  __syncthreads();
  const float m_c = warp_max_nan(lane < (T >> 5) ? s_m[lane] : neg_inf());

  // Pass 1b: sum of e^(x - m_c) over the on-chip part, one FFMA + exp2 per
  // element; the rounding of c = -m_c log2 e is common to every term and is
  // corrected once (stats_correct).
  float sum = 0.0f;
  if (m_c != neg_inf()) {
    const bool huge = !(fabsf(m_c) < 1e38f);
    const float c = huge ? 0.0f : __fmul_rn(-m_c, L2E_HI);
    auto term = [&](float v) {
      return huge ? ex2_ftz(__fmul_rn(__fsub_rn(v, m_c), L2E_HI)) : ex2_ftz(__fmaf_rn(v, L2E_HI, c));
    };
    for (int64_t vi = t; vi < s_nv; vi += T) {
      float f[V];
      unpack16<InT>(*reinterpret_cast<const uint4*>(sx + vi * V), f);
      mask_tail<V>(f, c0 + vi * V, L);
      float e[V];
#pragma unroll
      for (int i = 0; i < V; ++i) e[i] = term(f[i]);
#pragma unroll
      for (int w = V / 2; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) e[i] = __fadd_rn(e[i], e[i + w]);
      sum = __fadd_rn(sum, e[0]);
    }
#pragma unroll
    for (int k = 0; k < RV; ++k) {
      float e[V];
#pragma unroll
      for (int i = 0; i < V; ++i) e[i] = term(r[k][i]);
#pragma unroll
      for (int w = V / 2; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) e[i] = __fadd_rn(e[i], e[i + w]);
      sum = __fadd_rn(sum, e[0]);
    }
    sum = stats_correct(sum, m_c);
  }
  // Streamed remainder (rows longer than the cluster holds), first read:
  // the per-thread tiled online update, merged with the on-chip summary.
  float m_s = neg_inf(), d_s = 0.0f;
  for (int64_t vi = b_nv + t; vi < v_nv; vi += T) {
    float f[V];
    load_vec16<InT>(xr + c0 + vi * V, f);
    mask_tail<V>(f, c0 + vi * V, L);
    online_fold<V>(m_s, d_s, f);
  }
  MD md = md_merge(MD{m_c, sum}, MD{m_s, d_s});

  // CTA summary: warp butterfly, then the per-warp summaries.
  md = warp_merge(md);
  __syncthreads();  // s_m is reused
  if (lane == 0) {
    s_m[warp] = md.m;
    s_d[warp] = md.d;
  }
  __syncthreads();
  md = warp_merge(lane < (T >> 5) ? MD{s_m[lane], s_d[lane]} : MD{neg_inf(), 0.0f});
  if (t == 0) {
    s_cta[0] = md.m;
    s_cta[1] = md.d;
  }
  // Exchange through distributed shared memory.
  __syncwarp();
  cluster_arrive();
  cluster_wait();
  MD all{neg_inf(), 0.0f};
  if (lane < (int)csize) all = MD{ld_peer_f32(&s_cta[0], lane), ld_peer_f32(&s_cta[1], lane)};
  // merge in rank order: a butterfly gives identical bits in every lane
  all = warp_merge(all);
  __syncwarp();
  cluster_arrive();  // my reads of the peers are done; matched by the wait at exit

  const float M = all.m, D = all.d;
  if constexpr (MODE == MODE_STATS) {
    if (crank == 0 && t == 0) {
      m_out[row] = M;
      d_out[row] = M == neg_inf() ? 0.0f : D;
    }
  } else {
    OutT* yr = y + row * cols;
    const bool zero_row = (M == neg_inf());
    const bool nan_row = !zero_row && (D != D);
    if (!zero_row && !nan_row) {
      constexpr float SC = ExpPolicy<OutT, MODE_SOFTMAX>::SCALE_LOG2;
      const bool huge = !(fabsf(M) < 1e38f);
      const float rD = recip_refined(D);
      float c2 = SC, c2_err = 0.0f;
      if (!huge) {
        const float a = __fmul_rn(-M, L2E_HI);
        const float e1 = __fmaf_rn(-M, L2E_HI, -a);  // exact residual of the product
        c2 = __fadd_rn(a, SC);
        const float bb = __fsub_rn(c2, a);           // TwoSum(a, SC) residual
        const float e2 = __fadd_rn(__fsub_rn(a, __fsub_rn(c2, bb)), __fsub_rn(SC, bb));
        c2_err = __fadd_rn(e1, e2);
      }
      // 2^-SC / D, times 2^(c2_err) ~ 1 + c2_err ln 2
      const float rD2 = __fmul_rn(__fmul_rn(rD, SC == 0.0f ? 1.0f : 0.00390625f),
                                  __fmaf_rn(c2_err, LN2, 1.0f));
      auto emit = [&](int64_t vi, const float (&f)[V]) {
        float p[V];
#pragma unroll
        for (int i = 0; i < V; ++i) {
          const float xv = huge ? __fsub_rn(f[i], M) : f[i];
          p[i] = cluster_out<OutT>(xv, huge ? 0.0f : M, c2, rD, rD2);
        }
        store_vec<OutT, V>(yr + c0 + vi * V, p);
      };
      for (int64_t vi = t; vi < a_nv; vi += T) {
        float f[V];
        if (vi < s_nv) {
          unpack16<InT>(*reinterpret_cast<const uint4*>(sx + vi * V), f);
          mask_tail<V>(f, c0 + vi * V, L);
        } else {
#pragma unroll
          for (int i = 0; i < V; ++i) f[i] = neg_inf();
        }
        emit(vi, f);
      }
#pragma unroll
      for (int k = 0; k < RV; ++k) {
        const int64_t vi = a_nv + (int64_t)k * T + t;
        if (vi < b_nv) emit(vi, r[k]);
      }
      for (int64_t vi = b_nv + t; vi < c_nv; vi += T) {  // streamed remainder, second read
        float f[V];
        if (vi < v_nv) {
          load_vec16<InT>(xr + c0 + vi * V, f);
          mask_tail<V>(f, c0 + vi * V, L);
        } else {
#pragma unroll
          for (int i = 0; i < V; ++i) f[i] = neg_inf();
        }
        emit(vi, f);
      }
    } else {
      // policy rows: zeros, or NaN in the valid lanes
      for (int64_t vi = t; vi < c_nv; vi += T) {
        const int64_t e0 = c0 + vi * V;
        float p[V];
#pragma unroll
        for (int i = 0; i < V; ++i) p[i] = (nan_row && e0 + i < L) ? qnan() : 0.0f;
        store_vec<OutT, V>(yr + e0, p);
      }
    }
  }

  if (timed_out) {
    atomicOr(status, DEV_TIMEOUT);
    // let this CTA's own copies land before its shared memory is released
    for (int p = 0; p < CLUSTER_PIECES; ++p) {
      const int64_t p0 = (int64_t)p * piece_nv;
      if (p0 >= s_nv) break;
      mbar_wait_bounded(smem_addr(&bars[p]), 0, int64_t(1) << 21);
    }
  }
  cluster_wait();  // no CTA leaves while a peer may still read its summary
}

}  // namespace smx
