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
//   - CTA c owns elements [c*chunk, (c+1)*chunk) of every row.  The first part
//     of the chunk is staged in shared memory by bulk asynchronous copies
//     (cp.async.bulk, the non-tensor TMA form) in NP pieces, one mbarrier each;
//     the next part is held in registers (RV 16-byte vectors per thread); any
//     remainder (rows longer than the cluster holds) is streamed from global
//     memory twice, a counted re-read.
//   - The CTA takes the exact maximum m_c of its on-chip part as pieces land,
//     then sum e^(x - m_c); a streamed remainder is folded with the tiled
//     online update ("Kernel visualization: online softmax", "Tiled version").
//   - The C CTA summaries are exchanged through distributed shared memory after
//     one cluster barrier; every CTA merges all C of them in rank order with a
//     butterfly, so all get identical (M, D).
//   - Each CTA writes its chunk: y = e^(x - M) / D from the on-chip copy.
//
// The cluster is persistent: it walks rows blockIdx.y, blockIdx.y + gridDim.y,
// ... and as soon as the normalise pass has consumed staged piece p of one row
// the copy of piece p of the next row is issued into it, so the next row's
// reads overlap this row's arithmetic and writes.  No multicast is used: each
// CTA fetches only its own chunk.  Every wait on an mbarrier is bounded; when a
// bound runs out the kernel records SMX_ERR_TIMEOUT in the device status word,
// still takes every cluster barrier, and lets its own copies land before exit.
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
// does not cancel and is carried explicitly.  With |M| near the top of the
// fp32 range (huge) the difference is taken first instead.
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
__device__ __forceinline__ float cluster_out(float x, const OutConst& k) {
  if constexpr (ExpPolicy<OutT, MODE_SOFTMAX>::ACCURATE) {
    return __fmul_rn(exp_shift_accurate(x, k.M), k.rD);
  } else {
    const float u = k.huge ? __fmaf_rn(__fsub_rn(x, k.M), L2E_HI, k.c2) : __fmaf_rn(x, L2E_HI, k.c2);
    return __fmul_rn(ex2_ftz(u), k.rD2);
  }
}

// Unpack one staged vector; only the vector holding the end of the valid
// prefix needs masking.
template <typename InT, int V>
__device__ __forceinline__ void staged_vec(const InT* sx, int vi, int v_nv_full, int64_t e0, int64_t L,
                                           float (&f)[V]) {
  unpack16<InT>(*reinterpret_cast<const uint4*>(sx + (int64_t)vi * V), f);
  if (vi >= v_nv_full) mask_tail<V>(f, e0, L);
}

template <typename InT, typename OutT, int RV, int MODE>
__global__ void __launch_bounds__(CLUSTER_THREADS, 1)
    k_rows_cluster(const InT* __restrict__ x, OutT* __restrict__ y, float* __restrict__ m_out,
                   float* __restrict__ d_out, int64_t rows, int64_t cols,
                   const int32_t* __restrict__ valid_len, int64_t chunk, int64_t smem_elems,
                   int64_t max_polls, int* __restrict__ status) {
  constexpr int V = Elem<InT>::V;
  constexpr int NP = CLUSTER_PIECES;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const InT* sx = reinterpret_cast<const InT*>(smem_raw);
  __shared__ __align__(8) uint64_t bars[NP];
  __shared__ __align__(8) uint64_t never_bar;  // the error-path probe: nothing signals it
  __shared__ float s_m[32], s_d[32];
  __shared__ float s_cta[2][2];  // this CTA's (m, d) per row parity, read by the peers

  const int T = CLUSTER_THREADS;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t crank = cluster_ctarank();
  const uint32_t csize = cluster_nctarank();

  // Chunk geometry in vectors, the same for every row (offsets are multiples of V).
  const int64_t c0 = (int64_t)crank * chunk;
  const int64_t c1 = c0 + chunk < cols ? c0 + chunk : cols;
  const int c_nv = c1 > c0 ? (int)((c1 - c0) / V) : 0;
  const int a_nv = smem_elems / V < c_nv ? (int)(smem_elems / V) : c_nv;  // staged region
  const int b_nv = a_nv + T * RV < c_nv ? a_nv + T * RV : c_nv;            // end of registers
  const int P = (a_nv + NP - 1) / NP;                                      // piece size

  auto length_of = [&](int64_t row) -> int64_t {
    if (valid_len == nullptr) return cols;
    const int64_t v = __ldg(valid_len + row);
    return v < 0 ? 0 : (v > cols ? cols : v);
  };
  // valid vectors of this chunk for a row of valid length L
  auto valid_vectors = [&](int64_t L) -> int {
    int64_t vend = (L + V - 1) / V * V;
    if (vend > c1) vend = c1;
    return vend > c0 ? (int)((vend - c0) / V) : 0;
  };
  // thread 0: issue the valid part of staged piece p of `row` (one phase of bars[p])
  auto fill_piece = [&](int64_t row, int s_nv, int p) {
    const int p0 = p * P;
    int p1 = p0 + P < s_nv ? p0 + P : s_nv;
    if (p1 > p0) {
      const uint32_t bytes = (uint32_t)(p1 - p0) * 16u;
      mbar_arrive_expect_tx(smem_addr(&bars[p]), bytes);
      bulk_load_g2s(smem_addr(smem_raw + (size_t)p0 * 16), x + row * cols + c0 + (int64_t)p0 * V, bytes,
                    smem_addr(&bars[p]));
    } else {
      mbar_arrive(smem_addr(&bars[p]));
    }
  };

  const int64_t row_first = blockIdx.y;
  if (t == 0) {
    for (int p = 0; p < NP; ++p) mbar_init(smem_addr(&bars[p]), 1);
    mbar_init(smem_addr(&never_bar), 1);
    mbar_fence_init();
    // max_polls < 0 asks for a probe of the error path: a wait of -max_polls
    // polls on a barrier nothing arrives on, which must run out and be reported
    if (max_polls < 0 && !mbar_wait_bounded(smem_addr(&never_bar), 0, -max_polls))
      atomicOr(status, DEV_TIMEOUT);
    if (row_first < rows) {
      const int s_nv0 = min(a_nv, valid_vectors(length_of(row_first)));
      for (int p = 0; p < NP; ++p) fill_piece(row_first, s_nv0, p);
    }
  }
  __syncthreads();

  if (max_polls < 0) max_polls = int64_t(1) << 21;
  bool timed_out = false;
  int par = 0;
  for (int64_t row = row_first; row < rows; row += gridDim.y, par ^= 1) {
    const int64_t L = length_of(row);
    const int v_nv = valid_vectors(L);                       // valid vectors in the chunk
    const int v_full = (int)((L > c0 ? (L - c0) : 0) / V);  // vectors wholly valid
    const int s_nv = a_nv < v_nv ? a_nv : v_nv;               // staged and valid
    const InT* xr = x + row * cols + c0;
    const int64_t next_row = row + gridDim.y;
    int next_s_nv = 0;
    if (t == 0 && next_row < rows) next_s_nv = min(a_nv, valid_vectors(length_of(next_row)));

    // Register part: vector a_nv + k*T + t of the chunk.
    float r[RV][V];
#pragma unroll
    for (int k = 0; k < RV; ++k) {
      const int vi = a_nv + k * T + t;
      if (vi < b_nv && vi < v_nv) {
        load_vec16<InT>(xr + (int64_t)vi * V, r[k]);
        if (vi >= v_full) mask_tail<V>(r[k], c0 + (int64_t)vi * V, L);
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) r[k][i] = neg_inf();
      }
    }

    // Pass 1a: exact maximum of the on-chip part, pieces processed as they land.
    float mx = neg_inf();
    for (int p = 0; p < NP; ++p) {
      // after one wait has run out, later waits get a single poll each
      if (!mbar_wait_bounded(smem_addr(&bars[p]), (uint32_t)par, timed_out ? 1 : max_polls))
        timed_out = true;
      const int p1 = (p + 1) * P < s_nv ? (p + 1) * P : s_nv;
      for (int vi = p * P + t; vi < p1; vi += T) {
        float f[V];
        staged_vec<InT, V>(sx, vi, v_full, c0 + (int64_t)vi * V, L, f);
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

    // Pass 1b: sum of e^(x - m_c) over the on-chip part: one FFMA + exp2 per
    // element; the rounding of c = -m_c log2 e, common to every term, is
    // corrected once (stats_correct).
    float sum = 0.0f;
    if (m_c != neg_inf()) {
      const bool huge = !(fabsf(m_c) < 1e38f);
      const float c = huge ? 0.0f : __fmul_rn(-m_c, L2E_HI);
      const float msub = huge ? m_c : 0.0f;
      for (int vi = t; vi < s_nv; vi += T) {
        float f[V];
        staged_vec<InT, V>(sx, vi, v_full, c0 + (int64_t)vi * V, L, f);
        float e[V];
#pragma unroll
        for (int i = 0; i < V; ++i) e[i] = ex2_ftz(__fmaf_rn(__fsub_rn(f[i], msub), L2E_HI, c));
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
        for (int i = 0; i < V; ++i) e[i] = ex2_ftz(__fmaf_rn(__fsub_rn(r[k][i], msub), L2E_HI, c));
#pragma unroll
        for (int w = V / 2; w > 0; w >>= 1)
#pragma unroll
          for (int i = 0; i < w; ++i) e[i] = __fadd_rn(e[i], e[i + w]);
        sum = __fadd_rn(sum, e[0]);
      }
      sum = stats_correct(sum, m_c);
    }
    // Streamed remainder, first read: the per-thread tiled online update.
    float m_s = neg_inf(), d_s = 0.0f;
    for (int vi = b_nv + t; vi < v_nv; vi += T) {
      float f[V];
      load_vec16<InT>(xr + (int64_t)vi * V, f);
      if (vi >= v_full) mask_tail<V>(f, c0 + (int64_t)vi * V, L);
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
      s_cta[par][0] = md.m;
      s_cta[par][1] = md.d;
    }
    if constexpr (MODE == MODE_STATS) {
      // all staged reads are done (the barriers above): refill every piece now
      if (t == 0 && next_row < rows && !timed_out)
        for (int p = 0; p < NP; ++p) fill_piece(next_row, next_s_nv, p);
    }
    // Exchange through distributed shared memory.  The summaries alternate
    // between two slots by row parity: a peer reads slot par of this row
    // before it reaches the next row's barrier, and this CTA rewrites slot par
    // only two rows later, after that barrier.
    __syncwarp();
    cluster_arrive();
    cluster_wait();
    MD all{neg_inf(), 0.0f};
    if (lane < (int)csize) all = MD{ld_peer_f32(&s_cta[par][0], lane), ld_peer_f32(&s_cta[par][1], lane)};
    all = warp_merge(all);  // rank order, identical bits in every lane

    const float M = all.m, D = all.d;
    if constexpr (MODE == MODE_STATS) {
      if (crank == 0 && t == 0) {
        m_out[row] = M;
        d_out[row] = M == neg_inf() ? 0.0f : D;
      }
    } else {
      OutT* yr = y + row * cols + c0;
      const bool zero_row = (M == neg_inf());
      const bool nan_row = !zero_row && (D != D);
      const OutConst kc = make_out_const<OutT>(M, D);
      auto emit = [&](int vi, const float (&f)[V], bool valid_vec) {
        float pv[V];
        if (!zero_row && !nan_row) {
#pragma unroll
          for (int i = 0; i < V; ++i) pv[i] = valid_vec ? cluster_out<OutT>(f[i], kc) : 0.0f;
        } else {
          const int64_t e0 = c0 + (int64_t)vi * V;
#pragma unroll
          for (int i = 0; i < V; ++i) pv[i] = (nan_row && e0 + i < L) ? qnan() : 0.0f;
        }
        store_vec<OutT, V>(yr + (int64_t)vi * V, pv);
      };
      for (int p = 0; p < NP; ++p) {
        const int p0 = p * P, p1 = (p + 1) * P < a_nv ? (p + 1) * P : a_nv;
        for (int vi = p0 + t; vi < p1; vi += T) {
          float f[V];
          const bool valid_vec = vi < s_nv;
          if (valid_vec) staged_vec<InT, V>(sx, vi, v_full, c0 + (int64_t)vi * V, L, f);
          emit(vi, f, valid_vec);
        }
        __syncthreads();  // piece p is consumed: refill it with the next row
        // (not after a wait of thread 0 ran out: that barrier's phase may
        // still be pending, and a second arrive on it is not allowed)
        if (t == 0 && next_row < rows && !timed_out) fill_piece(next_row, next_s_nv, p);
      }
#pragma unroll
      for (int k = 0; k < RV; ++k) {
        const int vi = a_nv + k * T + t;
        if (vi < b_nv) emit(vi, r[k], true);
      }
      for (int vi = b_nv + t; vi < c_nv; vi += T) {  // streamed remainder, second read
        float f[V];
        const bool valid_vec = vi < v_nv;
        if (valid_vec) {
          load_vec16<InT>(xr + (int64_t)vi * V, f);
          if (vi >= v_full) mask_tail<V>(f, c0 + (int64_t)vi * V, L);
        }
        emit(vi, f, valid_vec);
      }
    }
  }

  if (timed_out) {
    atomicOr(status, DEV_TIMEOUT);
    // let this CTA's own copies land before its shared memory is released
    const int last = rows > row_first ? (int)(((rows - 1 - row_first) / gridDim.y) & 1) : 0;
    for (int p = 0; p < NP; ++p) mbar_wait_bounded(smem_addr(&bars[p]), (uint32_t)last, int64_t(1) << 21);
  }
  // no CTA leaves while a peer may still read its last summary
  __syncwarp();
  cluster_arrive();
  cluster_wait();
}

}  // namespace smx
