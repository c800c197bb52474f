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

// Unpack one staged vector; only the vector holding the end of the valid
// prefix needs masking.
template <typename InT, int V>
__device__ __forceinline__ void staged_vec(const InT* sx, int vi, int v_nv_full, int64_t e0, int64_t L,
                                           float (&f)[V]) {
  unpack16<InT>(*reinterpret_cast<const uint4*>(sx + (int64_t)vi * V), f);
  if (vi >= v_nv_full) mask_tail<V>(f, e0, L);
}

// cp.async.wait_group with a run-time count (0..7).
__device__ __forceinline__ void cp_async_wait_dyn(int n) {
  switch (n) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
  }
}

// Staging of the shared-memory part.  TMA: thread 0 issues one bulk copy per
// piece and every thread waits on the piece's mbarrier.  Otherwise every thread
// copies its own vectors of the piece with cp.async (one commit group per
// piece) and waits on its own groups; every pass visits the staged region with
// the same thread-to-vector map (piece p, vectors p*P + t + k*T), so a thread
// only ever reads what it staged itself and the stage needs no barrier.
template <typename InT, typename OutT, int RV, int MODE, bool TMA>
__global__ void __launch_bounds__(CLUSTER_THREADS, 1)
    k_rows_cluster(const InT* __restrict__ x, OutT* __restrict__ y, float* __restrict__ m_out,
                   float* __restrict__ d_out, int64_t rows, int64_t cols,
                   const int32_t* __restrict__ valid_len, int64_t chunk, int64_t smem_elems,
                   int64_t max_polls, int* __restrict__ status) {
  constexpr int V = Elem<InT>::V;
  constexpr int NP = CLUSTER_PIECES;
  // fp32 in and out: the sum pass computes the compensated e^(x - m_c) once and
  // keeps it (in place of x in shared memory, and in the register part); the
  // normalise pass is then one multiply by e^(m_c - M) / D
  constexpr bool KEEP_E = ExpPolicy<OutT, MODE>::ACCURATE && std::is_same<InT, float>::value;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const InT* sx = reinterpret_cast<const InT*>(smem_raw);
  float* se = reinterpret_cast<float*>(smem_raw);  // the kept exponentials (KEEP_E)
  __shared__ __align__(8) uint64_t bars[NP];
  __shared__ __align__(8) uint64_t never_bar;  // the error-path probe: nothing signals it
  __shared__ float s_m[32], s_d[32];
  // every CTA's (m, d) for the row, pushed here by its owner; two slots by row
  // parity (see the exchange below)
  __shared__ float s_all[2][16][2];

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
  auto piece_end = [&](int p, int lim) { return (p + 1) * P < lim ? (p + 1) * P : lim; };
  // thread 0 (TMA): bit p = parity of the number of fills issued on piece p's
  // barrier, so that the last issued fill's phase is known after a timeout
  uint32_t fill_par = 0;
  // stage the valid part of piece p of `row` (s_nv staged-and-valid vectors)
  auto fill_piece = [&](int64_t row, int s_nv, int p) {
    const InT* src = x + row * cols + c0;
    if constexpr (TMA) {
      if (t != 0) return;
      // order this CTA's earlier generic-proxy accesses of the piece (reads,
      // and the kept exponentials' writes) before the copy's async-proxy writes
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      const int p0 = p * P, p1 = piece_end(p, s_nv);
      if (p1 > p0) {
        const uint32_t bytes = (uint32_t)(p1 - p0) * 16u;
        mbar_arrive_expect_tx(smem_addr(&bars[p]), bytes);
        bulk_load_g2s(smem_addr(smem_raw + (size_t)p0 * 16), src + (int64_t)p0 * V, bytes,
                      smem_addr(&bars[p]));
      } else {
        mbar_arrive(smem_addr(&bars[p]));
      }
      fill_par ^= 1u << p;
    } else {
      const int p1 = piece_end(p, s_nv);
      for (int vi = p * P + t; vi < p1; vi += T)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_raw + (size_t)vi * 16)),
                     "l"(src + (int64_t)vi * V)
                     : "memory");
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
  };
  auto load_regs = [&](int64_t row, float (&r)[RV][V]) {
    const int64_t L = length_of(row);
    const int v_nv = valid_vectors(L);
    const int v_full = (int)((L > c0 ? (L - c0) : 0) / V);
    const InT* src = x + row * cols + c0;
#pragma unroll
    for (int k = 0; k < RV; ++k) {
      const int vi = a_nv + k * T + t;
      if (vi < b_nv && vi < v_nv) {
        load_vec16<InT>(src + (int64_t)vi * V, r[k]);
        if (vi >= v_full) mask_tail<V>(r[k], c0 + (int64_t)vi * V, L);
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) r[k][i] = neg_inf();
      }
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
  }
  __syncthreads();
  float r[RV][V];
  if (row_first < rows) {
    const int s_nv0 = min(a_nv, valid_vectors(length_of(row_first)));
    for (int p = 0; p < NP; ++p) fill_piece(row_first, s_nv0, p);
    load_regs(row_first, r);
  }

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
    const int next_s_nv = next_row < rows ? min(a_nv, valid_vectors(length_of(next_row))) : 0;

    // Pass 1a: exact maximum of the on-chip part, pieces processed as they land.
    float mx = neg_inf();
    for (int p = 0; p < NP; ++p) {
      if constexpr (TMA) {
        // after one wait has run out, later waits get a single poll each
        if (!mbar_wait_bounded(smem_addr(&bars[p]), (uint32_t)par, timed_out ? 1 : max_polls))
          timed_out = true;
      } else {
        cp_async_wait_dyn(NP - 1 - p);  // this thread's copies of pieces 0..p have landed
      }
      const int p1 = piece_end(p, s_nv);
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

    // Pass 1b: sum of e^(x - m_c) over the on-chip part.
    float sum = 0.0f;
    if (KEEP_E && m_c != neg_inf()) {
      for (int p = 0; p < NP; ++p) {
        const int p1 = piece_end(p, s_nv);
        for (int vi = p * P + t; vi < p1; vi += T) {
          float f[V];
          staged_vec<InT, V>(sx, vi, v_full, c0 + (int64_t)vi * V, L, f);
#pragma unroll
          for (int i = 0; i < V; i += 2) exp_shift_accurate2(f[i], f[i + 1], m_c, f[i], f[i + 1]);
          *reinterpret_cast<float4*>(se + (int64_t)vi * V) = make_float4(f[0], f[1], f[2], f[3]);
          sum = __fadd_rn(sum, __fadd_rn(__fadd_rn(f[0], f[1]), __fadd_rn(f[2], f[3])));
        }
      }
#pragma unroll
      for (int k = 0; k < RV; ++k) {
#pragma unroll
        for (int i = 0; i < V; i += 2) exp_shift_accurate2(r[k][i], r[k][i + 1], m_c, r[k][i], r[k][i + 1]);
        sum = __fadd_rn(sum, __fadd_rn(__fadd_rn(r[k][0], r[k][1]), __fadd_rn(r[k][2], r[k][3])));
      }
    } else if (m_c != neg_inf()) {
      // one FFMA + exp2 per element; the rounding of c = -m_c log2 e, common to
      // every term, is corrected once (stats_correct)
      const bool huge = !(fabsf(m_c) < 1e38f);
      const float c = huge ? 0.0f : __fmul_rn(-m_c, L2E_HI);
      const float msub = huge ? m_c : 0.0f;
      auto add_terms = [&](const float (&f)[V]) {
        float e[V];
#pragma unroll
        for (int i = 0; i < V; ++i) e[i] = ex2_ftz(__fmaf_rn(__fsub_rn(f[i], msub), L2E_HI, c));
#pragma unroll
        for (int w = V / 2; w > 0; w >>= 1)
#pragma unroll
          for (int i = 0; i < w; ++i) e[i] = __fadd_rn(e[i], e[i + w]);
        sum = __fadd_rn(sum, e[0]);
      };
      for (int p = 0; p < NP; ++p) {
        const int p1 = piece_end(p, s_nv);
        for (int vi = p * P + t; vi < p1; vi += T) {
          float f[V];
          staged_vec<InT, V>(sx, vi, v_full, c0 + (int64_t)vi * V, L, f);
          add_terms(f);
        }
      }
#pragma unroll
      for (int k = 0; k < RV; ++k) add_terms(r[k]);
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
    // CTA summary.  Every thread's on-chip sum is relative to the same m_c, so
    // without a streamed remainder the summary is (m_c, plain sum); with one,
    // the threads' (m, d) pairs are merged.
    MD md;
    if (b_nv >= v_nv) {
      float ssum = warp_sum(sum);
      __syncthreads();  // s_m is reused
      if (lane == 0) s_d[warp] = ssum;
      __syncthreads();
      md = MD{m_c, warp_sum(lane < (T >> 5) ? s_d[lane] : 0.0f)};
    } else {
      md = warp_merge(md_merge(MD{m_c, sum}, MD{m_s, d_s}));
      __syncthreads();  // s_m is reused
      if (lane == 0) {
        s_m[warp] = md.m;
        s_d[warp] = md.d;
      }
      __syncthreads();
      md = warp_merge(lane < (T >> 5) ? MD{s_m[lane], s_d[lane]} : MD{neg_inf(), 0.0f});
    }
    // push this CTA's summary into slot [par][crank] of every CTA of the cluster
    if (warp == 0 && lane < (int)csize) {
      st_peer_f32(&s_all[par][crank][0], lane, md.m);
      st_peer_f32(&s_all[par][crank][1], lane, md.d);
    }
    if constexpr (MODE == MODE_STATS) {
      // all staged reads are done (the barriers above): refill every piece now
      if (next_row < rows && !timed_out)
        for (int p = 0; p < NP; ++p) fill_piece(next_row, next_s_nv, p);
    }
    // Exchange through distributed shared memory: the pushes above, then one
    // cluster barrier (release/acquire) makes every summary visible locally.
    // The slots alternate by row parity: slot par of every CTA is read before
    // that CTA reaches the next row's barrier, and is written again only two
    // rows later, after that barrier.
    __syncwarp();
    cluster_arrive();
    cluster_wait();
    MD all{neg_inf(), 0.0f};
    if (lane < (int)csize) all = MD{s_all[par][lane][0], s_all[par][lane][1]};
    all = warp_merge(all);  // rank order, identical bits in every lane

    const float M = all.m, D = all.d;
    if constexpr (MODE == MODE_STATS) {
      if (crank == 0 && t == 0) {
        m_out[row] = M;
        d_out[row] = M == neg_inf() ? 0.0f : D;
      }
      if (next_row < rows) load_regs(next_row, r);
    } else {
      OutT* yr = y + row * cols + c0;
      const bool zero_row = (M == neg_inf());
      const bool nan_row = !zero_row && (D != D);
      const OutConst kc = make_out_const<OutT>(M, D);
      // KEEP_E: e^(m_c - M) / D, the one factor between a kept e and y
      const float scale_c = (m_c == neg_inf() || zero_row || nan_row)
                                ? 0.0f
                                : __fmul_rn(rescale_factor(m_c, M), kc.rD);
      // f holds kept exponentials (is_e: the on-chip part with KEEP_E) or inputs
      auto emit = [&](int vi, const float (&f)[V], bool valid_vec, bool is_e) {
        float pv[V];
        if (!zero_row && !nan_row) {
          if (KEEP_E && is_e) {
#pragma unroll
            for (int i = 0; i < V; ++i) pv[i] = valid_vec ? __fmul_rn(f[i], scale_c) : 0.0f;
          } else {
            out_values<OutT, V>(f, kc, pv);
#pragma unroll
            for (int i = 0; i < V; ++i) pv[i] = valid_vec ? pv[i] : 0.0f;
          }
        } else {
          const int64_t e0 = c0 + (int64_t)vi * V;
#pragma unroll
          for (int i = 0; i < V; ++i) pv[i] = (nan_row && e0 + i < L) ? qnan() : 0.0f;
        }
        store_vec<OutT, V>(yr + (int64_t)vi * V, pv);
      };
      for (int p = 0; p < NP; ++p) {
        const int p1 = piece_end(p, a_nv);
        for (int vi = p * P + t; vi < p1; vi += T) {
          float f[V];
          const bool valid_vec = vi < s_nv;
          if (valid_vec) {
            if constexpr (KEEP_E) {
              const float4 e4 = *reinterpret_cast<const float4*>(se + (int64_t)vi * V);
              f[0] = e4.x; f[1] = e4.y; f[2] = e4.z; f[3] = e4.w;
            } else {
              staged_vec<InT, V>(sx, vi, v_full, c0 + (int64_t)vi * V, L, f);
            }
          }
          emit(vi, f, valid_vec, true);
        }
        // piece p is consumed: refill it with the next row (TMA: after every
        // thread is done with it; a wait of thread 0 that ran out leaves that
        // barrier's phase pending, and a second arrive on it is not allowed)
        if constexpr (TMA) __syncthreads();
        if (next_row < rows && !timed_out) fill_piece(next_row, next_s_nv, p);
      }
#pragma unroll
      for (int k = 0; k < RV; ++k) {
        const int vi = a_nv + k * T + t;
        if (vi < b_nv) emit(vi, r[k], vi < v_nv, true);
      }
      if (next_row < rows) load_regs(next_row, r);  // in flight while the remainder is written
      for (int vi = b_nv + t; vi < c_nv; vi += T) {  // streamed remainder, second read
        float f[V];
        const bool valid_vec = vi < v_nv;
        if (valid_vec) {
          load_vec16<InT>(xr + (int64_t)vi * V, f);
          if (vi >= v_full) mask_tail<V>(f, c0 + (int64_t)vi * V, L);
        }
        emit(vi, f, valid_vec, false);
      }
    }
  }

  if constexpr (TMA) {
    if (timed_out) {
      atomicOr(status, DEV_TIMEOUT);
      // Thread 0 issued every copy.  After its own wait ran out it stopped
      // refilling, so each piece has at most one phase still pending: the one
      // its last issued fill completes (fill k completes phase k, parity k & 1).
      // Let those copies land before this CTA's shared memory is released.
      if (t == 0 && row_first < rows)
        for (int p = 0; p < NP; ++p)
          mbar_wait_bounded(smem_addr(&bars[p]), ((fill_par >> p) & 1u) ^ 1u, int64_t(1) << 21);
    }
  } else {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
  }
  // no CTA leaves while a peer may still read its last summary
  __syncwarp();
  cluster_arrive();
  cluster_wait();
}

}  // namespace smx
