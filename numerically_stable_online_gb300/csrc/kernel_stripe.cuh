// Long rows read once: every row is cut into Q column stripes, one per CTA of
// a row group, and each CTA keeps its stripe on chip from the summary to the
// normalisation.
//
// The pages' long-row answer is the block summary: each block of a row gets
// its own (m, d), the summaries are merged by rescaling both sums to the
// larger maximum, and the merged pair normalises every block ("Stable softmax:
// keep the normalizer consistent as tiles arrive", third paragraph; "Online
// stable softmax", "Derive the update for two blocks").  The traffic account
// asks that a row be read once and written once where on-chip capacity allows
// ("Softmax numerics architecture...", "Fusion and the memory-traffic
// account"; "Kernel visualization: online softmax", "Tiled version").  Here a
// block is a column stripe of about row_bytes / Q, and on-chip capacity is the
// shared memory of all the SMs together:
//
//   - A persistent cooperative grid of groups x Q CTAs (every CTA resident).
//     Group g takes rows g, g + groups, ...; CTA q of a group always owns
//     vectors [q nvec / Q, (q + 1) nvec / Q) of its rows.
//   - Compute thread 0 keeps the stripes of the next rows in flight: one bulk
//     copy (cp.async.bulk global -> shared, no multicast) per stripe into a
//     ring of NSLOT shared-memory slots, one mbarrier each.
//   - Compute warps, row i: the exact stripe maximum m_q, then sum e^(x - m_q);
//     fp32 inputs with fp32 outputs keep the compensated exponentials in the
//     slot.  The pair (m_q, d_q) goes to the sync warps through a shared
//     word and an mbarrier.  Then they normalise row i - LAG from the slot it
//     still occupies (its (M, D) arrive from the sync warps) and store it: one
//     HBM read and one HBM write per element.
//   - Two sync warps, alternating rows: publish (m_q, d_q) to global memory
//     and count it into the row's completion counter (release), wait for the
//     row's Q stripes (relaxed polls, then an acquire fence; bounded), merge
//     the Q summaries in rank order (identical bits in every CTA), and hand the
//     row's constants to the compute warps.  The compute warps never wait on a
//     global-memory round trip: LAG rows of slack cover the exchange.
//
// Modes: softmax, log_softmax, and cross-entropy with its gradient (the loss
// is written by the thread holding x_t).  Every wait is bounded; a wait that
// runs out records SMX_ERR_TIMEOUT in the device status word, and thread 0
// lets its own bulk copies land before the CTA exits.
#pragma once

#include "kernel_stream.cuh"
#include "smx_async.cuh"
#include "smx_launch.h"

namespace smx {

struct StripeArgs {
  int64_t rows, cols;
  int Q;            // stripes (CTAs) per row
  int groups;       // row groups; the grid is groups x Q CTAs
  int nslots;       // shared-memory ring slots
  int slot_vecs;    // 16-byte vectors per slot (>= the longest stripe)
  float2* sums;     // [rows][Q] stripe summaries (m, d)
  unsigned* count;  // [rows] stripes published (zero at launch)
  unsigned* count_next;  // the other counter array: zeroed here for the next call
  int64_t count_next_n;
  const int64_t* target;  // cross-entropy
  float* loss;
  int64_t max_polls;  // bound of each wait
  int64_t probe;      // > 0: the sync warps wait for one stripe more than exists (the error-path probe)
  int* status;
};

// The row constants the sync warps hand to the compute warps.
struct StripeRow {
  float M, D, ld;  // merged maximum and sum, log D
  float F;         // kept exponentials: e^(m_q - M) / D (0 for an empty stripe)
  OutConst kc;     // recomputed exponentials: constants of out_value
  int zero_row, nan_row;
};

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ float2 ld_cg_f2(const float2* p) {
  float2 v;
  asm volatile("ld.global.cg.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p) : "memory");
  return v;
}

template <typename InT, typename OutT, int MODE>
struct StripePolicy {
  // fp32 in and out: the compensated exponentials of the sum pass are kept in
  // the slot, in place of x, and the normalisation is one multiply
  static constexpr bool KEEP_E = (MODE == MODE_SOFTMAX || MODE == MODE_CE) &&
                                 ExpPolicy<OutT, MODE_SOFTMAX>::ACCURATE &&
                                 std::is_same<InT, float>::value;
};

template <typename InT, typename OutT, int MODE>
__global__ void __launch_bounds__(STRIPE_THREADS, 1)
    k_rows_stripe(const InT* __restrict__ x, OutT* __restrict__ y, StripeArgs a,
                  const int32_t* __restrict__ valid_len) {
  static_assert(MODE == MODE_SOFTMAX || MODE == MODE_LOG || MODE == MODE_CE, "modes of the stripe kernel");
  constexpr int V = Elem<InT>::V;
  constexpr bool KEEP_E = StripePolicy<InT, OutT, MODE>::KEEP_E;
  constexpr int LAG = STRIPE_LAG, RING = STRIPE_RING;
  extern __shared__ __align__(128) uint4 slots[];  // [nslots][slot_vecs]
  __shared__ __align__(8) uint64_t full_bar[STRIPE_MAX_SLOTS];
  __shared__ __align__(8) uint64_t summ_bar[RING], row_bar[RING];
  __shared__ int64_t slot_len[STRIPE_MAX_SLOTS];    // the row's valid length
  __shared__ long long slot_t[STRIPE_MAX_SLOTS];    // cross-entropy: the target, -1 if ignored
  __shared__ float slot_xt[STRIPE_MAX_SLOTS];       // cross-entropy: x_t when this stripe holds it
  __shared__ float2 summ[RING];
  __shared__ StripeRow rowc[RING];
  __shared__ float s_max[2][32], s_sum[32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NC = (int)(blockDim.x >> 5) - STRIPE_SYNC_WARPS;  // compute warps
  const int TC = NC * 32;
  const int grp = (int)(blockIdx.x / (unsigned)a.Q), q = (int)(blockIdx.x % (unsigned)a.Q);
  const int64_t nvec = a.cols / V;
  const int64_t sv0 = (int64_t)q * nvec / a.Q, sv1 = (int64_t)(q + 1) * nvec / a.Q;
  const int nvq = (int)(sv1 - sv0);     // vectors of this stripe
  const int64_t col0 = sv0 * V;          // its first column
  const int64_t nr = grp < a.rows ? (a.rows - 1 - grp) / a.groups + 1 : 0;  // rows of this group
  const int nslots = a.nslots;
  auto row_of = [&](int64_t i) -> int64_t { return grp + i * a.groups; };
  // elements of the stripe inside a row's valid prefix L
  auto stripe_valid = [&](int64_t L) -> int {
    const int64_t v = L - col0;
    return (int)(v < 0 ? 0 : (v > (int64_t)nvq * V ? (int64_t)nvq * V : v));
  };

  // the counters of the next call start at zero
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + tid; i < a.count_next_n;
       i += (int64_t)gridDim.x * blockDim.x)
    a.count_next[i] = 0;

  if (tid == 0) {
    for (int s = 0; s < nslots; ++s) mbar_init(smem_addr(&full_bar[s]), 1);
    for (int k = 0; k < RING; ++k) {
      mbar_init(smem_addr(&summ_bar[k]), 1);
      mbar_init(smem_addr(&row_bar[k]), 1);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp < NC) {
    // ------------------------------------------------------------ compute warps
    const int c = tid;
    int64_t filled = -1;  // thread 0: the last row whose stripe copy was issued
    // thread 0 loads the next fill's row length (and target) one fill ahead,
    // so that issuing a copy never waits on a global load
    int64_t next_L = a.cols;
    long long next_t = -1;
    auto load_row_values = [&](int64_t i) {
      if (i >= nr) return;
      const int64_t row = row_of(i);
      next_L = a.cols;
      if (valid_len != nullptr) {
        const int64_t v = __ldg(valid_len + row);
        next_L = v < 0 ? 0 : (v > a.cols ? a.cols : v);
      }
      if constexpr (MODE == MODE_CE) next_t = __ldg(a.target + row);
    };
    // stripe of local row i into slot i % nslots (compute thread 0; rows in order)
    auto fill = [&](int64_t i) {
      const int s = (int)(i % nslots);
      const int64_t row = row_of(i);
      const int64_t L = next_L;
      slot_len[s] = L;
      if constexpr (MODE == MODE_CE) slot_t[s] = (next_t < 0 || next_t >= L) ? -1 : next_t;
      const int nv = (stripe_valid(L) + V - 1) / V;
      // the slot's earlier generic-proxy reads and writes come before the copy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      const uint32_t bar = smem_addr(&full_bar[s]);
      if (nv > 0) {
        mbar_arrive_expect_tx(bar, (uint32_t)nv * 16u);
        bulk_load_g2s(smem_addr(slots + (size_t)s * a.slot_vecs), x + row * a.cols + col0,
                      (uint32_t)nv * 16u, bar);
      } else {
        mbar_arrive(bar);  // an empty stripe: the phase completes with no bytes
      }
      filled = i;
      load_row_values(i + 1);
    };
    if (c == 0) {
      load_row_values(0);
      for (int64_t i = 0; i < nslots && i < nr; ++i) fill(i);
    }

    bool timed_out = false;  // after one wait ran out, later waits poll once
    int par = 0;
    for (int64_t i = 0; i < nr + LAG; ++i, par ^= 1) {
      if (i < nr) {
        // ---- the stripe of row i: exact maximum, then its sum
        const int s = (int)(i % nslots);
        if (!mbar_wait_bounded(smem_addr(&full_bar[s]), (uint32_t)((i / nslots) & 1),
                               timed_out ? 1 : a.max_polls))
          timed_out = true;
        const int Lv = stripe_valid(slot_len[s]);
        const InT* sx = reinterpret_cast<const InT*>(slots + (size_t)s * a.slot_vecs);
        float mx = neg_inf();
        for (int k = c; k * V < Lv; k += TC) {
          float f[V];
          load_masked<InT, true>(sx + k * V, k * V, Lv, f);
#pragma unroll
          for (int u = 0; u < V; ++u) mx = fmax_nan(mx, f[u]);
        }
        mx = warp_max_nan(mx);
        if (lane == 0) s_max[par][warp] = mx;
        named_bar_sync(1, TC);
        const float mq = warp_max_nan(lane < NC ? s_max[par][lane] : neg_inf());
        // every compute thread has normalised row i - LAG - 1 (previous
        // iteration): its slot takes the row nslots later
        if (c == 0 && !timed_out) {  // after a wait ran out, thread 0 issues no more copies
          const int64_t j = i - LAG - 1;
          if (j >= 0 && j + nslots < nr) fill(j + nslots);
        }
        if constexpr (MODE == MODE_CE) {
          // x_t, kept by the thread that holds it before the slot's x may be overwritten
          const int64_t t = slot_t[s] - col0;
          if (t >= 0 && t < Lv && (int)(t / V) % TC == c)
            slot_xt[s] = Elem<InT>::to_f32(sx[t]);
        }
        float dq = 0.0f;
        if (mq != neg_inf()) {
          float sum = 0.0f;
          for (int k = c; k * V < Lv; k += TC) {
            float f[V];
            load_masked<InT, true>(sx + k * V, k * V, Lv, f);
            if constexpr (KEEP_E) {
#pragma unroll
              for (int u = 0; u < V; u += 2) exp_shift_accurate2(f[u], f[u + 1], mq, f[u], f[u + 1]);
              *reinterpret_cast<float4*>(slots + (size_t)s * a.slot_vecs + k) = make_float4(f[0], f[1], f[2], f[3]);
              sum = __fadd_rn(sum, __fadd_rn(__fadd_rn(f[0], f[1]), __fadd_rn(f[2], f[3])));
            } else {
              float g1[1][V];
#pragma unroll
              for (int u = 0; u < V; ++u) g1[0][u] = f[u];
              sum = __fadd_rn(sum, sum_exp<1, V>(g1, mq));
            }
          }
          sum = warp_sum(sum);
          if (lane == 0) s_sum[warp] = sum;
          named_bar_sync(1, TC);
          const float S = warp_sum(lane < NC ? s_sum[lane] : 0.0f);
          dq = KEEP_E ? S : stats_correct(S, mq);
        }
        if (c == 0) {
          summ[i % RING] = make_float2(mq, dq);
          mbar_arrive(smem_addr(&summ_bar[i % RING]));
        }
      }
      if (i >= LAG) {
        // ---- normalise row r = i - LAG from its slot
        const int64_t r = i - LAG;
        const int s = (int)(r % nslots), kr = (int)(r % RING);
        if (!mbar_wait_bounded(smem_addr(&row_bar[kr]), (uint32_t)((r / RING) & 1),
                               timed_out ? 1 : a.max_polls))
          timed_out = true;
        const StripeRow rc = rowc[kr];
        const int Lv = stripe_valid(slot_len[s]);
        const int64_t row = row_of(r);
        OutT* yr = y + row * a.cols + col0;
        const InT* sx = reinterpret_cast<const InT*>(slots + (size_t)s * a.slot_vecs);
        const float* se = reinterpret_cast<const float*>(slots + (size_t)s * a.slot_vecs);
        bool zero_out = rc.zero_row, nan_out = rc.nan_row;
        int64_t tl = -1;
        if constexpr (MODE == MODE_CE) {
          const bool ignored = slot_t[s] < 0;
          nan_out = !ignored && (rc.zero_row || rc.nan_row);
          zero_out = ignored;
          tl = ignored ? -1 : slot_t[s] - col0;
          if (tl >= Lv) tl = -1;  // the target lies in another stripe (or before this one: tl < 0)
        }
        for (int k = c; k < nvq; k += TC) {
          const int e0 = k * V;
          float o[V];
          if constexpr (MODE == MODE_LOG) {
            if (nan_out || zero_out) {
#pragma unroll
              for (int u = 0; u < V; ++u) o[u] = (nan_out && e0 + u < Lv) ? qnan() : neg_inf();
            } else {
              float f[V];
              load_masked<InT, true>(sx + e0, e0, Lv, f);
              const unsigned long long nm = pk(-rc.M, -rc.M), nl = pk(-rc.ld, -rc.ld);
#pragma unroll
              for (int u = 0; u < V; u += 2) {
                const unsigned long long t2 = add2(add2(pk(f[u], f[u + 1]), nm), nl);
                o[u] = pk_lo(t2);
                o[u + 1] = pk_hi(t2);
              }
            }
          } else {
            // (kept exponentials: F = 0 also for a stripe with no finite
            // element, whose slot still holds x)
            if (nan_out || zero_out || e0 >= Lv || (KEEP_E && rc.F == 0.0f)) {
#pragma unroll
              for (int u = 0; u < V; ++u) o[u] = (nan_out && e0 + u < Lv) ? qnan() : 0.0f;
            } else if constexpr (KEEP_E) {
              const float4 e4 = *reinterpret_cast<const float4*>(se + e0);
              const float ev[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
              for (int u = 0; u < V; ++u) o[u] = e0 + u < Lv ? __fmul_rn(ev[u], rc.F) : 0.0f;
            } else {
              float f[V];
              load_masked<InT, true>(sx + e0, e0, Lv, f);
              out_values<OutT, V>(f, rc.kc, o);
            }
          }
          store_vec<OutT, V>(yr + e0, o);
        }
        if constexpr (MODE == MODE_CE) {
          if (tl >= 0 && (int)(tl / V) % TC == c) {
            // the owner of x_t: the loss, and p_t - 1 over its own store of p_t
            const bool bad = rc.zero_row || rc.nan_row;
            const float xt = slot_xt[s];
            a.loss[row] = bad ? qnan() : __fadd_rn(__fsub_rn(rc.M, xt), rc.ld);
            if (!bad) {
              float pt;
              if constexpr (KEEP_E) {
                pt = __fmul_rn(se[tl], rc.F);
              } else {
                pt = out_value<OutT>(xt, rc.kc);
              }
              yr[tl] = Elem<OutT>::from_f32(__fsub_rn(pt, 1.0f));
            }
          }
          if (slot_t[s] < 0 && q == 0 && c == 0) a.loss[row] = 0.0f;
        }
      }
    }
    if (c == 0 && filled >= 0 && timed_out) {
      // a wait ran out and the ring stopped: let the copies still in flight
      // land before this CTA's shared memory is released (each slot's last
      // issued fill is its pending phase, if any)
      for (int s = 0; s < nslots; ++s) {
        int64_t j = filled - ((filled - s) % nslots + nslots) % nslots;  // last row filled into slot s
        if (j >= 0) mbar_wait_bounded(smem_addr(&full_bar[s]), (uint32_t)((j / nslots) & 1), int64_t(1) << 21);
      }
    }
  } else {
    // --------------------------------------------------------------- sync warps
    const int sw = warp - NC;
    const unsigned need = (unsigned)a.Q + (a.probe > 0 ? 1u : 0u);
    const int64_t polls_max = a.probe > 0 ? a.probe : a.max_polls;
    bool timed_out = false;
    for (int64_t r = sw; r < nr; r += STRIPE_SYNC_WARPS) {
      const int kr = (int)(r % RING);
      if (!mbar_wait_bounded(smem_addr(&summ_bar[kr]), (uint32_t)((r / RING) & 1),
                             timed_out ? 1 : a.max_polls))
        timed_out = true;
      const float2 mine = summ[kr];
      const int64_t row = row_of(r);
      float2* rs = a.sums + row * a.Q;
      int late = 0;
      if (lane == 0) {
        rs[q] = mine;
        red_release_add(a.count + row, 1u);
        int64_t polls = 0;
        while (ld_relaxed_u32(a.count + row) < need) {
          if (timed_out || ++polls > polls_max) {
            late = 1;
            break;
          }
          __nanosleep(32);
        }
        fence_acq_rel_gpu();  // the summaries counted above are visible from here on
        if (late) atomicOr(a.status, DEV_TIMEOUT);
      }
      if (__shfl_sync(0xffffffffu, late, 0)) timed_out = true;
      __syncwarp();
      float2 b[STRIPE_MAX_Q / 32];
#pragma unroll
      for (int u = 0; u < STRIPE_MAX_Q / 32; ++u) {
        const int t = lane + 32 * u;
        b[u] = t < a.Q ? ld_cg_f2(rs + t) : make_float2(neg_inf(), 0.0f);
      }
      MD acc{neg_inf(), 0.0f};
#pragma unroll
      for (int u = 0; u < STRIPE_MAX_Q / 32; ++u) acc = md_merge(acc, MD{b[u].x, b[u].y});
      acc = warp_merge(acc);  // rank order: the same bits in every CTA of the group
      if (lane == 0) {
        StripeRow rc;
        rc.M = acc.m;
        rc.D = acc.d;
        rc.zero_row = acc.m == neg_inf();
        rc.nan_row = !rc.zero_row && (acc.d != acc.d || acc.m != acc.m || acc.m == pos_inf());
        rc.ld = rc.zero_row ? 0.0f : logf(acc.d);
        if constexpr (MODE != MODE_LOG) {
          rc.kc = make_out_const<OutT>(acc.m, acc.d);
          rc.F = (mine.x == neg_inf() || rc.zero_row || rc.nan_row)
                     ? 0.0f
                     : __fmul_rn(rescale_factor(mine.x, acc.m), rc.kc.rD);
        } else {
          rc.F = 0.0f;
        }
        rowc[kr] = rc;
        mbar_arrive(smem_addr(&row_bar[kr]));
      }
      __syncwarp();
    }
  }
}

}  // namespace smx
