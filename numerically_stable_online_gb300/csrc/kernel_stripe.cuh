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
// block is what one warp holds of a column stripe, and on-chip capacity is the
// shared memory of all the SMs together:
//
//   - A persistent cooperative grid of groups x Q CTAs (every CTA resident).
//     Group g takes rows g, g + groups, ...; CTA q of a group always owns
//     vectors [q nvec / Q, (q + 1) nvec / Q) of its rows.
//   - The producer warp keeps the stripes of the next rows in flight: one bulk
//     copy (cp.async.bulk global -> shared, no multicast) per stripe into a
//     ring of shared-memory slots, one mbarrier each; a slot is refilled once
//     every compute warp has signalled (another mbarrier) that it is done with
//     the row it held.
//   - Compute warps, each on its own (no block barrier): row i, the warp's
//     part of the stripe into registers once, its exact maximum m_w, then
//     sum e^(x - m_w); fp32 inputs with fp32 outputs keep those compensated
//     exponentials in the slot.  (m_w, d_w) goes to the publisher warp through
//     shared memory and an mbarrier.  Then the warp normalises row i - LAG
//     from the slot, with its own factor e^(m_w - M) / D once the row's (M, D)
//     has arrived: one HBM read and one HBM write per element.
//   - The publisher warp folds the warps' pairs into the stripe's (m_q, d_q),
//     stores it in global memory and counts it into the row's completion
//     counter (release); it never waits on another CTA.
//   - Collector warps, rows round robin: wait for the row's Q stripes
//     (acquire polls, bounded), load the Q summaries and merge them.
//
// Every merge here, of warps and of stripes, is the pages' two-block update
// applied to all blocks at once: the maximum M exactly (a NaN-propagating warp
// maximum), then D = sum_b d_b e^(m_b - M) in a fixed order, so every CTA of a
// group gets the same bits.  Modes: softmax, log_softmax, cross-entropy
// with its gradient (the loss is written by the thread holding x_t), and the
// softmax backward ("Softmax numerics architecture...", "The Jacobian, and the
// backward pass that never divides": dx = p (g - s), s = sum g p): a slot holds
// the row's stripes of p and of g, the warps' and the stripes' partial dots are
// added in a fixed order in place of the (m, d) merge, and dx is formed from
// the slot -- two reads and one write per element.  Every
// wait is bounded; a wait that runs out records SMX_ERR_TIMEOUT in the device
// status word, and the producer lets its bulk copies land before it exits.
#pragma once

#include "kernel_stream.cuh"
#include "smx_async.cuh"
#include "smx_launch.h"

namespace smx {

// the stripe kernel's mode value of the softmax backward
constexpr int MODE_BWD = CALL_BACKWARD;

struct StripeArgs {
  int64_t rows, cols;
  int Q;            // stripes (CTAs) per row
  int groups;       // row groups; the grid is groups x Q CTAs
  int nslots;       // shared-memory ring slots
  int slot_vecs;    // 16-byte vectors per slot (>= the longest stripe; the backward: two stripes,
                    // p in the first half, g in the second)
  const void* g;    // the backward's upstream gradient (x is the forward output p)
  float2* sums;     // [rows][Q] stripe summaries (m, d)
  unsigned* count;  // [rows] stripes published (zero at launch)
  unsigned* count_next;  // the other counter array: zeroed here for the next call
  int64_t count_next_n;
  const int64_t* target;  // cross-entropy
  float* loss;
  int64_t max_polls;  // bound of each wait
  int64_t probe;      // > 0: the collectors wait for one stripe more than exists (the error-path probe)
  int lag;            // rows between a stripe's summary and its normalisation (1..STRIPE_LAG)
  int piece_bytes;    // bulk copies of at most this many bytes per stripe (0: one copy)
  int l2_ahead;       // the producer prefetches into L2 the stripe this many rows past each fill (0: off)
  int* status;
};

// The row constants a collector warp hands to the compute warps.
struct StripeRow {
  float M, D, ld;  // merged maximum and sum, log D
  OutConst kc;     // constants of out_value (its rD is 1/D)
  int zero_row, nan_row;
  float F[32];     // kept exponentials: compute warp w's factor e^(m_w - M) / D
                   // (0 when the warp held no finite element, or on a zero / NaN row)
};

// The flat merge of up to 32 summaries, one per lane (lanes without one pass
// (-inf, 0)): M the NaN-propagating maximum, D = sum d e^(m - M) over the
// lanes in butterfly order, with the merge's policy for the special maxima (a
// NaN maximum poisons both, all empty gives (-inf, 0), +inf gives (+inf, NaN)).
// Every lane returns the same bits.
__device__ __forceinline__ MD warp_flat_merge(float m, float d) {
  const float M = warp_max_nan(m);
  if (M != M) return MD{qnan(), qnan()};
  if (M == neg_inf()) return MD{neg_inf(), 0.0f};
  if (M == pos_inf()) return MD{pos_inf(), qnan()};
  const float t = m == neg_inf() ? 0.0f : __fmul_rn(d, rescale_factor(m, M));
  return MD{M, warp_sum(t)};
}
__device__ __forceinline__ float2 ld_cg_f2(const float2* p) {
  float2 v;
  asm volatile("ld.global.cg.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p) : "memory");
  return v;
}

// SMX_STRIPE_TRACE (a build-time diagnostic, off in the library build): the
// kernel stamps %globaltimer at its waits, per CTA and row, into a device
// array read back with smx_debug_stripe_trace().
#ifdef SMX_STRIPE_TRACE
constexpr int STRIPE_TRACE_CTAS = 160, STRIPE_TRACE_ROWS = 256, STRIPE_TRACE_EVENTS = 8;
__device__ unsigned long long g_stripe_trace[STRIPE_TRACE_CTAS][STRIPE_TRACE_ROWS][STRIPE_TRACE_EVENTS];
__device__ __forceinline__ void stripe_stamp(int64_t r, int ev) {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  if (blockIdx.x < STRIPE_TRACE_CTAS && r < STRIPE_TRACE_ROWS) g_stripe_trace[blockIdx.x][r][ev] = t;
}
#define SMX_STAMP(r, ev) stripe_stamp((r), (ev))
#else
#define SMX_STAMP(r, ev) ((void)0)
#endif

template <typename InT, typename OutT, int MODE>
struct StripePolicy {
  // fp32 in and out: the compensated exponentials of the sum pass are kept in
  // the slot, in place of x, and the normalisation is one multiply
  static constexpr bool KEEP_E = (MODE == MODE_SOFTMAX || MODE == MODE_CE) &&
                                 ExpPolicy<OutT, MODE_SOFTMAX>::ACCURATE &&
                                 std::is_same<InT, float>::value;
};

template <typename InT, typename OutT, int MODE, int VPT>
__global__ void __launch_bounds__(STRIPE_THREADS, 1)
    k_rows_stripe(const InT* __restrict__ x, OutT* __restrict__ y, StripeArgs a,
                  const int32_t* __restrict__ valid_len) {
  static_assert(MODE == MODE_SOFTMAX || MODE == MODE_LOG || MODE == MODE_CE || MODE == MODE_BWD,
                "modes of the stripe kernel");
  constexpr bool BWD = MODE == MODE_BWD;
  constexpr int V = Elem<InT>::V;
  constexpr bool KEEP_E = StripePolicy<InT, OutT, MODE>::KEEP_E;
  constexpr int RING = STRIPE_RING;
  const int LAG = a.lag;
  constexpr int NC = STRIPE_COMPUTE_WARPS;
  constexpr int TC = NC * 32;
  extern __shared__ __align__(128) uint4 slots[];  // [nslots][slot_vecs]
  __shared__ __align__(8) uint64_t full_bar[STRIPE_MAX_SLOTS], free_bar[STRIPE_MAX_SLOTS];
  __shared__ __align__(8) uint64_t summ_bar[RING], row_bar[RING];
  __shared__ int64_t slot_len[STRIPE_MAX_SLOTS];    // the row's valid length
  __shared__ long long slot_t[STRIPE_MAX_SLOTS];    // cross-entropy: the target, -1 if ignored
  __shared__ float slot_xt[STRIPE_MAX_SLOTS];       // cross-entropy: x_t when this stripe holds it
  __shared__ float2 warp_md[RING][32];              // each compute warp's (m_w, d_w) of a row
  __shared__ int warp_fast[RING][32];               // ... and whether it kept fast exponentials
  __shared__ StripeRow rowc[RING];
  __shared__ uint4 neg_vec;                         // a vector of -inf (read in place of vectors past the stripe)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = (int)(blockIdx.x / (unsigned)a.Q), q = (int)(blockIdx.x % (unsigned)a.Q);
  const int64_t nvec = a.cols / V;
  const int64_t sv0 = (int64_t)q * nvec / a.Q, sv1 = (int64_t)(q + 1) * nvec / a.Q;
  const int nvq = (int)(sv1 - sv0);     // vectors of this stripe (<= VPT * TC)
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
    const unsigned ninf = std::is_same<InT, float>::value ? 0xff800000u
                          : (std::is_same<InT, __half>::value ? 0xfc00fc00u : 0xff80ff80u);
    neg_vec = make_uint4(ninf, ninf, ninf, ninf);
    for (int s = 0; s < nslots; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&free_bar[s]), NC);
    }
    for (int k = 0; k < RING; ++k) {
      mbar_init(smem_addr(&summ_bar[k]), NC);
      mbar_init(smem_addr(&row_bar[k]), 1);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp < NC) {
    // ------------------------------------------------------------ compute warps
    // Thread c holds vectors c, c + TC, ... of the stripe; those at or past
    // nvq are read clamped to the stripe's last vector and discarded.  The
    // per-vector work is branch-free: the row-uniform cases (a stripe cut by
    // the valid prefix, zero and NaN rows) are decided once per row.
    const int c = tid;
    bool timed_out = false;  // after one wait ran out, later waits poll once
    // slots, fill parities and rows of rows i and i - LAG, kept incrementally
    // (no division in the loop)
    int sA = 0, sB = 0;
    uint32_t pA = 0;
    int64_t rowA = grp, rowB = grp;
    for (int64_t i = 0; i < nr + LAG; ++i) {
      if (i < nr) {
        // ---- row i: this warp's part of the stripe, its maximum, its sum
        const int s = sA, kr = (int)(i & (RING - 1));
        if (c == 0) SMX_STAMP(i, 0);
        if (!mbar_wait_bounded(smem_addr(&full_bar[s]), pA, timed_out ? 1 : a.max_polls))
          timed_out = true;
        if (c == 0) SMX_STAMP(i, 1);
        const int Lv = stripe_valid(slot_len[s]);
        const bool cut = Lv != nvq * V;  // the valid prefix ends inside the stripe
        uint4* sv = slots + (size_t)s * a.slot_vecs;
        if constexpr (BWD) {
          // this warp's part of sum g p over the valid lanes (an FMA chain per
          // thread, then the warp's butterfly)
          const uint4* sg = sv + a.slot_vecs / 2;
          float acc = 0.0f;
#pragma unroll
          for (int j = 0; j < VPT; ++j) {
            const int k = j * TC + c;
            if (k < nvq) {
              float fp[V], fg[V];
              unpack16<InT>(sv[k], fp);
              unpack16<InT>(sg[k], fg);
#pragma unroll
              for (int u = 0; u < V; ++u)
                if (!cut || k * V + u < Lv) acc = __fmaf_rn(fg[u], fp[u], acc);
            }
          }
          const float dw = warp_sum(acc);
          if (lane == 0) {
            warp_md[kr][warp] = make_float2(dw, 0.0f);
            mbar_arrive(smem_addr(&summ_bar[kr]));
          }
          if (++sA == nslots) {
            sA = 0;
            pA ^= 1u;
          }
          rowA += a.groups;
        } else {
        float f[VPT][V];
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
          const int k = j * TC + c;
          unpack16<InT>(*(k < nvq ? sv + k : &neg_vec), f[j]);
        }
        if (cut) {
#pragma unroll
          for (int j = 0; j < VPT; ++j)
#pragma unroll
            for (int u = 0; u < V; ++u) f[j][u] = (j * TC + c) * V + u < Lv ? f[j][u] : neg_inf();
        }
        if constexpr (MODE == MODE_CE) {
          // x_t, kept by the thread that holds it (the slot's x may be overwritten)
          const int64_t t = slot_t[s] - col0;
          const InT* sx = reinterpret_cast<const InT*>(sv);
          if (t >= 0 && t < Lv && (int)(t / V) % TC == c) slot_xt[s] = Elem<InT>::to_f32(sx[t]);
        }
        const float mw = warp_max_nan(local_max(f));
        float dw = 0.0f;
        int fast = 0;
        if (mw != neg_inf()) {
          if constexpr (KEEP_E) {
            // Kept exponentials.  When every element the warp holds lies
            // within STRIPE_FAST_RANGE of m_w, the plain form 2^(fma(x,
            // log2e_hi, c)) is accurate enough: its argument, below 16 in
            // magnitude, rounds with an error under 2^-21 (the exponential's
            // relative error stays near 3e-7 plus the unit's own 1.4e-7, and
            // log2e_hi's representation adds at most 11 * 2^-25.7), and the
            // rounding of c = RN(-m_w log2e_hi) is common to the warp: its
            // exact residual is applied to d_w here and to the warp's factor
            // by the collector.  Otherwise (a wider range, masked or special
            // values) the compensated exponential.
            float mn = f[0][0];
#pragma unroll
            for (int j = 0; j < VPT; ++j)
#pragma unroll
              for (int u = 0; u < V; u += 2) mn = fmin3(mn, f[j][u], f[j][u + 1]);
            mn = warp_min(mn);
            fast = (fabsf(mw) < 1e38f && mn >= __fsub_rn(mw, STRIPE_FAST_RANGE)) ? 1 : 0;
            unsigned long long acc = pk(0.0f, 0.0f);
            if (fast) {
              const float cw = __fmul_rn(-mw, L2E_HI);
              const unsigned long long k2 = pk(L2E_HI, L2E_HI), c2 = pk(cw, cw);
#pragma unroll
              for (int j = 0; j < VPT; ++j) {
                const int k = j * TC + c;
#pragma unroll
                for (int u = 0; u < V; u += 2) {
                  const unsigned long long uu = fma2(pk(f[j][u], f[j][u + 1]), k2, c2);
                  f[j][u] = ex2_ftz(pk_lo(uu));
                  f[j][u + 1] = ex2_ftz(pk_hi(uu));
                }
                if (k < nvq) *reinterpret_cast<float4*>(sv + k) = make_float4(f[j][0], f[j][1], f[j][2], f[j][3]);
                acc = add2(acc, add2(pk(f[j][0], f[j][1]), pk(f[j][2], f[j][3])));
              }
              dw = stats_correct(warp_sum(__fadd_rn(pk_lo(acc), pk_hi(acc))), mw);
            } else {
#pragma unroll
              for (int j = 0; j < VPT; ++j) {
                const int k = j * TC + c;
#pragma unroll
                for (int u = 0; u < V; u += 2) exp_shift_accurate2(f[j][u], f[j][u + 1], mw, f[j][u], f[j][u + 1]);
                if (k < nvq) *reinterpret_cast<float4*>(sv + k) = make_float4(f[j][0], f[j][1], f[j][2], f[j][3]);
                acc = add2(acc, add2(pk(f[j][0], f[j][1]), pk(f[j][2], f[j][3])));
              }
              dw = warp_sum(__fadd_rn(pk_lo(acc), pk_hi(acc)));
            }
          } else {
            dw = stats_correct(warp_sum(sum_exp(f, mw)), mw);
          }
        }
        if (lane == 0) {
          warp_md[kr][warp] = make_float2(mw, dw);
          warp_fast[kr][warp] = fast;
          mbar_arrive(smem_addr(&summ_bar[kr]));
        }
        if (++sA == nslots) {
          sA = 0;
          pA ^= 1u;
        }
        rowA += a.groups;
        }
      }
      if (i >= LAG) {
        // ---- normalise row r = i - LAG from its slot
        const int64_t r = i - LAG;
        const int s = sB, kr = (int)(r & (RING - 1));
        if (c == 0) SMX_STAMP(r, 2);
        if (!mbar_wait_bounded(smem_addr(&row_bar[kr]), (uint32_t)((r / RING) & 1),
                               timed_out ? 1 : a.max_polls))
          timed_out = true;
        if (c == 0) SMX_STAMP(r, 3);
        const StripeRow& rc = rowc[kr];
        const int Lv = stripe_valid(slot_len[s]);
        const bool cut = Lv != nvq * V;
        const int64_t row = rowB;
        OutT* yr = y + row * a.cols + col0;
        const uint4* sv = slots + (size_t)s * a.slot_vecs;
        if constexpr (BWD) {
          // dx = p (g - s) over the valid lanes, +0 past them
          const float sd = rc.M;
          const uint4* sg = sv + a.slot_vecs / 2;
#pragma unroll
          for (int j = 0; j < VPT; ++j) {
            const int k = j * TC + c;
            if (k < nvq) {
              float fp[V], fg[V], o[V];
              unpack16<InT>(sv[k], fp);
              unpack16<InT>(sg[k], fg);
#pragma unroll
              for (int u = 0; u < V; ++u)
                o[u] = (!cut || k * V + u < Lv) ? __fmul_rn(fp[u], __fsub_rn(fg[u], sd)) : 0.0f;
              store_vec<OutT, V>(yr + k * V, o);
            }
          }
        } else {
        bool zero_out = rc.zero_row, nan_out = rc.nan_row;
        int64_t tl = -1;
        if constexpr (MODE == MODE_CE) {
          const bool ignored = slot_t[s] < 0;
          nan_out = !ignored && (rc.zero_row || rc.nan_row);
          zero_out = ignored;
          tl = ignored ? -1 : slot_t[s] - col0;
          if (tl >= Lv) tl = -1;  // the target lies in another stripe (or before this one: tl < 0)
        }
        // kept exponentials: this warp's factor (0 also when it held no finite
        // element: its part of the slot still holds x)
        const float F = KEEP_E ? rc.F[warp] : 0.0f;
        if (zero_out || nan_out || (KEEP_E && F == 0.0f)) {
          // the policy's rows: +0 (log: -inf), NaN in the valid lanes of NaN rows
          const float fill = (MODE == MODE_LOG) ? neg_inf() : 0.0f;
#pragma unroll
          for (int j = 0; j < VPT; ++j) {
            const int k = j * TC + c;
            float o[V];
#pragma unroll
            for (int u = 0; u < V; ++u) o[u] = (nan_out && k * V + u < Lv) ? qnan() : fill;
            if (k < nvq) store_vec<OutT, V>(yr + k * V, o);
          }
        } else {
          const float M = rc.M;
#pragma unroll
          for (int j = 0; j < VPT; ++j) {
            const int k = j * TC + c;
            const uint4 raw = *(k < nvq ? sv + k : &neg_vec);  // (past the stripe: not stored)
            float o[V];
            if constexpr (KEEP_E) {
              // past the valid prefix the slot holds kept zeros (exponentials of -inf)
              const unsigned long long f2 = pk(F, F);
              const unsigned long long p0 = mul2(pk(__uint_as_float(raw.x), __uint_as_float(raw.y)), f2);
              const unsigned long long p1 = mul2(pk(__uint_as_float(raw.z), __uint_as_float(raw.w)), f2);
              o[0] = pk_lo(p0);
              o[1] = pk_hi(p0);
              o[2] = pk_lo(p1);
              o[3] = pk_hi(p1);
            } else {
              float fv[V];
              unpack16<InT>(raw, fv);
              if (cut) {
#pragma unroll
                for (int u = 0; u < V; ++u) fv[u] = k * V + u < Lv ? fv[u] : neg_inf();
              }
              if constexpr (MODE == MODE_LOG) {
                const unsigned long long nm = pk(-M, -M), nl = pk(-rc.ld, -rc.ld);
#pragma unroll
                for (int u = 0; u < V; u += 2) {
                  const unsigned long long t2 = add2(add2(pk(fv[u], fv[u + 1]), nm), nl);
                  o[u] = pk_lo(t2);
                  o[u + 1] = pk_hi(t2);
                }
              } else {
                out_values<OutT, V>(fv, rc.kc, o);
              }
            }
            if (k < nvq) store_vec<OutT, V>(yr + k * V, o);
          }
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
                pt = __fmul_rn(reinterpret_cast<const float*>(sv)[tl], F);
              } else {
                pt = out_value<OutT>(xt, rc.kc);
              }
              yr[tl] = Elem<OutT>::from_f32(__fsub_rn(pt, 1.0f));
            }
          }
          if (slot_t[s] < 0 && q == 0 && c == 0) a.loss[row] = 0.0f;
        }
        }
        // this warp is done with the slot
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&free_bar[s]));
        if (c == 0) SMX_STAMP(r, 4);
        if (++sB == nslots) sB = 0;
        rowB += a.groups;
      }
    }
  } else if (warp == NC) {
    // ----------------------------------------------------------- producer warp
    if (lane == 0) {
      bool timed_out = false;
      int64_t filled = -1;  // the last row whose stripe copy was issued
      int s = 0;            // slot of row j (kept incrementally)
      int64_t wraps = 0;    // j / nslots
      int64_t row = grp;
      for (int64_t j = 0; j < nr; ++j, row += a.groups) {
        if (j >= nslots) {
          // every compute warp has normalised row j - nslots from this slot
          if (!mbar_wait_bounded(smem_addr(&free_bar[s]), (uint32_t)((wraps - 1) & 1), a.max_polls)) {
            timed_out = true;
            break;  // stop refilling; the copies in flight are drained below
          }
        }
        int64_t L = a.cols;
        if (valid_len != nullptr) {
          const int64_t v = __ldg(valid_len + row);
          L = v < 0 ? 0 : (v > a.cols ? a.cols : v);
        }
        slot_len[s] = L;
        if constexpr (MODE == MODE_CE) {
          const int64_t t = __ldg(a.target + row);
          slot_t[s] = (t < 0 || t >= L) ? -1 : t;
        }
        const int nv = (stripe_valid(L) + V - 1) / V;
        // the slot's earlier generic-proxy reads and writes come before the copy
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        const uint32_t bar = smem_addr(&full_bar[s]);
        if (nv > 0) {
          // one expect-tx for the stripe (the backward: both stripes), then its
          // bytes in pieces of at most piece_bytes (several copies in flight)
          const uint32_t total = (uint32_t)nv * 16u;
          const uint32_t piece = a.piece_bytes > 0 ? (uint32_t)a.piece_bytes : total;
          mbar_arrive_expect_tx(bar, BWD ? 2u * total : total);
          const char* src = reinterpret_cast<const char*>(x + row * a.cols + col0);
          const uint32_t dst = smem_addr(slots + (size_t)s * a.slot_vecs);
          for (uint32_t off = 0; off < total; off += piece)
            bulk_load_g2s(dst + off, src + off, total - off < piece ? total - off : piece, bar);
          if constexpr (BWD) {
            const char* gsrc = reinterpret_cast<const char*>(static_cast<const InT*>(a.g) + row * a.cols + col0);
            const uint32_t gdst = dst + (uint32_t)(a.slot_vecs / 2) * 16u;
            for (uint32_t off = 0; off < total; off += piece)
              bulk_load_g2s(gdst + off, gsrc + off, total - off < piece ? total - off : piece, bar);
          }
        } else {
          mbar_arrive(bar);  // an empty stripe: the phase completes with no bytes
        }
        filled = j;
        SMX_STAMP(j, 5);
        // the stripe of a row further ahead, into L2 only (no shared memory)
        const int64_t jp = j + a.l2_ahead;
        if (a.l2_ahead > 0 && jp < nr && jp >= nslots) {
          const int64_t rp = row_of(jp);
          int64_t Lp = a.cols;
          if (valid_len != nullptr) {
            const int64_t v = __ldg(valid_len + rp);
            Lp = v < 0 ? 0 : (v > a.cols ? a.cols : v);
          }
          const int nvp = (stripe_valid(Lp) + V - 1) / V;
          if (nvp > 0) {
            bulk_prefetch_l2(x + rp * a.cols + col0, (uint32_t)nvp * 16u);
            if constexpr (BWD) bulk_prefetch_l2(static_cast<const InT*>(a.g) + rp * a.cols + col0, (uint32_t)nvp * 16u);
          }
        }
        if (++s == nslots) {
          s = 0;
          ++wraps;
        }
      }
      // no bulk copy may outlive the CTA: wait (bounded) for each slot's last
      // issued fill (normally long complete)
      for (int s = 0; s < nslots; ++s) {
        const int64_t j = filled - ((filled - s) % nslots + nslots) % nslots;  // last row filled into slot s
        if (j >= 0) mbar_wait_bounded(smem_addr(&full_bar[s]), (uint32_t)((j / nslots) & 1), int64_t(1) << 21);
      }
      if (timed_out) atomicOr(a.status, DEV_TIMEOUT);
    }
  } else if (warp == NC + 1) {
    // ---------------------------------------------------------- publisher warp
    bool timed_out = false;
    for (int64_t r = 0; r < nr; ++r) {
      const int kr = (int)(r % RING);
      if (!mbar_wait_bounded(smem_addr(&summ_bar[kr]), (uint32_t)((r / RING) & 1),
                             timed_out ? 1 : a.max_polls))
        timed_out = true;
      float2 outv;
      if constexpr (BWD) {
        // the warps' partial dots, added in a fixed (butterfly) order
        outv = make_float2(warp_sum(lane < NC ? warp_md[kr][lane].x : 0.0f), 0.0f);
      } else {
        const float2 p = lane < NC ? warp_md[kr][lane] : make_float2(neg_inf(), 0.0f);
        const MD md = warp_flat_merge(p.x, p.y);
        outv = make_float2(md.m, md.d);
      }
      if (lane == 0) {
        const int64_t row = row_of(r);
        a.sums[row * a.Q + q] = outv;
        red_release_add(a.count + row, 1u);
        SMX_STAMP(r, 6);
      }
      __syncwarp();
    }
  } else {
    // --------------------------------------------------------- collector warps
    const int cw = warp - NC - 2;
    const unsigned need = (unsigned)a.Q + (a.probe > 0 ? 1u : 0u);
    const int64_t polls_max = a.probe > 0 ? a.probe : a.max_polls;
    bool timed_out = false;
    for (int64_t r = cw; r < nr; r += STRIPE_COLLECT_WARPS) {
      const int kr = (int)(r % RING);
      const int64_t row = row_of(r);
      const float2* rs = a.sums + row * a.Q;
      int late = 0;
      if (lane == 0) {
        int64_t polls = 0;
        while (ld_acquire_u32(a.count + row) < need) {
          if (timed_out || ++polls > polls_max) {
            late = 1;
            break;
          }
          __nanosleep(64);
        }
        if (late) atomicOr(a.status, DEV_TIMEOUT);
        SMX_STAMP(r, 7);
      }
      if (__shfl_sync(0xffffffffu, late, 0)) timed_out = true;
      __syncwarp();  // lane 0's acquire orders the summaries for the warp
      float2 b[STRIPE_MAX_Q / 32];
#pragma unroll
      for (int u = 0; u < STRIPE_MAX_Q / 32; ++u) {
        const int t = lane + 32 * u;
        b[u] = t < a.Q ? ld_cg_f2(rs + t) : make_float2(neg_inf(), 0.0f);
      }
      if constexpr (BWD) {
        // the row's dot: each lane's partials in order, then the lanes
        float sl = 0.0f;
#pragma unroll
        for (int u = 0; u < STRIPE_MAX_Q / 32; ++u) sl = __fadd_rn(sl, lane + 32 * u < a.Q ? b[u].x : 0.0f);
        const float sd = warp_sum(sl);
        if (lane == 0) {
          StripeRow& rc = rowc[kr];
          rc.M = sd;
          rc.D = 0.0f;
          rc.zero_row = 0;
          rc.nan_row = 0;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&row_bar[kr]));
        __syncwarp();
        continue;
      }
      // each lane's summaries first (the same merge, lane-local), then the lanes
      float ml = neg_inf();
#pragma unroll
      for (int u = 0; u < STRIPE_MAX_Q / 32; ++u) ml = fmax_nan(ml, b[u].x);
      float dl = 0.0f;
      if (ml == ml && ml != neg_inf() && ml != pos_inf()) {
#pragma unroll
        for (int u = 0; u < STRIPE_MAX_Q / 32; ++u)
          if (b[u].x != neg_inf()) dl = __fadd_rn(dl, __fmul_rn(b[u].y, rescale_factor(b[u].x, ml)));
      }
      const MD md = warp_flat_merge(ml, dl);
      const bool zero_row = md.m == neg_inf();
      const bool nan_row = !zero_row && (md.d != md.d || md.m != md.m || md.m == pos_inf());
      const OutConst kc = make_out_const<OutT>(md.m, md.d);
      StripeRow& rc = rowc[kr];
      if constexpr (KEEP_E) {
        // lane w: compute warp w's factor e^(m_w - M) / D (its m_w is in
        // warp_md until the compute warps reach row r + RING, after row r)
        if (lane < NC) {
          const float mw = warp_md[kr][lane].x;
          float F = (mw == neg_inf() || zero_row || nan_row) ? 0.0f : __fmul_rn(rescale_factor(mw, md.m), kc.rD);
          if (warp_fast[kr][lane]) {
            // the warp's fast exponentials carry 2^(-delta), delta the exact
            // residual of RN(-m_w log2e_hi): the factor takes 2^(delta) back
            const float cw = __fmul_rn(-mw, L2E_HI);
            const float delta = __fmaf_rn(-mw, L2E_HI, -cw);
            F = __fmaf_rn(F, __fmul_rn(delta, LN2), F);
          }
          rc.F[lane] = F;
        }
      }
      if (lane == 0) {
        rc.M = md.m;
        rc.D = md.d;
        rc.zero_row = zero_row;
        rc.nan_row = nan_row;
        rc.ld = zero_row ? 0.0f : logf(md.d);
        rc.kc = kc;
      }
      __syncwarp();  // every lane's fields are written before lane 0 releases the row
      if (lane == 0) mbar_arrive(smem_addr(&row_bar[kr]));
      __syncwarp();
    }
  }
}

}  // namespace smx
