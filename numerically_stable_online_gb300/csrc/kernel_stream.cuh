// Persistent row softmax that keeps the next items' reads in flight while it
// reduces the current one.
//
// An item is a whole row (rows of up to 32 KiB), or one chunk of a long row.
// The arithmetic is the register-resident kernel's (kernel_regs.cuh, via
// row_core.cuh): exact maximum, exponentials against it with their fp32 sum,
// one normalising multiply; one HBM read and one HBM write per element.  The
// register kernel's CTA holds no reads in flight while it reduces its row;
// here a persistent CTA of G threads walks its items and every thread
// prefetches its own 16-byte vectors of the next DEPTH items into its own
// shared-memory words with cp.async (one commit group per item).  Each thread
// reads back only what it copied itself, so the prefetch needs no barrier; an
// item's group is awaited with cp.async.wait_group just before the item is used.
//
// Whole rows (CHUNKED = false) are dealt round robin: CTA b takes rows
// b, b + gridDim.x, ...  With WARP = true each warp is such a walker on its own
// (a row per warp, rows b NW + w, stepping by gridDim.x NW): short rows then
// need no block barrier at all, only warp shuffles.  Chunks (CHUNKED = true)
// are dealt in contiguous runs: CTA b takes items [b n / gridDim.x,
// (b + 1) n / gridDim.x), so a CTA meets each of its rows in consecutive items.
//
// Modes (the same walk):
//   MODE_SOFTMAX  whole rows: y = e^(x - m) / d.
//   MODE_STATS    the (m, d) block summary of each item ("Stable softmax: keep
//                 the normalizer consistent as tiles arrive", third paragraph),
//                 at m_out[k], d_out[k] (k counted from the launch's first item;
//                 for whole rows, the row - row0).  With d_out == nullptr
//                 (whole rows) m_out receives LSE = m + log d instead
//                 ("Softmax numerics architecture...", "Log-sum-exp:
//                 log-probabilities without probabilities").
//   MODE_LOG      whole rows: log_softmax y = (x - m) - log d, the same section;
//                 -inf in masked lanes (the log of their +0 probability).
//   MODE_APPLY    chunks only: the row's (M, D) -- given per row (Items::
//                 row_stats), or merged from the row's chunk summaries m_in,
//                 d_in ("Online stable softmax", "Derive the update for two
//                 blocks"; once per row a CTA meets) -- normalises the chunk:
//                 the step that completes a softmax whose summaries were
//                 computed apart.
//   MODE_APPLY_LOG  as MODE_APPLY, writing log_softmax.
//   MODE_CE       whole rows: cross-entropy with logits (the same section and
//                 "The Jacobian, and the backward pass that never divides"):
//                 loss = LSE - x_t = (m - x_t) + log d, and, when y is given,
//                 the fused gradient y = p - onehot(t): the row's p is stored,
//                 then the thread that holds x_t stores p_t - 1 over its own
//                 p_t.  A target outside the valid prefix is ignored: loss 0
//                 and a zero gradient row.
//   MODE_APPLY_CE   chunks: MODE_CE with the row's merged (M, D).
#pragma once

#include "row_core.cuh"

namespace smx {

enum : int { MODE_APPLY = 2, MODE_LOG = 3, MODE_APPLY_LOG = 4, MODE_CE = 5, MODE_APPLY_CE = 6 };

// The items of one launch: item k is chunk k % nchunks of row row0 + k / nchunks.
struct Items {
  int64_t n;     // items in the launch
  int64_t row0;  // first row
  int64_t cols;  // row length
  int chunk;     // elements per item (a multiple of the vector width; a row's last item may be shorter)
  int nchunks;   // items per row (1: whole rows)
  int l2_hint;   // chunked reads only: 0 none, 1 keep in L2 (evict_last), 2 evict_first
  int row_stats; // apply modes: 1 = (m_in[r], d_in[r]) per row, 0 = merge the row's chunk summaries
};

__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_dst), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async16_hint(uint32_t smem_dst, const void* gsrc, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_dst),
               "l"(gsrc), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t smem_dst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_dst), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t smem_dst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_dst), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint64_t l2_policy(int hint) {
  uint64_t p = 0;
  if (hint == 1)
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  else
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// SMX_STREAM_MAXNREG (a build-time tuning knob) caps the registers per thread,
// trading spills for resident CTAs.
// The warp walkers run 128-thread CTAs, so their register budget is not the
// 1024-thread one.
// SMX_WARP_MIN_CTAS (a build-time tuning knob) asks the compiler to fit that
// many 128-thread warp-walker CTAs per SM (a register budget).  Measured on
// GB300 (masked fp16 rows of 1024): 6 (at most 85 registers) against no budget
// (92): softmax 21.0 -> 20.5 us, log_softmax 23.0 -> 20.6 us, cross-entropy
// 26.0 -> 25.2 us; 8 (64 registers) spills and is slower.
#ifndef SMX_WARP_MIN_CTAS
#define SMX_WARP_MIN_CTAS 6
#endif
#ifdef SMX_STREAM_MAXNREG
#define SMX_STREAM_REGS __maxnreg__(SMX_STREAM_MAXNREG)
#else
#define SMX_STREAM_REGS __launch_bounds__(WARP ? 128 : 1024, WARP ? SMX_WARP_MIN_CTAS : 1)
#endif

template <typename InT, typename OutT, int VPT, int MODE, int DEPTH, bool CHUNKED, bool WARP = false>
__global__ void SMX_STREAM_REGS
    k_rows_stream(const InT* __restrict__ x, OutT* __restrict__ y, float* __restrict__ m_out,
                  float* __restrict__ d_out, const float* __restrict__ m_in,
                  const float* __restrict__ d_in, Items it, const int32_t* __restrict__ valid_len,
                  const int64_t* __restrict__ target, float* __restrict__ loss) {
  constexpr bool APPLY = (MODE == MODE_APPLY || MODE == MODE_APPLY_LOG || MODE == MODE_APPLY_CE);
  constexpr bool CE = (MODE == MODE_CE || MODE == MODE_APPLY_CE);
  static_assert(CHUNKED || !APPLY || (MODE == MODE_APPLY && WARP),
                "the apply modes walk chunks, or (given per-row statistics) whole rows a warp each");
  static_assert(!(WARP && CHUNKED), "a warp walks whole rows");
  constexpr int V = Elem<InT>::V;
  // [walkers][DEPTH][VPT][G] uint4: thread g of a walker owns column g; then
  // [DEPTH][blockDim.x] 8-byte words: each thread's copy of its item's per-row
  // value (the target, or the given (m, d))
  extern __shared__ __align__(16) uint4 sbuf[];
  // s_max alternates between items: an item with no valid lane skips the sum's
  // barrier, so only the next item's max barrier separates reads from rewrites
  // (s_mm, s_dd alternate between row merges for the same reason)
  __shared__ float s_max[2][32], s_sum[32], s_mm[2][32], s_dd[2][32];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int G = WARP ? 32 : blockDim.x, g = WARP ? lane : threadIdx.x;
  uint4* ring = sbuf + (WARP ? (size_t)warp * DEPTH * VPT * 32 : 0);
  const uint32_t my_slot = static_cast<uint32_t>(__cvta_generic_to_shared(ring + g));
  const uint32_t slot_stride = (uint32_t)(VPT * G * 16);  // bytes between ring slots
  uint2* aux = reinterpret_cast<uint2*>(sbuf + (size_t)DEPTH * VPT * blockDim.x);
  const uint32_t my_aux = static_cast<uint32_t>(__cvta_generic_to_shared(aux + threadIdx.x));
  const int ncols = (int)(CHUNKED ? it.chunk : it.cols);

  // An item's place: k, its row r (from row0) and chunk c.  Two cursors walk
  // the walker's items without dividing: `cur` at the item being reduced, `pf`
  // DEPTH items ahead at the next one to prefetch.
  struct Cursor {
    int64_t k, r;
    int c;
  };
  int64_t k_end;
  Cursor cur;
  int64_t step = gridDim.x;
  if constexpr (CHUNKED) {
    const int64_t kb = (int64_t)blockIdx.x * it.n / gridDim.x;
    k_end = (int64_t)(blockIdx.x + 1) * it.n / gridDim.x;
    cur = Cursor{kb, kb / it.nchunks, (int)(kb % it.nchunks)};
  } else if constexpr (WARP) {
    k_end = it.n;
    const int64_t k0 = (int64_t)blockIdx.x * nw + warp;
    cur = Cursor{k0, k0, 0};
    step = (int64_t)gridDim.x * nw;
  } else {
    k_end = it.n;
    cur = Cursor{(int64_t)blockIdx.x, (int64_t)blockIdx.x, 0};
  }
  auto advance = [&](Cursor& q) {
    if constexpr (CHUNKED) {
      ++q.k;
      if (++q.c == it.nchunks) {
        q.c = 0;
        ++q.r;
      }
    } else {
      q.k += step;
      q.r = q.k;
    }
  };
  // elements of an item, and its share of the row's valid prefix
  auto item_len = [&](const Cursor& q) -> int {
    if constexpr (CHUNKED) {
      const int64_t rest = it.cols - (int64_t)q.c * it.chunk;
      return rest < it.chunk ? (int)rest : it.chunk;
    } else {
      return ncols;
    }
  };
  // the item's share of its row's valid prefix, from the row's raw valid
  // length v (loaded one item ahead, see vl_pf below)
  auto item_valid = [&](const Cursor& q, int32_t vraw) -> int {
    const int len = item_len(q);
    if (valid_len == nullptr) return len;
    const int64_t v = vraw;
    const int64_t L = (v < 0 ? 0 : (v > it.cols ? it.cols : v)) - (int64_t)q.c * ncols;
    return (int)(L < 0 ? 0 : (L > len ? len : L));
  };
  auto row_valid = [&](int64_t row) -> int64_t {  // the row's valid prefix length
    if (valid_len == nullptr) return it.cols;
    const int64_t v = __ldg(valid_len + row);
    return v < 0 ? 0 : (v > it.cols ? it.cols : v);
  };
  // reductions over the walker (the CTA, or one warp)
  auto walker_max = [&](float m, int par) -> float {
    m = warp_max_nan(m);
    if constexpr (WARP) {
      return m;
    } else {
      if (lane == 0) s_max[par][warp] = m;
      __syncthreads();
      return warp_max_nan(lane < nw ? s_max[par][lane] : neg_inf());
    }
  };
  auto walker_sum = [&](float t) -> float {
    t = warp_sum(t);
    if constexpr (WARP) {
      return t;
    } else {
      if (lane == 0) s_sum[warp] = t;
      __syncthreads();
      return warp_sum(lane < nw ? s_sum[lane] : 0.0f);
    }
  };
  const uint64_t pol = (CHUNKED && it.l2_hint != 0) ? l2_policy(it.l2_hint) : 0;
  // per-row values the item needs (the target; the given statistics) travel
  // with the item: lane 0 of each warp copies them into its own word of the
  // slot in the same cp.async group (so no register waits on their loads) and
  // hands them to the other lanes by shuffle once the group has landed
  constexpr bool AUX = CE || APPLY;
  auto prefetch_row_values = [&](const Cursor& q, int d) {
    if constexpr (AUX) {
      if (lane == 0 && q.k < k_end) {  // one copy per warp, shuffled to the lanes
        const uint32_t dst = my_aux + d * blockDim.x * 8;
        if constexpr (CE) cp_async8(dst, target + it.row0 + q.r);
        if constexpr (APPLY) {
          if (it.row_stats) {
            cp_async4(dst, m_in + q.r);
            cp_async4(dst + 4, d_in + q.r);
          }
        }
      }
    }
  };
  // the raw valid length of the item the next prefetch copies, loaded as soon
  // as the prefetch cursor reaches it, one item ahead of its use, so that no
  // prefetch waits on a load of its own length.  Measured on GB300 (masked
  // fp16 rows of 1024): faster for the softmax, log_softmax and cross-entropy
  // rows, slower for the statistics and apply rows, which load it in place.
  constexpr bool VL_AHEAD = MODE == MODE_SOFTMAX || MODE == MODE_LOG || MODE == MODE_CE;
  // copy this thread's vectors of item q into ring slot d; always one group
  auto prefetch = [&](const Cursor& q, int d, int32_t vraw) -> int {
    int Lk = 0;
    if (q.k < k_end) {
      if constexpr (!VL_AHEAD) vraw = valid_len != nullptr ? __ldg(valid_len + it.row0 + q.r) : 0;
      Lk = item_valid(q, vraw);
      const InT* xr = x + (it.row0 + q.r) * it.cols + (int64_t)q.c * ncols;
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
        const int e0 = (j * G + g) * V;
        if (e0 < Lk) {
          const uint32_t dst = my_slot + d * slot_stride + j * G * 16;
          if (CHUNKED && it.l2_hint != 0)
            cp_async16_hint(dst, xr + e0, pol);
          else
            cp_async16(dst, xr + e0);
        }
      }
    }
    prefetch_row_values(q, d);
    cp_async_commit();
    return Lk;
  };

  // the raw valid length of the item the next prefetch copies (VL_AHEAD modes)
  auto load_vl = [&](const Cursor& q) -> int32_t {
    if constexpr (VL_AHEAD) {
      return (valid_len != nullptr && q.k < k_end) ? __ldg(valid_len + it.row0 + q.r) : 0;
    } else {
      return 0;
    }
  };
  Cursor pf = cur;
  int32_t vl_pf = load_vl(pf);
  int Ls[DEPTH];
#pragma unroll
  for (int d = 0; d < DEPTH; ++d) {
    Ls[d] = prefetch(pf, d, vl_pf);
    advance(pf);
    vl_pf = load_vl(pf);
  }

  // the apply modes' summary of the row they are in
  int64_t have_row = -1;
  MD row_md{neg_inf(), 0.0f};
  float row_ld = 0.0f;  // log of row_md.d (the log and cross-entropy modes)
  int mpar = 0;

  for (int d = 0, par = 0; cur.k < k_end; advance(cur), par ^= 1) {
    cp_async_wait<DEPTH - 1>();  // this thread's copies of the item have landed
    const int L = Ls[0];
    const int len = item_len(cur);
    const int64_t row = it.row0 + cur.r;
    const int64_t begin = (int64_t)cur.c * ncols;
    float v[VPT][V];
    const InT* sx = reinterpret_cast<const InT*>(ring + (size_t)d * VPT * G);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int e0 = (j * G + g) * V;
      load_masked<InT, true>(sx + e0, e0, L, v[j]);
    }
    // cross-entropy: the target's place in this item, and x_t, read by the
    // thread that copied it (the slot holds the item in element order) before
    // the slot is refilled
    int64_t t_item = -1;
    float m_item = 0.0f, d_item = 0.0f;
    if constexpr (AUX) {
      const uint2 w0 = aux[d * blockDim.x + threadIdx.x];  // meaningful in lane 0
      const uint2 w = make_uint2(__shfl_sync(0xffffffffu, w0.x, 0), __shfl_sync(0xffffffffu, w0.y, 0));
      if constexpr (CE) t_item = (long long)(((unsigned long long)w.y << 32) | w.x);
      if constexpr (APPLY) {
        m_item = __uint_as_float(w.x);
        d_item = __uint_as_float(w.y);
      }
    }
    int tl = -1;
    bool t_mine = false;
    float xt = 0.0f;
    if constexpr (CE) {
      const int64_t tl64 = t_item - begin;
      if (tl64 >= 0 && tl64 < L) tl = (int)tl64;
      t_mine = tl >= 0 && (tl / V) % G == g;
      if (t_mine) xt = Elem<InT>::to_f32(sx[tl]);
    }
    // the slot's words are in registers now: refill it with the item DEPTH ahead
#pragma unroll
    for (int i = 0; i + 1 < DEPTH; ++i) Ls[i] = Ls[i + 1];
    Ls[DEPTH - 1] = prefetch(pf, d, vl_pf);
    advance(pf);
    vl_pf = load_vl(pf);
    d = d + 1 == DEPTH ? 0 : d + 1;

    if constexpr (APPLY) {
      if (cur.r != have_row) {  // uniform: every thread walks the same items
        if (it.row_stats || WARP) {  // a warp walker has the row's statistics given
          row_md = MD{m_item, d_item};
        } else {
          MD acc{neg_inf(), 0.0f};
          const int64_t k0 = cur.r * it.nchunks;
          for (int i = g; i < it.nchunks; i += G)
            acc = md_merge(acc, MD{__ldg(m_in + k0 + i), __ldg(d_in + k0 + i)});
          acc = warp_merge(acc);
          if (lane == 0) {
            s_mm[mpar][warp] = acc.m;
            s_dd[mpar][warp] = acc.d;
          }
          __syncthreads();
          row_md = warp_merge(lane < nw ? MD{s_mm[mpar][lane], s_dd[mpar][lane]} : MD{neg_inf(), 0.0f});
          mpar ^= 1;
        }
        have_row = cur.r;
        row_ld = logf(row_md.d);
      }
      const float M = row_md.m, Dr = row_md.d;
      const bool zero_row = (M == neg_inf());
      const bool nan_row = !zero_row && (Dr != Dr || M != M || M == pos_inf());
      OutT* yr = y + row * it.cols + begin;
      if constexpr (MODE == MODE_APPLY_LOG) {
        store_log<OutT, VPT, V>(yr, G, g, len, L, v, zero_row, nan_row, M, row_ld);
      } else {
        // cross-entropy: an ignored target zeroes the row, a bad row is NaN
        // in its valid lanes; the owner of x_t writes the loss
        bool zero_out = zero_row, nan_out = nan_row;
        if constexpr (MODE == MODE_APPLY_CE) {
          const bool ignored = t_item < 0 || t_item >= row_valid(row);
          const bool bad = zero_row || nan_row;
          zero_out = ignored;
          nan_out = !ignored && bad;
          if (t_mine) loss[row] = bad ? qnan() : __fadd_rn(__fsub_rn(M, xt), row_ld);
          if (ignored && cur.c == 0 && g == 0) loss[row] = 0.0f;
        }
        if (MODE != MODE_APPLY_CE || y != nullptr) {
          const OutConst kc = make_out_const<OutT>(M, Dr);
#pragma unroll
          for (int j = 0; j < VPT; ++j) {
            const int e0 = (j * G + g) * V;
            if (e0 < len) {
              float p[V];
              if (!zero_out && !nan_out) {
                out_values<OutT, V>(v[j], kc, p);
              } else {
#pragma unroll
                for (int i = 0; i < V; ++i) p[i] = (nan_out && e0 + i < L) ? qnan() : 0.0f;
              }
              store_vec<OutT, V>(yr + e0, p);
            }
          }
          if constexpr (MODE == MODE_APPLY_CE) {
            // p_t - 1 over the owner's own earlier store of p_t
            if (t_mine && !zero_out && !nan_out)
              yr[tl] = Elem<OutT>::from_f32(__fsub_rn(out_value<OutT>(xt, kc), 1.0f));
          }
        }
      }
    } else {
      const float M = walker_max(local_max(v), par);
      float Dsum = 0.0f;
      if (M != neg_inf()) {
        float sum;
        if constexpr (MODE == MODE_LOG) {
          sum = sum_exp(v, M);  // v keeps x
        } else if constexpr (MODE == MODE_CE) {
          // with a gradient, exponentials in place as the softmax forms them;
          // the loss alone needs only their sum
          sum = y != nullptr ? exp_and_sum<OutT, MODE_SOFTMAX>(v, M) : sum_exp(v, M);
        } else {
          sum = exp_and_sum<OutT, MODE>(v, M);
        }
        Dsum = walker_sum(sum);
      }
      const bool zero_row = (M == neg_inf());
      const bool nan_row = !zero_row && (Dsum != Dsum);
      if constexpr (MODE == MODE_STATS) {
        if (g == 0) {
          const float dk = zero_row ? 0.0f : stats_correct(Dsum, M);
          if (d_out != nullptr) {
            m_out[cur.k] = M;
            d_out[cur.k] = dk;
          } else {
            m_out[cur.k] = zero_row ? neg_inf() : __fadd_rn(M, logf(dk));
          }
        }
      } else if constexpr (MODE == MODE_CE) {
        const bool ignored = tl < 0;  // a whole row: the item's valid length is the row's
        const bool bad = zero_row || nan_row;
        if (t_mine) {
          const float ld = y != nullptr ? __fmaf_rn(-softmax_sum_offset_log2<OutT>(M), LN2, logf(Dsum))
                                        : logf(stats_correct(Dsum, M));
          loss[row] = bad ? qnan() : __fadd_rn(__fsub_rn(M, xt), ld);
        }
        if (ignored && g == 0) loss[row] = 0.0f;
        if (y != nullptr) {
          OutT* yr = y + row * it.cols;
          const float rD = recip_refined(Dsum);
          store_row<OutT, VPT, V>(yr, G, g, len, L, v, ignored, !ignored && bad, rD);
          // p_t - 1 over the owner's own earlier store of p_t
          if (t_mine && !bad)
            yr[tl] = Elem<OutT>::from_f32(__fsub_rn(__fmul_rn(exp_like_softmax<OutT>(xt, M), rD), 1.0f));
        }
      } else if constexpr (MODE == MODE_LOG) {
        const float ld = zero_row ? 0.0f : logf(stats_correct(Dsum, M));
        store_log<OutT, VPT, V>(y + row * it.cols, G, g, len, L, v, zero_row, nan_row, M, ld);
      } else {
        store_row<OutT, VPT, V>(y + row * it.cols, G, g, len, L, v, zero_row, nan_row,
                                recip_refined(Dsum));
      }
    }
  }
  cp_async_wait<0>();  // no copy may still target this CTA's shared memory at exit
}

// Row statistics of long rows: merge each row's nchunks chunk summaries
// (consecutive in m_in, d_in) into (m_out[r], d_out[r]), or into
// m_out[r] = LSE when d_out is null; one CTA per row.
template <int THREADS>
__global__ void __launch_bounds__(THREADS)
    k_merge_chunk_stats(const float* __restrict__ m_in, const float* __restrict__ d_in, int nchunks,
                        float* __restrict__ m_out, float* __restrict__ d_out) {
  __shared__ float s_mm[THREADS / 32], s_dd[THREADS / 32];
  const int g = threadIdx.x, lane = g & 31, warp = g >> 5;
  const int64_t k0 = (int64_t)blockIdx.x * nchunks;
  MD acc{neg_inf(), 0.0f};
  for (int i = g; i < nchunks; i += THREADS) acc = md_merge(acc, MD{m_in[k0 + i], d_in[k0 + i]});
  acc = warp_merge(acc);
  if (lane == 0) {
    s_mm[warp] = acc.m;
    s_dd[warp] = acc.d;
  }
  __syncthreads();
  if (warp == 0) {
    acc = warp_merge(lane < THREADS / 32 ? MD{s_mm[lane], s_dd[lane]} : MD{neg_inf(), 0.0f});
    if (lane == 0) {
      const float d = acc.m == neg_inf() ? 0.0f : acc.d;
      if (d_out != nullptr) {
        m_out[blockIdx.x] = acc.m;
        d_out[blockIdx.x] = d;
      } else {  // LSE = m + log d
        m_out[blockIdx.x] = acc.m == neg_inf() ? neg_inf() : __fadd_rn(acc.m, logf(d));
      }
    }
  }
}

// Cross-entropy loss of long rows without a gradient: merge each row's chunk
// summaries, read x_t, write loss = (M - x_t) + log D (0 for an ignored target);
// one CTA per row of the slab starting at row0.
template <typename InT, int THREADS>
__global__ void __launch_bounds__(THREADS)
    k_merge_chunk_ce(const float* __restrict__ m_in, const float* __restrict__ d_in, int nchunks,
                     const InT* __restrict__ x, int64_t cols, const int64_t* __restrict__ target,
                     const int32_t* __restrict__ valid_len, int64_t row0, float* __restrict__ loss) {
  __shared__ float s_mm[THREADS / 32], s_dd[THREADS / 32];
  const int g = threadIdx.x, lane = g & 31, warp = g >> 5;
  const int64_t k0 = (int64_t)blockIdx.x * nchunks;
  MD acc{neg_inf(), 0.0f};
  for (int i = g; i < nchunks; i += THREADS) acc = md_merge(acc, MD{m_in[k0 + i], d_in[k0 + i]});
  acc = warp_merge(acc);
  if (lane == 0) {
    s_mm[warp] = acc.m;
    s_dd[warp] = acc.d;
  }
  __syncthreads();
  if (g == 0) {
    acc = MD{neg_inf(), 0.0f};
    for (int w = 0; w < THREADS / 32; ++w) acc = md_merge(acc, MD{s_mm[w], s_dd[w]});
    const int64_t row = row0 + blockIdx.x;
    int64_t L = cols;
    if (valid_len != nullptr) {
      const int64_t v = valid_len[row];
      L = v < 0 ? 0 : (v > cols ? cols : v);
    }
    const int64_t t = target[row];
    float out = 0.0f;
    if (t >= 0 && t < L) {
      const bool bad = acc.m == neg_inf() || acc.m != acc.m || acc.m == pos_inf() || acc.d != acc.d;
      const float xt = Elem<InT>::to_f32(x[row * cols + t]);
      out = bad ? qnan() : __fadd_rn(__fsub_rn(acc.m, xt), logf(acc.d));
    }
    loss[row] = out;
  }
}

}  // namespace smx
