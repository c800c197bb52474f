// Long rows in one persistent launch: the chunk summaries of a slab of rows,
// then the normalisation of the same chunks, slab after slab.
//
// A row of many chunks (4096 elements each) is the pages' tiled case ("Kernel
// visualization: online softmax", "Tiled version"; "Online stable softmax",
// "Derive the update for two blocks"): every chunk's (m, d) summary is formed
// on its own and the row's summaries are merged before the chunk is
// normalised.  Each CTA of a cooperative grid owns the same contiguous range
// of a slab's chunks in both phases:
//   A  each chunk's summary (exact chunk maximum, fp32 sum) -> ms/ds[row, c];
//      after its range, thread 0 adds its chunk count to every row it touched
//      (release: a device fence, then the atomics);
//   B  for each row it meets, thread 0 waits (acquire, bounded) until the row's
//      count reaches the number of chunks, the CTA merges the row's summaries
//      and normalises its chunks of the row, re-reading them (from L2 when
//      the slab fits there).
// The cp.async prefetch ring (kernel_stream.cuh) runs straight through the
// phase and slab changes, so phase B's first chunks are in flight while the
// CTA waits.  Phase A never waits, so with every CTA resident (a cooperative
// launch) every wait ends; a wait that runs past its bound records
// SMX_ERR_TIMEOUT in the device status word and the CTA carries on.
#pragma once

#include "kernel_stream.cuh"
#include "smx_async.cuh"

namespace smx {

struct SplitArgs {
  int64_t rows, cols;
  int nchunks;       // chunks per row
  int64_t slab;      // rows per slab
  float* ms;         // [rows][nchunks] chunk maxima
  float* ds;         // [rows][nchunks] chunk sums (natural units)
  unsigned* count;   // [rows] chunks summarised so far (zero at launch)
  const int64_t* target;
  float* loss;
  int64_t max_polls;
  int64_t probe;     // > 0: each count wait asks for one chunk more than the row has (error-path probe)
  int* status;
};

template <typename InT, typename OutT, int MODE, int VPT, int DEPTH>
__global__ void __launch_bounds__(256, 3)
    k_rows_split(const InT* __restrict__ x, OutT* __restrict__ y, SplitArgs a,
                 const int32_t* __restrict__ valid_len) {
  static_assert(MODE == MODE_SOFTMAX || MODE == MODE_LOG || MODE == MODE_CE, "modes of the split");
  constexpr int V = Elem<InT>::V;
  extern __shared__ __align__(16) uint4 sbuf[];  // [DEPTH][VPT][G]
  __shared__ float s_max[2][32], s_sum[32], s_mm[2][32], s_dd[2][32];
  __shared__ float s_row[3];  // the row's M, D, log D
  __shared__ long long s_t;   // the row's target (-1: ignored)

  const int G = blockDim.x, g = threadIdx.x, lane = g & 31, warp = g >> 5, nw = G >> 5;
  const uint32_t my_slot = static_cast<uint32_t>(__cvta_generic_to_shared(sbuf + g));
  const uint32_t slot_stride = (uint32_t)(VPT * G * 16);
  const int chunk = G * VPT * V;
  const int nch = a.nchunks;
  const int64_t nslabs = (a.rows + a.slab - 1) / a.slab;

  // the virtual walk: slab s, phase p (0 = A, 1 = B), item k of the slab
  // (row r = k / nch of the slab, chunk c = k % nch)
  struct Cur {
    int64_t s, k, r, kend;
    int p, c;
  };
  auto range = [&](int64_t s, int64_t& kb, int64_t& ke) {
    const int64_t r0 = s * a.slab;
    const int64_t n = (a.rows - r0 < a.slab ? a.rows - r0 : a.slab) * nch;
    kb = (int64_t)blockIdx.x * n / gridDim.x;
    ke = (int64_t)(blockIdx.x + 1) * n / gridDim.x;
  };
  auto start = [&](Cur& q, int64_t s, int p) {  // first item of (s, p), skipping empty ranges
    for (; s < nslabs; ++s, p = 0) {
      int64_t kb, ke;
      range(s, kb, ke);
      if (kb < ke) {
        q = Cur{s, kb, kb / nch, ke, p, (int)(kb % nch)};
        return;
      }
    }
    q = Cur{nslabs, 0, 0, 0, 0, 0};
  };
  auto advance = [&](Cur& q) {
    ++q.k;
    if (++q.c == nch) {
      q.c = 0;
      ++q.r;
    }
    if (q.k == q.kend) {
      if (q.p == 0) {
        start(q, q.s, 1);
      } else {
        start(q, q.s + 1, 0);
      }
    }
  };
  auto valid_of = [&](int64_t row, int c, int& len) -> int {
    const int64_t begin = (int64_t)c * chunk;
    len = (int)(a.cols - begin < chunk ? a.cols - begin : chunk);
    int64_t L = a.cols;
    if (valid_len != nullptr) {
      const int64_t v = __ldg(valid_len + row);
      L = v < 0 ? 0 : (v > a.cols ? a.cols : v);
    }
    L -= begin;
    return (int)(L < 0 ? 0 : (L > len ? len : L));
  };
  auto prefetch = [&](const Cur& q, int d) -> int {
    int Lk = 0;
    if (q.s < nslabs) {
      const int64_t row = q.s * a.slab + q.r;
      int len;
      Lk = valid_of(row, q.c, len);
      const InT* xr = x + row * a.cols + (int64_t)q.c * chunk;
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
        const int e0 = (j * G + g) * V;
        if (e0 < Lk) cp_async16(my_slot + d * slot_stride + j * G * 16, xr + e0);
      }
    }
    cp_async_commit();
    return Lk;
  };

  Cur cur;
  start(cur, 0, 0);
  Cur pf = cur;
  int Ls[DEPTH];
#pragma unroll
  for (int d = 0; d < DEPTH; ++d) {
    Ls[d] = prefetch(pf, d);
    advance(pf);
  }
  int64_t have_row = -1;  // phase B: the row whose (M, D) s_row holds
  int mpar = 0;

  for (int d = 0, par = 0; cur.s < nslabs; par ^= 1) {
    cp_async_wait<DEPTH - 1>();
    const int L = Ls[0];
    const int64_t row = cur.s * a.slab + cur.r;
    int len;
    valid_of(row, cur.c, len);
    float v[VPT][V];
    const InT* sx = reinterpret_cast<const InT*>(sbuf + (size_t)d * VPT * G);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int e0 = (j * G + g) * V;
      load_masked<InT, true>(sx + e0, e0, L, v[j]);
    }
#pragma unroll
    for (int i = 0; i + 1 < DEPTH; ++i) Ls[i] = Ls[i + 1];
    Ls[DEPTH - 1] = prefetch(pf, d);
    advance(pf);
    d = d + 1 == DEPTH ? 0 : d + 1;

    if (cur.p == 0) {
      // ---- phase A: the chunk's summary
      const float M = warp_max_nan(local_max(v));
      if (lane == 0) s_max[par][warp] = M;
      __syncthreads();
      const float Mc = warp_max_nan(lane < nw ? s_max[par][lane] : neg_inf());
      float Dc = 0.0f;
      if (Mc != neg_inf()) {
        const float sum = warp_sum(exp_and_sum<float, MODE_STATS>(v, Mc));
        if (lane == 0) s_sum[warp] = sum;
        __syncthreads();
        Dc = stats_correct(warp_sum(lane < nw ? s_sum[lane] : 0.0f), Mc);
      }
      if (g == 0) {
        a.ms[row * nch + cur.c] = Mc;
        a.ds[row * nch + cur.c] = Dc;
      }
      if (cur.k + 1 == cur.kend) {
        // end of the range: publish the chunk counts of the rows it touched
        if (g == 0) {
          int64_t kb, ke;
          range(cur.s, kb, ke);
          __threadfence();
          for (int64_t r = kb / nch; r <= (ke - 1) / nch; ++r) {
            const int64_t lo = r * nch > kb ? r * nch : kb;
            const int64_t hi = (r + 1) * nch < ke ? (r + 1) * nch : ke;
            atomicAdd(a.count + cur.s * a.slab + r, (unsigned)(hi - lo));
          }
        }
      }
    } else {
      // ---- phase B: the row's merged (M, D), then the chunk's outputs
      if (row != have_row) {
        if (g == 0) {
          const unsigned need = (unsigned)nch + (a.probe > 0 ? 1u : 0u);
          const int64_t limit = a.probe > 0 ? a.probe : a.max_polls;
          int64_t polls = 0;
          while (ld_acquire_u32(a.count + row) < need) {
            if (++polls > limit) {
              atomicOr(a.status, DEV_TIMEOUT);
              break;
            }
            __nanosleep(200);
          }
        }
        __syncthreads();  // thread 0's acquire orders the summaries for the CTA
        MD acc{neg_inf(), 0.0f};
        for (int i = g; i < nch; i += G)
          acc = md_merge(acc, MD{__ldcg(a.ms + row * nch + i), __ldcg(a.ds + row * nch + i)});
        acc = warp_merge(acc);
        if (lane == 0) {
          s_mm[mpar][warp] = acc.m;
          s_dd[mpar][warp] = acc.d;
        }
        __syncthreads();
        acc = warp_merge(lane < nw ? MD{s_mm[mpar][lane], s_dd[mpar][lane]} : MD{neg_inf(), 0.0f});
        mpar ^= 1;
        if (g == 0) {
          s_row[0] = acc.m;
          s_row[1] = acc.d;
          s_row[2] = logf(acc.d);
          if constexpr (MODE == MODE_CE) {
            const int64_t t = __ldg(a.target + row);
            int64_t Lr = a.cols;
            if (valid_len != nullptr) {
              const int64_t vv = __ldg(valid_len + row);
              Lr = vv < 0 ? 0 : (vv > a.cols ? a.cols : vv);
            }
            s_t = (t < 0 || t >= Lr) ? -1 : t;  // an ignored target is kept as -1
          }
        }
        __syncthreads();
        have_row = row;
      }
      const float Mr = s_row[0], Dr = s_row[1], ldr = s_row[2];
      const bool zero_row = (Mr == neg_inf());
      const bool nan_row = !zero_row && (Dr != Dr || Mr != Mr || Mr == pos_inf());
      OutT* yr = y + row * a.cols + (int64_t)cur.c * chunk;
      if constexpr (MODE == MODE_LOG) {
        store_log<OutT, VPT, V>(yr, G, g, len, L, v, zero_row, nan_row, Mr, ldr);
      } else {
        bool zero_out = zero_row, nan_out = nan_row;
        // cross-entropy: the target's place in this chunk, and x_t from the
        // registers of the thread that holds it
        int tl = -1;
        float xt = 0.0f;
        if constexpr (MODE == MODE_CE) {
          const int64_t t_row = s_t;
          const bool ignored = t_row < 0;
          const bool bad = zero_row || nan_row;
          zero_out = ignored;
          nan_out = !ignored && bad;
          const int64_t t = t_row - (int64_t)cur.c * chunk;
          tl = (!ignored && t >= 0 && t < L) ? (int)t : -1;
          if (tl >= 0 && (tl / V) % G == g) {
            const int jo = tl / V / G, io = tl % V;
#pragma unroll
            for (int j = 0; j < VPT; ++j)
#pragma unroll
              for (int i = 0; i < V; ++i)
                if (j == jo && i == io) xt = v[j][i];
          }
        }
        const OutConst kc = make_out_const<OutT>(Mr, Dr);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
          const int e0 = (j * G + g) * V;
          if (e0 < len) {
            float q[V];
            if (!zero_out && !nan_out) {
              out_values<OutT, V>(v[j], kc, q);
            } else {
#pragma unroll
              for (int i = 0; i < V; ++i) q[i] = (nan_out && e0 + i < L) ? qnan() : 0.0f;
            }
            store_vec<OutT, V>(yr + e0, q);
          }
        }
        if constexpr (MODE == MODE_CE) {
          if (tl >= 0 && (tl / V) % G == g) {
            const bool bad = zero_row || nan_row;
            a.loss[row] = bad ? qnan() : __fadd_rn(__fsub_rn(Mr, xt), ldr);
            if (!bad) yr[tl] = Elem<OutT>::from_f32(__fsub_rn(out_value<OutT>(xt, kc), 1.0f));
          }
          if (s_t < 0 && cur.c == 0 && g == 0) a.loss[row] = 0.0f;
        }
      }
    }
    advance(cur);
  }
  cp_async_wait<0>();
}

}  // namespace smx
