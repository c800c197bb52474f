// Softmax backward: the vector-Jacobian product of "Softmax numerics
// architecture - max subtract, fp32 accumulate, fusion, online", section "The
// Jacobian, and the backward pass that never divides": for the stored softmax
// p of a row and the upstream gradient g,
//     dx_j = p_j (g_j - s),   s = sum_k g_k p_k,
// over the row's valid prefix; masked lanes (where the forward output is the
// constant +0) get dx = 0.  One dot product and one pass: two reads and one
// write per element, so the kernel is HBM-bound like the forward.
//
// The walk is the streamed forward kernel's (kernel_stream.cuh): a persistent
// CTA of G threads, each thread prefetching its own 16-byte vectors of p and g
// for the next DEPTH items into its own shared-memory words with cp.async.
// Whole rows are dealt round robin; long rows in chunks, in contiguous runs per
// CTA, in two launches: BWD_DOT writes each chunk's partial dot, BWD_APPLY adds
// the row's partials (once per row a CTA meets) and writes the chunk's dx.
#pragma once

#include "kernel_stream.cuh"

namespace smx {

enum : int { BWD_ROWS = 0, BWD_DOT = 1, BWD_APPLY = 2 };

template <typename InT, typename OutT, int VPT, int MODE, int DEPTH>
__global__ void __launch_bounds__(1024)
    k_backward(const InT* __restrict__ p, const InT* __restrict__ gr, OutT* __restrict__ dx,
               float* __restrict__ part_out, const float* __restrict__ part_in, Items it,
               const int32_t* __restrict__ valid_len) {
  constexpr bool CHUNKED = (MODE != BWD_ROWS);
  constexpr int V = Elem<InT>::V;
  extern __shared__ __align__(16) uint4 sbuf[];  // [DEPTH][2][VPT][G]: p then g
  __shared__ float s_dot[2][32];

  const int G = blockDim.x, g = threadIdx.x, lane = g & 31, warp = g >> 5, nw = G >> 5;
  const uint32_t my_slot = static_cast<uint32_t>(__cvta_generic_to_shared(sbuf + g));
  const uint32_t half_stride = (uint32_t)(VPT * G * 16);  // p part to g part
  const uint32_t slot_stride = 2 * half_stride;
  const int ncols = (int)(CHUNKED ? it.chunk : it.cols);

  struct Cursor {
    int64_t k, r;
    int c;
  };
  int64_t k_end;
  Cursor cur;
  if constexpr (CHUNKED) {
    const int64_t kb = (int64_t)blockIdx.x * it.n / gridDim.x;
    k_end = (int64_t)(blockIdx.x + 1) * it.n / gridDim.x;
    cur = Cursor{kb, kb / it.nchunks, (int)(kb % it.nchunks)};
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
      q.k += gridDim.x;
      q.r = q.k;
    }
  };
  auto item_len = [&](const Cursor& q) -> int {
    if constexpr (CHUNKED) {
      const int64_t rest = it.cols - (int64_t)q.c * it.chunk;
      return rest < it.chunk ? (int)rest : it.chunk;
    } else {
      return ncols;
    }
  };
  auto item_valid = [&](const Cursor& q) -> int {
    const int len = item_len(q);
    if (valid_len == nullptr) return len;
    const int64_t v = __ldg(valid_len + it.row0 + q.r);
    const int64_t L = (v < 0 ? 0 : (v > it.cols ? it.cols : v)) - (int64_t)q.c * ncols;
    return (int)(L < 0 ? 0 : (L > len ? len : L));
  };
  // the dot pass reads only the valid lanes; the apply pass only the valid
  // lanes too (dx is 0 beyond them whatever p and g hold)
  auto prefetch = [&](const Cursor& q, int d) -> int {
    int Lk = 0;
    if (q.k < k_end) {
      Lk = item_valid(q);
      const int64_t off = (it.row0 + q.r) * it.cols + (int64_t)q.c * ncols;
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
        const int e0 = (j * G + g) * V;
        if (e0 < Lk) {
          const uint32_t dst = my_slot + d * slot_stride + j * G * 16;
          cp_async16(dst, p + off + e0);
          cp_async16(dst + half_stride, gr + off + e0);
        }
      }
    }
    cp_async_commit();
    return Lk;
  };

  Cursor pf = cur;
  int Ls[DEPTH];
#pragma unroll
  for (int d = 0; d < DEPTH; ++d) {
    Ls[d] = prefetch(pf, d);
    advance(pf);
  }
  int64_t have_row = -1;
  float row_s = 0.0f;
  int spar = 0;

  for (int d = 0, par = 0; cur.k < k_end; advance(cur), par ^= 1) {
    cp_async_wait<DEPTH - 1>();
    const int L = Ls[0];
    const int len = item_len(cur);
    const int64_t row = it.row0 + cur.r;
    // masked lanes load as -inf; the products below only ever see valid lanes
    float vp[VPT][V], vg[VPT][V];
    const InT* sp = reinterpret_cast<const InT*>(sbuf + (size_t)d * 2 * VPT * G);
    const InT* sg = reinterpret_cast<const InT*>(sbuf + (size_t)d * 2 * VPT * G + VPT * G);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int e0 = (j * G + g) * V;
      load_masked<InT, true>(sp + e0, e0, L, vp[j]);
      load_masked<InT, true>(sg + e0, e0, L, vg[j]);
    }
#pragma unroll
    for (int i = 0; i + 1 < DEPTH; ++i) Ls[i] = Ls[i + 1];
    Ls[DEPTH - 1] = prefetch(pf, d);
    advance(pf);
    d = d + 1 == DEPTH ? 0 : d + 1;

    float s;
    if constexpr (MODE == BWD_APPLY) {
      if (cur.r != have_row) {  // the row's partial dots, added once per row
        float acc = 0.0f;
        const int64_t k0 = cur.r * it.nchunks;
        for (int i = g; i < it.nchunks; i += G) acc = __fadd_rn(acc, __ldg(part_in + k0 + i));
        acc = warp_sum(acc);
        if (lane == 0) s_dot[spar][warp] = acc;
        __syncthreads();
        row_s = warp_sum(lane < nw ? s_dot[spar][lane] : 0.0f);
        spar ^= 1;
        have_row = cur.r;
      }
      s = row_s;
    } else {
      // this thread's share of sum g p over its valid lanes
      float acc = 0.0f;
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
        const int e0 = (j * G + g) * V;
#pragma unroll
        for (int i = 0; i < V; ++i)
          if (e0 + i < L) acc = __fmaf_rn(vg[j][i], vp[j][i], acc);
      }
      acc = warp_sum(acc);
      if (lane == 0) s_dot[par][warp] = acc;
      __syncthreads();
      s = warp_sum(lane < nw ? s_dot[par][lane] : 0.0f);
    }
    if constexpr (MODE == BWD_DOT) {
      if (g == 0) part_out[cur.k] = s;
    } else {
      OutT* yr = dx + row * it.cols + (int64_t)cur.c * ncols;
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
        const int e0 = (j * G + g) * V;
        if (e0 < len) {
          float q[V];
#pragma unroll
          for (int i = 0; i < V; ++i)
            q[i] = e0 + i < L ? __fmul_rn(vp[j][i], __fsub_rn(vg[j][i], s)) : 0.0f;
          store_vec<OutT, V>(yr + e0, q);
        }
      }
    }
  }
  cp_async_wait<0>();
}

// Any alignment and any cols: one CTA per row, the dot then dx, scalar loads.
template <typename InT, typename OutT>
__global__ void __launch_bounds__(256)
    k_backward_generic(const InT* __restrict__ p, const InT* __restrict__ gr, OutT* __restrict__ dx,
                       int64_t cols, const int32_t* __restrict__ valid_len, int64_t row0) {
  __shared__ float s_dot[8];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t row = row0 + blockIdx.x;
  int64_t L = cols;
  if (valid_len != nullptr) {
    const int64_t v = __ldg(valid_len + row);
    L = v < 0 ? 0 : (v > cols ? cols : v);
  }
  const InT* pr = p + row * cols;
  const InT* gq = gr + row * cols;
  float acc = 0.0f;
  for (int64_t j = t; j < L; j += 256)
    acc = __fmaf_rn(Elem<InT>::to_f32(gq[j]), Elem<InT>::to_f32(pr[j]), acc);
  acc = warp_sum(acc);
  if (lane == 0) s_dot[warp] = acc;
  __syncthreads();
  const float s = warp_sum(lane < 8 ? s_dot[lane] : 0.0f);
  OutT* yr = dx + row * cols;
  for (int64_t j = t; j < cols; j += 256) {
    float q = 0.0f;
    if (j < L)
      q = __fmul_rn(Elem<InT>::to_f32(pr[j]), __fsub_rn(Elem<InT>::to_f32(gq[j]), s));
    yr[j] = Elem<OutT>::from_f32(q);
  }
}

}  // namespace smx
