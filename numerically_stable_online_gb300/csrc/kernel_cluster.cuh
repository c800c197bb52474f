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

#include "kernel_regs.cuh"
#include "smx_launch.h"

namespace smx {

constexpr int CLUSTER_PIECES = 8;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_peer_f32(const float* local, uint32_t rank) {
  uint32_t raddr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(smem_addr(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(raddr) : "memory");
  return v;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: at most max_polls polls, backing off with nanosleep.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, int64_t max_polls) {
  for (int64_t i = 0; i < max_polls; ++i) {
    if (mbar_test_wait(bar, parity)) return true;
    if (i >= 16) __nanosleep(64);
  }
  return false;
}
__device__ __forceinline__ void bulk_load_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

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
  const int64_t v_nv = vend > c0 ? (vend - c0) / V : 0;           // valid vectors
  const int64_t a_nv = smem_elems / V < c_nv ? smem_elems / V : c_nv;  // staged region
  const int64_t s_nv = a_nv < v_nv ? a_nv : v_nv;                 // staged and valid
  const int64_t b_nv = a_nv + (int64_t)T * RV < c_nv ? a_nv + (int64_t)T * RV : c_nv;

  // Piece layout of the staged region.
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

  // Register part: vector A + k*T + t of the chunk.
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

  // Pass 1: this thread's running (m, d).
  float m = neg_inf(), d = 0.0f;
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
      online_fold<V>(m, d, f);
    }
  }
#pragma unroll
  for (int k = 0; k < RV; ++k) online_fold<V>(m, d, r[k]);
  for (int64_t vi = b_nv + t; vi < v_nv; vi += T) {  // streamed remainder, first read
    float f[V];
    load_vec16<InT>(xr + c0 + vi * V, f);
    mask_tail<V>(f, c0 + vi * V, L);
    online_fold<V>(m, d, f);
  }

  // CTA summary: warp butterfly, then the per-warp summaries.
  MD md = warp_merge(MD{m, d});
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
    const float rD = recip_refined(D);
    auto emit = [&](int64_t vi, const float (&f)[V]) {
      const int64_t e0 = c0 + vi * V;
      float p[V];
#pragma unroll
      for (int i = 0; i < V; ++i) {
        if (zero_row) p[i] = 0.0f;
        else if (nan_row) p[i] = (e0 + i < L) ? qnan() : 0.0f;
        else p[i] = __fmul_rn(exp_for<OutT, MODE_SOFTMAX>(f[i], M), rD);
      }
      store_vec<OutT, V>(yr + e0, p);
    };
    // staged region (vectors past the valid data were never loaded: zeros)
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
  }

  if (timed_out) {
    atomicOr(status, DEV_TIMEOUT);
    // let this CTA's own copies land before its shared memory is released
    for (int p = 0; p < CLUSTER_PIECES; ++p) {
      const int64_t p0 = (int64_t)p * piece_nv;
      if (p0 >= s_nv) break;
      mbar_wait_bounded(smem_addr(&bars[p]), 0, int64_t(1) << 22);
    }
  }
  cluster_wait();  // no CTA leaves while a peer may still read its summary
}

}  // namespace smx
