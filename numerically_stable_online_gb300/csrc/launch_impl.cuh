// Kernel selection and launch for one input type.  Included once per input
// type by inst_f32.cu, inst_f16.cu and inst_bf16.cu (so the instantiations
// compile in parallel) with SMX_IN_T and SMX_SUFFIX defined.
#pragma once

#include <mutex>
#include <unordered_map>

#include "kernel_backward.cuh"
#include "kernel_cluster.cuh"
#include "kernel_generic.cuh"
#include "kernel_stream.cuh"
#include "kernel_regs.cuh"
#include "kernel_split_fused.cuh"
#include "kernel_stripe.cuh"
#include "smx_launch.h"

namespace smx {
namespace {

constexpr int64_t MAX_GRID_X_ROWS = int64_t(1) << 30;

// The dynamic-shared-memory limit of a kernel is only ever raised: launches and
// occupancy queries of one kernel with different sizes share the attribute, so
// lowering it for one would make another's launch fail.  The largest value set
// per (device, kernel) is kept here.
inline cudaError_t smem_raise(const void* kern, int64_t bytes) {
  static std::mutex mu;
  static std::unordered_map<const void*, int64_t> set[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  int64_t& have = set[dev][kern];
  if (have >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}
constexpr int64_t MAX_GRID_Y = 65535;

template <typename InT, typename OutT, int MODE, int VPT, bool WR>
cudaError_t launch_regs_vpt(const Call& c, const Plan& p) {
  constexpr int V = Elem<InT>::V;
  if constexpr (VPT * V > 32) {
    return cudaErrorInvalidValue;
  } else {
    const int rows_per_cta = WR ? p.threads / 32 : 1;
    for (int64_t r0 = 0; r0 < c.rows; r0 += MAX_GRID_X_ROWS) {
      const int64_t n = c.rows - r0 < MAX_GRID_X_ROWS ? c.rows - r0 : MAX_GRID_X_ROWS;
      const unsigned grid = (unsigned)((n + rows_per_cta - 1) / rows_per_cta);
      note_launch();
      k_rows_regs<InT, OutT, VPT, WR, MODE><<<grid, p.threads, 0, c.stream>>>(
          static_cast<const InT*>(c.x), static_cast<OutT*>(c.y), c.m_out, c.d_out, r0 + n, c.cols,
          c.valid_len, r0);
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
}

template <typename InT, typename OutT, int MODE, bool WR>
cudaError_t launch_regs_wr(const Call& c, const Plan& p) {
  switch (p.vpt) {
    case 1: return launch_regs_vpt<InT, OutT, MODE, 1, WR>(c, p);
    case 2: return launch_regs_vpt<InT, OutT, MODE, 2, WR>(c, p);
    case 4: return launch_regs_vpt<InT, OutT, MODE, 4, WR>(c, p);
    case 8: return launch_regs_vpt<InT, OutT, MODE, 8, WR>(c, p);
    default: return cudaErrorInvalidValue;
  }
}

template <typename InT, typename OutT, int MODE, bool TMA>
cudaError_t prepare_cluster_kernel(int64_t smem_bytes) {
  auto kern = k_rows_cluster<InT, OutT, CLUSTER_RV, MODE, TMA>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  static bool nonportable[64] = {};
  if (!nonportable[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    nonportable[dev] = true;
  }
  return smem_raise(reinterpret_cast<const void*>(kern), smem_bytes);
}

template <typename InT, typename OutT, int MODE, bool TMA>
cudaError_t launch_cluster_t(const Call& c, const Plan& p) {
  const int64_t smem_bytes = p.smem_elems * (int64_t)sizeof(InT) > 16
                                 ? p.smem_elems * (int64_t)sizeof(InT)
                                 : 16;
  cudaError_t e = prepare_cluster_kernel<InT, OutT, MODE, TMA>(smem_bytes);
  if (e != cudaSuccess) return e;
  // persistent: p.ctas clusters, each walking its rows
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.cluster, (unsigned)p.ctas, 1);
  cfg.blockDim = dim3(CLUSTER_THREADS, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem_bytes;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  note_launch();
  return cudaLaunchKernelEx(&cfg, k_rows_cluster<InT, OutT, CLUSTER_RV, MODE, TMA>,
                            static_cast<const InT*>(c.x), static_cast<OutT*>(c.y), c.m_out, c.d_out,
                            c.rows, c.cols, c.valid_len, p.chunk, p.smem_elems, c.max_polls,
                            c.status);
}

template <typename InT, typename OutT, int MODE>
cudaError_t launch_cluster(const Call& c, const Plan& p) {
  return p.stage_tma ? launch_cluster_t<InT, OutT, MODE, true>(c, p)
                     : launch_cluster_t<InT, OutT, MODE, false>(c, p);
}

// One launch of the streamed kernel over the items `it`.
template <typename InT, typename OutT, int MODE, int VPT, int DEPTH, bool CHUNKED, bool WARP = false>
cudaError_t launch_stream_k(const Call& c, const Plan& p, const Items& it, float* m_out, float* d_out,
                            const float* m_in, const float* d_in) {
  constexpr int V = Elem<InT>::V;
  // at most 16 elements per thread with the compensated exponential (fp32
  // outputs) or a per-element exponential after the sum, and 32 otherwise
  constexpr bool PER_ELEMENT_EXP = ExpPolicy<OutT, MODE>::ACCURATE ||
                                   (MODE == MODE_APPLY && (!WARP || ExpPolicy<OutT, MODE_SOFTMAX>::ACCURATE)) ||
                                   MODE == MODE_APPLY_CE ||
                                   (MODE == MODE_CE && ExpPolicy<OutT, MODE_SOFTMAX>::ACCURATE);
  if constexpr (VPT * V > (PER_ELEMENT_EXP ? 16 : 32)) {
    return cudaErrorInvalidValue;
  } else {
    auto kern = k_rows_stream<InT, OutT, VPT, MODE, DEPTH, CHUNKED, WARP>;
    const int64_t smem = stream_smem_bytes(DEPTH, VPT, p.threads);  // walkers x their rings
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    e = smem_raise(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    const int64_t walkers = WARP ? p.threads / 32 : 1;  // rows a CTA walks at once
    const int64_t need = (it.n + walkers - 1) / walkers;
    const int64_t grid = need < p.ctas ? need : p.ctas;
    note_launch();
    kern<<<(unsigned)grid, p.threads, (size_t)smem, c.stream>>>(
        static_cast<const InT*>(c.x), static_cast<OutT*>(c.y), m_out, d_out, m_in, d_in, it,
        c.valid_len, c.target, c.loss);
    return cudaGetLastError();
  }
}

template <typename InT, typename OutT, int MODE, int VPT>
cudaError_t launch_stream_v(const Call& c, const Plan& p, const Items& it) {
  if (p.warp_rows) {  // a row per warp, p.stages rows prefetched per warp
    switch (p.stages) {
      case 3: return launch_stream_k<InT, OutT, MODE, VPT, 3, false, true>(c, p, it, c.m_out, c.d_out, nullptr, nullptr);
      case 4: return launch_stream_k<InT, OutT, MODE, VPT, 4, false, true>(c, p, it, c.m_out, c.d_out, nullptr, nullptr);
      default: return launch_stream_k<InT, OutT, MODE, VPT, 2, false, true>(c, p, it, c.m_out, c.d_out, nullptr, nullptr);
    }
  }
  switch (p.stages) {
    case 3: return launch_stream_k<InT, OutT, MODE, VPT, 3, false>(c, p, it, c.m_out, c.d_out, nullptr, nullptr);
    case 4: return launch_stream_k<InT, OutT, MODE, VPT, 4, false>(c, p, it, c.m_out, c.d_out, nullptr, nullptr);
    default: return launch_stream_k<InT, OutT, MODE, VPT, 2, false>(c, p, it, c.m_out, c.d_out, nullptr, nullptr);
  }
}

// Whole rows: softmax, row statistics (or LSE), log_softmax; or the apply mode
// with the given per-row statistics, each row one chunk.
template <typename InT, typename OutT, int MODE>
cudaError_t launch_stream(const Call& c, const Plan& p) {
  if constexpr (MODE == MODE_APPLY) {
    const Items it{c.rows, 0, c.cols, (int)c.cols, 1, 0, 1};
    if (p.warp_rows) {  // whole rows a warp each (16-bit outputs), the given statistics per row
      switch (p.vpt) {
        case 1: return launch_stream_k<InT, OutT, MODE, 1, 2, false, true>(c, p, it, nullptr, nullptr, c.m_in, c.d_in);
        case 2: return launch_stream_k<InT, OutT, MODE, 2, 2, false, true>(c, p, it, nullptr, nullptr, c.m_in, c.d_in);
        case 4: return launch_stream_k<InT, OutT, MODE, 4, 2, false, true>(c, p, it, nullptr, nullptr, c.m_in, c.d_in);
        case 8: return launch_stream_k<InT, OutT, MODE, 8, 2, false, true>(c, p, it, nullptr, nullptr, c.m_in, c.d_in);
        default: return cudaErrorInvalidValue;
      }
    }
    switch (p.vpt) {
      case 1: return launch_stream_k<InT, OutT, MODE, 1, 2, true>(c, p, it, nullptr, nullptr, c.m_in, c.d_in);
      case 2: return launch_stream_k<InT, OutT, MODE, 2, 2, true>(c, p, it, nullptr, nullptr, c.m_in, c.d_in);
      case 4: return launch_stream_k<InT, OutT, MODE, 4, 2, true>(c, p, it, nullptr, nullptr, c.m_in, c.d_in);
      default: return cudaErrorInvalidValue;
    }
  } else {
    const Items it{c.rows, 0, c.cols, (int)c.cols, 1, 0, 0};
    switch (p.vpt) {
      case 1: return launch_stream_v<InT, OutT, MODE, 1>(c, p, it);
      case 2: return launch_stream_v<InT, OutT, MODE, 2>(c, p, it);
      case 4: return launch_stream_v<InT, OutT, MODE, 4>(c, p, it);
      case 8: return launch_stream_v<InT, OutT, MODE, 8>(c, p, it);
      default: return cudaErrorInvalidValue;
    }
  }
}

// One cooperative launch over all slabs: chunk summaries, per-row completion
// counts, merge and normalise (kernel_split_fused.cuh).  Scratch: the chunk
// summaries of every row and one counter per row, zeroed on the stream first.
template <typename InT, typename OutT, int MODE>
cudaError_t launch_split_fused(const Call& c, const Plan& p) {
  constexpr int SV = 16 / Elem<InT>::V;
  auto kern = k_rows_split<InT, OutT, MODE, SV, 2>;
  const int64_t smem = 2LL * SV * p.threads * 16;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  e = smem_raise(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  // every CTA of a cooperative grid must be resident: size it by this
  // instantiation's own occupancy
  static int resident[64][2] = {};  // per device: threads asked, CTAs resident (asked once)
  if (resident[dev][0] != p.threads) {
    int occ = 0, sms = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, p.threads, (size_t)smem)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    if (occ <= 0) return cudaErrorInvalidConfiguration;
    resident[dev][1] = occ * sms;
    resident[dev][0] = p.threads;
  }
  const int grid = p.fused_ctas < resident[dev][1] ? p.fused_ctas : resident[dev][1];
  const size_t n_sum = (size_t)c.rows * p.nchunks;
  char* base = reinterpret_cast<char*>(p.scratch);  // the library's per-device scratch
  if (base == nullptr) return cudaErrorInvalidValue;
  SplitArgs a;
  a.rows = c.rows;
  a.cols = c.cols;
  a.nchunks = p.nchunks;
  a.slab = p.slab_rows < c.rows ? p.slab_rows : c.rows;
  a.ms = reinterpret_cast<float*>(base);
  a.ds = a.ms + n_sum;
  a.count = reinterpret_cast<unsigned*>(a.ds + n_sum);
  a.target = c.target;
  a.loss = c.loss;
  a.max_polls = c.max_polls;
  a.probe = p.stripe_probe;
  a.status = c.status;
  e = cudaMemsetAsync(a.count, 0, (size_t)c.rows * sizeof(unsigned), c.stream);
  if (e != cudaSuccess) return e;
  const InT* xp = static_cast<const InT*>(c.x);
  OutT* yp = static_cast<OutT*>(c.y);
  const int32_t* vl = c.valid_len;
  void* args[] = {(void*)&xp, (void*)&yp, (void*)&a, (void*)&vl};
  note_launch();
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3((unsigned)grid),
                                     dim3((unsigned)p.threads), args, (size_t)smem, c.stream);
}

// Long rows read once (kernel_stripe.cuh): one cooperative launch of
// groups x Q CTAs, each row's stripes kept in shared memory from their
// summary to their normalisation.  p.scratch holds the stripe summaries;
// p.stripe_count / p.stripe_count_next the two counter arrays (this call's,
// zero; the next call's, zeroed by the kernel).
template <typename InT, typename OutT, int MODE, int VPT>
cudaError_t launch_stripe_v(const Call& c, const Plan& p) {
  auto kern = k_rows_stripe<InT, OutT, MODE, VPT>;
  const int64_t smem = (int64_t)p.stripe_slots * p.stripe_slot_vecs * 16;
  cudaError_t e = smem_raise(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  if (p.scratch == nullptr || p.stripe_count == nullptr) return cudaErrorInvalidValue;
  // a compute thread's vectors of one stripe (the backward's slots hold two)
  if (p.stripe_slot_vecs / (MODE == MODE_BWD ? 2 : 1) > VPT * STRIPE_COMPUTE_THREADS) return cudaErrorInvalidValue;
  StripeArgs a;
  a.rows = c.rows;
  a.cols = c.cols;
  a.Q = p.stripe_q;
  a.groups = p.stripe_groups;
  a.nslots = p.stripe_slots;
  a.slot_vecs = p.stripe_slot_vecs;
  a.g = c.g;
  a.sums = reinterpret_cast<float2*>(p.scratch);
  a.count = p.stripe_count;
  a.count_next = p.stripe_count_next;
  a.count_next_n = p.stripe_count_next_n;
  a.target = c.target;
  a.loss = c.loss;
  a.max_polls = c.max_polls;
  a.probe = p.stripe_probe;
  a.lag = p.stripe_lag;
  a.piece_bytes = p.stripe_piece;
  a.l2_ahead = p.stripe_l2_ahead;
  a.status = c.status;
  const InT* xp = static_cast<const InT*>(c.x);
  OutT* yp = static_cast<OutT*>(c.y);
  const int32_t* vl = c.valid_len;
  void* args[] = {(void*)&xp, (void*)&yp, (void*)&a, (void*)&vl};
  note_launch();
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern),
                                     dim3((unsigned)(p.stripe_q * p.stripe_groups)), dim3(STRIPE_THREADS),
                                     args, (size_t)smem, c.stream);
}

template <typename InT, typename OutT, int MODE>
cudaError_t launch_stripe(const Call& c, const Plan& p) {
  switch (p.vpt) {
    case 2: return launch_stripe_v<InT, OutT, MODE, 2>(c, p);
    case 4: return launch_stripe_v<InT, OutT, MODE, 4>(c, p);
    default: return cudaErrorInvalidValue;
  }
}

// Resident CTAs per SM of the stripe kernel with `smem` bytes of ring (every
// mode and output type must fit as many; the fp32 softmax, the bf16 and fp32
// cross-entropy, the log_softmax and the fp32 backward stand for them).
template <typename InT>
int stripe_occupancy(int64_t smem) {
  auto query = [&](auto kern) -> int {
    int n = 0;
    if (smem_raise(reinterpret_cast<const void*>(kern), smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, STRIPE_THREADS, (size_t)smem) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return n;
  };
  int n = query(k_rows_stripe<InT, float, MODE_SOFTMAX, STRIPE_MAX_VPT>);
  const int n2 = query(k_rows_stripe<InT, __nv_bfloat16, MODE_CE, STRIPE_MAX_VPT>);
  const int n3 = query(k_rows_stripe<InT, float, MODE_CE, STRIPE_MAX_VPT>);
  const int n4 = query(k_rows_stripe<InT, __nv_bfloat16, MODE_LOG, STRIPE_MAX_VPT>);
  const int n5 = query(k_rows_stripe<InT, float, MODE_BWD, STRIPE_MAX_VPT>);
  n = n2 < n ? n2 : n;
  n = n3 < n ? n3 : n;
  n = n5 < n ? n5 : n;
  return n4 < n ? n4 : n;
}

// Static shared memory of the stripe kernel (the ring is dynamic).
template <typename InT>
int stripe_static_smem() {
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, k_rows_stripe<InT, float, MODE_CE, STRIPE_MAX_VPT>) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return (int)fa.sharedSizeBytes;
}

// Resident CTAs per SM of the one-launch long-row kernel (the fp32-output
// softmax stands for the family).
template <typename InT>
int split_fused_occupancy(int threads) {
  constexpr int SV = 16 / Elem<InT>::V;
  auto kern = k_rows_split<InT, float, MODE_SOFTMAX, SV, 2>;
  const int64_t smem = 2LL * SV * threads * 16;
  int n = 0;
  if (smem_raise(reinterpret_cast<const void*>(kern), smem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, (size_t)smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  // every output type must fit as many
  auto kb = k_rows_split<InT, __nv_bfloat16, MODE_CE, SV, 2>;
  int n2 = 0;
  if (smem_raise(reinterpret_cast<const void*>(kb), smem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n2, kb, threads, (size_t)smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  auto kc = k_rows_split<InT, float, MODE_CE, SV, 2>;
  int n3 = 0;
  if (smem_raise(reinterpret_cast<const void*>(kc), smem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n3, kc, threads, (size_t)smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  n = n2 < n ? n2 : n;
  return n3 < n ? n3 : n;
}

// Long rows in chunks of 16 elements per thread.  Softmax and log_softmax, in
// slabs of rows: the streamed kernel computes every chunk's summary, then
// normalises every chunk with its row's merged (M, D); row statistics (or LSE)
// merge the summaries instead.  The summaries live in a stream-ordered scratch
// allocation for the call, or in p.scratch when given.  The apply mode has its
// statistics and takes one pass over all rows.
template <typename InT, typename OutT, int MODE>
cudaError_t launch_split(const Call& c, const Plan& p) {
  constexpr int SV = 16 / Elem<InT>::V;
  if constexpr (MODE == MODE_APPLY) {
    const Items it{c.rows * p.nchunks, 0, c.cols, (int)p.chunk, p.nchunks, 0, 1};
    return launch_stream_k<InT, OutT, MODE_APPLY, SV, 2, true>(c, p, it, nullptr, nullptr, c.m_in,
                                                               c.d_in);
  } else {
    // softmax, log_softmax and the cross-entropy with its gradient: one
    // persistent cooperative launch (kernel_split_fused.cuh) when planned
    if (split_uses_fused(c, p)) {
      if constexpr (MODE == MODE_SOFTMAX || MODE == MODE_LOG || MODE == MODE_CE)
        return launch_split_fused<InT, OutT, MODE>(c, p);
    }
    // the statistics-only calls (row statistics, LSE, the loss alone) read
    // every element once: one slab of all rows
    const bool read_once = split_read_once(c, p);
    // a slab is never more rows than the call has (the scratch is sized by it)
    const int64_t slab = (read_once || p.slab_rows > c.rows) ? c.rows : p.slab_rows;
    const size_t part_n = (size_t)slab * p.nchunks;
    char* base = reinterpret_cast<char*>(p.scratch);  // the library's or the caller's scratch
    if (base == nullptr) return cudaErrorInvalidValue;
    cudaError_t e = cudaSuccess;
    float* pm = reinterpret_cast<float*>(base);
    float* pd = pm + part_n;
    for (int64_t r0 = 0; r0 < c.rows && e == cudaSuccess; r0 += slab) {
      const int64_t n = c.rows - r0 < slab ? c.rows - r0 : slab;
      const Items st{n * p.nchunks, r0, c.cols, (int)p.chunk, p.nchunks, p.l2_hint_stats, 0};
      e = launch_stream_k<InT, float, MODE_STATS, SV, 2, true>(c, p, st, pm, pd, nullptr, nullptr);
      if (e != cudaSuccess) break;
      const Items ap{n * p.nchunks, r0, c.cols, (int)p.chunk, p.nchunks, p.l2_hint_apply, 0};
      if constexpr (MODE == MODE_SOFTMAX) {
        e = launch_stream_k<InT, OutT, MODE_APPLY, SV, 2, true>(c, p, ap, nullptr, nullptr, pm, pd);
      } else if constexpr (MODE == MODE_LOG) {
        e = launch_stream_k<InT, OutT, MODE_APPLY_LOG, SV, 2, true>(c, p, ap, nullptr, nullptr, pm, pd);
      } else if constexpr (MODE == MODE_CE) {
        if (c.y != nullptr) {
          e = launch_stream_k<InT, OutT, MODE_APPLY_CE, SV, 2, true>(c, p, ap, nullptr, nullptr, pm, pd);
        } else {
          note_launch();
          k_merge_chunk_ce<InT, 256><<<(unsigned)n, 256, 0, c.stream>>>(
              pm, pd, p.nchunks, static_cast<const InT*>(c.x), c.cols, c.target, c.valid_len, r0, c.loss);
          e = cudaGetLastError();
        }
      } else {
        note_launch();
        k_merge_chunk_stats<256><<<(unsigned)n, 256, 0, c.stream>>>(
            pm, pd, p.nchunks, c.m_out + r0, c.d_out == nullptr ? nullptr : c.d_out + r0);
        e = cudaGetLastError();
      }
    }
    return e;
  }
}

template <typename InT, typename OutT, int MODE>
cudaError_t launch_generic(const Call& c) {
  for (int64_t r0 = 0; r0 < c.rows; r0 += MAX_GRID_X_ROWS) {
    const int64_t n = c.rows - r0 < MAX_GRID_X_ROWS ? c.rows - r0 : MAX_GRID_X_ROWS;
    note_launch();
    k_rows_generic<InT, OutT, MODE><<<(unsigned)n, GENERIC_THREADS, 0, c.stream>>>(
        static_cast<const InT*>(c.x), static_cast<OutT*>(c.y), c.m_out, c.d_out, c.m_in, c.d_in,
        r0 + n, c.cols, c.valid_len, r0, c.target, c.loss);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ---------------------------------------------------------------------------
// Softmax backward.  c.x = p, c.g = g, c.y = dx.
template <typename InT, typename OutT, int VPT, int MODE>
cudaError_t launch_bwd_k(const Call& c, const Plan& p, const Items& it, float* part_out,
                         const float* part_in) {
  auto kern = k_backward<InT, OutT, VPT, MODE, 2>;
  const int64_t smem = 2 * stream_smem_bytes(2, VPT, p.threads);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  e = smem_raise(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = it.n < p.ctas ? it.n : p.ctas;
  note_launch();
  kern<<<(unsigned)grid, p.threads, (size_t)smem, c.stream>>>(
      static_cast<const InT*>(c.x), static_cast<const InT*>(c.g), static_cast<OutT*>(c.y), part_out,
      part_in, it, c.valid_len);
  return cudaGetLastError();
}

template <typename InT, typename OutT>
cudaError_t launch_backward(const Call& c, const Plan& p) {
  constexpr int V = Elem<InT>::V;
  constexpr int SV = 16 / V;
  if (p.path == PATH_STRIPE) return launch_stripe<InT, OutT, MODE_BWD>(c, p);
  if (p.path == PATH_GENERIC) {
    for (int64_t r0 = 0; r0 < c.rows; r0 += MAX_GRID_X_ROWS) {
      const int64_t n = c.rows - r0 < MAX_GRID_X_ROWS ? c.rows - r0 : MAX_GRID_X_ROWS;
      note_launch();
      k_backward_generic<InT, OutT><<<(unsigned)n, 256, 0, c.stream>>>(
          static_cast<const InT*>(c.x), static_cast<const InT*>(c.g), static_cast<OutT*>(c.y), c.cols,
          c.valid_len, r0);
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  if (p.path == PATH_STREAM) {
    const Items it{c.rows, 0, c.cols, (int)c.cols, 1, 0, 0};
    switch (p.vpt) {
      case 1: return launch_bwd_k<InT, OutT, 1, BWD_ROWS>(c, p, it, nullptr, nullptr);
      case 2: return launch_bwd_k<InT, OutT, 2, BWD_ROWS>(c, p, it, nullptr, nullptr);
      case 4:
        if constexpr (4 * V <= 16) return launch_bwd_k<InT, OutT, 4, BWD_ROWS>(c, p, it, nullptr, nullptr);
        return cudaErrorInvalidValue;
      default: return cudaErrorInvalidValue;
    }
  }
  if (p.path != PATH_SPLIT) return cudaErrorInvalidValue;
  // long rows: per slab, the chunks' partial dots, then dx per chunk
  const int64_t slab = p.slab_rows < c.rows ? p.slab_rows : c.rows;  // sizes the scratch
  float* part = p.scratch;  // the library's per-device scratch
  if (part == nullptr) return cudaErrorInvalidValue;
  cudaError_t e = cudaSuccess;
  for (int64_t r0 = 0; r0 < c.rows && e == cudaSuccess; r0 += slab) {
    const int64_t n = c.rows - r0 < slab ? c.rows - r0 : slab;
    const Items it{n * p.nchunks, r0, c.cols, (int)p.chunk, p.nchunks, 0, 0};
    e = launch_bwd_k<InT, float, SV, BWD_DOT>(c, p, it, part, nullptr);
    if (e == cudaSuccess) e = launch_bwd_k<InT, OutT, SV, BWD_APPLY>(c, p, it, nullptr, part);
  }
  return e;
}

template <typename InT>
int backward_occupancy(int vpt, int threads) {
  constexpr int V = Elem<InT>::V;
  auto query = [&](auto kern, int v) -> int {
    const int64_t smem = 2 * stream_smem_bytes(2, v, threads);
    int n = 0;
    if (smem_raise(reinterpret_cast<const void*>(kern), smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, (size_t)smem) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return n;
  };
  switch (vpt) {
    case 0: {  // chunks: the fp32-output apply kernel stands for both passes
      const int a = query(k_backward<InT, float, 16 / V, BWD_APPLY, 2>, 16 / V);
      const int b = query(k_backward<InT, float, 16 / V, BWD_DOT, 2>, 16 / V);
      return a < b ? a : b;
    }
    case 1: return query(k_backward<InT, float, 1, BWD_ROWS, 2>, 1);
    case 2: return query(k_backward<InT, float, 2, BWD_ROWS, 2>, 2);
    case 4:
      if constexpr (4 * V <= 16) return query(k_backward<InT, float, 4, BWD_ROWS, 2>, 4);
      return 0;
    default: return 0;
  }
}

template <typename InT, typename OutT, int MODE>
cudaError_t launch_typed(const Call& c, const Plan& p) {
  constexpr bool CLASSIC = (MODE == MODE_SOFTMAX || MODE == MODE_STATS);
  switch (p.path) {
    case PATH_REGS:
      if constexpr (CLASSIC)
        return p.warp_rows ? launch_regs_wr<InT, OutT, MODE, true>(c, p)
                           : launch_regs_wr<InT, OutT, MODE, false>(c, p);
      return cudaErrorInvalidValue;
    case PATH_CLUSTER:
      if constexpr (CLASSIC) return launch_cluster<InT, OutT, MODE>(c, p);
      return cudaErrorInvalidValue;
    case PATH_GENERIC: return launch_generic<InT, OutT, MODE>(c);
    case PATH_STREAM: return launch_stream<InT, OutT, MODE>(c, p);
    case PATH_SPLIT: return launch_split<InT, OutT, MODE>(c, p);
    case PATH_STRIPE:
      if constexpr (MODE == MODE_SOFTMAX || MODE == MODE_LOG || MODE == MODE_CE) {
        if (MODE != MODE_CE || c.y != nullptr) return launch_stripe<InT, OutT, MODE>(c, p);
      }
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

template <typename InT, int MODE>
cudaError_t launch_out(const Call& c, const Plan& p) {
  switch (c.out_dtype) {
    case 0: return launch_typed<InT, float, MODE>(c, p);
    case 1: return launch_typed<InT, __half, MODE>(c, p);
    case 2: return launch_typed<InT, __nv_bfloat16, MODE>(c, p);
    default: return cudaErrorInvalidValue;
  }
}

template <typename InT>
cudaError_t launch_in(const Call& c, const Plan& p) {
  if (c.mode == CALL_BACKWARD) {
    switch (c.out_dtype) {
      case 0: return launch_backward<InT, float>(c, p);
      case 1: return launch_backward<InT, __half>(c, p);
      case 2: return launch_backward<InT, __nv_bfloat16>(c, p);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (c.mode) {
    case MODE_SOFTMAX: return launch_out<InT, MODE_SOFTMAX>(c, p);
    case MODE_STATS: return launch_typed<InT, float, MODE_STATS>(c, p);
    case MODE_APPLY: return launch_out<InT, MODE_APPLY>(c, p);
    case MODE_LOG: return launch_out<InT, MODE_LOG>(c, p);
    case MODE_CE:
      // the loss alone: no output type; a half type keeps the 32-element shapes
      return c.y == nullptr ? launch_typed<InT, __nv_bfloat16, MODE_CE>(c, p)
                            : launch_out<InT, MODE_CE>(c, p);
    default: return cudaErrorInvalidValue;
  }
}

template <typename InT>
int cluster_capacity(int cluster, int64_t smem_bytes) {
  // the softmax kernel with fp32 output stands for the family (same resources)
  if (prepare_cluster_kernel<InT, float, MODE_SOFTMAX, true>(smem_bytes) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cluster, 1, 1);
  cfg.blockDim = dim3(CLUSTER_THREADS, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem_bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_rows_cluster<InT, float, CLUSTER_RV, MODE_SOFTMAX, true>,
                                     &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <typename InT, typename OutT, int MODE>
int stream_occupancy_mode(int vpt, int threads, int depth, bool warp) {
  const int64_t smem = stream_smem_bytes(depth, vpt, threads);
  auto query = [&](auto kern) -> int {
    int n = 0;
    if (smem_raise(reinterpret_cast<const void*>(kern), smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, (size_t)smem) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return n;
  };
  constexpr int V = Elem<InT>::V;
  constexpr bool CH = (MODE == MODE_APPLY);  // the apply mode runs the chunked kernel, depth 2
  auto by_depth = [&](auto k2, auto k3, auto k4) {
    if (CH) return query(k2);
    return depth == 3 ? query(k3) : (depth == 4 ? query(k4) : query(k2));
  };
  if constexpr (CH) {
    if (warp) {  // the apply mode's warp walkers prefetch 2 rows
      switch (vpt) {
        case 1: return query(k_rows_stream<InT, OutT, 1, MODE, 2, false, true>);
        case 2: return query(k_rows_stream<InT, OutT, 2, MODE, 2, false, true>);
        case 4: return query(k_rows_stream<InT, OutT, 4, MODE, 2, false, true>);
        case 8:
          if constexpr (8 * V <= 32) return query(k_rows_stream<InT, OutT, 8, MODE, 2, false, true>);
          return 0;
        default: return 0;
      }
    }
  }
  if constexpr (!CH) {
    if (warp) {
      auto wd = [&](auto k2, auto k3, auto k4) { return depth == 3 ? query(k3) : (depth == 4 ? query(k4) : query(k2)); };
      switch (vpt) {
        case 1:
          return wd(k_rows_stream<InT, OutT, 1, MODE, 2, false, true>, k_rows_stream<InT, OutT, 1, MODE, 3, false, true>,
                    k_rows_stream<InT, OutT, 1, MODE, 4, false, true>);
        case 2:
          return wd(k_rows_stream<InT, OutT, 2, MODE, 2, false, true>, k_rows_stream<InT, OutT, 2, MODE, 3, false, true>,
                    k_rows_stream<InT, OutT, 2, MODE, 4, false, true>);
        case 4:
          return wd(k_rows_stream<InT, OutT, 4, MODE, 2, false, true>, k_rows_stream<InT, OutT, 4, MODE, 3, false, true>,
                    k_rows_stream<InT, OutT, 4, MODE, 4, false, true>);
        case 8:
          if constexpr (8 * V <= 32)
            return wd(k_rows_stream<InT, OutT, 8, MODE, 2, false, true>, k_rows_stream<InT, OutT, 8, MODE, 3, false, true>,
                      k_rows_stream<InT, OutT, 8, MODE, 4, false, true>);
          return 0;
        default: return 0;
      }
    }
  }
  switch (vpt) {
    case 1:
      return by_depth(k_rows_stream<InT, OutT, 1, MODE, 2, CH>, k_rows_stream<InT, OutT, 1, MODE, CH ? 2 : 3, CH>,
                      k_rows_stream<InT, OutT, 1, MODE, CH ? 2 : 4, CH>);
    case 2:
      return by_depth(k_rows_stream<InT, OutT, 2, MODE, 2, CH>, k_rows_stream<InT, OutT, 2, MODE, CH ? 2 : 3, CH>,
                      k_rows_stream<InT, OutT, 2, MODE, CH ? 2 : 4, CH>);
    case 4:
      if constexpr (4 * V <= 16 || !CH)
        return by_depth(k_rows_stream<InT, OutT, 4, MODE, 2, CH>,
                        k_rows_stream<InT, OutT, 4, MODE, CH ? 2 : 3, CH>,
                        k_rows_stream<InT, OutT, 4, MODE, CH ? 2 : 4, CH>);
      return 0;
    case 8:
      if constexpr (8 * V <= 32 && !CH)
        return by_depth(k_rows_stream<InT, OutT, 8, MODE, 2, CH>, k_rows_stream<InT, OutT, 8, MODE, 3, CH>,
                        k_rows_stream<InT, OutT, 8, MODE, 4, CH>);
      return 0;
    default: return 0;
  }
}

// Resident CTAs per SM of the streamed kernel of `mode` (a half-precision
// output stands for the output types; statistics write fp32).
template <typename InT>
int stream_occupancy(int vpt, int threads, int depth, int mode, bool warp) {
  switch (mode) {
    case MODE_STATS: return stream_occupancy_mode<InT, float, MODE_STATS>(vpt, threads, depth, warp);
    case MODE_LOG: return stream_occupancy_mode<InT, __nv_bfloat16, MODE_LOG>(vpt, threads, depth, warp);
    case MODE_CE: return stream_occupancy_mode<InT, __nv_bfloat16, MODE_CE>(vpt, threads, depth, warp);
    case MODE_APPLY:
      return stream_occupancy_mode<InT, __nv_bfloat16, MODE_APPLY>(vpt, threads, depth, warp);
    default: return stream_occupancy_mode<InT, __nv_bfloat16, MODE_SOFTMAX>(vpt, threads, depth, warp);
  }
}

// Resident CTAs per SM of the long-row kernels (the fp32-output apply kernel,
// the largest, and the statistics kernel) at `threads` threads.
template <typename InT>
int split_occupancy(int threads) {
  constexpr int SV = 16 / Elem<InT>::V;
  const int64_t smem = stream_smem_bytes(2, SV, threads);
  auto query = [&](auto kern) -> int {
    int n = 0;
    if (smem_raise(reinterpret_cast<const void*>(kern), smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, (size_t)smem) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return n;
  };
  const int a = query(k_rows_stream<InT, float, SV, MODE_APPLY, 2, true>);
  const int b = query(k_rows_stream<InT, float, SV, MODE_STATS, 2, true>);
  return a < b ? a : b;
}

}  // namespace
}  // namespace smx
