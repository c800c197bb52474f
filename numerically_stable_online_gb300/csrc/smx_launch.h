// Internal interface between the host API (smx_api.cu) and the per-input-type
// kernel instantiation units (inst_*.cu).  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace smx {

enum Path : int {
  PATH_AUTO = 0, PATH_REGS = 1, PATH_CLUSTER = 2, PATH_GENERIC = 3, PATH_STREAM = 4, PATH_SPLIT = 5,
  PATH_STRIPE = 6
};

struct Call {
  const void* x;
  void* y;
  float* m_out;
  float* d_out;
  int64_t rows, cols;
  const int32_t* valid_len;
  int in_dtype, out_dtype;  // smx_dtype values
  int mode;                 // 0 softmax, 1 row statistics (LSE if d_out is null), 2 apply given
                            // statistics, 3 log_softmax, 5 cross-entropy (the kernels' MODE_*
                            // values), CALL_BACKWARD
  cudaStream_t stream;
  int* status;              // device status word
  int64_t max_polls;        // bound of each staging wait
  const float* m_in = nullptr;  // apply: per-row statistics
  const float* d_in = nullptr;
  const void* g = nullptr;      // backward: the upstream gradient (x is the forward output p)
  const int64_t* target = nullptr;  // cross-entropy: target index per row
  float* loss = nullptr;            // cross-entropy: loss per row
};

// Call::mode of the softmax backward (past the kernels' MODE_* values).
constexpr int CALL_BACKWARD = 8;

struct Plan {
  int path = PATH_GENERIC;
  // register-resident rows
  int threads = 256;  // threads per CTA
  int vpt = 1;        // 16-byte vectors per thread
  bool warp_rows = false;
  // streamed rows: `stages` rows prefetched per CTA (2 or 3), `ctas` CTAs
  int stages = 0, ctas = 0;
  // cluster rows
  int cluster = 1;
  int64_t chunk = 0;       // elements per CTA
  int64_t smem_elems = 0;  // staged elements per CTA
  bool stage_tma = true;   // stage with bulk copies (TMA) or per-thread cp.async
  // split rows: slabs of slab_rows rows, chunks of `chunk` elements
  int64_t slab_rows = 0;
  bool fused_split = false;  // long rows in one cooperative launch of fused_ctas (all resident)
  int fused_ctas = 0;
  int l2_hint_stats = 0;  // L2 policies of the two passes' reads (Items::l2_hint)
  int l2_hint_apply = 0;
  int resident_clusters = 0;
  int nchunks = 0;
  float* scratch = nullptr;  // the long-row paths' summaries (the library's per-device scratch)
  bool fixed_scratch = false;  // scratch is the fixed array of smx_softmax_rows_fixed_scratch
  // read-once long rows (kernel_stripe.cuh): Q stripes per row, row groups,
  // shared-memory ring slots of slot_vecs 16-byte vectors; the per-row
  // counter arrays (this call's and the next call's)
  int stripe_q = 0, stripe_groups = 0, stripe_slots = 0, stripe_slot_vecs = 0;
  unsigned* stripe_count = nullptr;
  unsigned* stripe_count_next = nullptr;
  int64_t stripe_count_next_n = 0;
  int64_t stripe_probe = 0;  // > 0: the count waits' error-path probe (paths 5 fused and 6)
  int stripe_lag = 4;    // path 6: rows between summary and normalisation
  int stripe_piece = 0;  // path 6: bytes per bulk copy of a stripe (0: one)
  int stripe_l2_ahead = 0;  // path 6: rows past a fill whose stripe is prefetched into L2 (0: off)
};

// The read-once long-row kernel (kernel_stripe.cuh).  SMX_STRIPE_COMPUTE_WARPS
// (a build-time tuning knob) sets its compute warps.
#ifndef SMX_STRIPE_COMPUTE_WARPS
#define SMX_STRIPE_COMPUTE_WARPS 27
#endif
constexpr int STRIPE_COLLECT_WARPS = 3;                       // collector warps (rows round robin)
constexpr int STRIPE_SYNC_WARPS = 2 + STRIPE_COLLECT_WARPS;   // + the producer and publisher warps
constexpr int STRIPE_COMPUTE_WARPS = SMX_STRIPE_COMPUTE_WARPS;
constexpr int STRIPE_THREADS = 32 * (STRIPE_COMPUTE_WARPS + STRIPE_SYNC_WARPS);
constexpr int STRIPE_COMPUTE_THREADS = 32 * STRIPE_COMPUTE_WARPS;
constexpr int STRIPE_MAX_VPT = 4;      // 16-byte vectors per compute thread (registers): 2 or 4
constexpr int STRIPE_LAG = 6;          // most rows between a stripe's summary and its normalisation
constexpr int STRIPE_RING = 8;         // summary / row-constant ring entries (>= LAG + 1)
constexpr int STRIPE_MAX_SLOTS = 16;   // shared-memory ring slots (>= lag + 2)
constexpr int STRIPE_MIN_SLOTS = 6;    // the planner's smallest ring (lag 4 and two copies in flight)
constexpr int STRIPE_MIN_SLOTS_TWO = 4;  // ... for the backward, whose slots hold two stripes (lag 2)
constexpr int STRIPE_MAX_Q = 256;      // stripes per row (at most 8 summaries per collector lane)
constexpr int STRIPE_DEFAULT_LAG = 6;  // rows of lag the planner gives (1..STRIPE_LAG, at most slots - 2)
constexpr float STRIPE_FAST_RANGE = 11.0f;  // kept exponentials: a warp's range for the plain exp2 form
constexpr int STRIPE_DEFAULT_PIECE = 0;  // bytes per bulk copy of a stripe (0: one copy)
constexpr int STRIPE_DEFAULT_L2_AHEAD = 2;  // rows past a fill whose stripe is prefetched into L2
static_assert(STRIPE_COMPUTE_WARPS <= 27 && STRIPE_THREADS <= 1024, "one CTA of at most 1024 threads");
static_assert(STRIPE_RING >= STRIPE_LAG + 1, "a row's summary and constants live until its normalisation");

constexpr int CLUSTER_RV = 2;  // register vectors per thread on the cluster path
constexpr int CLUSTER_THREADS = 1024;

// Kernels launched by the calling thread's current library call (a testing
// and benchmarking count; reset by each entry point).
extern thread_local int t_kernel_launches;
inline void note_launch() { ++t_kernel_launches; }

// Attention forward (inst_attention.cu): q [heads][sq][d], k, v [heads][sk][d],
// o like q, lse [heads][sq] fp32 or null; d 64 or 128; dtype fp16 (1) or bf16 (2).
struct AttnCall {
  const void *q, *k, *v;
  void* o;
  float* lse;
  int64_t heads, sq, sk;
  int d;
  double scale;
  int causal;
  int dtype;
  cudaStream_t stream;
  int* status = nullptr;   // device status word (bounded waits of the tcgen05 kernel)
  int64_t max_polls = 0;
  int64_t probe_polls = 0;    // > 0: the tcgen05 kernel's error-path probe (a wait that runs out)
  int kernel = 0;              // ATTN_TILE, ATTN_TMA1, ATTN_MMA_SYNC or ATTN_TMA2
  int sm_count = 0;            // the persistent kernels' grid
};
// attention kernels (tcgen05 unless named): one 128-row query tile per CTA,
// operands copied by the row threads (cp.async); one tile per CTA, operands
// fetched by tensor-map copies in their own warps; mma.sync; two tiles per
// CTA sharing the tensor-map fetched stages
constexpr int ATTN_TILE = 0, ATTN_TMA1 = 1, ATTN_MMA_SYNC = 2, ATTN_TMA2 = 3;
cudaError_t launch_attention(const AttnCall& c);

// Launch the planned kernel(s) for one input type; returns the first CUDA error.
cudaError_t launch_in_f32(const Call& c, const Plan& p);
cudaError_t launch_in_f16(const Call& c, const Plan& p);
cudaError_t launch_in_bf16(const Call& c, const Plan& p);

// Clusters of `cluster` CTAs with `smem_bytes` of dynamic shared memory each that
// can be resident at once (0 if that cluster size cannot launch).
int cluster_capacity_f32(int cluster, int64_t smem_bytes);
int cluster_capacity_f16(int cluster, int64_t smem_bytes);
int cluster_capacity_bf16(int cluster, int64_t smem_bytes);

// Resident CTAs per SM of the streamed kernel for this input type and shape.
int stream_occupancy_f32(int vpt, int threads, int depth, int mode, bool warp);
int stream_occupancy_f16(int vpt, int threads, int depth, int mode, bool warp);
int stream_occupancy_bf16(int vpt, int threads, int depth, int mode, bool warp);
int split_occupancy_f32(int threads);
int split_occupancy_f16(int threads);
int split_occupancy_bf16(int threads);
int split_fused_occupancy_f32(int threads);
int split_fused_occupancy_f16(int threads);
int split_fused_occupancy_bf16(int threads);
// ... of the read-once long-row kernel with `smem` bytes of ring, and its
// static shared memory (-1 if the query failed).
int stripe_occupancy_f32(int64_t smem);
int stripe_occupancy_f16(int64_t smem);
int stripe_occupancy_bf16(int64_t smem);
int stripe_static_smem_f32();
int stripe_static_smem_f16();
int stripe_static_smem_bf16();
// ... of the backward kernels: whole rows (vpt, threads) or chunks (vpt = 0).
int backward_occupancy_f32(int vpt, int threads);
int backward_occupancy_f16(int vpt, int threads);
int backward_occupancy_bf16(int vpt, int threads);

constexpr int BWD_MAX_ROW_BYTES = 16384;  // whole rows per CTA; longer rows in chunks

constexpr int STREAM_MAX_ROW_BYTES = 32768;
constexpr int WARP_WALKER_THREADS = 128;  // CTA of the warp walkers: 4 independent warps

// Scratch of the long-row slab path for slabs of `slab` rows of `nchunks`
// chunks: the chunk summaries (m, then d).
inline size_t split_scratch_bytes(int64_t slab, int64_t nchunks) {
  return (size_t)(2 * slab * nchunks) * sizeof(float);
}

// The split path's single cooperative launch (kernel_split_fused.cuh): when
// planned, for the softmax, log_softmax and the cross-entropy with a gradient.
inline bool split_uses_fused(const Call& c, const Plan& p) {
  return p.fused_split && !p.fixed_scratch &&
         (c.mode == 0 || c.mode == 3 || (c.mode == 5 && c.y != nullptr));
}
// The split path's statistics-only calls (row statistics, LSE, the loss
// alone) read every element once, in one slab of all rows.
inline bool split_read_once(const Call& c, const Plan& p) {
  return (c.mode == 1 || (c.mode == 5 && c.y == nullptr)) &&
         c.rows * p.nchunks <= ((int64_t)1 << 31) && !p.fixed_scratch;
}

// Device scratch (bytes) a planned call needs: the long-row paths' summaries.
inline size_t plan_scratch_bytes(const Call& c, const Plan& p) {
  if (p.path == PATH_STRIPE) return (size_t)c.rows * p.stripe_q * 2 * sizeof(float);
  if (p.path != PATH_SPLIT) return 0;
  const int64_t slab = p.slab_rows < c.rows ? p.slab_rows : c.rows;
  if (c.mode == CALL_BACKWARD) return (size_t)slab * p.nchunks * sizeof(float);
  if (c.mode == 2) return 0;  // the apply mode has its statistics
  if (split_uses_fused(c, p))
    return split_scratch_bytes(c.rows, p.nchunks) + (size_t)c.rows * sizeof(unsigned);
  return split_scratch_bytes(split_read_once(c, p) ? c.rows : slab, p.nchunks);
}

// Dynamic shared memory of the streamed kernel: `depth` rows of vpt 16-byte
// vectors for each of the CTA's threads, and an 8-byte word per thread per row
// for the row's own values (target, given statistics).
inline int64_t stream_smem_bytes(int depth, int vpt, int threads) {
  return (int64_t)depth * vpt * threads * 16 + (int64_t)depth * threads * 8;
}

cudaError_t launch_merge(const float* m_a, const float* d_a, const float* m_b, const float* d_b,
                         float* m_o, float* d_o, int64_t n, cudaStream_t stream);

}  // namespace smx
