// Host side of the C ABI declared in include/smx.h: argument checks, the
// per-device property cache, the choice of kernel, and launches.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "../../include/smx.h"
#include "kernel_generic.cuh"
#include "smx_launch.h"

// Scratch of smx_softmax_rows_fixed_scratch: 2 floats per chunk, 32768 chunks
// of one slab (256 KiB); larger slabs are cut to fit (a 4 MiB fp32 row is 256
// chunks, so a slab holds 128 such rows).
constexpr int64_t FIXED_SCRATCH_FLOATS = 65536;
static __device__ __align__(256) float g_fixed_scratch[FIXED_SCRATCH_FLOATS];

namespace smx {
thread_local int t_kernel_launches = 0;
namespace {

constexpr int MAX_DEVICES = 64;
constexpr uint64_t SCRATCH_POOL_KEEP_BYTES = 64ull << 20;  // scratch memory kept between calls
constexpr int64_t DEFAULT_MAX_POLLS = int64_t(1) << 21;
// shared memory kept back from the cluster kernel's staging area for its
// static arrays (barriers, per-warp partials, the CTA summary)
constexpr int64_t CLUSTER_STATIC_SMEM = 1024;

// A device buffer of the library's that only grows: reserved at the first call
// that needs it and reallocated only when a call needs more than any before.
struct ScratchBuf {
  char* base = nullptr;
  size_t bytes = 0;
};

// The per-device scratch of the long-row paths and of the staged host-buffer
// call.  Calls that use it are ordered on the device: a call on another stream
// than the previous user's first waits for the event recorded after it, so
// calls on different streams never share the buffers at once.  Held (mutex)
// from the reservation to the event record.
struct ScratchState {
  std::mutex mu;
  cudaEvent_t done = nullptr;       // recorded after the last call that used the scratch
  cudaStream_t last = nullptr;      // that call's stream
  bool used = false;
  ScratchBuf work;                  // chunk / stripe summaries, backward partial dots
  ScratchBuf counts;                // the stripe kernel's two per-row counter arrays, zeroed at growth
  int64_t count_cap = 0;            // rows each counter array holds
  int count_parity = 0;             // which array the next stripe call counts in
  ScratchBuf staging;               // the host-buffer call's device slots
  cudaEvent_t computed[4] = {}, copied[4] = {}, host_done = nullptr;  // the host-buffer call's events
};

struct DeviceInfo {
  std::atomic<bool> ready{false};
  bool supported = false;
  int sm_count = 0;
  int64_t smem_optin = 0;
  int64_t l2_bytes = 0;
  int* status = nullptr;   // device status word
  cudaMemPool_t pool = nullptr;  // the long-row paths' scratch (keeps its memory between calls)
  std::atomic<int> max_cluster[3] = {0, 0, 0};  // per input type, 0 = not queried yet
  bool coop = false;                // cooperative launches supported
  cudaStream_t copy_stream = nullptr;  // the host-buffer call's copies back (created on first use)
  ScratchState scratch;
  int stripe_smem_static[3] = {-1, -1, -1};  // per input type, queried once
};

DeviceInfo g_dev[MAX_DEVICES];
std::mutex g_mutex;

// testing hooks
std::atomic<int> g_force_path{0};
std::atomic<int> g_max_cluster{0};
std::atomic<int64_t> g_smem_cap{0};
std::atomic<int64_t> g_wait_limit{0};
std::atomic<int> g_regs_threads{0};
std::atomic<int> g_regs_vpt{0};
std::atomic<int> g_stream_depth{0};
std::atomic<int> g_stream_ctas_per_sm{0};
std::atomic<int> g_cluster_stage{0};  // 0 automatic, 1 bulk copies, 2 cp.async
std::atomic<int64_t> g_split_slab_bytes{0};
std::atomic<int> g_split_hint_stats{-1}, g_split_hint_apply{-1};
std::atomic<int64_t> g_bwd_inflight{48 * 1024};  // backward: reads in flight per SM
std::atomic<int> g_stream_warp{0};
std::atomic<int> g_split_fused{0};
std::atomic<int64_t> g_host_chunk{0};  // host-buffer call: input bytes a chunk (0 = default)
std::atomic<int> g_host_slots{0};      // host-buffer call: device staging slots (0 = default)
std::atomic<int> g_host_staged{0};     // host-buffer call: 1 = always through the staging slots
std::atomic<int> g_attention_kernel{-1};  // -1: by the call (causal: ATTN_TMA2, else ATTN_TILE); or one of them
std::atomic<int64_t> g_read_only_inflight{96 * 1024};  // LSE / statistics: reads in flight per SM

// Device allocations, events and streams the library has created (a testing
// count: a steady loop of calls adds none).
std::atomic<int64_t> g_alloc_calls{0};
std::atomic<int64_t> g_count_probe{0};
std::atomic<int> g_stripe_lag{0};    // path 6: rows of lag (0: default)
std::atomic<int> g_stripe_piece{-1};  // path 6: bytes per bulk copy (-1: default)
std::atomic<int> g_stripe_l2_ahead{-1};  // path 6: rows prefetched into L2 past a fill (-1: default)  // > 0: the cooperative long-row kernels' error-path probe (polls)

thread_local int t_last_cuda_error = 0;
thread_local int t_last_path = 0;

int elem_size(int dtype) { return dtype == SMX_F32 ? 4 : 2; }
bool valid_dtype(int d) { return d == SMX_F32 || d == SMX_F16 || d == SMX_BF16; }

bool overlaps(const void* a, int64_t na, const void* b, int64_t nb) {
  if (a == nullptr || b == nullptr || na <= 0 || nb <= 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + (uintptr_t)nb && b0 < a0 + (uintptr_t)na;
}

smx_status cuda_fail(cudaError_t e, smx_status code) {
  t_last_cuda_error = (int)e;
  return code;
}

// Current device's cached properties; allocates its status word on first use.
smx_status device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, SMX_ERR_UNSUPPORTED);
  if (dev < 0 || dev >= MAX_DEVICES) return SMX_ERR_UNSUPPORTED;
  DeviceInfo& d = g_dev[dev];
  if (!d.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!d.ready.load(std::memory_order_relaxed)) {
      int major = 0, minor = 0, sms = 0, optin = 0, l2 = 0;
      if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
              cudaSuccess ||
          (e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev)) != cudaSuccess)
        return cuda_fail(e, SMX_ERR_DEVICE);
      d.supported = (major == 10 && minor == 3);
      d.sm_count = sms;
      d.smem_optin = optin;
      d.l2_bytes = l2;
      int coop = 0;
      if ((e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess)
        return cuda_fail(e, SMX_ERR_DEVICE);
      d.coop = coop != 0;
      if (d.supported) {
        int* s = nullptr;
        if ((e = cudaMalloc(&s, sizeof(int))) != cudaSuccess) return cuda_fail(e, SMX_ERR_DEVICE);
        ++g_alloc_calls;
        if ((e = cudaMemset(s, 0, sizeof(int))) != cudaSuccess) return cuda_fail(e, SMX_ERR_DEVICE);
        d.status = s;
        // a pool of the library's own, so that the per-call scratch of the
        // long-row paths reuses memory instead of mapping it anew after every
        // synchronisation (the default pool returns its memory then)
        cudaMemPoolProps props;
        std::memset(&props, 0, sizeof(props));
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if ((e = cudaMemPoolCreate(&pool, &props)) != cudaSuccess) return cuda_fail(e, SMX_ERR_DEVICE);
        uint64_t keep = SCRATCH_POOL_KEEP_BYTES;
        if ((e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess)
          return cuda_fail(e, SMX_ERR_DEVICE);
        d.pool = pool;
        ++g_alloc_calls;
      }
      d.ready.store(true, std::memory_order_release);
    }
  }
  if (!d.supported) return SMX_ERR_UNSUPPORTED;
  *out = &d;
  return SMX_OK;
}

// Make `b` hold at least `bytes` for a call on `stream` (caller holds st.mu).
// Orders the call after the scratch's previous user when that ran on another
// stream; grows the buffer (stream-ordered, zeroed when asked) only when the
// call needs more than any call before.
cudaError_t scratch_reserve(DeviceInfo& d, ScratchBuf& b, size_t bytes, cudaStream_t stream, bool zero) {
  ScratchState& st = d.scratch;
  cudaError_t e;
  if (st.done == nullptr) {
    if ((e = cudaEventCreateWithFlags(&st.done, cudaEventDisableTiming)) != cudaSuccess) return e;
    ++g_alloc_calls;
  }
  if (st.used && st.last != stream) {
    if ((e = cudaStreamWaitEvent(stream, st.done, 0)) != cudaSuccess) return e;
    st.last = stream;  // later reservations of this call need no second wait
  }
  if (bytes <= b.bytes) return cudaSuccess;
  size_t nb = b.bytes + b.bytes / 2;
  if (nb < bytes) nb = bytes;
  nb = (nb + 4095) / 4096 * 4096;
  if (b.base != nullptr) {
    if ((e = cudaFreeAsync(b.base, stream)) != cudaSuccess) return e;
    b.base = nullptr;
    b.bytes = 0;
  }
  if ((e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&b.base), nb, d.pool, stream)) != cudaSuccess) {
    b.base = nullptr;
    return e;
  }
  ++g_alloc_calls;
  b.bytes = nb;
  if (zero && (e = cudaMemsetAsync(b.base, 0, nb, stream)) != cudaSuccess) return e;
  return cudaSuccess;
}

// The call on `stream` has enqueued its last use of the scratch (caller holds st.mu).
cudaError_t scratch_release(DeviceInfo& d, cudaStream_t stream) {
  ScratchState& st = d.scratch;
  const cudaError_t e = cudaEventRecord(st.done, stream);
  if (e == cudaSuccess) {
    st.last = stream;
    st.used = true;
  }
  return e;
}

// Residency answers (occupancy queries) are properties of the device and the
// kernel's shape, so each is asked of the runtime once and kept: a query costs
// microseconds of host time, more than a short call's kernel.
std::mutex g_occ_mutex;
std::unordered_map<uint64_t, int> g_occ_cache;

template <typename F>
int cached_query(uint64_t key, F&& query) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return query();
  key = key * 64 + (uint64_t)(dev & 63);
  {
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    const auto it = g_occ_cache.find(key);
    if (it != g_occ_cache.end()) return it->second;
  }
  const int v = query();
  if (v > 0) {  // failures are not kept
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    g_occ_cache[key] = v;
  }
  return v;
}

// key fields: kind (4 bits), input type (2), then the query's own numbers
uint64_t occ_key(int kind, int in_dtype, uint64_t a, uint64_t b = 0, uint64_t c = 0, uint64_t d = 0) {
  return ((((((uint64_t)kind * 4 + (uint64_t)in_dtype) * 65536 + a) * 65536 + b) * 64 + c) * 16) + d;
}

int cluster_capacity(int in_dtype, int cluster, int64_t smem_bytes) {
  return cached_query(occ_key(1, in_dtype, (uint64_t)cluster, (uint64_t)(smem_bytes / 16)), [&] {
    switch (in_dtype) {
      case SMX_F32: return cluster_capacity_f32(cluster, smem_bytes);
      case SMX_F16: return cluster_capacity_f16(cluster, smem_bytes);
      default: return cluster_capacity_bf16(cluster, smem_bytes);
    }
  });
}

int64_t cluster_smem_cap_bytes(const DeviceInfo& d) {
  int64_t cap = d.smem_optin - CLUSTER_STATIC_SMEM;
  const int64_t dbg = g_smem_cap.load();
  if (dbg > 0 && dbg < cap) cap = dbg;
  return cap / 16 * 16;
}

// Largest cluster size (power of two up to 16) that can be resident with the
// full staging area; cached per device and input type.
int max_cluster_size(DeviceInfo& d, int in_dtype) {
  if (d.max_cluster[in_dtype] == 0) {
    std::lock_guard<std::mutex> lock(g_mutex);
    const int64_t smem = d.smem_optin - CLUSTER_STATIC_SMEM;
    int best = 1;
    for (int c = 16; c >= 2; c >>= 1) {
      if (cluster_capacity(in_dtype, c, smem / 16 * 16) > 0) {
        best = c;
        break;
      }
    }
    d.max_cluster[in_dtype] = best;
  }
  int c = d.max_cluster[in_dtype];
  const int dbg = g_max_cluster.load();
  if (dbg > 0 && dbg < c) c = dbg;
  return c;
}

// read_heavy: the statistics / LSE and cross-entropy rows, whose per-row
// reductions dominate; the others write a row per row read.
bool plan_regs(int64_t cols, int in_dtype, bool accurate_exp, Plan* p, bool read_heavy = false) {
  const int V = 16 / elem_size(in_dtype);
  const int64_t nvec = cols / V;
  // the compensated exponential (fp32 outputs) keeps more live registers per
  // element: at most 16 elements per thread there, 32 otherwise
  const int max_vpt = (accurate_exp ? 16 : 32) / V;
  int vpt = 0;
  int64_t G = 0;
  const int dbg_t = g_regs_threads.load(), dbg_v = g_regs_vpt.load();
  if (dbg_t > 0 && dbg_v > 0 && dbg_v <= max_vpt && (dbg_t % 32) == 0 && dbg_t <= 1024 &&
      (int64_t)dbg_t * dbg_v >= nvec) {
    vpt = dbg_v;
    G = dbg_t;
  } else {
    // measured on GB300 (CTA shapes per mode over bf16/f16/f32 rows of 1K-8K
    // elements): rows that write an output are fastest with two vectors per
    // thread and 64..512 threads, then four, one, eight vectors; the
    // read-heavy rows with four vectors per thread and 64..256 threads (fewer
    // threads per row: cheaper reductions), then two, eight, one
    const int order_w[4] = {2, 4, 1, 8}, order_r[4] = {4, 2, 8, 1};
    const int* order = read_heavy ? order_r : order_w;
    const int64_t g_hi = read_heavy ? 256 : 512;
    for (int pass = 0; pass < 2 && vpt == 0; ++pass) {
      for (int k = 0; k < 4; ++k) {
        const int v = order[k];
        if (v > max_vpt) continue;
        const int64_t g = ((nvec + v - 1) / v + 31) / 32 * 32;
        if (pass == 0 ? (g >= 64 && g <= g_hi) : g <= 1024) {
          vpt = v;
          G = g;
          break;
        }
      }
    }
    if (vpt == 0) return false;
  }
  p->path = PATH_REGS;
  p->vpt = vpt;
  p->warp_rows = (G == 32);
  p->threads = p->warp_rows ? 256 : (int)G;
  return true;
}

int stream_occupancy(int in_dtype, int vpt, int threads, int depth, int mode, bool warp) {
  return cached_query(occ_key(2, in_dtype, (uint64_t)vpt, (uint64_t)threads, (uint64_t)depth * 8 + mode,
                              warp ? 1 : 0),
                      [&] {
                        switch (in_dtype) {
                          case SMX_F32: return stream_occupancy_f32(vpt, threads, depth, mode, warp);
                          case SMX_F16: return stream_occupancy_f16(vpt, threads, depth, mode, warp);
                          default: return stream_occupancy_bf16(vpt, threads, depth, mode, warp);
                        }
                      });
}

// Streamed path for rows of at most 32 KiB: the CTA shape of the register path
// (threads per row, vectors per thread; at least two warps), two rows
// prefetched per CTA, and enough persistent CTAs per SM to keep about 48 KiB of
// row reads in flight on every SM (measured on GB300: fewer CTAs starve HBM,
// more only contend; with lengths given, rows are taken as half valid).
constexpr int64_t STREAM_INFLIGHT_BYTES = 48 * 1024;
constexpr int64_t CE_INFLIGHT_BYTES = 64 * 1024;
constexpr int64_t CLUSTER_MAX_ROW_BYTES = 4 << 20;
constexpr int64_t ATTN_MAX_POLLS = int64_t(1) << 24;  // each tensor-core wait: tens of ms at most

bool plan_stream(DeviceInfo& d, int64_t rows, int64_t cols, int in_dtype, bool accurate_exp,
                 bool has_lengths, int mode, int64_t inflight, Plan* p, bool apply_out16 = false) {
  const bool apply = mode == MODE_APPLY;
  const int es = elem_size(in_dtype);
  if (cols * es > STREAM_MAX_ROW_BYTES) return false;
  const int V = 16 / es;
  const int64_t nvec = cols / V;
  const int max_vpt = (accurate_exp ? 16 : 32) / V;
  Plan r;
  // a row that fits one warp is walked by one warp (no block barrier), unless
  // a CTA shape is forced or the warp walkers are switched off
  // (the apply rows too when their outputs are 16-bit: no compensated
  // exponential, so a lane holds up to 32 elements, as the softmax's do)
  bool warp = false;
  const int warp_vpt = (apply && apply_out16) ? 32 / V : max_vpt;
  if ((!apply || apply_out16) && g_stream_warp.load() == 0 && g_regs_threads.load() == 0 &&
      nvec <= 32LL * warp_vpt) {
    r.vpt = 1;
    while (32LL * r.vpt < nvec) r.vpt <<= 1;
    r.threads = WARP_WALKER_THREADS;
    warp = true;
  } else if (!plan_regs(cols, in_dtype, accurate_exp, &r, mode == MODE_STATS || mode == MODE_CE) ||
             r.warp_rows) {
    r.threads = 64;
    r.vpt = 1;
    while (64LL * r.vpt < nvec) r.vpt <<= 1;
    if (r.vpt * V > (accurate_exp ? 16 : 32)) return false;
  }
  const int dd = g_stream_depth.load();
  // the apply kernel prefetches 2 items; the other walkers 2 unless set
  const int depth = (!apply && (dd == 3 || dd == 4)) ? dd : 2;
  const int occ_max = stream_occupancy(in_dtype, r.vpt, r.threads, depth, mode, warp);
  if (occ_max <= 0) return false;
  int occ = occ_max;
  int64_t row_read = cols * es;
  if (has_lengths) row_read = (row_read + 1) / 2;
  const int64_t walkers = warp ? r.threads / 32 : 1;
  int64_t want = inflight / ((int64_t)depth * walkers * (row_read > 0 ? row_read : 1));
  if (want < 1) want = 1;
  if (want < occ) occ = (int)want;
  const int forced = g_stream_ctas_per_sm.load();
  if (forced > 0) occ = forced < occ_max ? forced : occ_max;
  const int64_t ctas = (int64_t)occ * d.sm_count;
  const int64_t need = (rows + walkers - 1) / walkers;
  p->path = PATH_STREAM;
  p->threads = r.threads;
  p->vpt = r.vpt;
  p->warp_rows = warp;
  p->stages = depth;
  p->ctas = (int)(need < ctas ? need : ctas);
  return true;
}

// Long rows: chunks of 16 elements per thread of 256-thread CTAs on the
// streamed kernel, the statistics of every chunk of a slab of rows, then the
// merge and the normalising pass over the same slab.
bool plan_split(DeviceInfo& d, int64_t cols, int in_dtype, Plan* p) {
  const int es = elem_size(in_dtype);
  const int V = 16 / es;
  const int vpt = 16 / V;  // 16 elements per thread: the compensated exponential fits
  const int threads = 256;
  const int64_t chunk = (int64_t)threads * vpt * V;
  const int64_t nchunks = (cols + chunk - 1) / chunk;
  if (nchunks > ((int64_t)1 << 30)) return false;
  // one slab of all rows by default: the normalising pass re-reads the input
  // from DRAM.  Measured on GB300 (64 rows of 4 MiB): slabs of up to half the
  // L2, which the second pass re-reads from L2, were slower (160 us against
  // 142 us) -- every slab costs a drain of both passes, more than the re-read
  // from DRAM saves
  int64_t slab_bytes = INT64_MAX;
  const int64_t dbg = g_split_slab_bytes.load();
  if (dbg > 0) slab_bytes = dbg;
  int64_t slab = slab_bytes / (cols * es);
  if (slab < 1) slab = 1;
  if (slab > ((int64_t)1 << 31) / nchunks) slab = ((int64_t)1 << 31) / nchunks;
  const int occ_max = cached_query(occ_key(3, in_dtype, (uint64_t)threads), [&] {
    switch (in_dtype) {
      case SMX_F32: return split_occupancy_f32(threads);
      case SMX_F16: return split_occupancy_f16(threads);
      default: return split_occupancy_bf16(threads);
    }
  });
  if (occ_max <= 0) return false;
  int occ = occ_max;
  const int forced = g_stream_ctas_per_sm.load();
  if (forced > 0) occ = forced < occ_max ? forced : occ_max;
  p->path = PATH_SPLIT;
  p->threads = threads;
  p->vpt = vpt;
  p->stages = 2;
  p->ctas = occ * d.sm_count;
  p->chunk = chunk;
  p->nchunks = (int)nchunks;
  p->slab_rows = slab;
  // one cooperative launch (every CTA resident; per-row completion counts
  // between the passes) when asked for and supported: measured on GB300 it
  // is not faster than two launches over one slab (153 us against 142 us)
  if (g_split_fused.load() != 0 && d.coop) {
    const int fo = cached_query(occ_key(4, in_dtype, (uint64_t)threads), [&] {
      switch (in_dtype) {
        case SMX_F32: return split_fused_occupancy_f32(threads);
        case SMX_F16: return split_fused_occupancy_f16(threads);
        default: return split_fused_occupancy_bf16(threads);
      }
    });
    if (fo > 0) {
      int fc = fo;
      if (forced > 0) fc = forced < fo ? forced : fo;
      p->fused_split = true;
      p->fused_ctas = fc * d.sm_count;
      p->stripe_probe = g_count_probe.load();
    }
  }
  const int hs = g_split_hint_stats.load(), ha = g_split_hint_apply.load();
  p->l2_hint_stats = hs >= 0 ? hs : 1;  // the statistics pass's reads stay for the re-read
  p->l2_hint_apply = ha >= 0 ? ha : 2;  // the normalising pass's reads are the last
  return true;
}

int stripe_occupancy(int in_dtype, int64_t smem) {
  return cached_query(occ_key(6, in_dtype, (uint64_t)(smem / 16)), [&] {
    switch (in_dtype) {
      case SMX_F32: return stripe_occupancy_f32(smem);
      case SMX_F16: return stripe_occupancy_f16(smem);
      default: return stripe_occupancy_bf16(smem);
    }
  });
}

// Long rows read once (kernel_stripe.cuh), for the softmax, log_softmax and
// the cross-entropy with a gradient: Q CTAs per row, each holding one column
// stripe of every row of its group in a ring of shared-memory slots.  The
// stripes are as short as the CTAs allow, so that the ring holds as many as
// possible (at least LAG + 2: LAG rows held between summary and
// normalisation, plus copies in flight); the preferred ring is 8 slots, then
// 6, then 4.  Not planned when a row needs more CTAs than the device holds or
// the device cannot launch cooperatively.
// `two`: the backward's slots hold two stripes (p and g), so fewer fit: down
// to four slots (two rows of lag) instead of STRIPE_MIN_SLOTS
bool plan_stripe(DeviceInfo& d, int64_t rows, int64_t cols, int in_dtype, Plan* p, bool two = false) {
  if (!d.coop) return false;
  const int es = elem_size(in_dtype);
  const int V = 16 / es;
  const int64_t nvec = cols / V;
  if (nvec <= 0) return false;
  int& st = d.stripe_smem_static[in_dtype];
  if (st < 0) {
    st = in_dtype == SMX_F32 ? stripe_static_smem_f32()
                             : (in_dtype == SMX_F16 ? stripe_static_smem_f16() : stripe_static_smem_bf16());
    if (st < 0) return false;
  }
  const int64_t ring_bytes = (d.smem_optin - st - 256) / 16 * 16;  // (256: the runtime's own reserve)
  const int64_t ring_vecs = ring_bytes / 16;
  const int64_t cap = d.sm_count < STRIPE_MAX_Q ? d.sm_count : STRIPE_MAX_Q;  // one CTA per SM
  // a compute thread holds at most STRIPE_MAX_VPT vectors of a stripe
  const int64_t vec_cap = (int64_t)STRIPE_MAX_VPT * STRIPE_COMPUTE_THREADS;
  const int per_slot = two ? 2 : 1;  // stripes a slot holds
  const int min_slots = two ? STRIPE_MIN_SLOTS_TWO : STRIPE_MIN_SLOTS;
  for (const int target : {8, STRIPE_MIN_SLOTS, STRIPE_MIN_SLOTS_TWO}) {
    if (target < min_slots) continue;
    int64_t slot_cap = ring_vecs / target / per_slot;  // vectors of one stripe
    if (slot_cap > vec_cap) slot_cap = vec_cap;
    if (slot_cap <= 0) continue;
    const int64_t q_min = (nvec + slot_cap - 1) / slot_cap;
    if (q_min > cap) continue;
    int64_t groups = d.sm_count / q_min;
    if (groups > rows) groups = rows;
    if (groups < 1) groups = 1;
    int64_t Q = d.sm_count / groups;
    if (Q > STRIPE_MAX_Q) Q = STRIPE_MAX_Q;
    if (Q > nvec) Q = nvec;
    const int64_t stripe_vecs = (nvec + Q - 1) / Q;
    const int64_t slot_vecs = stripe_vecs * per_slot;
    int64_t nslots = ring_vecs / slot_vecs;
    if (nslots > STRIPE_MAX_SLOTS) nslots = STRIPE_MAX_SLOTS;
    if (nslots < min_slots) continue;
    const int64_t smem = nslots * slot_vecs * 16;
    if (stripe_occupancy(in_dtype, smem) < 1) return false;
    p->path = PATH_STRIPE;
    p->vpt = stripe_vecs <= 2LL * STRIPE_COMPUTE_THREADS ? 2 : 4;
    p->stripe_q = (int)Q;
    p->stripe_groups = (int)groups;
    p->stripe_slots = (int)nslots;
    p->stripe_slot_vecs = (int)slot_vecs;
    p->ctas = (int)(Q * groups);
    p->stripe_probe = g_count_probe.load();
    const int lg = g_stripe_lag.load(), pc = g_stripe_piece.load();
    p->stripe_lag = lg > 0 && lg < nslots - 1 ? lg : (STRIPE_DEFAULT_LAG < nslots - 1 ? STRIPE_DEFAULT_LAG : (int)nslots - 2);
    p->stripe_piece = pc >= 0 ? pc : STRIPE_DEFAULT_PIECE;
    const int la = g_stripe_l2_ahead.load();
    // measured on GB300 (64 rows of 4 MiB fp32 / bf16, 512 rows of 256 KiB
    // bf16; lag 4 / 6; prefetch 0, 2, 4, 6 rows ahead): 2 rows ahead and lag 6
    // fastest on all three (fp32: 115 -> 103 us)
    p->stripe_l2_ahead = la >= 0 ? la : STRIPE_DEFAULT_L2_AHEAD;
    return true;
  }
  return false;
}

bool plan_cluster(DeviceInfo& d, int64_t rows, int64_t cols, int in_dtype, Plan* p) {
  const int es = elem_size(in_dtype);
  const int V = 16 / es;
  const int64_t smem_elems_cap = cluster_smem_cap_bytes(d) / es;
  const int64_t per_cta = smem_elems_cap + (int64_t)CLUSTER_THREADS * CLUSTER_RV * V;
  const int maxc = max_cluster_size(d, in_dtype);
  int c = 1;
  while (c < maxc && (int64_t)c * per_cta < cols) c <<= 1;
  int64_t chunk = (cols + c - 1) / c;
  chunk = (chunk + V - 1) / V * V;
  // in-chunk vector indices are 32-bit
  if (chunk / V > (int64_t)1 << 30) return false;
  const int64_t smem_elems = chunk < smem_elems_cap ? chunk : smem_elems_cap;
  const int64_t smem_bytes = smem_elems * es > 16 ? smem_elems * es : 16;
  const int resident = cluster_capacity(in_dtype, c, smem_bytes);
  if (resident <= 0) return false;
  p->path = PATH_CLUSTER;
  p->cluster = c;
  p->chunk = chunk;
  p->smem_elems = smem_elems;
  p->ctas = (int)(rows < resident ? rows : resident);  // persistent clusters
  p->resident_clusters = resident;
  p->stage_tma = g_cluster_stage.load() != 2;
  return true;
}

int backward_occupancy(int in_dtype, int vpt, int threads) {
  return cached_query(occ_key(5, in_dtype, (uint64_t)vpt, (uint64_t)threads), [&] {
    switch (in_dtype) {
      case SMX_F32: return backward_occupancy_f32(vpt, threads);
      case SMX_F16: return backward_occupancy_f16(vpt, threads);
      default: return backward_occupancy_bf16(vpt, threads);
    }
  });
}

// Softmax backward: rows of up to 16 KiB per CTA (at most 16 elements per
// thread: two inputs held), with enough persistent CTAs for about 48 KiB of
// reads in flight per SM; longer rows in chunks of 4096 elements (two passes,
// by default over one slab of all rows); the scalar kernel for unaligned shapes.
void plan_backward(DeviceInfo& d, const Call& c, bool vec_ok, Plan* p) {
  p->path = PATH_GENERIC;
  if (!vec_ok) return;
  const int force = g_force_path.load();
  if (force == PATH_GENERIC) return;
  const int es = elem_size(c.in_dtype);
  const int V = 16 / es;
  const int64_t row_bytes = c.cols * es;
  if (row_bytes <= BWD_MAX_ROW_BYTES && force != PATH_SPLIT) {
    const int64_t nvec = c.cols / V;
    int vpt = 1;
    while (vpt * V < 16 && (nvec + vpt - 1) / vpt > 256) vpt <<= 1;
    int64_t threads = ((nvec + vpt - 1) / vpt + 31) / 32 * 32;
    if (threads < 64) threads = 64;
    if (threads <= 1024) {
      const int occ_max = backward_occupancy(c.in_dtype, vpt, (int)threads);
      if (occ_max > 0) {
        int64_t read = 2 * row_bytes;
        if (c.valid_len != nullptr) read = (read + 1) / 2;
        const int64_t per_cta = 2 * (read > 0 ? read : 1);  // two items prefetched
        int64_t want = (g_bwd_inflight.load() + per_cta - 1) / per_cta;
        if (want < 1) want = 1;
        int occ = want < occ_max ? (int)want : occ_max;
        const int forced = g_stream_ctas_per_sm.load();
        if (forced > 0) occ = forced < occ_max ? forced : occ_max;
        const int64_t ctas = (int64_t)occ * d.sm_count;
        p->path = PATH_STREAM;
        p->threads = (int)threads;
        p->vpt = vpt;
        p->stages = 2;
        p->ctas = (int)(c.rows < ctas ? c.rows : ctas);
        return;
      }
    }
  }
  // long rows read once in column stripes (p and g of a row kept on chip
  // from its dot to dx) when the stripes fit the SMs' shared memory
  if (force != PATH_SPLIT && (force == 0 || force == PATH_STRIPE) &&
      plan_stripe(d, c.rows, c.cols, c.in_dtype, p, true))
    return;
  const int vpt = 16 / V;
  const int threads = 256;
  const int64_t chunk = (int64_t)threads * vpt * V;
  const int64_t nchunks = (c.cols + chunk - 1) / chunk;
  if (nchunks > ((int64_t)1 << 30)) return;
  const int occ_max = backward_occupancy(c.in_dtype, 0, threads);
  if (occ_max <= 0) return;
  int occ = occ_max;
  const int forced = g_stream_ctas_per_sm.load();
  if (forced > 0) occ = forced < occ_max ? forced : occ_max;
  // one slab of all rows by default, as for the softmax (measured on GB300,
  // 64 rows of 4 MiB: 215 us against 232 us with slabs of half the L2)
  int64_t slab_bytes = INT64_MAX;
  const int64_t dbg = g_split_slab_bytes.load();
  if (dbg > 0) slab_bytes = dbg;
  int64_t slab = slab_bytes / (2 * row_bytes);
  if (slab < 1) slab = 1;
  if (slab > ((int64_t)1 << 31) / nchunks) slab = ((int64_t)1 << 31) / nchunks;
  p->path = PATH_SPLIT;
  p->threads = threads;
  p->vpt = vpt;
  p->stages = 2;
  p->ctas = occ * d.sm_count;
  p->chunk = chunk;
  p->nchunks = (int)nchunks;
  p->slab_rows = slab;
}

smx_status launch_planned(Call& c, DeviceInfo& dev, Plan p);

smx_status run_backward(Call& c, DeviceInfo& dev) {
  const int es = elem_size(c.in_dtype);
  const bool vec_ok = (reinterpret_cast<uintptr_t>(c.x) % 16 == 0) &&
                      (reinterpret_cast<uintptr_t>(c.g) % 16 == 0) &&
                      (reinterpret_cast<uintptr_t>(c.y) % 16 == 0) && ((c.cols * es) % 16 == 0);
  Plan p;
  plan_backward(dev, c, vec_ok, &p);
  return launch_planned(c, dev, p);
}

// The kernel family and launch shape for a call (no launch).
Plan plan_call(const Call& c, DeviceInfo& dev) {
  const int es_in = elem_size(c.in_dtype);
  const bool vec_ok =
      (reinterpret_cast<uintptr_t>(c.x) % 16 == 0) &&
      (c.y == nullptr || reinterpret_cast<uintptr_t>(c.y) % 16 == 0) &&
      ((c.cols * es_in) % 16 == 0) && c.cols > 0;
  // softmax and (m, d) statistics run on every kernel; LSE, log_softmax and
  // the apply mode on the streamed, long-row and generic ones
  const bool classic = c.mode == MODE_SOFTMAX || (c.mode == MODE_STATS && c.d_out != nullptr);
  const bool stripe_mode = c.mode == MODE_SOFTMAX || c.mode == MODE_LOG || (c.mode == MODE_CE && c.y != nullptr);
  Plan p;
  const int force = g_force_path.load();
  bool planned = false;
  if (vec_ok) {
    if (force == PATH_CLUSTER && classic) {
      planned = plan_cluster(dev, c.rows, c.cols, c.in_dtype, &p);
    } else if (force == PATH_STRIPE && stripe_mode) {
      planned = plan_stripe(dev, c.rows, c.cols, c.in_dtype, &p);
    } else if (force == PATH_SPLIT) {
      planned = plan_split(dev, c.cols, c.in_dtype, &p);
    } else if (force != PATH_GENERIC) {
      // the compensated exponential (fp32 softmax outputs, and every apply
      // output) holds 16 elements per thread at most
      const bool acc = (c.mode == MODE_SOFTMAX && c.out_dtype == SMX_F32) ||
                       (c.mode == MODE_CE && c.y != nullptr && c.out_dtype == SMX_F32) ||
                       c.mode == MODE_APPLY;
      if (force != PATH_REGS || !classic) {
        // read-only rows (statistics, LSE) and the cross-entropy (longer per-row
        // epilogue) keep more rows in flight (measured on GB300)
        const int64_t inflight = c.mode == MODE_STATS ? g_read_only_inflight.load()
                                 : c.mode == MODE_CE  ? CE_INFLIGHT_BYTES
                                                      : STREAM_INFLIGHT_BYTES;
        planned = plan_stream(dev, c.rows, c.cols, c.in_dtype, acc, c.valid_len != nullptr, c.mode,
                              inflight, &p, c.mode == MODE_APPLY && c.out_dtype != SMX_F32);
      }
      if (!planned && classic) planned = plan_regs(c.cols, c.in_dtype, acc, &p);
      // rows longer than one CTA holds: read once in column stripes over all
      // SMs when the stripes fit the SMs' shared memory (softmax, log_softmax,
      // cross-entropy with a gradient); the statistics rows a row per
      // thread-block cluster when the rows fill every resident cluster and
      // are shorter than 4 MiB; else chunks (path 5), which spread every row
      // over all SMs
      if (!planned && stripe_mode) planned = plan_stripe(dev, c.rows, c.cols, c.in_dtype, &p);
      if (!planned && classic && c.cols * es_in < CLUSTER_MAX_ROW_BYTES) {
        planned = plan_cluster(dev, c.rows, c.cols, c.in_dtype, &p);
        if (planned && c.rows < p.resident_clusters) planned = false;
      }
      if (!planned) planned = plan_split(dev, c.cols, c.in_dtype, &p);
      if (!planned && classic) planned = plan_cluster(dev, c.rows, c.cols, c.in_dtype, &p);
    }
  }
  if (!planned) p.path = PATH_GENERIC;
  return p;
}

cudaError_t launch_typed_in(const Call& c, const Plan& p) {
  switch (c.in_dtype) {
    case SMX_F32: return launch_in_f32(c, p);
    case SMX_F16: return launch_in_f16(c, p);
    default: return launch_in_bf16(c, p);
  }
}

// Launch a planned call.  The long-row paths take their summaries (and the
// stripe kernel its counters) from the device's scratch, which grows only when
// a call needs more than any before: a steady loop of calls allocates nothing.
smx_status launch_planned(Call& c, DeviceInfo& dev, Plan p) {
  c.status = dev.status;
  const int64_t wl = g_wait_limit.load();
  c.max_polls = wl != 0 ? wl : DEFAULT_MAX_POLLS;
  const size_t need = plan_scratch_bytes(c, p);
  cudaError_t e = cudaSuccess;
  if (need == 0 || p.scratch != nullptr) {
    e = launch_typed_in(c, p);
  } else {
    ScratchState& st = dev.scratch;
    std::lock_guard<std::mutex> lock(st.mu);
    e = scratch_reserve(dev, st.work, need, c.stream, false);
    if (e == cudaSuccess && p.path == PATH_STRIPE && c.rows > st.count_cap) {
      // both counter arrays (this call's and the next's), zero
      e = scratch_reserve(dev, st.counts, (size_t)2 * c.rows * sizeof(unsigned), c.stream, true);
      if (e == cudaSuccess) {
        st.count_cap = (int64_t)(st.counts.bytes / (2 * sizeof(unsigned)));
        st.count_parity = 0;
      }
    }
    if (e == cudaSuccess) {
      p.scratch = reinterpret_cast<float*>(st.work.base);
      if (p.path == PATH_STRIPE) {
        unsigned* cb = reinterpret_cast<unsigned*>(st.counts.base);
        p.stripe_count = cb + (size_t)st.count_parity * st.count_cap;
        p.stripe_count_next = cb + (size_t)(1 - st.count_parity) * st.count_cap;
        p.stripe_count_next_n = st.count_cap;
      }
      e = launch_typed_in(c, p);
      // the next stripe call counts in the array this one zeroed
      if (e == cudaSuccess && p.path == PATH_STRIPE) st.count_parity ^= 1;
      const cudaError_t f = scratch_release(dev, c.stream);
      if (e == cudaSuccess) e = f;
    }
  }
  t_last_path = p.path;
  if (e != cudaSuccess) return cuda_fail(e, SMX_ERR_LAUNCH);
  return SMX_OK;
}

smx_status run(Call& c, DeviceInfo& dev) { return launch_planned(c, dev, plan_call(c, dev)); }


// ---------------------------------------------------------------------------
// smx_softmax_rows_fixed_scratch: the long-row path with its chunk summaries in
// a fixed device array instead of a per-call allocation.


struct FixedSetup {
  std::atomic<bool> ready{false};
  bool supported = false;
  int sm_count = 0;
  int64_t l2_bytes = 0;
  int64_t smem_optin = 0;
  float* scratch = nullptr;  // this device's copy of g_fixed_scratch
};
FixedSetup g_fixed[MAX_DEVICES];

// Current device's properties and scratch address; no allocation.
smx_status fixed_setup(FixedSetup** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, SMX_ERR_UNSUPPORTED);
  if (dev < 0 || dev >= MAX_DEVICES) return SMX_ERR_UNSUPPORTED;
  FixedSetup& f = g_fixed[dev];
  if (!f.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!f.ready.load(std::memory_order_relaxed)) {
      int major = 0, minor = 0, sms = 0, l2 = 0, optin = 0;
      if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return cuda_fail(e, SMX_ERR_DEVICE);
      f.supported = (major == 10 && minor == 3);
      f.sm_count = sms;
      f.l2_bytes = l2;
      f.smem_optin = optin;
      if (f.supported) {
        void* a = nullptr;
        if ((e = cudaGetSymbolAddress(&a, g_fixed_scratch)) != cudaSuccess)
          return cuda_fail(e, SMX_ERR_DEVICE);
        f.scratch = static_cast<float*>(a);
      }
      f.ready.store(true, std::memory_order_release);
    }
  }
  if (!f.supported) return SMX_ERR_UNSUPPORTED;
  *out = &f;
  return SMX_OK;
}

// Chunks per row of the long-row path (4096 elements each, any type).
int64_t fixed_chunks(int64_t cols) { return (cols + 4095) / 4096; }

}  // namespace

// Element-wise merge of two arrays of (m, d) summaries; may run in place.
__global__ void __launch_bounds__(256)
    k_merge_stats(const float* m_a, const float* d_a, const float* m_b, const float* d_b,
                  float* m_o, float* d_o, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const MD r = md_merge(MD{m_a[i], d_a[i]}, MD{m_b[i], d_b[i]});
    m_o[i] = r.m;
    d_o[i] = r.d;
  }
}


cudaError_t launch_merge(const float* m_a, const float* d_a, const float* m_b, const float* d_b,
                         float* m_o, float* d_o, int64_t n, cudaStream_t stream) {
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  note_launch();
  k_merge_stats<<<(unsigned)blocks, 256, 0, stream>>>(m_a, d_a, m_b, d_b, m_o, d_o, n);
  return cudaGetLastError();
}

}  // namespace smx

using namespace smx;

extern "C" {

smx_status smx_softmax_rows(const void* x, void* y, int64_t rows, int64_t cols,
                            const int32_t* valid_len, smx_dtype in_dtype, smx_dtype out_dtype,
                            smx_stream_t stream) {
  t_kernel_launches = 0;
  if (rows < 0 || cols < 0 || !valid_dtype(in_dtype) || !valid_dtype(out_dtype))
    return SMX_ERR_INVALID_ARG;
  if (rows > 0 && cols > INT64_MAX / 4 / rows) return SMX_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return SMX_OK;
  if (x == nullptr || y == nullptr) return SMX_ERR_INVALID_ARG;
  const int64_t nx = rows * cols * elem_size(in_dtype), ny = rows * cols * elem_size(out_dtype);
  if (overlaps(x, nx, y, ny)) return SMX_ERR_ALIAS;
  if (valid_len && overlaps(valid_len, rows * 4, y, ny)) return SMX_ERR_ALIAS;
  DeviceInfo* dev = nullptr;
  smx_status s = device_info(&dev);
  if (s != SMX_OK) return s;
  Call c{x, y, nullptr, nullptr, rows, cols, valid_len, (int)in_dtype, (int)out_dtype,
         MODE_SOFTMAX, reinterpret_cast<cudaStream_t>(stream), nullptr, 0};
  return run(c, *dev);
}

// The host-buffer call stages rows through device slots of about this much
// input each (enough rows per launch; several chunks to overlap).
constexpr int64_t HOST_CHUNK_BYTES = int64_t(16) << 20;
constexpr int HOST_SLOTS = 2, HOST_MAX_SLOTS = 4;

// The device's address of a page-locked host buffer mapped into its address
// space (cudaHostAlloc / cudaHostRegister memory), else null.
const void* mapped_host(const void* h) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

smx_status smx_softmax_rows_host(const void* x, void* y, int64_t rows, int64_t cols,
                                 const int32_t* valid_len, smx_dtype in_dtype, smx_dtype out_dtype,
                                 smx_stream_t stream) {
  t_kernel_launches = 0;
  if (rows < 0 || cols < 0 || !valid_dtype(in_dtype) || !valid_dtype(out_dtype))
    return SMX_ERR_INVALID_ARG;
  if (rows > 0 && cols > INT64_MAX / 4 / rows) return SMX_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return SMX_OK;
  if (x == nullptr || y == nullptr) return SMX_ERR_INVALID_ARG;
  const int64_t ies = elem_size(in_dtype), oes = elem_size(out_dtype);
  const int64_t nx = rows * cols * ies, ny = rows * cols * oes;
  if (overlaps(x, nx, y, ny)) return SMX_ERR_ALIAS;
  if (valid_len && overlaps(valid_len, rows * 4, y, ny)) return SMX_ERR_ALIAS;
  DeviceInfo* dev = nullptr;
  smx_status s = device_info(&dev);
  if (s != SMX_OK) return s;
  cudaError_t e;
  cudaStream_t B = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (dev->copy_stream == nullptr) {
      if ((e = cudaStreamCreateWithFlags(&dev->copy_stream, cudaStreamNonBlocking)) != cudaSuccess) {
        dev->copy_stream = nullptr;
        return cuda_fail(e, SMX_ERR_DEVICE);
      }
      ++g_alloc_calls;
    }
    B = dev->copy_stream;
  }
  const cudaStream_t A = reinterpret_cast<cudaStream_t>(stream);
  if (g_host_staged.load() == 0) {
    // Page-locked buffers mapped into the device's address space are read
    // and written in place, over the host link, by the kernels that read
    // each input element once with plain or per-thread asynchronous loads
    // (the streamed and register-resident rows).  The long-row kernels read
    // the input twice, so those rows take the staging slots below; so do
    // the cluster kernel's rows (bulk copies).  Measured on GB300 (bf16
    // 16384 x 4096 / f16 32768 x 1024 with lengths / f32 64 x 1M): 305 / 335 /
    // 181 GB/s in place against 261 / 232 / 246 GB/s staged.
    const void* mx = mapped_host(x);
    void* my = const_cast<void*>(mapped_host(y));
    const int32_t* mvl = valid_len ? static_cast<const int32_t*>(mapped_host(valid_len)) : nullptr;
    if (mx && my && (!valid_len || mvl)) {
      Call c{mx, my, nullptr, nullptr, rows, cols, mvl, (int)in_dtype, (int)out_dtype, MODE_SOFTMAX, A, nullptr, 0};
      const Plan p = plan_call(c, *dev);
      if (p.path == PATH_STREAM || p.path == PATH_REGS) return launch_planned(c, *dev, p);
    }
  }
  const int64_t chunk_bytes = g_host_chunk.load() > 0 ? g_host_chunk.load() : HOST_CHUNK_BYTES;
  const int gs = g_host_slots.load();
  const int nslots = gs >= 2 && gs <= HOST_MAX_SLOTS ? gs : HOST_SLOTS;
  int64_t cr = chunk_bytes / (cols * ies);  // rows a chunk
  if (cr < 1) cr = 1;
  if (cr > rows) cr = rows;
  auto up16 = [](int64_t b) { return (b + 15) / 16 * 16; };
  const int64_t in_b = up16(cr * cols * ies), out_b = up16(cr * cols * oes);
  const int64_t slot = in_b + out_b + (valid_len ? up16(cr * 4) : 0);
  // The staging slots and the events live in the device's scratch (grown only
  // when a call needs more; events created once); the whole call holds it.
  ScratchState& sst = dev->scratch;
  std::lock_guard<std::mutex> lock(sst.mu);
  if ((e = scratch_reserve(*dev, sst.staging, (size_t)(nslots * slot), A, false)) != cudaSuccess)
    return cuda_fail(e, SMX_ERR_DEVICE);
  for (int i = 0; i < HOST_MAX_SLOTS && e == cudaSuccess; ++i) {
    if (sst.computed[i] == nullptr && (e = cudaEventCreateWithFlags(&sst.computed[i], cudaEventDisableTiming)) == cudaSuccess)
      ++g_alloc_calls;
    if (e == cudaSuccess && sst.copied[i] == nullptr &&
        (e = cudaEventCreateWithFlags(&sst.copied[i], cudaEventDisableTiming)) == cudaSuccess)
      ++g_alloc_calls;
  }
  if (e == cudaSuccess && sst.host_done == nullptr &&
      (e = cudaEventCreateWithFlags(&sst.host_done, cudaEventDisableTiming)) == cudaSuccess)
    ++g_alloc_calls;
  if (e != cudaSuccess) return cuda_fail(e, SMX_ERR_DEVICE);
  char* base = sst.staging.base;
  // per slot: its chunk computed (on A), its output copied back (on B)
  cudaEvent_t* computed = sst.computed;
  cudaEvent_t* copied = sst.copied;
  int launches = 0;
  for (int64_t i = 0, r0 = 0; e == cudaSuccess && r0 < rows; ++i, r0 += cr) {
    const int sl = (int)(i % nslots);
    const int64_t n = rows - r0 < cr ? rows - r0 : cr;
    char* dx = base + sl * slot;
    char* dy = dx + in_b;
    int32_t* dvl = valid_len ? reinterpret_cast<int32_t*>(dy + out_b) : nullptr;
    // in on A (the slot's previous chunk was computed earlier on A)
    if ((e = cudaMemcpyAsync(dx, static_cast<const char*>(x) + r0 * cols * ies, (size_t)(n * cols * ies),
                             cudaMemcpyHostToDevice, A)) != cudaSuccess)
      break;
    if (dvl && (e = cudaMemcpyAsync(dvl, valid_len + r0, (size_t)(n * 4), cudaMemcpyHostToDevice, A)) !=
                   cudaSuccess)
      break;
    // the slot's output buffer is free once its previous chunk's copy back is done
    if (i >= nslots && (e = cudaStreamWaitEvent(A, copied[sl], 0)) != cudaSuccess) break;
    Call c{dx, dy, nullptr, nullptr, n, cols, dvl, (int)in_dtype, (int)out_dtype, MODE_SOFTMAX, A, nullptr, 0};
    Plan p = plan_call(c, *dev);
    if (plan_scratch_bytes(c, p) > 0) {
      // the long-row kernels' summaries: the work buffer of the scratch held here
      if ((e = scratch_reserve(*dev, sst.work, plan_scratch_bytes(c, p), A, false)) != cudaSuccess) break;
      p.scratch = reinterpret_cast<float*>(sst.work.base);
      if (p.path == PATH_STRIPE) {
        if (c.rows > sst.count_cap) {
          if ((e = scratch_reserve(*dev, sst.counts, (size_t)2 * c.rows * sizeof(unsigned), A, true)) != cudaSuccess)
            break;
          sst.count_cap = (int64_t)(sst.counts.bytes / (2 * sizeof(unsigned)));
          sst.count_parity = 0;
        }
        unsigned* cb = reinterpret_cast<unsigned*>(sst.counts.base);
        p.stripe_count = cb + (size_t)sst.count_parity * sst.count_cap;
        p.stripe_count_next = cb + (size_t)(1 - sst.count_parity) * sst.count_cap;
        p.stripe_count_next_n = sst.count_cap;
      }
    }
    t_kernel_launches = 0;
    s = launch_planned(c, *dev, p);
    launches += t_kernel_launches;
    if (s != SMX_OK) break;
    if (p.path == PATH_STRIPE) sst.count_parity ^= 1;
    // out on B, after the chunk's softmax
    if ((e = cudaEventRecord(computed[sl], A)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(B, computed[sl], 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(static_cast<char*>(y) + r0 * cols * oes, dy, (size_t)(n * cols * oes),
                             cudaMemcpyDeviceToHost, B)) != cudaSuccess ||
        (e = cudaEventRecord(copied[sl], B)) != cudaSuccess)
      break;
  }
  // the call completes on the caller's stream: A waits for B's last copy; the
  // scratch's next user is ordered after that point of A
  cudaError_t f = cudaEventRecord(sst.host_done, B);
  if (f == cudaSuccess) f = cudaStreamWaitEvent(A, sst.host_done, 0);
  const cudaError_t g = scratch_release(*dev, A);
  t_kernel_launches = launches;
  if (s != SMX_OK) return s;
  if (e == cudaSuccess) e = f;
  if (e == cudaSuccess) e = g;
  if (e != cudaSuccess) return cuda_fail(e, SMX_ERR_DEVICE);
  return SMX_OK;
}

smx_status smx_softmax_rows_fixed_scratch(const void* x, void* y, int64_t rows, int64_t cols,
                                          const int32_t* valid_len, smx_dtype in_dtype,
                                          smx_dtype out_dtype, smx_stream_t stream) {
  t_kernel_launches = 0;
  if (rows < 0 || cols < 0 || !valid_dtype(in_dtype) || !valid_dtype(out_dtype))
    return SMX_ERR_INVALID_ARG;
  if (rows > 0 && cols > INT64_MAX / 4 / rows) return SMX_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return SMX_OK;
  if (x == nullptr || y == nullptr) return SMX_ERR_INVALID_ARG;
  const int64_t nx = rows * cols * elem_size(in_dtype), ny = rows * cols * elem_size(out_dtype);
  if (overlaps(x, nx, y, ny)) return SMX_ERR_ALIAS;
  if (valid_len && overlaps(valid_len, rows * 4, y, ny)) return SMX_ERR_ALIAS;
  const bool vec_ok = (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                      (reinterpret_cast<uintptr_t>(y) % 16 == 0) &&
                      ((cols * elem_size(in_dtype)) % 16 == 0);
  // one row's chunk summaries must fit (a slab holds at least one row)
  if (vec_ok && 2 * fixed_chunks(cols) > FIXED_SCRATCH_FLOATS) return SMX_ERR_TOO_LARGE;
  FixedSetup* f = nullptr;
  smx_status s = fixed_setup(&f);
  if (s != SMX_OK) return s;
  Call c{x, y, nullptr, nullptr, rows, cols, valid_len, (int)in_dtype, (int)out_dtype,
         MODE_SOFTMAX, reinterpret_cast<cudaStream_t>(stream), nullptr, 0};
  // The streamed and register-resident kernels need no scratch: rows they
  // take run exactly as smx_softmax_rows runs them.  Longer rows take the
  // chunked long-row kernels (never the cooperative ones, nor the cluster
  // kernel, whose bounded waits report through the library's status word)
  // with their summaries in the fixed array, in slabs cut to fit it.  No
  // kernel launched here writes the status word, so c.status stays null.
  Plan p;
  if (vec_ok) {
    DeviceInfo d;
    d.sm_count = f->sm_count;
    d.l2_bytes = f->l2_bytes;
    d.smem_optin = f->smem_optin;
    d.coop = false;
    const bool acc = out_dtype == SMX_F32;
    bool planned = plan_stream(d, rows, cols, in_dtype, acc, valid_len != nullptr, MODE_SOFTMAX,
                               STREAM_INFLIGHT_BYTES, &p);
    if (!planned) planned = plan_regs(cols, in_dtype, acc, &p);
    if (!planned) {
      if (!plan_split(d, cols, in_dtype, &p)) return SMX_ERR_UNSUPPORTED;
      const int64_t cap = FIXED_SCRATCH_FLOATS / (2 * (int64_t)p.nchunks);
      if (p.slab_rows > cap) p.slab_rows = cap;
      p.scratch = f->scratch;
      p.fixed_scratch = true;
    }
  } else {
    p.path = PATH_GENERIC;  // the scalar kernel takes no scratch
  }
  cudaError_t e;
  switch (c.in_dtype) {
    case SMX_F32: e = launch_in_f32(c, p); break;
    case SMX_F16: e = launch_in_f16(c, p); break;
    default: e = launch_in_bf16(c, p); break;
  }
  t_last_path = p.path;
  if (e != cudaSuccess) return cuda_fail(e, SMX_ERR_LAUNCH);
  return SMX_OK;
}

smx_status smx_softmax_row_stats(const void* x, float* m_out, float* d_out, int64_t rows,
                                 int64_t cols, const int32_t* valid_len, smx_dtype in_dtype,
                                 smx_stream_t stream) {
  t_kernel_launches = 0;
  if (rows < 0 || cols < 0 || !valid_dtype(in_dtype)) return SMX_ERR_INVALID_ARG;
  if (rows > 0 && cols > INT64_MAX / 4 / rows) return SMX_ERR_INVALID_ARG;
  if (rows == 0) return SMX_OK;
  if (m_out == nullptr || d_out == nullptr || (cols > 0 && x == nullptr)) return SMX_ERR_INVALID_ARG;
  const int64_t nx = rows * cols * elem_size(in_dtype);
  if (overlaps(x, nx, m_out, rows * 4) || overlaps(x, nx, d_out, rows * 4) ||
      overlaps(m_out, rows * 4, d_out, rows * 4))
    return SMX_ERR_ALIAS;
  if (valid_len && (overlaps(valid_len, rows * 4, m_out, rows * 4) ||
                    overlaps(valid_len, rows * 4, d_out, rows * 4)))
    return SMX_ERR_ALIAS;
  DeviceInfo* dev = nullptr;
  smx_status s = device_info(&dev);
  if (s != SMX_OK) return s;
  Call c{x, nullptr, m_out, d_out, rows, cols, valid_len, (int)in_dtype, SMX_F32, MODE_STATS,
         reinterpret_cast<cudaStream_t>(stream), nullptr, 0};
  return run(c, *dev);
}

smx_status smx_log_softmax_rows(const void* x, void* y, int64_t rows, int64_t cols,
                                const int32_t* valid_len, smx_dtype in_dtype, smx_dtype out_dtype,
                                smx_stream_t stream) {
  t_kernel_launches = 0;
  if (rows < 0 || cols < 0 || !valid_dtype(in_dtype) || !valid_dtype(out_dtype))
    return SMX_ERR_INVALID_ARG;
  if (rows > 0 && cols > INT64_MAX / 4 / rows) return SMX_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return SMX_OK;
  if (x == nullptr || y == nullptr) return SMX_ERR_INVALID_ARG;
  const int64_t nx = rows * cols * elem_size(in_dtype), ny = rows * cols * elem_size(out_dtype);
  if (overlaps(x, nx, y, ny)) return SMX_ERR_ALIAS;
  if (valid_len && overlaps(valid_len, rows * 4, y, ny)) return SMX_ERR_ALIAS;
  DeviceInfo* dev = nullptr;
  smx_status s = device_info(&dev);
  if (s != SMX_OK) return s;
  Call c{x, y, nullptr, nullptr, rows, cols, valid_len, (int)in_dtype, (int)out_dtype,
         MODE_LOG, reinterpret_cast<cudaStream_t>(stream), nullptr, 0};
  return run(c, *dev);
}

smx_status smx_softmax_lse(const void* x, float* lse_out, int64_t rows, int64_t cols,
                           const int32_t* valid_len, smx_dtype in_dtype, smx_stream_t stream) {
  t_kernel_launches = 0;
  if (rows < 0 || cols < 0 || !valid_dtype(in_dtype)) return SMX_ERR_INVALID_ARG;
  if (rows > 0 && cols > INT64_MAX / 4 / rows) return SMX_ERR_INVALID_ARG;
  if (rows == 0) return SMX_OK;
  if (lse_out == nullptr || (cols > 0 && x == nullptr)) return SMX_ERR_INVALID_ARG;
  const int64_t nx = rows * cols * elem_size(in_dtype);
  if (overlaps(x, nx, lse_out, rows * 4)) return SMX_ERR_ALIAS;
  if (valid_len && overlaps(valid_len, rows * 4, lse_out, rows * 4)) return SMX_ERR_ALIAS;
  DeviceInfo* dev = nullptr;
  smx_status s = device_info(&dev);
  if (s != SMX_OK) return s;
  Call c{x, nullptr, lse_out, nullptr, rows, cols, valid_len, (int)in_dtype, SMX_F32, MODE_STATS,
         reinterpret_cast<cudaStream_t>(stream), nullptr, 0};
  return run(c, *dev);
}

smx_status smx_softmax_apply_stats(const void* x, const float* m_in, const float* d_in, void* y,
                                   int64_t rows, int64_t cols, const int32_t* valid_len,
                                   smx_dtype in_dtype, smx_dtype out_dtype, smx_stream_t stream) {
  t_kernel_launches = 0;
  if (rows < 0 || cols < 0 || !valid_dtype(in_dtype) || !valid_dtype(out_dtype))
    return SMX_ERR_INVALID_ARG;
  if (rows > 0 && cols > INT64_MAX / 4 / rows) return SMX_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return SMX_OK;
  if (x == nullptr || y == nullptr || m_in == nullptr || d_in == nullptr) return SMX_ERR_INVALID_ARG;
  const int64_t nx = rows * cols * elem_size(in_dtype), ny = rows * cols * elem_size(out_dtype);
  if (overlaps(x, nx, y, ny) || overlaps(m_in, rows * 4, y, ny) || overlaps(d_in, rows * 4, y, ny))
    return SMX_ERR_ALIAS;
  if (valid_len && overlaps(valid_len, rows * 4, y, ny)) return SMX_ERR_ALIAS;
  DeviceInfo* dev = nullptr;
  smx_status s = device_info(&dev);
  if (s != SMX_OK) return s;
  Call c{x, y, nullptr, nullptr, rows, cols, valid_len, (int)in_dtype, (int)out_dtype,
         MODE_APPLY, reinterpret_cast<cudaStream_t>(stream), nullptr, 0, m_in, d_in};
  return run(c, *dev);
}

smx_status smx_softmax_backward(const void* p, const void* g, void* dx, int64_t rows, int64_t cols,
                                const int32_t* valid_len, smx_dtype dtype, smx_dtype dx_dtype,
                                smx_stream_t stream) {
  t_kernel_launches = 0;
  if (rows < 0 || cols < 0 || !valid_dtype(dtype) || !valid_dtype(dx_dtype)) return SMX_ERR_INVALID_ARG;
  if (rows > 0 && cols > INT64_MAX / 4 / rows) return SMX_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return SMX_OK;
  if (p == nullptr || g == nullptr || dx == nullptr) return SMX_ERR_INVALID_ARG;
  const int64_t n = rows * cols * elem_size(dtype), nd = rows * cols * elem_size(dx_dtype);
  if (overlaps(p, n, dx, nd) || overlaps(g, n, dx, nd)) return SMX_ERR_ALIAS;
  if (valid_len && overlaps(valid_len, rows * 4, dx, nd)) return SMX_ERR_ALIAS;
  DeviceInfo* dev = nullptr;
  smx_status s = device_info(&dev);
  if (s != SMX_OK) return s;
  Call c{p, dx, nullptr, nullptr, rows, cols, valid_len, (int)dtype, (int)dx_dtype, CALL_BACKWARD,
         reinterpret_cast<cudaStream_t>(stream), nullptr, 0};
  c.g = g;
  return run_backward(c, *dev);
}

smx_status smx_cross_entropy(const void* x, const int64_t* target, float* loss, void* grad,
                             int64_t rows, int64_t cols, const int32_t* valid_len, smx_dtype in_dtype,
                             smx_dtype grad_dtype, smx_stream_t stream) {
  t_kernel_launches = 0;
  if (rows < 0 || cols < 0 || !valid_dtype(in_dtype) || !valid_dtype(grad_dtype))
    return SMX_ERR_INVALID_ARG;
  if (rows > 0 && cols > INT64_MAX / 4 / rows) return SMX_ERR_INVALID_ARG;
  if (rows == 0) return SMX_OK;
  if (loss == nullptr || target == nullptr || (cols > 0 && x == nullptr)) return SMX_ERR_INVALID_ARG;
  const int64_t nx = rows * cols * elem_size(in_dtype), ng = rows * cols * elem_size(grad_dtype);
  if (overlaps(loss, rows * 4, x, nx) || overlaps(loss, rows * 4, target, rows * 8) ||
      (valid_len && overlaps(loss, rows * 4, valid_len, rows * 4)))
    return SMX_ERR_ALIAS;
  if (grad != nullptr &&
      (overlaps(grad, ng, x, nx) || overlaps(grad, ng, target, rows * 8) ||
       overlaps(grad, ng, loss, rows * 4) || (valid_len && overlaps(grad, ng, valid_len, rows * 4))))
    return SMX_ERR_ALIAS;
  DeviceInfo* dev = nullptr;
  smx_status s = device_info(&dev);
  if (s != SMX_OK) return s;
  Call c{x, cols > 0 ? grad : nullptr, nullptr, nullptr, rows, cols, valid_len, (int)in_dtype,
         (int)grad_dtype, MODE_CE, reinterpret_cast<cudaStream_t>(stream), nullptr, 0};
  c.target = target;
  c.loss = loss;
  return run(c, *dev);
}

smx_status smx_attention_forward(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int64_t heads, int64_t seq_q, int64_t seq_k, int head_dim,
                                 double scale, int causal, smx_dtype dtype, smx_stream_t stream) {
  t_kernel_launches = 0;
  if (heads < 0 || seq_q < 0 || seq_k < 0 || (dtype != SMX_F16 && dtype != SMX_BF16) ||
      !(scale > 0.0) || !(scale < 1e30))
    return SMX_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return SMX_ERR_UNSUPPORTED;
  if (heads > 65535) return SMX_ERR_UNSUPPORTED;
  if (heads > 0 && (seq_q > INT64_MAX / 4 / heads / head_dim || seq_k > INT64_MAX / 4 / heads / head_dim))
    return SMX_ERR_INVALID_ARG;
  if (heads == 0 || seq_q == 0) return SMX_OK;
  if (q == nullptr || o == nullptr || (seq_k > 0 && (k == nullptr || v == nullptr)))
    return SMX_ERR_INVALID_ARG;
  const auto misaligned = [](const void* p) { return p != nullptr && reinterpret_cast<uintptr_t>(p) % 16 != 0; };
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(o)) return SMX_ERR_INVALID_ARG;
  const int64_t nq = heads * seq_q * head_dim * 2, nk = heads * seq_k * head_dim * 2;
  if (overlaps(o, nq, q, nq) || overlaps(o, nq, k, nk) || overlaps(o, nq, v, nk) ||
      (lse && (overlaps(lse, heads * seq_q * 4, o, nq) || overlaps(lse, heads * seq_q * 4, q, nq) ||
               overlaps(lse, heads * seq_q * 4, k, nk) || overlaps(lse, heads * seq_q * 4, v, nk))))
    return SMX_ERR_ALIAS;
  DeviceInfo* dev = nullptr;
  smx_status s = device_info(&dev);
  if (s != SMX_OK) return s;
  AttnCall c{q, k, v, o, lse, heads, seq_q, seq_k, head_dim, scale, causal ? 1 : 0, (int)dtype,
             reinterpret_cast<cudaStream_t>(stream)};
  c.status = dev->status;
  const int64_t wl = g_wait_limit.load();
  c.max_polls = wl > 0 ? wl : ATTN_MAX_POLLS;
  c.probe_polls = wl < 0 ? -wl : 0;
  // measured on the pages' 4096 x 4096 shape: the two-tile persistent kernel
  // balances causal work best (1276 against 1194 TFLOP/s); the one-tile
  // kernel is level or ahead without a mask (1423 against 1407)
  const int which = g_attention_kernel.load();
  c.kernel = which >= 0 ? which : (causal ? ATTN_TMA2 : ATTN_TILE);
  c.sm_count = dev->sm_count;
  const cudaError_t e = launch_attention(c);
  if (e != cudaSuccess) return cuda_fail(e, SMX_ERR_LAUNCH);
  return SMX_OK;
}

smx_status smx_softmax_merge_stats(const float* m_a, const float* d_a, const float* m_b,
                                   const float* d_b, float* m_out, float* d_out, int64_t n,
                                   smx_stream_t stream) {
  t_kernel_launches = 0;
  if (n < 0) return SMX_ERR_INVALID_ARG;
  if (n == 0) return SMX_OK;
  if (!m_a || !d_a || !m_b || !d_b || !m_out || !d_out) return SMX_ERR_INVALID_ARG;
  if (n > INT64_MAX / 4) return SMX_ERR_INVALID_ARG;
  const int64_t nb = n * 4;
  const void* ins[4] = {m_a, d_a, m_b, d_b};
  const void* outs[2] = {m_out, d_out};
  if (overlaps(m_out, nb, d_out, nb)) return SMX_ERR_ALIAS;
  for (const void* o : outs)
    for (const void* i : ins)
      if (o != i && overlaps(o, nb, i, nb)) return SMX_ERR_ALIAS;
  DeviceInfo* dev = nullptr;
  smx_status s = device_info(&dev);
  if (s != SMX_OK) return s;
  const cudaError_t e =
      launch_merge(m_a, d_a, m_b, d_b, m_out, d_out, n, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, SMX_ERR_LAUNCH);
  return SMX_OK;
}

smx_status smx_last_device_status(smx_stream_t stream) {
  t_kernel_launches = 0;
  DeviceInfo* dev = nullptr;
  smx_status s = device_info(&dev);
  if (s != SMX_OK) return s;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, SMX_ERR_DEVICE);
  int v = 0;
  if ((e = cudaMemcpy(&v, dev->status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, SMX_ERR_DEVICE);
  if (v != 0 && (e = cudaMemset(dev->status, 0, sizeof(int))) != cudaSuccess)
    return cuda_fail(e, SMX_ERR_DEVICE);
  if (e != cudaSuccess) return cuda_fail(e, SMX_ERR_DEVICE);
  return v == 0 ? SMX_OK : (smx_status)(v & DEV_TIMEOUT ? SMX_ERR_TIMEOUT : SMX_ERR_DEVICE);
}

const char* smx_status_string(smx_status status) {
  switch (status) {
    case SMX_OK: return "ok";
    case SMX_ERR_INVALID_ARG: return "invalid argument";
    case SMX_ERR_UNSUPPORTED: return "no sm_103 CUDA device";
    case SMX_ERR_ALIAS: return "input and output overlap";
    case SMX_ERR_LAUNCH: return "kernel launch failed";
    case SMX_ERR_TIMEOUT: return "device: bounded wait for staged data ran out";
    case SMX_ERR_DEVICE: return "CUDA runtime call failed";
    case SMX_ERR_TOO_LARGE: return "row too long for the fixed scratch";
    default: return "unknown status";
  }
}

int smx_last_cuda_error(void) { return t_last_cuda_error; }

int smx_version(void) { return 100; }

void smx_debug_force_path(int path) { g_force_path.store(path >= 0 && path <= 6 ? path : 0); }

int64_t smx_debug_alloc_count(void) { return g_alloc_calls.load(); }

void smx_debug_set_count_probe(int64_t polls) { g_count_probe.store(polls > 0 ? polls : 0); }

void smx_debug_set_stripe_tuning(int lag, int piece_bytes, int l2_ahead) {
  g_stripe_lag.store(lag >= 1 && lag <= STRIPE_LAG ? lag : 0);
  g_stripe_piece.store(piece_bytes >= 0 && piece_bytes % 16 == 0 ? piece_bytes : -1);
  g_stripe_l2_ahead.store(l2_ahead >= 0 && l2_ahead <= 64 ? l2_ahead : -1);
}

void smx_debug_set_cluster(int max_cluster, int64_t smem_bytes) {
  g_max_cluster.store(max_cluster > 0 ? max_cluster : 0);
  g_smem_cap.store(smem_bytes > 0 ? smem_bytes : 0);
}

void smx_debug_set_wait_limit(int64_t polls) { g_wait_limit.store(polls); }

int smx_debug_last_path(void) { return t_last_path; }

int smx_debug_last_launches(void) { return t_kernel_launches; }

void smx_debug_set_stream_depth(int depth) { g_stream_depth.store(depth > 0 ? depth : 0); }

void smx_debug_set_split_slab(int64_t bytes) { g_split_slab_bytes.store(bytes > 0 ? bytes : 0); }

void smx_debug_set_inflight(int64_t read_only_bytes, int64_t backward_bytes) {
  g_read_only_inflight.store(read_only_bytes > 0 ? read_only_bytes : 96 * 1024);
  g_bwd_inflight.store(backward_bytes > 0 ? backward_bytes : 48 * 1024);
}

void smx_debug_set_stream_warp(int off) { g_stream_warp.store(off ? 1 : 0); }

void smx_debug_set_split_fused(int on) { g_split_fused.store(on ? 1 : 0); }
void smx_debug_set_host_chunk(int64_t bytes, int slots, int staged) {
  g_host_chunk.store(bytes > 0 ? bytes : 0);
  g_host_slots.store(slots >= 2 && slots <= HOST_MAX_SLOTS ? slots : 0);
  g_host_staged.store(staged ? 1 : 0);
}

void smx_debug_set_attention_kernel(int which) {
  g_attention_kernel.store(which == ATTN_TILE || which == ATTN_TMA1 || which == ATTN_MMA_SYNC || which == ATTN_TMA2
                               ? which
                               : -1);
}

void smx_debug_set_split_hints(int stats, int apply) {
  g_split_hint_stats.store(stats >= 0 && stats <= 2 ? stats : -1);
  g_split_hint_apply.store(apply >= 0 && apply <= 2 ? apply : -1);
}

void smx_debug_set_cluster_staging(int mode) { g_cluster_stage.store(mode == 1 || mode == 2 ? mode : 0); }

void smx_debug_set_stream_ctas(int per_sm) { g_stream_ctas_per_sm.store(per_sm > 0 ? per_sm : 0); }

void smx_debug_set_regs_shape(int threads, int vpt) {
  g_regs_threads.store(threads > 0 ? threads : 0);
  g_regs_vpt.store(vpt > 0 ? vpt : 0);
}

}  // extern "C"
