// Attention forward with warp-specialised operand fetching: the running
// state (m, l, o) of "Online stable softmax" ("Carry a weighted value
// numerator for attention") and "Softmax numerics architecture..." ("From
// online softmax to tiled attention") on the 5th-generation tensor cores.
//
// Persistent CTAs walk work items (a head's block of TILES x 128 query rows;
// items of one head are consecutive, so concurrent items share K and V in
// L2; under causal masking each head's longest items come first).  Tile t of
// an item is 128 query rows (warps 4t .. 4t + 3, row thread r = TMEM lane r
// of the tile's accumulators); keys go in blocks of 64.  TILES = 1: two CTAs
// an SM; TILES = 2: one CTA an SM whose two tiles read the same K and V
// stages (a key block crosses from L2 to shared memory once per 256 query
// rows).  Tensor memory:
//   O_t            columns t D ..                          (fp32, D wide)
//   S_t, buffer i  columns TILES D + 128 t + 64 i ..        (fp32, 64 wide; P,
//                  packed two to a column, over its first 32)
// Warp roles: the row warps (the per-block softmax of tc_rows_block: mask,
// maximum, exponentials, sum, P into tensor memory, O rescaled when the
// reference maximum moves; then the item's output); one issuing warp per
// tile, whose lane 0 issues that tile's tcgen05.mma (one issuing thread was
// measured to leave the tensor core idle with two tiles' 64-key products:
// issuing a product waits for room in the tensor pipe); one warp that
// fetches the K stages and one that fetches Q and the V stages, each by
// tensor-map bulk copies (cp.async.bulk.tensor, 128-byte swizzle, no
// multicast) completing on full barriers.  The row warps issue no copies.
//
// Issue rounds.  For each item, tile t's issuing lane issues its products in
// rounds: round 0 is S_t(0), round 1 S_t(1), and round b + 2 (once the
// tile's rows finished block b: named barrier) is O_t += P_t(b) V(b)
// followed by S_t(b + 2) (n blocks make rounds 0 .. n + 1; an item without
// keys for the tile makes none).  Rounds are numbered across the CTA's items
// and each ends with one tcgen05.commit, on round barrier R_t[r % 16]; it
// completes when every product of the round (and before it) has finished.
// Everything else waits on those: the rows for their scores (round b), a
// rescale for the previous O += P V (round b + 1), the output for the last
// one (round n + 1), the K fetcher for a stage's previous scores, and the V
// fetcher for a stage's previous O += P V and for the item's last scores
// before it refills Q.  The round 16 later on the same barrier cannot finish
// before the waiter has moved on: it needs the waiter's own progress (rows
// it has not yet let through, or at least five stages it has not yet
// fetched: a round per block plus two per item never outruns the fetches
// three to one), so a phase parity names one round.  One commit a round:
// each commit is costly for the issuing thread, and a 64-key round is short.
// The next item's first scores are issued right after the current item's
// last round, so they overlap the rows' output; eight blocks before an item
// ends, the fetchers bring the next item's Q and first K and V stages into L2.  Rows past the end of the query or key range
// are zero in shared memory (the copies fill them) and masked.  Every
// mbarrier wait is bounded; running out records SMX_ERR_TIMEOUT.
#pragma once

#include <cuda.h>

#include "kernel_attention_tc.cuh"
#include "smx_async.cuh"

namespace smx {

constexpr int ATM_BM = 128;  // query rows per tile
constexpr int ATM_BN = 64;   // keys per block
constexpr int ATM_NBAR = 44;

template <int TILES>
struct AtmShape {
  static_assert(TILES == 1 || TILES == 2, "one or two query tiles a CTA");
  static constexpr int NK = TILES == 2 ? 4 : 3;  // K stages
  static constexpr int NV = TILES == 2 ? 4 : 2;  // V stages
  static constexpr int ROW_THREADS = TILES * ATM_BM;
  static constexpr int ISSUE_WARP = ROW_THREADS / 32;        // tile t: ISSUE_WARP + t
  static constexpr int KLOAD_WARP = ISSUE_WARP + TILES;
  static constexpr int VLOAD_WARP = KLOAD_WARP + 1;
  static constexpr int BLOCK = (VLOAD_WARP + 1) * 32;
  static constexpr int CTAS_PER_SM = TILES == 2 ? 1 : 2;
  static constexpr uint32_t TCOLS = TILES == 2 ? 512 : 256;
  // output staging (two tiles a CTA): 2 KB a row warp, 32 rows x 64 bytes,
  // through which the rows' output goes out in coalesced pieces
  static constexpr int STAGE_BYTES = TILES == 2 ? TILES * 4 * 2048 : 0;
  // shared memory: Q [TILES][128][D], K [NK][64][D], V [NV][64][D] (16-bit),
  // then the output staging
  template <int D>
  __host__ __device__ static constexpr int tile_bytes() {
    return (TILES * ATM_BM * D + (NK + NV) * ATM_BN * D) * 2 + STAGE_BYTES;
  }
  // the launch adds 1024 bytes so that the tiles start on a 1024-byte
  // boundary (the 128-byte swizzle's atom); the barriers and the TMEM
  // address (ATM_NBAR * 8 + 4 bytes, under half of it) sit in that slack
  template <int D>
  __host__ __device__ static constexpr int smem_bytes() {
    return tile_bytes<D>() + 1024;
  }
};

struct AttnTmaArgs {
  AttnArgs a;
  int64_t nq;     // work items of a head (query blocks of TILES x 128 rows)
  int64_t items;  // heads x nq
  int* status;
  int64_t max_polls;
  int64_t probe_polls;  // > 0: thread 0 first waits this many polls on a barrier nothing
                        // signals and records SMX_ERR_TIMEOUT (a probe of the error path)
};

// box (x = column, y = row, z = head) of a 3-D tensor map into shared memory,
// completing its bytes on the mbarrier
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
// the same box into L2 only
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// A stage fetcher's wait for a free stage: its copies run stages ahead of
// their use, so it polls at leisure (a sleep between polls keeps it off the
// issue slots the row warps need).  Bounded like tc_wait.
__device__ __forceinline__ bool atm_wait_lazy(uint32_t bar, uint32_t parity, int64_t max_polls, const int* status) {
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (int64_t it = 0; it < max_polls; ++it) {
    if (mbar_test_wait(bar, parity)) return true;
    __nanosleep(256);
    if ((it & 15) == 15) {
      if (*reinterpret_cast<const volatile int*>(status) & DEV_TIMEOUT) return false;
      uint64_t t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > 200000000ull) return false;
    }
  }
  return false;
}

#ifdef SMX_ATM_TRACE
// per key block, SM clock stamps of two CTAs (tuning builds only): [cta][event][block]
// events: 0/1 issuer past tile t's named barrier, 2/3 issuer done issuing for
// tile t, 4/5 tile t's rows past their score wait, 6/7 tile t's rows arrive,
// 8 K fetch issued, 9 V fetch issued; by item: 10 Q fetch issued, 11 tile 0's
// issuer past its Q wait, 12 tile 0's issuer done with round 0, 13 tile 0's
// rows done with the output
__device__ long long g_atm_trace[2][14][256];
#define ATM_STAMP(ev, blk)                                                                   \
  do {                                                                                      \
    if (trace_slot >= 0 && (blk) < 256) g_atm_trace[trace_slot][ev][blk] = clock64();        \
  } while (0)
#else
#define ATM_STAMP(ev, blk) \
  do {                     \
  } while (0)
#endif

// Work item w of a CTA: its head, first query row and the key blocks of
// each tile (0 for a tile wholly past the query rows or without valid keys).
template <int TILES>
struct AtmItem {
  int64_t head, q0;
  int n[2];
  int nmax;
  __device__ __forceinline__ AtmItem(int64_t w, const AttnArgs& a, int64_t nq) {
    head = w / nq;
    const int64_t qb = w - head * nq;
    q0 = (a.causal ? nq - 1 - qb : qb) * (TILES * ATM_BM);
    n[0] = n[1] = 0;
#pragma unroll
    for (int t = 0; t < TILES; ++t) {
      const int64_t r0 = q0 + t * ATM_BM;
      int64_t kv_end = a.sk;
      if (r0 >= a.sq) {
        kv_end = 0;
      } else if (a.causal) {
        const int64_t last = r0 + ATM_BM - 1 < a.sq - 1 ? r0 + ATM_BM - 1 : a.sq - 1;
        kv_end = last + a.sk - a.sq + 1;
        if (kv_end > a.sk) kv_end = a.sk;
        if (kv_end < 0) kv_end = 0;
      }
      n[t] = (int)((kv_end + ATM_BN - 1) / ATM_BN);
    }
    nmax = n[0] > n[1] ? n[0] : n[1];
  }
  // tile t's key blocks (t not a compile-time constant: a select, not an
  // indexed load)
  __device__ __forceinline__ int nt(int t) const { return t ? n[1] : n[0]; }
};

// The CTA's k-th work item: rounds of gridDim.x items, dealt to the CTAs in
// alternating directions (under causal masking an item's work falls along a
// head's items, and alternate directions even it out between CTAs); -1 past
// the end.
__device__ __forceinline__ int64_t atm_item_of(int64_t k, int64_t items) {
  const int64_t g = gridDim.x, c = blockIdx.x;
  const int64_t w = k * g + ((k & 1) ? g - 1 - c : c);
  return w < items ? w : -1;
}

template <typename T, int D, int TILES>
__global__ void __launch_bounds__(AtmShape<TILES>::BLOCK, AtmShape<TILES>::CTAS_PER_SM)
    k_attention_tma(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, T* __restrict__ o, float* __restrict__ lse,
                    AttnTmaArgs args) {
  static_assert(D == 64 || D == 128, "head dimension");
  using S = AtmShape<TILES>;
  using Item = AtmItem<TILES>;
  constexpr int BM = ATM_BM, BN = ATM_BN, NK = S::NK, NV = S::NV;
  constexpr int QT = BM * D * 2;  // bytes of a Q tile
  constexpr int KT = BN * D * 2;  // bytes of a K or V stage
  // barrier indices: round barriers R_t[i] at B_R + 16 t + i, full barriers
  // of the K and V stages, Q, the probe's, the issuing lanes' drains
  constexpr int B_R = 0, B_KF = 32, B_VF = 36, B_Q = 40, B_PROBE = 41, B_DRAIN = 42;
  static_assert(NK <= 4 && NV <= 4 && B_DRAIN + 2 == ATM_NBAR, "barrier layout");
  auto rnd = [](int t, int r) { return B_R + 16 * t + (r & 15); };
  auto rpar = [](int r) { return (uint32_t)((r >> 4) & 1); };
  extern __shared__ __align__(16) uint8_t smem_raw[];

  const AttnArgs& a = args.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#ifdef SMX_ATM_TRACE
  const int trace_slot = blockIdx.x == 0 ? 0 : (blockIdx.x == 64 ? 1 : -1);
#endif

  const uint32_t raw = tc_su32(smem_raw);
  const uint32_t pad = (1024 - (raw & 1023)) & 1023;
  uint8_t* base = smem_raw + pad;
  const uint32_t sQ = tc_su32(base), sK = sQ + TILES * QT, sV = sK + NK * KT, sO = sV + NV * KT;
  // the barriers: in the alignment gap when it has room, else after the tiles
  constexpr uint32_t AUX = ATM_NBAR * 8 + 4;
  static_assert(2 * AUX < 1024, "barriers fit the alignment slack");
  uint8_t* aux = pad >= AUX ? smem_raw : base + S::template tile_bytes<D>();
  uint64_t* bars = reinterpret_cast<uint64_t*>(aux);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + ATM_NBAR);
  const uint32_t bar0 = tc_su32(bars);
  auto bar = [bar0](int i) { return bar0 + 8u * (uint32_t)i; };

  if (warp == S::ISSUE_WARP) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tc_su32(tmem_slot)),
                 "r"(S::TCOLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < ATM_NBAR; ++i) mbar_init(bar(i), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  // the error-path probe: a wait on a barrier nothing signals runs out
  if (args.probe_polls > 0 && tid == 0 && !tc_wait(bar(B_PROBE), 0u, args.probe_polls, args.status))
    atomicOr(args.status, DEV_TIMEOUT);
  auto t_o = [tmem](int t) { return tmem + (uint32_t)(t * D); };
  auto t_s = [tmem](int t, int i) { return tmem + (uint32_t)(TILES * D + 128 * t + 64 * i); };
  bool ok = true;
  auto wait_or_flag = [&](uint32_t b_, uint32_t par) {
    if (!tc_wait(b_, par, args.max_polls, args.status)) {
      ok = false;
      atomicOr(args.status, DEV_TIMEOUT);
    }
  };
  // counters every role keeps alike over the CTA's items: rounds and blocks
  // of each tile, K / V fetches, Q loads
  int R0[2] = {0, 0}, G[2] = {0, 0}, J = 0, QC = 0;
  auto sel = [](const int (&v)[2], int t) { return t ? v[1] : v[0]; };
  auto advance = [&](const Item& it) {
#pragma unroll
    for (int t = 0; t < TILES; ++t) {
      R0[t] += it.n[t] > 0 ? it.n[t] + 2 : 0;
      G[t] += it.n[t];
    }
    J += it.nmax;
    QC += it.nmax > 0 ? 1 : 0;
  };

  if (warp >= S::ISSUE_WARP && warp < S::ISSUE_WARP + TILES) {
    // the issuing warp of tile t
    const int t = warp - S::ISSUE_WARP;
    const uint32_t id_s = tc_idesc<T>(BM, BN), id_o = tc_idesc<T>(BM, D, true);
    const uint32_t qb = sQ + (uint32_t)(t * QT);
    // S_t = Q_t K^T for the block with (CTA-wide) index g of this tile and
    // fetch f: D / 16 steps of K = 16 (two per 32 bytes of a 128-byte row)
    auto issue_s = [&](int g, int f) {
      const uint32_t kb = sK + (uint32_t)((f % NK) * KT);
#pragma unroll
      for (int st = 0; st < D / 16; ++st) {
        const uint32_t koff = (uint32_t)((st & 3) * 32);
        const uint64_t da = tc_sdesc(qb + (uint32_t)((st >> 2) * BM * 128) + koff);
        const uint64_t db = tc_sdesc(kb + (uint32_t)((st >> 2) * BN * 128) + koff);
        tc_mma(t_s(t, g & 1), da, db, id_s, st > 0 ? 1u : 0u);
      }
    };
    // O_t += P_t V: BN / 16 steps of K = 16 keys, P from the score tile's
    // first columns (8 a step), V as the MN-major B operand (two 8-key
    // groups, 2048 bytes, a step); the item's first block overwrites O_t
    auto issue_pv = [&](int g, int f, bool first) {
      const uint32_t vb = sV + (uint32_t)((f % NV) * KT), pb = t_s(t, g & 1);
#pragma unroll
      for (int s2 = 0; s2 < BN / 16; ++s2) {
        const uint64_t db = tc_sdesc_mn(vb + (uint32_t)(s2 * 2048), (uint32_t)(BN * 128));
        tc_mma_ta(t_o(t), pb + (uint32_t)(s2 * 8), db, id_o, (!first || s2 > 0) ? 1u : 0u);
      }
    };
    for (int64_t k = 0, w; (w = atm_item_of(k, args.items)) >= 0; ++k) {
      const Item it(w, a, args.nq);
      const int n = it.nt(t), r0 = sel(R0, t), g0 = sel(G, t);
      if (n > 0) {
        // rounds 0 and 1 (a round with nothing to issue still commits, so
        // every round completes its barrier's phase)
        if (lane == 0) {
          wait_or_flag(bar(B_Q), (uint32_t)(QC & 1));
          if (t == 0) ATM_STAMP(11, (int)k);
          for (int r = 0; r < 2; ++r) {
            if (r < n) {
              wait_or_flag(bar(B_KF + (J + r) % NK), (uint32_t)(((J + r) / NK) & 1));
              issue_s(g0 + r, J + r);
            }
            tc_commit(bar(rnd(t, r0 + r)));
            if (t == 0 && r == 0) ATM_STAMP(12, (int)k);
          }
        }
        __syncwarp();
        for (int b = 0; b < n; ++b) {
          // the tile's rows finished block b (P_t in tensor memory, O_t
          // rescaled): named barrier 1 + 2 t + (g & 1); the rows are at most
          // one block ahead of this warp, so two barriers never mix generations
          const int g = g0 + b;
          const int nbar = 1 + 2 * t + (g & 1);
          asm volatile("barrier.sync.aligned %0, %1;" ::"r"(nbar), "n"(ATM_BM + 32) : "memory");
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          if (lane == 0) {
            ATM_STAMP(t, g);
            // round b + 2
            wait_or_flag(bar(B_VF + (J + b) % NV), (uint32_t)(((J + b) / NV) & 1));
            issue_pv(g, J + b, b == 0);
            if (b + 2 < n) {
              wait_or_flag(bar(B_KF + (J + b + 2) % NK), (uint32_t)(((J + b + 2) / NK) & 1));
              issue_s(g + 2, J + b + 2);
            }
            tc_commit(bar(rnd(t, r0 + b + 2)));
            ATM_STAMP(2 + t, g);
          }
          __syncwarp();
        }
      }
      advance(it);
    }
    // every product this lane issued has finished before the tensor memory is
    // freed (the row threads' waits cover them on the normal path; after a
    // wait ran out they may not): one more commit, waited by wall time only
    if (lane == 0 && sel(R0, t) > 0) {
      tc_commit(bar(B_DRAIN + t));
      tc_wait_drain(bar(B_DRAIN + t), 0u);
    }
    __syncwarp();
  } else if (warp == S::KLOAD_WARP || warp == S::VLOAD_WARP) {
    // the stage fetchers: K, or Q and V.  A stage is refilled once every tile
    // that read its previous block is done with it: the round of that
    // block's scores (K) or of its O += P V (V), kept for the last NS fetches
    // (-1: no tile of the block had it).  Q waits for each tile's last scores
    // of the previous item, so its fetcher is the V one: the K stages of the
    // next item fill while the current item's last blocks run.  Eight blocks
    // before an item's end, each fetcher brings the next item's first stages
    // (and Q) into L2.
    const bool is_k = warp == S::KLOAD_WARP;
    const CUtensorMap* map = is_k ? &tm_k : &tm_v;
    const uint32_t stages = is_k ? sK : sV;
    const int full0 = is_k ? B_KF : B_VF;
    constexpr int NS = NK > NV ? NK : NV;  // the longer ring; the shorter uses its tail
    const int ns = is_k ? NK : NV;
    int rec[2][NS];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int i = 0; i < NS; ++i) rec[t][i] = -1;
    int qwait[2] = {-1, -1};  // each tile's round of its last scores so far (the Q tile is free after it)
    if (lane == 0) {
      tma_prefetch_map(map);
      if (!is_k) tma_prefetch_map(&tm_q);
      for (int64_t k = 0, w; (w = atm_item_of(k, args.items)) >= 0; ++k) {
        const Item it(w, a, args.nq);
        const int64_t wn = atm_item_of(k + 1, args.items);
        if (it.nmax > 0) {
          if (!is_k) {
            // the Q tiles, once each tile's last scores have read them (rows
            // past the query range land as zeros); a tight wait: the next
            // item's first scores wait for this copy
#pragma unroll
            for (int t = 0; t < TILES; ++t)
              if (qwait[t] >= 0 && !tc_wait(bar(rnd(t, qwait[t])), rpar(qwait[t]), args.max_polls, args.status)) {
                ok = false;
                atomicOr(args.status, DEV_TIMEOUT);
              }
            ATM_STAMP(10, (int)k);
            mbar_arrive_expect_tx(bar(B_Q), (uint32_t)(TILES * QT));
#pragma unroll
            for (int t = 0; t < TILES; ++t)
#pragma unroll
              for (int h = 0; h < D / 64; ++h)
                tma_load_3d(sQ + (uint32_t)(t * QT + h * BM * 128), &tm_q, h * 64, (int)(it.q0 + t * BM),
                            (int)it.head, bar(B_Q));
#pragma unroll
            for (int t = 0; t < TILES; ++t)
              if (it.n[t] > 0) qwait[t] = R0[t] + it.n[t] - 1;
          }
          const int pre_at = it.nmax > 8 ? it.nmax - 8 : 0;
          for (int j = 0; j < it.nmax; ++j) {
            if (j == pre_at && wn >= 0) {
              const Item nx(wn, a, args.nq);
              for (int jj = 0; jj < ns && jj < nx.nmax; ++jj)
#pragma unroll
                for (int h = 0; h < D / 64; ++h) tma_prefetch_l2_3d(map, h * 64, jj * BN, (int)nx.head);
              if (!is_k)
#pragma unroll
                for (int t = 0; t < TILES; ++t)
#pragma unroll
                  for (int h = 0; h < D / 64; ++h)
                    tma_prefetch_l2_3d(&tm_q, h * 64, (int)(nx.q0 + t * BM), (int)nx.head);
            }
            const int f = J + j, s = f % ns;
            // the stage's previous block: recorded ns fetches ago
#pragma unroll
            for (int t = 0; t < TILES; ++t) {
              const int r = is_k ? rec[t][NS - NK] : rec[t][NS - NV];
              if (r >= 0 && !atm_wait_lazy(bar(rnd(t, r)), rpar(r), args.max_polls, args.status)) {
                ok = false;
                atomicOr(args.status, DEV_TIMEOUT);
              }
            }
#pragma unroll
            for (int t = 0; t < TILES; ++t) {
#pragma unroll
              for (int i = 0; i + 1 < NS; ++i) rec[t][i] = rec[t][i + 1];
              rec[t][NS - 1] = j < it.n[t] ? R0[t] + (is_k ? j : j + 2) : -1;
            }
            ATM_STAMP(is_k ? 8 : 9, f);
            mbar_arrive_expect_tx(bar(full0 + s), (uint32_t)KT);
#pragma unroll
            for (int h = 0; h < D / 64; ++h)
              tma_load_3d(stages + (uint32_t)(s * KT + h * BN * 128), map, h * 64, j * BN, (int)it.head,
                          bar(full0 + s));
          }
        }
        advance(it);
      }
      // every copy this lane issued has landed before the CTA ends (already
      // so on the normal path: the issuing lanes waited for each)
      for (int s = 0; s < ns && s < J; ++s) {
        const int fl = s + ((J - 1 - s) / ns) * ns;  // the last fetch into stage s
        tc_wait_drain(bar(full0 + s), (uint32_t)((fl / ns) & 1));
      }
      if (!is_k && QC > 0) tc_wait_drain(bar(B_Q), (uint32_t)((QC - 1) & 1));
    }
    __syncwarp();
  } else {
    // row threads: tile t, TMEM lane rt of the tile
    const int t = tid >> 7, rt = tid & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float cs = a.scale_log2;
    for (int64_t k = 0, w; (w = atm_item_of(k, args.items)) >= 0; ++k) {
      const Item it(w, a, args.nq);
      const int n = it.nt(t), r0 = sel(R0, t), g0 = sel(G, t);
      const int64_t qi = it.q0 + t * BM + rt;
      const int64_t lim = a.causal ? qi + a.sk - a.sq : a.sk - 1;  // keys j <= lim are valid
      const int64_t jmax = lim < a.sk - 1 ? lim : a.sk - 1;
      float m_ref = neg_inf(), l = 0.0f;
      for (int b = 0; b < n; ++b) {
        const int g = g0 + b, r = r0 + b;
        // S_t done: round r (round r + 16 needs rows this thread has not yet
        // let through)
        if (!tc_wait(bar(rnd(t, r)), rpar(r), args.max_polls, args.status)) {
          ok = false;
          atomicOr(args.status, DEV_TIMEOUT);
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (rt == 0) ATM_STAMP(4 + t, g);
        // a rescale waits for the previous O_t += P_t V: round r + 1 (issued
        // once the previous block's named barrier passed)
        tc_rows_block<T, D>(t_s(t, g & 1) + lane_off, t_o(t) + lane_off, b, (int64_t)b * BN, jmax, cs, m_ref, l,
                            ok, bar(rnd(t, r + 1)), rpar(r + 1), args.max_polls, args.status);
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        const int nbar = 1 + 2 * t + (g & 1);
        if (rt == 0) ATM_STAMP(6 + t, g);
        asm volatile("barrier.arrive.aligned %0, %1;" ::"r"(nbar), "n"(ATM_BM + 32) : "memory");
      }
      // the tile's last O += P V: round n + 1
      if (n > 0 && !tc_wait(bar(rnd(t, r0 + n + 1)), rpar(r0 + n + 1), args.max_polls, args.status))
        ok = false;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      // o = O / l in the input type; LSE = m ln 2 + log l; an empty row: 0,
      // -inf.  The TMEM loads are warp-collective, so every row thread loads;
      // rows past the end store nothing.
      const float inv = l > 0.0f ? recip_refined(l) : 0.0f;
      if constexpr (S::STAGE_BYTES > 0) {
        // 32 columns at a time: each lane packs its row's 64 bytes into the
        // warp's staging rows (16-byte chunks XOR-ed with the row's bits 1-2,
        // so that eight lanes cover all 32 banks), then the warp stores eight
        // rows' 64-byte pieces an instruction (lane L: row 8 i + L / 4, chunk
        // L % 4) instead of 32 rows' 16 bytes
        const uint32_t stg = sO + (uint32_t)(warp * 2048);
        const int64_t row0 = it.q0 + t * BM + (warp & 3) * 32;  // the warp's first query row
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t pkd[16];
#pragma unroll
          for (int h = 0; h < 32; h += 16) {
            float t16[16];
            if (n > 0) {
              tc_ld16(t_o(t) + lane_off + (uint32_t)(c + h), t16);
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) t16[i] = 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 16; i += 2) pkd[(h + i) / 2] = pack2<T>(t16[i] * inv, t16[i + 1] * inv);
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t addr = stg + (uint32_t)(lane * 64 + ((q ^ ((lane >> 1) & 3)) * 16));
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pkd[4 * q]),
                         "r"(pkd[4 * q + 1]), "r"(pkd[4 * q + 2]), "r"(pkd[4 * q + 3])
                         : "memory");
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int rr = 8 * i + (lane >> 2), q = lane & 3;
            const uint32_t addr = stg + (uint32_t)(rr * 64 + ((q ^ ((rr >> 1) & 3)) * 16));
            uint4 v;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(addr)
                         : "memory");
            if (row0 + rr < a.sq)
              *reinterpret_cast<uint4*>(o + (it.head * a.sq + row0 + rr) * D + c + q * 8) = v;
          }
          __syncwarp();
        }
      } else {
        T* orow = o + (it.head * a.sq + (qi < a.sq ? qi : 0)) * D;
#pragma unroll
        for (int c = 0; c < D; c += 16) {
          float t16[16];
          if (n > 0) {
            tc_ld16(t_o(t) + lane_off + (uint32_t)c, t16);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) t16[i] = 0.0f;
          }
          if (qi < a.sq) {
            uint4 w0, w1;
            w0.x = pack2<T>(t16[0] * inv, t16[1] * inv);
            w0.y = pack2<T>(t16[2] * inv, t16[3] * inv);
            w0.z = pack2<T>(t16[4] * inv, t16[5] * inv);
            w0.w = pack2<T>(t16[6] * inv, t16[7] * inv);
            w1.x = pack2<T>(t16[8] * inv, t16[9] * inv);
            w1.y = pack2<T>(t16[10] * inv, t16[11] * inv);
            w1.z = pack2<T>(t16[12] * inv, t16[13] * inv);
            w1.w = pack2<T>(t16[14] * inv, t16[15] * inv);
            *reinterpret_cast<uint4*>(orow + c) = w0;
            *reinterpret_cast<uint4*>(orow + c + 8) = w1;
          }
        }
      }
      if (qi < a.sq && lse != nullptr)
        lse[it.head * a.sq + qi] = l > 0.0f ? __fmaf_rn(m_ref, LN2, logf(l)) : neg_inf();
      if (tid == 0) ATM_STAMP(13, (int)k);
      advance(it);
    }
  }
  if (!ok) atomicOr(args.status, DEV_TIMEOUT);
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == S::ISSUE_WARP) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(S::TCOLS) : "memory");
  }
}

}  // namespace smx
