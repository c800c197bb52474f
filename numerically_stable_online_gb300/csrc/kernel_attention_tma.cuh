// Attention forward with warp-specialised operand fetching: the running
// state (m, l, o) of "Online stable softmax" ("Carry a weighted value
// numerator for attention") and "Softmax numerics architecture..." ("From
// online softmax to tiled attention") on the 5th-generation tensor cores.
//
// A CTA takes TILES tiles of 128 query rows of one head (tile t: warps
// 4t .. 4t + 3, row thread r = TMEM lane r of the tile's accumulators) and
// walks the head's keys in blocks of 64.  TILES = 1: two CTAs an SM; TILES =
// 2: one CTA an SM whose two tiles read the same K and V stages (a key block
// crosses from L2 to shared memory once per 256 query rows).  Tensor memory:
//   O_t            columns t D ..                          (fp32, D wide)
//   S_t, buffer i  columns TILES D + 128 t + 64 i ..        (fp32, 64 wide; P,
//                  packed two to a column, over its first 32)
// Warp roles: the row warps (the per-block softmax of tc_rows_block: mask,
// maximum, exponentials, sum, P into tensor memory, O rescaled when the
// reference maximum moves); one issuing warp per tile, whose lane 0 issues
// that tile's tcgen05.mma (one issuing thread was measured to leave the
// tensor core idle with two tiles' 64-key products: issuing a product waits
// for room in the tensor pipe); one warp that fetches Q and the K stages and
// one that fetches the V stages, each by tensor-map bulk copies
// (cp.async.bulk.tensor, 128-byte swizzle, no multicast) completing on full
// barriers.  The row warps issue no copies.
//
// Issue rounds.  Tile t's issuing lane issues its products in rounds: round
// 0 is S_t(0), round 1 S_t(1), and round b + 2 (once the tile's rows finished
// block b: named barrier) is O_t += P_t(b) V(b) followed by S_t(b + 2) (the
// tile's n blocks make rounds 0 .. n + 1).  Each round ends with one
// tcgen05.commit, on round barrier R_t[r % 8]; it completes when every
// product of the round (and before it) has finished.  Everything else waits
// on those: the rows for their scores (round b), a rescale for the previous
// O += P V (round b + 1), the epilogue for the last one (round n + 1), the K
// fetcher for a stage's previous scores (K stage j % NK is free after round
// j - NK) and the V fetcher for its previous O += P V (V stage j % NV is free
// after round j - NV + 2).  In each case the next round on the same barrier
// (eight rounds later) cannot finish before the waiter has moved on -- it
// needs rows the waiter has not yet let through, or a stage it has not yet
// fetched -- so a phase parity names one round.  One commit a round: each
// commit is costly for the issuing thread, and a tile's 64-key rounds are
// short.  Rows past the end of the query or key range are zero in shared
// memory (the copies fill them) and masked.  Every mbarrier wait is bounded;
// running out records SMX_ERR_TIMEOUT.
#pragma once

#include <cuda.h>

#include "kernel_attention_tc.cuh"
#include "smx_async.cuh"

namespace smx {

constexpr int ATM_BM = 128;  // query rows per tile
constexpr int ATM_BN = 64;   // keys per block
constexpr int ATM_NBAR = 28;

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
  // shared memory: Q [TILES][128][D], K [NK][64][D], V [NV][64][D] (16-bit)
  template <int D>
  __host__ __device__ static constexpr int tile_bytes() {
    return (TILES * ATM_BM * D + (NK + NV) * ATM_BN * D) * 2;
  }
  // the launch adds 1024 bytes so that the tiles start on a 1024-byte
  // boundary (the 128-byte swizzle's atom); the barriers and the TMEM
  // address (ATM_NBAR * 8 + 4 bytes) sit in that slack
  template <int D>
  __host__ __device__ static constexpr int smem_bytes() {
    return tile_bytes<D>() + 1024;
  }
};

struct AttnTmaArgs {
  AttnArgs a;
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
// 8 K fetch issued, 9 V fetch issued
__device__ long long g_atm_trace[2][10][64];
#define ATM_STAMP(ev, blk)                                                                   \
  do {                                                                                      \
    if (trace_slot >= 0 && (blk) < 64) g_atm_trace[trace_slot][ev][blk] = clock64();        \
  } while (0)
#else
#define ATM_STAMP(ev, blk) \
  do {                     \
  } while (0)
#endif

template <typename T, int D, int TILES>
__global__ void __launch_bounds__(AtmShape<TILES>::BLOCK, AtmShape<TILES>::CTAS_PER_SM)
    k_attention_tma(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, T* __restrict__ o, float* __restrict__ lse,
                    AttnTmaArgs args) {
  static_assert(D == 64 || D == 128, "head dimension");
  using S = AtmShape<TILES>;
  constexpr int BM = ATM_BM, BN = ATM_BN, NK = S::NK, NV = S::NV;
  constexpr int QT = BM * D * 2;  // bytes of a Q tile
  constexpr int KT = BN * D * 2;  // bytes of a K or V stage
  // barrier indices: round barriers R_t[i] at B_R + 8 t + i, full barriers
  // of the K and V stages, Q, the probe's, the issuing lanes' drains
  constexpr int B_R = 0, B_KF = 16, B_VF = 20, B_Q = 24, B_PROBE = 25, B_DRAIN = 26;
  static_assert(NK <= 4 && NV <= 4 && B_DRAIN + 2 == ATM_NBAR, "barrier layout");
  auto rnd = [](int t, int r) { return B_R + 8 * t + (r & 7); };
  auto rpar = [](int r) { return (uint32_t)((r >> 3) & 1); };
  extern __shared__ __align__(16) uint8_t smem_raw[];

  const AttnArgs& a = args.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t head = blockIdx.y;
  // causal: the CTAs with the most key blocks start first
  const int64_t qblk = a.causal ? (int64_t)(gridDim.x - 1 - blockIdx.x) : (int64_t)blockIdx.x;
  const int64_t q0 = qblk * (TILES * BM);
#ifdef SMX_ATM_TRACE
  const int trace_slot = blockIdx.x == 0 ? (blockIdx.y == 0 ? 0 : (blockIdx.y == 64 ? 1 : -1)) : -1;
#endif

  const uint32_t raw = tc_su32(smem_raw);
  const uint32_t pad = (1024 - (raw & 1023)) & 1023;
  uint8_t* base = smem_raw + pad;
  const uint32_t sQ = tc_su32(base), sK = sQ + TILES * QT, sV = sK + NK * KT;
  // the barriers: in the alignment gap when it has room, else after the tiles
  constexpr uint32_t AUX = ATM_NBAR * 8 + 4;
  uint8_t* aux = pad >= AUX ? smem_raw : base + S::template tile_bytes<D>();
  uint64_t* bars = reinterpret_cast<uint64_t*>(aux);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + ATM_NBAR);
  const uint32_t bar0 = tc_su32(bars);
  auto bar = [bar0](int i) { return bar0 + 8u * (uint32_t)i; };

  // key blocks of each tile (0 for a tile wholly past the query rows)
  int nb0 = 0, nb1 = 0;
#pragma unroll
  for (int t = 0; t < TILES; ++t) {
    const int64_t r0 = q0 + t * BM;
    int64_t kv_end = a.sk;
    if (r0 >= a.sq) {
      kv_end = 0;
    } else if (a.causal) {
      const int64_t last = r0 + BM - 1 < a.sq - 1 ? r0 + BM - 1 : a.sq - 1;
      kv_end = last + a.sk - a.sq + 1;
      if (kv_end > a.sk) kv_end = a.sk;
      if (kv_end < 0) kv_end = 0;
    }
    (t ? nb1 : nb0) = (int)((kv_end + BN - 1) / BN);
  }
  const int nmax = nb0 > nb1 ? nb0 : nb1;

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

  if (warp >= S::ISSUE_WARP && warp < S::ISSUE_WARP + TILES) {
    // the issuing warp of tile t
    const int t = warp - S::ISSUE_WARP;
    const int n = t ? nb1 : nb0;
    const uint32_t id_s = tc_idesc<T>(BM, BN), id_o = tc_idesc<T>(BM, D, true);
    const uint32_t qb = sQ + (uint32_t)(t * QT);
    // S_t(j) = Q_t K(j)^T: D / 16 steps of K = 16 (two per 32 bytes of a
    // 128-byte row)
    auto issue_s = [&](int j) {
      const uint32_t kb = sK + (uint32_t)((j % NK) * KT);
#pragma unroll
      for (int st = 0; st < D / 16; ++st) {
        const uint32_t koff = (uint32_t)((st & 3) * 32);
        const uint64_t da = tc_sdesc(qb + (uint32_t)((st >> 2) * BM * 128) + koff);
        const uint64_t db = tc_sdesc(kb + (uint32_t)((st >> 2) * BN * 128) + koff);
        tc_mma(t_s(t, j & 1), da, db, id_s, st > 0 ? 1u : 0u);
      }
    };
    // O_t += P_t(j) V(j): BN / 16 steps of K = 16 keys, P from the score
    // tile's first columns (8 a step), V as the MN-major B operand (two 8-key
    // groups, 2048 bytes, a step)
    auto issue_pv = [&](int j) {
      const uint32_t vb = sV + (uint32_t)((j % NV) * KT), pb = t_s(t, j & 1);
#pragma unroll
      for (int s2 = 0; s2 < BN / 16; ++s2) {
        const uint64_t db = tc_sdesc_mn(vb + (uint32_t)(s2 * 2048), (uint32_t)(BN * 128));
        tc_mma_ta(t_o(t), pb + (uint32_t)(s2 * 8), db, id_o, (j > 0 || s2 > 0) ? 1u : 0u);
      }
    };
    auto wait_or_flag = [&](uint32_t b_, uint32_t par) {
      if (!tc_wait(b_, par, args.max_polls, args.status)) {
        ok = false;
        atomicOr(args.status, DEV_TIMEOUT);
      }
    };
    // rounds 0 and 1 (a round with nothing to issue still commits, so every
    // round 0 .. n + 1 completes its barrier's phase)
    if (lane == 0 && n > 0) {
      wait_or_flag(bar(B_Q), 0u);
      for (int r = 0; r < 2; ++r) {
        if (r < n) {
          wait_or_flag(bar(B_KF + r % NK), (uint32_t)((r / NK) & 1));
          issue_s(r);
        }
        tc_commit(bar(rnd(t, r)));
      }
    }
    __syncwarp();
    for (int b = 0; b < n; ++b) {
      // the tile's rows finished block b (P_t(b) in tensor memory, O_t
      // rescaled): named barrier 1 + 2 t + (b & 1); the rows are at most one
      // block ahead of this warp, so two barriers never mix generations
      const int nbar = 1 + 2 * t + (b & 1);
      asm volatile("barrier.sync.aligned %0, %1;" ::"r"(nbar), "n"(ATM_BM + 32) : "memory");
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (lane == 0) {
        ATM_STAMP(t, b);
        // round b + 2
        wait_or_flag(bar(B_VF + b % NV), (uint32_t)((b / NV) & 1));
        issue_pv(b);
        if (b + 2 < n) {
          wait_or_flag(bar(B_KF + (b + 2) % NK), (uint32_t)(((b + 2) / NK) & 1));
          issue_s(b + 2);
        }
        tc_commit(bar(rnd(t, b + 2)));
        ATM_STAMP(2 + t, b);
      }
      __syncwarp();
    }
    // every product this lane issued has finished before the tensor memory is
    // freed (the row threads' waits cover them on the normal path; after a
    // wait ran out they may not): one more commit, waited by wall time only
    if (lane == 0 && n > 0) {
      tc_commit(bar(B_DRAIN + t));
      tc_wait_drain(bar(B_DRAIN + t), 0u);
    }
    __syncwarp();
  } else if (warp == S::KLOAD_WARP || warp == S::VLOAD_WARP) {
    // the stage fetchers: Q and K, or V
    const bool is_k = warp == S::KLOAD_WARP;
    const CUtensorMap* map = is_k ? &tm_k : &tm_v;
    const uint32_t stages = is_k ? sK : sV;
    const int full0 = is_k ? B_KF : B_VF;
    const int ns = is_k ? NK : NV;
    if (lane == 0 && nmax > 0) {
      tma_prefetch_map(map);
      if (is_k) {
        tma_prefetch_map(&tm_q);
        // the Q tiles (rows past the query range land as zeros)
        mbar_arrive_expect_tx(bar(B_Q), (uint32_t)(TILES * QT));
#pragma unroll
        for (int t = 0; t < TILES; ++t)
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tma_load_3d(sQ + (uint32_t)(t * QT + h * BM * 128), &tm_q, h * 64, (int)(q0 + t * BM), (int)head,
                        bar(B_Q));
      }
      for (int j = 0; j < nmax; ++j) {
        const int s = j % ns;
        // the stage's previous block (j - ns) has been read by every tile that
        // has it: its scores (round j - NK) or its O += P V (round j - NV + 2)
        // finished
        const int r = is_k ? j - NK : j - NV + 2;
#pragma unroll
        for (int t = 0; t < TILES; ++t) {
          if (j >= ns && j - ns < (t ? nb1 : nb0) &&
              !atm_wait_lazy(bar(rnd(t, r)), rpar(r), args.max_polls, args.status)) {
            ok = false;
            atomicOr(args.status, DEV_TIMEOUT);
          }
        }
        ATM_STAMP(is_k ? 8 : 9, j);
        mbar_arrive_expect_tx(bar(full0 + s), (uint32_t)KT);
#pragma unroll
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(stages + (uint32_t)(s * KT + h * BN * 128), map, h * 64, j * BN, (int)head, bar(full0 + s));
      }
      // every copy this lane issued has landed before the CTA ends (already
      // so on the normal path: the issuing lanes waited for each)
      for (int s = 0; s < ns && s < nmax; ++s) {
        const int jl = s + ((nmax - 1 - s) / ns) * ns;  // the last block fetched into stage s
        tc_wait_drain(bar(full0 + s), (uint32_t)((jl / ns) & 1));
      }
      if (is_k) tc_wait_drain(bar(B_Q), 0u);
    }
    __syncwarp();
  } else {
    // row threads: tile t, query row qi (TMEM lane rt of the tile)
    const int t = tid >> 7, rt = tid & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int64_t qi = q0 + t * BM + rt;
    const int64_t lim = a.causal ? qi + a.sk - a.sq : a.sk - 1;  // keys j <= lim are valid
    const int64_t jmax = lim < a.sk - 1 ? lim : a.sk - 1;
    const float cs = a.scale_log2;
    float m_ref = neg_inf(), l = 0.0f;
    const int n = t ? nb1 : nb0;
    for (int b = 0; b < n; ++b) {
      // S_t(b) done: round b (round b + 8 needs block b + 6's named barrier)
      if (!tc_wait(bar(rnd(t, b)), rpar(b), args.max_polls, args.status)) {
        ok = false;
        atomicOr(args.status, DEV_TIMEOUT);
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (rt == 0) ATM_STAMP(4 + t, b);
      // a rescale waits for O_t += P_t(b - 1) V(b - 1): round b + 1 (issued
      // once block b - 1's named barrier passed; round b + 9 needs block
      // b + 7)
      tc_rows_block<T, D>(t_s(t, b & 1) + lane_off, t_o(t) + lane_off, b, (int64_t)b * BN, jmax, cs, m_ref, l, ok,
                          bar(rnd(t, b + 1)), rpar(b + 1), args.max_polls, args.status);
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      const int nbar = 1 + 2 * t + (b & 1);
      if (rt == 0) ATM_STAMP(6 + t, b);
      asm volatile("barrier.arrive.aligned %0, %1;" ::"r"(nbar), "n"(ATM_BM + 32) : "memory");
    }
    // the tile's last O += P V: round n + 1, the last
    if (n > 0 && !tc_wait(bar(rnd(t, n + 1)), rpar(n + 1), args.max_polls, args.status)) ok = false;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    // o = O / l in the input type; LSE = m ln 2 + log l; an empty row: 0, -inf.
    // The TMEM loads are warp-collective, so every row thread loads; rows
    // past the end store nothing.
    const float inv = l > 0.0f ? recip_refined(l) : 0.0f;
    T* orow = o + (head * a.sq + (qi < a.sq ? qi : 0)) * D;
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
    if (qi < a.sq && lse != nullptr)
      lse[head * a.sq + qi] = l > 0.0f ? __fmaf_rn(m_ref, LN2, logf(l)) : neg_inf();
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
