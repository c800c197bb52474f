// Attention forward on the 5th-generation tensor cores (tcgen05, TMEM): the
// same running state (m, l, o) as kernel_attention.cuh ("Online stable
// softmax", "Carry a weighted value numerator for attention" and "Reference
// summary"; "Softmax numerics architecture...", "From online softmax to tiled
// attention"), with both products issued by one thread as tcgen05.mma and
// accumulated in tensor memory:
//   S  (128 x 64 fp32, TMEM columns [D, D + 64))  = Q K_B^T
//   O  (128 x D fp32,  TMEM columns [0, D))      += P V_B
// One CTA of 128 threads takes 128 query rows of one head; thread r owns query
// row r, which is TMEM lane r, so the row's maximum and sum need no exchange.
// Operands sit in shared memory K-major with the 128-byte swizzle (8-row atoms
// of 1024 bytes; 16-byte chunks XOR-ed with the row): Q and K as stored, P
// written by the row threads, V transposed while it is staged (V^T rows are
// the head dimension, so the second product's B operand is K-major too).
//
// Per key block: one thread issues S = Q K^T and commits to an mbarrier (the
// commit also covers the previous block's O += P V^T); the next block's K
// (cp.async, second buffer) and V (registers) are fetched meanwhile; each row
// thread reads its 64 scores from TMEM,
// masks, updates (m, l), writes P (the input type) to shared memory and, when
// its reference maximum has to move, rescales its O row in TMEM; one thread
// issues O += P V^T and commits.  The reference maximum moves only when the
// block's maximum exceeds it by more than 8 (base-2 units): the exponentials
// then stay below 2^8, and l and o always share one reference, so the result
// is the same quotient (the rescale is exact bookkeeping, not an
// approximation).  Two CTAs share an SM (shared memory 97 KiB and up to 256
// TMEM columns each) so that one's softmax overlaps the other's products.  Every mbarrier wait is bounded; running out records
// SMX_ERR_TIMEOUT in the device status word.
#pragma once

#include <type_traits>

#include "kernel_attention.cuh"

namespace smx {

constexpr int ATT_TC_BM = 128;  // query rows per CTA (one per thread, one per TMEM lane)
constexpr int ATT_TC_BN = 64;   // keys per block
constexpr int ATT_TC_THREADS = 128;

struct AttnTcArgs {
  AttnArgs a;
  int* status;
  int64_t max_polls;
};

__device__ __forceinline__ uint32_t tc_su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// byte offset of element (r, k) of a K-major tile of `rows` rows with the
// 128-byte swizzle: 64-element column blocks of rows x 128 bytes, 8-row atoms
// of 1024 bytes, 16-byte chunks XOR-ed with the row in its atom
__device__ __forceinline__ uint32_t tc_off(int r, int k, int rows) {
  return (uint32_t)((k >> 6) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 +
                    ((((k & 63) >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}

// shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (the leading offset is not used by this layout)
__device__ __forceinline__ uint64_t tc_sdesc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// instruction descriptor of kind::f16: fp32 accumulator, A and B of type T,
// both K-major, M x N
template <typename T>
__device__ __forceinline__ uint32_t tc_idesc(int M, int N) {
  const uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(da), "l"(db), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
               : "memory");
}
// Wait for an mbarrier phase, bounded: at most max_polls polls and 200 ms of
// wall time, and no wait at all once the status word records a timeout (so a
// failure ends every CTA's waits quickly).  Returns false when it gave up.
__device__ __forceinline__ bool tc_wait(uint32_t mbar, uint32_t parity, int64_t max_polls,
                                        const int* status) {
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (int64_t it = 0; it < max_polls; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(mbar), "r"(parity)
        : "memory");
    if (done) return true;
    if ((it & 15) == 15) {
      if (*reinterpret_cast<const volatile int*>(status) & DEV_TIMEOUT) return false;
      uint64_t t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > 200000000ull) return false;
    }
  }
  return false;
}
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tc_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

template <typename T, int D>
__global__ void __launch_bounds__(ATT_TC_THREADS)
    k_attention_tc(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   T* __restrict__ o, float* __restrict__ lse, AttnTcArgs args) {
  static_assert(D == 64 || D == 128, "head dimension");
  constexpr int BM = ATT_TC_BM, BN = ATT_TC_BN;
  constexpr uint32_t TCOLS = D == 128 ? 256 : 128;  // O then S, a power of two
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t mbar[1];  // products done (S each block, then the last O)
  __shared__ uint32_t tmem_base;

  const AttnArgs& a = args.a;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int64_t head = blockIdx.y;
  const int64_t q0 = (int64_t)blockIdx.x * BM;
  const T* qh = q + head * a.sq * D;
  const T* kh = k + head * a.sk * D;
  const T* vh = v + head * a.sk * D;

  // 1024-aligned operand tiles: Q [BM][D], K [2][BN][D], V^T [D][BN], P [BM][BN]
  const uint32_t raw = tc_su32(smem_raw);
  uint8_t* base = smem_raw + ((1024 - (raw & 1023)) & 1023);
  uint8_t* sQ = base;
  uint8_t* sK0 = sQ + BM * D * 2;
  constexpr int KT = BN * D * 2;  // bytes of one K or V^T tile
  uint8_t* sVt = sK0 + 2 * KT;
  uint8_t* sP = sVt + KT;

  int64_t kv_end = a.sk;
  if (a.causal) {
    const int64_t last = q0 + BM - 1 < a.sq - 1 ? q0 + BM - 1 : a.sq - 1;
    kv_end = last + a.sk - a.sq + 1;
    if (kv_end > a.sk) kv_end = a.sk;
    if (kv_end < 0) kv_end = 0;
  }
  const int nblocks = (int)((kv_end + BN - 1) / BN);

  // Q: 16-byte chunks straight into the swizzled layout; rows past sq zero
  for (int i = tid; i < BM * (D / 8); i += ATT_TC_THREADS) {
    const int r = i / (D / 8), c = (i % (D / 8)) * 8;
    const uint32_t dst = tc_su32(sQ + tc_off(r, c, BM));
    if (q0 + r < a.sq)
      att_cp16(dst, qh + (q0 + r) * D + c);
    else
      asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0) : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tc_su32(&tmem_base)),
                 "r"(TCOLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_su32(&mbar[0])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base;
  const uint32_t t_o = tmem, t_s = tmem + D;
  // this thread's TMEM lane (its query row) in the warp's 32-lane slice
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  const int64_t qi = q0 + tid;
  const int64_t lim = a.causal ? qi + a.sk - a.sq : a.sk - 1;  // keys j <= lim are valid

  const uint32_t id_s = tc_idesc<T>(BM, BN), id_o = tc_idesc<T>(BM, D);
  bool ok = true;
  float m_ref = neg_inf(), l = 0.0f;

  // staging of key block b: K by cp.async into buffer (b & 1); V into
  // registers (vr) one block ahead, then transposed into V^T with eight 2-byte
  // stores per 16-byte chunk (lanes over consecutive keys, so a warp fills
  // whole chunks)
  constexpr int VCH = BN * (D / 8) / ATT_TC_THREADS;  // 16-byte V chunks per thread
  uint4 vr[VCH];
  auto stage_k = [&](int blk) {
    const int64_t key0 = (int64_t)blk * BN;
    uint8_t* sK = sK0 + (blk & 1) * KT;
    for (int i = tid; i < BN * (D / 8); i += ATT_TC_THREADS) {
      const int r = i / (D / 8), c = (i % (D / 8)) * 8;
      const uint32_t dst = tc_su32(sK + tc_off(r, c, BN));
      if (key0 + r < a.sk)
        att_cp16(dst, kh + (key0 + r) * D + c);
      else
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  auto load_v = [&](int blk) {
    const int64_t key0 = (int64_t)blk * BN;
#pragma unroll
    for (int u = 0; u < VCH; ++u) {
      const int i = tid + u * ATT_TC_THREADS;
      const int j = i % BN, c = (i / BN) * 8;
      vr[u] = make_uint4(0, 0, 0, 0);
      if (key0 + j < a.sk) vr[u] = __ldg(reinterpret_cast<const uint4*>(vh + (key0 + j) * D + c));
    }
  };
  auto store_vt = [&]() {
#pragma unroll
    for (int u = 0; u < VCH; ++u) {
      const int i = tid + u * ATT_TC_THREADS;
      const int j = i % BN, c = (i / BN) * 8;
      const uint16_t* e = reinterpret_cast<const uint16_t*>(&vr[u]);
#pragma unroll
      for (int t = 0; t < 8; ++t) *reinterpret_cast<uint16_t*>(sVt + tc_off(c + t, j, D)) = e[t];
    }
  };
  // block 0's K and V before the loop
  if (nblocks > 0) {
    stage_k(0);
    load_v(0);
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

  for (int b = 0; b < nblocks; ++b) {
    const int64_t key0 = (int64_t)b * BN;
    // S = Q K^T: D / 16 steps of K = 16 (two per 32 bytes of a 128-byte row)
    if (tid == 0) {
      const uint32_t kbase = tc_su32(sK0 + (b & 1) * KT);
#pragma unroll
      for (int s = 0; s < D / 16; ++s) {
        const uint32_t koff = (uint32_t)((s & 3) * 32);
        const uint64_t da = tc_sdesc(tc_su32(sQ) + (uint32_t)((s >> 2) * BM * 128) + koff);
        const uint64_t db = tc_sdesc(kbase + (uint32_t)((s >> 2) * BN * 128) + koff);
        tc_mma(t_s, da, db, id_s, s > 0 ? 1u : 0u);
      }
      tc_commit(tc_su32(&mbar[0]));
    }
    // the next block's K in flight while this one runs (its buffer's last
    // reader, the previous S, has finished)
    const bool more = b + 1 < nblocks;
    if (more) stage_k(b + 1);
    // S done; its commit covers every earlier product of the issuing thread,
    // so O += P V^T of the previous block has finished too: P, O and V^T may
    // be rewritten
    if (!tc_wait(tc_su32(&mbar[0]), (uint32_t)(b & 1), args.max_polls, args.status)) {
      ok = false;
      atomicOr(args.status, DEV_TIMEOUT);
    }
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    // this block's V^T from the registers, then the next block's V into them
    store_vt();
    if (more) load_v(b + 1);
    // this row's 64 scores: mask, block maximum in scaled base-2 units
    float s[BN];
#pragma unroll
    for (int c = 0; c < BN; c += 16) {
      float t16[16];
      tc_ld16(t_s + lane_off + (uint32_t)c, t16);
#pragma unroll
      for (int i = 0; i < 16; ++i) s[c + i] = t16[i];
    }
    float mx = neg_inf();
#pragma unroll
    for (int i = 0; i < BN; ++i) {
      const int64_t j = key0 + i;
      s[i] = (j > lim || j >= a.sk) ? neg_inf() : s[i] * a.scale_log2;
      mx = fmaxf(mx, s[i]);
    }
    // move the reference only when needed (see the header); alpha rescales l and O
    float alpha = 1.0f;
    if (mx > m_ref + 8.0f) {
      alpha = m_ref == neg_inf() ? 0.0f : ex2_full(m_ref - mx);
      m_ref = mx;
    }
    const float sub = m_ref == neg_inf() ? 0.0f : m_ref;
    float ps = 0.0f;
    // P row into shared memory, 8 keys (16 bytes) at a time
#pragma unroll
    for (int c = 0; c < BN; c += 8) {
      float p8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        p8[i] = ex2_full(s[c + i] - sub);
        ps += p8[i];
      }
      const uint4 w = make_uint4(pack2<T>(p8[0], p8[1]), pack2<T>(p8[2], p8[3]), pack2<T>(p8[4], p8[5]),
                                 pack2<T>(p8[6], p8[7]));
      *reinterpret_cast<uint4*>(sP + tc_off(tid, c, BM)) = w;
    }
    l = __fmaf_rn(l, alpha, ps);
    // TMEM loads and stores are warp-collective: a warp rescales when any of
    // its rows must (the others multiply by 1, exactly)
    if (b > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
      // O row *= alpha (the previous product has finished: waited above)
#pragma unroll
      for (int c = 0; c < D; c += 16) {
        float t16[16];
        tc_ld16(t_o + lane_off + (uint32_t)c, t16);
#pragma unroll
        for (int i = 0; i < 16; ++i) t16[i] *= alpha;
        tc_st16(t_o + lane_off + (uint32_t)c, t16);
      }
    }
    // P and V^T written, the next block's K landed
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    // O += P V^T: BN / 16 steps of K = 16 over the block's keys
    if (tid == 0) {
#pragma unroll
      for (int s2 = 0; s2 < BN / 16; ++s2) {
        const uint32_t koff = (uint32_t)((s2 & 3) * 32);
        const uint64_t da = tc_sdesc(tc_su32(sP) + (uint32_t)((s2 >> 2) * BM * 128) + koff);
        const uint64_t db = tc_sdesc(tc_su32(sVt) + (uint32_t)((s2 >> 2) * D * 128) + koff);
        tc_mma(t_o, da, db, id_o, (b > 0 || s2 > 0) ? 1u : 0u);
      }
    }
  }
  // the last O += P V^T: one more commit on the same barrier (every earlier
  // phase has been waited, so the parity names this one)
  if (nblocks > 0) {
    if (tid == 0) tc_commit(tc_su32(&mbar[0]));
    if (!tc_wait(tc_su32(&mbar[0]), (uint32_t)(nblocks & 1), args.max_polls, args.status)) ok = false;
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (!ok) atomicOr(args.status, DEV_TIMEOUT);

  // o = O / l in the input type; LSE = m ln 2 + log l; the empty row: 0, -inf.
  // The TMEM loads are warp-collective, so every thread loads; rows past the
  // end store nothing.
  const float inv = l > 0.0f ? recip_refined(l) : 0.0f;
  T* orow = o + (head * a.sq + (qi < a.sq ? qi : 0)) * D;
#pragma unroll
  for (int c = 0; c < D; c += 16) {
    float t16[16];
    if (nblocks > 0) {
      tc_ld16(t_o + lane_off + (uint32_t)c, t16);
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
  if (qi < a.sq && lse != nullptr) lse[head * a.sq + qi] = l > 0.0f ? __fmaf_rn(m_ref, LN2, logf(l)) : neg_inf();
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TCOLS) : "memory");
  }
}

}  // namespace smx
