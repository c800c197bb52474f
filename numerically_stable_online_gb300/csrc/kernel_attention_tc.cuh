// Attention forward on the 5th-generation tensor cores (tcgen05, TMEM): the
// same running state (m, l, o) as kernel_attention.cuh ("Online stable
// softmax", "Carry a weighted value numerator for attention" and "Reference
// summary"; "Softmax numerics architecture...", "From online softmax to tiled
// attention"), with both products issued by one thread as tcgen05.mma and
// accumulated in tensor memory:
//   S  (128 x 64 fp32, TMEM columns D + 64 (b & 1) onward) = Q K_b^T
//   O  (128 x D fp32,  TMEM columns [0, D))              += P_b V_b
// One CTA takes 128 query rows of one head: row thread r (warps 0-3) owns
// query row r, which is TMEM lane r, so the row's maximum and sum need no
// exchange; a fifth warp issues the products.
// Operands sit in shared memory with the 128-byte swizzle (8-row atoms of
// 1024 bytes; 16-byte chunks XOR-ed with the row), all tiles in one layout:
// rows of 64 16-bit elements.  Q and K are K-major operands; V, staged as
// stored ([key][head dim]), is the second product's B operand in MN-major
// form, so nothing is transposed.  P (the input type) stays in tensor memory:
// each row thread writes its packed row over the first 32 columns of the
// score tile it has just read, and the second product takes A from there.
//
// Pipeline, per key block b: S(b + 1) is already issued (two S tiles in TMEM,
// two K and three V buffers in shared memory) when the row threads take
// S(b), so the tensor core computes the next scores and the previous
// O += P V while the rows compute this block's exponentials.  Each row thread
// masks its 64 scores, updates (m, l), writes P, and -- only when its
// reference maximum has to move -- waits for the previous O += P V and
// rescales its O row in TMEM; it then arrives (without waiting) on a named
// barrier, on which the issuing warp waits before it issues O += P V and the
// scores two blocks ahead.  K and V of later blocks are copied by cp.async as
// soon as their buffers are free (known from S(b): one thread's products
// finish in issue order).  The reference maximum moves only when the block's
// maximum exceeds it by more than 8 (base-2 units): the exponentials then
// stay below 2^8, and l and o always share one reference, so the result is
// the same quotient (the rescale is exact bookkeeping, not an
// approximation).  Two CTAs share an SM (shared memory 113 KiB and 256 TMEM
// columns each) so that one's softmax overlaps the other's products.
// Every mbarrier wait is bounded; running out records SMX_ERR_TIMEOUT in the
// device status word.
#pragma once

#include <type_traits>

#include "kernel_attention.cuh"

namespace smx {

constexpr int ATT_TC_BM = 128;  // query rows per CTA (one per thread, one per TMEM lane)
constexpr int ATT_TC_BN = 64;   // keys per block
constexpr int ATT_TC_THREADS = 128;                 // row threads (warps 0-3)
constexpr int ATT_TC_BLOCK = ATT_TC_THREADS + 32;   // plus one warp that issues the products
// shared memory of the operand tiles: Q [128][D], K [2][64][D], V [3][64][D]
// (16-bit elements); the launch adds 1024 bytes so that the tiles can start on
// a 1024-byte boundary, and the barriers live in that slack
template <int D>
__host__ __device__ constexpr int att_tc_tile_bytes() {
  return (ATT_TC_BM * D + 5 * ATT_TC_BN * D) * 2;
}

struct AttnTcArgs {
  AttnArgs a;
  int* status;
  int64_t max_polls;
  int64_t probe_polls;  // > 0: thread 0 first waits this many polls on a barrier nothing
                        // signals and records SMX_ERR_TIMEOUT (a probe of the error path)
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

// the same for an MN-major operand (each 128-byte row holds 64 consecutive
// N-elements of one K index; 8 K-rows make a 1024-byte atom): 8-row groups
// along K are 1024 bytes apart (stride offset), the 64-element halves along N
// are `lbo` bytes apart (leading offset)
__device__ __forceinline__ uint64_t tc_sdesc_mn(uint32_t saddr, uint32_t lbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// instruction descriptor of kind::f16: fp32 accumulator, A and B of type T,
// A K-major, B K-major or (b_mn) MN-major, M x N
template <typename T>
__device__ __forceinline__ uint32_t tc_idesc(int M, int N, bool b_mn = false) {
  const uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(da), "l"(db), "r"(idesc), "r"(acc)
      : "memory");
}
// the same with the A operand in tensor memory: M rows in the lanes, K
// 16-bit elements packed two to a 32-bit column (element 2c in the low half)
__device__ __forceinline__ void tc_mma_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t db, uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem_d),
      "r"(tmem_a), "l"(db), "r"(idesc), "r"(acc)
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
  // a phase that has already completed costs one test (no timer read)
  {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(mbar), "r"(parity)
        : "memory");
    if (done) return true;
  }
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
// Wait for an mbarrier phase bounded by wall time only (200 ms): the drain of
// the kernel's own asynchronous work before it frees tensor memory, which
// must end also after another wait has run out.
__device__ __forceinline__ bool tc_wait_drain(uint32_t mbar, uint32_t parity) {
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (;;) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(mbar), "r"(parity)
        : "memory");
    if (done) return true;
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > 200000000ull) return false;
  }
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
// 64 consecutive columns of this warp's 32 lanes; the wait is part of the same
// statement, so no use of the values can be scheduled before it
__device__ __forceinline__ void tc_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
      "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
      "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
      "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
// three-input maximum (one instruction on this architecture)
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// 32 consecutive columns of this warp's 32 lanes from registers; the wait is
// part of the same statement
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {"
      "%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
        "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
        "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
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

// One key block of one row thread's online softmax on tensor-memory tiles
// (the thread's query row is its TMEM lane; ts and to carry the warp's lane
// offset): read the row's 64 scores at ts, mask keys past jmax, update the
// reference maximum m_ref and the sum l, rescale the row's O at `to` when the
// reference moves (after the previous O += P V: the o_bar phase of parity
// o_par), and write P (type T, packed two to a column) over the first 32
// columns of the score tile.  The reference moves only when the block's
// maximum exceeds it by more than 8 (base-2 units): the exponentials stay
// below 2^8, and l and O always share one reference.
template <typename T, int D>
__device__ __forceinline__ void tc_rows_block(uint32_t ts, uint32_t to, int b, int64_t key0, int64_t jmax, float cs,
                                              float& m_ref, float& l, bool& ok, uint32_t o_bar,
                                              uint32_t o_par, int64_t max_polls, int* status) {
  constexpr int BN = 64;
  float sc[BN];
  tc_ld64(ts, sc);
  const int64_t nv64 = jmax - key0 + 1;
  const int nv = nv64 < 0 ? 0 : (nv64 > BN ? BN : (int)nv64);
  if (nv < BN) {
#pragma unroll
    for (int i = 0; i < BN; ++i)
      if (i >= nv) sc[i] = neg_inf();
  }
  // block maximum (four chains of three-input max), in scaled base-2 units
  float mx4[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) mx4[j] = fmaxf(sc[2 * j], sc[2 * j + 1]);
#pragma unroll
  for (int i = 8; i < BN; i += 8)
#pragma unroll
    for (int j = 0; j < 4; ++j) mx4[j] = max3(mx4[j], sc[i + 2 * j], sc[i + 2 * j + 1]);
  const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * cs;
  float alpha = 1.0f;
  if (mx > m_ref + 8.0f) {
    alpha = m_ref == neg_inf() ? 0.0f : ex2_full(m_ref - mx);
    m_ref = mx;
  }
  const float nsub = m_ref == neg_inf() ? 0.0f : -m_ref;
  // p = 2^(s cs - m_ref) (pairs by one f32x2 FMA), packed to the input type;
  // two f32x2 partial sums
  uint32_t pk2[BN / 2];
  const unsigned long long cs2 = pk(cs, cs), ns2 = pk(nsub, nsub);
  unsigned long long acc2[2] = {0ull, 0ull};
#pragma unroll
  for (int i = 0; i < BN; i += 2) {
    const unsigned long long e = fma2(pk(sc[i], sc[i + 1]), cs2, ns2);
    const float p0 = ex2_ftz(pk_lo(e)), p1 = ex2_ftz(pk_hi(e));
    acc2[(i >> 1) & 1] = add2(acc2[(i >> 1) & 1], pk(p0, p1));
    pk2[i / 2] = pack2<T>(p0, p1);
  }
  const float ps = (pk_lo(acc2[0]) + pk_hi(acc2[0])) + (pk_lo(acc2[1]) + pk_hi(acc2[1]));
  l = __fmaf_rn(l, alpha, ps);
  // TMEM loads and stores are warp-collective: a warp rescales when any of
  // its rows must (the others multiply by 1, exactly)
  if (b > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
    // O += P(b - 1) V(b - 1) finished first
    if (!tc_wait(o_bar, o_par, max_polls, status)) {
      ok = false;
      atomicOr(status, DEV_TIMEOUT);
    }
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
    for (int c = 0; c < D; c += 16) {
      float t16[16];
      tc_ld16(to + (uint32_t)c, t16);
#pragma unroll
      for (int i = 0; i < 16; ++i) t16[i] *= alpha;
      tc_st16(to + (uint32_t)c, t16);
    }
  }
  tc_st32(ts, pk2);
}

template <typename T, int D>
__global__ void __launch_bounds__(ATT_TC_BLOCK, 2)
    k_attention_tc(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   T* __restrict__ o, float* __restrict__ lse, AttnTcArgs args) {
  static_assert(D == 64 || D == 128, "head dimension");
  constexpr int BM = ATT_TC_BM, BN = ATT_TC_BN;
  constexpr uint32_t TCOLS = 256;  // O (D columns) then two S buffers of 64: a power of two
  extern __shared__ __align__(16) uint8_t smem_raw[];

  const AttnArgs& a = args.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool row_thread = tid < ATT_TC_THREADS;
  const int64_t head = blockIdx.y;
  const int64_t q0 = (int64_t)blockIdx.x * BM;
  const T* qh = q + head * a.sq * D;
  const T* kh = k + head * a.sk * D;
  const T* vh = v + head * a.sk * D;

  // 1024-aligned operand tiles: Q [BM][D], K [2][BN][D], V [3][BN][D]
  const uint32_t raw = tc_su32(smem_raw);
  const uint32_t pad = (1024 - (raw & 1023)) & 1023;
  uint8_t* base = smem_raw + pad;
  uint8_t* sQ = base;
  uint8_t* sK0 = sQ + BM * D * 2;
  constexpr int KT = BN * D * 2;  // bytes of one K or V tile
  uint8_t* sV0 = sK0 + 2 * KT;
  // six mbarriers (S of even / odd key blocks; O += P V; the last O += P V;
  // the probe's, never signalled; the issuing lane's drain) and the TMEM
  // address: in the alignment gap when it has room, else after the tiles (the
  // launch's 1024 spare bytes hold the gap plus these 52 bytes)
  uint8_t* aux = pad >= 64 ? smem_raw : base + att_tc_tile_bytes<D>();
  uint64_t* mbar = reinterpret_cast<uint64_t*>(aux);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aux + 48);

  int64_t kv_end = a.sk;
  if (a.causal) {
    const int64_t last = q0 + BM - 1 < a.sq - 1 ? q0 + BM - 1 : a.sq - 1;
    kv_end = last + a.sk - a.sq + 1;
    if (kv_end > a.sk) kv_end = a.sk;
    if (kv_end < 0) kv_end = 0;
  }
  const int nblocks = (int)((kv_end + BN - 1) / BN);

  // Q: 16-byte chunks straight into the swizzled layout; rows past sq zero
  if (row_thread) {
    for (int i = tid; i < BM * (D / 8); i += ATT_TC_THREADS) {
      const int r = i / (D / 8), c = (i % (D / 8)) * 8;
      const uint32_t dst = tc_su32(sQ + tc_off(r, c, BM));
      if (q0 + r < a.sq)
        att_cp16(dst, qh + (q0 + r) * D + c);
      else
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0) : "memory");
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tc_su32(tmem_slot)),
                 "r"(TCOLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < 6; ++i) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_su32(mbar + i)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  // the error-path probe: a wait on a barrier nothing signals runs out
  if (args.probe_polls > 0 && tid == 0 &&
      !tc_wait(tc_su32(&mbar[4]), 0u, args.probe_polls, args.status))
    atomicOr(args.status, DEV_TIMEOUT);
  const uint32_t t_o = tmem, t_s = tmem + D;
  // this thread's TMEM lane (its query row) in the warp's 32-lane slice
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  const int64_t qi = q0 + tid;
  const int64_t lim = a.causal ? qi + a.sk - a.sq : a.sk - 1;  // keys j <= lim are valid

  const uint32_t id_s = tc_idesc<T>(BM, BN), id_o = tc_idesc<T>(BM, D, true);
  bool ok = true;
  float m_ref = neg_inf(), l = 0.0f;
  // keys j <= jmax are valid for this row
  const int64_t jmax = lim < a.sk - 1 ? lim : a.sk - 1;
  const float cs = a.scale_log2;  // > 0, so the raw maximum scales to the scaled one

  // key block blk of K or V into tile buffer (blk % nbuf) by cp.async, rows past
  // the keys zero; one commit group each, empty past the last block (so the
  // group count per block is fixed).  V keeps its stored layout: it is the
  // second product's B operand in MN-major form (N = head dimension).
  // this thread's chunks of a tile: column c0 of rows r0 + RS u (RS a
  // multiple of 8, so the swizzle phase is fixed and the shared offset
  // advances by whole atoms)
  constexpr int CPR = D / 8;                   // 16-byte chunks a row
  constexpr int RS = ATT_TC_THREADS / CPR;    // rows a pass
  constexpr int NU = BN / RS;                  // passes a tile
  const int r0 = tid / CPR, c0 = (tid % CPR) * 8;
  const uint32_t soff = tc_off(r0, c0, BN);
  auto stage = [&](const T* src, uint8_t* tiles, int nbuf, int blk) {
    if (blk < nblocks) {
      const int64_t key0 = (int64_t)blk * BN;
      const uint32_t dst = tc_su32(tiles + (blk % nbuf) * KT) + soff;
      const T* g = src + (key0 + r0) * D + c0;
      if (key0 + BN <= a.sk) {
#pragma unroll
        for (int u = 0; u < NU; ++u) att_cp16(dst + (uint32_t)(u * RS * 128), g + (int64_t)u * RS * D);
      } else {
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          if (key0 + r0 + u * RS < a.sk)
            att_cp16(dst + (uint32_t)(u * RS * 128), g + (int64_t)u * RS * D);
          else
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst + (uint32_t)(u * RS * 128)), "r"(0)
                         : "memory");
        }
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  // S(blk) = Q K(blk)^T into TMEM buffer (blk & 1): D / 16 steps of K = 16
  // (two per 32 bytes of a 128-byte row); committed to mbar[blk & 1]
  auto issue_s = [&](int blk) {
    const uint32_t kbase = tc_su32(sK0 + (blk & 1) * KT);
#pragma unroll
    for (int st = 0; st < D / 16; ++st) {
      const uint32_t koff = (uint32_t)((st & 3) * 32);
      const uint64_t da = tc_sdesc(tc_su32(sQ) + (uint32_t)((st >> 2) * BM * 128) + koff);
      const uint64_t db = tc_sdesc(kbase + (uint32_t)((st >> 2) * BN * 128) + koff);
      tc_mma(t_s + (uint32_t)((blk & 1) * BN), da, db, id_s, st > 0 ? 1u : 0u);
    }
    tc_commit(tc_su32(&mbar[blk & 1]));
  };
  // O += P(blk) V(blk): BN / 16 steps of K = 16 over the block's keys, P from
  // the first BN / 2 columns of the block's TMEM score tile (8 columns a
  // step), V (buffer blk % 3) two 8-key groups, 2048 bytes, a step; committed
  // to mbar[2], and the last block's also to mbar[3]
  auto issue_pv = [&](int blk) {
    const uint32_t vbase = tc_su32(sV0 + (blk % 3) * KT);
    const uint32_t pbase = t_s + (uint32_t)((blk & 1) * BN);
#pragma unroll
    for (int s2 = 0; s2 < BN / 16; ++s2) {
      const uint64_t db = tc_sdesc_mn(vbase + (uint32_t)(s2 * 2048), (uint32_t)(BN * 128));
      tc_mma_ta(t_o, pbase + (uint32_t)(s2 * 8), db, id_o, (blk > 0 || s2 > 0) ? 1u : 0u);
    }
    tc_commit(tc_su32(&mbar[2]));
    if (blk == nblocks - 1) tc_commit(tc_su32(&mbar[3]));
  };

  // blocks 0 and 1's K and block 0's V before the loop
  if (row_thread) {
    stage(kh, sK0, 2, 0);
    stage(vh, sV0, 3, 0);
    stage(kh, sK0, 2, 1);
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

  if (!row_thread) {
    // The issuing warp.  Tensor-core order: S(0), S(1), then per block b,
    // once the row threads have finished it (named barrier 1 + (b & 1): P(b)
    // in TMEM, O rescaled, V(b) and K(b + 2) landed), O += P(b) V(b) and
    // S(b + 2) into the score tile that holds P(b).  One thread's products
    // run in issue order, so S(b + 2) overwrites P(b) only after O += P(b) V(b)
    // has read it.
    if (lane == 0 && nblocks > 0) {
      issue_s(0);
      if (nblocks > 1) issue_s(1);
    }
    __syncwarp();
    for (int b = 0; b < nblocks; ++b) {
      // named barrier 1 + (b & 1): the row threads can be at most one block
      // ahead of this warp (they need S(b + 1), issued after the previous
      // barrier), so two barriers never mix generations
      if (b & 1)
        asm volatile("barrier.sync.aligned 2, %0;" ::"n"(ATT_TC_BLOCK) : "memory");
      else
        asm volatile("barrier.sync.aligned 1, %0;" ::"n"(ATT_TC_BLOCK) : "memory");
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (lane == 0) {
        issue_pv(b);
        if (b + 2 < nblocks) issue_s(b + 2);
      }
      __syncwarp();
    }
    // every product this lane issued has finished before the tensor memory is
    // freed (the row threads' waits cover them on the normal path; after a
    // wait ran out they may not): one more commit, waited by wall time only
    if (lane == 0 && nblocks > 0) {
      tc_commit(tc_su32(&mbar[5]));
      tc_wait_drain(tc_su32(&mbar[5]), 0u);
    }
    __syncwarp();
  } else {
    for (int b = 0; b < nblocks; ++b) {
      const int64_t key0 = (int64_t)b * BN;
      // S(b) done.  mbar[x] takes every other block's commit, and S(b + 2)
      // is issued only after every row thread finished block b (so after
      // this wait): the phase parity is unambiguous
      if (!tc_wait(tc_su32(&mbar[b & 1]), (uint32_t)((b >> 1) & 1), args.max_polls, args.status)) {
        ok = false;
        atomicOr(args.status, DEV_TIMEOUT);
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      // S(b) finished, so did every product issued before it: the K buffer
      // S(b) read takes block b + 2, the V buffer O += P(b - 2) V(b - 2) read
      // takes block b + 1
      stage(kh, sK0, 2, b + 2);
      stage(vh, sV0, 3, b + 1);

      // a rescale waits for O += P(b - 1) V(b - 1) on mbar[2] (S(b) finished, so
      // every product issued before it did, O += P(b - 2) V(b - 2) included,
      // and O += P(b) V(b) waits for this block: the completed phases are
      // b - 1 or b, and the parity names b - 1 alone)
      tc_rows_block<T, D>(t_s + lane_off + (uint32_t)((b & 1) * BN), t_o + lane_off, b, key0, jmax, cs, m_ref, l,
                          ok, tc_su32(&mbar[2]), (uint32_t)((b - 1) & 1), args.max_polls, args.status);
      // P written; block b + 2's K and block b's V landed (block b + 1's V,
      // the newest group, may still be in flight); hand the block to the
      // issuing warp without waiting for it
      asm volatile("cp.async.wait_group 1;" ::: "memory");
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      if (b & 1)
        asm volatile("barrier.arrive.aligned 2, %0;" ::"n"(ATT_TC_BLOCK) : "memory");
      else
        asm volatile("barrier.arrive.aligned 1, %0;" ::"n"(ATT_TC_BLOCK) : "memory");
    }
    // the last O += P V (its own barrier: mbar[2]'s phases are not all waited)
    if (nblocks > 0 && !tc_wait(tc_su32(&mbar[3]), 0u, args.max_polls, args.status)) ok = false;
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (!ok) atomicOr(args.status, DEV_TIMEOUT);

  // o = O / l in the input type; LSE = m ln 2 + log l; the empty row: 0, -inf.
  // The TMEM loads are warp-collective, so every row thread loads; rows past
  // the end store nothing.
  const float inv = l > 0.0f ? recip_refined(l) : 0.0f;
  T* orow = o + (head * a.sq + (qi < a.sq ? qi : 0)) * D;
  if (row_thread) {
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
  }
  if (row_thread && qi < a.sq && lse != nullptr)
    lse[head * a.sq + qi] = l > 0.0f ? __fmaf_rn(m_ref, LN2, logf(l)) : neg_inf();
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TCOLS) : "memory");
  }
}

}  // namespace smx
