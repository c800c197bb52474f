// Attention forward with the online weighted numerator: the pages' running
// state (m, l, o) ("Online stable softmax", sections "Carry a weighted value
// numerator for attention" and "Reference summary"; "Softmax numerics
// architecture...", "From online softmax to tiled attention"):
//   for each key block B:  m' = max(m, max S_B),  l' = e^(m - m') l + sum e^(S_B - m'),
//                          o' = e^(m - m') o + e^(S_B - m') V_B;   finally o / l,
// with S = scale Q K^T.  The score and probability matrices never leave the
// chip.
//
// One CTA of 4 warps takes 64 query rows of one head; each warp holds 16 rows.
// Key/value blocks of 64 rows are double-buffered into shared memory with
// cp.async (16-byte chunks, XOR-swizzled by row so that ldmatrix reads are
// free of bank conflicts).  Both products run on the tensor cores with
// mma.sync m16n8k16 (16-bit inputs, fp32 accumulation): S_B = Q K_B^T from
// ldmatrix fragments, P = e^(S_B - m') rounded to the input type and reused in
// registers as the A operand of O += P V_B (V read with ldmatrix.trans).  The
// exponent is one FFMA: 2^(s log2(e) scale - m'), m' kept in that scaled base-2
// unit.  Masked scores (causal, key tails) are -inf before the maximum; a row
// with no valid key is the declared empty row: o = 0, LSE = -inf.
#pragma once

#include "smx_device.cuh"

namespace smx {

constexpr int ATT_BM = 64;       // query rows per CTA (4 warps x 16)
constexpr int ATT_BN = 64;       // keys per block
constexpr int ATT_THREADS = 128;

struct AttnArgs {
  int64_t sq, sk;   // query / key rows per head
  int64_t heads;    // batch x heads
  float scale_log2; // scale * log2(e)
  int causal;       // 1: key j valid for query i when j <= i + sk - sq
};

__device__ __forceinline__ void att_cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// byte offset of 16-byte chunk c of row r in a [rows][D] tile (D / 8 chunks a row)
template <int D>
__device__ __forceinline__ uint32_t att_off(int r, int c) {
  return (uint32_t)(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <typename T>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<__half>(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                 uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <typename T, int D>
__global__ void __launch_bounds__(ATT_THREADS, 2)
    k_attention(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                T* __restrict__ o, float* __restrict__ lse, AttnArgs a) {
  constexpr int CH = D / 8;                 // 16-byte chunks per row
  constexpr int TILE = ATT_BN * D * 2;      // bytes of one K or V block
  extern __shared__ __align__(128) uint8_t smem[];  // Q [64][D], K[2], V[2]
  const uint32_t s_base = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  const uint32_t sQ = s_base, sK = sQ + ATT_BM * D * 2, sV = sK + 2 * TILE;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t head = blockIdx.y;
  const int64_t q0 = (int64_t)blockIdx.x * ATT_BM;
  const T* qh = q + head * a.sq * D;
  const T* kh = k + head * a.sk * D;
  const T* vh = v + head * a.sk * D;

  // keys this block can see: all, or up to the causal limit of its last row
  int64_t kv_end = a.sk;
  if (a.causal) {
    const int64_t last = q0 + ATT_BM - 1 < a.sq - 1 ? q0 + ATT_BM - 1 : a.sq - 1;
    kv_end = last + a.sk - a.sq + 1;
    if (kv_end > a.sk) kv_end = a.sk;
    if (kv_end < 0) kv_end = 0;
  }
  const int nblocks = (int)((kv_end + ATT_BN - 1) / ATT_BN);

  // rows of a 64 x D tile into shared memory: rows past `valid` are zeroed
  auto load_tile = [&](uint32_t dst, const T* src, int64_t row0, int64_t valid) {
    for (int i = tid; i < ATT_BM * CH; i += ATT_THREADS) {
      const int r = i / CH, c = i % CH;
      const uint32_t d = dst + att_off<D>(r, c);
      if (row0 + r < valid) {
        att_cp16(d, src + (row0 + r) * D + c * 8);
      } else {
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(d), "r"(0) : "memory");
      }
    }
  };

  load_tile(sQ, qh, q0, a.sq);
  if (nblocks > 0) {
    load_tile(sK, kh, 0, a.sk);
    load_tile(sV, vh, 0, a.sk);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");

  // this thread's two rows of the warp's 16, in the CTA's 64 and in the head
  const int r_lo = warp * 16 + (lane >> 2), r_hi = r_lo + 8;
  const int64_t qi_lo = q0 + r_lo, qi_hi = q0 + r_hi;
  // causal limit per row (keys j <= lim are valid)
  const int64_t lim_lo = a.causal ? qi_lo + a.sk - a.sq : a.sk - 1;
  const int64_t lim_hi = a.causal ? qi_hi + a.sk - a.sq : a.sk - 1;

  float m_lo = neg_inf(), m_hi = neg_inf(), l_lo = 0.0f, l_hi = 0.0f;
  float acc_o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc_o[n][i] = 0.0f;
  uint32_t qf[D / 16][4];

  for (int b = 0; b < nblocks; ++b) {
    const int stage = b & 1;
    // the next block into the other stage, then wait for this one
    if (b + 1 < nblocks) {
      load_tile(sK + (stage ^ 1) * TILE, kh, (int64_t)(b + 1) * ATT_BN, a.sk);
      load_tile(sV + (stage ^ 1) * TILE, vh, (int64_t)(b + 1) * ATT_BN, a.sk);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncthreads();
    if (b == 0) {
      // Q fragments once: rows warp*16 + (lane % 16), chunk 2 kk + lane / 16
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        ldsm_x4(sQ + att_off<D>(warp * 16 + (lane & 15), 2 * kk + (lane >> 4)), qf[kk][0], qf[kk][1],
                qf[kk][2], qf[kk][3]);
    }
    const uint32_t kb = sK + stage * TILE, vb = sV + stage * TILE;

    // S = Q K^T for 16 rows x 64 keys: 8 n-tiles of 8 keys
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) s[n][i] = 0.0f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {  // two n-tiles per ldmatrix.x4
        const int mi = lane >> 3;
        const int key = np * 16 + (lane & 7) + (mi >> 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + att_off<D>(key, 2 * kk + (mi & 1)), b0, b1, b2, b3);
        mma16816<T>(s[2 * np], qf[kk], b0, b1);
        mma16816<T>(s[2 * np + 1], qf[kk], b2, b3);
      }
    }

    // mask, then the running state of this thread's two rows
    const int64_t key0 = (int64_t)b * ATT_BN;
    float mx_lo = neg_inf(), mx_hi = neg_inf();
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int64_t j = key0 + n * 8 + (lane & 3) * 2 + i;
        if (j > lim_lo || j >= a.sk) s[n][i] = neg_inf();
        if (j > lim_hi || j >= a.sk) s[n][2 + i] = neg_inf();
        mx_lo = fmaxf(mx_lo, s[n][i]);
        mx_hi = fmaxf(mx_hi, s[n][2 + i]);
      }
    }
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
    // m' = max(m, max S_B) in the scaled base-2 unit; the empty prefix (-inf)
    // gets the factor 0 selected, never -inf - (-inf)
    const float mn_lo = fmaxf(m_lo, mx_lo * a.scale_log2), mn_hi = fmaxf(m_hi, mx_hi * a.scale_log2);
    const float al_lo = m_lo == neg_inf() ? 0.0f : ex2_full(m_lo - mn_lo);
    const float al_hi = m_hi == neg_inf() ? 0.0f : ex2_full(m_hi - mn_hi);
    const float sub_lo = mn_lo == neg_inf() ? 0.0f : mn_lo, sub_hi = mn_hi == neg_inf() ? 0.0f : mn_hi;
    float ps_lo = 0.0f, ps_hi = 0.0f;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        s[n][i] = ex2_full(__fmaf_rn(s[n][i], a.scale_log2, -sub_lo));
        s[n][2 + i] = ex2_full(__fmaf_rn(s[n][2 + i], a.scale_log2, -sub_hi));
        ps_lo += s[n][i];
        ps_hi += s[n][2 + i];
      }
    }
    l_lo = __fmaf_rn(l_lo, al_lo, ps_lo);  // the row sum is finished after the loop
    l_hi = __fmaf_rn(l_hi, al_hi, ps_hi);
    m_lo = mn_lo;
    m_hi = mn_hi;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      acc_o[n][0] *= al_lo;
      acc_o[n][1] *= al_lo;
      acc_o[n][2] *= al_hi;
      acc_o[n][3] *= al_hi;
    }
    // O += P V: P from the score registers (4 k-steps of 16 keys)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack2<T>(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack2<T>(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack2<T>(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack2<T>(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {  // two d n-tiles per ldmatrix.x4.trans
        const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + att_off<D>(key, 2 * np + (lane >> 4)), b0, b1, b2, b3);
        mma16816<T>(acc_o[2 * np], pa, b0, b1);
        mma16816<T>(acc_o[2 * np + 1], pa, b2, b3);
      }
    }
    __syncthreads();  // this stage is refilled two blocks on
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");

  // l over the row's four threads, then o / l and LSE = m ln 2 + log l
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
  const float inv_lo = l_lo > 0.0f ? recip_refined(l_lo) : 0.0f;
  const float inv_hi = l_hi > 0.0f ? recip_refined(l_hi) : 0.0f;
  T* oh = o + head * a.sq * D;
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    const int col = n * 8 + (lane & 3) * 2;
    if (qi_lo < a.sq)
      *reinterpret_cast<uint32_t*>(oh + qi_lo * D + col) =
          pack2<T>(acc_o[n][0] * inv_lo, acc_o[n][1] * inv_lo);
    if (qi_hi < a.sq)
      *reinterpret_cast<uint32_t*>(oh + qi_hi * D + col) =
          pack2<T>(acc_o[n][2] * inv_hi, acc_o[n][3] * inv_hi);
  }
  if ((lane & 3) == 0 && lse != nullptr) {
    if (qi_lo < a.sq)
      lse[head * a.sq + qi_lo] = l_lo > 0.0f ? __fmaf_rn(m_lo, LN2, logf(l_lo)) : neg_inf();
    if (qi_hi < a.sq)
      lse[head * a.sq + qi_hi] = l_hi > 0.0f ? __fmaf_rn(m_hi, LN2, logf(l_hi)) : neg_inf();
  }
}

}  // namespace smx
