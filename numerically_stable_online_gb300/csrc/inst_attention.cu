// Kernel instantiations of the attention forward (kernel_attention.cuh).
#include <mutex>
#include <unordered_map>

#include <cudaTypedefs.h>

#include "kernel_attention.cuh"
#include "kernel_attention_tc.cuh"
#include "kernel_attention_tma.cuh"
#include "smx_launch.h"

namespace smx {
namespace {

template <typename T, int D>
cudaError_t launch_attention_t(const AttnCall& c) {
  auto kern = k_attention<T, D>;
  const int64_t smem = (int64_t)(ATT_BM + 4 * ATT_BN) * D * 2;  // Q, K x 2, V x 2
  static std::mutex mu;
  static bool set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!set[dev]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      set[dev] = true;
    }
  }
  AttnArgs a;
  a.sq = c.sq;
  a.sk = c.sk;
  a.heads = c.heads;
  a.scale_log2 = (float)(c.scale * 1.4426950408889634);
  a.causal = c.causal;
  const dim3 grid((unsigned)((c.sq + ATT_BM - 1) / ATT_BM), (unsigned)c.heads);
  note_launch();
  kern<<<grid, ATT_THREADS, (size_t)smem, c.stream>>>(static_cast<const T*>(c.q), static_cast<const T*>(c.k),
                                                      static_cast<const T*>(c.v), static_cast<T*>(c.o), c.lse,
                                                      a);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_attention_tc_t(const AttnCall& c) {
  auto kern = k_attention_tc<T, D>;
  // the operand tiles and 1024 bytes for their alignment and the barriers
  const int64_t smem = (int64_t)att_tc_tile_bytes<D>() + 1024;
  static std::mutex mu;
  static bool set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!set[dev]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      // two CTAs of (D = 128) 113 KiB each need the largest shared-memory carveout
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
      set[dev] = true;
    }
  }
  AttnTcArgs a;
  a.a.sq = c.sq;
  a.a.sk = c.sk;
  a.a.heads = c.heads;
  a.a.scale_log2 = (float)(c.scale * 1.4426950408889634);
  a.a.causal = c.causal;
  a.status = c.status;
  a.max_polls = c.max_polls;
  a.probe_polls = c.probe_polls;
  const dim3 grid((unsigned)((c.sq + ATT_TC_BM - 1) / ATT_TC_BM), (unsigned)c.heads);
  note_launch();
  kern<<<grid, ATT_TC_BLOCK, (size_t)smem, c.stream>>>(static_cast<const T*>(c.q), static_cast<const T*>(c.k),
                                                          static_cast<const T*>(c.v), static_cast<T*>(c.o), c.lse,
                                                          a);
  return cudaGetLastError();
}

// The driver's tensor-map encoder, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [heads][rows][d] 16-bit tensor as a 3-D tensor map read in boxes of 64
// columns x box_rows rows with the 128-byte swizzle; rows past the end read
// as zeros
bool encode_rows_map(CUtensorMap* m, const void* ptr, int64_t heads, int64_t rows, int d, int box_rows,
                     int dtype) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)heads};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)(rows * d * 2)};
  const cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = enc(m, dtype == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                         const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename T, int D, int TILES>
cudaError_t launch_attention_tma_t(const AttnCall& c) {
  using S = AtmShape<TILES>;
  auto kern = k_attention_tma<T, D, TILES>;
  const int smem = S::template smem_bytes<D>();
  static std::mutex mu;
  static bool set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!set[dev]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
      set[dev] = true;
    }
  }
  CUtensorMap mq, mk, mv;
  if (!encode_rows_map(&mq, c.q, c.heads, c.sq, D, ATM_BM, c.dtype) ||
      !encode_rows_map(&mk, c.k, c.heads, c.sk, D, ATM_BN, c.dtype) ||
      !encode_rows_map(&mv, c.v, c.heads, c.sk, D, ATM_BN, c.dtype))
    return cudaErrorInvalidValue;
  AttnTmaArgs a;
  a.a.sq = c.sq;
  a.a.sk = c.sk;
  a.a.heads = c.heads;
  a.a.scale_log2 = (float)(c.scale * 1.4426950408889634);
  a.a.causal = c.causal;
  a.status = c.status;
  a.max_polls = c.max_polls;
  a.probe_polls = c.probe_polls;
  // persistent CTAs: as many as fit at once, each walking items grid-stride
  a.nq = (c.sq + TILES * ATM_BM - 1) / (TILES * ATM_BM);
  a.items = a.nq * c.heads;
  const int64_t resident = (int64_t)(c.sm_count > 0 ? c.sm_count : 1) * S::CTAS_PER_SM;
  const unsigned grid = (unsigned)(a.items < resident ? a.items : resident);
  note_launch();
  kern<<<grid, S::BLOCK, (size_t)smem, c.stream>>>(mq, mk, mv, static_cast<T*>(c.o), c.lse, a);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_attention_tma_tiles(const AttnCall& c) {
  return c.kernel == ATTN_TMA2 ? launch_attention_tma_t<T, D, 2>(c) : launch_attention_tma_t<T, D, 1>(c);
}

}  // namespace

cudaError_t launch_attention(const AttnCall& c) {
  // the tensor-map kernels need keys (their maps cover them) and rows that
  // fit a tensor map's 32-bit coordinates; otherwise the one-tile kernel
  if ((c.kernel == ATTN_TMA1 || c.kernel == ATTN_TMA2) && c.sk > 0 && c.sq < (int64_t(1) << 31) &&
      c.sk < (int64_t(1) << 31)) {
    if (c.dtype == 2)
      return c.d == 64 ? launch_attention_tma_tiles<__nv_bfloat16, 64>(c)
                       : launch_attention_tma_tiles<__nv_bfloat16, 128>(c);
    return c.d == 64 ? launch_attention_tma_tiles<__half, 64>(c) : launch_attention_tma_tiles<__half, 128>(c);
  }
  if (c.kernel != ATTN_MMA_SYNC) {
    if (c.dtype == 2)
      return c.d == 64 ? launch_attention_tc_t<__nv_bfloat16, 64>(c) : launch_attention_tc_t<__nv_bfloat16, 128>(c);
    return c.d == 64 ? launch_attention_tc_t<__half, 64>(c) : launch_attention_tc_t<__half, 128>(c);
  }
  if (c.dtype == 2) {
    return c.d == 64 ? launch_attention_t<__nv_bfloat16, 64>(c) : launch_attention_t<__nv_bfloat16, 128>(c);
  }
  return c.d == 64 ? launch_attention_t<__half, 64>(c) : launch_attention_t<__half, 128>(c);
}

}  // namespace smx

#ifdef SMX_ATM_TRACE
extern "C" int smx_debug_atm_trace(long long* out) {
  return (int)cudaMemcpyFromSymbol(out, smx::g_atm_trace, sizeof(smx::g_atm_trace));
}
#endif
