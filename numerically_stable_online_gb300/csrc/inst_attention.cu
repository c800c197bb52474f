// Kernel instantiations of the attention forward (kernel_attention.cuh).
#include <mutex>
#include <unordered_map>

#include "kernel_attention.cuh"
#include "kernel_attention_tc.cuh"
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

}  // namespace

cudaError_t launch_attention(const AttnCall& c) {
  if (c.tensor_memory) {
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
