// Kernel instantiations for f32 inputs (one translation unit per input type).
#include "launch_impl.cuh"

namespace smx {
cudaError_t launch_in_f32(const Call& c, const Plan& p) { return launch_in<float>(c, p); }
int cluster_capacity_f32(int cluster, int64_t smem_bytes) {
  return cluster_capacity<float>(cluster, smem_bytes);
}
int stream_occupancy_f32(int vpt, int threads, int depth, int mode, bool warp) {
  return stream_occupancy<float>(vpt, threads, depth, mode, warp);
}
int split_occupancy_f32(int threads) { return split_occupancy<float>(threads); }
int split_fused_occupancy_f32(int threads) { return split_fused_occupancy<float>(threads); }
int backward_occupancy_f32(int vpt, int threads) {
  return backward_occupancy<float>(vpt, threads);
}
int stripe_occupancy_f32(int64_t smem) { return stripe_occupancy<float>(smem); }
int stripe_static_smem_f32() { return stripe_static_smem<float>(); }
}  // namespace smx

#ifdef SMX_STRIPE_TRACE
// The stripe kernel's wait stamps (build-time diagnostic; see kernel_stripe.cuh).
extern "C" int smx_debug_stripe_trace(void* host, int64_t bytes) {
  const int64_t n = (int64_t)sizeof(smx::g_stripe_trace);
  return cudaMemcpyFromSymbol(host, smx::g_stripe_trace, (size_t)(bytes < n ? bytes : n)) == cudaSuccess ? 0 : 1;
}
#endif
