// Kernel instantiations for f16 inputs (one translation unit per input type).
#include "launch_impl.cuh"

namespace smx {
cudaError_t launch_in_f16(const Call& c, const Plan& p) { return launch_in<__half>(c, p); }
int cluster_capacity_f16(int cluster, int64_t smem_bytes) {
  return cluster_capacity<__half>(cluster, smem_bytes);
}
int stream_occupancy_f16(int vpt, int threads, int depth, int mode, bool warp) {
  return stream_occupancy<__half>(vpt, threads, depth, mode, warp);
}
int split_occupancy_f16(int threads) { return split_occupancy<__half>(threads); }
int split_fused_occupancy_f16(int threads) { return split_fused_occupancy<__half>(threads); }
int backward_occupancy_f16(int vpt, int threads) {
  return backward_occupancy<__half>(vpt, threads);
}
int stripe_occupancy_f16(int64_t smem) { return stripe_occupancy<__half>(smem); }
int stripe_static_smem_f16() { return stripe_static_smem<__half>(); }
}  // namespace smx
