// Kernel instantiations for bf16 inputs (one translation unit per input type).
#include "launch_impl.cuh"

namespace smx {
cudaError_t launch_in_bf16(const Call& c, const Plan& p) { return launch_in<__nv_bfloat16>(c, p); }
int cluster_capacity_bf16(int cluster, int64_t smem_bytes) {
  return cluster_capacity<__nv_bfloat16>(cluster, smem_bytes);
}
int stream_occupancy_bf16(int vpt, int threads, int depth, int mode, bool warp) {
  return stream_occupancy<__nv_bfloat16>(vpt, threads, depth, mode, warp);
}
int split_occupancy_bf16(int threads) { return split_occupancy<__nv_bfloat16>(threads); }
int split_fused_occupancy_bf16(int threads) { return split_fused_occupancy<__nv_bfloat16>(threads); }
int backward_occupancy_bf16(int vpt, int threads) {
  return backward_occupancy<__nv_bfloat16>(vpt, threads);
}
int stripe_occupancy_bf16(int64_t smem) { return stripe_occupancy<__nv_bfloat16>(smem); }
int stripe_static_smem_bf16() { return stripe_static_smem<__nv_bfloat16>(); }
}  // namespace smx
