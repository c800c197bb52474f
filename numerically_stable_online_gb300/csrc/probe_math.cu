// Testing entry point: the library's own exponential and reciprocal
// primitives (smx_device.cuh) evaluated on caller-given arguments, so that
// their error can be measured against fp64 on the host.  The pages warn that
// approximate exponential instructions carry an error of their own ("Stable
// softmax: keep the normalizer consistent as tiles arrive", first paragraph;
// "Online stable softmax", "Masks, empty rows, and precision"); the kernels
// evaluate e^z as 2^(z log2 e) ("Softmax numerics architecture...", "On CPU,
// and the pitfalls worth naming").
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/smx.h"
#include "row_core.cuh"
#include "smx_launch.h"

namespace smx {
namespace {

// which: 0 ex2.approx.ftz (a), 1 ex2.approx (a), 2 rcp.approx.ftz (a), 3 the
// refined reciprocal 1/a, 4 the compensated e^(a - b), 5 the fast e^(a - b)
// as the statistics path forms one term: 2^(fma(a, log2e_hi, RN(-b log2e_hi)))
// times 2^(c_lo) (stats_correct of a one-term sum)
__global__ void __launch_bounds__(256) k_probe_math(const float* __restrict__ a, const float* __restrict__ b,
                                                    float* __restrict__ out, int64_t n, int which) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float u = a[i];
    float r;
    switch (which) {
      case 0: r = ex2_ftz(u); break;
      case 1: r = ex2_full(u); break;
      case 2: asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(u)); break;
      case 3: r = recip_refined(u); break;
      case 4: r = exp_shift_accurate(u, b[i]); break;
      default: {
        const float m = b[i];
        const float c = __fmul_rn(-m, L2E_HI);
        r = stats_correct(ex2_ftz(__fmaf_rn(u, L2E_HI, c)), m);
        break;
      }
    }
    out[i] = r;
  }
}

}  // namespace
}  // namespace smx

extern "C" smx_status smx_debug_probe_math(const float* a, const float* b, float* out, int64_t n, int which,
                                           smx_stream_t stream) {
  if (n < 0 || which < 0 || which > 5) return SMX_ERR_INVALID_ARG;
  if (n == 0) return SMX_OK;
  if (a == nullptr || out == nullptr || ((which == 4 || which == 5) && b == nullptr)) return SMX_ERR_INVALID_ARG;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  smx::k_probe_math<<<(unsigned)blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a, b, out, n, which);
  return cudaGetLastError() == cudaSuccess ? SMX_OK : SMX_ERR_LAUNCH;
}
