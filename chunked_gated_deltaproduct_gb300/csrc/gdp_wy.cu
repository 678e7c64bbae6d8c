// gdp_wy.cu -- the prep + WY kernel for bfloat16 q / k / v with fp32 beta and natural-log g;
// the method and the layout are described in gdp_wy_body.cuh.  The kernels for the other input
// types are in gdp_wy_variants.cu.
#include "gdp_wy_body.cuh"

namespace gdp {
namespace {
GDP_WY_KERNEL(gdp_wy_kernel, false, false)
}  // namespace

cudaError_t launch_wy(const Problem &p, cudaStream_t stream) {
  if (p.ntdp_pad == 0) return cudaSuccess;
  const bool typed = (p.beta && p.beta_type != kTypeF32) || (p.g && (p.g_type != kTypeF32 || p.g_alpha));
  if (p.f16 || typed) return launch_wy_variant(p, stream, p.f16 != 0, typed);
  return launch_wy_kernel(gdp_wy_kernel, p, stream);
}

}  // namespace gdp
