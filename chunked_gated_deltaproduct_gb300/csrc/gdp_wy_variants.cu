// gdp_wy_variants.cu -- the prep + WY kernels for float16 q / k / v and / or 16-bit or
// linear-space gates (FlashInfer page, parameters q, k, v, g, beta): the body of
// gdp_wy_body.cuh with those types.
#include "gdp_wy_body.cuh"

namespace gdp {
namespace {
GDP_WY_KERNEL(gdp_wy_kernel_typed, false, true)
GDP_WY_KERNEL(gdp_wy_kernel_f16, true, false)
GDP_WY_KERNEL(gdp_wy_kernel_f16_typed, true, true)
}  // namespace

cudaError_t launch_wy_variant(const Problem &p, cudaStream_t stream, bool f16, bool typed) {
  if (f16) return launch_wy_kernel(typed ? gdp_wy_kernel_f16_typed : gdp_wy_kernel_f16, p, stream);
  return launch_wy_kernel(gdp_wy_kernel_typed, p, stream);
}

}  // namespace gdp
