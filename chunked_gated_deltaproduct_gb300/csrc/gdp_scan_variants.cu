// gdp_scan_variants.cu -- the scan kernels for float16 inputs and output and / or a bfloat16
// dense initial state (FlashInfer page, parameters q, k, v and initial_state): the body of
// gdp_scan_body.cuh with those types.
#include "gdp_scan_body.cuh"

namespace gdp {
namespace {
GDP_SCAN_KERNEL(gdp_scan_kernel_init16, false, true)
GDP_SCAN_KERNEL(gdp_scan_kernel_f16, true, false)
GDP_SCAN_KERNEL(gdp_scan_kernel_f16_init16, true, true)
}  // namespace

cudaError_t launch_scan_variant(const Problem &p, cudaStream_t stream, bool f16, bool init16) {
  if (f16) return launch_scan_kernel(init16 ? gdp_scan_kernel_f16_init16 : gdp_scan_kernel_f16, p, stream);
  return launch_scan_kernel(gdp_scan_kernel_init16, p, stream);
}

}  // namespace gdp
