// gdp_scan.cu -- the inter-chunk state scan and output kernel for bfloat16 inputs and an
// fp32 (or no) initial state; the method, the data layout and the roles of the warps are
// described in gdp_scan_body.cuh.  The kernels for float16 inputs or a bfloat16 initial
// state are in gdp_scan_variants.cu.
#include "gdp_scan_body.cuh"

namespace gdp {
namespace {
GDP_SCAN_KERNEL(gdp_scan_kernel, false, false)
}  // namespace

cudaError_t launch_scan(const Problem &p, cudaStream_t stream) {
  if (p.N == 0) return cudaSuccess;
  const bool init16 = p.init && p.init_bf16 && !p.cache;
  if (p.f16 || init16) return launch_scan_variant(p, stream, p.f16 != 0, init16);
  return launch_scan_kernel(gdp_scan_kernel, p, stream);
}

}  // namespace gdp
