// gdp_static_scratch.cu -- gdp_prefill_varlen_static_scratch: the prefill for
// callers that cannot allocate device memory.
//
// Some callers have no way to provide the caller-owned workspace the main
// entry point asks for: a plugin running inside another runtime that owns all
// device memory through its own pool, or a C host program with no caching
// allocator that must not call cudaMalloc in its serving loop (cudaMalloc can
// synchronise the device and stall every other stream).  This entry point
// takes the same arguments but ignores args->workspace / workspace_bytes and
// uses a scratch array that lives in the library itself: a file-scope
// __device__ array of GDP_STATIC_SCRATCH_BYTES bytes, which every GPU that
// loads the library keeps for the life of the process.
//
// Host code cannot use the array's name as a device address (on the host it
// names a stand-in object), so the device address is looked up once per device
// with cudaGetSymbolAddress, with that device current, on the first call made
// on that device, and cached.  Make that first call outside any stream capture.
//
// Nothing in the scratch has to start at zero: every byte a kernel reads was
// written earlier in the same call.  All calls share the one array, so two
// calls whose kernels overlap on the GPU (different streams, or different host
// threads) race on it; serialise them.
#include <mutex>

#include "gdp_internal.cuh"

#define GDP_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kScratchBytes = GDP_STATIC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char gdp_static_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(int dev, void **out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, gdp_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

GDP_EXPORT gdp_status gdp_prefill_varlen_static_scratch(const gdp_prefill_args *args, void *stream) {
  if (!args) {
    gdp::set_last_error("args is NULL");
    return GDP_ERR_INVALID_ARG;
  }
  const size_t need = gdp_prefill_workspace_bytes(args->T, args->N, args->H, args->K, args->V,
                                                  args->num_householder);
  if (need == 0) {
    gdp::set_last_error("bad shape T=%lld N=%lld H=%d K=%d V=%d M=%d", (long long)args->T, (long long)args->N,
                        args->H, args->K, args->V, args->num_householder);
    return GDP_ERR_INVALID_ARG;
  }
  if (need > kScratchBytes) {
    gdp::set_last_error("this shape needs %zu bytes of scratch, more than the %zu-byte static scratch of "
                        "gdp_prefill_varlen_static_scratch; use gdp_prefill_varlen with a caller workspace",
                        need, kScratchBytes);
    return GDP_ERR_WORKSPACE;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    gdp::set_last_error("cudaGetDevice: %s", e != cudaSuccess ? cudaGetErrorString(e) : "device index too large");
    return GDP_ERR_CUDA;
  }
  void *scratch = nullptr;
  e = scratch_address(dev, &scratch);
  if (e != cudaSuccess) {
    gdp::set_last_error("cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
    return GDP_ERR_CUDA;
  }
  gdp_prefill_args local = *args;
  local.workspace = scratch;
  local.workspace_bytes = kScratchBytes;
  return gdp_prefill_varlen(&local, stream);
}
