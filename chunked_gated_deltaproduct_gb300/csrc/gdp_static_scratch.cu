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
// names a stand-in object).  Each CUDA context loads its own copy of the
// library's device code, so the array has one device address per context: the
// first call made in a context (with that context current) looks the address up
// with cudaGetSymbolAddress and caches it under the context's unique ID (which
// CUDA never reuses within a process, so a context destroyed by
// cudaDeviceReset and its successor never share an entry).  Make the first call
// in each context outside any stream capture.
//
// Nothing in the scratch has to start at zero: every byte a kernel reads was
// written earlier in the same call.  All calls share the one array, so two
// calls whose kernels overlap on the GPU (different streams, or different host
// threads) race on it; serialise them.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gdp_internal.cuh"

#define GDP_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kScratchBytes = GDP_STATIC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char gdp_static_scratch[kScratchBytes];

// Driver calls that name the current context, fetched through the runtime's driver entry
// point so that the library keeps linking against the runtime only.
struct CtxApi {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};
const CtxApi &ctx_api() {
  static CtxApi api;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      api.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      api.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  return api;
}

// The unique ID of the current context; false when none is current or the driver lacks the calls.
bool current_context_id(unsigned long long *id) {
  const CtxApi &api = ctx_api();
  CUcontext ctx = nullptr;
  if (!api.get_current || !api.get_id || api.get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return api.get_id(ctx, id) == CUDA_SUCCESS;
}

constexpr int kCacheEntries = 64;
struct Entry {
  unsigned long long ctx_id;
  void *addr;
};
std::mutex g_mutex;
Entry g_cache[kCacheEntries] = {};
int g_used = 0;

// Device address of the scratch array in the current context.  The lookup also makes the
// device's primary context current when no context is, so the context is named after it.
cudaError_t scratch_address(void **out) {
  unsigned long long id = 0;
  if (current_context_id(&id)) {
    std::lock_guard<std::mutex> lock(g_mutex);
    for (int i = 0; i < g_used; ++i)
      if (g_cache[i].ctx_id == id) {
        *out = g_cache[i].addr;
        return cudaSuccess;
      }
  }
  void *p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, gdp_static_scratch);
  if (e != cudaSuccess) return e;
  if (current_context_id(&id)) {  // cached for this context (looked up on every call once the table is full)
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_used < kCacheEntries) g_cache[g_used++] = Entry{id, p};
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

GDP_EXPORT size_t gdp_static_scratch_bytes(void) { return kScratchBytes; }

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
  void *scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    gdp::set_last_error("cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
    return GDP_ERR_CUDA;
  }
  gdp_prefill_args local = *args;
  local.workspace = scratch;
  local.workspace_bytes = kScratchBytes;
  return gdp_prefill_varlen(&local, stream);
}
