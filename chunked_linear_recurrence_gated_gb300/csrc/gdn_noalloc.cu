// gdn_chunk_fwd_noalloc: the chunk forward with its scratch memory in a
// fixed, library-owned device array instead of a caller-provided workspace.
//
// Some callers cannot hand the library a workspace: they run inside a host
// framework that owns all device memory and exposes no allocator, or they must
// never trigger a device allocation (which can synchronise the device) while
// they run. This entry point serves them. Its scratch is one file-scope
// __device__ array of GDN_NOALLOC_SCRATCH_BYTES that every GPU which loads the
// library keeps until the process exits; the caller still passes every input
// and output buffer. The array's first word is the status word the kernels
// record device-side conditions in; gdn_noalloc_status reads it.
#include <cuda.h>

#include <mutex>

#include "../../include/gdn.h"
#include "../../include/gdn_profile.h"

namespace {

// Device-resident scratch shared by every call on a device.
static __device__ __align__(256) unsigned char g_scratch[GDN_NOALLOC_SCRATCH_BYTES];

// The host-side name g_scratch is only a stand-in: kernels must be given the
// device address, which is looked up with the device current. The address
// belongs to the device's context: after cudaDeviceReset the module is loaded
// again into a new context, so the cache is keyed on (device, context).
constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Entry {
  void* ctx;
  void* ptr;
};
Entry g_cache[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The current context of the calling thread (nullptr if none is current yet
// or the CUDA driver-API entry point is unavailable).
void* current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (CtxGetCurrentFn)f;
    looked_up = true;
  }
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return (void*)c;
}

gdn_status scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  void* ctx = current_context();
  Entry& e = g_cache[dev];
  if (!e.ptr || !ctx || e.ctx != ctx) {
    // (also makes the device's primary context current if none was)
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
    e.ptr = p;
    e.ctx = current_context();
  }
  *out = e.ptr;
  return GDN_OK;
}

}  // namespace

namespace gdn {
gdn_status chunk_fwd_unsplit(const gdn_shape* shape, const void* q, const void* k, const void* v,
                             const void* g, const void* beta, const float* S_in, void* o,
                             float* S_out, void* workspace, size_t workspace_bytes, void* stream);
}

extern "C" gdn_status gdn_chunk_fwd_noalloc(const gdn_shape* shape, const void* q, const void* k,
                                            const void* v, const void* g, const void* beta,
                                            const float* S_in, void* o, float* S_out,
                                            void* stream) {
  const size_t need = gdn_chunk_workspace_bytes(shape, 0);
  if (need == 0)  // invalid or unsupported shape: report it exactly as gdn_chunk_fwd does
    return gdn_chunk_fwd(shape, q, k, v, g, beta, S_in, o, S_out, nullptr, 0, stream);
  if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_WORKSPACE;
  void* scratch = nullptr;
  const gdn_status s = scratch_for_current_device(&scratch);
  if (s != GDN_OK) return s;
  return gdn::chunk_fwd_unsplit(shape, q, k, v, g, beta, S_in, o, S_out, scratch,
                                (size_t)GDN_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" gdn_status gdn_noalloc_status(void* stream) {
  void* scratch = nullptr;
  const gdn_status s = scratch_for_current_device(&scratch);
  if (s != GDN_OK) return s;
  return gdn_workspace_status(scratch, stream);
}

extern "C" int gdn_diag_wait_timeout_noalloc(int limit_log2, void* stream) {
  void* scratch = nullptr;
  const gdn_status s = scratch_for_current_device(&scratch);
  if (s != GDN_OK) return s;
  return gdn_diag_wait_timeout(scratch, limit_log2, stream);
}
