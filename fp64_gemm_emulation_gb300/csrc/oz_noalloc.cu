// oz_noalloc.cu -- ozaki2_dgemm_noalloc: the Scheme II product without any allocation.
//
// Some callers cannot allocate device memory at the time they multiply: a process whose
// memory manager has already reserved the whole GPU and forbids outside cudaMalloc, or
// code that must not allocate after start-up (a fixed-budget or real-time loop where an
// allocation may block or fail at the worst moment).  This entry point serves them: its
// workspace lives in a fixed array compiled into the library instead of coming from
// cudaMalloc / cudaMallocAsync / the caller.
//
// The array is a file-scope __device__ buffer of OZ_NOALLOC_SCRATCH_BYTES: every GPU that
// loads the library holds it until the process exits.  Host code cannot use the array's
// name as a device address, so the first call on each device (with that device current)
// looks the address up with cudaGetSymbolAddress and keeps it, together with the unique
// id of the CUDA context it belongs to.  A later call in another context (after
// cudaDeviceReset, for instance, the library's module is loaded again and the array may
// sit elsewhere) sees a different id and looks the address up again; where the context id
// cannot be read, every call looks it up.  All calls share the one buffer: calls whose
// work overlaps on the GPU (different streams, or different host threads) race on it.
// Nothing in it needs to start at zero -- each step writes everything the next one reads.
#include <cuda.h>

#include <mutex>

#include "oz_internal.h"

namespace oz {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[OZ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct ScratchEntry {
  unsigned long long ctx_id;  // id of the context the address belongs to (0: none yet)
  void* addr;
};
std::mutex g_scratch_mu;  // several host threads may call at once
ScratchEntry g_scratch[kMaxDevices] = {};

typedef CUresult (*PFN_ctxGetCurrent)(CUcontext*);
typedef CUresult (*PFN_ctxGetId)(CUcontext, unsigned long long*);

template <typename F>
F driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return reinterpret_cast<F>(p);
}

// Unique id of the context current on this thread; false if there is none or the driver
// cannot tell.
bool current_context_id(unsigned long long* id) {
  static const PFN_ctxGetCurrent get_current = driver_fn<PFN_ctxGetCurrent>("cuCtxGetCurrent");
  static const PFN_ctxGetId get_id = driver_fn<PFN_ctxGetId>("cuCtxGetId");
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS && *id != 0;
}

// Device address of the scratch array in the current device's context.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return OZ_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return OZ_ENODEV;
  unsigned long long id = 0;
  if (current_context_id(&id)) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch[dev].addr && g_scratch[dev].ctx_id == id) {
      *out = g_scratch[dev].addr;
      return OZ_OK;
    }
  }
  void* p = nullptr;  // set-up: the lookup also makes the device's context current
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return OZ_ECUDA;
  }
  if (current_context_id(&id)) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    g_scratch[dev].ctx_id = id;
    g_scratch[dev].addr = p;
  }
  *out = p;
  return OZ_OK;
}

}  // namespace
}  // namespace oz

extern "C" int ozaki2_dgemm_noalloc(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                                    double* C, int ldc, int num_moduli, cudaStream_t stream) {
  // the argument checks of ozaki2_dgemm, in its order; the buffer's limit comes last
  if (m < 0 || n < 0 || k < 0) return OZ_EINVAL;
  if (lda < (m > 1 ? m : 1) || ldb < (k > 1 ? k : 1) || ldc < (m > 1 ? m : 1)) return OZ_EINVAL;
  if (num_moduli < OZ_MIN_MODULI || num_moduli > OZ_MAX_MODULI) return OZ_EINVAL;
  if (m == 0 || n == 0) return OZ_OK;
  if (!C) return OZ_EINVAL;
  if (k == 0) return ozaki2_dgemm_ws(m, n, k, A, lda, B, ldb, C, ldc, num_moduli, nullptr, 0, stream);  // C = +0
  if (!A || !B) return OZ_EINVAL;
  {
    int kA;
    const int rc = ozaki2_choose_k(num_moduli, k, &kA);
    if (rc != OZ_OK) return rc;
  }
  const size_t need = ozaki2_workspace_bytes(m, n, k, num_moduli);
  if (need == 0 || need > static_cast<size_t>(OZ_NOALLOC_SCRATCH_BYTES)) return OZ_ENOMEM;
  void* scratch = nullptr;
  const int rc = oz::scratch_address(&scratch);
  if (rc != OZ_OK) return rc;
  return ozaki2_dgemm_ws(m, n, k, A, lda, B, ldb, C, ldc, num_moduli, scratch,
                         static_cast<size_t>(OZ_NOALLOC_SCRATCH_BYTES), stream);
}
