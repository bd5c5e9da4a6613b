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
// name as a device address, so on the first call on each device (with that device
// current) the library looks the address up with cudaGetSymbolAddress and keeps it.
// All calls share the one buffer: calls whose work overlaps on the GPU (different
// streams, or different host threads) race on it.  Nothing in it needs to start at
// zero -- each step writes everything the next one reads.
#include <atomic>

#include "oz_internal.h"

namespace oz {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[OZ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices] = {};  // several host threads may call at once

// Device address of the scratch array on the current device (looked up once per device;
// concurrent first calls look up the same address).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return OZ_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return OZ_ENODEV;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return OZ_ECUDA;
    }
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return OZ_OK;
}

}  // namespace
}  // namespace oz

extern "C" int ozaki2_dgemm_noalloc(int m, int n, int k, const double* A, int lda, const double* B, int ldb,
                                    double* C, int ldc, int num_moduli, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 0) return OZ_EINVAL;
  if (lda < (m > 1 ? m : 1) || ldb < (k > 1 ? k : 1) || ldc < (m > 1 ? m : 1)) return OZ_EINVAL;
  if (num_moduli < OZ_MIN_MODULI || num_moduli > OZ_MAX_MODULI) return OZ_EINVAL;
  if (m == 0 || n == 0) return OZ_OK;
  if (k > 0) {
    const size_t need = ozaki2_workspace_bytes(m, n, k, num_moduli);
    if (need == 0 || need > static_cast<size_t>(OZ_NOALLOC_SCRATCH_BYTES)) return OZ_ENOMEM;
  }
  void* scratch = nullptr;
  const int rc = oz::scratch_address(&scratch);
  if (rc != OZ_OK) return rc;
  return ozaki2_dgemm_ws(m, n, k, A, lda, B, ldb, C, ldc, num_moduli, scratch,
                         static_cast<size_t>(OZ_NOALLOC_SCRATCH_BYTES), stream);
}
