// mm_swiglu_ffn_noalloc: the dense SwiGLU FFN for callers that cannot
// allocate device memory (see include/mm.h).  Its scratch is a fixed,
// library-owned device array; everything else is the regular
// mm_swiglu_ffn_ex path.
#include <mutex>

#include "mm_kernels.cuh"

namespace {

// Library-owned scratch: allocated by the CUDA runtime when this library's
// module is loaded on a device and held until the process exits.  Shared by
// every call; it keeps the last call's contents.
constexpr size_t kNoAllocScratchBytes = MM_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The symbol's
// name is only a host-side stand-in; the address comes from the runtime,
// looked up once per device with that device current.
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return MM_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MM_OK;
}

}  // namespace

extern "C" int mm_swiglu_ffn_noalloc(const void* x, const void* Wg, const void* Wu, const void* Wd,
                                     void* y, int64_t T, int H, int I, int dtype, void* stream) {
  if (mm_swiglu_ffn_workspace_bytes(T, H, I, dtype) == 0) return MM_ERR_INVALID_ARG;
  if (T == 0) return MM_OK;
  // the automatic path when its scratch fits, else the tensor-core GEMMs
  int path = MM_PATH_AUTO;
  size_t need = mm::dense_workspace_for_path(T, H, I, dtype, path);
  if (need == 0 || need > kNoAllocScratchBytes) {
    path = MM_PATH_TENSOR;
    need = mm::dense_workspace_for_path(T, H, I, dtype, path);
  }
  if (need == 0 || need > kNoAllocScratchBytes) return MM_ERR_UNSUPPORTED;   // beyond the scratch
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != MM_OK) return rc;
  // The array's first 256 bytes hold the streaming kernels' grid-barrier
  // counters and the watchdog word.  A call whose wait gave up leaves them
  // non-zero, and nobody can read or clear them through mm_check_status, so
  // every call zeroes them first, in order on its own stream (a memset
  // allocates nothing).
  const cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(mm::WsHeader),
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return MM_ERR_CUDA;
  return mm_swiglu_ffn_ex(x, Wg, Wu, Wd, y, T, H, I, dtype, scratch, kNoAllocScratchBytes, stream,
                          path);
}
