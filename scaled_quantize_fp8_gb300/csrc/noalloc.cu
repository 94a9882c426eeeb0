// fp8_quantize_static_scratch: fp8_quantize without a caller-provided workspace.
//
// Some callers cannot hand this library a device workspace, for example code embedded in a
// host framework whose allocator owns the whole device memory pool (an extra cudaMalloc
// would fail or fragment it), or latency-critical loops that must never pay for cudaMalloc's
// implicit device synchronisation. For them the tensorwise and delayed recipes reduce their
// amax partials in a fixed scratch array that lives in this library's device image.
#include <mutex>

#include "internal.cuh"

namespace fp8lin {

// Scratch for the amax partials: 65536 x 4 bytes = 256 KiB on every device that loads the
// library, held until the process exits.
constexpr size_t kStaticScratchWords = 65536;
static __device__ __align__(256) uint32_t g_static_scratch[kStaticScratchWords];

namespace {
// The array's device address in the context where it was last looked up, per device. A
// cudaDeviceReset, or a context of the caller's own made current, gives the device a new
// context (with a new id) in which the library image, and the array, may sit elsewhere.
struct ScratchSlot {
  unsigned long long ctx;
  void* ptr;
};
std::mutex g_mu;
ScratchSlot g_slot[kMaxDevices] = {};

// Device address of the scratch array in the current context (looked up once per context).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  if (id != 0 && g_slot[dev].ctx == id) {
    *out = g_slot[dev].ptr;
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess) return e;
  if (id == 0) id = current_context_id();   // the lookup may have made the context current
  g_slot[dev] = ScratchSlot{id, p};          // id 0 (unknown) never matches: looked up again
  *out = p;
  return cudaSuccess;
}
}  // namespace

}  // namespace fp8lin

using namespace fp8lin;

extern "C" fp8_status fp8_quantize_static_scratch(const fp8_recipe* recipe, const void* x_bf16,
                                                  int64_t rows, int64_t cols, int32_t role,
                                                  int32_t want_row, int32_t want_col,
                                                  fp8_tensor* out, int32_t* dev_status,
                                                  cudaStream_t stream) {
  if (recipe == nullptr) return FP8_ERR_NULL;
  const size_t need = quantize_workspace_bytes(recipe->kind, rows, cols);
  if (need > kStaticScratchWords * sizeof(uint32_t)) return FP8_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    const fp8_status st = cuda_status(scratch_address(&scratch));
    if (st != FP8_OK) return st;
  }
  return fp8_quantize(recipe, x_bf16, rows, cols, role, want_row, want_col, out, scratch,
                      need, dev_status, stream);
}
