// W12 GEMM entry point that allocates nothing.
//
// w12_gemm takes a caller-supplied workspace for its split-K scratch (one
// counter per output tile, two fp32 partial slots per CTA). Some callers
// cannot provide one: code embedded in a host application that owns every
// device allocation and exposes no allocator, and latency-critical loops that
// are not allowed to call cudaMalloc/cudaFree (or a framework allocator) while
// they run. w12_gemm_noalloc serves them from a fixed-size scratch array in
// device memory that this library holds for as long as it is loaded.
#include <mutex>

#include "w12_dev.cuh"
#include "w12_host.h"

namespace w12 {

// Largest shape the fixed scratch serves: M <= 16 rows, at most 4096 output
// tiles of 128 (N <= 524288), at most 192 SMs.
constexpr int kNoAllocMaxM = 16;
constexpr size_t kNoAllocCounterBytes = sizeof(int32_t) * 4096;
constexpr size_t kNoAllocPartBytes = sizeof(float) * 2ull * 192 * 16 * 128;
constexpr size_t kNoAllocBytes = kNoAllocCounterBytes + kNoAllocPartBytes;  // 3,162,112 bytes

// Zero-initialised when the library's module loads on a device; every GPU that
// loads the library holds these bytes until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// Device address of g_noalloc_scratch on the current device. In host code the
// array's name only stands in for the symbol, so the address is looked up
// once per device (with that device current) and cached.
static int noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return W12_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return W12_ERR_CUDA;
    }
    addr[dev] = p;
  }
  *out = addr[dev];
  return W12_OK;
}

}  // namespace w12

using namespace w12;

extern "C" int w12_gemm_noalloc(const uint16_t* X, int64_t M, const w12_weights* W, float* Y, int32_t* dev_status,
                                void* stream) {
  if (!W) return W12_ERR_ARG;
  GemmShape sh;
  int st = gemm_shape(M, W->N, W->K, &sh);
  if (st) return st;
  const WsLayout L = ws_layout(sh, 0);
  if (M > kNoAllocMaxM || L.total > kNoAllocBytes) return W12_ERR_WORKSPACE;  // beyond the fixed scratch
  if (!device_supported()) return W12_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st) return st;
  // The tile counters must start at zero. A successful call leaves them zero,
  // but one that stopped early (an expired wait) may not, so clear them.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(static_cast<uint8_t*>(scratch) + L.counters, 0, sizeof(int32_t) * size_t(sh.tiles), s) !=
      cudaSuccess)
    return W12_ERR_CUDA;
  return launch_gemm(true, false, X, M, W, nullptr, W->N, W->K, Y, nullptr, nullptr, scratch, kNoAllocBytes,
                     dev_status, s);
}
