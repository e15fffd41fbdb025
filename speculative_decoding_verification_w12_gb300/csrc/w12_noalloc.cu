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

// Device address of g_noalloc_scratch in the current CUDA context. In host
// code the array's name only stands in for the symbol, so the address is
// looked up once per context (with that context current) and cached under the
// context's unique id: a context created later (cuCtxCreate, or a primary
// context re-created after cudaDeviceReset) gets its own lookup, never a stale
// address from another context.
static int noalloc_scratch(void** out) {
  struct Entry {
    unsigned long long ctx;
    void* addr;
  };
  constexpr int kSlots = 64;
  static std::mutex mu;
  static Entry cache[kSlots];
  static int used = 0, next = 0;
  unsigned long long id = 0;
  bool have_id = current_context_id(&id);
  std::lock_guard<std::mutex> lock(mu);
  if (have_id)
    for (int i = 0; i < used; ++i)
      if (cache[i].ctx == id) {
        *out = cache[i].addr;
        return W12_OK;
      }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return W12_ERR_CUDA;
  }
  if (!have_id) have_id = current_context_id(&id);  // the lookup made the primary context current
  if (have_id) {
    const int slot = used < kSlots ? used++ : (next++ % kSlots);
    cache[slot] = Entry{id, p};
  }
  *out = p;
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
