// Shared host code of libw12.so: status strings, device queries, tensor-map
// encoding, workspace layout, the wait bound and the timeout self-test.
#include <atomic>
#include <cstring>
#include <mutex>

#include "w12_dev.cuh"
#include "w12_host.h"

namespace w12 {

static std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

static std::atomic<int> g_overlap{1};

bool overlap_enabled() { return g_overlap.load(std::memory_order_relaxed) != 0; }

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cache[dev] = n;
  }
  return cache[dev];
}

bool device_supported() {
  static int cache[64] = {0};  // 0 unknown, 1 yes, 2 no
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev] == 1;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  const bool ok = major == 10 && minor == 3;
  if (dev >= 0 && dev < 64) cache[dev] = ok ? 1 : 2;
  return ok;
}

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    else
      cudaGetLastError();
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    else
      cudaGetLastError();
  });
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
    } else {
      cudaGetLastError();
    }
  });
  return fn;
}

// A tensor map depends only on these fields (the address, not the data), so
// encoded maps are cached: repeated calls on the same buffers skip the driver.
struct TmapKey {
  int dtype, swizzle;
  void* base;
  uint64_t inner, outer, stride;
  uint32_t box_inner, box_outer;
  bool operator==(const TmapKey& o) const {
    return dtype == o.dtype && swizzle == o.swizzle && base == o.base && inner == o.inner && outer == o.outer &&
           stride == o.stride && box_inner == o.box_inner && box_outer == o.box_outer;
  }
};

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  constexpr int kSlots = 512;
  static std::mutex mu;
  static TmapKey keys[kSlots];
  static CUtensorMap maps[kSlots];
  static bool used[kSlots] = {false};
  const TmapKey key{int(dtype), int(swizzle), base, inner, outer, row_stride_bytes, box_inner, box_outer};
  const uint64_t h = (reinterpret_cast<uint64_t>(base) >> 8) ^ (inner * 0x9E3779B97F4A7C15ull) ^ (outer << 7) ^
                     (uint64_t(box_outer) << 17) ^ uint64_t(dtype) ^ (uint64_t(swizzle) << 3);
  const int slot = int(h % kSlots);
  {
    std::lock_guard<std::mutex> lock(mu);
    if (used[slot] && keys[slot] == key) {
      *map = maps[slot];
      return true;
    }
  }
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dtype, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lock(mu);
  keys[slot] = key;
  maps[slot] = *map;
  used[slot] = true;
  return true;
}

bool encode_tmap_4d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, const uint64_t dims[4],
                    const uint64_t strides_bytes[3], const uint32_t box[4], CUtensorMapSwizzle swizzle) {
  constexpr int kSlots = 64;
  struct Key {
    int dtype, swizzle;
    void* base;
    uint64_t dims[4], strides[3];
    uint32_t box[4];
  };
  static std::mutex mu;
  static Key keys[kSlots];
  static CUtensorMap maps[kSlots];
  static bool used[kSlots] = {false};
  Key key{};
  key.dtype = int(dtype);
  key.swizzle = int(swizzle);
  key.base = base;
  for (int i = 0; i < 4; ++i) key.dims[i] = dims[i], key.box[i] = box[i];
  for (int i = 0; i < 3; ++i) key.strides[i] = strides_bytes[i];
  auto same = [](const Key& a, const Key& b) { return std::memcmp(&a, &b, sizeof(Key)) == 0; };
  uint64_t h = (reinterpret_cast<uint64_t>(base) >> 8) ^ uint64_t(dtype) ^ (uint64_t(swizzle) << 3);
  for (int i = 0; i < 4; ++i) h = h * 0x9E3779B97F4A7C15ull + dims[i] + (uint64_t(box[i]) << 40);
  const int slot = int(h % kSlots);
  {
    std::lock_guard<std::mutex> lock(mu);
    if (used[slot] && same(keys[slot], key)) {
      *map = maps[slot];
      return true;
    }
  }
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t st[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
  cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, dtype, 4, base, d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lock(mu);
  keys[slot] = key;
  maps[slot] = *map;
  used[slot] = true;
  return true;
}

int gemm_shape(int64_t M, int64_t N, int64_t K, GemmShape* s) {
  if (M < 1 || M > kMaxM || N < kGroup || K < kGroup || N % kGroup || K % kGroup) return W12_ERR_SHAPE;
  if (N > (int64_t(1) << 30) || K > (int64_t(1) << 30)) return W12_ERR_SHAPE;
  s->M = static_cast<int>(M);
  s->Mpad = static_cast<int>(round_up(M, 16));
  s->N = static_cast<int>(N);
  s->K = static_cast<int>(K);
  s->KB = static_cast<int>(K / kGroup);
  s->tiles = static_cast<int>(N / kGroup);
  s->units = int64_t(s->tiles) * s->KB;
  int sms = device_sm_count();
  if (sms <= 0) sms = 256;  // sizing without a device: an upper bound
  s->grid = static_cast<int>(s->units < sms ? s->units : sms);
  return W12_OK;
}

WsLayout ws_layout(const GemmShape& s, int64_t partial_tiles) {
  WsLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off += static_cast<size_t>(round_up(static_cast<int64_t>(bytes), 256));
    return at;
  };
  L.counters = take(sizeof(int32_t) * s.tiles);
  L.parts = take(sizeof(float) * size_t(2) * s.grid * s.Mpad * kGroup);
  L.amax_val = take(sizeof(float) * size_t(partial_tiles) * s.Mpad);
  L.amax_idx = take(sizeof(int32_t) * size_t(partial_tiles) * s.Mpad);
  L.argmax = take(sizeof(int32_t) * s.Mpad);
  L.done = take(sizeof(int32_t) * 4);
  L.total = off;
  return L;
}

// ---------------------------------------------------------------------------
// Timeout self-test: a barrier that nothing ever arrives at.
// ---------------------------------------------------------------------------

__global__ void selftest_timeout_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  cta_sync();
  if (threadIdx.x == 0) {
    if (!mbar_wait(&bar, 0, limit_ns)) set_status(status, W12_ERR_TIMEOUT);
  }
  cta_sync();
}

// ---------------------------------------------------------------------------
// Copy kernel for the host path of a step: inputs from page-locked host memory
// into device buffers, results back. As a kernel (not a copy-engine transfer)
// it takes part in launch overlap: it lets the next kernel on the stream start
// at once (a GEMM then requests its first weight tiles while the inputs are
// still arriving) and waits for the previous kernel before it reads or writes.
// ---------------------------------------------------------------------------

constexpr int kCopyThreads = 256;
constexpr int kCopyBlocks = 16;  // few CTAs: the next GEMM needs whole SMs for its own CTAs

__global__ void __launch_bounds__(kCopyThreads) copy_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                            int64_t n16, uint8_t* __restrict__ dtail,
                                                            const uint8_t* __restrict__ stail, int tail) {
  grid_dep_launch();
  grid_dep_wait();
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  // Four 16-byte loads in flight per thread before the stores. Loads skip
  // the caches (the source may be host memory the CPU rewrote since the last
  // launch) and stores write through (the destination may be host memory).
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = __ldcv(src + i), b = __ldcv(src + i + stride), c = __ldcv(src + i + 2 * stride),
                d = __ldcv(src + i + 3 * stride);
    __stwt(dst + i, a);
    __stwt(dst + i + stride, b);
    __stwt(dst + i + 2 * stride, c);
    __stwt(dst + i + 3 * stride, d);
  }
  for (; i < n16; i += stride) __stwt(dst + i, __ldcv(src + i));
  if (blockIdx.x == 0 && int(threadIdx.x) < tail) {
    const uint8_t v = *reinterpret_cast<const volatile uint8_t*>(stail + threadIdx.x);
    *reinterpret_cast<volatile uint8_t*>(dtail + threadIdx.x) = v;
  }
}

// Device address of p (device, managed or page-locked host memory), or null.
static const void* device_address(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return p;
  if (a.type == cudaMemoryTypeHost) return a.devicePointer;
  return nullptr;
}

}  // namespace w12

using namespace w12;

extern "C" {

const char* w12_status_string(int status) {
  switch (status) {
    case W12_OK: return "ok";
    case W12_ERR_ARG: return "invalid argument";
    case W12_ERR_SHAPE: return "unsupported shape (N, K multiples of 128; 1 <= M <= 256)";
    case W12_ERR_WORKSPACE: return "workspace or exception capacity too small";
    case W12_ERR_BAD_TREE: return "malformed draft tree (parents[0] != -1 or parents[i] not in [0, i))";
    case W12_ERR_CORRUPT: return "packed weights failed a consistency check";
    case W12_ERR_TIMEOUT: return "a device-side bounded wait expired";
    case W12_ERR_CUDA: return "CUDA runtime error";
    case W12_ERR_UNSUPPORTED: return "unsupported device or feature (needs an sm_103a GPU)";
    default: return "unknown status";
  }
}

int w12_version(void) { return 200; }

int w12_set_wait_limit_us(int64_t limit_us) {
  if (limit_us < 1) return W12_ERR_ARG;
  g_wait_limit_ns.store(static_cast<uint64_t>(limit_us) * 1000ull, std::memory_order_relaxed);
  return W12_OK;
}

int w12_set_overlap(int enable) {
  g_overlap.store(enable ? 1 : 0, std::memory_order_relaxed);
  return W12_OK;
}

int w12_selftest_timeout(int32_t* dev_status, int limit_us, void* stream) {
  if (!dev_status || limit_us < 1) return W12_ERR_ARG;
  if (!device_supported()) return W12_ERR_UNSUPPORTED;
  selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_status,
                                                                           uint64_t(limit_us) * 1000ull);
  return cuda_status(cudaGetLastError());
}

int w12_copy(void* dst, const void* src, size_t bytes, void* stream) {
  if (!dst || !src || !aligned(dst, 16) || !aligned(src, 16)) return W12_ERR_ARG;
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
  if (bytes > 0 && s0 < d0 + bytes && d0 < s0 + bytes) return W12_ERR_ARG;  // overlapping
  if (!device_supported()) return W12_ERR_UNSUPPORTED;
  if (bytes == 0) return W12_OK;
  void* dd = const_cast<void*>(device_address(dst));
  const void* sd = device_address(src);
  if (!dd || !sd) return W12_ERR_ARG;
  const int64_t n16 = int64_t(bytes / 16);
  const int tail = int(bytes % 16);
  int64_t blocks = (n16 + kCopyThreads - 1) / kCopyThreads;
  blocks = blocks < 1 ? 1 : (blocks > kCopyBlocks ? kCopyBlocks : blocks);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(blocks));
  cfg.blockDim = dim3(unsigned(kCopyThreads));
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_enabled() ? 1 : 0;
  uint8_t* dt = static_cast<uint8_t*>(dd) + n16 * 16;
  const uint8_t* st = static_cast<const uint8_t*>(sd) + n16 * 16;
  return cuda_status(cudaLaunchKernelEx(&cfg, copy_kernel, static_cast<uint4*>(dd), static_cast<const uint4*>(sd),
                                        n16, dt, st, tail));
}

size_t w12_gemm_ws_bytes(int64_t M, int64_t N, int64_t K) {
  GemmShape s;
  if (gemm_shape(M, N, K, &s) != W12_OK) return 0;
  return ws_layout(s, 0).total;
}

size_t w12_verify_ws_bytes(int64_t M, int64_t V) {
  // The fused head needs the GEMM slots at K >= 128 and per-tile partials;
  // the logits path needs per-chunk partials. Size for the larger of both.
  GemmShape s;
  int64_t Vr = round_up(V < kGroup ? kGroup : V, kGroup);
  if (gemm_shape(M, Vr, kGroup, &s) != W12_OK) return 0;
  int sms = device_sm_count();
  s.grid = sms > 0 ? sms : 256;  // the fused head runs one CTA per SM
  int64_t parts = s.tiles;
  return ws_layout(s, parts).total;
}

}  // extern "C"
