// Host-side internals shared by the translation units of libw12.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/w12.h"

namespace w12 {

constexpr int kGroup = 128;            // K elements per exponent group / exception block column
constexpr int kMaxM = 256;             // verified rows per call
constexpr int kMaxProb = 4;            // GEMMs in one grouped launch
constexpr int kOffCap = 1024;          // exception offsets staged in shared memory per CTA
constexpr int kEntCap = 2048;          // exception entries staged in shared memory per CTA
constexpr int kTreeMax = 256;          // nodes per draft tree

// Wall-time bound for every device-side wait (nanoseconds).
uint64_t wait_limit_ns();

// Whether launches may overlap the previous kernel on the stream
// (programmatic dependent launch); on by default.
bool overlap_enabled();

// Number of SMs of the current device (cached per device); 0 if no device.
int device_sm_count();

// True if the current device is an sm_103 part this library was built for.
bool device_supported();

// Unique id of the CUDA context current on this thread (unique for the
// process lifetime, unlike the context handle). False if none is current.
bool current_context_id(unsigned long long* id);

// Encode a 2-D tiled tensor map (inner dimension first). Returns false on failure.
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);

// Encode a 4-D tiled tensor map (dims and box inner first; strides of dims 1..3
// in bytes). Returns false on failure.
bool encode_tmap_4d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, const uint64_t dims[4],
                    const uint64_t strides_bytes[3], const uint32_t box[4], CUtensorMapSwizzle swizzle);

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? W12_OK : W12_ERR_CUDA; }

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

inline int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Stream-K schedule shared by the GEMM launcher and its workspace sizing.
struct GemmShape {
  int M, Mpad, N, K, KB, tiles, grid;
  int64_t units;
};
int gemm_shape(int64_t M, int64_t N, int64_t K, GemmShape* s);

// Workspace carve-up for the GEMM (counters + split-K partial slots) and the
// verify tail (per-tile argmax partials, argmax vector, completion counter).
struct WsLayout {
  size_t counters, parts, amax_val, amax_idx, argmax, done, total;
};
WsLayout ws_layout(const GemmShape& s, int64_t partial_tiles);

// Launchers implemented in the .cu files.
int launch_gemm(bool w12_mode, bool argmax_mode, const uint16_t* X, int64_t M, const w12_weights* W,
                const uint16_t* Wbf16, int64_t N, int64_t K, float* Y, float* amax_val, int32_t* amax_idx,
                void* ws, size_t ws_bytes, int32_t* dev_status, cudaStream_t stream);

int launch_logits_partials(const float* logits, int64_t V, int M, int Mstride, int chunk, float* pv, int32_t* pi,
                           cudaStream_t stream);

int launch_reduce_accept(const float* pv, const int32_t* pi, int nparts, int Mstride, int M, int mode, int B, int T,
                         int T_rows, const int32_t* draft, const int32_t* parents, int32_t* accept_len, int32_t* bonus,
                         int32_t* path, int32_t* path_len, int32_t* argmax_ws, int32_t* argmax_out, int32_t* done,
                         int32_t* dev_status, cudaStream_t stream);

}  // namespace w12
