// Commit of the accepted path after verification.
//
// The verify pass writes a key/value row for every draft node: node i of
// request b at position prefix_len[b] + i of each cache. Once acceptance has
// chosen the path root -> ... -> node (root first, node indices strictly
// increasing, because a parent's index is below its child's), the path's rows
// must sit contiguously after the committed prefix before the next step; a
// target with recurrent layers keeps the state of the path's last node
// (SpecPilot paper digest, "Reasons" bullet 2: tree verification for targets
// with recurrent layers; JetSpec article, "Technical architecture": every
// draft token is conditioned on its root-to-node path).
//
// kv_commit_kernel: one thread per 16-byte column of a cache row, for one
// request of one cache. Each thread moves its column of rows prefix+path[k]
// to prefix+k in increasing k. Since path[k] >= k, the row a step reads is
// never one an earlier step wrote, and no other thread touches the column,
// so the move is in place without barriers. A request whose path is invalid
// is left unchanged and flagged.
#include "w12_dev.cuh"
#include "w12_host.h"

namespace w12 {

constexpr int kCommitThreads = 128;
constexpr int kMaxCaches = 64;  // caches per launch (more are done in several launches)

struct CommitParams {
  uint8_t* caches[kMaxCaches];
  int n_caches, B, path_stride, flag_new_len;
  int64_t S_max, row_bytes;
  const int32_t* prefix_len;
  const int32_t* path;
  const int32_t* path_len;
  int32_t* new_len;
  int32_t* status;
};

// Validity of request b's path (every thread of the request evaluates it).
__device__ __forceinline__ bool path_ok(const int32_t* pb, int n, int stride, int64_t P0, int64_t S_max) {
  if (n < 1 || n > stride || P0 < 0) return false;
  int prev = -1;
  for (int k = 0; k < n; ++k) {
    const int v = pb[k];
    if (v <= prev) return false;
    prev = v;
  }
  return P0 + prev < S_max;
}

__global__ void __launch_bounds__(kCommitThreads) kv_commit_kernel(const __grid_constant__ CommitParams P) {
  const int b = blockIdx.y, ci = blockIdx.z;
  const int64_t ncol = P.row_bytes / 16;
  const int64_t col = int64_t(blockIdx.x) * kCommitThreads + threadIdx.x;
  const int64_t P0 = P.prefix_len[b];
  const int n = P.path_len[b];
  const int32_t* pb = P.path + int64_t(b) * P.path_stride;
  const bool ok = path_ok(pb, n, P.path_stride, P0, P.S_max);
  if (blockIdx.x == 0 && ci == 0 && threadIdx.x == 0) {
    if (!ok) set_status(P.status, W12_ERR_BAD_TREE);
    if (P.flag_new_len) P.new_len[b] = int32_t(ok ? P0 + n : P0);
  }
  if (!ok || col >= ncol) return;
  uint4* base = reinterpret_cast<uint4*>(P.caches[ci] + int64_t(b) * P.S_max * P.row_bytes) + col;
  for (int k = 0; k < n; ++k) {
    const int src = pb[k];
    if (src != k) base[(P0 + k) * ncol] = base[(P0 + src) * ncol];
  }
}

// out[b] = states[b, path[b, path_len[b] - 1]] (16-byte columns).
__global__ void __launch_bounds__(kCommitThreads)
    state_select_kernel(const uint8_t* __restrict__ states, int T, int64_t row_bytes, const int32_t* __restrict__ path,
                        int path_stride, const int32_t* __restrict__ path_len, uint8_t* __restrict__ out,
                        int32_t* status) {
  const int b = blockIdx.y;
  const int64_t ncol = row_bytes / 16;
  const int64_t col = int64_t(blockIdx.x) * kCommitThreads + threadIdx.x;
  const int n = path_len[b];
  const int node = (n >= 1 && n <= path_stride) ? path[int64_t(b) * path_stride + n - 1] : -1;
  const bool ok = node >= 0 && node < T;
  if (!ok) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, W12_ERR_BAD_TREE);
    return;
  }
  if (col >= ncol) return;
  const uint4* src = reinterpret_cast<const uint4*>(states + (int64_t(b) * T + node) * row_bytes) + col;
  reinterpret_cast<uint4*>(out + int64_t(b) * row_bytes)[col] = *src;
}

}  // namespace w12

using namespace w12;

extern "C" {

int w12_kv_commit(void* const* caches, int n_caches, int B, int64_t S_max, int64_t row_bytes,
                  const int32_t* prefix_len, const int32_t* path, int path_stride, const int32_t* path_len,
                  int32_t* new_len, int32_t* dev_status, void* stream) {
  if (!caches || n_caches < 1 || B < 1 || B > 65535 || S_max < 1 || row_bytes < 16 || row_bytes % 16 ||
      path_stride < 1 || !prefix_len || !path || !path_len)
    return W12_ERR_ARG;
  for (int i = 0; i < n_caches; ++i)
    if (!caches[i] || !aligned(caches[i], 16)) return W12_ERR_ARG;
  if (!device_supported()) return W12_ERR_UNSUPPORTED;
  const int64_t ncol = row_bytes / 16;
  const int64_t gx = (ncol + kCommitThreads - 1) / kCommitThreads;
  if (gx > 0x7FFFFFFF) return W12_ERR_SHAPE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int i0 = 0; i0 < n_caches; i0 += kMaxCaches) {
    CommitParams P{};
    P.n_caches = n_caches - i0 < kMaxCaches ? n_caches - i0 : kMaxCaches;
    for (int i = 0; i < P.n_caches; ++i) P.caches[i] = static_cast<uint8_t*>(caches[i0 + i]);
    P.B = B;
    P.path_stride = path_stride;
    P.S_max = S_max;
    P.row_bytes = row_bytes;
    P.prefix_len = prefix_len;
    P.path = path;
    P.path_len = path_len;
    P.new_len = new_len;
    P.flag_new_len = (new_len && i0 == 0) ? 1 : 0;  // every launch reads the same prefix lengths
    P.status = dev_status;
    kv_commit_kernel<<<dim3(unsigned(gx), unsigned(B), unsigned(P.n_caches)), kCommitThreads, 0, s>>>(P);
    const int st = cuda_status(cudaGetLastError());
    if (st) return st;
  }
  return W12_OK;
}

int w12_state_select(const void* states, int B, int T, int64_t row_bytes, const int32_t* path, int path_stride,
                     const int32_t* path_len, void* out, int32_t* dev_status, void* stream) {
  if (!states || !out || !path || !path_len || B < 1 || B > 65535 || T < 1 || row_bytes < 16 || row_bytes % 16 ||
      path_stride < 1 || !aligned(states, 16) || !aligned(out, 16))
    return W12_ERR_ARG;
  if (!device_supported()) return W12_ERR_UNSUPPORTED;
  const int64_t gx = (row_bytes / 16 + kCommitThreads - 1) / kCommitThreads;
  if (gx > 0x7FFFFFFF) return W12_ERR_SHAPE;
  state_select_kernel<<<dim3(unsigned(gx), unsigned(B)), kCommitThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t*>(states), T, row_bytes, path, path_stride, path_len, static_cast<uint8_t*>(out),
      dev_status);
  return cuda_status(cudaGetLastError());
}

}  // extern "C"
