// Greedy block and tree verification.
//
// A drafted token is accepted iff it equals the target's greedy choice at the
// preceding position (SpecPilot paper digest, "Risks" bullet 3); block
// drafters propose a whole block per step (SpecPilot write-up, "Main
// challenge"); tree drafts are causal, every token conditioned on its
// root-to-node path (JetSpec article, "Technical architecture").
//
// Kernels:
//   logits_partials_kernel  row-chunk (max, index) partials of fp32 logits
//   reduce_accept_kernel    one CTA per verified row reduces the partials to
//                           the row argmax; the last CTA to finish runs the
//                           acceptance walk for every request (warp per
//                           request: ballot over the block, or pointer jumping
//                           over the tree).
// The fused entry points produce the same partials from the W12 LM head
// (w12_gemm.cu, argmax epilogue) and reuse reduce_accept_kernel.
#include <float.h>

#include "w12_dev.cuh"
#include "w12_host.h"

namespace w12 {

constexpr int kLogitChunk = 4096;

__device__ __forceinline__ void better(float& bv, int& bi, float v, int i) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

__device__ __forceinline__ void warp_argmax(float& bv, int& bi) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
    const int i = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
    better(bv, bi, v, i);
  }
}

// Block of 256 threads; returns the block-wide result in thread 0.
__device__ __forceinline__ void block_argmax(float& bv, int& bi) {
  __shared__ float sv[8];
  __shared__ int si[8];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  warp_argmax(bv, bi);
  if (lane == 0) {
    sv[w] = bv;
    si[w] = bi;
  }
  cta_sync();
  if (w == 0) {
    bv = lane < 8 ? sv[lane] : -INFINITY;
    bi = lane < 8 ? si[lane] : 0x7FFFFFFF;
    warp_argmax(bv, bi);
  }
}

__global__ void __launch_bounds__(256) logits_partials_kernel(const float* __restrict__ logits, int64_t V,
                                                              int Mstride, int chunk, float* __restrict__ pv,
                                                              int32_t* __restrict__ pi) {
  grid_dep_wait();
  const int m = blockIdx.y, cidx = blockIdx.x;
  const int64_t beg = int64_t(cidx) * chunk;
  const int64_t end = beg + chunk < V ? beg + chunk : V;
  const float* rowp = logits + int64_t(m) * V;
  float bv = -INFINITY;
  int bi = 0x7FFFFFFF;
  for (int64_t j = beg + threadIdx.x; j < end; j += blockDim.x) better(bv, bi, __ldg(rowp + j), int(j));
  block_argmax(bv, bi);
  if (threadIdx.x == 0) {
    pv[int64_t(cidx) * Mstride + m] = bv;
    pi[int64_t(cidx) * Mstride + m] = bi;
  }
}

// Greedy acceptance of request b by one warp.
__device__ void accept_greedy(int b, int T, int T_rows, const int32_t* draft, const int32_t* amax,
                              int32_t* accept_len, int32_t* bonus) {
  const int lane = threadIdx.x & 31;
  int L = T;
  for (int j0 = 0; j0 < T; j0 += 32) {
    const int j = j0 + lane;
    const bool miss = j < T && draft[int64_t(b) * T + j] != __ldcg(amax + int64_t(b) * T_rows + j);
    const uint32_t mask = __ballot_sync(0xFFFFFFFFu, miss);
    if (mask) {
      L = j0 + __ffs(mask) - 1;
      break;
    }
  }
  if (lane == 0) {
    accept_len[b] = L;
    bonus[b] = L < T_rows ? __ldcg(amax + int64_t(b) * T_rows + L) : -1;
  }
}

// Tree acceptance of tree b by one warp, with per-warp scratch of 3*kTreeMax ints.
__device__ void accept_tree(int b, int T, const int32_t* parents, const int32_t* draft, const int32_t* amax,
                            int32_t* path, int32_t* path_len, int32_t* accept_len, int32_t* bonus, int* anc,
                            int* dist, int* okv, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int32_t* par = parents + int64_t(b) * T;
  const int32_t* dr = draft + int64_t(b) * T;
  const int32_t* am = amax + int64_t(b) * T;
  bool valid = true;
  for (int i = lane; i < T; i += 32) {
    const int p = par[i];
    if (i == 0 ? p != -1 : (p < 0 || p >= i)) valid = false;
  }
  valid = __all_sync(0xFFFFFFFFu, valid);
  if (!valid) {
    for (int i = lane; i < T; i += 32) path[int64_t(b) * T + i] = -1;
    if (lane == 0) {
      path_len[b] = -1;
      accept_len[b] = -1;
      bonus[b] = -1;
      set_status(status, W12_ERR_BAD_TREE);
    }
    return;
  }
  for (int i = lane; i < T; i += 32) {
    if (i == 0) {
      anc[0] = 0;
      dist[0] = 0;
      okv[0] = 1;
    } else {
      const int p = par[i];
      anc[i] = p;
      dist[i] = 1;
      okv[i] = dr[i] == __ldcg(am + p) ? 1 : 0;
    }
  }
  __syncwarp();
  // Pointer jumping: after round r, anc[i] is the 2^r-th ancestor (or the
  // root), dist[i] the number of edges to it, okv[i] whether every node on
  // the way (i included, anc[i] excluded) matched its parent's target.
  for (int span = 1; span < T; span <<= 1) {
    int na[kTreeMax / 32], nd[kTreeMax / 32], no[kTreeMax / 32];
    int k = 0;
    for (int i = lane; i < T; i += 32, ++k) {
      const int a = anc[i];
      na[k] = anc[a];
      nd[k] = dist[i] + dist[a];
      no[k] = okv[i] & okv[a];
    }
    __syncwarp();
    k = 0;
    for (int i = lane; i < T; i += 32, ++k) {
      anc[i] = na[k];
      dist[i] = nd[k];
      okv[i] = no[k];
    }
    __syncwarp();
  }
  // Deepest accepted node, lowest index among equals.
  int bd = -1, bn = 0x7FFFFFFF;
  for (int i = lane; i < T; i += 32) {
    const int d = okv[i] ? dist[i] : -1;
    if (d > bd) {
      bd = d;
      bn = i;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const int d = __shfl_xor_sync(0xFFFFFFFFu, bd, o);
    const int n = __shfl_xor_sync(0xFFFFFFFFu, bn, o);
    if (d > bd || (d == bd && n < bn)) {
      bd = d;
      bn = n;
    }
  }
  for (int i = lane; i < T; i += 32)
    if (i > bd) path[int64_t(b) * T + i] = -1;
  if (lane == 0) {
    int node = bn;
    for (int d = bd; d >= 0; --d) {
      path[int64_t(b) * T + d] = node;
      node = par[node];
    }
    path_len[b] = bd + 1;
    accept_len[b] = bd;
    bonus[b] = __ldcg(am + bn);
  }
}

// mode 0 = greedy blocks, mode 1 = trees.
__global__ void __launch_bounds__(256) reduce_accept_kernel(
    const float* __restrict__ pv, const int32_t* __restrict__ pi, int nparts, int Mstride, int M, int mode, int B,
    int T, int T_rows, const int32_t* __restrict__ draft, const int32_t* __restrict__ parents,
    int32_t* __restrict__ accept_len, int32_t* __restrict__ bonus, int32_t* __restrict__ path,
    int32_t* __restrict__ path_len, int32_t* argmax_ws, int32_t* argmax_out, int32_t* done, int32_t* status) {
  __shared__ int is_last;
  __shared__ int tree_scratch[8][3][kTreeMax];
  grid_dep_wait();
  grid_dep_launch();
  const int m = blockIdx.x;
  float bv = -INFINITY;
  int bi = 0x7FFFFFFF;
  // Eight partials per thread in flight before the comparisons: one L2 round
  // trip per batch (1,187 partials per row over 256 threads for the 151,936
  // vocabulary: one batch) instead of one per partial.
  constexpr int kBatch = 8;
  for (int p0 = threadIdx.x; p0 < nparts; p0 += kBatch * int(blockDim.x)) {
    float vv[kBatch];
    int32_t ii[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int p = p0 + j * int(blockDim.x);
      vv[j] = p < nparts ? pv[int64_t(p) * Mstride + m] : -INFINITY;
      ii[j] = p < nparts ? pi[int64_t(p) * Mstride + m] : 0x7FFFFFFF;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) better(bv, bi, vv[j], ii[j]);
  }
  block_argmax(bv, bi);
  if (threadIdx.x == 0) {
    argmax_ws[m] = bi;
    if (argmax_out) argmax_out[m] = bi;
    __threadfence();
    const int old = atomicAdd(done, 1);
    is_last = old == M - 1;
  }
  cta_sync();
  if (!is_last) return;
  __threadfence();
  if (threadIdx.x == 0) *done = 0;
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int b = w; b < B; b += nw) {
    if (mode == 0)
      accept_greedy(b, T, T_rows, draft, argmax_ws, accept_len, bonus);
    else
      accept_tree(b, T, parents, draft, argmax_ws, path, path_len, accept_len, bonus, tree_scratch[w][0],
                  tree_scratch[w][1], tree_scratch[w][2], status);
  }
}

int launch_logits_partials(const float* logits, int64_t V, int M, int Mstride, int chunk, float* pv, int32_t* pi,
                           cudaStream_t stream) {
  const int64_t nparts = (V + chunk - 1) / chunk;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nparts), static_cast<unsigned>(M));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_enabled() ? 1 : 0;
  return cuda_status(cudaLaunchKernelEx(&cfg, logits_partials_kernel, logits, V, Mstride, chunk, pv, pi));
}

int launch_reduce_accept(const float* pv, const int32_t* pi, int nparts, int Mstride, int M, int mode, int B, int T,
                         int T_rows, const int32_t* draft, const int32_t* parents, int32_t* accept_len, int32_t* bonus,
                         int32_t* path, int32_t* path_len, int32_t* argmax_ws, int32_t* argmax_out, int32_t* done,
                         int32_t* dev_status, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(M));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_enabled() ? 1 : 0;
  return cuda_status(cudaLaunchKernelEx(&cfg, reduce_accept_kernel, pv, pi, nparts, Mstride, M, mode, B, T, T_rows,
                                        draft, parents, accept_len, bonus, path, path_len, argmax_ws, argmax_out, done,
                                        dev_status));
}

static int check_greedy(int B, int T, int T_rows) {
  if (B < 1 || T < 1 || (T_rows != T && T_rows != T + 1)) return W12_ERR_ARG;
  if (int64_t(B) * T_rows > kMaxM) return W12_ERR_SHAPE;
  return W12_OK;
}

static int check_tree(int B, int T) {
  if (B < 1 || T < 1 || T > kTreeMax) return W12_ERR_ARG;
  if (int64_t(B) * T > kMaxM) return W12_ERR_SHAPE;
  return W12_OK;
}

// Carve the verify workspace for M rows over a vocabulary of V.
static int verify_ws(int64_t M, int64_t V, int64_t K, void* ws, size_t ws_bytes, GemmShape* sh, WsLayout* L) {
  int st = gemm_shape(M, (V + kGroup - 1) / kGroup * kGroup, K, sh);
  if (st) return st;
  const int sms = device_sm_count();
  GemmShape sz = *sh;
  sz.grid = sms > 0 ? sms : 256;
  *L = ws_layout(sz, sh->tiles);
  if (!ws) return W12_ERR_ARG;
  if (ws_bytes < L->total) return W12_ERR_WORKSPACE;
  return W12_OK;
}

static int verify_logits(const float* logits, int64_t V, int mode, const int32_t* parents, const int32_t* draft,
                         int B, int T, int T_rows, int32_t* path, int32_t* path_len, int32_t* accept_len,
                         int32_t* bonus, int32_t* argmax_out, void* ws, size_t ws_bytes, int32_t* dev_status,
                         cudaStream_t stream) {
  if (!logits || V < 1 || !draft || !accept_len || !bonus) return W12_ERR_ARG;
  const int M = B * T_rows;
  GemmShape sh;
  WsLayout L;
  int st = verify_ws(M, V, kGroup, ws, ws_bytes, &sh, &L);
  if (st) return st;
  if (!device_supported()) return W12_ERR_UNSUPPORTED;
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* pv = reinterpret_cast<float*>(w + L.amax_val);
  int32_t* pi = reinterpret_cast<int32_t*>(w + L.amax_idx);
  const int nparts = int((V + kLogitChunk - 1) / kLogitChunk);
  st = launch_logits_partials(logits, V, M, sh.Mpad, kLogitChunk, pv, pi, stream);
  if (st) return st;
  return launch_reduce_accept(pv, pi, nparts, sh.Mpad, M, mode, B, T, T_rows, draft, parents, accept_len, bonus, path,
                              path_len, reinterpret_cast<int32_t*>(w + L.argmax), argmax_out,
                              reinterpret_cast<int32_t*>(w + L.done), dev_status, stream);
}

static int verify_fused(const uint16_t* H, const w12_weights* head, int mode, const int32_t* parents,
                        const int32_t* draft, int B, int T, int T_rows, int32_t* path, int32_t* path_len,
                        int32_t* accept_len, int32_t* bonus, int32_t* argmax_out, void* ws, size_t ws_bytes,
                        int32_t* dev_status, cudaStream_t stream) {
  if (!H || !head || !draft || !accept_len || !bonus) return W12_ERR_ARG;
  const int M = B * T_rows;
  GemmShape sh;
  WsLayout L;
  int st = verify_ws(M, head->N, head->K, ws, ws_bytes, &sh, &L);
  if (st) return st;
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* pv = reinterpret_cast<float*>(w + L.amax_val);
  int32_t* pi = reinterpret_cast<int32_t*>(w + L.amax_idx);
  st = launch_gemm(true, true, H, M, head, nullptr, head->N, head->K, nullptr, pv, pi, ws, ws_bytes, dev_status,
                   stream);
  if (st) return st;
  return launch_reduce_accept(pv, pi, sh.tiles, sh.Mpad, M, mode, B, T, T_rows, draft, parents, accept_len, bonus,
                              path, path_len, reinterpret_cast<int32_t*>(w + L.argmax), argmax_out,
                              reinterpret_cast<int32_t*>(w + L.done), dev_status, stream);
}

}  // namespace w12

using namespace w12;

extern "C" {

int w12_verify_greedy(const float* logits, int64_t V, const int32_t* draft, int B, int T, int T_rows,
                      int32_t* accept_len, int32_t* bonus, int32_t* argmax_out, void* ws, size_t ws_bytes,
                      int32_t* dev_status, void* stream) {
  int st = check_greedy(B, T, T_rows);
  if (st) return st;
  return verify_logits(logits, V, 0, nullptr, draft, B, T, T_rows, nullptr, nullptr, accept_len, bonus, argmax_out,
                       ws, ws_bytes, dev_status, static_cast<cudaStream_t>(stream));
}

int w12_verify_greedy_fused(const uint16_t* H, const w12_weights* head, const int32_t* draft, int B, int T,
                            int T_rows, int32_t* accept_len, int32_t* bonus, int32_t* argmax_out, void* ws,
                            size_t ws_bytes, int32_t* dev_status, void* stream) {
  int st = check_greedy(B, T, T_rows);
  if (st) return st;
  return verify_fused(H, head, 0, nullptr, draft, B, T, T_rows, nullptr, nullptr, accept_len, bonus, argmax_out, ws,
                      ws_bytes, dev_status, static_cast<cudaStream_t>(stream));
}

int w12_verify_tree(const float* logits, int64_t V, const int32_t* parents, const int32_t* draft, int B, int T,
                    int32_t* path, int32_t* path_len, int32_t* accept_len, int32_t* bonus, int32_t* argmax_out,
                    void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  int st = check_tree(B, T);
  if (st) return st;
  if (!parents || !path || !path_len) return W12_ERR_ARG;
  return verify_logits(logits, V, 1, parents, draft, B, T, T, path, path_len, accept_len, bonus, argmax_out, ws,
                       ws_bytes, dev_status, static_cast<cudaStream_t>(stream));
}

int w12_verify_tree_fused(const uint16_t* H, const w12_weights* head, const int32_t* parents, const int32_t* draft,
                          int B, int T, int32_t* path, int32_t* path_len, int32_t* accept_len, int32_t* bonus,
                          int32_t* argmax_out, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  int st = check_tree(B, T);
  if (st) return st;
  if (!parents || !path || !path_len) return W12_ERR_ARG;
  return verify_fused(H, head, 1, parents, draft, B, T, T, path, path_len, accept_len, bonus, argmax_out, ws,
                      ws_bytes, dev_status, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
