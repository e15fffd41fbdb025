// W12 pack and unpack (SpecPilot paper digest, "Reasons" bullet 2: BF16 split
// into three 4-bit planes, restored bitwise). Offline, bit-exact kernels.
#include "w12_dev.cuh"
#include "w12_host.h"

namespace w12 {

// One CTA per 128x128 block u (row tile, K group); thread r handles row r of
// the block. COUNT pass: exception count of the block -> counts[u].
// WRITE pass: planes, ebase and the block's exception entries, placed at
// exc_off[u] in (row, column) order.
template <bool kWrite>
__global__ void __launch_bounds__(128) pack_block_kernel(const uint16_t* __restrict__ W, int N, int K,
                                                         uint8_t* __restrict__ p0, uint8_t* __restrict__ p1,
                                                         uint8_t* __restrict__ p2, uint8_t* __restrict__ ebase,
                                                         uint32_t* __restrict__ exc_off,
                                                         uint32_t* __restrict__ exc_ent, int64_t capacity) {
  const int KB = K / kGroup;
  const int u = blockIdx.x;
  const int bn = u / KB, bk = u % KB;
  const int r = threadIdx.x;
  const int64_t n = int64_t(bn) * kGroup + r;
  const uint16_t* row = W + n * K + int64_t(bk) * kGroup;
  const uint4* row4 = reinterpret_cast<const uint4*>(row);

  // emax over finite nonzero normal values.
  int emax = 0;
#pragma unroll 4
  for (int v = 0; v < 16; ++v) {
    uint4 q = row4[v];
    uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int e = (w4[j] >> (16 * hh + 7)) & 0xFF;
        if (e >= 1 && e <= 254 && e > emax) emax = e;
      }
    }
  }
  const int eb = emax > 15 ? emax - 15 : 0;

  // Codes, planes and exception count.
  int cnt = 0;
  const int64_t prow = n * (K / 2) + int64_t(bk) * (kGroup / 2);
  for (int q8 = 0; q8 < 16; ++q8) {  // 8 elements per step
    uint4 q = row4[q8];
    uint32_t h[8] = {q.x & 0xFFFFu, q.x >> 16, q.y & 0xFFFFu, q.y >> 16,
                     q.z & 0xFFFFu, q.z >> 16, q.w & 0xFFFFu, q.w >> 16};
    uint32_t w0 = 0, w1 = 0, w2 = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t b = h[j];
      const int s = b >> 15, e = (b >> 7) & 0xFF, m = b & 0x7F;
      uint32_t code = 0;
      if (e >= 1 && e <= 254 && e > eb) {
        code = (uint32_t(s) << 11) | (uint32_t(e - eb) << 7) | uint32_t(m);
      } else {
        ++cnt;
      }
      // element j of the group: byte j%4, low nibble for j<4, high nibble for j>=4
      const int sh = 8 * (j & 3) + 4 * (j >> 2);
      w0 |= (code & 0xFu) << sh;
      w1 |= ((code >> 4) & 0xFu) << sh;
      w2 |= ((code >> 8) & 0xFu) << sh;
    }
    if (kWrite) {
      reinterpret_cast<uint32_t*>(p0 + prow)[q8] = w0;
      reinterpret_cast<uint32_t*>(p1 + prow)[q8] = w1;
      reinterpret_cast<uint32_t*>(p2 + prow)[q8] = w2;
    }
  }
  if (kWrite) ebase[int64_t(bk) * N + n] = static_cast<uint8_t>(eb);

  // Block-wide exclusive scan of the per-row counts.
  __shared__ int warp_tot[4];
  __shared__ int block_tot;
  const int lane = r & 31, wid = r >> 5;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[wid] = incl;
  cta_sync();
  int before = 0;
  for (int w = 0; w < wid; ++w) before += warp_tot[w];
  if (r == 0) block_tot = warp_tot[0] + warp_tot[1] + warp_tot[2] + warp_tot[3];
  cta_sync();
  const int excl = before + incl - cnt;

  if (!kWrite) {
    if (r == 0) exc_off[u] = static_cast<uint32_t>(block_tot);
    return;
  }
  if (cnt == 0) return;
  const int64_t base = int64_t(exc_off[u]) + excl;
  if (base + cnt > capacity) return;  // the host checked the total already
  int k = 0;
  for (int c = 0; c < kGroup; ++c) {
    const uint32_t b = row[c];
    const int e = (b >> 7) & 0xFF;
    if (!(e >= 1 && e <= 254 && e > eb)) {
      exc_ent[base + k] = (uint32_t(r) << 23) | (uint32_t(c) << 16) | b;
      ++k;
    }
  }
}

// In-place exclusive scan: counts[0..U) -> offsets[0..U], offsets[U] = total.
__global__ void __launch_bounds__(1024) exclusive_scan_kernel(uint32_t* data, int64_t U) {
  __shared__ uint64_t warp_sum[32];
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  const int64_t per = (U + blockDim.x - 1) / blockDim.x;
  const int64_t beg = t * per, end = beg + per < U ? beg + per : U;
  uint64_t local = 0;
  for (int64_t i = beg; i < end; ++i) local += data[i];
  uint64_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint64_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sum[wid] = incl;
  cta_sync();
  uint64_t before = 0;
  for (int w = 0; w < wid; ++w) before += warp_sum[w];
  uint64_t run = before + incl - local;
  for (int64_t i = beg; i < end; ++i) {
    const uint32_t c = data[i];
    data[i] = static_cast<uint32_t>(run);
    run += c;
  }
  cta_sync();
  if (t == blockDim.x - 1) {
    uint64_t tot = 0;
    for (int w = 0; w < 32; ++w) tot += warp_sum[w];
    data[U] = static_cast<uint32_t>(tot);
  }
}

// One thread per 8 elements: three plane words -> four bf16 pairs.
__global__ void __launch_bounds__(256) unpack_main_kernel(const uint8_t* __restrict__ p0,
                                                          const uint8_t* __restrict__ p1,
                                                          const uint8_t* __restrict__ p2,
                                                          const uint8_t* __restrict__ ebase, int N, int K,
                                                          uint16_t* __restrict__ out) {
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t per_row = K / 8;
  if (gid >= int64_t(N) * per_row) return;
  const int64_t n = gid / per_row, q = gid % per_row;
  const uint32_t A = reinterpret_cast<const uint32_t*>(p0)[gid];
  const uint32_t B = reinterpret_cast<const uint32_t*>(p1)[gid];
  const uint32_t C = reinterpret_cast<const uint32_t*>(p2)[gid];
  const uint32_t eb = ebase[(q * 8 / kGroup) * N + n];
  uint32_t w[4];
  decode8(A, B, C, (eb << 7) * 0x00010001u, w);
  reinterpret_cast<uint4*>(out + n * K)[q] = make_uint4(w[0], w[1], w[2], w[3]);
}

// One CTA per 128x128 block: overwrite the block's exception positions.
__global__ void __launch_bounds__(128) unpack_exc_kernel(const uint32_t* __restrict__ exc_off,
                                                         const uint32_t* __restrict__ exc_ent, int64_t n_exc,
                                                         int N, int K, uint16_t* __restrict__ out,
                                                         int32_t* status) {
  const int KB = K / kGroup;
  const int u = blockIdx.x;
  const int bn = u / KB, bk = u % KB;
  const uint32_t o0 = exc_off[u], o1 = exc_off[u + 1];
  if (o1 < o0 || int64_t(o1) > n_exc) {
    if (threadIdx.x == 0) set_status(status, W12_ERR_CORRUPT);
    return;
  }
  for (uint32_t i = o0 + threadIdx.x; i < o1; i += blockDim.x) {
    const uint32_t e = exc_ent[i];
    // A valid entry has bits 31..30 clear (row field < 128); anything else
    // would address a row outside the block, so it is reported, not written.
    if (e >> 30) {
      set_status(status, W12_ERR_CORRUPT);
      continue;
    }
    const int64_t n = int64_t(bn) * kGroup + (e >> 23);
    const int64_t k = int64_t(bk) * kGroup + ((e >> 16) & 0x7F);
    out[n * K + k] = static_cast<uint16_t>(e & 0xFFFF);
  }
}

static int check_pack_shape(int64_t N, int64_t K) {
  if (N < kGroup || K < kGroup || N % kGroup || K % kGroup) return W12_ERR_SHAPE;
  if ((N / kGroup) * (K / kGroup) >= (int64_t(1) << 31)) return W12_ERR_SHAPE;
  return W12_OK;
}

}  // namespace w12

using namespace w12;

extern "C" {

size_t w12_pack_ws_bytes(int64_t N, int64_t K) {
  if (check_pack_shape(N, K) != W12_OK) return 0;
  return sizeof(uint32_t) * size_t((N / kGroup) * (K / kGroup) + 1);
}

int w12_pack_query(const uint16_t* W, int64_t N, int64_t K, w12_sizes* out, void* ws, size_t ws_bytes,
                   void* stream) {
  if (!W || !out || !ws) return W12_ERR_ARG;
  int st = check_pack_shape(N, K);
  if (st) return st;
  if (!aligned(W, 16)) return W12_ERR_ARG;
  const int64_t U = (N / kGroup) * (K / kGroup);
  if (ws_bytes < w12_pack_ws_bytes(N, K)) return W12_ERR_WORKSPACE;
  if (!device_supported()) return W12_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* counts = static_cast<uint32_t*>(ws);
  pack_block_kernel<false><<<static_cast<unsigned>(U), 128, 0, s>>>(W, int(N), int(K), nullptr, nullptr, nullptr,
                                                                   nullptr, counts, nullptr, 0);
  exclusive_scan_kernel<<<1, 1024, 0, s>>>(counts, U);
  uint32_t total = 0;
  if (cudaMemcpyAsync(&total, counts + U, sizeof(total), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return W12_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return W12_ERR_CUDA;
  out->plane_bytes = N * K / 2;
  out->ebase_bytes = (K / kGroup) * N;
  out->exc_off_count = U + 1;
  out->n_exc = total;
  out->total_bytes = 3 * out->plane_bytes + out->ebase_bytes + 4 * (U + 1) + 4 * int64_t(total);
  return W12_OK;
}

int w12_pack(const uint16_t* W, int64_t N, int64_t K, const w12_weights* dst, void* stream) {
  if (!W || !dst) return W12_ERR_ARG;
  int st = check_pack_shape(N, K);
  if (st) return st;
  if (dst->N != N || dst->K != K) return W12_ERR_ARG;
  if (!dst->p0 || !dst->p1 || !dst->p2 || !dst->ebase || !dst->exc_off) return W12_ERR_ARG;
  if (dst->n_exc > 0 && !dst->exc_ent) return W12_ERR_ARG;
  if (!aligned(W, 16) || !aligned(dst->p0, 16) || !aligned(dst->p1, 16) || !aligned(dst->p2, 16))
    return W12_ERR_ARG;
  if (!device_supported()) return W12_ERR_UNSUPPORTED;
  const int64_t U = (N / kGroup) * (K / kGroup);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  pack_block_kernel<false><<<static_cast<unsigned>(U), 128, 0, s>>>(W, int(N), int(K), nullptr, nullptr, nullptr,
                                                                   nullptr, dst->exc_off, nullptr, 0);
  exclusive_scan_kernel<<<1, 1024, 0, s>>>(dst->exc_off, U);
  uint32_t total = 0;
  if (cudaMemcpyAsync(&total, dst->exc_off + U, sizeof(total), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return W12_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return W12_ERR_CUDA;
  if (int64_t(total) > dst->n_exc) return W12_ERR_WORKSPACE;
  pack_block_kernel<true><<<static_cast<unsigned>(U), 128, 0, s>>>(W, int(N), int(K), dst->p0, dst->p1, dst->p2,
                                                                  dst->ebase, dst->exc_off, dst->exc_ent,
                                                                  dst->n_exc);
  if (cudaGetLastError() != cudaSuccess) return W12_ERR_CUDA;
  return cuda_status(cudaStreamSynchronize(s));
}

int w12_unpack(const w12_weights* src, uint16_t* W_out, int32_t* dev_status, void* stream) {
  if (!src || !W_out) return W12_ERR_ARG;
  int st = check_pack_shape(src->N, src->K);
  if (st) return st;
  if (!src->p0 || !src->p1 || !src->p2 || !src->ebase || !src->exc_off) return W12_ERR_ARG;
  if (src->n_exc > 0 && !src->exc_ent) return W12_ERR_ARG;
  if (!aligned(W_out, 16) || !aligned(src->p0, 4) || !aligned(src->p1, 4) || !aligned(src->p2, 4))
    return W12_ERR_ARG;
  if (!device_supported()) return W12_ERR_UNSUPPORTED;
  const int64_t N = src->N, K = src->K;
  const int64_t U = (N / kGroup) * (K / kGroup);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t groups = N * K / 8;
  unpack_main_kernel<<<static_cast<unsigned>((groups + 255) / 256), 256, 0, s>>>(src->p0, src->p1, src->p2,
                                                                                src->ebase, int(N), int(K), W_out);
  unpack_exc_kernel<<<static_cast<unsigned>(U), 128, 0, s>>>(src->exc_off, src->exc_ent, src->n_exc, int(N), int(K),
                                                            W_out, dev_status);
  return cuda_status(cudaGetLastError());
}

}  // extern "C"
