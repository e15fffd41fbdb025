// Tree-masked verify attention on the tensor cores.
//
// The verify pass scores a causal draft tree (a block of drafted tokens is the
// chain tree) in one forward pass: each draft node's query attends to the
// committed prefix and to the draft nodes on its own root-to-node path (JetSpec
// article, "Technical architecture": every draft token is conditioned on the
// path that leads to it; SpecPilot digest, "Reasons" bullet 2: tree
// verification). Query row (b, t, h) reads key/value head h / (Hq / Hkv); node
// i's key and value sit at cache position prefix_len[b] + i.
//
// One CTA takes 128 query rows of one (request, kv head) -- the rows (head hh
// of the group, node t) in head-major order, so every row of the CTA reads the
// same keys -- over one contiguous range of 128-key blocks (a split of the
// request's keys when there are too few (request, kv head, row tile) items to
// fill the GPU). Per key block:
//   S = Q K^T        tcgen05.mma, A = Q (smem), B = K (smem, both K-major),
//                    D = S in TMEM (double-buffered so S of the next block is
//                    computed while this one is in the softmax);
//   P = exp2(c S - m) two softmax warpgroups, one per 64-key half, read their
//                    half of each row of S from TMEM, mask it, and write P as
//                    bf16 pairs over the first 32 of the half's S columns;
//   O_h += P_h V_h   tcgen05.mma, A = P_h (TMEM), B = V (smem, MN-major: the
//                    cache's head dimension is contiguous), D = O_h in TMEM,
//                    one accumulator per half, merged in the epilogue.
// Each half's running maximum m only moves when a block's maximum exceeds it
// by more than 8 (in log2 units), so P <= 256 and O_h is rescaled rarely; the
// output is (sum_h 2^(m_h - M) O_h) / (sum_h 2^(m_h - M) l_h) with l_h the fp32
// sum of the half's P (P itself enters P V rounded to bf16). With several
// splits each CTA writes (O, m, l) and attn_combine_kernel merges them.
//
// Warp roles (384 threads): warps 0 and 2 issue the TMA copies of K and of V
// (separate rings: a K stage frees once S of its block is done, a V stage once
// P V is), warps 1 and 3 issue the S and the P V MMAs (warp 1 also allocates
// TMEM; S of block j waits for P V of block j - 2, whose P sits in the buffer
// S overwrites), warps 4-7 and 8-11 (warpgroups: warp w reads TMEM lanes
// 32 (w % 4) ..) run the softmax of the first and second key half and the
// epilogue. All warps load Q.
#include "w12_dev.cuh"
#include "w12_host.h"

namespace w12 {
namespace attn_impl {

#define W12_TIE8(v, o)                                                                                   \
  "+r"(v[o]), "+r"(v[o + 1]), "+r"(v[o + 2]), "+r"(v[o + 3]), "+r"(v[o + 4]), "+r"(v[o + 5]), "+r"(v[o + 6]), \
      "+r"(v[o + 7])

// Wait for every outstanding tcgen05.ld of this thread; ties all 128 values
// to the wait (for loads issued as several 16-column pieces).
__device__ __forceinline__ void tmem_ld_wait64(uint32_t (&v)[64]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : W12_TIE8(v, 0), W12_TIE8(v, 8), W12_TIE8(v, 16), W12_TIE8(v, 24), W12_TIE8(v, 32), W12_TIE8(v, 40),
                 W12_TIE8(v, 48), W12_TIE8(v, 56)
               :
               : "memory");
}

__device__ __forceinline__ void tmem_ld_wait128(uint32_t (&v)[128]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : W12_TIE8(v, 0), W12_TIE8(v, 8), W12_TIE8(v, 16), W12_TIE8(v, 24), W12_TIE8(v, 32), W12_TIE8(v, 40),
                 W12_TIE8(v, 48), W12_TIE8(v, 56), W12_TIE8(v, 64), W12_TIE8(v, 72), W12_TIE8(v, 80),
                 W12_TIE8(v, 88), W12_TIE8(v, 96), W12_TIE8(v, 104), W12_TIE8(v, 112), W12_TIE8(v, 120)
               :
               : "memory");
}

constexpr int kD = 128;                         // head dimension
constexpr int kKeys = 128;                      // keys per block
constexpr int kThreads = 384;
constexpr int kCombineThreads = 256;            // merge kernel: one warp per output row
constexpr int kStages = 3;
constexpr int kMaxT = 128;                      // draft nodes per request
constexpr uint32_t kHalf = 128u * 128u;         // 128 rows x 64 bf16 (one 128-byte swizzled half)
constexpr uint32_t kTile = 2u * kHalf;          // 128 rows x 128 bf16
constexpr uint32_t kQOff = 0;
constexpr uint32_t kKOff = kTile;                                  // K ring: stage s at kKOff + s * kTile
constexpr uint32_t kVOff = kKOff + uint32_t(kStages) * kTile;      // V ring
constexpr uint32_t kBarOff = kVOff + uint32_t(kStages) * kTile;
constexpr uint32_t kSmemBytes = kBarOff + 256 + 1024;  // barriers + misc + alignment slack
constexpr uint32_t kTmemCols = 512;
// TMEM: S of even / odd blocks (each key half's P over its first 32 columns),
// and the O accumulators of the two key halves.
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColOA = 256, kColOB = 384;
constexpr int kCtaOverheadBlocks = 4;          // a CTA's start and finish, in key blocks
constexpr float kRescale = 8.0f;                // log2 growth of the maximum that triggers a rescale

struct AttnParams {
  const uint16_t* Q;          // [B, T, Hq, 128]
  uint16_t* O;                // [B, T, Hq, 128]
  const int32_t* prefix_len;  // [B]
  const int32_t* parents;     // [B, T]
  float* part_o;              // [items, nsplit, 128, 128] (nsplit > 1)
  float2* part_ml;            // [items, nsplit, 128]: (m, l)
  int32_t* status;
  int B, T, Hq, Hkv, G, ntile, nsplit, bps, max_len;
  float c;                    // scale * log2(e)
  uint64_t limit_ns;
};

// Shared-memory matrix descriptor of an MN-major operand stored with the
// 128-byte swizzle: rows along K are 128 bytes of 64 MN-consecutive values,
// 8-row groups 1024 bytes apart (stride byte offset), and the next 64 values
// along MN `lbo` bytes further (leading byte offset).
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            int32_t w, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 values -> one word of bf16 (round to nearest even): lo in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t word_sel(const uint32_t (&a)[4], int i) {
  return i == 0 ? a[0] : i == 1 ? a[1] : i == 2 ? a[2] : i == 3 ? a[3] : 0u;
}

// Bits sh .. sh+31 of the 128-bit value a (zero outside [0, 128)).
__device__ __forceinline__ uint32_t bits32(const uint32_t (&a)[4], int sh) {
  if (sh <= -32 || sh >= 128) return 0u;
  const int wi = sh >= 0 ? sh >> 5 : -1;
  const int r = sh - wi * 32;  // 0..31
  const uint32_t lo = word_sel(a, wi), hi = word_sel(a, wi + 1);
  return r == 0 ? lo : (lo >> r) | (hi << (32 - r));
}

// Ancestors of node t (itself included) in a parent array as a 128-bit set;
// a malformed parent array sets W12_ERR_BAD_TREE and ends the walk.
__device__ __forceinline__ void tree_ancestors(const int32_t* pb, int t, int T, uint32_t (&anc)[4], int32_t* status) {
  anc[0] = anc[1] = anc[2] = anc[3] = 0u;
  int j = t;
  for (int step = 0; step <= T && j >= 0; ++step) {
    const uint32_t bit = 1u << (j & 31);
#pragma unroll
    for (int w = 0; w < 4; ++w) anc[w] |= (j >> 5) == w ? bit : 0u;
    const int pj = pb[j];
    if ((j == 0) ? (pj != -1) : (pj < 0 || pj >= j)) {
      set_status(status, W12_ERR_BAD_TREE);
      break;
    }
    j = pj;
  }
}

// Scores of keys key0 .. key0+127 that the row may not see become -inf: it
// sees all of the prefix (keys < Pb) and the draft keys Pb + j of its
// ancestors j; none past the request's keys.
template <int N>
__device__ __forceinline__ void mask_block(uint32_t (&v)[N], int key0, int Pb, const uint32_t (&anc)[4], bool valid) {
#pragma unroll
  for (int w = 0; w < N / 32; ++w) {
    const int lim_w = Pb - key0 - 32 * w;  // keys 32w + k with k < lim_w are prefix keys
    const uint32_t pre = lim_w >= 32 ? ~0u : lim_w <= 0 ? 0u : ((1u << lim_w) - 1u);
    const uint32_t allow = valid ? (pre | bits32(anc, key0 + 32 * w - Pb)) : 0u;
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (!((allow >> k) & 1u)) v[32 * w + k] = __float_as_uint(-INFINITY);
  }
}

// Maximum of the N scores (eight independent chains).
template <int N>
__device__ __forceinline__ float block_max(const uint32_t (&v)[N]) {
  float mx8[8];
#pragma unroll
  for (int a = 0; a < 8; ++a) mx8[a] = __uint_as_float(v[a]);
#pragma unroll
  for (int k = 8; k < N; ++k) mx8[k & 7] = fmaxf(mx8[k & 7], __uint_as_float(v[k]));
  return fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])), fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
}

// Two lanes of fp32 in one instruction (sm_100 family): d = a * b + c and
// d = a + b, each lane rounded as its scalar form.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// P_k = 2^(c s_k + negm), packed as bf16 pairs into v[0 .. N/2-1] in place
// (pair k overwrites v[k], which pair k/2 has already read); returns the fp32 sum.
// The scale and the sum run two lanes per instruction (the softmax is bound
// by instruction issue, not by the exp2 unit).
template <int N>
__device__ __forceinline__ float exp_pack(uint32_t (&v)[N], float c, float negm) {
  float2 ps4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  const float2 c2 = make_float2(c, c), m2 = make_float2(negm, negm);
#pragma unroll
  for (int k = 0; k < N / 2; ++k) {
    const float2 x = fma2(make_float2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1])), c2, m2);
    const float2 p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
    ps4[k & 3] = add2(ps4[k & 3], p);
    v[k] = pack_bf16x2(p.x, p.y);
  }
  const float2 s = add2(add2(ps4[0], ps4[1]), add2(ps4[2], ps4[3]));
  return s.x + s.y;
}

// O row *= f (warp-collective: every lane of the warp calls it).
__device__ __forceinline__ void rescale_row(uint32_t o_row, float f) {
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    uint32_t o[16];
    tmem_ld16(o_row + uint32_t(ch * 16), o);
    tmem_ld_wait(o);
#pragma unroll
    for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
    tmem_st16(o_row + uint32_t(ch * 16), o);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ AttnParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + kBarOff);  // K of block i landed (stage i % kStages)
  uint64_t* kempty = kfull + kStages;                                 // S of the stage's block done
  uint64_t* vfull = kempty + kStages;                                 // V of block i landed
  uint64_t* vempty = vfull + kStages;                                 // P V of the stage's block done
  uint64_t* s_full = vempty + kStages;  // [2]: S of block i in buffer i % 2
  uint64_t* p_full = s_full + 2;        // [2][2]: P of block i (buffer i % 2), key half h
  uint64_t* o_done = p_full + 4;        // [2]: P V of block i (both halves) complete
  uint64_t* o_final = o_done + 2;       // every MMA of the CTA complete
  uint32_t* misc = reinterpret_cast<uint32_t*>(o_final + 1);
  volatile uint32_t* tmem_slot = misc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int idx = blockIdx.x;
  const int tile = idx % P.ntile;
  idx /= P.ntile;
  const int split = idx % P.nsplit;
  idx /= P.nsplit;
  const int g = idx % P.Hkv;
  const int b = idx / P.Hkv;
  const int T = P.T;
  const int item = (b * P.Hkv + g) * P.ntile + tile;

  // Everything below reads what the previous kernel on the stream wrote.
  grid_dep_wait();
  int Pb = P.prefix_len[b];
  if (Pb < 0 || Pb + T > P.max_len) {
    if (threadIdx.x == 0 && tile == 0 && split == 0 && g == 0) set_status(P.status, W12_ERR_ARG);
    Pb = Pb < 0 ? 0 : P.max_len - T;
  }
  const int L = Pb + T;                             // keys of this request
  const int nkb = (L + kKeys - 1) / kKeys;
  const int j0 = split * P.bps;
  const int j1 = min(j0 + P.bps, nkb);
  const int n = j1 - j0;                            // key blocks of this CTA
  if (n <= 0) {
    // Nothing to attend to in this split: an empty partial (m = -inf).
    if (threadIdx.x < 128)
      P.part_ml[(size_t(item) * P.nsplit + split) * 128 + threadIdx.x] = make_float2(-INFINITY, 0.f);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&s_full[k], 1);
      mbar_init(&o_done[k], 1);
    }
    for (int k = 0; k < 4; ++k) mbar_init(&p_full[k], 128);
    mbar_init(o_final, 2);  // one commit from each MMA issuer
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(const_cast<uint32_t*>(tmem_slot), kTmemCols);
    tmem_relinquish();
  }

  // Q tile: 128 rows (head hh of the group, node t) in head-major order, rows
  // past G*T zero; two 128-byte-swizzled halves of 64 dims.
  const int Rg = P.G * T;
  {
    uint8_t* qs = smem + kQOff;
    for (int cid = threadIdx.x; cid < 128 * 16; cid += kThreads) {
      const int r = cid >> 4, c = cid & 15;
      const int rr = tile * 128 + r;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (rr < Rg) {
        const int hh = rr / T, t = rr - hh * T;
        const uint16_t* src = P.Q + ((size_t(b) * T + t) * P.Hq + size_t(g) * P.G + hh) * kD + c * 8;
        v = *reinterpret_cast<const uint4*>(src);
      }
      *reinterpret_cast<uint4*>(qs + (c >> 3) * kHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint64_t lim = P.limit_ns;

  auto fail = [&](int code) {
    set_status(P.status, code);
    *abort_flag = 1;
  };
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0; i < 0x80000000u; ++i) {
      if (mbar_try_wait(bar, parity)) return true;
      if ((i & 63u) == 63u) {
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > lim) {
          fail(W12_ERR_TIMEOUT);
          return false;
        }
      }
    }
    fail(W12_ERR_TIMEOUT);
    return false;
  };

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------------ TMA
    // Warp 0 streams K, warp 2 streams V, each through its own ring: a K stage
    // frees once S of its block is done, well before P V frees the V stage.
    if (lane == 0) {
      const bool isK = warp == 0;
      const CUtensorMap* tm = isK ? &tm_k : &tm_v;
      uint64_t* fullb = isK ? kfull : vfull;
      uint64_t* emptyb = isK ? kempty : vempty;
      uint8_t* ring = smem + (isK ? kKOff : kVOff);
      prefetch_tmap(tm);
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      for (; issued < n; ++issued) {
        const int s = issued % kStages;
        if (issued >= kStages && !wait(&emptyb[s], uint32_t((issued / kStages) - 1) & 1u)) break;
        uint8_t* st = ring + uint32_t(s) * kTile;
        const int key0 = (j0 + issued) * kKeys;
        mbar_arrive_expect_tx(&fullb[s], kTile);
        tma_load_4d(st, tm, 0, g, key0, b, &fullb[s], pol);
        tma_load_4d(st + kHalf, tm, 64, g, key0, b, &fullb[s], pol);
      }
      if (isK) grid_dep_launch();
      if (*abort_flag) {
        for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
          mbar_wait(&fullb[i % kStages], uint32_t(i / kStages) & 1u, drain_limit_ns(lim));
      }
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------------ MMA
    // Two issuing threads on different SM sub-partitions. Warp 1 issues
    // S_j = Q K_j^T into TMEM buffer j % 2 once K_j has landed and P V of block
    // j - 2 is complete (its P sits in that buffer). Warp 3 issues, for each
    // key half h, O_h += P_h V_h once V_j has landed and that half's P is written.
    if (lane == 0) {
      const uint32_t sbase = smem_u32(smem);
      const bool is_s = warp == 1;
      // Descriptors are computed once; a stage or K step only adds a constant
      // (byte offset >> 4) to the 14-bit start-address field, which cannot
      // overflow (shared memory < 256 KB).
      const uint64_t qd = sdesc_k_sw128(sbase + kQOff);
      const uint64_t kd0 = sdesc_k_sw128(sbase + kKOff);
      const uint64_t vd0 = sdesc_mn_sw128(sbase + kVOff, kHalf);
      const uint32_t idesc_s = idesc_bf16(128, 128);
      const uint32_t idesc_o = idesc_bf16(128, 128) | (1u << 16);  // B (V) MN-major
      for (int j = 0; j < n; ++j) {
        const int s = j % kStages;
        const uint32_t sb = tmem + ((j & 1) ? kColS1 : kColS0);
        if (is_s) {
          if (!wait(&kfull[s], uint32_t(j / kStages) & 1u)) break;
          if (j >= 2 && !wait(&o_done[j & 1], uint32_t((j - 2) >> 1) & 1u)) break;
          tc_fence_after();
          const uint64_t kd = kd0 + uint64_t((uint32_t(s) * kTile) >> 4);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t off = uint64_t((uint32_t(ks >> 2) * kHalf + uint32_t(ks & 3) * 32u) >> 4);
            mma_bf16_ss(sb, qd + off, kd + off, idesc_s, ks > 0 ? 1u : 0u);
          }
          tc_commit(&s_full[j & 1]);
          tc_commit(&kempty[s]);
        } else {
          if (!wait(&vfull[s], uint32_t(j / kStages) & 1u)) break;
          const uint64_t vd = vd0 + uint64_t((uint32_t(s) * kTile) >> 4);
          bool got = true;
          for (int h = 0; h < 2; ++h) {
            if (!wait(&p_full[(j & 1) * 2 + h], uint32_t(j >> 1) & 1u)) {
              got = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              // Keys 64h + 16ks ..: V rows 128 bytes apart (the dims' second half kHalf further);
              // P_h sits over the first 32 of this half's 64 S columns.
              const uint64_t off = uint64_t((uint32_t(h) * 8192u + uint32_t(ks) * 2048u) >> 4);
              mma_bf16_ts(tmem + (h ? kColOB : kColOA), sb + uint32_t(64 * h + 8 * ks), vd + off, idesc_o,
                          (j > 0 || ks > 0) ? 1u : 0u);
            }
          }
          if (!got) break;
          tc_commit(&o_done[j & 1]);
          tc_commit(&vempty[s]);
        }
      }
      tc_commit(o_final);  // also drains this thread's MMAs before TMEM is released
      mbar_wait(o_final, 0, drain_limit_ns(lim));
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------ softmax, epilogue
    // Warp w handles rows 32 (w % 4) .. of the tile (its TMEM lanes), one row
    // per thread, over the keys of half h = (w - 4) / 4 (64 keys of every
    // block) with its own running maximum, sum and O accumulator; the two
    // halves are merged in the epilogue.
    const int q = warp & 3;
    const int h = (warp - 4) >> 2;
    const int r = q * 32 + lane;                   // row of the tile = TMEM lane
    const int rr = tile * 128 + r;
    const bool valid = rr < Rg;
    const int hh = valid ? rr / T : 0;
    const int t = valid ? rr - hh * T : 0;
    const uint32_t lane_off = uint32_t(q * 32) << 16;
    const uint32_t o_own = tmem + lane_off + (h ? kColOB : kColOA);
    uint32_t anc[4] = {0u, 0u, 0u, 0u};
    if (valid) tree_ancestors(P.parents + size_t(b) * T, t, T, anc, P.status);
    // Warps whose 32 rows are all padding keep the barrier protocol but skip the math.
    const bool warp_live = __any_sync(0xFFFFFFFFu, valid);
    float m_ref = -INFINITY, l = 0.f;   // this half's running maximum (log2 units) and sum of P
    const float c = P.c;                 // > 0
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      const int kb = (j0 + i) * kKeys + 64 * h;     // first key of this half
      // Waits are one decision per warp: the TMEM loads and stores below are warp-collective.
      if (!__all_sync(0xFFFFFFFFu, wait(&s_full[i & 1], uint32_t(i >> 1) & 1u))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool edge = kb + 64 > Pb;               // draft keys or keys past the request
      if (edge && L - kb < 64) {
        // Cache rows past the request's keys may hold anything: zero this
        // half's such rows in the V stage so that P = 0 never meets a
        // non-finite value (thread r takes row 64h + r / 2, dims half r % 2).
        const int s = i % kStages;
        if (!__all_sync(0xFFFFFFFFu, wait(&vfull[s], uint32_t(i / kStages) & 1u))) {
          ok = false;
          break;
        }
        if ((r >> 1) >= L - kb) {
          uint8_t* vrow = smem + kVOff + uint32_t(s) * kTile + uint32_t(r & 1) * kHalf + uint32_t(kb - (j0 + i) * kKeys + (r >> 1)) * 128u;
#pragma unroll
          for (int k = 0; k < 8; ++k) *reinterpret_cast<uint4*>(vrow + k * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      if (warp_live) {
        const uint32_t sc = tmem + lane_off + ((i & 1) ? kColS1 : kColS0) + uint32_t(64 * h);
        uint32_t v[64];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) tmem_ld16(sc + uint32_t(ch * 16), *reinterpret_cast<uint32_t(*)[16]>(&v[ch * 16]));
        tmem_ld_wait64(v);
        if (edge) mask_block<64>(v, kb, Pb, anc, valid);
        const float mx = block_max<64>(v) * c;
        float factor = 1.f;
        if (mx > m_ref + kRescale) {
          factor = fast_exp2(m_ref - mx);  // 0 while m_ref = -inf
          m_ref = mx;
        }
        const float psum = exp_pack<64>(v, c, m_ref == -INFINITY ? 0.f : -m_ref);
        // Rescale this half's O row when its maximum moved (warp-uniform: the
        // TMEM accesses are collective), once P V of the previous block is done.
        const bool resc = i > 0 && factor < 1.f && l > 0.f;
        if (__any_sync(0xFFFFFFFFu, resc)) {
          if (!__all_sync(0xFFFFFFFFu, wait(&o_done[(i - 1) & 1], uint32_t((i - 1) >> 1) & 1u))) {
            ok = false;
            break;
          }
          tc_fence_after();
          rescale_row(o_own, resc ? factor : 1.f);
        }
        l = l * factor + psum;
        // P over the first 32 of this half's S columns (this thread has read them).
        tmem_st16(sc, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
        tmem_st16(sc + 16u, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&p_full[(i & 1) * 2 + h]);
    }
    // Epilogue: merge the halves, O = (2^(ma-M) Oa + 2^(mb-M) Ob) / (2^(ma-M) la + 2^(mb-M) lb).
    // Every softmax thread reaches the exchange barrier, also after a failed wait.
    const bool fin = __all_sync(0xFFFFFFFFu, ok && wait(o_final, 0));
    float2* xch = reinterpret_cast<float2*>(smem + kKOff);  // the K ring is idle once every MMA is done
    xch[h * 128 + r] = make_float2(m_ref, l);
    named_bar_sync(1, 256);
    if (fin && warp_live) {
      tc_fence_after();
      const float2 other = xch[(1 - h) * 128 + r];
      const float ma = h ? other.x : m_ref, la = h ? other.y : l;
      const float mb = h ? m_ref : other.x, lb = h ? l : other.y;
      const float M = fmaxf(ma, mb);
      const float wa = ma == -INFINITY ? 0.f : fast_exp2(ma - M);
      const float wb = mb == -INFINITY ? 0.f : fast_exp2(mb - M);
      const float den = wa * la + wb * lb;
      // This thread writes dims 64h .. 64h+63 of its row.
      uint32_t v[128];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        tmem_ld16(tmem + lane_off + kColOA + uint32_t(64 * h + ch * 16), *reinterpret_cast<uint32_t(*)[16]>(&v[ch * 16]));
        tmem_ld16(tmem + lane_off + kColOB + uint32_t(64 * h + ch * 16),
                  *reinterpret_cast<uint32_t(*)[16]>(&v[64 + ch * 16]));
      }
      tmem_ld_wait128(v);
      if (P.nsplit == 1) {
        if (valid) {
          const float inv = den > 0.f ? 1.f / den : 0.f;
          uint4* dst = reinterpret_cast<uint4*>(P.O + ((size_t(b) * T + t) * P.Hq + size_t(g) * P.G + hh) * kD + 64 * h);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              o[e] = (wa * __uint_as_float(v[8 * k + e]) + wb * __uint_as_float(v[64 + 8 * k + e])) * inv;
            uint4 w;
            w.x = pack_bf16x2(o[0], o[1]);
            w.y = pack_bf16x2(o[2], o[3]);
            w.z = pack_bf16x2(o[4], o[5]);
            w.w = pack_bf16x2(o[6], o[7]);
            dst[k] = w;
          }
        }
      } else {
        const size_t prow = (size_t(item) * P.nsplit + split) * 128 + r;
        float4* dst = reinterpret_cast<float4*>(P.part_o + prow * kD + 64 * h);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          float o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) o[e] = wa * __uint_as_float(v[4 * k + e]) + wb * __uint_as_float(v[64 + 4 * k + e]);
          dst[k] = make_float4(o[0], o[1], o[2], o[3]);
        }
        if (h == 0) P.part_ml[prow] = make_float2(M, den);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge the splits of every output row: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
// One warp per output row (b, t, h); lane k owns dims 4k .. 4k+3.
__global__ void __launch_bounds__(kCombineThreads) attn_combine_kernel(const __grid_constant__ AttnParams P) {
  grid_dep_wait();
  const int64_t row = int64_t(blockIdx.x) * (kCombineThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int64_t rows = int64_t(P.B) * P.T * P.Hq;
  if (row >= rows) return;
  const int h = int(row % P.Hq);
  const int64_t bt = row / P.Hq;
  const int t = int(bt % P.T), b = int(bt / P.T);
  const int g = h / P.G, hh = h - g * P.G;
  const int r = hh * P.T + t;
  const int tile = r / 128, rit = r % 128;
  const size_t item = size_t(b * P.Hkv + g) * P.ntile + tile;
  float M = -INFINITY;
  for (int s = 0; s < P.nsplit; ++s) M = fmaxf(M, P.part_ml[(item * P.nsplit + s) * 128 + rit].x);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < P.nsplit; ++s) {
      const size_t prow = (item * P.nsplit + s) * 128 + rit;
      const float2 ml = P.part_ml[prow];
      if (ml.x == -INFINITY) continue;
      const float w = fast_exp2(ml.x - M);
      const float4 o = reinterpret_cast<const float4*>(P.part_o + prow * kD)[lane];
      acc.x += w * o.x;
      acc.y += w * o.y;
      acc.z += w * o.z;
      acc.w += w * o.w;
      den += w * ml.y;
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint2 out;
  out.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  out.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  reinterpret_cast<uint2*>(P.O + size_t(row) * kD)[lane] = out;
}

struct AttnPlan {
  int ntile, nkb, nsplit, bps;
  int64_t items;   // (request, kv head, row tile) items, one CTA each per split
};

// Splits of each (request, kv head, row tile) item's key blocks: the count that
// minimises waves x (blocks per split + a CTA's fixed cost) on `sms` SMs (one
// CTA per SM), smallest on ties.
static AttnPlan plan_attn(int B, int T, int Hq, int Hkv, int64_t max_len, int sms) {
  AttnPlan p{};
  const int G = Hq / Hkv;
  p.ntile = (G * T + 127) / 128;
  p.nkb = int((max_len + kKeys - 1) / kKeys);
  p.items = int64_t(B) * Hkv * p.ntile;
  int best = 1;
  int64_t best_cost = -1;
  for (int s = 1; s <= p.nkb && s <= 64; ++s) {
    const int64_t waves = (p.items * s + sms - 1) / sms;
    const int64_t cost = waves * ((p.nkb + s - 1) / s + kCtaOverheadBlocks);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  p.bps = (p.nkb + best - 1) / best;
  p.nsplit = (p.nkb + p.bps - 1) / p.bps;
  return p;
}

static int sms_or_default() {
  const int sms = device_sm_count();
  return sms > 0 ? sms : 152;
}

static bool shape_ok(int B, int T, int Hq, int Hkv, int head_dim, int64_t S_max, int64_t max_len) {
  return B >= 1 && B <= 65535 && T >= 1 && T <= kMaxT && Hkv >= 1 && Hq >= Hkv && Hq % Hkv == 0 && Hq <= 1024 &&
         head_dim == kD && S_max >= T && S_max < (int64_t(1) << 31) && max_len >= T && max_len <= S_max;
}

static size_t ws_bytes_of(const AttnPlan& p) {
  if (p.nsplit <= 1) return 256;
  const size_t rows = size_t(p.items) * p.nsplit * 128;
  return rows * kD * sizeof(float) + rows * sizeof(float2) + 256;
}

}  // namespace attn_impl
}  // namespace w12

using namespace w12;
using namespace w12::attn_impl;

extern "C" {

size_t w12_tree_attention_ws_bytes(int B, int T, int Hq, int Hkv, int64_t max_kv_len) {
  if (!shape_ok(B, T, Hq, Hkv, kD, max_kv_len, max_kv_len)) return 0;
  return ws_bytes_of(plan_attn(B, T, Hq, Hkv, max_kv_len, sms_or_default()));
}

int w12_tree_attention(const uint16_t* Q, const uint16_t* K_cache, const uint16_t* V_cache, int B, int T, int Hq,
                       int Hkv, int head_dim, int64_t S_max, int64_t max_kv_len, const int32_t* prefix_len,
                       const int32_t* parents, float scale, uint16_t* O, void* ws, size_t ws_bytes,
                       int32_t* dev_status, void* stream) {
  if (!Q || !K_cache || !V_cache || !prefix_len || !parents || !O || !aligned(Q, 16) || !aligned(K_cache, 16) ||
      !aligned(V_cache, 16) || !aligned(O, 16) || !(scale > 0.f) || scale > 1e30f)
    return W12_ERR_ARG;
  if (!shape_ok(B, T, Hq, Hkv, head_dim, S_max, max_kv_len)) return W12_ERR_SHAPE;
  if (!device_supported()) return W12_ERR_UNSUPPORTED;
  const AttnPlan pl = plan_attn(B, T, Hq, Hkv, max_kv_len, sms_or_default());
  if (pl.items * pl.nsplit > 0x7FFFFFFF) return W12_ERR_SHAPE;
  if (pl.nsplit > 1 && (!ws || !aligned(ws, 16) || ws_bytes < ws_bytes_of(pl))) return W12_ERR_WORKSPACE;

  AttnParams P{};
  P.Q = Q;
  P.O = O;
  P.prefix_len = prefix_len;
  P.parents = parents;
  if (pl.nsplit > 1) {
    const size_t rows = size_t(pl.items) * pl.nsplit * 128;
    P.part_o = static_cast<float*>(ws);
    P.part_ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(ws) + rows * kD * sizeof(float));
  }
  P.status = dev_status;
  P.B = B;
  P.T = T;
  P.Hq = Hq;
  P.Hkv = Hkv;
  P.G = Hq / Hkv;
  P.ntile = pl.ntile;
  P.nsplit = pl.nsplit;
  P.bps = pl.bps;
  P.max_len = int(max_kv_len);
  P.c = float(double(scale) * 1.4426950408889634);
  P.limit_ns = wait_limit_ns();

  // Caches [B, S_max, Hkv, 128] as 4-D maps (dim, head, position, request):
  // a box is 128 positions x 64 dims of one head, so a block never reads
  // another request's rows (positions past S_max read as zero).
  CUtensorMap tk, tv;
  const uint64_t dims[4] = {uint64_t(kD), uint64_t(Hkv), uint64_t(S_max), uint64_t(B)};
  const uint64_t strides[3] = {uint64_t(kD) * 2, uint64_t(Hkv) * kD * 2, uint64_t(S_max) * Hkv * kD * 2};
  const uint32_t box[4] = {64, 1, uint32_t(kKeys), 1};
  if (!encode_tmap_4d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<uint16_t*>(K_cache), dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_4d(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<uint16_t*>(V_cache), dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
    return W12_ERR_CUDA;

  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return W12_ERR_CUDA;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes)) !=
        cudaSuccess)
      return W12_ERR_CUDA;
    attr_set[dev] = true;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(pl.items * pl.nsplit));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_enabled() ? 1 : 0;
  int st = cuda_status(cudaLaunchKernelEx(&cfg, attn_kernel, tk, tv, P));
  if (st || pl.nsplit == 1) return st;
  const int64_t rows = int64_t(B) * T * Hq;
  cudaLaunchConfig_t cfg2 = cfg;
  cfg2.gridDim = dim3(unsigned((rows + kCombineThreads / 32 - 1) / (kCombineThreads / 32)));
  cfg2.blockDim = dim3(kCombineThreads);
  cfg2.dynamicSmemBytes = 0;
  return cuda_status(cudaLaunchKernelEx(&cfg2, attn_combine_kernel, P));
}

}  // extern "C"
