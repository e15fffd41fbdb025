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
// Work unit: 128 query rows of one (request, kv head) -- the rows (head hh of
// the group, node t) in head-major order, so every row reads the same keys --
// against one 128-key block; an item is such a row tile with all its key
// blocks. The kernel is persistent: one CTA per SM takes an even run of the
// item-major sequence of units (stream-K), so a run covers the tail of one
// item, whole items, and the head of another, and no SM idles in a second
// wave. Per key block:
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
// sum of the half's P (P itself enters P V rounded to bf16). A segment that
// is a whole item writes O directly; otherwise it stores its (O, m, l) and adds
// its block count to the item's count, and the segment that completes the
// count merges the item's partials (merge_item) and resets the count.
//
// Warp roles (384 threads): warps 0 and 2 issue the TMA copies of K and of V
// (separate rings: a K stage frees once S of its block is done, a V stage once
// P V is), warps 1 and 3 issue the S and the P V MMAs (warp 1 also allocates
// TMEM; S of block j waits for P V of block j - 2, whose P sits in the buffer
// S overwrites), warps 4-7 and 8-11 (warpgroups: warp w reads TMEM lanes
// 32 (w % 4) ..) run the softmax of the first and second key half and the
// epilogue. All warps load the first segment's Q; the softmax warps load the
// next one's once the MMAs of a segment are done.
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
constexpr float kRescale = 8.0f;                // log2 growth of the maximum that triggers a rescale
constexpr int kEarlyBlocks = 1;                 // K/V blocks copied before the setup barrier
constexpr int kMergeBatch = 1;                  // partials whose loads a merge step keeps in flight

struct AttnParams {
  const uint16_t* Q;          // [B, T, Hq, 128]
  uint16_t* O;                // [B, T, Hq, 128]
  const int32_t* prefix_len;  // [B]
  const int32_t* parents;     // [B, T]
  uint4* part_o;              // [grid, 2 slots, 16 chunks of 8 dims, 128 rows]: partial O / (l sc), fp16
  float2* part_ml;            // [grid, 2 slots, 128 rows]: (m, l) of the partial
  float* part_sc;             // [grid, 2 slots, 2 halves, 128 rows]: scale sc of the half row
  int32_t* cnt;               // [items]: key blocks of the item done (zero between calls)
  int32_t* status;
  int64_t U;                  // B x Hkv x nkb (request, kv head, key block) units
  int B, T, Hq, Hkv, G, ntile, nkb, max_len;
  int ngroups;                // CTA groups; CTA c is row tile c % ntile of group c / ntile
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

// The same for fp16, and back.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float2 unpack_f16x2(uint32_t v) {
  float lo, hi;
  asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(v));
  return make_float2(lo, hi);
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

// A request's parent row spread over the warp: lane l holds parents[l + 32k]
// in pr[k] (one round of loads).
__device__ __forceinline__ void parent_row(const int32_t* pb, int T, int (&pr)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = lane + 32 * k;
    pr[k] = -1;
    if (32 * k < T && i < T) pr[k] = __ldg(pb + i);
  }
}

// Ancestors of node t (itself included) as a 128-bit set, for every lane of
// the warp at once (warp-collective), from the parent row the warp holds
// (parent_row): each lane walks its node's path by shuffles. A malformed row
// (parents[0] != -1, or parents[i] outside [0, i)) sets W12_ERR_BAD_TREE and
// every lane keeps only its own node.
__device__ __forceinline__ void tree_ancestors(const int (&pr)[4], int t, int T, bool active, uint32_t (&anc)[4],
                                               int32_t* status) {
  const int lane = threadIdx.x & 31;
  bool bad = false;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = lane + 32 * k;
    if (i < T) bad |= i == 0 ? pr[k] != -1 : (pr[k] < 0 || pr[k] >= i);
  }
  anc[0] = anc[1] = anc[2] = anc[3] = 0u;
  const bool row_bad = __any_sync(0xFFFFFFFFu, bad);
  if (row_bad && lane == 0) set_status(status, W12_ERR_BAD_TREE);
  int j = active ? t : -1;
  if (row_bad && j >= 0) {
#pragma unroll
    for (int w = 0; w < 4; ++w) anc[w] = (j >> 5) == w ? 1u << (j & 31) : 0u;
    j = -1;
  }
  // Parents strictly decrease along a valid path: at most T steps.
  for (int step = 0; step <= T && __any_sync(0xFFFFFFFFu, j >= 0); ++step) {
    const int jj = j >= 0 ? j : 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) anc[w] |= (j >= 0 && (jj >> 5) == w) ? 1u << (jj & 31) : 0u;
    // Only the words that hold nodes < T are exchanged (T is uniform).
    const int w = jj >> 5;
    int pj = __shfl_sync(0xFFFFFFFFu, pr[0], jj & 31);
    if (T > 32) {
      const int p1 = __shfl_sync(0xFFFFFFFFu, pr[1], jj & 31);
      pj = w == 1 ? p1 : pj;
    }
    if (T > 64) {
      const int p2 = __shfl_sync(0xFFFFFFFFu, pr[2], jj & 31);
      pj = w == 2 ? p2 : pj;
    }
    if (T > 96) {
      const int p3 = __shfl_sync(0xFFFFFFFFu, pr[3], jj & 31);
      pj = w == 3 ? p3 : pj;
    }
    j = j >= 0 ? pj : -1;
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

// Runs: group k of ntile CTAs takes units [start(k), start(k+1)) of the
// (request, kv head)-major sequence of U units, start(k) = k U / ngroups, as
// even as integers allow; CTA (k, tile) computes row tile `tile` of every unit
// of the run, so the group's CTAs read each K/V block at about the same time
// and all but the first find it in L2.
__device__ __forceinline__ int64_t run_start(const AttnParams& P, int k) {
  return int64_t(k) * P.U / int64_t(P.ngroups);
}

// The group whose run holds unit x: the largest k with start(k) <= x.
__device__ __forceinline__ int run_of(const AttnParams& P, int64_t x) {
  return int(((x + 1) * int64_t(P.ngroups) - 1) / P.U);
}

// One segment of a CTA's run: key blocks [j0, j1) of one item (row tile of a
// request's kv head). A run's first segment keeps its partial result in slot 0
// of the CTA, a later one (only the last can be partial) in slot 1.
struct Seg {
  int item, b, g, tile, j0, j1;
  int n;       // key blocks with keys of the request (the rest of [j0, j1) is past its end)
  int Pb;      // prefix length (clamped into range when invalid)
  int slot;
  bool whole;  // the segment is the whole item: no partial, no merge
};

// The segment's indices (no memory access).
__device__ __forceinline__ bool seg_at(const AttnParams& P, int64_t& pos, int64_t end, int64_t run0, Seg& s) {
  if (pos >= end) return false;
  const int kvh = int(pos / P.nkb);  // request x Hkv + kv head
  s.j0 = int(pos - int64_t(kvh) * P.nkb);
  s.j1 = int(min(int64_t(P.nkb), int64_t(s.j0) + (end - pos)));
  s.slot = pos == run0 ? 0 : 1;
  s.whole = s.j0 == 0 && s.j1 == P.nkb;
  pos = int64_t(kvh) * P.nkb + s.j1;
  s.tile = int(blockIdx.x) % P.ntile;
  s.item = kvh * P.ntile + s.tile;
  s.g = kvh % P.Hkv;
  s.b = kvh / P.Hkv;
  return true;
}

// The segment's request length: its prefix and the key blocks with keys.
__device__ __forceinline__ void seg_keys(const AttnParams& P, Seg& s) {
  int Pb = P.prefix_len[s.b];
  if (Pb < 0 || Pb + P.T > P.max_len) {
    if (threadIdx.x == 0) set_status(P.status, W12_ERR_ARG);
    Pb = Pb < 0 ? 0 : P.max_len - P.T;
  }
  s.Pb = Pb;
  const int nkb_b = (Pb + P.T + kKeys - 1) / kKeys;
  s.n = max(0, min(s.j1, nkb_b) - s.j0);
}

__device__ __forceinline__ bool next_seg(const AttnParams& P, int64_t& pos, int64_t end, int64_t run0, Seg& s) {
  if (!seg_at(P, pos, end, run0, s)) return false;
  seg_keys(P, s);
  return true;
}

__device__ __forceinline__ uint4 ld_no_l1(const void* p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Q rows of a tile for the Q area: 128 rows (head hh of the group, node t) in
// head-major order, rows past G*T zero; two 128-byte-swizzled halves of 64
// dims. Thread `tid` of `kNth` takes pieces tid, tid + kNth, ..; all its loads
// are issued before any is used (one round trip).
template <int kNth>
__device__ __forceinline__ void load_q_regs(const AttnParams& P, uint4 (&qv)[(128 * 16 + kNth - 1) / kNth], int b,
                                            int g, int tile, int tid) {
  constexpr int kIter = (128 * 16 + kNth - 1) / kNth;
  const int Rg = P.G * P.T;
#pragma unroll
  for (int j = 0; j < kIter; ++j) {
    const int cid = tid + j * kNth;
    const int r = cid >> 4, c = cid & 15;
    const int rr = tile * 128 + r;
    qv[j] = make_uint4(0, 0, 0, 0);
    if (cid < 128 * 16 && rr < Rg) {
      const int hh = rr / P.T, t = rr - hh * P.T;
      qv[j] = ld_no_l1(P.Q + ((size_t(b) * P.T + t) * P.Hq + size_t(g) * P.G + hh) * kD + c * 8);
    }
  }
}

template <int kNth>
__device__ __forceinline__ void store_q_regs(uint8_t* qs, const uint4 (&qv)[(128 * 16 + kNth - 1) / kNth], int tid) {
  constexpr int kIter = (128 * 16 + kNth - 1) / kNth;
#pragma unroll
  for (int j = 0; j < kIter; ++j) {
    const int cid = tid + j * kNth;
    const int r = cid >> 4, c = cid & 15;
    if (cid < 128 * 16) *reinterpret_cast<uint4*>(qs + (c >> 3) * kHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = qv[j];
  }
}

// Row of the output: O[b, t, g*G + hh, 64h .. 64h+63] = o / den, as bf16.
__device__ __forceinline__ void store_row(const AttnParams& P, int b, int g, int hh, int t, int h, const float (&o)[64],
                                          float den) {
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint4* dst = reinterpret_cast<uint4*>(P.O + ((size_t(b) * P.T + t) * P.Hq + size_t(g) * P.G + hh) * kD + 64 * h);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    uint4 w;
    w.x = pack_bf16x2(o[8 * k] * inv, o[8 * k + 1] * inv);
    w.y = pack_bf16x2(o[8 * k + 2] * inv, o[8 * k + 3] * inv);
    w.z = pack_bf16x2(o[8 * k + 4] * inv, o[8 * k + 5] * inv);
    w.w = pack_bf16x2(o[8 * k + 6] * inv, o[8 * k + 7] * inv);
    dst[k] = w;
  }
}

// A partial result of this thread's half row: (M, den) and o as
// u = o / (den sc) in fp16, sc the largest |o / den| of the half row (so
// |u| <= 1 and u keeps 11 significant bits relative to the row's largest
// value); chunk-major, so a warp's stores of one chunk cover 32 consecutive
// rows.
__device__ __forceinline__ void store_partial(const AttnParams& P, size_t sb, int r, int h, float M, float den,
                                              const float (&o)[64]) {
  const float inv = den > 0.f ? 1.f / den : 0.f;
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 64; ++k) amax = fmaxf(amax, fabsf(o[k]));
  amax *= inv;
  const float sc = amax > 0.f ? amax : 1.f;
  const float f = inv / sc;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint4 w;
    w.x = pack_f16x2(o[8 * c] * f, o[8 * c + 1] * f);
    w.y = pack_f16x2(o[8 * c + 2] * f, o[8 * c + 3] * f);
    w.z = pack_f16x2(o[8 * c + 4] * f, o[8 * c + 5] * f);
    w.w = pack_f16x2(o[8 * c + 6] * f, o[8 * c + 7] * f);
    P.part_o[(sb * 16 + 8 * h + c) * 128 + r] = w;
  }
  P.part_sc[(sb * 2 + h) * 128 + r] = sc;
  if (h == 0) P.part_ml[sb * 128 + r] = make_float2(M, den);
}

// Merge of an item's partial results by the segment that finished last: it
// folds every partial of the item into (M, den, o), O = sum_s 2^(m_s - M) O_s /
// sum_s 2^(m_s - M) l_s, with O_s = l_s sc_s u_s. With `own` the caller's
// (M, den, o) already hold this CTA's part and its slot is skipped; otherwise
// they start empty and its slot is read like the others. Partials are read
// through L2 (ld.cg) after the acquire that made them visible, kMergeBatch
// CTAs' at a time with all their loads in flight together; an empty partial
// (m = -inf, l = 0) adds nothing.
__device__ void merge_item(const AttnParams& P, const Seg& sg, int r, int h, float M, float den, float (&o)[64],
                           bool own) {
  const int64_t x0 = int64_t(sg.item / P.ntile) * P.nkb;
  const int k0 = run_of(P, x0), k1 = run_of(P, x0 + P.nkb - 1);
  for (int k = k0; k <= k1; k += kMergeBatch) {
    float2 ml[kMergeBatch];
    float scv[kMergeBatch];
    uint4 u[kMergeBatch][8];
#pragma unroll
    for (int e = 0; e < kMergeBatch; ++e) {
      const int kk = k + e;
      const int cc = kk * P.ntile + sg.tile;
      ml[e] = make_float2(-INFINITY, 0.f);
      scv[e] = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) u[e][c] = make_uint4(0, 0, 0, 0);
      if (kk <= k1 && !(own && cc == int(blockIdx.x))) {
        const size_t sb = size_t(cc) * 2 + (run_start(P, kk) >= x0 ? 0 : 1);
        ml[e] = __ldcg(&P.part_ml[sb * 128 + r]);
        scv[e] = __ldcg(&P.part_sc[(sb * 2 + h) * 128 + r]);
#pragma unroll
        for (int c = 0; c < 8; ++c) u[e][c] = __ldcg(&P.part_o[(sb * 16 + 8 * h + c) * 128 + r]);
      }
    }
#pragma unroll
    for (int e = 0; e < kMergeBatch; ++e) {
      const float Mn = fmaxf(M, ml[e].x);
      const float a = M == Mn ? 1.f : fast_exp2(M - Mn);  // 0 while M = -inf
      const float w = ml[e].x == Mn ? 1.f : fast_exp2(ml[e].x - Mn);
      const float f = w * ml[e].y * scv[e];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t ww[4] = {u[e][c].x, u[e][c].y, u[e][c].z, u[e][c].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 v = unpack_f16x2(ww[q]);
          o[8 * c + 2 * q] = o[8 * c + 2 * q] * a + f * v.x;
          o[8 * c + 2 * q + 1] = o[8 * c + 2 * q + 1] * a + f * v.y;
        }
      }
      den = den * a + w * ml[e].y;
      M = Mn;
    }
  }
  const int rr = sg.tile * 128 + r;
  if (rr < P.G * P.T) {
    const int hh = rr / P.T;
    store_row(P, sg.b, sg.g, hh, rr - hh * P.T, h, o, den);
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
  uint64_t* o_final = o_done + 2;       // every MMA of the segment complete (one phase per segment)
  uint64_t* seg_ready = o_final + 1;    // the next segment's Q stored and O read (one phase per boundary)
  uint64_t* drained = seg_ready + 1;    // [2]: each MMA issuer's last MMAs complete
  uint32_t* misc = reinterpret_cast<uint32_t*>(drained + 2);
  volatile uint32_t* tmem_slot = misc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile int* merge_here = reinterpret_cast<volatile int*>(misc + 2);  // this CTA merges the segment's item

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = int(blockIdx.x) / P.ntile;
  const int64_t run0 = run_start(P, grp), run1 = run_start(P, grp + 1);

  // Everything below reads what the previous kernel on the stream wrote.
  grid_dep_wait();
  Seg first;
  int64_t pos_first = run0;              // where the run continues after the first segment
  next_seg(P, pos_first, run1, run0, first);  // run1 > run0: every CTA has at least one unit

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
      mbar_init(&drained[k], 1);
    }
    for (int k = 0; k < 4; ++k) mbar_init(&p_full[k], 128);
    mbar_init(o_final, 2);      // one commit from each MMA issuer
    mbar_init(seg_ready, 256);  // every softmax thread
    *abort_flag = 0;
    fence_barrier_init();
    // The first K and V block do not depend on Q: their copies start now,
    // under the Q load and the setup barrier (the rest of the ring after it,
    // so that Q and the first block are not queued behind them).
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    const uint64_t pol = policy_evict_first();
    for (int i = 0; i < min(kEarlyBlocks, first.n); ++i) {
      const int key0 = (first.j0 + i) * kKeys;
      uint8_t* ks = smem + kKOff + uint32_t(i) * kTile;
      uint8_t* vs = smem + kVOff + uint32_t(i) * kTile;
      mbar_arrive_expect_tx(&kfull[i], kTile);
      tma_load_4d(ks, &tm_k, 0, first.g, key0, first.b, &kfull[i], pol);
      tma_load_4d(ks + kHalf, &tm_k, 64, first.g, key0, first.b, &kfull[i], pol);
      mbar_arrive_expect_tx(&vfull[i], kTile);
      tma_load_4d(vs, &tm_v, 0, first.g, key0, first.b, &vfull[i], pol);
      tma_load_4d(vs + kHalf, &tm_v, 64, first.g, key0, first.b, &vfull[i], pol);
    }
  }
  if (warp == 1) {
    tmem_alloc(const_cast<uint32_t*>(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  // The softmax warps find their rows' ancestor sets for the first segment
  // while the Q loads are in flight.
  uint32_t anc_first[4] = {0u, 0u, 0u, 0u};
  {
    uint4 qv[(128 * 16 + kThreads - 1) / kThreads];
    load_q_regs<kThreads>(P, qv, first.b, first.g, first.tile, threadIdx.x);
    if (warp >= 4) {
      int pr[4];
      parent_row(P.parents + size_t(first.b) * P.T, P.T, pr);
      const int rr = first.tile * 128 + int(threadIdx.x & 127);
      const bool valid = rr < P.G * P.T;
      tree_ancestors(pr, valid ? rr % P.T : 0, P.T, valid && first.n > 0, anc_first, P.status);
    }
    store_q_regs<kThreads>(smem + kQOff, qv, threadIdx.x);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  cta_sync();
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
    // Block numbers (ring stages and phases) run on across segments.
    if (lane == 0) {
      const bool isK = warp == 0;
      const CUtensorMap* tm = isK ? &tm_k : &tm_v;
      uint64_t* fullb = isK ? kfull : vfull;
      uint64_t* emptyb = isK ? kempty : vempty;
      uint8_t* ring = smem + (isK ? kKOff : kVOff);
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      int skip = min(kEarlyBlocks, first.n);  // issued during setup
      bool ok = true;
      int64_t pos = pos_first;
      Seg sg = first;
      for (bool more = true; ok && more; more = next_seg(P, pos, run1, run0, sg)) {
        for (int i = 0; i < sg.n; ++i) {
          if (skip > 0) {
            --skip;
            ++issued;
            continue;
          }
          const int s = issued % kStages;
          if (issued >= kStages && !wait(&emptyb[s], uint32_t((issued / kStages) - 1) & 1u)) {
            ok = false;
            break;
          }
          uint8_t* st = ring + uint32_t(s) * kTile;
          const int key0 = (sg.j0 + i) * kKeys;
          mbar_arrive_expect_tx(&fullb[s], kTile);
          tma_load_4d(st, tm, 0, sg.g, key0, sg.b, &fullb[s], pol);
          tma_load_4d(st + kHalf, tm, 64, sg.g, key0, sg.b, &fullb[s], pol);
          ++issued;
        }
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
    // key half h, O_h += P_h V_h once V_j has landed and that half's P is
    // written. A segment after the first starts once its Q is stored and the
    // previous segment's O has been read out (seg_ready).
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
      int base = 0, si = 0;
      bool ok = true;
      int64_t pos = pos_first;
      Seg sg = first;
      for (bool more = true; more; more = next_seg(P, pos, run1, run0, sg)) {
        if (si > 0 && !wait(seg_ready, uint32_t(si - 1) & 1u)) ok = false;
        for (int j = 0; ok && j < sg.n; ++j) {
          const int gj = base + j;
          const int s = gj % kStages;
          const uint32_t sb = tmem + ((gj & 1) ? kColS1 : kColS0);
          if (is_s) {
            if (!wait(&kfull[s], uint32_t(gj / kStages) & 1u)) {
              ok = false;
              break;
            }
            if (gj >= 2 && !wait(&o_done[gj & 1], uint32_t((gj - 2) >> 1) & 1u)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t kd = kd0 + uint64_t((uint32_t(s) * kTile) >> 4);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint64_t off = uint64_t((uint32_t(ks >> 2) * kHalf + uint32_t(ks & 3) * 32u) >> 4);
              mma_bf16_ss(sb, qd + off, kd + off, idesc_s, ks > 0 ? 1u : 0u);
            }
            tc_commit(&s_full[gj & 1]);
            tc_commit(&kempty[s]);
          } else {
            if (!wait(&vfull[s], uint32_t(gj / kStages) & 1u)) {
              ok = false;
              break;
            }
            const uint64_t vd = vd0 + uint64_t((uint32_t(s) * kTile) >> 4);
            for (int h = 0; h < 2; ++h) {
              if (!wait(&p_full[(gj & 1) * 2 + h], uint32_t(gj >> 1) & 1u)) {
                ok = false;
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
            if (!ok) break;
            tc_commit(&o_done[gj & 1]);
            tc_commit(&vempty[s]);
          }
        }
        if (!ok) break;
        tc_commit(o_final);
        base += sg.n;
        ++si;
      }
      tc_commit(&drained[is_s ? 0 : 1]);  // drains this thread's MMAs before TMEM is released
      mbar_wait(&drained[is_s ? 0 : 1], 0, drain_limit_ns(lim));
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------------- softmax
    // Warps 4-7 take keys 0-63 of every block, warps 8-11 keys 64-127; thread
    // (warp w, lane) owns row 32 (w % 4) + lane. The two halves keep separate
    // running maxima and sums and separate O accumulators (no exchange per
    // block); they are merged at the end of each segment.
    const int q = warp & 3;
    const int h = (warp - 4) >> 2;
    const int r = q * 32 + lane;                   // row of the tile = TMEM lane
    const uint32_t lane_off = uint32_t(q * 32) << 16;
    const uint32_t o_own = tmem + lane_off + (h ? kColOB : kColOA);
    const float c = P.c;                           // > 0
    const int Rg = P.G * P.T;
    float2* xch = reinterpret_cast<float2*>(smem + kQOff);  // the Q area, once the segment's MMAs are done
    int base = 0, si = 0;
    int64_t pos = pos_first;
    Seg sg = first;
    bool more = true;
    uint32_t anc[4] = {anc_first[0], anc_first[1], anc_first[2], anc_first[3]};  // this row's ancestor set
    while (more) {
      Seg nx;
      int64_t pos2 = pos;
      const bool has_next = seg_at(P, pos2, run1, run0, nx);
      const int T = P.T;
      const int rr = sg.tile * 128 + r;
      const bool valid = rr < Rg;
      const int hh = valid ? rr / T : 0;
      const int t = valid ? rr - hh * T : 0;
      // Warps whose 32 rows are all padding keep the barrier protocol but skip the math.
      const bool warp_live = __any_sync(0xFFFFFFFFu, valid);
      const int Pb = sg.Pb, L = Pb + T;
      float m_ref = -INFINITY, l = 0.f;   // this half's running maximum (log2 units) and sum of P
      bool ok = true;
      for (int i = 0; i < sg.n; ++i) {
        const int gi = base + i;
        const int kb = (sg.j0 + i) * kKeys + 64 * h;  // first key of this half
        // Waits are one decision per warp: the TMEM loads and stores below are warp-collective.
        if (!__all_sync(0xFFFFFFFFu, wait(&s_full[gi & 1], uint32_t(gi >> 1) & 1u))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const bool edge = kb + 64 > Pb;               // draft keys or keys past the request
        if (edge && L - kb < 64) {
          // Cache rows past the request's keys may hold anything: zero this
          // half's such rows in the V stage so that P = 0 never meets a
          // non-finite value (thread r takes row 64h + r / 2, dims half r % 2).
          const int s = gi % kStages;
          if (!__all_sync(0xFFFFFFFFu, wait(&vfull[s], uint32_t(gi / kStages) & 1u))) {
            ok = false;
            break;
          }
          if ((r >> 1) >= L - kb) {
            uint8_t* vrow = smem + kVOff + uint32_t(s) * kTile + uint32_t(r & 1) * kHalf + uint32_t(64 * h + (r >> 1)) * 128u;
#pragma unroll
            for (int k = 0; k < 8; ++k) *reinterpret_cast<uint4*>(vrow + k * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        if (warp_live) {
          const uint32_t sc = tmem + lane_off + ((gi & 1) ? kColS1 : kColS0) + uint32_t(64 * h);
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
            if (!__all_sync(0xFFFFFFFFu, wait(&o_done[(gi - 1) & 1], uint32_t((gi - 1) >> 1) & 1u))) {
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
        mbar_arrive(&p_full[(gi & 1) * 2 + h]);
      }
      // Epilogue: merge the halves, O = (2^(ma-M) Oa + 2^(mb-M) Ob) / (2^(ma-M) la + 2^(mb-M) lb).
      // Every softmax thread takes the same barriers, also after a failed wait;
      // a failure anywhere ends the loop for all 256 together.
      const bool fin = __all_sync(0xFFFFFFFFu, ok && wait(o_final, uint32_t(si) & 1u));
      if (named_bar_any(1, 256, !fin)) break;
      xch[h * 128 + r] = make_float2(m_ref, l);
      named_bar_sync(1, 256);
      const float2 other = xch[(1 - h) * 128 + r];
      const float ma = h ? other.x : m_ref, la = h ? other.y : l;
      const float mb = h ? m_ref : other.x, lb = h ? l : other.y;
      const float M = fmaxf(ma, mb);
      const float wa = ma == -INFINITY ? 0.f : fast_exp2(ma - M);
      const float wb = mb == -INFINITY ? 0.f : fast_exp2(mb - M);
      const float den = wa * la + wb * lb;
      // This thread's dims 64h .. 64h+63 of its row.
      float o[64];
      if (sg.n > 0 && warp_live) {
        tc_fence_after();
        uint32_t v[128];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          tmem_ld16(tmem + lane_off + kColOA + uint32_t(64 * h + ch * 16), *reinterpret_cast<uint32_t(*)[16]>(&v[ch * 16]));
          tmem_ld16(tmem + lane_off + kColOB + uint32_t(64 * h + ch * 16),
                    *reinterpret_cast<uint32_t(*)[16]>(&v[64 + ch * 16]));
        }
        tmem_ld_wait128(v);
#pragma unroll
        for (int k = 0; k < 64; ++k) o[k] = wa * __uint_as_float(v[k]) + wb * __uint_as_float(v[64 + k]);
      } else {
#pragma unroll
        for (int k = 0; k < 64; ++k) o[k] = 0.f;
      }
      tc_fence_before();
      // The next segment's request length and parent row are loaded before
      // this segment's stores (a partial result to this CTA's slot), its Q
      // right after them, so that their latency passes under the stores.
      constexpr int kQIter = 128 * 16 / 256;
      uint4 qv[kQIter];
      int pr[4];
      if (has_next) {
        seg_keys(P, nx);
        parent_row(P.parents + size_t(nx.b) * T, T, pr);
      }
      if (!sg.whole) {
        store_partial(P, size_t(blockIdx.x) * 2 + sg.slot, r, h, sg.n > 0 && warp_live ? M : -INFINITY, den, o);
      } else if (valid) {
        store_row(P, sg.b, sg.g, hh, t, h, o, den);
      }
      if (has_next) {
        load_q_regs<256>(P, qv, nx.b, nx.g, nx.tile, threadIdx.x - 128);
        // The next segment's ancestor sets, while the loads are in flight.
        const int rn = nx.tile * 128 + r;
        const bool vn = rn < Rg;
        tree_ancestors(pr, vn ? rn % T : 0, T, vn && nx.n > 0, anc, P.status);
      }
      if (has_next) {
        // Every thread has read the exchange: the Q area takes the next
        // segment's Q, and the MMA issuers may start on it.
        named_bar_sync(1, 256);
        store_q_regs<256>(smem + kQOff, qv, threadIdx.x - 128);
        fence_proxy_async_smem();
        mbar_arrive(seg_ready);
      }
      if (!sg.whole) {
        // Count this segment's key blocks in once every thread's partial is
        // visible. The segment whose count completes the item's nkb blocks
        // merges them all and resets the count.
        fence_acq_rel_gpu();
        named_bar_sync(1, 256);
        if (threadIdx.x == 128) {
          const int add = sg.j1 - sg.j0;
          *merge_here = atomic_add_acq_rel_gpu(&P.cnt[sg.item], add) + add == P.nkb;
        }
        named_bar_sync(1, 256);
        if (*merge_here) {
          fence_acq_rel_gpu();
          if (has_next) {
            // o is not kept past the next segment's loads: this CTA's part is
            // read back from its slot like the others.
#pragma unroll
            for (int k = 0; k < 64; ++k) o[k] = 0.f;
            merge_item(P, sg, r, h, -INFINITY, 0.f, o, false);
          } else {
            merge_item(P, sg, r, h, sg.n > 0 && warp_live ? M : -INFINITY, den, o, true);
          }
          if (threadIdx.x == 128) P.cnt[sg.item] = 0;
        }
      }
      base += sg.n;
      ++si;
      sg = nx;
      pos = pos2;
      more = has_next;
    }
  }

  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

struct AttnPlan {
  int ntile, nkb, ngroups, grid;
  int64_t items;   // (request, kv head, row tile) items
  int64_t U;       // B x Hkv x nkb (request, kv head, key block) units
};

// CTAs whose K/V streams together saturate HBM (each streams one 64 KB block
// per about 0.8 us of tensor and softmax work).
constexpr int64_t kHbmCtas = 80;

// Cost of running the units on ng groups, in key blocks: the longer of the
// longest run (blocks, a start-up of about two blocks per segment, and a merge
// step per other partial of an item) and the HBM time of the K/V blocks plus
// the partial results (written and read back: about two blocks each).
static int64_t plan_cost(const AttnPlan& p, int64_t ng) {
  int64_t worst = 0, max_parts = 1, partials = 0;
  for (int64_t k = 0; k < ng; ++k) {
    const int64_t a = k * p.U / ng, e = (k + 1) * p.U / ng;
    const int64_t segs = (e - 1) / p.nkb - a / p.nkb + 1;
    const int64_t whole = std::max<int64_t>(0, e / p.nkb - (a + p.nkb - 1) / p.nkb);
    partials += segs - whole;
    worst = std::max(worst, (e - a) + 2 * segs);
  }
  const int64_t kvh = p.U / p.nkb;
  for (int64_t it = 0; it < kvh && it < 4096; ++it) {
    const int64_t x0 = it * p.nkb, x1 = x0 + p.nkb - 1;
    max_parts = std::max(max_parts, ((x1 + 1) * ng - 1) / p.U - ((x0 + 1) * ng - 1) / p.U + 1);
  }
  const int64_t crit = worst + (max_parts > 1 ? 2 * (max_parts - 1) : 0);
  const int64_t hbm = (p.U + 2 * partials * p.ntile) / kHbmCtas;
  return std::max(crit, hbm);
}

// Work split over the CTAs: even runs of units (stream-K) on as many groups of
// ntile CTAs as the SMs hold, or on a whole multiple of the (request, kv head)
// count below that (fewer or no partials), whichever the cost model rates lower.
static AttnPlan plan_attn(int B, int T, int Hq, int Hkv, int64_t max_len, int sms) {
  AttnPlan p{};
  const int G = Hq / Hkv;
  p.ntile = (G * T + 127) / 128;
  p.nkb = int((max_len + kKeys - 1) / kKeys);
  p.items = int64_t(B) * Hkv * p.ntile;
  const int64_t kvh = int64_t(B) * Hkv;
  p.U = kvh * p.nkb;
  const int64_t gmax = std::max<int64_t>(1, std::min<int64_t>(sms / p.ntile, p.U));
  int64_t best_cost = plan_cost(p, gmax);
  p.ngroups = int(gmax);
  for (int64_t ng = kvh; ng < gmax; ng += kvh) {
    const int64_t cost = plan_cost(p, ng);
    if (cost < best_cost) {
      best_cost = cost;
      p.ngroups = int(ng);
    }
  }
  p.grid = p.ngroups * p.ntile;
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

// Whether some CTA's run starts inside an item (then items are merged from partials).
static bool has_partials(const AttnPlan& p) {
  for (int k = 1; k < p.ngroups; ++k)
    if ((int64_t(k) * p.U / p.ngroups) % p.nkb != 0) return true;
  return false;
}

static size_t part_o_bytes(const AttnPlan& p) { return size_t(p.grid) * 2 * 128 * kD * 2; }
static size_t part_ml_bytes(const AttnPlan& p) { return size_t(p.grid) * 2 * 128 * sizeof(float2); }
static size_t part_sc_bytes(const AttnPlan& p) { return size_t(p.grid) * 2 * 2 * 128 * sizeof(float); }

static size_t ws_bytes_of(const AttnPlan& p) {
  if (!has_partials(p)) return 256;
  return part_o_bytes(p) + part_ml_bytes(p) + part_sc_bytes(p) + size_t(p.items) * sizeof(int32_t) + 256;
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
  if (pl.items > 0x7FFFFFFF || pl.U > (int64_t(1) << 40)) return W12_ERR_SHAPE;
  const bool parts = has_partials(pl);
  if (parts && (!ws || !aligned(ws, 16) || ws_bytes < ws_bytes_of(pl))) return W12_ERR_WORKSPACE;

  AttnParams P{};
  P.Q = Q;
  P.O = O;
  P.prefix_len = prefix_len;
  P.parents = parents;
  if (parts) {
    uint8_t* w = static_cast<uint8_t*>(ws);
    P.part_o = reinterpret_cast<uint4*>(w);
    P.part_ml = reinterpret_cast<float2*>(w + part_o_bytes(pl));
    P.part_sc = reinterpret_cast<float*>(w + part_o_bytes(pl) + part_ml_bytes(pl));
    P.cnt = reinterpret_cast<int32_t*>(w + part_o_bytes(pl) + part_ml_bytes(pl) + part_sc_bytes(pl));
  }
  P.status = dev_status;
  P.B = B;
  P.T = T;
  P.Hq = Hq;
  P.Hkv = Hkv;
  P.G = Hq / Hkv;
  P.ntile = pl.ntile;
  P.nkb = pl.nkb;
  P.U = pl.U;
  P.ngroups = pl.ngroups;
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
  cfg.gridDim = dim3(unsigned(pl.grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_enabled() ? 1 : 0;
  return cuda_status(cudaLaunchKernelEx(&cfg, attn_kernel, tk, tv, P));
}

}  // extern "C"
