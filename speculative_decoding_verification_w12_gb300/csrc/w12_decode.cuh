// Decode warps of the W12 GEMM kernels (the single-GEMM kernel and the grouped
// one share this code): the loop that restores each unit's 128 x 128 bf16
// weights from the three 4-bit planes in a shared-memory stage, patches the
// unit's exception entries in, and stores the result as the MMA's A operand
// in tensor memory.
//
// A unit's row r (one thread's W row) is 128 values: 64 bytes in each plane
// (`planes` at stage + r * 64 in 8 KB planes, 128-byte swizzle in 16-byte
// chunks), the group's exponent base in the stage's ebase bytes. Exception
// entry e (row << 23 | col << 16 | bits16, row and col within the unit) sets
// value (row, col) to its 16 stored bits; an entry with a row field >= 128
// (bits 31..30 set) is corrupt: never applied, and reported by the caller
// from the OR of the entries read. Entries of a unit are read from the
// staged window in shared memory when it fits, else from global memory.
#pragma once

#include "w12_dev.cuh"
#include "w12_host.h"

namespace w12 {

#ifndef W12_DEC_GROUPS
#define W12_DEC_GROUPS 2
#endif
#ifndef W12_DEC_SPLIT
#define W12_DEC_SPLIT 1
#endif
static_assert(W12_DEC_GROUPS >= 1 && W12_DEC_GROUPS <= 3, "decode groups: 1..3");
static_assert(W12_DEC_SPLIT == 1 || W12_DEC_SPLIT == 2 || W12_DEC_SPLIT == 4, "decode split: 1, 2 or 4");
constexpr int kDecGroups = W12_DEC_GROUPS;       // decode groups: group g takes units g, g + kDecGroups, ...
constexpr int kDecSplit = W12_DEC_SPLIT;         // warps sharing one unit row
constexpr int kAColsPerBuf = 64;                 // 128 K values = 64 TMEM columns of bf16 pairs
constexpr uint32_t kInvalidEnt = 0xFFFFFFFFu;
// From kWideMinMpad padded rows (a ring of two or three stages, so a unit's
// restore sits on the critical path) the kernels lay the same decode warps
// out as one group of kWideSplit warps per lane quarter instead of kDecGroups
// groups: one unit at a time, each restored kWideSplit times sooner.
constexpr int kWideMinMpad = 128;
constexpr int kWideSplit = kDecGroups * kDecSplit;
static_assert(kWideSplit == 1 || kWideSplit == 2 || kWideSplit == 4, "wide decode layout");

// A CTA's exception window over units [ub, ub + n) of one problem, staged by
// one warp (all 32 lanes): the n + 1 offsets exc_off[ub ..] into soff (n + 1
// <= kOffCap, which the host checks), and the entries they span,
// exc_ent[e0 .. e1), into sent when they fit (kEntCap). Every load of a batch
// is issued before the batch's first store, so the window costs one memory
// round trip per batch rather than one per 32 values (the decoders cannot
// start before it is done). bad: the window's ends are inconsistent (e1 < e0
// or past n_exc).
struct ExcWindow {
  uint32_t e0, e1;
  bool bad, fits;
};

__device__ __forceinline__ ExcWindow stage_window(const uint32_t* exc_off, const uint32_t* exc_ent, int64_t n_exc,
                                                  int64_t ub, int n, uint32_t* soff, uint32_t* sent) {
  const int lane = threadIdx.x & 31;
  const int nwin = n + 1;
  {
    uint32_t v[kOffCap / 32];
#pragma unroll
    for (int j = 0; j < kOffCap / 32; ++j)
      if (lane + 32 * j < nwin) v[j] = exc_off[ub + lane + 32 * j];
#pragma unroll
    for (int j = 0; j < kOffCap / 32; ++j)
      if (lane + 32 * j < nwin) soff[lane + 32 * j] = v[j];
  }
  __syncwarp();
  ExcWindow w;
  w.e0 = soff[0];
  w.e1 = soff[nwin - 1];
  w.bad = w.e1 < w.e0 || int64_t(w.e1) > n_exc;
  w.fits = !w.bad && (w.e1 - w.e0) <= uint32_t(kEntCap);
  if (w.fits) {
    constexpr int kBatch = 16;  // entries per lane in flight
    const uint32_t cnt = w.e1 - w.e0;
    for (uint32_t b0 = 0; b0 < cnt; b0 += 32 * kBatch) {
      uint32_t v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (b0 + lane + 32 * j < cnt) v[j] = exc_ent[w.e0 + b0 + lane + 32 * j];
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (b0 + lane + 32 * j < cnt) sent[b0 + lane + 32 * j] = v[j];
    }
  }
  __syncwarp();
  return w;
}

// What the decode loop needs from its kernel.
struct DecodeCtx {
  const uint8_t* smem;       // stage 0 (stages stage_bytes apart)
  uint32_t stage_bytes;
  uint32_t eb_off;           // the stage's ebase bytes (one per row)
  int S;                     // ring stages
  int n_units;               // units of this CTA
  uint64_t* full;            // [S] weight bytes of a stage landed
  uint64_t* a_full;          // [S] decoded A of a stage stored (128 * split width arrivals)
  uint32_t a_tmem;           // TMEM address of A buffer 0 at this warp's lane quarter
  const uint32_t* soff;      // per unit: first entry position (n_units + 1 values)
  const uint32_t* sent;      // staged entries (when in_smem)
  uint32_t e_base;           // position of sent[0]
  bool in_smem;
  int32_t* status;
};

// The decode warp's loop. dw = warp index among the decode warps. wait(bar,
// parity) is the kernel's bounded wait (false: give up); bad(i, o0, o1) says
// whether unit i's entry positions [o0, o1) fail a consistency check (then the
// unit is decoded without exceptions and W12_ERR_CORRUPT is set); gptr(i)
// gives the pointer p with entry position o of unit i at p[o] when entries are
// not staged. Returns the OR of the entries read.
//
// kGroups x kSplitW sets how the 4 * kGroups * kSplitW decode warps share the
// work (a_full counts 128 * kSplitW arrivals): more groups decode more units
// at once, a wider split restores each unit sooner.
template <int kGroups = kDecGroups, int kSplitW = kDecSplit, class Wait, class Bad, class Gptr>
__device__ __forceinline__ uint32_t decode_units(const DecodeCtx& c, int dw, Wait&& wait, Bad&& bad, Gptr&& gptr) {
  static_assert(kGroups >= 1 && (kSplitW == 1 || kSplitW == 2 || kSplitW == 4), "decode layout");
  constexpr int kChunksPerThread = 4 / kSplitW;
  const int lane = threadIdx.x & 31;
  const int q = (threadIdx.x >> 5) & 3;       // TMEM lane quarter of this warp
  const int grp = (dw >> 2) / kSplitW;        // decode group
  const int h = (dw >> 2) % kSplitW;          // slice of the unit row (kChunksPerThread chunks of 32 values)
  const int row = q * 32 + lane;              // W row within the unit
  const uint32_t tm_a = c.a_tmem + (uint32_t(q * 32) << 16);
  uint32_t seen = 0;

  // Exceptions of unit i that fall in this warp's rows: the lane-held entry
  // (first 32 of the unit) and one ballot mask per 32-value chunk. Prepared
  // one unit ahead so this bookkeeping overlaps the previous unit's stores.
  struct Exc {
    uint32_t o0, o1, ent, mask[kChunksPerThread];
  };
  auto prep = [&](int i, Exc& x) {
    x.o0 = c.soff[i];
    x.o1 = c.soff[i + 1];
    if (bad(i, x.o0, x.o1)) {
      if (lane == 0) set_status(c.status, W12_ERR_CORRUPT);
      x.o1 = x.o0;
    }
    const uint32_t nex = x.o1 - x.o0;
    x.ent = kInvalidEnt;
#pragma unroll
    for (int cc = 0; cc < kChunksPerThread; ++cc) x.mask[cc] = 0;
    if (nex > 0) {
      if (uint32_t(lane) < nex) {
        const uint32_t v = c.in_smem ? c.sent[x.o0 - c.e_base + lane] : __ldg(gptr(i) + x.o0 + lane);
        seen |= v;
        x.ent = (v >> 30) ? kInvalidEnt : v;
      }
      const bool mine = x.ent != kInvalidEnt && ((x.ent >> 28) & 3u) == uint32_t(q);
      const uint32_t ch = (x.ent >> 21) & 3u;
#pragma unroll
      for (int cc = 0; cc < kChunksPerThread; ++cc)
        x.mask[cc] = __ballot_sync(0xFFFFFFFFu, mine && ch == uint32_t(h * kChunksPerThread + cc));
    }
  };
  Exc cur;
  if (grp < c.n_units) prep(grp, cur);

  int s = 0;
  uint32_t ph = 0;
  for (int k = 0; k < grp; ++k)
    if (++s == c.S) {
      s = 0;
      ph ^= 1u;
    }
  for (int i = grp; i < c.n_units; i += kGroups) {
    // Stage s's copies can only have landed after the MMA that last read
    // its TMEM A buffer committed, so the buffer is free once this returns.
    // One decision per warp: the loop uses warp-collective instructions.
    if (!__all_sync(0xFFFFFFFFu, wait(&c.full[s], ph))) break;
    tc_fence_after();
    const uint8_t* st = c.smem + s * c.stage_bytes;
    const uint8_t* pl = st + row * 64;
    const uint32_t swz = uint32_t(row >> 1) & 3u;
    uint4 a[kChunksPerThread], b[kChunksPerThread], g[kChunksPerThread];
#pragma unroll
    for (int cc = 0; cc < kChunksPerThread; ++cc) {
      const uint32_t off = ((uint32_t(h * kChunksPerThread + cc) ^ swz) << 4);
      a[cc] = *reinterpret_cast<const uint4*>(pl + off);
      b[cc] = *reinterpret_cast<const uint4*>(pl + 8192 + off);
      g[cc] = *reinterpret_cast<const uint4*>(pl + 16384 + off);
    }
    const uint32_t eb = st[c.eb_off + row];
    const uint32_t E2 = (eb << 7) * 0x00010001u;

#pragma unroll
    for (int cc = 0; cc < kChunksPerThread; ++cc) {
      const uint32_t lc = uint32_t(h * kChunksPerThread + cc);  // 16-byte plane chunk = 32 values
      uint32_t w[16];
      decode8(a[cc].x, b[cc].x, g[cc].x, E2, w + 0);
      decode8(a[cc].y, b[cc].y, g[cc].y, E2, w + 4);
      decode8(a[cc].z, b[cc].z, g[cc].z, E2, w + 8);
      decode8(a[cc].w, b[cc].w, g[cc].w, E2, w + 12);
      if (kSplitW <= 2) {
        if (cur.mask[cc] != 0u) {
          // Patch through shared memory: the chunk's 16 words go to bytes of
          // the stage that only this thread reads and has already loaded (its
          // own row's slices of the planes), the lane holding each exception
          // of the chunk stores its 16 bits at the target (row, column), and
          // the words are read back. Scratch slot k (16 bytes) is plane
          // k / kChunksPerThread, chunk slice h * kChunksPerThread + k %
          // kChunksPerThread of the row, in the planes' swizzle.
          uint8_t* const stw = const_cast<uint8_t*>(st);
          auto slot_addr = [&](uint32_t r, uint32_t k) {
            return stw + (k / kChunksPerThread) * 8192u + r * 64u +
                   (((uint32_t(h * kChunksPerThread) + k % kChunksPerThread) ^ ((r >> 1) & 3u)) << 4);
          };
#pragma unroll
          for (int k = 0; k < 4; ++k)
            *reinterpret_cast<uint4*>(slot_addr(uint32_t(row), uint32_t(k))) =
                make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
          __syncwarp();
          if ((cur.mask[cc] >> lane) & 1u) {
            const uint32_t col = (cur.ent >> 16) & 31u;  // byte 2 * col of the chunk's 64
            const uint32_t r = uint32_t(q * 32) + ((cur.ent >> 23) & 31u);
            *reinterpret_cast<uint16_t*>(slot_addr(r, col >> 3) + ((col & 7u) << 1)) = uint16_t(cur.ent & 0xFFFFu);
          }
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 v = *reinterpret_cast<const uint4*>(slot_addr(uint32_t(row), uint32_t(k)));
            w[4 * k] = v.x, w[4 * k + 1] = v.y, w[4 * k + 2] = v.z, w[4 * k + 3] = v.w;
          }
        }
      } else {
        uint32_t mk = cur.mask[cc];
        while (mk) {
          const int src = __ffs(mk) - 1;
          mk &= mk - 1;
          const uint32_t e = __shfl_sync(0xFFFFFFFFu, cur.ent, src);
          if (uint32_t(lane) == ((e >> 23) & 31u)) patch_word(w, (e >> 16) & 31u, e & 0xFFFFu);
        }
      }
      if (cur.o1 - cur.o0 > 32) {
        // Rare: more than 32 exceptions in the unit; walk the rest in batches.
        for (uint32_t bst = cur.o0 + 32; bst < cur.o1; bst += 32) {
          uint32_t e2 = kInvalidEnt;
          if (bst + lane < cur.o1) {
            const uint32_t v = c.in_smem ? c.sent[bst - c.e_base + lane] : __ldg(gptr(i) + bst + lane);
            seen |= v;
            e2 = (v >> 30) ? kInvalidEnt : v;
          }
          const bool mine2 = e2 != kInvalidEnt && ((e2 >> 28) & 3u) == uint32_t(q) && ((e2 >> 21) & 3u) == lc;
          uint32_t mk2 = __ballot_sync(0xFFFFFFFFu, mine2);
          while (mk2) {
            const int src = __ffs(mk2) - 1;
            mk2 &= mk2 - 1;
            const uint32_t e = __shfl_sync(0xFFFFFFFFu, e2, src);
            if (uint32_t(lane) == ((e >> 23) & 31u)) patch_word(w, (e >> 16) & 31u, e & 0xFFFFu);
          }
        }
      }
      tmem_st16(tm_a + uint32_t(s * kAColsPerBuf) + lc * 16u, w);
    }
    if (i + kGroups < c.n_units) prep(i + kGroups, cur);  // overlaps the stores in flight
    tmem_st_wait();
    tc_fence_before();
    // This thread's reads of the stage (generic proxy) come before the copy
    // (async proxy) that refills it once the MMA has committed. Without the
    // fence, a refill issued soon after the reads was seen to land under
    // them in about 1 % of launches.
    fence_proxy_async_smem();
    mbar_arrive(&c.a_full[s]);
    for (int k = 0; k < kGroups; ++k)
      if (++s == c.S) {
        s = 0;
        ph ^= 1u;
      }
  }
  return seen;
}

}  // namespace w12
