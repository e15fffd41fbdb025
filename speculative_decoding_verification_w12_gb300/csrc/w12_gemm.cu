// W12 verify GEMM and the in-tree BF16 baseline on sm_103a.
//
// Y[M, N] = X[M, K] * W[N, K]^T with M (verified rows) small: the verify pass
// streams every target weight to score a 16-token draft block (SpecPilot
// paper digest, summary paragraph), so the kernel is bound by HBM reads of W.
// W is stored in W12 and restored bitwise in registers before the tensor-core
// contraction (SpecPilot digest, "Reasons" bullet 2).
//
// Design (one persistent CTA per SM, stream-K over 128x128 units of W):
//   warp 0      TMA producer: three plane tiles (3 x 128x64 B, 64-byte
//               swizzle), the 128 ebase bytes, and the X tile (2 boxes of
//               Mpad x 64 bf16, 128-byte swizzle) per unit into a smem ring.
//   warp 1      MMA issuer (one thread): swap-AB tcgen05.mma kind::f16,
//               D[128 x Mpad] (TMEM, fp32) += A[128 x 16] (TMEM, decoded W)
//               x B[16 x Mpad] (smem, X), 8 instructions per unit.
//   warp 2      TMEM allocation / release.
//   warp 3      stages the CTA's exception offsets and entries in smem.
//   decode warps (4 + 4*groups*split of them): each thread restores its
//               row's share of the unit from the planes (LDS.128), patches
//               exceptions in registers, and writes bf16 pairs into TMEM
//               (tcgen05.st); decode groups take units in turn (at large M
//               one group of wider split restores each unit sooner).
//   last 4 warps epilogue: tcgen05.ld of the accumulator; unsplit tiles write
//               Y directly; split tiles write partial slots and the last CTA
//               to arrive sums them in a fixed order (deterministic).
// The BF16 baseline uses the same skeleton with A loaded by TMA into smem.
// In argmax mode (fused LM head) the epilogue reduces each 128-row vocab
// tile to a per-row (max, index) pair instead of writing logits.
#include "w12_decode.cuh"
#include "w12_dev.cuh"
#include "w12_host.h"

namespace w12 {

// Decode warps: W12_DEC_GROUPS groups of 4 x W12_DEC_SPLIT warps. Each warp
// serves one TMEM lane quarter (32 rows); the W12_DEC_SPLIT warps of a
// quarter in a group split the unit's 4 chunks of 32 values; groups take
// units in turn (unit i goes to group i % W12_DEC_GROUPS).
constexpr int kMaxStages = 8;         // smem ring depth limit (one TMEM A buffer per stage)
constexpr int kEpiBar = 1;            // named barrier id of the epilogue warps
constexpr int kScratchStride = 129;   // floats per column in the argmax transpose buffer
constexpr int kDeferMinMpad = 128;    // from this many padded rows, split tiles may be summed by a second kernel

struct GemmParams {
  int M, Mpad, N, K, KB, tiles, grid, stages, issuers;
  int defer;  // split tiles only write their partials; splitk_reduce_kernel sums them
  int64_t units;
  const uint8_t* ebase;
  const uint32_t* exc_off;
  const uint32_t* exc_ent;
  int64_t n_exc;
  float* Y;
  float* parts;
  int32_t* counters;
  float* amax_val;
  int32_t* amax_idx;
  int32_t* status;
  uint64_t limit_ns;
};

template <bool kW12>
struct Cfg {
  static constexpr int kDecWarps = kW12 ? 4 * kDecGroups * kDecSplit : 0;
  static constexpr int kEpiWarp0 = 4 + kDecWarps;
  static constexpr int kThreads = (kEpiWarp0 + 4) * 32;
  static constexpr uint32_t kABytes = kW12 ? 3 * 8192 : 2 * 16384;  // A operand bytes per stage
  static constexpr uint32_t kEbBytes = kW12 ? 1024 : 0;             // ebase (128 B used)
  static constexpr uint32_t kTmemCols = kW12 ? 512 : 256;
};

// Shared memory carve-up (identical on host and device).
struct SmemPlan {
  uint32_t stage_bytes, x_off, eb_off, stages;
  uint32_t scratch_off, red_off, soff_off, sent_off, bar_off, misc_off, total;
};

template <bool kW12>
__host__ __device__ inline SmemPlan smem_plan(int Mpad, int stages) {
  SmemPlan p;
  p.eb_off = Cfg<kW12>::kABytes;
  p.x_off = p.eb_off + Cfg<kW12>::kEbBytes;
  p.stage_bytes = p.x_off + 2u * Mpad * 128u;
  p.stages = stages;
  uint32_t off = p.stage_bytes * stages;
  p.scratch_off = off;
  off += 16 * kScratchStride * 4;
  p.red_off = off;
  off += 4 * 16 * 8;
  p.soff_off = off;
  off += kW12 ? (kOffCap + 4) * 4 : 0;
  p.sent_off = off;
  off += kW12 ? kEntCap * 4 : 0;
  off = (off + 15) & ~15u;
  p.bar_off = off;
  off += 64 * 8;
  p.misc_off = off;
  off += 64;
  p.total = off + 1024;  // slack for 1024-byte alignment of the base
  return p;
}

__device__ __forceinline__ int64_t unit_begin(int c, int64_t U, int G) { return int64_t(c) * U / G; }

// CTA that owns unit u: the largest c with floor(c*U/G) <= u.
__device__ __forceinline__ int unit_owner(int64_t u, int64_t U, int G) {
  return static_cast<int>(((u + 1) * G + U - 1) / U - 1);
}

struct Bars {
  uint64_t* full;
  uint64_t* empty;
  uint64_t* a_full;
  uint64_t* acc_full;
  uint64_t* acc_empty;
  uint64_t* exc_ready;
  uint64_t* drain;
  uint64_t* gather;
};

template <bool kW12, bool kArgmax, bool kWide>
__global__ void __launch_bounds__(Cfg<kW12>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
                const __grid_constant__ CUtensorMap tm_a2, const __grid_constant__ CUtensorMap tm_x,
                const GemmParams P) {
  using C = Cfg<kW12>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const SmemPlan plan = smem_plan<kW12>(P.Mpad, P.stages);
  const int S = P.stages;
  const int NACC = P.Mpad <= 128 ? 2 : 1;

  uint64_t* bar_base = reinterpret_cast<uint64_t*>(smem + plan.bar_off);
  Bars B;
  B.full = bar_base;
  B.empty = bar_base + S;
  B.a_full = bar_base + 2 * S;
  B.acc_full = B.a_full + S;
  B.acc_empty = B.acc_full + 2;
  B.exc_ready = B.acc_empty + 2;
  B.drain = B.exc_ready + 1;
  B.gather = B.drain + 1;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + plan.misc_off);
  volatile uint32_t* tmem_slot = misc + 0;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(misc + 2);
  volatile int* ent_in_smem = reinterpret_cast<volatile int*>(misc + 3);
  volatile uint32_t* ent_base = misc + 4;
  volatile uint32_t* ent_end = misc + 5;
  volatile int* pref_flag = reinterpret_cast<volatile int*>(misc + 6);
  volatile int* fast_flag = reinterpret_cast<volatile int*>(misc + 7);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int64_t U = P.units;
  const int G = P.grid;
  const int64_t ub = unit_begin(c, U, G), ue = unit_begin(c + 1, U, G);
  const int KB = P.KB;
  const uint64_t lim = P.limit_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&B.full[s], 1);
      mbar_init(&B.empty[s], 1);
    }
    if (kW12) {  // decoded-operand handshakes exist only when there are decode warps
      for (int a = 0; a < S; ++a) mbar_init(&B.a_full[a], 128 * (kWide ? kWideSplit : kDecSplit));
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&B.acc_full[a], P.issuers);  // one commit per MMA issuer per segment
      mbar_init(&B.acc_empty[a], 128);
    }
    mbar_init(B.exc_ready, 1);
    mbar_init(B.drain, P.issuers);
    mbar_init(B.gather, 1);
    *abort_flag = 0;
    *last_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(const_cast<uint32_t*>(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // TMEM columns: accumulators [0, NACC*issuers*Mpad) (buffer b, issuer k at
  // column (b*issuers + k)*Mpad), then one 64-column A buffer per stage.
  const int NISS = P.issuers;
  const uint32_t a_col0 = uint32_t((NACC * NISS * P.Mpad + 63) & ~63);

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

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      prefetch_tmap(&tm_x);
      prefetch_tmap(&tm_a0);
      if (kW12) {
        prefetch_tmap(&tm_a1);
        prefetch_tmap(&tm_a2);
      }
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      const uint32_t xbox = uint32_t(P.Mpad) * 128u;
      const uint32_t tx = C::kABytes + (kW12 ? 128u : 0u) + 2u * xbox;
      // Per-unit state kept incrementally in 32-bit registers (no 64-bit
      // division in this single-thread loop).
      int t = int(ub / KB), kb = int(ub % KB);
      const int n_units = int(ue - ub);
      // The first ring-full of weight tiles is requested before waiting for
      // the previous kernel on the stream (launch overlap); X is loaded, and
      // anything else is read or written, only after that wait.
      const int prefill = n_units < S ? n_units : S;
      {
        int t0 = t, kb0 = kb;
        for (int i = 0; i < prefill; ++i) {
          uint8_t* st = smem + i * plan.stage_bytes;
          mbar_arrive_expect_tx(&B.full[i], tx);
          if (kW12) {
            tma_load_2d_hint(st, &tm_a0, kb0 * 64, t0 * 128, &B.full[i], pol_w);
            tma_load_2d_hint(st + 8192, &tm_a1, kb0 * 64, t0 * 128, &B.full[i], pol_w);
            tma_load_2d_hint(st + 16384, &tm_a2, kb0 * 64, t0 * 128, &B.full[i], pol_w);
            bulk_load(st + plan.eb_off, P.ebase + int64_t(kb0) * P.N + int64_t(t0) * 128, 128u, &B.full[i]);
          } else {
            tma_load_2d_hint(st, &tm_a0, kb0 * 128, t0 * 128, &B.full[i], pol_w);
            tma_load_2d_hint(st + 16384, &tm_a0, kb0 * 128 + 64, t0 * 128, &B.full[i], pol_w);
          }
          if (++kb0 == KB) {
            kb0 = 0;
            ++t0;
          }
        }
      }
      grid_dep_wait();
      int s = 0;
      uint32_t ph = 0;
      int issued = 0;
      for (; issued < n_units; ++issued) {
        uint8_t* st = smem + s * plan.stage_bytes;
        if (issued >= prefill) {
          if (!wait(&B.empty[s], ph ^ 1u)) break;
          mbar_arrive_expect_tx(&B.full[s], tx);
          if (kW12) {
            tma_load_2d_hint(st, &tm_a0, kb * 64, t * 128, &B.full[s], pol_w);
            tma_load_2d_hint(st + 8192, &tm_a1, kb * 64, t * 128, &B.full[s], pol_w);
            tma_load_2d_hint(st + 16384, &tm_a2, kb * 64, t * 128, &B.full[s], pol_w);
            bulk_load(st + plan.eb_off, P.ebase + int64_t(kb) * P.N + int64_t(t) * 128, 128u, &B.full[s]);
          } else {
            tma_load_2d_hint(st, &tm_a0, kb * 128, t * 128, &B.full[s], pol_w);
            tma_load_2d_hint(st + 16384, &tm_a0, kb * 128 + 64, t * 128, &B.full[s], pol_w);
          }
        }
        tma_load_2d_hint(st + plan.x_off, &tm_x, kb * 128, 0, &B.full[s], pol_x);
        tma_load_2d_hint(st + plan.x_off + xbox, &tm_x, kb * 128 + 64, 0, &B.full[s], pol_x);
        if (++kb == KB) {
          kb = 0;
          ++t;
        }
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      grid_dep_launch();
      if (*abort_flag) {
        // Let the copies already issued land before the CTA can exit.
        for (int i = issued > S ? issued - S : 0; i < issued; ++i)
          mbar_wait(&B.full[i % S], uint32_t(i / S) & 1u, drain_limit_ns(lim));
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------------ MMA
    // Issuer k (warp 1 + k, one thread) takes the units i with i % issuers == k
    // into its own accumulator: one thread can only issue a kind::f16 MMA
    // every few tens of cycles, so two issuers double the issue rate.
    const int k = warp - 1;
    if (lane == 0 && k < NISS) {
      const uint32_t idesc = idesc_bf16(128, uint32_t(P.Mpad));
      const uint32_t xbox = uint32_t(P.Mpad) * 128u;
      // Descriptors of stage 0; other stages and K steps add (byte offset >> 4)
      // to the 14-bit start-address field, which cannot overflow (smem < 256 KB).
      const uint32_t st0 = smem_u32(smem);
      const uint64_t bdesc0 = sdesc_k_sw128(st0 + plan.x_off);
      const uint64_t adesc0 = sdesc_k_sw128(st0);
      const uint32_t a_tmem0 = tmem_base + a_col0;
      const int n_units = int(ue - ub);
      int kb = int(ub % KB);
      int s = 0, accb = 0;
      uint32_t ph = 0, accph = 0;
      bool started = false;  // this issuer has written its accumulator in the current segment
      for (int i = 0; i < n_units; ++i) {
        const bool first = (i == 0) || (kb == 0);
        const bool last = (i + 1 == n_units) || (kb + 1 == KB);
        if (first) {
          if (!wait(&B.acc_empty[accb], accph ^ 1u)) break;
          tc_fence_after();
          started = false;
        }
        if (i % NISS == k) {
          // W12: the decoders waited for the stage's copies before arriving on
          // a_full, so "decoded" implies "landed" for X as well.
          if (kW12 ? !wait(&B.a_full[s], ph) : !wait(&B.full[s], ph)) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + uint32_t(accb * NISS + k) * uint32_t(P.Mpad);
          const uint64_t soff16 = uint64_t((uint32_t(s) * plan.stage_bytes) >> 4);
          const uint32_t a_tmem = a_tmem0 + uint32_t(s * kAColsPerBuf);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t koff = uint64_t(((uint32_t(kk >> 2) * xbox) + uint32_t(kk & 3) * 32u) >> 4);
            const uint64_t bdesc = bdesc0 + soff16 + koff;
            const uint32_t acc = (started || kk > 0) ? 1u : 0u;
            if (kW12) {
              mma_bf16_ts(d_tmem, a_tmem + uint32_t(kk * 8), bdesc, idesc, acc);
            } else {
              const uint64_t aoff = uint64_t((uint32_t(kk >> 2) * 16384u + uint32_t(kk & 3) * 32u) >> 4);
              mma_bf16_ss(d_tmem, adesc0 + soff16 + aoff, bdesc, idesc, acc);
            }
          }
          started = true;
          tc_commit(&B.empty[s]);  // frees the smem stage and its TMEM A buffer
        }
        if (last) {
          tc_commit(&B.acc_full[accb]);  // every issuer arrives once per segment
          if (++accb == NACC) {
            accb = 0;
            accph ^= 1u;
          }
        }
        if (++kb == KB) kb = 0;
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      // Make sure no MMA is in flight before TMEM is released.
      tc_commit(B.drain);
      mbar_wait(B.drain, 0, drain_limit_ns(lim));
    }
  } else if (warp == 3) {
    // ---------------------------------------------- exception metadata (W12)
    if (kW12) {
      const ExcWindow w = stage_window(P.exc_off, P.exc_ent, P.n_exc, ub, int(ue - ub),
                                       reinterpret_cast<uint32_t*>(smem + plan.soff_off),
                                       reinterpret_cast<uint32_t*>(smem + plan.sent_off));
      if (lane == 0) {
        if (w.bad) set_status(P.status, W12_ERR_CORRUPT);
        *ent_in_smem = w.fits ? 1 : 0;
        *ent_base = w.e0;
        *ent_end = w.bad ? w.e0 : w.e1;
        mbar_arrive(B.exc_ready);
      }
    }
  } else if (kW12 && warp >= 4 && warp < 4 + C::kDecWarps) {
    // --------------------------------------------------------------- decode
    // One decision per warp: the decode loop uses warp-collective instructions.
    if (__all_sync(0xFFFFFFFFu, wait(B.exc_ready, 0))) {
      DecodeCtx d;
      d.smem = smem;
      d.stage_bytes = plan.stage_bytes;
      d.eb_off = plan.eb_off;
      d.S = S;
      d.n_units = int(ue - ub);
      d.full = B.full;
      d.a_full = B.a_full;
      d.a_tmem = tmem_base + a_col0;
      d.soff = reinterpret_cast<const uint32_t*>(smem + plan.soff_off);
      d.sent = reinterpret_cast<const uint32_t*>(smem + plan.sent_off);
      d.e_base = *ent_base;
      d.in_smem = *ent_in_smem;
      d.status = P.status;
      const uint32_t e_end = *ent_end;
      const uint32_t seen = decode_units<kWide ? 1 : kDecGroups, kWide ? kWideSplit : kDecSplit>(
          d, warp - 4, wait,
          [&](int, uint32_t o0, uint32_t o1) {
            return o1 < o0 || int64_t(o1) > P.n_exc || o0 < d.e_base || o1 > e_end;
          },
          [&](int) { return P.exc_ent; });
      // Every entry of the window is read by a decode warp: a corrupt one
      // (row field >= 128) shows in the OR.
      if ((seen >> 30) != 0) set_status(P.status, W12_ERR_CORRUPT);
    }
  } else if (warp >= C::kEpiWarp0) {
    // ------------------------------------------------------------- epilogue
    const int ew = warp & 3;            // TMEM lane quarter
    const int row = ew * 32 + lane;
    const uint32_t tm_lane = uint32_t(ew * 32) << 16;
    const int et = threadIdx.x - C::kEpiWarp0 * 32;  // 0..127
    float* scratch = reinterpret_cast<float*>(smem + plan.scratch_off);
    float* red_v = reinterpret_cast<float*>(smem + plan.red_off);
    int32_t* red_i = reinterpret_cast<int32_t*>(smem + plan.red_off + 4 * 16 * 4);
    const int first_tile = int(ub / KB);
    const int nchunks = P.Mpad / 16;

    // Tile argmax over a 16-column chunk: v[r] = logit of vocab row `row`
    // for token mc*16 + r. Lowest vocab index wins ties.
    auto argmax_chunk = [&](const float (&v)[16], int t, int mc) {
#pragma unroll
      for (int r = 0; r < 16; ++r) scratch[r * kScratchStride + row] = v[r];
      named_bar_sync(kEpiBar, 128);
      if (lane < 16) {
        const float* col = scratch + lane * kScratchStride + ew * 32;
        float best = col[0];
        int bi = 0;
        for (int k = 1; k < 32; ++k) {
          const float x = col[k];
          if (x > best) {
            best = x;
            bi = k;
          }
        }
        red_v[ew * 16 + lane] = best;
        red_i[ew * 16 + lane] = ew * 32 + bi;
      }
      named_bar_sync(kEpiBar, 128);
      if (ew == 0 && lane < 16) {
        float best = red_v[lane];
        int bi = red_i[lane];
        for (int w2 = 1; w2 < 4; ++w2) {
          const float x = red_v[w2 * 16 + lane];
          if (x > best) {
            best = x;
            bi = red_i[w2 * 16 + lane];
          }
        }
        const int m = mc * 16 + lane;
        P.amax_val[int64_t(t) * P.Mpad + m] = best;
        P.amax_idx[int64_t(t) * P.Mpad + m] = t * 128 + bi;
      }
      named_bar_sync(kEpiBar, 128);
    };
    auto store_chunk = [&](const float (&v)[16], int t, int mc) {
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const int m = mc * 16 + r;
        if (m < P.M) P.Y[int64_t(m) * P.N + int64_t(t) * 128 + row] = v[r];
      }
    };

    grid_dep_wait();
    int accb = 0;
    uint32_t accph = 0;
    int gather_pending = -1;  // phase of a gather of partials that was given up on
    int t = first_tile;
    for (int64_t u = ub; u < ue; ++t) {
      const int64_t seg_begin = u;
      const int64_t seg_end = (int64_t(t) + 1) * KB < ue ? (int64_t(t) + 1) * KB : ue;
      u = seg_end;
      const int cur = accb;
      const uint32_t cur_ph = accph;
      if (++accb == NACC) {
        accb = 0;
        accph ^= 1u;
      }
      const int c_first = unit_owner(int64_t(t) * KB, U, G);
      const int c_last = unit_owner((int64_t(t) + 1) * KB - 1, U, G);
      const int nsplit = c_last - c_first + 1;
      // Partial slots are laid out [chunk][quarter][row][4] floats: the 16
      // values a thread holds for a chunk are four 16-byte pieces 2 KB apart,
      // so each warp-wide access covers 512 contiguous bytes (whole sectors).
      auto slot_of = [&](int cc) {
        const int ft = int(unit_begin(cc, U, G) / KB);
        return 2 * cc + (t == ft ? 0 : 1);
      };
      // The CTA's final segment ends the kernel. When its tile has one other
      // piece and that piece is already done (it was the first piece its CTA
      // processed, so it usually is), its partial is fetched while this
      // segment's last units are still in flight, and the tile is finished
      // here without writing a partial or taking a counter round trip.
      const int me = c - c_first;
      int pref = 0;
      if (!P.defer && seg_end == ue && nsplit == 2 && nchunks == 1) {
        if (et == 0) {
          int done = 0;
          const uint64_t t0 = globaltimer_ns();
          for (;;) {
            if (ld_acquire_gpu(&P.counters[t]) == nsplit - 1) {
              done = 1;
              break;
            }
            if (mbar_try_wait(&B.acc_full[cur], cur_ph)) {
              done = ld_acquire_gpu(&P.counters[t]) == nsplit - 1;
              break;
            }
            if (*abort_flag || globaltimer_ns() - t0 > lim) break;  // the wait below reports it
          }
          *pref_flag = done;
        }
        named_bar_sync(kEpiBar, 128);
        pref = *pref_flag;
        if (pref) {
          const float4* s0 =
              reinterpret_cast<const float4*>(P.parts + size_t(slot_of(c_first + 1 - me)) * P.Mpad * 128) + row;
          // Parked in this thread's own column of the transpose buffer (free
          // until this segment's epilogue writes the same places).
          float* sc = scratch + row;
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const float4 f = __ldcg(s0 + x * 128);
            sc[(4 * x) * kScratchStride] = f.x;
            sc[(4 * x + 1) * kScratchStride] = f.y;
            sc[(4 * x + 2) * kScratchStride] = f.z;
            sc[(4 * x + 3) * kScratchStride] = f.w;
          }
        }
      }
      // One decision for the 128 epilogue threads, which meet at named barriers below.
      if (named_bar_any(kEpiBar, 128, !wait(&B.acc_full[cur], cur_ph))) break;
      tc_fence_after();
      // Issuer k wrote accumulator (cur, k) iff the segment holds a unit i
      // (counted from the CTA's first unit) with i % issuers == k.
      const int ia = int(seg_begin - ub), nseg = int(seg_end - seg_begin);
      const uint32_t d_tmem = tmem_base + tm_lane + uint32_t(cur * NISS) * uint32_t(P.Mpad);
      auto load_acc = [&](int mc, float (&v)[16]) {
        bool have = false;
        for (int kq = 0; kq < NISS; ++kq) {
          if (!(nseg >= NISS || (ia % NISS) == kq)) continue;
          uint32_t r[16];
          tmem_ld16(d_tmem + uint32_t(kq * P.Mpad + mc * 16), r);
          tmem_ld_wait(r);
#pragma unroll
          for (int x = 0; x < 16; ++x) v[x] = have ? v[x] + __uint_as_float(r[x]) : __uint_as_float(r[x]);
          have = true;
        }
      };
      if (nsplit == 1 || pref) {
        for (int mc = 0; mc < nchunks; ++mc) {
          float v[16];
          load_acc(mc, v);
          if (pref) {
            // Same slot-order sum as the fixup below (own piece at position me).
#pragma unroll
            for (int x = 0; x < 16; ++x) {
              const float o = scratch[x * kScratchStride + row];
              float acc = 0.0f;
              acc += me == 0 ? v[x] : o;
              acc += me == 0 ? o : v[x];
              v[x] = acc;
            }
          }
          if (kArgmax) argmax_chunk(v, t, mc);
          else store_chunk(v, t, mc);
        }
        tc_fence_before();
        mbar_arrive(&B.acc_empty[cur]);
        if (pref && et == 0) P.counters[t] = 0;  // every other contributor has already counted
      } else {
        // In the final segment every stage of the ring has been consumed (the
        // segment's MMAs completed), so the other pieces' partials can be
        // brought into it with bulk copies, as many chunks per round trip as
        // fit. This CTA's own piece is then taken from TMEM. If every other
        // piece is already counted, the tile is finished here without writing
        // this piece or taking the counter round trip.
        //
        // With P.defer a piece only goes to its partial slot and the sum is
        // left to splitk_reduce_kernel, which spreads it over every SM: at
        // large M a split tile's partial is Mpad x 128 fp32 (up to 128 KB), and
        // one CTA summing three or more of them alone takes longer than its
        // main loop.
        const uint32_t ring_bytes = uint32_t(S) * plan.stage_bytes;
        const int cb_max = int(ring_bytes / (uint32_t(nsplit - 1) * 8192u));  // chunks per gather batch
        const bool gather = !P.defer && seg_end == ue && cb_max >= 1;
        int fast = 0;
        if (gather) {
          if (et == 0) *fast_flag = ld_acquire_gpu(&P.counters[t]) == nsplit - 1;
          named_bar_sync(kEpiBar, 128);
          fast = *fast_flag;
        }
        if (!fast) {
          const int slot = 2 * c + (t == first_tile ? 0 : 1);
          float4* my = reinterpret_cast<float4*>(P.parts + size_t(slot) * P.Mpad * 128);
          for (int mc = 0; mc < nchunks; ++mc) {
            float v[16];
            load_acc(mc, v);
            float4* dst = my + size_t(mc) * 512 + row;
#pragma unroll
            for (int x = 0; x < 4; ++x) dst[x * 128] = make_float4(v[4 * x], v[4 * x + 1], v[4 * x + 2], v[4 * x + 3]);
          }
        }
        tc_fence_before();
        mbar_arrive(&B.acc_empty[cur]);
        if (!fast && !P.defer) {
          // The barrier orders every epilogue thread's partial stores before
          // the single release-acquire increment; the last contributor's
          // readers are ordered after that increment by the second barrier.
          named_bar_sync(kEpiBar, 128);
          if (et == 0) {
            const int old = atomic_add_acq_rel_gpu(&P.counters[t], 1);
            *last_flag = (old == nsplit - 1) ? 1 : 0;
          }
          named_bar_sync(kEpiBar, 128);
        }
        const bool last = !P.defer && (fast || *last_flag != 0);
        uint32_t gph = 0;
        for (int mc0 = 0; last && mc0 < nchunks;) {
          const int nb = gather ? (nchunks - mc0 < cb_max ? nchunks - mc0 : cb_max) : nchunks;
          if (gather) {
            if (mc0 > 0) {
              // The previous batch has been read (generic proxy) by every
              // thread before the next bulk copies (async proxy) overwrite it.
              fence_proxy_async_smem();
              named_bar_sync(kEpiBar, 128);
            }
            if (et == 0) {
              mbar_arrive_expect_tx(B.gather, uint32_t(nsplit - 1) * uint32_t(nb) * 8192u);
              int j = 0;
              for (int sp = 0; sp < nsplit; ++sp) {
                if (sp == me) continue;
                const float* src = P.parts + size_t(slot_of(c_first + sp)) * P.Mpad * 128;
                for (int b2 = 0; b2 < nb; ++b2)
                  bulk_load(smem + uint32_t(j * nb + b2) * 8192u, src + size_t(mc0 + b2) * 128 * 16, 8192u,
                            B.gather);
                ++j;
              }
            }
            if (named_bar_any(kEpiBar, 128, !wait(B.gather, gph))) {
              gather_pending = int(gph);  // drained before the CTA exits
              break;
            }
            gph ^= 1u;
          }
          for (int b2 = 0; b2 < nb; ++b2) {
            const int mc = mc0 + b2;
            float r[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) r[k] = 0.0f;
            // Slot order, so the sum does not depend on which CTA finishes
            // the tile or by which path.
            for (int sp = 0, j = 0; sp < nsplit; ++sp) {
              float q[16];
              if (gather && sp == me) {
                load_acc(mc, q);
              } else {
                const float4* src =
                    gather ? reinterpret_cast<const float4*>(smem + uint32_t(j++ * nb + b2) * 8192u) + row
                           : reinterpret_cast<const float4*>(P.parts + size_t(slot_of(c_first + sp)) * P.Mpad * 128) +
                                 size_t(mc) * 512 + row;
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                  const float4 f = gather ? src[x * 128] : __ldcg(src + x * 128);
                  q[4 * x] = f.x, q[4 * x + 1] = f.y, q[4 * x + 2] = f.z, q[4 * x + 3] = f.w;
                }
              }
#pragma unroll
              for (int x = 0; x < 16; ++x) r[x] += q[x];
            }
            if (kArgmax) argmax_chunk(r, t, mc);
            else store_chunk(r, t, mc);
          }
          mc0 += nb;
        }
        if (last && et == 0) P.counters[t] = 0;
        named_bar_sync(kEpiBar, 128);
      }
    }
    // Partials requested into shared memory must land before the CTA exits.
    if (gather_pending >= 0) mbar_wait(B.gather, uint32_t(gather_pending), drain_limit_ns(lim));
  }

  cta_sync();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// Sum of the split tiles' partials (large M): block (t, mc) adds, for output
// tile t and tokens mc*16 .. mc*16+15, the partial slots of the CTAs that
// hold pieces of t, in CTA order (the same order as the in-kernel sum, so the
// result does not depend on the path), and writes Y. Unsplit tiles were
// written by the GEMM.
__global__ void __launch_bounds__(128) splitk_reduce_kernel(const float* __restrict__ parts, float* __restrict__ Y,
                                                            int M, int Mpad, int N, int KB, int64_t U, int G) {
  grid_dep_wait();
  grid_dep_launch();
  const int t = blockIdx.x, mc = blockIdx.y, row = threadIdx.x;
  const int c_first = unit_owner(int64_t(t) * KB, U, G);
  const int c_last = unit_owner((int64_t(t) + 1) * KB - 1, U, G);
  if (c_first == c_last) return;
  float r[16];
#pragma unroll
  for (int x = 0; x < 16; ++x) r[x] = 0.0f;
  // Pieces in batches of 4, every load of a batch issued before its first add
  // (one L2 round trip per batch); the adds keep CTA order.
  constexpr int kBatch = 4;
  for (int c0 = c_first; c0 <= c_last; c0 += kBatch) {
    float4 f[kBatch][4];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int cc = c0 + j;
      if (cc <= c_last) {
        const int ft = int(unit_begin(cc, U, G) / KB);
        const int slot = 2 * cc + (t == ft ? 0 : 1);
        const float4* src =
            reinterpret_cast<const float4*>(parts + size_t(slot) * Mpad * 128) + size_t(mc) * 512 + row;
#pragma unroll
        for (int x = 0; x < 4; ++x) f[j][x] = __ldcg(src + x * 128);
      }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      if (c0 + j <= c_last) {
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          r[4 * x] += f[j][x].x;
          r[4 * x + 1] += f[j][x].y;
          r[4 * x + 2] += f[j][x].z;
          r[4 * x + 3] += f[j][x].w;
        }
      }
    }
  }
#pragma unroll
  for (int x = 0; x < 16; ++x) {
    const int m = mc * 16 + x;
    if (m < M) Y[int64_t(m) * N + int64_t(t) * 128 + row] = r[x];
  }
}

template <bool kW12, bool kArgmax>
static int launch_impl(const GemmShape& sh, const GemmParams& P0, const CUtensorMap& a0, const CUtensorMap& a1,
                       const CUtensorMap& a2, const CUtensorMap& x, cudaStream_t stream) {
  GemmParams P = P0;
  // Deepest ring that fits next to the fixed carve-up.
  const int smem_max = 232448;
  const int nacc = sh.Mpad <= 128 ? 2 : 1;
  // Two MMA issuers when their accumulators fit in half of TMEM (Mpad <= 64).
  const int issuers = nacc * 2 * sh.Mpad <= 256 ? 2 : 1;
  const int a_col0 = (nacc * issuers * sh.Mpad + 63) & ~63;
  int stages = kMaxStages;
  while (stages > 2 && (smem_plan<kW12>(sh.Mpad, stages).total > uint32_t(smem_max) ||
                        (kW12 && a_col0 + stages * kAColsPerBuf > 512)))
    --stages;
  if (kW12 && a_col0 + stages * kAColsPerBuf > 512) return W12_ERR_UNSUPPORTED;
  const SmemPlan plan = smem_plan<kW12>(sh.Mpad, stages);
  if (plan.total > uint32_t(smem_max)) return W12_ERR_UNSUPPORTED;
  P.stages = stages;
  P.issuers = issuers;
  const bool wide = kW12 && sh.Mpad >= kWideMinMpad;
  auto kern = wide ? gemm_kernel<kW12, kArgmax, kW12> : gemm_kernel<kW12, kArgmax, false>;
  static bool attr_set[2][64] = {};  // per kernel and device; setting it twice is harmless
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return W12_ERR_CUDA;
  if (!attr_set[wide][dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max) != cudaSuccess)
      return W12_ERR_CUDA;
    attr_set[wide][dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(P.grid));
  cfg.blockDim = dim3(unsigned(Cfg<kW12>::kThreads));
  cfg.dynamicSmemBytes = plan.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_enabled() ? 1 : 0;
  int st = cuda_status(cudaLaunchKernelEx(&cfg, kern, a0, a1, a2, x, P));
  if (st || !P.defer) return st;
  cudaLaunchConfig_t rcfg = cfg;
  rcfg.gridDim = dim3(unsigned(P.tiles), unsigned(P.Mpad / 16));
  rcfg.blockDim = dim3(128);
  rcfg.dynamicSmemBytes = 0;
  return cuda_status(cudaLaunchKernelEx(&rcfg, splitk_reduce_kernel, static_cast<const float*>(P.parts), P.Y, P.M,
                                        P.Mpad, P.N, P.KB, P.units, P.grid));
}

int launch_gemm(bool w12_mode, bool argmax_mode, const uint16_t* X, int64_t M, const w12_weights* W,
                const uint16_t* Wbf16, int64_t N, int64_t K, float* Y, float* amax_val, int32_t* amax_idx,
                void* ws, size_t ws_bytes, int32_t* dev_status, cudaStream_t stream) {
  GemmShape sh;
  int st = gemm_shape(M, N, K, &sh);
  if (st) return st;
  if (!X || !aligned(X, 16) || !ws || !aligned(ws, 16)) return W12_ERR_ARG;
  if (argmax_mode ? (!amax_val || !amax_idx) : !Y) return W12_ERR_ARG;
  if (w12_mode) {
    if (!W || !W->p0 || !W->p1 || !W->p2 || !W->ebase || !W->exc_off) return W12_ERR_ARG;
    if (W->n_exc > 0 && !W->exc_ent) return W12_ERR_ARG;
    if (!aligned(W->p0, 16) || !aligned(W->p1, 16) || !aligned(W->p2, 16) || !aligned(W->ebase, 16))
      return W12_ERR_ARG;
  } else {
    if (!Wbf16 || !aligned(Wbf16, 16)) return W12_ERR_ARG;
  }
  if (!device_supported()) return W12_ERR_UNSUPPORTED;
  if (w12_mode && (sh.units + sh.grid - 1) / sh.grid + 1 > kOffCap) return W12_ERR_SHAPE;
  const WsLayout L = ws_layout(sh, 0);
  if (ws_bytes < L.total) return W12_ERR_WORKSPACE;

  GemmParams P{};
  P.M = sh.M;
  P.Mpad = sh.Mpad;
  P.N = sh.N;
  P.K = sh.K;
  P.KB = sh.KB;
  P.tiles = sh.tiles;
  P.grid = sh.grid;
  P.units = sh.units;
  P.ebase = w12_mode ? W->ebase : nullptr;
  P.exc_off = w12_mode ? W->exc_off : nullptr;
  P.exc_ent = w12_mode ? W->exc_ent : nullptr;
  P.n_exc = w12_mode ? W->n_exc : 0;
  P.Y = Y;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  P.counters = reinterpret_cast<int32_t*>(wsb + L.counters);
  P.parts = reinterpret_cast<float*>(wsb + L.parts);
  P.amax_val = amax_val;
  P.amax_idx = amax_idx;
  P.status = dev_status;
  P.limit_ns = wait_limit_ns();
  // At large M a split tile's partial is Mpad x 128 fp32 (up to 128 KB), and
  // the last contributor summing three or more of them alone takes longer
  // than its whole main loop: such launches (some tile split three or more
  // ways, i.e. a CTA's range shorter than a tile) leave the sum to a second
  // kernel. Two-piece splits and the fused head keep the in-kernel sum.
  P.defer = (!argmax_mode && sh.Mpad >= kDeferMinMpad && sh.units < int64_t(sh.KB) * sh.grid) ? 1 : 0;

  CUtensorMap tx, t0, t1, t2;
  if (!encode_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<uint16_t*>(X), uint64_t(K), uint64_t(M),
                      uint64_t(K) * 2, 64, uint32_t(sh.Mpad), CU_TENSOR_MAP_SWIZZLE_128B))
    return W12_ERR_CUDA;
  if (w12_mode) {
    const uint64_t half = uint64_t(K) / 2;
    if (!encode_tmap_2d(&t0, CU_TENSOR_MAP_DATA_TYPE_UINT8, W->p0, half, uint64_t(N), half, 64, 128,
                        CU_TENSOR_MAP_SWIZZLE_64B) ||
        !encode_tmap_2d(&t1, CU_TENSOR_MAP_DATA_TYPE_UINT8, W->p1, half, uint64_t(N), half, 64, 128,
                        CU_TENSOR_MAP_SWIZZLE_64B) ||
        !encode_tmap_2d(&t2, CU_TENSOR_MAP_DATA_TYPE_UINT8, W->p2, half, uint64_t(N), half, 64, 128,
                        CU_TENSOR_MAP_SWIZZLE_64B))
      return W12_ERR_CUDA;
    return argmax_mode ? launch_impl<true, true>(sh, P, t0, t1, t2, tx, stream)
                       : launch_impl<true, false>(sh, P, t0, t1, t2, tx, stream);
  }
  if (!encode_tmap_2d(&t0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<uint16_t*>(Wbf16), uint64_t(K),
                      uint64_t(N), uint64_t(K) * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return W12_ERR_CUDA;
  if (argmax_mode) return W12_ERR_UNSUPPORTED;
  return launch_impl<false, false>(sh, P, t0, t0, t0, tx, stream);
}

}  // namespace w12

using namespace w12;

extern "C" {

int w12_gemm(const uint16_t* X, int64_t M, const w12_weights* W, float* Y, void* ws, size_t ws_bytes,
             int32_t* dev_status, void* stream) {
  if (!W) return W12_ERR_ARG;
  return launch_gemm(true, false, X, M, W, nullptr, W->N, W->K, Y, nullptr, nullptr, ws, ws_bytes, dev_status,
                     static_cast<cudaStream_t>(stream));
}

int w12_gemm_bf16_ref(const uint16_t* X, int64_t M, const uint16_t* W, int64_t N, int64_t K, float* Y, void* ws,
                      size_t ws_bytes, int32_t* dev_status, void* stream) {
  return launch_gemm(false, false, X, M, nullptr, W, N, K, Y, nullptr, nullptr, ws, ws_bytes, dev_status,
                     static_cast<cudaStream_t>(stream));
}

}  // extern "C"
