// Grouped verify GEMMs: several W12 (or bf16) GEMMs of one layer in one
// persistent launch, optionally with the gate/up -> SwiGLU -> down dependency
// inside the launch.
//
// The verify pass reads every target weight each step (SpecPilot paper
// digest, summary paragraph); the layer's GEMMs all share M, so their
// 128x128 units can be split over the SMs as one stream: the launch pays one
// ramp-up and one tail for the group instead of one per GEMM. With a SwiGLU
// link the launch has three phases (the gate/up source; the other problems;
// the down projection, whose X is the gated activation of the gate/up output)
// and every CTA works through its share of each in turn; each down k-block
// waits (bounded) for a per-block ready flag written by the CTA that completes
// the block's two gate/up tiles. Flags carry a launch epoch, moved on by the
// last CTA to finish, so one workspace serves consecutive launches. A count of
// the blocks written so far lets a CTA that finds every block ready stop
// reading flags: a flag read is a round trip to L2 that the copy thread would
// otherwise take once per down unit.
//
// The kernel body follows the single-GEMM kernel of this library (warp roles,
// ring, TMEM buffers, stream-K fixup), generalised from one problem to a list
// of problems; it lives in its own translation unit and namespace so that the
// single-GEMM kernel keeps its own tuned code.
#include <cstring>

#include "w12_decode.cuh"
#include "w12_dev.cuh"
#include "w12_host.h"

namespace w12 {
namespace grouped_impl {

// Decode warps: W12_DEC_GROUPS groups of 4 x W12_DEC_SPLIT warps. Each warp
// serves one TMEM lane quarter (32 rows); the W12_DEC_SPLIT warps of a
// quarter in a group split the unit's 4 chunks of 32 values; groups take
// units in turn (unit i goes to group i % W12_DEC_GROUPS).
constexpr int kMaxStages = 8;         // smem ring depth limit (one TMEM A buffer per stage)
constexpr int kEpiBar = 1;            // named barrier id of the epilogue warps
constexpr int kScratchStride = 129;   // floats per column in the argmax transpose buffer

// One GEMM of a launch. A launch runs up to kMaxProb GEMMs (problems) that
// share M, in up to three phases (problems are ordered by phase). In every
// phase the CTAs are split over the phase's problems in proportion to their
// units; the CTAs of one problem share its units evenly (stream-K over the
// problem), so each CTA runs one job per phase: a range of consecutive units
// of one problem. The last phase holds the problem whose X is produced inside
// the launch (the SwiGLU link below).
struct ProbParams {
  int N, K, KB, tiles, phase, tile0;  // tile0: first of its tiles in the launch-wide tile numbering
  int cta0, cta1;                     // the problem's CTAs [cta0, cta1) in its phase
  const uint8_t* ebase;
  const uint32_t* exc_off;
  const uint32_t* exc_ent;
  int64_t n_exc;
  float* Y;
};

struct GemmParams {
  int M, Mpad, grid, stages, issuers, nprob, nphase;
  ProbParams pr[kMaxProb];
  float* parts;                       // split-K partial slots: 2 per CTA per phase
  int32_t* counters;                  // one per tile of the launch
  float* amax_val;
  int32_t* amax_idx;
  // SwiGLU link: problem glu_to multiplies act = bf16(silu(g) * u), where
  // [g | u] = Y of problem glu_from split in two halves along N; act block j
  // (columns j*128 .. j*128+127) is written by the CTA that completes the
  // second of its two Y tiles (j and j + N/256).
  int glu_from, glu_to, glu_blocks;
  // Pairs: the source phase gives CTA c < glu_blocks the two whole tiles c and
  // c + glu_blocks (gate and up of act block c) instead of an even share of
  // the source's units, so no source tile is split and each act block is
  // written by the CTA that computed both of its tiles, at the end of its
  // first phase rather than after the last of several pieces.
  int glu_pairs;
  uint16_t* act;
  int32_t* glu_cnt;                   // per block: tiles completed (reset to 0 by the writer)
  int32_t* glu_ready;                 // per block: epoch + 1 once written
  int32_t* epoch;                     // [0] launch epoch, [1] CTAs finished, [2] act blocks written (this launch)
  int32_t* status;
  uint64_t limit_ns;
};

// Tensor maps per problem: three planes (or the bf16 matrix in slot 0) and X.
struct GemmMaps {
  CUtensorMap m[kMaxProb][4];
};

// A CTA's job in one phase: units [b, b + n) of problem p, whose U units are
// shared by G CTAs, this one at place cl (G = 0: whole tiles that no other
// CTA shares); s0 = index of the job's first unit in the CTA's sequence. Exception entries of the job: positions [e0, e1) of
// the CTA's staged window, entry g0 + (position - e0) of the problem's list.
struct Job {
  int p, f, cl, G, U, b, n, s0;
  uint32_t e0, e1, g0, pad;
};

// Position of a unit in a CTA's sequence: job j (problem p), the problem's
// tile t and k-block kb, with the problem's KB cached; left = units of the
// job still to come (this one included), pos = this unit's place in the job.
struct Cur {
  int j, p, t, kb, KB, left, pos;
};

__device__ __forceinline__ int64_t unit_begin(int c, int64_t U, int G) { return int64_t(c) * U / G; }

// CTA that owns unit u: the largest c with floor(c*U/G) <= u.
__device__ __forceinline__ int unit_owner(int64_t u, int64_t U, int G) {
  return static_cast<int>(((u + 1) * G + U - 1) / U - 1);
}

// Cursor at unit ub of problem p, n units to go in the job.
__device__ __forceinline__ void cur_at(const GemmParams& P, int j, int p, int ub, int n, Cur& x) {
  x.j = j;
  x.p = p;
  x.KB = P.pr[p].KB;
  x.t = ub / x.KB;
  x.kb = ub % x.KB;
  x.left = n;
  x.pos = 0;
}

// Next unit of a job-table sequence (the next job's first unit after the
// last unit of a job).
__device__ __forceinline__ void cur_step(const GemmParams& P, const Job* J, int njobs, Cur& x) {
  if (--x.left > 0) {
    ++x.pos;
    if (++x.kb == x.KB) {
      x.kb = 0;
      ++x.t;
    }
  } else if (x.j + 1 < njobs) {
    const int j = x.j + 1;
    cur_at(P, j, J[j].p, J[j].b, J[j].n, x);
  }
}

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
  uint32_t scratch_off, red_off, soff_off, sent_off, uprob_off, bar_off, misc_off, job_off, total;
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
  p.uprob_off = off;
  off += kW12 ? kOffCap : 0;
  off = (off + 15) & ~15u;
  p.bar_off = off;
  off += 64 * 8;
  p.misc_off = off;
  off += 64;
  p.job_off = off;
  off += (kMaxProb + 1) * sizeof(Job);
  p.total = off + 1024;  // slack for 1024-byte alignment of the base
  return p;
}

struct Bars {
  uint64_t* full;     // weight bytes of a stage landed (decoders wait on this)
  uint64_t* full_x;   // X bytes of a stage landed (the MMA waits on this too)
  uint64_t* empty;
  uint64_t* a_full;
  uint64_t* acc_full;
  uint64_t* acc_empty;
  uint64_t* exc_ready;
  uint64_t* drain;
  uint64_t* gather;
};

template <bool kW12, bool kArgmax, int kMode, bool kWide>
__global__ void __launch_bounds__(Cfg<kW12>::kThreads, 1)
    gemm_kernel(const __grid_constant__ GemmMaps TM, const __grid_constant__ GemmParams P) {
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
  B.full_x = B.gather + 1;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + plan.misc_off);
  volatile uint32_t* tmem_slot = misc + 0;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(misc + 2);
  volatile int* ent_in_smem = reinterpret_cast<volatile int*>(misc + 3);
  volatile uint32_t* ent_base = misc + 4;
  volatile uint32_t* ent_end = misc + 5;
  volatile int* pref_flag = reinterpret_cast<volatile int*>(misc + 6);
  volatile int* fast_flag = reinterpret_cast<volatile int*>(misc + 7);
  volatile int* glu_flag = reinterpret_cast<volatile int*>(misc + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // kMode 0: one phase of independent problems, each CTA on one of them
  // (with one problem, every CTA on it): the one-problem code, on problem pc
  // at place c among its G CTAs. kMode 2: the phases of a SwiGLU link, one job
  // per phase (gate/up; the other problems; down), read from the CTA's job
  // table. The link's code (job table, flag polling, act blocks) is compiled
  // only into mode 2: the hot loops of every role stay small (instruction
  // cache) and within registers.
  constexpr bool kMulti = kMode == 2;
  constexpr bool kGlu = kMode == 2;
  constexpr bool single = !kMulti;
  Job* J = reinterpret_cast<Job*>(smem + plan.job_off);
  int pc = 0, c = blockIdx.x, G = P.grid;
  if constexpr (single) {
    while (pc + 1 < P.nprob && c >= P.pr[pc].cta1) ++pc;
    c -= P.pr[pc].cta0;
    G = P.pr[pc].cta1 - P.pr[pc].cta0;
  }
  // One-problem code: the problem's units, split evenly over Gc CTAs.
  const int64_t Uc = single ? int64_t(P.pr[pc].KB) * P.pr[pc].tiles : 0;
  const int Gc = single ? (Uc < G ? int(Uc) : G) : 0;
  auto sbegin = [&](int cc) { return unit_begin(cc < Gc ? cc : Gc, Uc, Gc); };
  int n_units = single ? int(sbegin(c + 1) - sbegin(c)) : 0;  // this CTA's units (job table: set below)
  int njobs = 1;
  const uint64_t lim = P.limit_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&B.full[s], 1);
      mbar_init(&B.full_x[s], 1);
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
    if (kMulti) {
      // Job table: this CTA's (nonempty) job in each phase, in phase order.
      int nj = 0, s0 = 0;
      for (int p = 0; p < P.nprob; ++p) {
        const ProbParams& q = P.pr[p];
        if (P.glu_pairs && p == P.glu_from) {
          if (int(blockIdx.x) < P.glu_blocks) {
            for (int h = 0; h < 2; ++h) {
              const int t = int(blockIdx.x) + h * P.glu_blocks;
              J[nj] = Job{p, q.phase, 0, 0, q.KB * q.tiles, t * q.KB, q.KB, s0, 0u, 0u, 0u, 0u};
              s0 += q.KB;
              ++nj;
            }
          }
          continue;
        }
        if (int(blockIdx.x) < q.cta0 || int(blockIdx.x) >= q.cta1) continue;
        const int U = q.KB * q.tiles, Gp = q.cta1 - q.cta0, cl = int(blockIdx.x) - q.cta0;
        const int b = int(unit_begin(cl, U, Gp)), e = int(unit_begin(cl + 1, U, Gp));
        if (e <= b) continue;
        J[nj] = Job{p, q.phase, cl, Gp, U, b, e - b, s0, 0u, 0u, 0u, 0u};
        s0 += e - b;
        ++nj;
      }
      misc[9] = uint32_t(nj);
      misc[10] = uint32_t(s0);
    }
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
  if (kMulti) {
    njobs = int(misc[9]);
    n_units = int(misc[10]);
  }
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
      for (int p = 0; p < P.nprob; ++p) {
        prefetch_tmap(&TM.m[p][3]);
        prefetch_tmap(&TM.m[p][0]);
        if (kW12) {
          prefetch_tmap(&TM.m[p][1]);
          prefetch_tmap(&TM.m[p][2]);
        }
      }
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      const uint32_t xbox = uint32_t(P.Mpad) * 128u;
      // Weights and X of a stage complete separately: the decoders can restore
      // a stage's weights while its X is still on the way (or, for the SwiGLU
      // target, not yet written).
      const uint32_t tx = C::kABytes + (kW12 ? 128u : 0u);
      const uint32_t txx = 2u * xbox;
      // Weight tile of the unit at cursor x into stage buffer st.
      auto load_w = [&](const Cur& x, uint8_t* st, uint64_t* bar) {
        const int pp = x.p;
        const CUtensorMap* m = TM.m[pp];
        if (kW12) {
          tma_load_2d_hint(st, &m[0], x.kb * 64, x.t * 128, bar, pol_w);
          tma_load_2d_hint(st + 8192, &m[1], x.kb * 64, x.t * 128, bar, pol_w);
          tma_load_2d_hint(st + 16384, &m[2], x.kb * 64, x.t * 128, bar, pol_w);
          bulk_load(st + plan.eb_off, P.pr[pp].ebase + int64_t(x.kb) * P.pr[pp].N + int64_t(x.t) * 128, 128u, bar);
        } else {
          tma_load_2d_hint(st, &m[0], x.kb * 128, x.t * 128, bar, pol_w);
          tma_load_2d_hint(st + 16384, &m[0], x.kb * 128 + 64, x.t * 128, bar, pol_w);
        }
      };
      // The first ring-full of weight tiles is requested before waiting for
      // the previous kernel on the stream (launch overlap); X is loaded, and
      // anything else is read or written, only after that wait.
      const int prefill = n_units < S ? n_units : S;
      Cur x;
      if (single)
        cur_at(P, 0, pc, int(sbegin(c)), n_units, x);
      else
        cur_at(P, 0, njobs > 0 ? J[0].p : 0, njobs > 0 ? J[0].b : 0, njobs > 0 ? J[0].n : 0, x);
      // One problem: plain (t, kb) counters, as cheap as possible per unit.
      auto step = [&](Cur& y) {
        if (kMulti) {
          cur_step(P, J, njobs, y);
        } else if (++y.kb == y.KB) {
          y.kb = 0;
          ++y.t;
        }
      };
      {
        Cur y = x;
        for (int i = 0; i < prefill; ++i) {
          mbar_arrive_expect_tx(&B.full[i], tx);
          load_w(y, smem + i * plan.stage_bytes, &B.full[i]);
          step(y);
        }
      }
      grid_dep_wait();
      const int32_t epoch = kGlu && P.glu_to >= 0 ? ld_acquire_gpu(P.epoch) : 0;
      int s = 0;
      uint32_t ph = 0;
      int issued = 0;
      bool gave_up = false;
      bool all_ready = false;  // every act block is written: no more flags to read
      for (; issued < n_units; ++issued) {
        uint8_t* st = smem + s * plan.stage_bytes;
        if (issued >= prefill) {
          if (!wait(&B.empty[s], ph ^ 1u)) break;
          mbar_arrive_expect_tx(&B.full[s], tx);
          load_w(x, st, &B.full[s]);
        }
        if (kGlu && x.p == P.glu_to && !gave_up && !all_ready) {
          // X of this problem is written by this launch: wait until its
          // k-block is ready (bounded), then make it visible to the copy. If
          // the wait gives up, the copies are still issued (of stale data) so
          // that every stage's byte count completes; the status word and the
          // abort flag already report the failure.
          all_ready = ld_acquire_gpu(P.epoch + 2) == P.glu_blocks;
          if (!all_ready) {
            const int32_t* rdy = P.glu_ready + x.kb;
            bool okr = ld_acquire_gpu(rdy) == epoch + 1;
            const uint64_t t0 = globaltimer_ns();
            while (!okr) {
              if (*abort_flag || globaltimer_ns() - t0 > lim) {
                fail(W12_ERR_TIMEOUT);
                gave_up = true;
                break;
              }
              __nanosleep(100);  // back off: every SM may be polling the same few flags
              okr = ld_acquire_gpu(rdy) == epoch + 1;
            }
          }
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        const CUtensorMap* mx = &TM.m[x.p][3];
        mbar_arrive_expect_tx(&B.full_x[s], txx);
        tma_load_2d_hint(st + plan.x_off, mx, x.kb * 128, 0, &B.full_x[s], pol_x);
        tma_load_2d_hint(st + plan.x_off + xbox, mx, x.kb * 128 + 64, 0, &B.full_x[s], pol_x);
        step(x);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      grid_dep_launch();
      if (*abort_flag) {
        // Let the copies already issued land before the CTA can exit. The
        // loop only stops at a stage boundary with every stage before it
        // fully issued (weights and X).
        for (int i = issued > S ? issued - S : 0; i < issued; ++i) {
          mbar_wait(&B.full[i % S], uint32_t(i / S) & 1u, drain_limit_ns(lim));
          mbar_wait(&B.full_x[i % S], uint32_t(i / S) & 1u, drain_limit_ns(lim));
        }
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
      Cur x;
      if (single)
        cur_at(P, 0, pc, int(sbegin(c)), n_units, x);
      else
        cur_at(P, 0, njobs > 0 ? J[0].p : 0, njobs > 0 ? J[0].b : 0, njobs > 0 ? J[0].n : 0, x);
      int s = 0, accb = 0;
      uint32_t ph = 0, accph = 0;
      bool started = false;  // this issuer has written its accumulator in the current segment
      for (int i = 0; i < n_units; ++i) {
        // A segment is the CTA's run of units of one tile.
        const bool first = (kMulti ? x.pos == 0 : i == 0) || (x.kb == 0);
        const bool last = (kMulti ? x.left == 1 : i + 1 == n_units) || (x.kb + 1 == x.KB);
        if (first) {
          if (!wait(&B.acc_empty[accb], accph ^ 1u)) break;
          tc_fence_after();
          started = false;
        }
        if (i % NISS == k) {
          // W12: the decoders waited for the stage's weights before arriving
          // on a_full; X completes on its own barrier.
          if (kW12 ? !wait(&B.a_full[s], ph) : !wait(&B.full[s], ph)) break;
          if (!wait(&B.full_x[s], ph)) break;
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
        if (kMulti) {
          cur_step(P, J, njobs, x);
        } else if (++x.kb == x.KB) {
          x.kb = 0;
        }
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
    if (kW12 && !single) {
      // Job table: the offsets of a job's units and its entries are one window
      // of its problem's lists. The offsets are rebased to positions in the
      // CTA's staged window (soff: n_units + 1 values; unit i's entries are at
      // positions soff[i] .. soff[i+1]) and ujob[i] names unit i's job. The
      // entries go to sent when every window fits; otherwise the decoders read
      // them from global memory.
      uint32_t* soff = reinterpret_cast<uint32_t*>(smem + plan.soff_off);
      uint32_t* sent = reinterpret_cast<uint32_t*>(smem + plan.sent_off);
      uint8_t* ujob = smem + plan.uprob_off;
      bool bad = false;
      uint32_t base = 0;
      for (int j = 0; j < njobs; ++j) {
        const ProbParams& q = P.pr[J[j].p];
        const int b = J[j].b, n = J[j].n, s0 = J[j].s0;  // n_units + 1 <= kOffCap (host)
        const uint32_t e0 = q.exc_off[b], e1 = q.exc_off[b + n];
        const bool badj = e1 < e0 || int64_t(e1) > q.n_exc;
        bad |= badj;
        const uint32_t w = badj ? 0u : e1 - e0;
        // Every load of a batch is issued before its first store.
        for (int k0 = 0; k0 < n; k0 += 32 * 8) {
          uint32_t v[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            if (k0 + lane + 32 * jj < n) v[jj] = q.exc_off[b + k0 + lane + 32 * jj];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int k = k0 + lane + 32 * jj;
            if (k < n) {
              soff[s0 + k] = v[jj] - e0 + base;  // checked against [e0, e1) of the job by the decoders
              ujob[s0 + k] = uint8_t(j);
            }
          }
        }
        if (lane == 0) {
          J[j].e0 = base;
          J[j].e1 = base + w;
          J[j].g0 = e0;
        }
        base += w;
      }
      if (lane == 0) soff[n_units] = base;
      __syncwarp();  // lane 0's job fields, for every lane
      const bool fits = base <= uint32_t(kEntCap);
      if (fits) {
        constexpr int kBatch = 16;  // entries per lane in flight
        for (int j = 0; j < njobs; ++j) {
          const uint32_t* src = P.pr[J[j].p].exc_ent + J[j].g0;
          uint32_t* dst = sent + J[j].e0;
          const uint32_t n = J[j].e1 - J[j].e0;
          for (uint32_t b0 = 0; b0 < n; b0 += 32 * kBatch) {
            uint32_t v[kBatch];
#pragma unroll
            for (int jj = 0; jj < kBatch; ++jj)
              if (b0 + lane + 32 * jj < n) v[jj] = src[b0 + lane + 32 * jj];
#pragma unroll
            for (int jj = 0; jj < kBatch; ++jj)
              if (b0 + lane + 32 * jj < n) dst[b0 + lane + 32 * jj] = v[jj];
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        if (bad) set_status(P.status, W12_ERR_CORRUPT);
        *ent_in_smem = fits ? 1 : 0;
        *ent_base = 0;
        *ent_end = base;
        mbar_arrive(B.exc_ready);
      }
    } else if (kW12) {
      const ExcWindow w = stage_window(P.pr[pc].exc_off, P.pr[pc].exc_ent, P.pr[pc].n_exc, sbegin(c), n_units,
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
      d.n_units = n_units;
      d.full = B.full;
      d.a_full = B.a_full;
      d.a_tmem = tmem_base + a_col0;
      d.soff = reinterpret_cast<const uint32_t*>(smem + plan.soff_off);
      d.sent = reinterpret_cast<const uint32_t*>(smem + plan.sent_off);
      d.e_base = *ent_base;
      d.in_smem = *ent_in_smem;
      d.status = P.status;
      const uint32_t e_end = *ent_end;
      const uint8_t* ujob = smem + plan.uprob_off;
      // One problem: the CTA's window of the problem's entries. Job table:
      // each job's window, positions [e0, e1) of the staged buffer for entries
      // g0 .. of the job's problem.
      const uint32_t seen = decode_units<kWide ? 1 : kDecGroups, kWide ? kWideSplit : kDecSplit>(
          d, warp - 4, wait,
          [&](int i, uint32_t o0, uint32_t o1) {
            if (single) return o1 < o0 || int64_t(o1) > P.pr[pc].n_exc || o0 < d.e_base || o1 > e_end;
            const Job& jb = J[ujob[i]];
            return o1 < o0 || o0 < jb.e0 || o1 > jb.e1;
          },
          [&](int i) -> const uint32_t* {
            if (single) return P.pr[pc].exc_ent;
            const Job& jb = J[ujob[i]];
            return P.pr[jb.p].exc_ent + (int64_t(jb.g0) - int64_t(jb.e0));
          });
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
    auto store_chunk = [&](const float (&v)[16], int pi, int t, int mc) {
      float* Y = P.pr[pi].Y;
      const int64_t N = P.pr[pi].N;
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const int m = mc * 16 + r;
        if (m < P.M) Y[int64_t(m) * N + int64_t(t) * 128 + row] = v[r];
      }
    };

    grid_dep_wait();
    const int32_t epoch = kGlu && P.glu_to >= 0 ? ld_acquire_gpu(P.epoch) : 0;
    // Tile t of the SwiGLU source problem is complete in Y: the CTA that
    // completes the second tile of block j writes act block j and publishes it.
    // This thread's column of act block j from both halves in Y: 8 rows per
    // batch, every load of a batch issued before its first use (one L2 round
    // trip per 8 rows).
    auto act_from_y = [&](int j) {
      const ProbParams& pg = P.pr[P.glu_from];
      const int64_t Nh = pg.N / 2;
      const int64_t col = int64_t(j) * 128 + et;
      for (int m0 = 0; m0 < P.M; m0 += 8) {
        float g[8], u[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int m = m0 + r < P.M ? m0 + r : P.M - 1;
          g[r] = __ldcg(pg.Y + int64_t(m) * pg.N + col);
          u[r] = __ldcg(pg.Y + int64_t(m) * pg.N + Nh + col);
        }
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (m0 + r < P.M) P.act[int64_t(m0 + r) * Nh + col] = f32_to_bf16_rne(g[r] / (1.0f + expf(-g[r])) * u[r]);
      }
    };
    // Pairs: tile t >= glu_blocks completes act block j = t - glu_blocks, whose
    // gate tile this CTA computed earlier. Each thread reads only the column it
    // stored itself in both tiles, so no barrier or count comes first; one
    // barrier orders every thread's act stores before the publication.
    auto glu_pair_done = [&](int j) {
      act_from_y(j);
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __threadfence();
      named_bar_sync(kEpiBar, 128);
      if (et == 0) {
        st_release_gpu(P.glu_ready + j, epoch + 1);
        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(P.epoch + 2) : "memory");
      }
    };
    auto glu_tile_done = [&](int t) {
      const int j = t < P.glu_blocks ? t : t - P.glu_blocks;
      named_bar_sync(kEpiBar, 128);  // every thread's Y stores of the tile are issued
      if (et == 0) {
        __threadfence();
        const int old = atomic_add_acq_rel_gpu(P.glu_cnt + j, 1);
        *glu_flag = old == 1 ? 1 : 0;
      }
      named_bar_sync(kEpiBar, 128);
      if (*glu_flag) {
        act_from_y(j);
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __threadfence();
        named_bar_sync(kEpiBar, 128);
        if (et == 0) {
          P.glu_cnt[j] = 0;
          st_release_gpu(P.glu_ready + j, epoch + 1);
          atomic_add_acq_rel_gpu(P.epoch + 2, 1);
        }
      }
    };
    int accb = 0;
    uint32_t accph = 0;
    int gather_pending = -1;  // phase of a gather of partials that was given up on
    // Walk the CTA's segments (its runs of units of one tile) job by job;
    // only the job and (next unit, end of the job's range) are carried
    // between segments. Unit numbers fit in 32 bits (the host checks every
    // problem's count).
    int jn = 0, un = 0, uen = 0;
    const int ub_single = single ? int(sbegin(c)) : 0;
    bool more;
    if (single) {
      un = ub_single;
      uen = int(sbegin(c + 1));
      more = un < uen;
    } else {
      more = njobs > 0;
      if (more) {
        un = J[0].b;
        uen = un + J[0].n;
      }
    }
    while (more) {
      // This segment's job (the cursor may move on to the next job below).
      const int f = single ? 0 : J[jn].f, cl = single ? c : J[jn].cl, Gf = single ? Gc : J[jn].G;
      const int ub = single ? ub_single : J[jn].b, ue = uen, ia0 = single ? 0 : J[jn].s0;
      const int64_t Uf = single ? Uc : J[jn].U;
      const int pi = single ? pc : J[jn].p;
      const int KBp = P.pr[pi].KB;
      const int t = un / KBp;
      const int tile_u0 = t * KBp;
      const int seg_begin = un;
      const int seg_end = tile_u0 + KBp < ue ? tile_u0 + KBp : ue;
      un = seg_end;
      more = un < uen;
      if (kMulti && !more && jn + 1 < njobs) {
        ++jn;
        un = J[jn].b;
        uen = un + J[jn].n;
        more = true;
      }
      const bool final_seg = !more;  // the CTA's last segment: the ring is idle once it is accumulated
      const int ia = ia0 + (seg_begin - ub), nseg = seg_end - seg_begin;
      const int gt = P.pr[pi].tile0 + t;   // launch-wide tile number (counters)
      const int cur = accb;
      const uint32_t cur_ph = accph;
      if (++accb == NACC) {
        accb = 0;
        accph ^= 1u;
      }
      // (A whole-tile job, Gf = 0, holds the only piece of its tiles.)
      const int c_first = Gf == 0 ? cl : unit_owner(tile_u0, Uf, Gf);
      const int c_last = Gf == 0 ? cl : unit_owner(tile_u0 + KBp - 1, Uf, Gf);
      const int nsplit = c_last - c_first + 1;
      // Partial slots are laid out [chunk][quarter][row][4] floats: the 16
      // values a thread holds for a chunk are four 16-byte pieces 2 KB apart,
      // so each warp-wide access covers 512 contiguous bytes (whole sectors).
      // CTA cc has two slots per phase: its first piece in the phase, and
      // its last.
      auto slot_of = [&](int cc) {
        const int64_t u0 = unit_begin(cc < Gf ? cc : Gf, Uf, Gf);
        const int cg = P.pr[pi].cta0 + cc;  // launch-wide CTA
        return 2 * (cg * P.nphase + f) + ((u0 >= tile_u0 && u0 < tile_u0 + KBp) ? 0 : 1);
      };
      // The CTA's final segment ends the kernel. When its tile has one other
      // piece and that piece is already done (it was the first piece its CTA
      // processed, so it usually is), its partial is fetched while this
      // segment's last units are still in flight, and the tile is finished
      // here without writing a partial or taking a counter round trip.
      const int me = cl - c_first;
      int pref = 0;
      // (Any phase's last segment qualifies: the prefetch goes to the
      // epilogue's own transpose buffer, not to the ring.)
      if (seg_end == ue && nsplit == 2 && nchunks == 1) {
        if (et == 0) {
          int done = 0;
          const uint64_t t0 = globaltimer_ns();
          for (;;) {
            if (ld_acquire_gpu(&P.counters[gt]) == nsplit - 1) {
              done = 1;
              break;
            }
            if (mbar_try_wait(&B.acc_full[cur], cur_ph)) {
              done = ld_acquire_gpu(&P.counters[gt]) == nsplit - 1;
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
          else store_chunk(v, pi, t, mc);
        }
        tc_fence_before();
        mbar_arrive(&B.acc_empty[cur]);
        if (pref && et == 0) P.counters[gt] = 0;  // every other contributor has already counted
        if (kGlu && pi == P.glu_from) {
          if (!P.glu_pairs) glu_tile_done(t);
          else if (t >= P.glu_blocks) glu_pair_done(t - P.glu_blocks);
        }
      } else {
        // In the final segment every stage of the ring has been consumed (the
        // segment's MMAs completed), so the other pieces' partials can be
        // brought into it with bulk copies, as many chunks per round trip as
        // fit. This CTA's own piece is then taken from TMEM. If every other
        // piece is already counted, the tile is finished here without writing
        // this piece or taking the counter round trip.
        const uint32_t ring_bytes = uint32_t(S) * plan.stage_bytes;
        const int cb_max = int(ring_bytes / (uint32_t(nsplit - 1) * 8192u));  // chunks per gather batch
        const bool gather = final_seg && cb_max >= 1;
        int fast = 0;
        if (gather) {
          if (et == 0) *fast_flag = ld_acquire_gpu(&P.counters[gt]) == nsplit - 1;
          named_bar_sync(kEpiBar, 128);
          fast = *fast_flag;
        }
        if (!fast) {
          const int slot = 2 * (int(blockIdx.x) * P.nphase + f) + (seg_begin == ub ? 0 : 1);
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
        if (!fast) {
          // The barrier orders every epilogue thread's partial stores before
          // the single release-acquire increment; the last contributor's
          // readers are ordered after that increment by the second barrier.
          named_bar_sync(kEpiBar, 128);
          if (et == 0) {
            const int old = atomic_add_acq_rel_gpu(&P.counters[gt], 1);
            *last_flag = (old == nsplit - 1) ? 1 : 0;
          }
          named_bar_sync(kEpiBar, 128);
        }
        const bool last = fast || *last_flag != 0;
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
            else store_chunk(r, pi, t, mc);
          }
          mc0 += nb;
        }
        if (last && et == 0) P.counters[gt] = 0;
        named_bar_sync(kEpiBar, 128);
        if (kGlu && last && pi == P.glu_from && !P.glu_pairs) glu_tile_done(t);  // (pairs never split a tile)
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
  if (kGlu && P.glu_to >= 0 && threadIdx.x == 0) {
    // The last CTA to finish moves the launch epoch on, so the next launch
    // on this workspace tells its ready flags from this one's.
    const int32_t e = *reinterpret_cast<volatile int32_t*>(P.epoch);
    if (atomic_add_acq_rel_gpu(P.epoch + 1, 1) == G - 1) {
      P.epoch[1] = 0;
      P.epoch[2] = 0;
      st_release_gpu(P.epoch, e + 1);
    }
  }
}

template <bool kW12, bool kArgmax, int kMode>
static int launch_impl(int Mpad, GemmParams& P, const GemmMaps& TM, cudaStream_t stream) {
  // Deepest ring that fits next to the fixed carve-up.
  const int smem_max = 232448;
  const int nacc = Mpad <= 128 ? 2 : 1;
  // Two MMA issuers when their accumulators fit in half of TMEM (Mpad <= 64).
  const int issuers = nacc * 2 * Mpad <= 256 ? 2 : 1;
  const int a_col0 = (nacc * issuers * Mpad + 63) & ~63;
  int stages = kMaxStages;
  while (stages > 2 && (smem_plan<kW12>(Mpad, stages).total > uint32_t(smem_max) ||
                        (kW12 && a_col0 + stages * kAColsPerBuf > 512)))
    --stages;
  if (kW12 && a_col0 + stages * kAColsPerBuf > 512) return W12_ERR_UNSUPPORTED;
  const SmemPlan plan = smem_plan<kW12>(Mpad, stages);
  if (plan.total > uint32_t(smem_max)) return W12_ERR_UNSUPPORTED;
  P.stages = stages;
  P.issuers = issuers;
  // Large M: one decode group of the widest split (a unit's restore sits on
  // the critical path of a two- or three-stage ring).
  const bool wide = kW12 && Mpad >= kWideMinMpad;
  auto kern = wide ? gemm_kernel<kW12, kArgmax, kMode, kW12> : gemm_kernel<kW12, kArgmax, kMode, false>;
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
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, TM, P));
}

// Tensor maps of one problem: planes (or the bf16 matrix) and X.
static int encode_problem(bool w12_mode, const uint16_t* X, int64_t M, int Mpad, const w12_weights* W,
                          const uint16_t* Wbf16, int64_t N, int64_t K, CUtensorMap* m) {
  if (!encode_tmap_2d(&m[3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<uint16_t*>(X), uint64_t(K), uint64_t(M),
                      uint64_t(K) * 2, 64, uint32_t(Mpad), CU_TENSOR_MAP_SWIZZLE_128B))
    return W12_ERR_CUDA;
  if (w12_mode) {
    const uint64_t half = uint64_t(K) / 2;
    if (!encode_tmap_2d(&m[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, W->p0, half, uint64_t(N), half, 64, 128,
                        CU_TENSOR_MAP_SWIZZLE_64B) ||
        !encode_tmap_2d(&m[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, W->p1, half, uint64_t(N), half, 64, 128,
                        CU_TENSOR_MAP_SWIZZLE_64B) ||
        !encode_tmap_2d(&m[2], CU_TENSOR_MAP_DATA_TYPE_UINT8, W->p2, half, uint64_t(N), half, 64, 128,
                        CU_TENSOR_MAP_SWIZZLE_64B))
      return W12_ERR_CUDA;
  } else {
    if (!encode_tmap_2d(&m[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<uint16_t*>(Wbf16), uint64_t(K),
                        uint64_t(N), uint64_t(K) * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
      return W12_ERR_CUDA;
    m[1] = m[0];
    m[2] = m[0];
  }
  return W12_OK;
}

static int check_weights(const w12_weights* W) {
  if (!W || !W->p0 || !W->p1 || !W->p2 || !W->ebase || !W->exc_off) return W12_ERR_ARG;
  if (W->n_exc > 0 && !W->exc_ent) return W12_ERR_ARG;
  if (!aligned(W->p0, 16) || !aligned(W->p1, 16) || !aligned(W->p2, 16) || !aligned(W->ebase, 16))
    return W12_ERR_ARG;
  return W12_OK;
}

static void set_problem(ProbParams& q, bool w12_mode, const w12_weights* W, int64_t N, int64_t K, float* Y) {
  q.N = int(N);
  q.K = int(K);
  q.KB = int(K / kGroup);
  q.tiles = int(N / kGroup);
  q.ebase = w12_mode ? W->ebase : nullptr;
  q.exc_off = w12_mode ? W->exc_off : nullptr;
  q.exc_ent = w12_mode ? W->exc_ent : nullptr;
  q.n_exc = w12_mode ? W->n_exc : 0;
  q.Y = Y;
}

// Grouped launch: problems in launch order with their phases, and the
// workspace carve-up.
struct Grouped {
  int n, order[kMaxProb], phase[kMaxProb], nphase, Mpad, grid, tiles, glu_from, glu_to, glu_blocks, glu_pairs;
  int cta0[kMaxProb], cta1[kMaxProb];  // launch problem j runs on CTAs [cta0[j], cta1[j]) of its phase
  int64_t N[kMaxProb], K[kMaxProb], phase_units[kMaxProb];
  size_t counters, glu_cnt, glu_ready, epoch, parts, total;
};

static int plan_grouped(const w12_problem* probs, int n, int64_t M, const w12_swiglu* link, bool w12_mode,
                        Grouped* g) {
  if (!probs || n < 1 || n > kMaxProb) return W12_ERR_ARG;
  if (M < 1 || M > kMaxM) return W12_ERR_SHAPE;
  memset(g, 0, sizeof(*g));
  g->n = n;
  g->glu_from = g->glu_to = -1;
  for (int i = 0; i < n; ++i) {
    const w12_weights* W = probs[i].W;
    g->N[i] = w12_mode ? (W ? W->N : 0) : probs[i].N;
    g->K[i] = w12_mode ? (W ? W->K : 0) : probs[i].K;
    GemmShape sh;
    const int st = gemm_shape(M, g->N[i], g->K[i], &sh);
    if (st) return st;
    g->Mpad = sh.Mpad;
  }
  int to = -1;
  if (link) {
    if (link->from < 0 || link->from >= n || link->to < 0 || link->to >= n || link->from == link->to)
      return W12_ERR_ARG;
    if (g->N[link->from] % (2 * kGroup) || g->K[link->to] != g->N[link->from] / 2) return W12_ERR_SHAPE;
    to = link->to;
  }
  // Phases. Independent problems form one phase. With a SwiGLU link the
  // source forms the first phase, the other problems the second (the
  // activation blocks complete while the CTAs work on them) and the target
  // the last.
  const int from = link ? link->from : -1;
  int k = 0;
  if (from >= 0) {
    g->order[k] = from;
    g->phase[k++] = 0;
  }
  for (int i = 0; i < n; ++i)
    if (i != to && i != from) {
      g->order[k] = i;
      g->phase[k++] = from >= 0 ? 1 : 0;
    }
  g->nphase = (from >= 0 ? 1 : 0) + (n - (from >= 0 ? 2 : 0) > 0 ? 1 : 0);
  if (to >= 0) {
    g->order[k] = to;
    g->phase[k++] = g->nphase++;
  }
  int64_t maxu = 0, U[kMaxProb];
  for (int j = 0; j < n; ++j) {
    const int i = g->order[j];
    U[j] = (g->N[i] / kGroup) * (g->K[i] / kGroup);
    g->phase_units[g->phase[j]] += U[j];
    g->tiles += int(g->N[i] / kGroup);
    // The kernel numbers a problem's units in 32 bits.
    if (U[j] > (int64_t(1) << 30)) return W12_ERR_SHAPE;
  }
  for (int f = 0; f < g->nphase; ++f) maxu = g->phase_units[f] > maxu ? g->phase_units[f] : maxu;
  int sms = device_sm_count();
  if (sms <= 0) sms = 256;  // sizing without a device: an upper bound
  // One CTA per SM at most: a CTA of the SwiGLU link may wait on work of any
  // other CTA, so all of them must be resident together.
  const int grid = int(maxu < sms ? maxu : sms);
  // CTAs [lo, hi) split over the problems of `sel` (a bit per launch problem)
  // so that the largest per-CTA share of units is as small as it can be: one
  // CTA at a time to the problem whose CTAs carry the most units each (units
  // weigh the same bytes in every problem), never more CTAs than units.
  // Returns that share, or -1 if there are fewer CTAs than problems.
  auto split = [&](int lo, int hi, unsigned sel) -> int64_t {
    int cnt[kMaxProb], np = 0;
    for (int j = 0; j < n; ++j) {
      cnt[j] = (sel >> j) & 1u;
      np += cnt[j];
    }
    if (np == 0) return 0;
    if (hi - lo < np) return -1;
    for (int left = hi - lo - np; left > 0; --left) {
      int best = -1;
      for (int j = 0; j < n; ++j)
        if (((sel >> j) & 1u) && cnt[j] < U[j] && (best < 0 || U[j] * cnt[best] > U[best] * cnt[j])) best = j;
      if (best < 0) break;
      ++cnt[best];
    }
    int at = lo;
    int64_t most = 0;
    for (int j = 0; j < n; ++j) {
      if (!((sel >> j) & 1u)) continue;
      g->cta0[j] = at;
      at += cnt[j];
      g->cta1[j] = at;
      const int64_t q = (U[j] + cnt[j] - 1) / cnt[j];
      most = q > most ? q : most;
    }
    return most;
  };
  unsigned in_phase[kMaxProb] = {0, 0, 0, 0};
  for (int j = 0; j < n; ++j) in_phase[g->phase[j]] |= 1u << j;
  int64_t most_of[kMaxProb] = {0, 0, 0, 0};
  for (int f = 0; f < g->nphase; ++f) {
    most_of[f] = split(0, grid, in_phase[f]);
    if (most_of[f] < 0) return W12_ERR_UNSUPPORTED;
  }
  g->grid = grid;
  if (to >= 0) {
    g->glu_from = 0;
    g->glu_to = n - 1;
    g->glu_blocks = int(g->N[link->from] / (2 * kGroup));
    // Whole gate/up pairs for the source phase when they spread over the CTAs
    // about as evenly as an even split would (at most 1.25 CTAs per pair):
    // one pair per CTA. The CTAs without a pair then take the middle phase's
    // problems that even out the first two phases best: each subset of them
    // on the free CTAs and the rest on the paired ones, against the middle
    // phase split over all CTAs, by the largest per-CTA load in units.
    const int pairs = g->glu_blocks;
    if (pairs <= grid && 4 * grid <= 5 * pairs) {
      g->glu_pairs = 1;
      const int64_t pair_units = 2 * (g->K[link->from] / kGroup);
      most_of[0] = pair_units;
      g->cta0[0] = 0;
      g->cta1[0] = pairs;
      const unsigned mid = g->nphase == 3 ? in_phase[1] : 0u;
      if (mid && grid > pairs) {
        int64_t best_load = pair_units + most_of[1];  // the middle phase over all CTAs
        unsigned best = ~0u;
        for (unsigned sub = mid;; sub = (sub - 1) & mid) {  // every subset of the middle problems
          const int64_t fr = split(pairs, grid, sub), pr = split(0, pairs, mid & ~sub);
          if (fr >= 0 && pr >= 0) {
            const int64_t load = fr > pair_units + pr ? fr : pair_units + pr;
            if (load < best_load) {
              best_load = load;
              best = sub;
            }
          }
          if (sub == 0) break;
        }
        if (best != ~0u) {
          const int64_t fr = split(pairs, grid, best), pr = split(0, pairs, mid & ~best);
          most_of[1] = fr > pr ? fr : pr;
        } else {
          most_of[1] = split(0, grid, mid);
        }
      }
    }
  }
  int64_t per_cta = 0;
  for (int f = 0; f < g->nphase; ++f) per_cta += most_of[f];
  g->grid = 0;  // CTAs past every problem's range (all capped at their units) are not launched
  for (int j = 0; j < n; ++j) g->grid = g->cta1[j] > g->grid ? g->cta1[j] : g->grid;
  if (w12_mode && per_cta + 1 > kOffCap) return W12_ERR_SHAPE;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += (bytes + 255) / 256 * 256;
    return at;
  };
  g->counters = take(sizeof(int32_t) * size_t(g->tiles));
  g->glu_cnt = take(sizeof(int32_t) * size_t(g->glu_blocks > 0 ? g->glu_blocks : 1));
  g->glu_ready = take(sizeof(int32_t) * size_t(g->glu_blocks > 0 ? g->glu_blocks : 1));
  g->epoch = take(sizeof(int32_t) * 4);
  g->parts = take(sizeof(float) * size_t(2) * g->nphase * g->grid * g->Mpad * kGroup);
  g->total = off;
  return W12_OK;
}

static int launch_grouped(bool w12_mode, const w12_problem* probs, int n, int64_t M, const w12_swiglu* link,
                          void* ws, size_t ws_bytes, int32_t* dev_status, cudaStream_t stream) {
  Grouped g;
  int st = plan_grouped(probs, n, M, link, w12_mode, &g);
  if (st) return st;
  if (!ws || !aligned(ws, 16)) return W12_ERR_ARG;
  if (ws_bytes < g.total) return W12_ERR_WORKSPACE;
  if (link && (!link->act || !aligned(link->act, 16) || !probs[link->from].Y)) return W12_ERR_ARG;
  for (int i = 0; i < n; ++i) {
    const bool is_to = link && i == link->to;
    if (!probs[i].Y) return W12_ERR_ARG;
    if (!is_to && (!probs[i].X || !aligned(probs[i].X, 16))) return W12_ERR_ARG;
    if (w12_mode) {
      if ((st = check_weights(probs[i].W))) return st;
    } else if (!probs[i].Wbf16 || !aligned(probs[i].Wbf16, 16)) {
      return W12_ERR_ARG;
    }
  }
  if (!device_supported()) return W12_ERR_UNSUPPORTED;

  GemmParams P{};
  P.M = int(M);
  P.Mpad = g.Mpad;
  P.grid = g.grid;
  P.nprob = n;
  P.nphase = g.nphase;
  GemmMaps TM;
  memset(&TM, 0, sizeof(TM));
  int tile0 = 0;
  for (int j = 0; j < n; ++j) {
    const int i = g.order[j];
    const bool is_to = link && i == link->to;
    ProbParams& q = P.pr[j];
    set_problem(q, w12_mode, probs[i].W, g.N[i], g.K[i], probs[i].Y);
    q.phase = g.phase[j];
    q.cta0 = g.cta0[j];
    q.cta1 = g.cta1[j];
    q.tile0 = tile0;
    tile0 += q.tiles;
    const uint16_t* X = is_to ? link->act : probs[i].X;
    if ((st = encode_problem(w12_mode, X, M, g.Mpad, probs[i].W, probs[i].Wbf16, g.N[i], g.K[i], TM.m[j])))
      return st;
  }
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  P.counters = reinterpret_cast<int32_t*>(wsb + g.counters);
  P.parts = reinterpret_cast<float*>(wsb + g.parts);
  P.glu_from = g.glu_from;
  P.glu_to = g.glu_to;
  P.glu_blocks = g.glu_blocks;
  P.glu_pairs = g.glu_pairs;
  P.act = link ? link->act : nullptr;
  P.glu_cnt = reinterpret_cast<int32_t*>(wsb + g.glu_cnt);
  P.glu_ready = reinterpret_cast<int32_t*>(wsb + g.glu_ready);
  P.epoch = reinterpret_cast<int32_t*>(wsb + g.epoch);
  P.status = dev_status;
  P.limit_ns = wait_limit_ns();
  // Independent problems run the one-problem form (each CTA on one problem);
  // a SwiGLU link the job-table form.
  if (link)
    return w12_mode ? launch_impl<true, false, 2>(g.Mpad, P, TM, stream)
                    : launch_impl<false, false, 2>(g.Mpad, P, TM, stream);
  return w12_mode ? launch_impl<true, false, 0>(g.Mpad, P, TM, stream)
                  : launch_impl<false, false, 0>(g.Mpad, P, TM, stream);
}

}  // namespace grouped_impl
}  // namespace w12

using namespace w12::grouped_impl;

extern "C" {

size_t w12_gemm_grouped_ws_bytes(const w12_problem* probs, int n, int64_t M, const w12_swiglu* link) {
  Grouped g;
  bool w12_mode = probs && n > 0 && probs[0].W;
  return plan_grouped(probs, n, M, link, w12_mode, &g) == W12_OK ? g.total : 0;
}

int w12_gemm_grouped(const w12_problem* probs, int n, int64_t M, const w12_swiglu* link, void* ws, size_t ws_bytes,
                     int32_t* dev_status, void* stream) {
  return launch_grouped(true, probs, n, M, link, ws, ws_bytes, dev_status, static_cast<cudaStream_t>(stream));
}

int w12_gemm_grouped_bf16_ref(const w12_problem* probs, int n, int64_t M, const w12_swiglu* link, void* ws,
                              size_t ws_bytes, int32_t* dev_status, void* stream) {
  return launch_grouped(false, probs, n, M, link, ws, ws_bytes, dev_status, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
