// bwd_kernel.cuh -- the deterministic attention backward tile kernel (the DASH hot path),
// instantiated by bwd.cu (uniform batches) and bwd_varlen.cu (packed variable-length batches).
//
// One persistent CTA per SM executes *workers* (sched.cuh): a worker owns one KV block j
// (or the pair c, N-1-c) of one (batch, kv head), keeps dK_j/dV_j in tensor memory for
// the whole segment (gist.science technical summary, section 2.1: one KV tile's
// operations run back to back on one SM with on-chip accumulation) and visits query
// tiles in the order of the selected schedule (section 2.2).  Per visited tile (128 query
// rows i, all in one query head h) it runs the five dense contractions on the tcgen05
// tensor cores, G4 split into the two 64-column halves a/b of the query tile:
//   G1  S^T  = K_j Q_i^T                   (128 x 128 x D)  -> TMEM
//   G2  dP^T = V_j dO_i^T                  (128 x 128 x D)  -> TMEM
//       P^T  = exp2(S^T * scale*log2e - LSE_i*log2e)   [causal: 0 above the diagonal]
//       dS^T = P^T o (dP^T - Dvec_i)                    (softmax-gradient warpgroups)
//   G3  dV_j += P^T dO_i                   (128 x D x 128)  A = P^T from TMEM
//   G4  dK_j += dS^T Q_i                   (128 x D x 128)  A = dS^T from TMEM
//   G5  dQ_part = dS K_j                   (128 x D x 128)  A = dS from shared memory
// and the epilogue warpgroup adds dQ_part into the fp32 dQ accumulator.  In the
// deterministic modes the addition into dQ tile (b,h,i) happens only when that tile's
// ordering semaphore equals this worker's rank in the tile's accumulation order, and the
// semaphore is advanced after the addition is globally visible (section 1: the dQ
// accumulation order is fixed; the schedules decide which order and how much waiting it
// costs).  In the atomic mode the additions are unordered.
//
// Pipeline (MMA issue order; every hand-off is an mbarrier):
//   segment start: G1(first) -> s_full
//   each step t:   [dQ(t-1) drained] G2(t) -> dp_full,
//                  [P^T(t) written] G3(t), G1(t+1) -> s_full   (G1 within the segment)
//                  [dS half a] G4a, [half b] G4b -> stage free,
//                  G5(t) -> g5_done
// The softmax-gradient warpgroups read S^T(t), compute P and write P^T (bf16) over the
// first half of the S^T columns they read, so G3(t) and then G1(t+1) run on the tensor pipe
// while they compute dS; they write dS^T over the dP^T columns they have just read, and only
// G4 and G5 remain between dS and the next step.  The epilogue copies the dQ partial to
// registers first and waits for its
// turn on the semaphore afterwards, so a waiting reduction does not hold tensor memory.
// The semaphore of a dQ tile counts the partials added to it; a poller warp watches the
// semaphores of this CTA's coming steps ahead of time, so the epilogue usually finds its
// turn already taken when the drain ends.  After the warpgroup's reductions one thread
// adds 1 with release semantics.
//
// Warp roles (512 threads; register budgets set per warpgroup with setmaxnreg):
//   warp 0      TMA producer (converged warp, one elected lane issues): K_j, V_j per
//               segment; Q_i, dO_i, LSE_i, Dvec_i per step into a ring of stages
//   warp 1      MMA issuer (converged warp, one elected lane issues): G1..G5 and the
//               tcgen05.commit arrivals
//   warp 2      allocates / frees the 512 TMEM columns
//   warp 3      deterministic modes: semaphore poller (acquires the epilogue's turns ahead)
//   warps 4-11  two softmax-gradient warpgroups; warpgroup w handles query columns
//               [64w, 64w+64) of the tile, thread = KV row (TMEM lane)
//   warps 12-15 epilogue warpgroup: dQ partial TMEM -> ordered/atomic fp32 reduction in
//               global memory; at D = 64 also dK/dV TMEM -> bf16 at the end of each
//               segment (at D = 128 the softmax-gradient warpgroups drain dK and dV)
// TMEM columns: S^T then P^T [0,128), dP^T then dS^T [128,256), dK [256,256+D), dV [256+D,256+2D);
// the dQ partial reuses [128,256) at D=128 and has its own columns [384,448) at D=64.
#pragma once
#include "common.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace dash {
namespace {

// The tile kernel's compile-time mode: bits 0-1 the mask (0 full, 1 causal, 2 causal with an
// odd tile count under Symmetric Shift), bit 2 the two-strand accumulation of
// DASH_SCHED_SHIFT_DUAL (ordered).  `odd` of the schedule the mode implies:
__host__ __device__ constexpr int odd_of(int mode) { return (mode & 3) == 2 ? 1 : 0; }
__host__ __device__ constexpr bool dual_of(int mode) { return (mode & 4) != 0; }
// Two strands, causal mask, D = 64: each epilogue warp releases its own reductions (the
// semaphore then counts four releases per partial) instead of handing them to the releaser
// warp.  Measured: +2.5-4 % for the causal mask at D = 64 (1k-16k), where the step is half
// as long and the releaser's one-at-a-time releases fall behind; -10 % for the full mask at
// D = 64 and far worse at D = 128, whose longer reductions hold each warp at its release.
template <int D, int MODE>
__host__ __device__ constexpr bool warp_release_of() {
  return dual_of(MODE) && D == 64 && (MODE & 3) != 0;
}
// bit 3: a packed variable-length batch (per-sequence lengths, tokens addressed through 3-D
// tensor maps over [T, heads, D], the packed shift traversal)
__host__ __device__ constexpr bool varlen_of(int mode) { return (mode & 8) != 0; }

// Depth of the ring of mbarriers through which the semaphore poller hands a dQ tile's turn
// to the epilogue (ordered variant): the poller runs at most this many steps ahead
// (measured: 8 at D = 64, where steps are half as long; at D = 128, 4 for the full mask
// (1.5 % ahead of 8) and 8 for the causal mask (2 % ahead of 4)).
template <int D, int MODE>
struct Turns {
  static constexpr int kN = (D == 64 || (MODE & 3) != 0) ? 8 : 4;
};

template <int D, bool DET, int MODE>
struct BwdLayout {
  static constexpr int kStages = (D == 64) ? (DET ? 4 : 3) : 2;
  // D = 64, atomic variant: the dQ partial goes out by one bulk (TMA) reduction from a
  // shared-memory staging tile instead of 2048 vector reductions per step.  At D = 128 there
  // is no room for the staging tile.  The ordered variant keeps the vector reductions: a
  // bulk reduction's completion (needed before the semaphore release) arrives more than a
  // step later, longer than the one-step gap between a dQ tile's contributors.
  static constexpr bool kBulkDQ = (D == 64 && !DET);
  static constexpr int kTileBytes = D * kTile * 2;  // one [128 x D] bf16 tile
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kStageBytes = 2 * kTileBytes;  // Q_i and dO_i
  static constexpr int offK = 0;
  static constexpr int offV = kTileBytes;
  static constexpr int offStage = 2 * kTileBytes;  // stage s: Q at +s*kStageBytes, dO after
  static constexpr int offDS = offStage + kStages * kStageBytes;
  static constexpr int kDSBytes = kTile * kTile * 2;
  static constexpr int offStg = offDS + kDSBytes;  // fp32 dQ partial, tile-native layout
  static constexpr int kStgBytes = kBulkDQ ? kTile * D * 4 : 0;
  static constexpr int offLSE = offStg + kStgBytes;
  static constexpr int offDVEC = offLSE + kStages * kTile * 4;
  static constexpr int offBar = offDVEC + kStages * kTile * 4;
  // Ordered: the poller hands each turn to the epilogue through an mbarrier ring, on which
  // the epilogue's thread waits suspended instead of spinning on a shared-memory counter
  // (measured: +3 % at D = 128, equal at D = 64).  Two-strand mode: a third ring (the
  // epilogue's reductions issued, for the releaser warp) and the ranks of the ring's steps
  // (misc words from offRanks).
  static constexpr bool kTurnRing = DET;
  static constexpr int kTurns = Turns<D, MODE>::kN;
  static constexpr int kNumBars = 2 * kStages + 15 + (kTurnRing ? 3 * kTurns : 0);
  static constexpr int offMisc = offBar + kNumBars * 8;
  static constexpr int offRanks = offMisc + 32;
  static constexpr int kBytes = offRanks + (kTurnRing ? 4 * kTurns : 0);
  static constexpr uint32_t tS = 0, tDP = 128, tDK = 256, tDV = 256 + D;
  static constexpr uint32_t tDQ = (D == 64) ? 384 : 128;
  static constexpr bool kDQOwnCols = (D == 64);  // dQ partial does not alias dP^T
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kBytes <= 232448, "shared memory budget");
  static_assert(offDS % 1024 == 0 && offStage % 1024 == 0, "swizzle atoms need 1 KB alignment");
};

// Register budgets per warpgroup: the launch gives every thread 128 registers
// (512 x 128 = the SM's 64 K); producer/MMA warpgroup gives some back, the others take them.
// At D=64 the epilogue holds only 64 dQ values, so the softmax-gradient warpgroups get more.
template <int D>
struct RegSplit {
  static constexpr uint32_t kLaunch = 128;  // 65536 registers / 512 threads
  static constexpr uint32_t kCtl = 88;
  static constexpr uint32_t kSoftmax = (D == 64) ? 152 : 136;
  static constexpr uint32_t kEpi = (D == 64) ? 120 : 152;
  static_assert(kCtl + 2 * kSoftmax + kEpi == 4 * kLaunch, "register split must sum to the launch");
};

// Pacing of the dQ reductions: a burst of red.global fills the SM's memory instruction
// queue and stalls the tcgen05 and shared-memory traffic of the other warps behind it, so
// the epilogue sleeps briefly after every kRedPaceEvery vector reductions (measured: +22% at
// S = 16k, full mask, D = 128, atomic variant).  The single-chain ordered reductions are not
// paced: a dQ tile's next contributor follows one lock step later, and spreading them out
// lengthens that chain of turns by more than the stalls cost.  The two-strand mode paces
// them: a strand's next contributor follows two lock steps later (measured: the two strands
// gain nothing unpaced, and 150-250 ns every 4 reductions all give the same +16 %).
constexpr int kRedPaceEvery = 4;
constexpr uint32_t kRedPaceNs = 200;

// Work of this CTA: worker u (head-major over all heads) runs on CTA (u mod grid), in order.
// The mask of a launch: a constant in the full-mask build; read from the parameters in the
// causal builds (measured: folding it there too cost 7 % on GQA shapes).
template <int MODE>
__device__ __forceinline__ int mode_causal(const BwdParams &p) {
  return (MODE & 3) == 0 ? 0 : p.causal;
}

struct Plan {
  int sched, W, first, stride, nunits;
};
template <int MODE = 0>
__device__ __forceinline__ Plan cta_plan(const BwdParams &p) {
  Plan pl;
  pl.sched = p.sched;
  pl.W = p.workers;
  pl.first = (int)blockIdx.x;
  pl.stride = (int)gridDim.x;
  pl.nunits = varlen_of(MODE) ? p.units : p.heads * pl.W;
  return pl;
}

// One worker of one (batch, kv head): where its head's data and its packed position are.
struct Unit {
  int b, hkv, w;
  int N, S, odd;   // the head's tile count, length and Symmetric-Shift parity
  int W;           // workers of the head
  int wbase;       // packed index of the head's first worker
  size_t tiles0;   // index of tile (b, query head 0, q 0) in the per-tile arrays
  size_t tok0;     // row of the sequence's first token in the BSHD tensors
};
template <int MODE>
__device__ __forceinline__ Unit decode_unit(const BwdParams &p, const Plan &pl, int u) {
  Unit r;
  if constexpr (varlen_of(MODE)) {
    // the sequence: the last table entry whose first worker is at or before u (the table
    // holds non-empty sequences only)
    int lo = 0, hi = p.batch;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p.seq_wprefix[mid] <= u) lo = mid;
      else hi = mid;
    }
    const int4 sq = p.seqs[lo];
    r.b = lo;
    r.S = sq.x;
    r.tok0 = (size_t)sq.y;
    r.tiles0 = (size_t)sq.z;
    r.N = sq.w;
    r.odd = mode_causal<MODE>(p) ? (r.N & 1) : 0;
    r.W = sched_workers(kShift, mode_causal<MODE>(p), r.N, r.odd);
    const int local = u - p.seq_wprefix[lo];
    r.hkv = local / r.W;
    r.w = local - r.hkv * r.W;
    r.wbase = p.seq_wprefix[lo] + r.hkv * r.W;
    return r;
  }
  r.w = u % pl.W;
  const int hd = u / pl.W;  // head index b * Hkv + hkv
  r.hkv = hd % p.Hkv;
  r.b = hd / p.Hkv;
  r.N = p.N;
  r.S = p.S;
  r.odd = odd_of(MODE);
  r.W = pl.W;
  r.wbase = hd * pl.W;
  r.tiles0 = (size_t)r.b * p.H * p.N;
  r.tok0 = (size_t)r.b * p.S;
  return r;
}
// Index of the per-tile arrays (row vectors, semaphores, accumulator) of query head h, tile q.
__device__ __forceinline__ size_t tile_of(const Unit &un, int h, int q) {
  return un.tiles0 + (size_t)h * un.N + q;
}

template <int D, bool DET, int MODE>
struct Bars {
  uint64_t *full, *empty, *kv_full, *kv_empty, *s_full, *p_ready, *dp_full, *pds, *g5_done,
      *dq_empty, *dkv_full, *dkv_empty, *drain, *turn_full, *turn_empty, *added;
  __device__ explicit Bars(uint8_t *smem) {
    using L = BwdLayout<D, DET, MODE>;
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + L::offBar);
    full = b;
    empty = b + L::kStages;
    b += 2 * L::kStages;
    kv_full = b + 0;
    kv_empty = b + 1;
    s_full = b + 2;   // S^T in TMEM (MMA commit)
    p_ready = b + 3;  // P^T written over S^T by both softmax-gradient warpgroups (8 warps)
    dp_full = b + 4;  // dP^T in TMEM (MMA commit)
    pds = b + 6;      // [2]: P^T, dS^T of half x in TMEM, dS in shared memory (4 warps)
    g5_done = b + 10;
    dq_empty = b + 11;
    dkv_full = b + 12;
    dkv_empty = b + 13;
    drain = b + 14;
    turn_full = L::kTurnRing ? b + 15 : nullptr;  // [kTurns]: the step's semaphore reached its rank
    turn_empty = L::kTurnRing ? b + 15 + L::kTurns : nullptr;  // [kTurns]: the step was released
    added = L::kTurnRing ? b + 15 + 2 * L::kTurns : nullptr;  // [kTurns]: additions issued (dual)
  }
};

// One [128 rows x 64 columns] box of a head's rows, starting at row `row` of the unit's
// sequence: a 4-D map (D, heads, S, B) for uniform batches (rows past S read as zeros), a 3-D
// map (D, heads, T) over the packed tokens for a variable-length batch (rows past the
// sequence read the next sequence's tokens, which the softmax-gradient warps mask).
template <int MODE>
__device__ __forceinline__ void load_rows(void *dst, const CUtensorMap *map, uint64_t *bar,
                                          int col, int head, int row, const Unit &un) {
  if constexpr (varlen_of(MODE))
    tma_load_3d(dst, map, bar, col, head, (int)un.tok0 + row);
  else
    tma_load_4d(dst, map, bar, col, head, row, un.b);
}

// ---------------------------------------------------------------------------------------
// TMA producer: the whole warp runs the loop; one elected lane issues the copies.
template <int D, bool DET, int MODE>
__device__ void bwd_producer(const CUtensorMap *tq, const CUtensorMap *tk, const CUtensorMap *tv,
                             const CUtensorMap *tdo, const BwdParams &p, uint8_t *smem,
                             const Bars<D, DET, MODE> &bar, const Abort &ab) {
  using L = BwdLayout<D, DET, MODE>;
  uint32_t it = 0, seg_it = 0;
  int last_full[L::kStages];
#pragma unroll
  for (int s = 0; s < L::kStages; ++s) last_full[s] = -1;
  int last_kv = -1;
  bool ok = true;
  const Plan pl = cta_plan<MODE>(p);
  for (int u = pl.first; ok && u < pl.nunits; u += pl.stride) {
    const Unit un = decode_unit<MODE>(p, pl, u);
    const int nseg = sched_segments(pl.sched, mode_causal<MODE>(p), un.N, un.w, un.odd);
    for (int seg = 0; ok && seg < nseg; ++seg) {
      const int kv = seg_kv(pl.sched, mode_causal<MODE>(p), un.N, un.w, seg, un.odd);
      const int nsteps = seg_steps(pl.sched, mode_causal<MODE>(p), un.N, un.w, seg, un.odd);
      if (!mbar_wait_warp(bar.kv_empty, (seg_it & 1) ^ 1, ab)) {
        ok = false;
        break;
      }
      if (elect_one()) {
        mbar_arrive_expect_tx(bar.kv_full, 2 * L::kTileBytes);
        // rows past S (partial last tile) are outside the tensor map and arrive as zeros
#pragma unroll
        for (int bx = 0; bx < L::kBoxes; ++bx) {
          load_rows<MODE>(smem + L::offK + bx * kBoxBytes, tk, bar.kv_full, bx * kBoxCols, un.hkv,
                          kv * kTile, un);
          load_rows<MODE>(smem + L::offV + bx * kBoxBytes, tv, bar.kv_full, bx * kBoxCols, un.hkv,
                          kv * kTile, un);
        }
      }
      __syncwarp();
      last_kv = seg_it & 1;
      ++seg_it;
      // GQA: the G query heads of a step are visited back to back, so every head keeps the
      // schedule's lock step
      for (int t = 0; ok && t < nsteps; ++t) {
        const int q = step_q(pl.sched, mode_causal<MODE>(p), un.N, un.w, seg, t, un.odd);
        for (int g = 0; g < p.G; ++g) {
          const int h = un.hkv * p.G + g;
          const int s = it % L::kStages;
          const uint32_t ph = (it / L::kStages) & 1;
          if (!mbar_wait_warp(&bar.empty[s], ph ^ 1, ab)) {
            ok = false;
            break;
          }
          if (elect_one()) {
            mbar_arrive_expect_tx(&bar.full[s], L::kStageBytes + 2 * kTile * 4);
            uint8_t *sq = smem + L::offStage + s * L::kStageBytes;
#pragma unroll
            for (int bx = 0; bx < L::kBoxes; ++bx) {
              load_rows<MODE>(sq + bx * kBoxBytes, tq, &bar.full[s], bx * kBoxCols, h, q * kTile,
                              un);
              load_rows<MODE>(sq + L::kTileBytes + bx * kBoxBytes, tdo, &bar.full[s],
                              bx * kBoxCols, h, q * kTile, un);
            }
            // row vectors are stored per whole tile ([B,H,N*128], zero padding)
            const size_t roff = tile_of(un, h, q) * kTile;
            bulk_load(smem + L::offLSE + s * kTile * 4, p.lse2 + roff, kTile * 4, &bar.full[s]);
            bulk_load(smem + L::offDVEC + s * kTile * 4, p.dvec + roff, kTile * 4, &bar.full[s]);
          }
          __syncwarp();
          last_full[s] = (int)ph;
          ++it;
        }
      }
    }
  }
  if (!ok) {  // leave no copy in flight into shared memory
#pragma unroll
    for (int s = 0; s < L::kStages; ++s)
      if (last_full[s] >= 0) mbar_wait_drain(&bar.full[s], (uint32_t)last_full[s], 100000000ull);
    if (last_kv >= 0) mbar_wait_drain(bar.kv_full, (uint32_t)last_kv, 100000000ull);
  }
}

// ---------------------------------------------------------------------------------------
// MMA issuer: the whole warp runs the loop (waits, descriptors and control flow stay
// warp-uniform); one elected lane issues each tcgen05 instruction.  Once the
// softmax-gradient warps have written P^T over the current S^T columns, G3 and then the
// next step's S^T product are issued, so both run while those warps compute dS.
template <int D, bool DET, int MODE>
__device__ void bwd_mma(const BwdParams &p, uint8_t *smem, uint32_t tmem, const Bars<D, DET, MODE> &bar,
                        const Abort &ab) {
  using L = BwdLayout<D, DET, MODE>;
  constexpr uint32_t kIdescSS = make_idesc_bf16(128, 128, false, false);  // G1, G2
  constexpr uint32_t kIdescTS = make_idesc_bf16(128, D, false, true);     // G3, G4x
  constexpr uint32_t kIdescG5 = make_idesc_bf16(128, D, true, true);      // G5
  const uint32_t sbase = smem_u32(smem);
  // K-major views (contraction over D): k step of 16 columns = +32 B inside a box, boxes
  // 16 KB apart.  MN-major views (contraction over rows): k step of 16 rows = +2 KB,
  // 64-column boxes 16 KB apart (the leading-dimension offset).
  const uint32_t loK = desc_lo(sbase + L::offK, 16), loV = desc_lo(sbase + L::offV, 16);
  const uint32_t loKmn = desc_lo(sbase + L::offK, kBoxBytes);
  const uint32_t loDS = desc_lo(sbase + L::offDS, kBoxBytes);
  auto stage_addr = [&](uint32_t step) { return sbase + L::offStage + (step % L::kStages) * L::kStageBytes; };
  // G1: S^T = K_j Q_i^T for the step whose Q_i sits in stage (step % kStages)
  auto issue_g1 = [&](uint32_t step) {
    const uint32_t loQ = desc_lo(stage_addr(step), 16);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t ko = ((k >> 2) * kBoxBytes + (k & 3) * 32) >> 4;
      mma_ss_e(tmem + L::tS, desc_of(loK + ko), desc_of(loQ + ko), kIdescSS, k > 0);
    }
    mma_commit_e(bar.s_full);
  };
  uint32_t it = 0, seg_it = 0;
  bool ok = true;
  const Plan pl = cta_plan<MODE>(p);
  for (int u = pl.first; ok && u < pl.nunits; u += pl.stride) {
    const Unit un = decode_unit<MODE>(p, pl, u);
    const int nseg = sched_segments(pl.sched, mode_causal<MODE>(p), un.N, un.w, un.odd);
    for (int seg = 0; ok && seg < nseg; ++seg) {
      const int nsteps = seg_steps(pl.sched, mode_causal<MODE>(p), un.N, un.w, seg, un.odd) * p.G;
      // segment prologue: new K_j/V_j and G1 of the first step (the previous step's G3,
      // the last reader of the S^T columns, was issued before and runs first)
      if (!mbar_wait_warp(bar.kv_full, seg_it & 1, ab) ||
          !mbar_wait_warp(&bar.full[it % L::kStages], (it / L::kStages) & 1, ab)) {
        ok = false;
        break;
      }
      tc_fence_after();
      DASH_TRACE(p, 0);
      issue_g1(it);
      for (int st = 0; st < nsteps; ++st, ++it) {
        const uint32_t par = it & 1;
        const uint32_t aQ = stage_addr(it);
        const uint32_t loDO = desc_lo(aQ + L::kTileBytes, 16);
        const uint32_t loQmn = desc_lo(aQ, kBoxBytes);
        const uint32_t loDOmn = desc_lo(aQ + L::kTileBytes, kBoxBytes);
        // at D=128 the dP^T columns still hold the previous step's dQ partial
        if (!L::kDQOwnCols && it > 0) {
          if (!mbar_wait_warp(bar.dq_empty, (it - 1) & 1, ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        // G2: dP^T = V_j dO_i^T
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t ko = ((k >> 2) * kBoxBytes + (k & 3) * 32) >> 4;
          mma_ss_e(tmem + L::tDP, desc_of(loV + ko), desc_of(loDO + ko), kIdescSS, k > 0);
        }
        mma_commit_e(bar.dp_full);
        DASH_TRACE(p, 1);
        const bool fresh = (st == 0);  // first step of a segment starts dK/dV from zero
        // G3: dV_j += P^T dO_i, as soon as both warpgroups have put P^T (bf16x2) over the
        // first 32 of their 64 S^T columns; it runs while they compute dS
        if (!mbar_wait_warp(bar.p_ready, par, ab) ||
            (fresh && seg_it > 0 && !mbar_wait_warp(bar.dkv_empty, (seg_it - 1) & 1, ab))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ts_e(tmem + L::tDV, tmem + L::tS + 64 * (k >> 2) + 8 * (k & 3),
                   desc_of(loDOmn + ((k * 2048) >> 4)), kIdescTS, (fresh && k == 0) ? 0u : 1u);
        DASH_TRACE(p, 2);
        // G1 of the next step of this segment, once Q_{i'} has landed (G3 above read the
        // S^T columns first: the tensor pipe runs a CTA's MMAs in issue order)
        if (st + 1 < nsteps) {
          if (!mbar_wait_warp(&bar.full[(it + 1) % L::kStages], ((it + 1) / L::kStages) & 1, ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_g1(it + 1);
        }
        // G4x: dK_j += dS^T Q_i over query half x, once warpgroup x has put dS^T of its half
        // into the dP^T columns: within the 32-column chunk c of the half, in columns 16..31
#pragma unroll 1
        for (int x = 0; x < 2; ++x) {
          if (!mbar_wait_warp(&bar.pds[x], par, ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
          DASH_TRACE(p, 3 + x);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t acol = L::tDP + 64 * x + 32 * (k >> 1) + 8 * (k & 1) + 16;
            mma_ts_e(tmem + L::tDK, tmem + acol, desc_of(loQmn + (((4 * x + k) * 2048) >> 4)),
                     kIdescTS, (fresh && x == 0 && k == 0) ? 0u : 1u);
          }
        }
        if (!ok) break;
        mma_commit_e(&bar.empty[it % L::kStages]);
        // D = 128: the segment's dK_j, dV_j are complete once its last G3 and G4 are, and
        // the softmax-gradient warps drain them while G5 runs
        if (D == 128 && st == nsteps - 1) mma_commit_e(bar.dkv_full);
        if (L::kDQOwnCols && it > 0) {
          if (!mbar_wait_warp(bar.dq_empty, (it - 1) & 1, ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        // G5: dQ_part = dS K_j  (contraction over the 128 KV rows; both operands MN-major)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ss_e(tmem + L::tDQ, desc_of(loDS + ((k * 2048) >> 4)),
                   desc_of(loKmn + ((k * 2048) >> 4)), kIdescG5, k > 0);
        mma_commit_e(bar.g5_done);
        DASH_TRACE(p, 5);
        if (st == nsteps - 1) {
          mma_commit_e(bar.kv_empty);
          if (D == 64) mma_commit_e(bar.dkv_full);
        }
      }
      ++seg_it;
    }
  }
  // leave no MMA in flight
  mma_commit_e(bar.drain);
  mbar_wait_drain(bar.drain, 0, 100000000ull);
}

// ---------------------------------------------------------------------------------------
// Softmax-gradient warpgroup x (query columns [64x, 64x+64) of the tile; thread = KV row):
// read S^T, compute P^T in registers and write it (bf16x2) over the first 32 of the S^T
// columns just read (the A operand of G3); then, when dP^T has arrived, compute
// dS^T = P^T (dP^T - Dvec) chunk by chunk and write it (bf16x2) back over the dP^T columns
// just read; dS also goes to shared memory for G5.
template <int D, bool DET, int MODE>
__device__ void bwd_softmax_grad(const BwdParams &p, uint8_t *smem, uint32_t tmem,
                                 const Bars<D, DET, MODE> &bar, const Abort &ab) {
  using L = BwdLayout<D, DET, MODE>;
  const int warp = warp_id(), lane = lane_id();
  const int x = (warp - 4) >> 2;  // query half: columns [64x, 64x + 64)
  const int quad = warp & 3;
  const int r = quad * 32 + lane;  // KV row of this thread = TMEM lane
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const int c0 = x * 64;
  uint8_t *ds_row = smem + L::offDS + x * kBoxBytes + r * 128;
  uint32_t it = 0, seg_it = 0;
  bool ok = true;
  const Plan pl = cta_plan<MODE>(p);
  for (int u = pl.first; ok && u < pl.nunits; u += pl.stride) {
    const Unit un = decode_unit<MODE>(p, pl, u);
    const int nseg = sched_segments(pl.sched, mode_causal<MODE>(p), un.N, un.w, un.odd);
    for (int seg = 0; ok && seg < nseg; ++seg) {
      const int kv = seg_kv(pl.sched, mode_causal<MODE>(p), un.N, un.w, seg, un.odd);
      const int nsteps = seg_steps(pl.sched, mode_causal<MODE>(p), un.N, un.w, seg, un.odd);
      for (int t = 0; ok && t < nsteps; ++t) {
        for (int g = 0; g < p.G; ++g, ++it) {
          const int q = step_q(pl.sched, mode_causal<MODE>(p), un.N, un.w, seg, t, un.odd);
          const bool diag = mode_causal<MODE>(p) && (q == kv);
          // a key row past S (partial last tile) reads zeros; its P is set to zero so that
          // nothing of it (not even an overflowing exp of -LSE) reaches dS
          const bool kv_pad = (un.S & (kTile - 1)) != 0 && kv * kTile + r >= un.S;
          const int s = it % L::kStages;
          const uint32_t ph = (it / L::kStages) & 1;
          const uint32_t par = it & 1;
          if (!mbar_wait_warp(bar.s_full, par, ab) || !mbar_wait_warp(&bar.full[s], ph, ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float *lse_s = reinterpret_cast<const float *>(smem + L::offLSE + s * kTile * 4);
          const float *dvec_s = reinterpret_cast<const float *>(smem + L::offDVEC + s * kTile * 4);
          // P^T of this half, packed bf16x2 (the values G3 consumes); dS uses the same bf16 P
          uint32_t pk[32];
          {
            uint32_t sv[64];
            tmem_ld32(tmem + lane_off + L::tS + c0, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
            tmem_ld32(tmem + lane_off + L::tS + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
            tmem_ld_wait();
            if (lane == 0 && warp == 4 + 4 * x) DASH_TRACE(p, 6 + 4 * x);
#pragma unroll
            for (int c = 0; c < 64; c += 4) {
              const float4 l4 = *reinterpret_cast<const float4 *>(lse_s + c0 + c);
              const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
              float pv[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                pv[e] = ex2_approx(fmaf(__uint_as_float(sv[c + e]), p.scale_log2, -lv[e]));
              }
              pk[c / 2] = pack_bf16(pv[0], pv[1]);
              pk[c / 2 + 1] = pack_bf16(pv[2], pv[3]);
            }
          }
          if (kv_pad) {  // uniform per thread: outside the exp loop
#pragma unroll
            for (int m = 0; m < 32; ++m) pk[m] = 0u;
          }
          // causal diagonal tile: query column < key row r is masked.  Applied to the packed
          // words once per diagonal step, not per element inside the exp loop (that loop is
          // bound by instruction issue: a per-element select cost 9 % at D = 64); the
          // unmasked exponentials computed there are overwritten here
          if (diag) {
#pragma unroll
            for (int m = 0; m < 32; ++m) {
              const int col = c0 + 2 * m;
              if (col + 1 < r) pk[m] = 0u;
              else if (col < r) pk[m] &= 0xFFFF0000u;
            }
          }
          // a packed variable-length batch: query rows past the sequence hold the next
          // sequence's tokens (not zeros), so their columns of P are cleared (once per partial
          // last tile, on the packed words)
          if (varlen_of(MODE) && (q + 1) * kTile > un.S) {
            const int lim = un.S - q * kTile;
#pragma unroll
            for (int m = 0; m < 32; ++m) {
              const int col = c0 + 2 * m;
              if (col >= lim) pk[m] = 0u;
              else if (col + 1 >= lim) pk[m] &= 0x0000FFFFu;
            }
          }
          // P^T (bf16x2) over the first 32 of this half's S^T columns, all read above: the
          // A operand of G3, which then runs while dS is computed
          tmem_st16(tmem + lane_off + L::tS + c0, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
          tmem_st16(tmem + lane_off + L::tS + c0 + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]));
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar.p_ready);
          if (lane == 0 && warp == 4 + 4 * x) DASH_TRACE(p, 7 + 4 * x);
          // Dvec of the first chunk into registers while dP^T is still being computed
          float dv[32];
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            *reinterpret_cast<float4 *>(&dv[c]) = *reinterpret_cast<const float4 *>(dvec_s + c0 + c);
          if (!mbar_wait_warp(bar.dp_full, par, ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0 && warp == 4 + 4 * x) DASH_TRACE(p, 8 + 4 * x);
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            const uint32_t col = L::tDP + c0 + 32 * ch;
            uint32_t dpv[32], dk[16];
            tmem_ld32(tmem + lane_off + col, dpv);
            tmem_ld_wait();
            if (lane == 0 && warp == 4) DASH_TRACE(p, 18 + 4 * ch);
#pragma unroll
            for (int m = 0; m < 16; ++m) {
              const uint32_t w = pk[16 * ch + m];
              const float p0 = __uint_as_float(w << 16), p1 = __uint_as_float(w & 0xFFFF0000u);
              dk[m] = pack_bf16(p0 * (__uint_as_float(dpv[2 * m]) - dv[2 * m]),
                                p1 * (__uint_as_float(dpv[2 * m + 1]) - dv[2 * m + 1]));
            }
            if (ch == 0) {  // next chunk's Dvec
#pragma unroll
              for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4 *>(&dv[c]) =
                    *reinterpret_cast<const float4 *>(dvec_s + c0 + 32 + c);
            }
            if (lane == 0 && warp == 4) DASH_TRACE(p, 19 + 4 * ch);
            // dS^T into columns 16..31 of the chunk's own (already read) dP^T columns
            tmem_st16(tmem + lane_off + col + 16, dk);
            if (lane == 0 && warp == 4) DASH_TRACE(p, 20 + 4 * ch);
            // dS into shared memory as the MN-major A operand of G5: row r of box x,
            // 16-byte chunk (4ch + j) at position (4ch + j) ^ (r % 8)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int cj = ch * 4 + j;
              *reinterpret_cast<uint4 *>(ds_row + ((cj ^ (r & 7)) << 4)) =
                  make_uint4(dk[4 * j], dk[4 * j + 1], dk[4 * j + 2], dk[4 * j + 3]);
            }
            if (lane == 0 && warp == 4) DASH_TRACE(p, 21 + 4 * ch);
          }
          fence_proxy_async_smem();
          if (lane == 0 && warp == 4) DASH_TRACE(p, 26);
          tmem_st_wait();
          if (lane == 0 && warp == 4) DASH_TRACE(p, 27);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&bar.pds[x]);
            mbar_arrive(&bar.empty[s]);
            if (warp == 4 + 4 * x) DASH_TRACE(p, 9 + 4 * x);
          }
        }
      }
      if (!ok) break;
      // segment end, D = 128: warpgroup 0 takes dK_j (scaled), warpgroup 1 dV_j, to bf16.
      // The two warpgroups are otherwise idle here (the next segment's S^T needs its K_j),
      // while the epilogue warpgroup still adds the segment's last dQ partial; drained by the
      // epilogue, dK/dV would wait behind those reductions and hold the next segment's G3
      // (measured: +4.5 % at S = 512, +1.5 % at 4k, full mask).  At D = 64, where these
      // warps bound the step, the epilogue keeps the drain (-1.3 % there otherwise).
      if constexpr (D == 128) {
        if (!mbar_wait_warp(bar.dkv_full, seg_it & 1, ab)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tcol = x == 0 ? L::tDK : L::tDV;
        const float mul = x == 0 ? p.scale : 1.f;
        __nv_bfloat16 *dst = (x == 0 ? p.dk : p.dv) +
                             ((un.tok0 + (size_t)kv * kTile + r) * p.Hkv + un.hkv) * D;
        const bool keep = kv * kTile + r < un.S;  // rows past S belong to no key
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t vv[32], pk2[16];
          tmem_ld32(tmem + lane_off + tcol + ch * 32, vv);
          tmem_ld_wait();
          if (ch == D / 32 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar.dkv_empty);
          }
#pragma unroll
          for (int m = 0; m < 16; ++m)
            pk2[m] = pack_bf16(__uint_as_float(vv[2 * m]) * mul,
                               __uint_as_float(vv[2 * m + 1]) * mul);
          if (keep) {
            uint4 *d4 = reinterpret_cast<uint4 *>(dst + ch * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              d4[j] = make_uint4(pk2[4 * j], pk2[4 * j + 1], pk2[4 * j + 2], pk2[4 * j + 3]);
          }
        }
        ++seg_it;
      } else {
        (void)seg_it;
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// The dQ-tile order of one worker: the rank of its contribution to query tile q from KV
// block kv.  Plain shift order when the head's workers share one round of the grid, else
// the packed-shift rank within the worker's phase (closed forms, sched.cuh), the phase being
// fixed for the whole unit.
struct UnitOrder {
  int ph_lo, ph_hi;
  bool split;
};
__device__ __forceinline__ UnitOrder unit_order(const BwdParams &p, const Unit &un) {
  UnitOrder o;
  o.ph_lo = 0;
  o.ph_hi = un.W;
  if (p.packed) packed_phase_at(un.wbase, un.W, (int)gridDim.x, un.w, &o.ph_lo, &o.ph_hi);
  o.split = p.packed && (o.ph_hi - o.ph_lo) != un.W;
  return o;
}
template <int MODE>
__device__ __forceinline__ int step_rank(const BwdParams &p, const Plan &pl, const Unit &un,
                                         const UnitOrder &o, int q, int kv) {
  if (!o.split) return dq_rank(pl.sched, mode_causal<MODE>(p), un.N, q, kv, un.odd);
  return rank_in_phase(mode_causal<MODE>(p), un.N, q, kv, o.ph_lo, o.ph_hi, un.odd);
}

// Semaphore poller (warp 3, deterministic modes): walks this CTA's steps in the
// epilogue's order and, for each, waits until the step's dQ tile semaphore (two strands:
// the semaphore of the partial's strand) has counted the partials before it, then hands the
// turn -- and, with two strands, the rank -- to the epilogue by arriving on the step's slot
// of the turn ring (it runs at most kTurns steps ahead).  The L2 round trips of the polling
// thus overlap the computation of the dQ partial instead of following its drain.
template <int D, bool DET, int MODE>
__device__ void bwd_sem_poller(const BwdParams &p, uint8_t *smem, const Abort &ab) {
  using L = BwdLayout<D, DET, MODE>;
  constexpr bool kDual = dual_of(MODE);
  volatile int *ranks = reinterpret_cast<volatile int *>(smem + L::offRanks);
  const int lane = lane_id();
  const Bars<D, DET, MODE> bar(smem);
  uint32_t it = 0;
  const Plan pl = cta_plan<MODE>(p);
  for (int u = pl.first; u < pl.nunits; u += pl.stride) {
    const Unit un = decode_unit<MODE>(p, pl, u);
    const UnitOrder o = unit_order(p, un);
    const int nseg = sched_segments(pl.sched, mode_causal<MODE>(p), un.N, un.w, un.odd);
    for (int seg = 0; seg < nseg; ++seg) {
      const int kv = seg_kv(pl.sched, mode_causal<MODE>(p), un.N, un.w, seg, un.odd);
      const int nsteps = seg_steps(pl.sched, mode_causal<MODE>(p), un.N, un.w, seg, un.odd);
      for (int t = 0; t < nsteps; ++t) {
        const int q = step_q(pl.sched, mode_causal<MODE>(p), un.N, un.w, seg, t, un.odd);
        const int rank = step_rank<MODE>(p, pl, un, o, q, kv);
        for (int g = 0; g < p.G; ++g, ++it) {
          const int h = un.hkv * p.G + g;
          // the step's semaphore: the tile's, or (two strands) that of strand rank % 2, on which
          // the partial's turn comes when the strand has counted its rank / 2 earlier partials
          const size_t ptile = tile_of(un, h, q);
          const int *sem = kDual ? p.sem + ptile * 2 + (rank & 1) : p.sem + ptile;
          const int want = (warp_release_of<D, MODE>() ? 4 : 1) * (kDual ? rank >> 1 : rank);
          int ok = 1;
          if (lane == 0) {
            // the slot is free once the step kTurns earlier has been released
            const uint32_t slot = it % L::kTurns, wrap = (it / L::kTurns) & 1;
            // (with per-warp releases the slot is free once the four warps have released)
            ok = mbar_wait(warp_release_of<D, MODE>() ? &bar.added[slot] : &bar.turn_empty[slot],
                           wrap ^ 1, ab)
                     ? 1
                     : 0;
            DASH_TRACE(p, 29);
            ok = ok && sem_wait(sem, want, ab) ? 1 : 0;
            DASH_TRACE(p, 30);
            if (ok) {
              ranks[slot] = rank;
              mbar_arrive(&bar.turn_full[slot]);
            }
            // audit record of the executed order (dash_attn_bwd_order_log)
            if (ok && p.order_log) p.order_log[ptile * p.log_stride + kv] = rank;
          }
          if (!__shfl_sync(0xffffffffu, ok, 0)) return;
        }
      }
    }
  }
}

// Releaser (warp 2 in the two-strand mode, after it has allocated the tensor memory): once
// the epilogue warpgroup has issued a step's reductions (each of its four warps arrived on
// the step's `added` slot after its own), advances the semaphore of the step's
// dQ tile and strand by one with gpu-scope release semantics -- which orders every one of
// those reductions before it -- and frees the turn-ring slot for the poller.  The release
// waits until the reductions are performed; done here, that wait does not hold the
// epilogue, which goes on to drain the next dQ partial (measured: +16 % together with the
// paced reductions at S = 16k, full mask; neither helps alone).
template <int D, bool DET, int MODE>
__device__ void bwd_releaser(const BwdParams &p, uint8_t *smem, const Bars<D, DET, MODE> &bar,
                             const Abort &ab) {
  using L = BwdLayout<D, DET, MODE>;
  const int lane = lane_id();
  const volatile int *ranks = reinterpret_cast<const volatile int *>(smem + L::offRanks);
  uint32_t it = 0;
  const Plan pl = cta_plan<MODE>(p);
  for (int u = pl.first; u < pl.nunits; u += pl.stride) {
    const Unit un = decode_unit<MODE>(p, pl, u);
    const int nseg = sched_segments(pl.sched, mode_causal<MODE>(p), un.N, un.w, un.odd);
    for (int seg = 0; seg < nseg; ++seg) {
      const int nsteps = seg_steps(pl.sched, mode_causal<MODE>(p), un.N, un.w, seg, un.odd);
      for (int t = 0; t < nsteps; ++t) {
        const int q = step_q(pl.sched, mode_causal<MODE>(p), un.N, un.w, seg, t, un.odd);
        for (int g = 0; g < p.G; ++g, ++it) {
          const size_t ptile = tile_of(un, un.hkv * p.G + g, q);
          int ok = 1;
          if (lane == 0) {
            const uint32_t slot = it % L::kTurns;
            ok = mbar_wait(&bar.added[slot], (it / L::kTurns) & 1, ab) ? 1 : 0;
            if (ok) {
              // the slot's rank stays valid until turn_empty lets the poller reuse the slot
              red_release_add(p.sem + ptile * 2 + (ranks[slot] & 1), 1);
              DASH_TRACE(p, 31);
              mbar_arrive(&bar.turn_empty[slot]);
            }
          }
          if (!__shfl_sync(0xffffffffu, ok, 0)) return;
        }
      }
    }
  }
}

// What the epilogue learns with its turn (ordered modes), from the partial's rank in its dQ
// tile: 1 + its strand (rank mod 2 with two strands, else 0) + 2 if it is its strand's first
// partial (rank < strands; used with two strands).  0 stands for a failed wait.
template <bool kDual>
__device__ __forceinline__ int turn_code(int rank) {
  constexpr int K = kDual ? 2 : 1;
  return 1 + (kDual ? (rank & 1) : 0) + (rank < K ? 2 : 0);
}

template <int D, bool DET, int MODE>
__device__ void bwd_epilogue(const BwdParams &p, uint8_t *smem, uint32_t tmem, const Bars<D, DET, MODE> &bar,
                             const Abort &ab) {
  using L = BwdLayout<D, DET, MODE>;
  constexpr bool kDual = dual_of(MODE);
  const int warp = warp_id(), lane = lane_id();
  const int et = threadIdx.x - 12 * 32;  // 0..127
  const int quad = warp & 3;
  const int r = quad * 32 + lane;  // query row (dQ) or KV row (dK/dV) = TMEM lane
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  // decisions taken by thread 0 and read by the warpgroup after a named barrier; two
  // slots alternate so a fast thread 0 never overwrites one that is still being read
  volatile int *decision = reinterpret_cast<volatile int *>(smem + L::offMisc + 8);
  uint32_t it = 0, seg_it = 0, dec = 0;
  bool ok = true;
  auto agree_int = [&](int mine) -> int {
    if (et == 0) decision[dec & 1] = mine;
    named_bar_sync(1, 128);
    return decision[dec++ & 1];
  };
  const volatile int *ranks = reinterpret_cast<const volatile int *>(smem + L::offRanks);
  constexpr bool kBulk = L::kBulkDQ && !DET;
  const Plan pl = cta_plan<MODE>(p);
  for (int u = pl.first; ok && u < pl.nunits; u += pl.stride) {
    const Unit un = decode_unit<MODE>(p, pl, u);
    const int nseg = sched_segments(pl.sched, mode_causal<MODE>(p), un.N, un.w, un.odd);
    for (int seg = 0; ok && seg < nseg; ++seg) {
      const int kv = seg_kv(pl.sched, mode_causal<MODE>(p), un.N, un.w, seg, un.odd);
      const int nsteps = seg_steps(pl.sched, mode_causal<MODE>(p), un.N, un.w, seg, un.odd);
      for (int t = 0; ok && t < nsteps; ++t) {
        for (int g = 0; g < p.G; ++g, ++it) {
          const int h = un.hkv * p.G + g;
          const int q = step_q(pl.sched, mode_causal<MODE>(p), un.N, un.w, seg, t, un.odd);
          const size_t tile_idx = tile_of(un, h, q);
          // two strands: thread 0 also takes the step's turn before the warpgroup meets, and
          // the strand travels with the decision, so no second barrier follows the drain (the
          // turn is normally ready thousands of cycles before the dQ partial; measured: the
          // separate wait and barrier after the drain cost ~540 cycles a step)
          int g5 = 1;
          if (et == 0) {
            g5 = mbar_wait(bar.g5_done, it & 1, ab) ? 1 : 0;
            if (kDual && g5)
              g5 = mbar_wait(&bar.turn_full[it % L::kTurns], (it / L::kTurns) & 1, ab)
                       ? turn_code<kDual>(ranks[it % L::kTurns])
                       : 0;
          }
          g5 = agree_int(g5);
          if (!g5) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (et == 0) DASH_TRACE(p, 14);
          // the whole dQ partial row to registers, then give the columns back
          uint32_t v[D / 32][32];
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) tmem_ld32(tmem + lane_off + L::tDQ + ch * 32, v[ch]);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar.dq_empty);
          if (et == 0) DASH_TRACE(p, 15);
          if constexpr (kBulk) {
            float *tile = p.dqacc + tile_idx * (size_t)(kTile * D);
            // the partial into the staging tile (same tile-native layout as the accumulator;
            // the previous reduction finished reading it before thread 0 left the last step)
            float4 *stg = reinterpret_cast<float4 *>(smem + L::offStg);
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                stg[(ch * 8 + j) * kTile + r] =
                    make_float4(__uint_as_float(v[ch][4 * j]), __uint_as_float(v[ch][4 * j + 1]),
                                __uint_as_float(v[ch][4 * j + 2]), __uint_as_float(v[ch][4 * j + 3]));
            }
            fence_proxy_async_smem();
            // every row staged: one thread adds the whole tile with a single bulk reduction
            named_bar_sync(1, 128);
            if (et == 0) {
              DASH_TRACE(p, 16);
              bulk_reduce_add_f32(tile, stg, kTile * D * 4);
              bulk_wait_read();
              DASH_TRACE(p, 17);
            }
            continue;
          }
          // the semaphore counts the partials added so far: the contributor of rank r goes
          // once rank r-1 has released it; the poller warp has been watching it (single
          // strand: the turn is taken here; two strands: with the G5 wait above, as 1 + the
          // strand of the partial)
          int turn = g5;
          if constexpr (DET && !kDual) {
            if (et == 0) {
              turn = mbar_wait(&bar.turn_full[it % L::kTurns], (it / L::kTurns) & 1, ab)
                         ? turn_code<kDual>(ranks[it % L::kTurns])
                         : 0;
              DASH_TRACE(p, 28);
            }
            turn = agree_int(turn);
          }
          if (turn == 0) {
            ok = false;
            break;
          }
          // two strands: the first partial of a strand is stored, so their accumulator needs
          // no clearing beforehand (measured: +12 % for the whole call at S = 512, neutral at
          // 16k; with one strand the second copy of the unrolled loop cost 3-5 % at long S,
          // so there the accumulator is cleared and every partial added)
          const bool first = kDual && ((turn - 1) >> 1) != 0;
          const size_t acc_idx = kDual ? tile_idx * 2 + ((turn - 1) & 1) : tile_idx;
          float *tile = p.dqacc + acc_idx * (size_t)(kTile * D);
          if (et == 0) DASH_TRACE(p, 16);
          // one branch per step (a branch per vector inside the unrolled loop cost 4-7 %:
          // the epilogue shares its SMSPs with the issue-bound softmax-gradient warps)
          auto out_partial = [&](auto op) {
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int c4 = ch * 8 + j;
                op(tile + ((size_t)c4 * kTile + r) * 4, __uint_as_float(v[ch][4 * j]),
                   __uint_as_float(v[ch][4 * j + 1]), __uint_as_float(v[ch][4 * j + 2]),
                   __uint_as_float(v[ch][4 * j + 3]));
                if ((!DET || kDual) && (c4 + 1) % kRedPaceEvery == 0 && c4 + 1 < D / 4)
                  __nanosleep(kRedPaceNs);
              }
            }
          };
          if (first)
            out_partial([](float *d, float a, float b, float c, float e) { st_v4(d, a, b, c, e); });
          else
            out_partial([](float *d, float a, float b, float c, float e) { red_add_v4(d, a, b, c, e); });
          if constexpr (warp_release_of<D, MODE>()) {  // each warp releases its own
            __syncwarp();
            if (lane == 0) {
              red_release_add(p.sem + tile_idx * 2 + ((turn - 1) & 1), 1);
              mbar_arrive(&bar.added[it % L::kTurns]);
            }
          } else if constexpr (kDual) {  // each warp's reductions issued: the releaser releases
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.added[it % L::kTurns]);
          } else if constexpr (DET) {  // one release for the warpgroup, after all reductions
            named_bar_sync(1, 128);
            if (et == 0) {
              red_release_add(p.sem + tile_idx, 1);
              mbar_arrive(&bar.turn_empty[it % L::kTurns]);
            }
          }
          if (et == 0) DASH_TRACE(p, 17);
        }
      }
      if (!ok) break;
      if constexpr (D == 64) {  // segment end: dK_j (scaled) and dV_j to bf16
        int got = 1;
        if (et == 0) got = mbar_wait(bar.dkv_full, seg_it & 1, ab) ? 1 : 0;
        if (!agree_int(got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const size_t orow = ((un.tok0 + (size_t)kv * kTile + r) * p.Hkv + un.hkv) * D;
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t kk[32], vv[32];
          tmem_ld32(tmem + lane_off + L::tDK + ch * 32, kk);
          tmem_ld32(tmem + lane_off + L::tDV + ch * 32, vv);
          tmem_ld_wait();
          if (ch == D / 32 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar.dkv_empty);
          }
          uint32_t kp[16], vp[16];
#pragma unroll
          for (int m = 0; m < 16; ++m) {
            kp[m] = pack_bf16(__uint_as_float(kk[2 * m]) * p.scale,
                              __uint_as_float(kk[2 * m + 1]) * p.scale);
            vp[m] = pack_bf16(__uint_as_float(vv[2 * m]), __uint_as_float(vv[2 * m + 1]));
          }
          uint4 *dkp = reinterpret_cast<uint4 *>(p.dk + orow + ch * 32);
          uint4 *dvp = reinterpret_cast<uint4 *>(p.dv + orow + ch * 32);
          if (kv * kTile + r < un.S) {  // rows past S belong to no key
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              dkp[j] = make_uint4(kp[4 * j], kp[4 * j + 1], kp[4 * j + 2], kp[4 * j + 3]);
              dvp[j] = make_uint4(vp[4 * j], vp[4 * j + 1], vp[4 * j + 2], vp[4 * j + 3]);
            }
          }
        }
        ++seg_it;
      } else {
        (void)kv;
        (void)seg_it;
      }
    }
  }
  // leave no bulk reduction in flight
  if (kBulk && et == 0) bulk_wait_done();
}

// ---------------------------------------------------------------------------------------
template <int D, bool DET, int MODE>
__global__ void __launch_bounds__(512, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const BwdParams p) {
  using L = BwdLayout<D, DET, MODE>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, kErrSmemAlign);
    return;
  }
  const Bars<D, DET, MODE> bar(smem);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + L::offMisc);
  int *s_abort = reinterpret_cast<int *>(smem + L::offMisc + 4);
  const Abort ab{s_abort, p.status, p.wait_ns};
  const int warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&bar.full[s], 1);
      mbar_init(&bar.empty[s], 1 + 8);  // MMA commit + 8 softmax-gradient warps
    }
    mbar_init(bar.kv_full, 1);
    mbar_init(bar.kv_empty, 1);
    mbar_init(bar.s_full, 1);
    mbar_init(bar.p_ready, 8);
    mbar_init(bar.dp_full, 1);
    mbar_init(&bar.pds[0], 4);
    mbar_init(&bar.pds[1], 4);
    mbar_init(bar.g5_done, 1);
    mbar_init(bar.dq_empty, 4);
    mbar_init(bar.dkv_full, 1);
    mbar_init(bar.dkv_empty, D == 128 ? 8 : 4);  // the warps that drain dK/dV
    mbar_init(bar.drain, 1);
    if constexpr (L::kTurnRing) {
      for (int i = 0; i < L::kTurns; ++i) {
        mbar_init(&bar.turn_full[i], 1);
        mbar_init(&bar.turn_empty[i], 1);
        mbar_init(&bar.added[i], 4);  // the four epilogue warps (two-strand mode)
      }
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == 2) {
    tmem_alloc(s_tmem, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp < 4) {
    regs_set<RegSplit<D>::kCtl, RegSplit<D>::kLaunch>();
    if (warp == 0) bwd_producer<D, DET, MODE>(&tm_q, &tm_k, &tm_v, &tm_do, p, smem, bar, ab);
    if (warp == 1) bwd_mma<D, DET, MODE>(p, smem, tmem, bar, ab);
    if constexpr (DET) {
      if (warp == 3) bwd_sem_poller<D, DET, MODE>(p, smem, ab);
      if constexpr (dual_of(MODE) && !warp_release_of<D, MODE>()) {
        if (warp == 2) bwd_releaser<D, DET, MODE>(p, smem, bar, ab);
      }
    }
  } else if (warp < 12) {
    regs_set<RegSplit<D>::kSoftmax, RegSplit<D>::kLaunch>();
    bwd_softmax_grad<D, DET, MODE>(p, smem, tmem, bar, ab);
  } else {
    regs_set<RegSplit<D>::kEpi, RegSplit<D>::kLaunch>();
    bwd_epilogue<D, DET, MODE>(p, smem, tmem, bar, ab);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int D, bool DET, int MODE>
cudaError_t launch_bwd_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         const CUtensorMap &tdo, const BwdParams &p, int grid, cudaStream_t stream) {
  using L = BwdLayout<D, DET, MODE>;
  auto kern = bwd_kernel<D, DET, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  // the per-warpgroup register split assumes exactly 128 registers per thread at launch
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != (int)RegSplit<D>::kLaunch) return cudaErrorInvalidConfiguration;
  // ordered schedules: workers wait on workers of other CTAs, so every CTA must be resident
  // at once; a cooperative launch makes the runtime guarantee that (or refuse the launch)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(512);
  cfg.dynamicSmemBytes = L::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = DET ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tdo, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

// MODE bits 0-1: 0 full mask, 1 causal, 2 causal with the padded (odd-N) Symmetric Shift;
// bit 2: two accumulation strands (ordered); bit 3: a packed variable-length batch.  The
// parity is a constant inside the kernel (per sequence at run time in the packed batch), and
// so is the mask in the full-mask build, which then carries no diagonal or schedule branches
// of the causal one (measured: +2 %).
template <int MODE>
cudaError_t launch_bwd_o(int D, bool deterministic, const CUtensorMap &tq, const CUtensorMap &tk,
                         const CUtensorMap &tv, const CUtensorMap &tdo, const BwdParams &p, int grid,
                         cudaStream_t stream) {
  if constexpr (dual_of(MODE)) {
    if (!deterministic) return cudaErrorInvalidValue;
    if (D == 64) return launch_bwd_t<64, true, MODE>(tq, tk, tv, tdo, p, grid, stream);
    return launch_bwd_t<128, true, MODE>(tq, tk, tv, tdo, p, grid, stream);
  } else {
    if (D == 64)
      return deterministic ? launch_bwd_t<64, true, MODE>(tq, tk, tv, tdo, p, grid, stream)
                           : launch_bwd_t<64, false, MODE>(tq, tk, tv, tdo, p, grid, stream);
    return deterministic ? launch_bwd_t<128, true, MODE>(tq, tk, tv, tdo, p, grid, stream)
                         : launch_bwd_t<128, false, MODE>(tq, tk, tv, tdo, p, grid, stream);
  }
}

}  // namespace dash
