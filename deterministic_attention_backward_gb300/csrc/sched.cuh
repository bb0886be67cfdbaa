// sched.cuh -- the DASH tile schedules as closed-form integer functions, shared by the
// backward kernel (device) and the host-side query entry points.
//
// A head has N = S/128 KV blocks and N query tiles.  A *worker* is the per-head unit of
// work that one persistent CTA executes without interruption: one KV block, or -- for the
// causal Symmetric Shift -- the pair (c, N-1-c).  A worker runs one or two *segments*
// (one KV block each, whose dK/dV stay in tensor memory for the whole segment); step t
// of a segment visits one query tile q and adds its dQ partial as the rank-th
// contribution to dQ tile q.
//
// Schedules (DASH pages, gist.science technical summary, section 2.2):
//  SERIAL (deterministic baseline, section 1): worker j visits q ascending
//    (full: 0..N-1, causal: j..N-1); tile q adds KV blocks in ascending order.
//  DESCENDING (section 2.2 A): visits q descending (full: N-1..0, causal: N-1..j); the
//    accumulation order is unchanged.
//  SHIFT, full mask (section 2.2 B): worker j visits q = (j + t) mod N.  All workers are
//    in lock step on distinct tiles, so tile q receives KV blocks q, q-1, ... (mod N):
//    rank = (q - kv) mod N.
//  SHIFT, causal mask = Symmetric Shift (section 2.2 B): h = N/2, worker c owns KV blocks
//    c and N-1-c.  Segment 0 (block c): phase 1, t < h: q = h + (c + t) mod h (the dense
//    lower-left rectangle q >= h, kv < h, cyclic); then q = c + (t - h) for t in
//    [h, N-c) (block c's rows of the upper-left triangle).  Segment 1 (block N-1-c):
//    q = N-1-t for t in [0, c].  In lock step the contributions to a tile arrive at
//    distinct steps; their step order gives the ranks
//      q <  h            : rank = q - kv
//      q >= h, kv <  h   : rank = (q - h - kv) mod h
//      q >= h, kv >= h   : rank = kv       (= h + (kv - h), after the h rectangle ones)
//    Odd N (the pages cover even N only): the head is padded with an empty KV block and
//    query tile N, the even schedule of Np = N+1 is laid out, and the steps that touch
//    the padding are dropped.  Worker 0 then owns block 0 alone and worker c >= 1 the
//    pair (c, N-c); every worker has N steps.  Ranks are the padded schedule's (formulas
//    above with h = Np/2): its lock-step order, in which the dropped steps are idle
//    slots.  Run with waits, a head finishes in N+1 steps, as for even N.
//  ATOMIC: no order; it visits tiles in the shift order (conflict-free and, for the causal
//    mask, balanced), the most favourable traversal, so that the deterministic schedules
//    are compared against the fastest non-deterministic backward.
#pragma once

#if defined(__CUDACC__)
#define DASH_HD __host__ __device__ __forceinline__
#else
#define DASH_HD inline
#endif

namespace dash {

// kShiftFill is the packed shift schedule (below): the shift workers of all heads dealt to
// every CTA of the grid; on the device it runs the kShift traversal with packed ranks.
// kShiftDual: the packed shift schedule with each dQ tile accumulated in two strands
// (partial of rank r into strand r mod 2, in rank order; strand 0 + strand 1 at the end).
enum Sched : int {
  kAtomic = 0,
  kSerial = 1,
  kDescending = 2,
  kShift = 3,
  kShiftFill = 4,
  kShiftDual = 6
};

// Which visiting order a schedule uses (ATOMIC borrows the shift order; the fill mode's
// shift heads use the shift order).
DASH_HD int traversal(int sched, int causal, int N) {
  (void)causal;
  (void)N;
  if (sched == kShiftFill || sched == kShiftDual || sched == kAtomic) return kShift;
  return sched;
}

DASH_HD bool sym_shift(int sched, int causal) { return sched == kShift && causal; }
// `odd` (below) is N & 1.  It only matters for Symmetric Shift; the backward kernel is
// compiled per mask and parity and receives it (and `causal`) as constants, so that an
// even N runs the plain even-N arithmetic.  The padded tile count of Symmetric Shift (N rounded up to even) and
// its half:
DASH_HD int sym_np(int N, int odd) { return N + odd; }
DASH_HD int sym_h(int N, int odd) { return (N + odd) >> 1; }

DASH_HD int sched_workers(int sched, int causal, int N, int odd) {
  return sym_shift(sched, causal) ? sym_h(N, odd) : N;
}
// Segments of worker w: two for a Symmetric Shift pair, one for worker 0 of an odd N (its
// partner would be the padding block).
DASH_HD int sched_segments(int sched, int causal, int N, int w, int odd) {
  (void)N;
  if (!sym_shift(sched, causal)) return 1;
  return (odd && w == 0) ? 1 : 2;
}
DASH_HD int seg_kv(int sched, int causal, int N, int w, int seg, int odd) {
  return (sym_shift(sched, causal) && seg == 1) ? sym_np(N, odd) - 1 - w : w;
}
DASH_HD int seg_steps(int sched, int causal, int N, int w, int seg, int odd) {
  if (!causal) return N;
  if (sched == kShift) return seg == 0 ? N - w : w + 1 - odd;
  return N - w;
}
DASH_HD int step_q(int sched, int causal, int N, int w, int seg, int t, int odd) {
  switch (sched) {
    case kDescending:
      return N - 1 - t;
    case kShift: {
      if (!causal) {
        int q = w + t;
        return q >= N ? q - N : q;
      }
      // t is the step among those kept; for odd N, skip the padded schedule's steps on
      // the padding tile (step h-1-w of segment 0, step 0 of segment 1)
      const int Np = sym_np(N, odd), h = sym_h(N, odd);
      if (seg == 1) return Np - 1 - (t + odd);
      if (odd && t >= h - 1 - w) ++t;
      if (t < h) {
        int r = w + t;
        r = r >= h ? r - h : r;
        return h + r;
      }
      return w + (t - h);
    }
    default:  // kSerial
      return causal ? w + t : t;
  }
}
DASH_HD int dq_rank(int sched, int causal, int N, int q, int kv, int odd) {
  if (sched != kShift) return kv;
  if (!causal) {
    int r = q - kv;
    return r < 0 ? r + N : r;
  }
  const int h = sym_h(N, odd);
  if (q < h) return q - kv;
  if (kv < h) {
    int r = q - h - kv;
    return r < 0 ? r + h : r;
  }
  return kv;
}

// ---------------------------------------------------------------------------------------
// Packed shift (kShiftFill).  The shift workers of all heads are laid out head-major and
// dealt round-robin to the P CTAs of the grid; every CTA runs its workers one per round.
// A head whose workers fall into two rounds runs as two lock-step phases (the workers of
// the earlier round first).  The visiting order of a worker is its head's shift order; the
// accumulation order of a dQ tile is the time order of its contributions: earlier phase
// first, then the step within the phase.  With W | P (no head split) this is exactly the
// shift order above.

// Worker (within its head) that owns KV block kv under the shift schedule.
DASH_HD int shift_worker_of(int causal, int N, int kv, int odd) {
  return (causal && kv >= sym_h(N, odd)) ? sym_np(N, odd) - 1 - kv : kv;
}
// Step, within its worker's program, at which the shift worker owning block kv visits
// query tile q; -1 if the tile is masked for that block (or kv is the padding block).
// For the causal mask this is the step of the padded (even) schedule, whose order is the
// accumulation order.
DASH_HD int shift_visit_step(int causal, int N, int kv, int q, int odd) {
  if (!causal) {
    const int t = q - kv;
    return t < 0 ? t + N : t;
  }
  if (q < kv) return -1;
  const int h = sym_h(N, odd), Np = sym_np(N, odd);
  if (kv < h) {  // worker c = kv, first segment
    if (q >= h) {
      const int t = q - h - kv;
      return t < 0 ? t + h : t;
    }
    return h + (q - kv);
  }
  const int c = Np - 1 - kv;  // worker c, second segment (block Np-1-c)
  return (Np - c) + (Np - 1 - q);
}
// The phase [lo, hi) of worker w of a head of W workers whose first worker has packed index
// s0: the workers of the head in w's round.
DASH_HD void packed_phase_at(long long s0, int W, int P, int w, int *lo, int *hi) {
  const long long round = (s0 + w) / P;
  long long a = round * P - s0, b = (round + 1) * P - s0;
  *lo = (int)(a < 0 ? 0 : a);
  *hi = (int)(b > W ? W : b);
}
// The same for head hd when every head has W workers (laid out head-major).
DASH_HD void packed_phase(int W, int P, int hd, int w, int *lo, int *hi) {
  packed_phase_at((long long)hd * W, W, P, w, lo, hi);
}
// Contributions to tile q from the workers [0, lo) of earlier rounds (all allowed blocks).
DASH_HD int packed_count_before(int causal, int N, int q, int lo, int odd) {
  if (!causal) return lo;
  const int a = lo < q + 1 ? lo : q + 1;             // blocks c <= q, c < lo
  const int b = lo - (sym_np(N, odd) - 1 - q);       // blocks Np-1-c <= q, c < lo
  return a + (b > 0 ? b : 0);
}
DASH_HD int span(int lo, int hi) { return hi > lo ? hi - lo : 0; }
DASH_HD int imax(int a, int b) { return a > b ? a : b; }
DASH_HD int imin(int a, int b) { return a < b ? a : b; }
// Contributions to tile q that precede (q, kv) in time and come from the workers c in
// [a, b) of kv's phase (all c < h), causal mask.  The Symmetric Shift visit steps of tile q
// by worker c are, per block,
//   block c, q >= h:      (q - h - c) mod h   = d - c (c <= d) or d - c + h (c > d), d = q - h
//   block c, q <  h:      h + q - c           (c <= q)
//   block Np-1-c:         (Np - c) + (Np-1-q) (c >= Np-1-q)
// and each is below tme on one contiguous range of c, so the count is a sum of range
// lengths.  Equal to the loop above (tested against the oracle's lock-step simulation).
DASH_HD int causal_count_in_phase(int N, int q, int kv, int a, int b, int odd) {
  const int tme = shift_visit_step(1, N, kv, q, odd);
  const int h = sym_h(N, odd), Np = sym_np(N, odd);
  const int bb = imin(b, h);
  int n;
  if (q >= h) {
    const int d = q - h;
    n = span(imax(imax(a, d - tme + 1), 0), imin(bb, d + 1)) +
        span(imax(imax(a, d + 1), d + h - tme + 1), bb);
  } else {
    n = span(imax(imax(a, h + q - tme + 1), 0), imin(bb, q + 1));
  }
  return n + span(imax(imax(a, Np - 1 - q), 2 * Np - q - tme), bb);
}
// Rank of block kv in dQ tile q of a head whose phase (kv's workers in kv's round) is
// [lo, hi): the earlier rounds' contributions, then the phase's earlier steps.  Full mask
// in closed form: the phase's Wp = hi - lo workers visit tile q at steps (q - c) mod N, so
// with base = (q - lo) mod N the worker c = lo + k comes at position base - k for k <= base
// and base + Wp - k otherwise, all workers past base being later than those up to it --
// unless base >= Wp - 1, when every worker of the phase comes in descending order.
DASH_HD int rank_in_phase(int causal, int N, int q, int kv, int lo, int hi, int odd) {
  if (!causal) {
    const int Wp = hi - lo, k = kv - lo;
    int base = q - lo;
    base = base < 0 ? base + N : base;
    const int in_phase = (base >= Wp - 1) ? Wp - 1 - k : (k <= base ? base - k : base + Wp - k);
    return lo + in_phase;
  }
  return packed_count_before(causal, N, q, lo, odd) + causal_count_in_phase(N, q, kv, lo, hi, odd);
}
// Rank of block kv in dQ tile q of head hd.
DASH_HD int packed_rank(int causal, int N, int P, int hd, int q, int kv, int odd) {
  const int W = causal ? sym_h(N, odd) : N;
  int lo, hi;
  packed_phase(W, P, hd, shift_worker_of(causal, N, kv, odd), &lo, &hi);
  return rank_in_phase(causal, N, q, kv, lo, hi, odd);
}

}  // namespace dash
