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
//  ATOMIC: no order; it visits tiles in the shift order (conflict-free and, for the causal
//    mask, balanced), the most favourable traversal, so that the deterministic schedules
//    are compared against the fastest non-deterministic backward; odd-N causal falls back
//    to the SERIAL traversal.
#pragma once

#if defined(__CUDACC__)
#define DASH_HD __host__ __device__ __forceinline__
#else
#define DASH_HD inline
#endif

namespace dash {

// kShiftFill is the shift schedule on as many SMs as hold whole heads, plus DESCENDING on
// the remaining SMs for a share of the heads (the host decides the split).
enum Sched : int { kAtomic = 0, kSerial = 1, kDescending = 2, kShift = 3, kShiftFill = 4 };

// Which visiting order a schedule uses (ATOMIC borrows the shift order when it exists; the
// fill mode's shift heads use the shift order).
DASH_HD int traversal(int sched, int causal, int N) {
  if (sched == kShiftFill) return kShift;
  if (sched != kAtomic) return sched;
  return (!causal || (N % 2) == 0) ? kShift : kSerial;
}

DASH_HD bool sym_shift(int sched, int causal) { return sched == kShift && causal; }

DASH_HD int sched_workers(int sched, int causal, int N) {
  return sym_shift(sched, causal) ? N / 2 : N;
}
DASH_HD int sched_segments(int sched, int causal) { return sym_shift(sched, causal) ? 2 : 1; }
DASH_HD int seg_kv(int sched, int causal, int N, int w, int seg) {
  return (sym_shift(sched, causal) && seg == 1) ? N - 1 - w : w;
}
DASH_HD int seg_steps(int sched, int causal, int N, int w, int seg) {
  if (!causal) return N;
  if (sched == kShift) return seg == 0 ? N - w : w + 1;
  return N - w;
}
DASH_HD int step_q(int sched, int causal, int N, int w, int seg, int t) {
  switch (sched) {
    case kDescending:
      return N - 1 - t;
    case kShift: {
      if (!causal) {
        int q = w + t;
        return q >= N ? q - N : q;
      }
      const int h = N >> 1;
      if (seg == 1) return N - 1 - t;
      if (t < h) {
        int r = w + t;
        r = r >= h ? r - h : r;
        return h + r;
      }
      return w + (t - h);
    }
    default:  // kAtomic, kSerial
      return causal ? w + t : t;
  }
}
DASH_HD int dq_rank(int sched, int causal, int N, int q, int kv) {
  if (sched != kShift) return kv;
  if (!causal) {
    int r = q - kv;
    return r < 0 ? r + N : r;
  }
  const int h = N >> 1;
  if (q < h) return q - kv;
  if (kv < h) {
    int r = q - h - kv;
    return r < 0 ? r + h : r;
  }
  return kv;
}

}  // namespace dash
