/*
 * dash_attn.h -- C ABI of libdash_attn.so: deterministic FlashAttention-style attention
 * backward (DASH tile schedules) for one NVIDIA GB300 GPU (sm_103a).
 *
 * The operation.  Softmax attention O = softmax(scale * Q K^T [masked]) V and its
 * gradient.  The DASH pages ("DASH: Deterministic Attention Scheduling for
 * High-throughput Reproducible LLM Training"; gist.science technical summary, section 1
 * "Problem statement") ask for a backward pass whose gradient accumulation -- dQ in
 * particular -- happens in a fixed order, so that repeated runs are bit-identical; the
 * order is given by one of the tile schedules of section 2.2 ("Scheduling strategies").
 *
 * Conventions shared by every entry point:
 *  - Layout BSHD, contiguous, bf16 (IEEE bfloat16 bit patterns):
 *      Q, O, dO, dQ : [B, S, H,   D]
 *      K, V, dK, dV : [B, S, Hkv, D]     Hkv = H / group
 *    LSE: [B, H, S] fp32, natural log of the softmax normaliser of each query row.
 *  - group = G >= 1 query heads share one K/V head; query head h uses kv head h / G
 *    (consecutive grouping).  G = 1 is plain multi-head attention.
 *  - mask: DASH_MASK_FULL, or DASH_MASK_CAUSAL = key j visible to query i iff j <= i
 *    (top-left aligned; queries and keys have the same length S).
 *  - scale <= 0 selects 1/sqrt(D).
 *  - Supported sizes: D in {64, 128}; S >= 1; B, H >= 1; H % group == 0.  The sequence
 *    is cut into N = ceil(S/128) tiles; when S is not a multiple of 128 the last tile is
 *    partial: its rows past S are read as zeros, their keys get zero attention weight, and
 *    nothing is written for them.  Anything else returns DASH_ERR_UNSUPPORTED (or DASH_ERR_INVALID for
 *    nonsensical values) synchronously and launches nothing.
 *  - Pointers: all tensor and workspace pointers are DEVICE pointers owned by the caller
 *    (for example allocated by PyTorch), 16-byte aligned (LSE: 4-byte aligned).  The library allocates no device
 *    memory, keeps no state between calls other than per-device kernel attributes, and is
 *    safe to call from several host threads on different streams.
 *  - Asynchrony: calls enqueue work on `stream` and return; argument errors are reported
 *    synchronously before anything is enqueued, launch failures as DASH_ERR_CUDA.
 *  - Device-side failures (a bounded wait that ran out, e.g. an ordering semaphore that
 *    was never released) do not hang or trap: the kernels record a code in the
 *    workspace's status word and return.  dash_attn_status() reads it.  One wait gives up
 *    after 2 s unless dash_attn_set_wait_limit() chose another limit.
 *  - Residency: the ordered backward schedules make workers wait on workers of other CTAs,
 *    so their tile kernel is launched cooperatively: the runtime starts it only once every
 *    CTA of its grid (at most one per SM) can be resident, also while other kernels share
 *    the GPU, and refuses the launch (DASH_ERR_CUDA) where that can never hold.
 */
#ifndef DASH_ATTN_H
#define DASH_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *dash_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum { DASH_MASK_FULL = 0, DASH_MASK_CAUSAL = 1 } dash_mask_t;

/* Tile schedules (gist.science technical summary, section 2.2).  N = ceil(S/128) tiles.
 *  DASH_SCHED_ATOMIC     -- non-deterministic reference: dQ partials are added with
 *                           unordered atomics (the "non-deterministic counterpart" of
 *                           section 1).  It visits tiles in the SHIFT order (cyclic /
 *                           symmetric), the fastest traversal, so that it is the speed reference for the
 *                           deterministic schedules.
 *  DASH_SCHED_SERIAL     -- deterministic baseline: the worker owning KV block j visits
 *                           query tiles in ascending order; every dQ tile adds the KV
 *                           blocks' partials in ascending kv order.
 *  DASH_SCHED_DESCENDING -- Descending Q-Tile Iteration (section 2.2 A): traversal
 *                           reversed (N-1 .. 0), accumulation order unchanged, so dQ is
 *                           bit-identical to SERIAL.
 *  DASH_SCHED_SHIFT      -- Shift Scheduling (section 2.2 B).  Full mask: the worker of
 *                           KV block j visits query tiles j, j+1, .., N-1, 0, .., j-1 and
 *                           tile q adds KV blocks q, q-1, .., q+1 (mod N).  Causal mask:
 *                           Symmetric Shift -- the worker c owns KV blocks c and N-1-c,
 *                           first the dense lower-left rectangle, then the folded
 *                           triangle.  Odd N (not covered by the pages): laid out as the
 *                           even schedule of N+1 tiles with the steps on the padding tile
 *                           dropped -- worker 0 owns block 0 alone, worker c >= 1 the
 *                           pair (c, N-c), (N+1)/2 workers of N steps each; the
 *                           accumulation order is the padded schedule's lock-step order.
 *  DASH_SCHED_SHIFT_FILL -- packed Shift Scheduling: the shift workers of all heads (W per
 *                           head: N, or ceil(N/2) for the causal mask) are dealt round-robin,
 *                           head-major, to every SM.  When W does not divide the SM count
 *                           a head's workers can fall into two consecutive rounds; such a
 *                           head runs as two lock-step phases, and each of its dQ tiles adds
 *                           the earlier phase's partials first, then the later phase's, each
 *                           phase in its shift (step) order.  Heads inside one round get
 *                           exactly the DASH_SCHED_SHIFT order.  Keeps every SM busy where
 *                           plain SHIFT leaves SMs waiting for a head's remaining workers,
 *                           and has no limit on N: a head with more workers than SMs runs
 *                           as several phases, each dQ tile adding the earlier phases'
 *                           partials first.  Deterministic for a given SM count (dash_sched_grid,
 *                           dash_sched_packed_rank give the order).
 *  DASH_SCHED_AUTO       -- the deterministic schedule that measured fastest on GB300 for
 *                           the mask, head dim, tile count N and group size G
 *                           (dash_sched_resolve names it): the pages leave the choice to the
 *                           user.  From whole-call timings (full mask H16 and causal H32 at
 *                           D = 128 and 64, S = 512 .. 16384, GQA 4:1) one schedule wins every
 *                           measured point: SHIFT_DUAL (against SHIFT_FILL: full mask +12 % at
 *                           N = 4, +19 % at N = 128; causal D = 128 +1-3 %, GQA +10 %; causal
 *                           D = 64 +2.5-4 %).  The mask, D, N and G remain arguments of
 *                           dash_sched_resolve for future entries.
 *  DASH_SCHED_SHIFT_DUAL -- packed Shift Scheduling (the SHIFT_FILL traversal, grid and ranks)
 *                           with each dQ tile accumulated in two strands: the partial of rank
 *                           r is added into strand r mod 2 as that strand's (r div 2)-th
 *                           addition, each strand in order under its own semaphore, and the
 *                           tile's dQ is bf16(scale * (strand 0 + strand 1)).  A fixed order,
 *                           deterministic for a given SM count like SHIFT_FILL, but not the
 *                           single chain of the pages: a strand's next contributor comes two
 *                           lock steps later instead of one, which lets the kernel spread its
 *                           reductions out and release each strand from a separate warp.
 */
typedef enum {
  DASH_SCHED_ATOMIC = 0,
  DASH_SCHED_SERIAL = 1,
  DASH_SCHED_DESCENDING = 2,
  DASH_SCHED_SHIFT = 3,
  DASH_SCHED_SHIFT_FILL = 4,
  DASH_SCHED_AUTO = 5,
  DASH_SCHED_SHIFT_DUAL = 6
} dash_sched_t;

typedef enum {
  DASH_OK = 0,
  DASH_ERR_INVALID = 1,     /* null pointer, non-positive size, misaligned pointer    */
  DASH_ERR_UNSUPPORTED = 2, /* valid but outside this library's support (D, N, GPU)  */
  DASH_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed            */
  DASH_ERR_TIMEOUT = 4,     /* a device-side bounded wait ran out (status word set)   */
  DASH_ERR_WORKSPACE = 5    /* workspace NULL or smaller than required                */
} dash_status_t;

/* Bytes of device workspace dash_attn_fwd needs (its status word); 0 on bad sizes. */
size_t dash_attn_fwd_workspace_bytes(int B, int S, int H, int D);

/* Forward pass: O = softmax(scale Q K^T + mask) V and LSE = log of each row's softmax
 * normaliser (natural log, fp32).  Provides the O and LSE the backward consumes; the
 * DASH pages take them as given (the method concerns the backward pass only).
 *   q [B,S,H,D] bf16, k/v [B,S,H/group,D] bf16        (inputs, read only)
 *   o [B,S,H,D] bf16, lse [B,H,S] fp32                  (outputs, fully overwritten)
 *   workspace: >= dash_attn_fwd_workspace_bytes(...) bytes of device memory. */
dash_status_t dash_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                            int B, int S, int H, int group, int D, float scale,
                            dash_mask_t mask, void *workspace, size_t workspace_bytes,
                            dash_stream_t stream);

/* Bytes of device workspace dash_attn_bwd needs, for any schedule: a status block (256 B),
 * the dQ ordering semaphores (room for two per dQ tile, B*H*(Sp/128)*8), two fp32 row
 * vectors (B*H*Sp*4 each) and the fp32 dQ accumulator (room for two strands, B*H*Sp*D*8),
 * Sp = 128*ceil(S/128), in this order, each part 256-byte aligned; 0 on bad sizes. */
size_t dash_attn_bwd_workspace_bytes(int B, int S, int H, int D);

/* Backward pass (the DASH hot path): given Q, K, V, O, dO and LSE, writes dQ, dK, dV.
 *   Steps, all on `stream`: clear the status word and the semaphores (and, unless the
 *   schedule is DASH_SCHED_SHIFT_DUAL, the accumulator); D_i = rowsum(dO_i * O_i); the
 *   tile kernel -- per KV block, dK/dV accumulate in tensor memory on one SM while every
 *   visited query tile's dQ partial is added to an fp32 accumulator in global memory in
 *   the order the schedule fixes, enforced by one ordering semaphore per dQ tile
 *   (section 2.1: one KV tile's operations stay on one SM; section 1: fixed dQ
 *   accumulation order; under DASH_SCHED_SHIFT_DUAL the first partial of each strand is
 *   stored rather than added); finally dQ = bf16(scale * accumulator).
 *   For group > 1, dK/dV of a KV head sum the group's query heads in ascending order.
 *   Deterministic schedules give bit-identical dQ/dK/dV on every run, for any grid size
 *   and under concurrent load; DASH_SCHED_ATOMIC does not.
 *   q, o, dout [B,S,H,D]; k, v [B,S,H/group,D]; lse [B,H,S]    (inputs, read only)
 *   dq [B,S,H,D]; dk, dv [B,S,H/group,D]                       (outputs, overwritten)
 *   workspace: >= dash_attn_bwd_workspace_bytes(B,S,H,D) bytes, caller-owned, contents
 *   need not be initialised; one workspace must not be used by two calls that may run
 *   concurrently.  DASH_SCHED_SHIFT requires a head's workers (N; ceil(N/2) for the
 *   causal mask) to fit on the SMs at once: they wait on one another. */
dash_status_t dash_attn_bwd(const void *q, const void *k, const void *v, const void *o,
                            const void *dout, const float *lse, void *dq, void *dk, void *dv,
                            int B, int S, int H, int group, int D, float scale,
                            dash_mask_t mask, dash_sched_t sched, void *workspace,
                            size_t workspace_bytes, dash_stream_t stream);

/* The same backward in separately launchable stages, for callers that time or overlap
 * them: DASH_BWD_PROLOGUE clears the workspace's status word and semaphores (and the
 * accumulator, except under DASH_SCHED_SHIFT_DUAL) and computes the row vectors
 * (rowsum(dO*O), LSE*log2 e); DASH_BWD_TILES runs the tile kernel (the five contractions
 * and the ordered dQ reduction, dK/dV written); DASH_BWD_EPILOGUE converts the dQ
 * accumulator to bf16.  Arguments as dash_attn_bwd; stages given in separate calls must
 * be issued in this order with identical arguments and workspace.  dash_attn_bwd is
 * dash_attn_bwd_stages(..., DASH_BWD_ALL). */
typedef enum {
  DASH_BWD_PROLOGUE = 1,
  DASH_BWD_TILES = 2,
  DASH_BWD_EPILOGUE = 4,
  DASH_BWD_ALL = 7
} dash_bwd_stage_t;
dash_status_t dash_attn_bwd_stages(const void *q, const void *k, const void *v, const void *o,
                                   const void *dout, const float *lse, void *dq, void *dk,
                                   void *dv, int B, int S, int H, int group, int D, float scale,
                                   dash_mask_t mask, dash_sched_t sched, void *workspace,
                                   size_t workspace_bytes, unsigned stages,
                                   dash_stream_t stream);

/* Synchronises `stream` and reads the status word of the last call that used
 * `workspace` (fwd or bwd workspace).  DASH_OK, or DASH_ERR_TIMEOUT when a bounded wait
 * ran out on the device (the outputs of that call are then undefined). */
dash_status_t dash_attn_status(void *workspace, dash_stream_t stream);
/* The same, under the backward's name. */
dash_status_t dash_attn_bwd_status(void *workspace, dash_stream_t stream);

/* Limit of one device-side bounded wait (an mbarrier phase, an ordering semaphore) for the
 * calls made after this one, process-wide: 1e-3 <= seconds <= 3600, default 2.  A wait
 * that runs out sets the status word (DASH_ERR_TIMEOUT) and the kernel returns.  Raise it
 * where the GPU is time-sliced with other processes for long periods. */
dash_status_t dash_attn_set_wait_limit(double seconds);
double dash_attn_wait_limit(void);

/* The backward of dash_attn_bwd that also records the accumulation order it executed: for
 * every (b, h, q, kv) pair the schedule visits, order_log[((b*H + h)*N + q)*N + kv] = the
 * rank at which KV block kv's partial was added into dQ tile q (the semaphore value the
 * addition waited for).  order_log: device int32
 * [B, H, N, N], N = ceil(S/128); entries of masked pairs are left as they were.  Ordered
 * schedules only (DASH_SCHED_ATOMIC records nothing).  For tests and audits. */
dash_status_t dash_attn_bwd_order_log(const void *q, const void *k, const void *v,
                                      const void *o, const void *dout, const float *lse,
                                      void *dq, void *dk, void *dv, int B, int S, int H,
                                      int group, int D, float scale, dash_mask_t mask,
                                      dash_sched_t sched, void *workspace,
                                      size_t workspace_bytes, int *order_log,
                                      dash_stream_t stream);

/* Allocation-free backward.  No counterpart on the DASH pages: this is a calling
 * convenience of this library.  It is for callers that cannot provide a workspace -- for
 * example a plugin inside an application whose memory pool owns the whole GPU and offers
 * plugins no allocator, or code where a cudaMalloc would implicitly synchronise the device.
 * Same arguments and results as dash_attn_bwd, without the workspace: the workspace is a
 * fixed device array of DASH_NOALLOC_SCRATCH_BYTES inside the library, present on every
 * GPU that loads the library until the process exits.  The call itself allocates nothing
 * (no cudaMalloc/cudaFree, no allocating library routine).
 *   - Limit: sizes whose dash_attn_bwd_workspace_bytes(B,S,H,D) exceeds
 *     DASH_NOALLOC_SCRATCH_BYTES are rejected with DASH_ERR_WORKSPACE before anything runs
 *     (64 MiB holds about B*H*S*(2D+2)*4 bytes: up to B*H*S = 64896 rows at D = 128).
 *   - The first call on a device (that device current) looks up the array's device address
 *     with cudaGetSymbolAddress; make that first call before any stream capture.
 *   - All calls on a device share the array: calls that may overlap on the GPU (e.g. on
 *     unordered streams) race and corrupt each other's results; order them on one stream.
 *     Each call re-zeroes the parts that must start at zero.
 *   - Device-side status (a bounded wait that ran out) is written into the array; read it
 *     with dash_attn_noalloc_status. */
#define DASH_NOALLOC_SCRATCH_BYTES (64u << 20)
dash_status_t dash_attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                                    const void *dout, const float *lse, void *dq, void *dk,
                                    void *dv, int B, int S, int H, int group, int D, float scale,
                                    dash_mask_t mask, dash_sched_t sched, dash_stream_t stream);
/* Synchronises `stream` and reads the status word of the last dash_attn_bwd_noalloc call on
 * the current device, as dash_attn_status does for a workspace: DASH_OK, or
 * DASH_ERR_TIMEOUT when a bounded wait ran out (that call's outputs are undefined). */
dash_status_t dash_attn_noalloc_status(dash_stream_t stream);

/* Variable-length batches.  `batch` sequences packed along the token axis:
 *   Q, O, dO, dQ : [T, H, D]        K, V, dK, dV : [T, Hkv, D]      T = cu_seqlens[batch]
 *   LSE          : the sequences' [H, S_b] blocks one after another (sequence b's block
 *                  starts at float offset H * cu_seqlens[b]); 4-byte aligned
 *   cu_seqlens   : HOST array of batch+1 ints, cu_seqlens[0] = 0, non-decreasing; sequence
 *                  b is tokens [cu_seqlens[b], cu_seqlens[b+1]) (S_b may be 0 or any length).
 * Each sequence is an independent attention problem (the mask applies within it).  The
 * forward runs each sequence as the B = 1 call on its slices.  The backward:
 *   - DASH_SCHED_SHIFT_FILL, DASH_SCHED_SHIFT_DUAL and DASH_SCHED_ATOMIC (and DASH_SCHED_AUTO,
 *     resolved once with the longest sequence's tile count, always to one of the first two)
 *     pack the workers of every sequence's heads onto the persistent grid in ONE tile-kernel
 *     launch per group of at most 1024 non-empty sequences: sequence b has its own
 *     N_b = ceil(S_b/128) tiles and, for causal masks, its own Symmetric Shift parity; the
 *     workers of all sequences are laid out sequence-major, then kv-head-major (the order
 *     of the uniform batch's heads) and dealt round-robin to the CTAs, so each dQ tile's
 *     accumulation order is the packed shift order at its sequence's position in that
 *     layout -- fixed by cu_seqlens, H, group, the mask and the SM count, hence bit-identical
 *     from run to run, but not in general the order of the B = 1 call on the sequence alone
 *     (equal where every head's workers fall in one round of the grid in both layouts);
 *   - DASH_SCHED_SERIAL, DASH_SCHED_DESCENDING, DASH_SCHED_SHIFT run each sequence as the
 *     B = 1 call on its slices, one after another on `stream`, with the results of that call.
 * The workspace is shared by the groups or sequences: size it with
 * dash_attn_bwd_varlen_workspace_bytes (the largest of the longest sequence's need and a
 * packed group's need: per-tile arrays for every tile of the group plus a 20.5 KB sequence
 * table).  The backward checks every sequence before it enqueues anything; the device
 * status word collects the flags of all groups or sequences.  Returns as the B = 1 calls
 * do, plus DASH_ERR_UNSUPPORTED where a packed group exceeds 2^30 tiles, tokens or workers. */
size_t dash_attn_bwd_varlen_workspace_bytes(const int *cu_seqlens, int batch, int H, int D);
dash_status_t dash_attn_fwd_varlen(const void *q, const void *k, const void *v, void *o,
                                   float *lse, const int *cu_seqlens, int batch, int H,
                                   int group, int D, float scale, dash_mask_t mask,
                                   void *workspace, size_t workspace_bytes,
                                   dash_stream_t stream);
dash_status_t dash_attn_bwd_varlen(const void *q, const void *k, const void *v, const void *o,
                                   const void *dout, const float *lse, void *dq, void *dk,
                                   void *dv, const int *cu_seqlens, int batch, int H, int group,
                                   int D, float scale, dash_mask_t mask, dash_sched_t sched,
                                   void *workspace, size_t workspace_bytes,
                                   dash_stream_t stream);
/* dash_attn_bwd_varlen with the audit record of dash_attn_bwd_order_log: order_log (device,
 * int32, 4-byte aligned, caller-owned) is [tiles][Nmax], Nmax = the longest sequence's tile
 * count and the tiles those of the non-empty sequences in order, each [H, N_b]: entry
 * [tile (b, h, q)][kv] receives the rank at which KV block kv's partial was added into dQ tile
 * q of sequence b (ordered schedules; entries of pairs not visited are left unchanged).
 * DASH_ERR_INVALID when order_log is NULL. */
dash_status_t dash_attn_bwd_varlen_order_log(const void *q, const void *k, const void *v,
                                             const void *o, const void *dout, const float *lse,
                                             void *dq, void *dk, void *dv, const int *cu_seqlens,
                                             int batch, int H, int group, int D, float scale,
                                             dash_mask_t mask, dash_sched_t sched,
                                             void *workspace, size_t workspace_bytes,
                                             int *order_log, dash_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char *dash_status_string(dash_status_t status);

/* Host-only view of the tile schedules the backward kernel executes (no GPU needed).
 * A head has N = ceil(S/128) KV blocks and query tiles.  Workers: the per-head units of work
 * (one KV block, or the pair c, N-1-c for causal DASH_SCHED_SHIFT); each worker runs
 * one or two segments (one KV block each) of steps; step t of a segment visits query
 * tile *q with KV block *kv, and its dQ partial is the rank-th addition into tile q.
 * Return -1 on unsupported arguments. */
int dash_sched_workers(int sched, int mask, int N);
/* The schedule dash_attn_bwd runs for `sched` (DASH_SCHED_AUTO resolved, every other value
 * returned unchanged) with `mask`, head dim D, N = ceil(S/128) tiles and `group` query heads
 * per KV head; -1 on bad arguments.  The table queries below resolve AUTO to SHIFT_FILL,
 * whose traversal SHIFT_DUAL shares. */
int dash_sched_resolve(int sched, int mask, int D, int N, int group);
/* Number of CTAs dash_attn_bwd launches for its tile kernel on a GPU with `sms` SMs, for
 * `heads` = B * H/group (batch, kv head) pairs; -1 where dash_attn_bwd would reject the
 * schedule arguments (e.g. DASH_SCHED_SHIFT with more workers per head than SMs). */
int dash_sched_grid(int sched, int mask, int N, int heads, int sms);
/* DASH_SCHED_SHIFT_FILL: position of KV block kv's partial in dQ tile q of head `head`
 * (0 <= head < heads) when the tile kernel runs on `grid` CTAs (dash_sched_grid); -1 on
 * bad arguments or a masked (q, kv). */
int dash_sched_packed_rank(int mask, int N, int heads, int grid, int head, int q, int kv);
int dash_sched_segments(int sched, int mask, int N, int worker);
int dash_sched_steps(int sched, int mask, int N, int worker, int segment);
int dash_sched_step(int sched, int mask, int N, int worker, int segment, int step, int *kv,
                    int *q, int *rank);

#ifdef __cplusplus
}
#endif
#endif /* DASH_ATTN_H */
