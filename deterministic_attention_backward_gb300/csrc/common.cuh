// common.cuh -- constants, parameter blocks and the internal launch interface shared by the
// translation units of libdash_attn.so.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dash {

constexpr int kTile = 128;                // rows of a query tile and of a KV block
constexpr int kBoxCols = 64;              // bf16 columns of one 128-byte-swizzled box
constexpr int kBoxBytes = kTile * 128;    // one [128 x 64] bf16 box = 16 KB
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// error codes written into a workspace status word (bit flags)
enum : uint32_t {
  kErrMbarTimeout = 1u,  // an mbarrier phase never completed
  kErrSemTimeout = 2u,   // a dQ ordering semaphore never reached the expected rank
  kErrSmemAlign = 4u,    // dynamic shared memory not 1024-byte aligned
  kErrAborted = 8u,      // the CTA stopped because another CTA reported an error
};

// Backward kernel parameters (besides the TMA descriptors of Q, K, V, dO).
struct BwdParams {
  const float *lse2;  // [B,H,N*128]  LSE * log2(e)
  const float *dvec;  // [B,H,N*128]  rowsum(dO * O)
  float *dqacc;       // fp32 dQ accumulator, tile-native [B,H,N][K][D/4][128][4], K strands
                      // (two strands: a strand's first partial is stored, no clearing needed)
  int *sem;           // [B,H,N][K] ordering semaphores (partials added so far, per strand)
  uint32_t *status;   // status word (error bit flags)
  __nv_bfloat16 *dk;  // [B,S,Hkv,D]
  __nv_bfloat16 *dv;  // [B,S,Hkv,D]
  int *order_log;     // optional [tiles][log_stride]: rank of (q, kv) in tile q's order, as
                      // executed, at [tile (b,h,q)][kv] ([B,H,N,N] for a uniform batch)
  int log_stride;
  // packed variable-length batch (mode bit 3): per sequence b, seqs[b] = {S_b, first token,
  // index of its first tile in the per-tile arrays, N_b}; seq_wprefix[b] = packed index of
  // its first worker (batch + 1 entries); units = all sequences' workers
  const int4 *seqs;
  const int *seq_wprefix;
  int batch, units;
  int B, S, H, Hkv, G, N;
  int causal;
  int heads;    // B * Hkv (b, kv head) pairs
  int sched;    // visiting order of the workers (sched.cuh)
  int workers;  // workers per head
  int packed;   // dQ ranks of the packed shift (workers dealt round-robin over the grid)
  unsigned long long wait_ns;  // limit of one bounded wait
  float scale_log2; // scale * log2(e)
  float scale;
  unsigned long long *trace;  // development trace build only: [64 steps][32 events] clock64
  int trace_cta;              // development trace build only: the CTA whose events are kept
};

// Development trace build (compiled with -DDASH_TRACE_BUILD into a separate library): the
// roles of one CTA record clock64() at fixed events of their first 64 steps, indexed by the
// role's own step counter `it`.  In the product build the macro expands to nothing.
#ifdef DASH_TRACE_BUILD
#define DASH_TRACE(p, slot)                                              \
  do {                                                                   \
    if ((p).trace && (int)blockIdx.x == (p).trace_cta && it < 64u)       \
      (p).trace[it * 32u + (slot)] = (unsigned long long)clock64();      \
  } while (0)
#else
#define DASH_TRACE(p, slot) \
  do {                      \
  } while (0)
#endif

struct FwdParams {
  __nv_bfloat16 *o;  // [B,S,H,D]
  float *lse;        // [B,H,S]
  uint32_t *status;
  unsigned long long wait_ns;  // limit of one bounded wait
  int B, S, H, Hkv, G, N;
  int causal;
  float scale_log2;
};

size_t fwd_smem_bytes(int D);

// mode: bits 0-1: 0 = full mask; 1 = causal mask; 2 = causal mask under Symmetric Shift
// (shift traversal) with an odd tile count, i.e. the padded schedule; bit 2 (value 4): two
// accumulation strands (ordered); bit 3 (value 8): a packed variable-length batch (3-D tensor
// maps over the tokens, per-sequence lengths, the packed shift traversal, odd tile counts
// read per sequence).  The tile kernel is compiled once per mode.
// The ordered (deterministic) launch is cooperative: the runtime starts it only with every
// CTA of the grid resident at once, so a worker never waits on a CTA that cannot start.
cudaError_t launch_bwd(int D, bool deterministic, int mode, const CUtensorMap &tq,
                       const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tdo,
                       const BwdParams &p, int grid, cudaStream_t stream);
// The packed variable-length launch (mode bit 3 set, the mask and the strands as given).
cudaError_t launch_bwd_varlen(int D, bool deterministic, bool causal, bool dual,
                              const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                              const CUtensorMap &tdo, const BwdParams &p, int grid,
                              cudaStream_t stream);
cudaError_t launch_fwd(int D, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const FwdParams &p, cudaStream_t stream);
cudaError_t launch_preprocess(const __nv_bfloat16 *o, const __nv_bfloat16 *dout,
                              const float *lse, float *dvec, float *lse2, int B, int S, int H,
                              int D, uint32_t *status, unsigned long long wait_ns,
                              cudaStream_t stream);
// dQ = bf16(scale * (strand 0 + ... + strand K-1)) for every row < S.  A strand s that
// received no partial (a tile with s or fewer: query tile 0 of a causal mask, or N = 1) is
// not read: the two-strand schedule stores each strand's first partial instead of clearing
// the accumulator.
cudaError_t launch_dq_convert(const float *dqacc, __nv_bfloat16 *dq, float scale, int B,
                              int S, int H, int D, int strands, int causal, uint32_t *status,
                              unsigned long long wait_ns, cudaStream_t stream);

// Packed variable-length batches: the sequence table (at most kMaxVarlenSeqs sequences) is
// written into the workspace by a one-block kernel that receives it as its parameter.
constexpr int kMaxVarlenSeqs = 1024;
struct VarlenTable {
  int4 seqs[kMaxVarlenSeqs];           // {S_b, first token, first tile, N_b}
  int wprefix[kMaxVarlenSeqs + 1];     // packed index of sequence b's first worker
  int batch;
};
cudaError_t launch_varlen_setup(const VarlenTable &t, int4 *seqs, int *wprefix,
                                cudaStream_t stream);
// preprocess and convert over a packed batch of T tokens (sequence table in device memory)
cudaError_t launch_preprocess_varlen(const __nv_bfloat16 *o, const __nv_bfloat16 *dout,
                                     const float *lse, float *dvec, float *lse2, const int4 *seqs,
                                     int batch, int T, int H, int D, uint32_t *status,
                                     unsigned long long wait_ns, cudaStream_t stream);
cudaError_t launch_dq_convert_varlen(const float *dqacc, __nv_bfloat16 *dq, float scale,
                                     const int4 *seqs, int batch, int ntiles, int H, int D,
                                     int strands, int causal, uint32_t *status,
                                     unsigned long long wait_ns, cudaStream_t stream);
// Strands a dQ tile's accumulation is split into (DASH_SCHED_SHIFT_DUAL: 2), at most:
constexpr int kMaxStrands = 2;

}  // namespace dash
