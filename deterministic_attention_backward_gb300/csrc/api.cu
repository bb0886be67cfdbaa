// api.cu -- the extern "C" boundary of libdash_attn.so (declared in include/dash_attn.h):
// argument validation, workspace carving, TMA descriptor construction and the launch
// sequence of the forward and backward passes.  No device memory is allocated here.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "dash_attn.h"
#include "sched.cuh"

namespace {

using dash::kTile;

// ------------------------------------------------------------------ driver entry point
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// [B, S, Hx, D] bf16 viewed as a 4-D tensor (D, Hx, S, B); box = 64 columns x 1 head x 128
// rows x 1 batch, 128-byte swizzle: one box lands in shared memory as 128 rows of 128 bytes.
// Rows of a tile past S (S not a multiple of 128) are outside the tensor and read as zeros.
bool make_bshd_map(CUtensorMap *m, const void *base, int B, int S, int Hx, int D) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hx, (cuuint64_t)S, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)Hx * D * 2,
                                 (cuuint64_t)S * Hx * D * 2};
  const cuuint32_t box[4] = {(cuuint32_t)dash::kBoxCols, 1, (cuuint32_t)kTile, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [T, Hx, D] bf16 packed tokens viewed as a 3-D tensor (D, Hx, T), same box and swizzle as
// make_bshd_map.  Rows past T read as zeros; a sequence's rows past its end are the next
// sequence's tokens, which the tile kernel masks.
bool make_thd_map(CUtensorMap *m, const void *base, int T, int Hx, int D) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hx, (cuuint64_t)T};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hx * D * 2};
  const cuuint32_t box[3] = {(cuuint32_t)dash::kBoxCols, 1, (cuuint32_t)kTile};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ device properties
struct DevInfo {
  int sms = 0, major = 0, minor = 0;
};
std::mutex g_dev_mu;
DevInfo g_dev[64];

dash_status_t device_info(DevInfo *out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DASH_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo &d = g_dev[dev];
  if (d.sms == 0) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      d.sms = 0;
      return DASH_ERR_CUDA;
    }
  }
  *out = d;
  // kernels are built for sm_103a only
  return (d.major == 10 && d.minor == 3) ? DASH_OK : DASH_ERR_UNSUPPORTED;
}

// ------------------------------------------------------------------ validation / workspace
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
int tiles(int S) { return (S + kTile - 1) / kTile; }  // N: a last, partial tile counts
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

dash_status_t check_sizes(int B, int S, int H, int group, int D) {
  if (B <= 0 || S <= 0 || H <= 0 || group <= 0 || D <= 0) return DASH_ERR_INVALID;
  if (H % group) return DASH_ERR_INVALID;
  if (D != 64 && D != 128) return DASH_ERR_UNSUPPORTED;
  // index arithmetic inside the kernels is 32-bit for row numbers
  if ((long long)B * tiles(S) * kTile >= (1LL << 31) / 2 ||
      (long long)B * H * tiles(S) >= (1LL << 30))
    return DASH_ERR_UNSUPPORTED;
  return DASH_OK;
}

constexpr size_t kStatusBytes = 256;

struct BwdWorkspace {
  uint32_t *status;
  float *dqacc, *lse2, *dvec;
  int *sem;
  size_t dqacc_bytes, sem_bytes, total;
};

// [status 256 B][semaphores][lse2][Dvec][dQ accumulator], each part 256-byte aligned; the
// status block and the semaphores are contiguous so that one clear covers both.  Row arrays
// are per tile: S padded up to N*128 rows per (b, h).  Semaphores and accumulator have room
// for kMaxStrands strands per dQ tile (a call with K strands uses [B,H,N][K]...).  `ntiles`
// dQ tiles in all (B*H*N for a uniform batch).
BwdWorkspace carve_tiles(void *ws, size_t ntiles, int D) {
  BwdWorkspace w{};
  const size_t rows = ntiles * kTile;
  char *base = static_cast<char *>(ws);
  size_t off = 0;
  w.status = reinterpret_cast<uint32_t *>(base + off);
  off += kStatusBytes;
  w.sem = reinterpret_cast<int *>(base + off);
  w.sem_bytes = ntiles * 4 * dash::kMaxStrands;
  off = align256(off + w.sem_bytes);
  w.lse2 = reinterpret_cast<float *>(base + off);
  off = align256(off + rows * 4);
  w.dvec = reinterpret_cast<float *>(base + off);
  off = align256(off + rows * 4);
  w.dqacc = reinterpret_cast<float *>(base + off);
  w.dqacc_bytes = rows * D * 4;  // one strand
  off = align256(off + w.dqacc_bytes * dash::kMaxStrands);
  w.total = off;
  return w;
}
BwdWorkspace carve_bwd(void *ws, int B, int S, int H, int D) {
  return carve_tiles(ws, (size_t)B * H * tiles(S), D);
}

// Limit of one bounded wait inside the kernels (dash_attn_set_wait_limit).
std::atomic<unsigned long long> g_wait_ns{2000000000ull};

#ifdef DASH_TRACE_BUILD
unsigned long long *g_trace = nullptr;  // development trace build only
int g_trace_cta = 0;
#endif

// How the backward tile kernel's grid is used: the workers of all heads, head-major, dealt
// round-robin to `grid` CTAs.
struct LaunchPlan {
  int sched, workers, grid, packed, strands;
};

bool sched_known(int sched) {
  return (sched >= DASH_SCHED_ATOMIC && sched <= DASH_SCHED_AUTO) || sched == DASH_SCHED_SHIFT_DUAL;
}

// DASH_SCHED_AUTO: the deterministic schedule measured fastest on GB300 for the mask, head
// dim D, tile count N and group size G (the table and its measurements are in the header).
// D = 0 asks for the traversal only (the schedule queries): SHIFT_FILL, whose tables
// DASH_SCHED_SHIFT_DUAL shares.
int resolve_sched(int sched, int mask, int D, int N, int G) {
  if (sched != DASH_SCHED_AUTO) return sched;
  (void)mask;
  (void)D;
  (void)N;
  (void)G;
  return DASH_SCHED_SHIFT_DUAL;
}

// False when plain SHIFT cannot have every worker of a head resident at once.  The packed
// schedules have no such limit: their ranks follow the time order of the rounds, so a head
// wider than the grid simply spans more rounds.
bool make_plan(int sched, int causal, int N, int heads, int sms, LaunchPlan *pl) {
  pl->sched = dash::traversal(sched, causal, N);
  pl->workers = dash::sched_workers(pl->sched, causal, N, N & 1);
  const long long total = (long long)heads * pl->workers;
  pl->grid = (int)(total < sms ? total : sms);
  pl->packed = sched == DASH_SCHED_SHIFT_FILL || sched == DASH_SCHED_SHIFT_DUAL;
  pl->strands = sched == DASH_SCHED_SHIFT_DUAL ? 2 : 1;
  return !(sched == DASH_SCHED_SHIFT && pl->workers > sms);
}

float resolve_scale(float scale, int D) {
  return scale > 0.f ? scale : 1.0f / std::sqrt((float)D);
}

// The tile kernel's parameters that uniform and packed batches fill alike: workspace
// arrays, outputs, the order log, heads, mask, scale, wait limit (and the development
// trace buffer).  The caller adds the batch geometry and the schedule.
dash::BwdParams base_params(const BwdWorkspace &w, void *dk, void *dv, int *order_log,
                            int log_stride, int H, int group, int causal, float sc) {
  dash::BwdParams p{};
  p.lse2 = w.lse2;
  p.dvec = w.dvec;
  p.dqacc = w.dqacc;
  p.sem = w.sem;
  p.status = w.status;
  p.dk = static_cast<__nv_bfloat16 *>(dk);
  p.dv = static_cast<__nv_bfloat16 *>(dv);
  p.order_log = order_log;
  p.log_stride = log_stride;
  p.H = H;
  p.Hkv = H / group;
  p.G = group;
  p.causal = causal;
  p.wait_ns = g_wait_ns.load();
  p.scale_log2 = sc * dash::kLog2e;
  p.scale = sc;
#ifdef DASH_TRACE_BUILD
  p.trace = g_trace;
  p.trace_cta = g_trace_cta;
#endif
  return p;
}

}  // namespace

extern "C" {

size_t dash_attn_fwd_workspace_bytes(int B, int S, int H, int D) {
  if (check_sizes(B, S, H, 1, D) != DASH_OK) return 0;
  return kStatusBytes;
}

size_t dash_attn_bwd_workspace_bytes(int B, int S, int H, int D) {
  if (check_sizes(B, S, H, 1, D) != DASH_OK) return 0;
  return carve_bwd(nullptr, B, S, H, D).total;
}

// keep_status: leave the workspace status word as it is (a later sequence of a varlen
// batch adds its error flags to the earlier ones' instead of clearing them).
static dash_status_t fwd_impl(const void *q, const void *k, const void *v, void *o, float *lse,
                              int B, int S, int H, int group, int D, float scale,
                              dash_mask_t mask, void *workspace, size_t workspace_bytes,
                              dash_stream_t stream, bool keep_status) {
  dash_status_t st = check_sizes(B, S, H, group, D);
  if (st != DASH_OK) return st;
  if (mask != DASH_MASK_FULL && mask != DASH_MASK_CAUSAL) return DASH_ERR_INVALID;
  if (!q || !k || !v || !o || !lse) return DASH_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse))
    return DASH_ERR_INVALID;
  if (!workspace || workspace_bytes < kStatusBytes || !aligned16(workspace))
    return DASH_ERR_WORKSPACE;
  DevInfo dev;
  if ((st = device_info(&dev)) != DASH_OK) return st;
  const int Hkv = H / group;
  CUtensorMap tq, tk, tv;
  if (!make_bshd_map(&tq, q, B, S, H, D) || !make_bshd_map(&tk, k, B, S, Hkv, D) ||
      !make_bshd_map(&tv, v, B, S, Hkv, D))
    return DASH_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!keep_status && cudaMemsetAsync(workspace, 0, kStatusBytes, s) != cudaSuccess)
    return DASH_ERR_CUDA;
  dash::FwdParams p{};
  p.o = static_cast<__nv_bfloat16 *>(o);
  p.lse = lse;
  p.status = static_cast<uint32_t *>(workspace);
  p.B = B;
  p.S = S;
  p.H = H;
  p.Hkv = Hkv;
  p.G = group;
  p.N = tiles(S);
  p.causal = mask == DASH_MASK_CAUSAL;
  p.scale_log2 = resolve_scale(scale, D) * dash::kLog2e;
  p.wait_ns = g_wait_ns.load();
  return dash::launch_fwd(D, tq, tk, tv, p, s) == cudaSuccess ? DASH_OK : DASH_ERR_CUDA;
}

dash_status_t dash_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                            int B, int S, int H, int group, int D, float scale,
                            dash_mask_t mask, void *workspace, size_t workspace_bytes,
                            dash_stream_t stream) {
  return fwd_impl(q, k, v, o, lse, B, S, H, group, D, scale, mask, workspace, workspace_bytes,
                  stream, false);
}

static dash_status_t bwd_impl(const void *q, const void *k, const void *v, const void *o,
                              const void *dout, const float *lse, void *dq, void *dk, void *dv,
                              int B, int S, int H, int group, int D, float scale,
                              dash_mask_t mask, dash_sched_t sched, void *workspace,
                              size_t workspace_bytes, unsigned stages, dash_stream_t stream,
                              bool keep_status, int *order_log, int log_stride = 0) {
  if (stages == 0 || (stages & ~unsigned(DASH_BWD_ALL))) return DASH_ERR_INVALID;
  dash_status_t st = check_sizes(B, S, H, group, D);
  if (st != DASH_OK) return st;
  if (mask != DASH_MASK_FULL && mask != DASH_MASK_CAUSAL) return DASH_ERR_INVALID;
  if (!sched_known(sched)) return DASH_ERR_INVALID;
  sched = (dash_sched_t)resolve_sched(sched, mask, D, tiles(S), group);
  const void *ptrs[] = {q, k, v, o, dout, dq, dk, dv};
  for (const void *ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return DASH_ERR_INVALID;
  if (!lse || !aligned4(lse)) return DASH_ERR_INVALID;
  if (order_log && !aligned4(order_log)) return DASH_ERR_INVALID;
  const int N = tiles(S);
  const int causal = mask == DASH_MASK_CAUSAL;
  const BwdWorkspace need = carve_bwd(nullptr, B, S, H, D);
  if (!workspace || !aligned16(workspace) || workspace_bytes < need.total)
    return DASH_ERR_WORKSPACE;
  DevInfo dev;
  if ((st = device_info(&dev)) != DASH_OK) return st;
  const int Hkv = H / group;
  LaunchPlan plan;
  // every worker of a head must be resident at once for the shift schedules
  if (!make_plan(sched, causal, N, B * Hkv, dev.sms, &plan)) return DASH_ERR_UNSUPPORTED;
  const bool ordered = sched != DASH_SCHED_ATOMIC;
  const int K = plan.strands;

  CUtensorMap tq, tk, tv, tdo;
  if (!make_bshd_map(&tq, q, B, S, H, D) || !make_bshd_map(&tk, k, B, S, Hkv, D) ||
      !make_bshd_map(&tv, v, B, S, Hkv, D) || !make_bshd_map(&tdo, dout, B, S, H, D))
    return DASH_ERR_CUDA;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const BwdWorkspace w = carve_bwd(workspace, B, S, H, D);
  const float sc = resolve_scale(scale, D);
  if (stages & DASH_BWD_PROLOGUE) {
    // status word and semaphores are contiguous; the accumulator is cleared unless it has
    // two strands (SHIFT_DUAL stores the first partial of each strand)
    if ((keep_status ? cudaMemsetAsync(w.sem, 0, w.sem_bytes, s)
                     : cudaMemsetAsync(w.status, 0, kStatusBytes + w.sem_bytes, s)) != cudaSuccess ||
        (K == 1 && cudaMemsetAsync(w.dqacc, 0, w.dqacc_bytes, s) != cudaSuccess))
      return DASH_ERR_CUDA;
    // a partial last tile: its padding rows of lse2 / Dvec must read as zero
    if ((S % kTile) &&
        cudaMemsetAsync(w.lse2, 0, reinterpret_cast<char *>(w.dqacc) - reinterpret_cast<char *>(w.lse2),
                        s) != cudaSuccess)
      return DASH_ERR_CUDA;
    if (dash::launch_preprocess(static_cast<const __nv_bfloat16 *>(o),
                                static_cast<const __nv_bfloat16 *>(dout), lse, w.dvec, w.lse2, B,
                                S, H, D, w.status, g_wait_ns.load(), s) != cudaSuccess)
      return DASH_ERR_CUDA;
  }
  if (!(stages & (DASH_BWD_TILES | DASH_BWD_EPILOGUE))) return DASH_OK;
  dash::BwdParams p = base_params(w, dk, dv, ordered ? order_log : nullptr,
                                  log_stride > 0 ? log_stride : N, H, group, causal, sc);
  p.B = B;
  p.S = S;
  p.N = N;
  p.heads = B * Hkv;
  p.sched = plan.sched;
  p.workers = plan.workers;
  p.packed = plan.packed;
  if ((stages & DASH_BWD_TILES) &&
      dash::launch_bwd(D, ordered,
                       (causal ? (((N & 1) && plan.sched == dash::kShift) ? 2 : 1) : 0) |
                           (K > 1 ? 4 : 0),
                       tq, tk, tv, tdo, p, plan.grid, s) != cudaSuccess)
    return DASH_ERR_CUDA;
  if ((stages & DASH_BWD_EPILOGUE) &&
      dash::launch_dq_convert(w.dqacc, static_cast<__nv_bfloat16 *>(dq), sc, B, S, H, D, K, causal,
                              w.status, g_wait_ns.load(), s) != cudaSuccess)
    return DASH_ERR_CUDA;
  return DASH_OK;
}

dash_status_t dash_attn_bwd_stages(const void *q, const void *k, const void *v, const void *o,
                                   const void *dout, const float *lse, void *dq, void *dk,
                                   void *dv, int B, int S, int H, int group, int D, float scale,
                                   dash_mask_t mask, dash_sched_t sched, void *workspace,
                                   size_t workspace_bytes, unsigned stages,
                                   dash_stream_t stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, S, H, group, D, scale, mask, sched,
                  workspace, workspace_bytes, stages, stream, false, nullptr);
}

dash_status_t dash_attn_bwd_order_log(const void *q, const void *k, const void *v,
                                      const void *o, const void *dout, const float *lse,
                                      void *dq, void *dk, void *dv, int B, int S, int H,
                                      int group, int D, float scale, dash_mask_t mask,
                                      dash_sched_t sched, void *workspace,
                                      size_t workspace_bytes, int *order_log,
                                      dash_stream_t stream) {
  if (!order_log) return DASH_ERR_INVALID;
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, S, H, group, D, scale, mask, sched,
                  workspace, workspace_bytes, DASH_BWD_ALL, stream, false, order_log);
}

dash_status_t dash_attn_set_wait_limit(double seconds) {
  if (!(seconds >= 1e-3 && seconds <= 3600.0)) return DASH_ERR_INVALID;
  g_wait_ns.store((unsigned long long)(seconds * 1e9));
  return DASH_OK;
}

double dash_attn_wait_limit(void) { return (double)g_wait_ns.load() * 1e-9; }

dash_status_t dash_attn_bwd(const void *q, const void *k, const void *v, const void *o,
                            const void *dout, const float *lse, void *dq, void *dk, void *dv,
                            int B, int S, int H, int group, int D, float scale,
                            dash_mask_t mask, dash_sched_t sched, void *workspace,
                            size_t workspace_bytes, dash_stream_t stream) {
  return dash_attn_bwd_stages(q, k, v, o, dout, lse, dq, dk, dv, B, S, H, group, D, scale, mask,
                              sched, workspace, workspace_bytes, DASH_BWD_ALL, stream);
}

// ------------------------------------------------------------------ variable-length batches
// The sequences of a packed batch are independent attention problems.  With the packed
// schedules (SHIFT_FILL, SHIFT_DUAL, AUTO, which resolves to one of them) and ATOMIC, the
// workers of every sequence's heads are dealt onto the persistent grid together, one launch
// per group of at most dash::kMaxVarlenSeqs non-empty sequences; each sequence keeps its own
// tile count and accumulation order (the packed shift ranks at the sequence's position in
// the launch).  The single-round schedules (SERIAL, DESCENDING, SHIFT) run each sequence as
// the B = 1 problem on its own slices, one after another on `stream`.
static dash_status_t check_seqlens(const int *cu, int batch, int *max_len) {
  if (!cu || batch <= 0 || cu[0] != 0) return DASH_ERR_INVALID;
  int mx = 0;
  for (int b = 0; b < batch; ++b) {
    if (cu[b + 1] < cu[b]) return DASH_ERR_INVALID;
    mx = cu[b + 1] - cu[b] > mx ? cu[b + 1] - cu[b] : mx;
  }
  *max_len = mx;
  return DASH_OK;
}

// One launch of the packed varlen path: sequences [b0, b1) of the batch (b1 - b0 non-empty
// ones at most dash::kMaxVarlenSeqs), their tokens [tok0, tok1), tiles and workers.
struct VarlenGroup {
  int b0, b1, tok0, tok1, nseq, units;
  size_t ntiles;
  bool ragged;
};

// The next group from sequence b on (empty sequences are skipped).
VarlenGroup next_group(const int *cu, int batch, int b, int H, int Hkv, int causal) {
  VarlenGroup g{};
  g.b0 = b;
  g.tok0 = cu[b];
  long long units = 0;
  while (b < batch && g.nseq < dash::kMaxVarlenSeqs) {
    const int S = cu[b + 1] - cu[b];
    ++b;
    if (S == 0) continue;
    const int N = tiles(S);
    g.ntiles += (size_t)H * N;
    units += (long long)Hkv * dash::sched_workers(dash::kShift, causal, N, causal ? (N & 1) : 0);
    g.ragged |= (S % kTile) != 0;
    ++g.nseq;
  }
  g.b1 = b;
  g.tok1 = cu[b];
  g.units = units > (1LL << 30) ? -1 : (int)units;
  return g;
}

size_t table_bytes() {
  return align256(sizeof(int4) * dash::kMaxVarlenSeqs) + align256(sizeof(int) * (dash::kMaxVarlenSeqs + 1));
}

size_t packed_bytes(const VarlenGroup &g, int D) {
  return carve_tiles(nullptr, g.ntiles, D).total + table_bytes();
}

bool packed_sched(int sched) {
  return sched == DASH_SCHED_ATOMIC || sched == DASH_SCHED_SHIFT_FILL ||
         sched == DASH_SCHED_SHIFT_DUAL;
}

// Workspace of the packed path: the largest group's; validates sizes (0 = invalid).
size_t varlen_packed_bytes(const int *cu, int batch, int H, int group, int D, int causal) {
  size_t need = 0;
  for (int b = 0; b < batch;) {
    const VarlenGroup g = next_group(cu, batch, b, H, H / group, causal);
    if (g.units < 0 || g.ntiles >= (size_t)1 << 30 || g.tok1 - g.tok0 >= (1 << 30)) return 0;
    const size_t n = packed_bytes(g, D);
    need = n > need ? n : need;
    b = g.b1;
  }
  return need;
}

size_t dash_attn_bwd_varlen_workspace_bytes(const int *cu_seqlens, int batch, int H, int D) {
  int mx = 0;
  if (check_seqlens(cu_seqlens, batch, &mx) != DASH_OK || mx == 0) return 0;
  const size_t single = dash_attn_bwd_workspace_bytes(1, mx, H, D);
  if (single == 0) return 0;
  // either mask (the causal workers differ, the tiles do not); group 1 (tiles do not depend on it)
  const size_t packed = varlen_packed_bytes(cu_seqlens, batch, H, 1, D, 1);
  if (packed == 0) return 0;
  return packed > single ? packed : single;
}

dash_status_t dash_attn_fwd_varlen(const void *q, const void *k, const void *v, void *o,
                                   float *lse, const int *cu_seqlens, int batch, int H,
                                   int group, int D, float scale, dash_mask_t mask,
                                   void *workspace, size_t workspace_bytes,
                                   dash_stream_t stream) {
  int mx = 0;
  dash_status_t st = check_seqlens(cu_seqlens, batch, &mx);
  if (st != DASH_OK) return st;
  if (H <= 0 || group <= 0 || H % group) return DASH_ERR_INVALID;
  const int Hkv = H / group;
  bool first = true;
  for (int b = 0; b < batch; ++b) {
    const int s0 = cu_seqlens[b], S = cu_seqlens[b + 1] - s0;
    if (S == 0) continue;
    st = fwd_impl(static_cast<const __nv_bfloat16 *>(q) + (size_t)s0 * H * D,
                  static_cast<const __nv_bfloat16 *>(k) + (size_t)s0 * Hkv * D,
                  static_cast<const __nv_bfloat16 *>(v) + (size_t)s0 * Hkv * D,
                  static_cast<__nv_bfloat16 *>(o) + (size_t)s0 * H * D, lse + (size_t)s0 * H, 1,
                  S, H, group, D, scale, mask, workspace, workspace_bytes, stream, !first);
    if (st != DASH_OK) return st;
    first = false;
  }
  return DASH_OK;
}

// One packed launch sequence (clears, sequence table, preprocess, tile kernel, dQ convert)
// for group g; pointers are the batch's, offset here to the group's first token.
static dash_status_t bwd_varlen_group(const VarlenGroup &g, const int *cu, const void *q,
                                      const void *k, const void *v, const void *o,
                                      const void *dout, const float *lse, void *dq, void *dk,
                                      void *dv, int H, int group, int D, float sc, int causal,
                                      int sched, int sms, void *workspace, cudaStream_t s,
                                      bool keep_status, int *order_log, int log_stride) {
  using bf = __nv_bfloat16;
  const int Hkv = H / group, T = g.tok1 - g.tok0;
  const size_t qo = (size_t)g.tok0 * H * D, ko = (size_t)g.tok0 * Hkv * D;
  const bool ordered = sched != DASH_SCHED_ATOMIC;
  const int K = sched == DASH_SCHED_SHIFT_DUAL ? 2 : 1;
  const BwdWorkspace w = carve_tiles(workspace, g.ntiles, D);
  int4 *seqs = reinterpret_cast<int4 *>(static_cast<char *>(workspace) + w.total);
  int *wprefix = reinterpret_cast<int *>(reinterpret_cast<char *>(seqs) +
                                         align256(sizeof(int4) * dash::kMaxVarlenSeqs));
  // the sequence table, tokens relative to the group's first
  static thread_local dash::VarlenTable t;
  int n = 0, tile = 0, unit = 0;
  for (int b = g.b0; b < g.b1; ++b) {
    const int S = cu[b + 1] - cu[b];
    if (S == 0) continue;
    const int N = tiles(S);
    t.seqs[n] = make_int4(S, cu[b] - g.tok0, tile, N);
    t.wprefix[n] = unit;
    tile += H * N;
    unit += Hkv * dash::sched_workers(dash::kShift, causal, N, causal ? (N & 1) : 0);
    ++n;
  }
  t.wprefix[n] = unit;
  t.batch = n;

  CUtensorMap tq, tk, tv, tdo;
  if (!make_thd_map(&tq, static_cast<const bf *>(q) + qo, T, H, D) ||
      !make_thd_map(&tk, static_cast<const bf *>(k) + ko, T, Hkv, D) ||
      !make_thd_map(&tv, static_cast<const bf *>(v) + ko, T, Hkv, D) ||
      !make_thd_map(&tdo, static_cast<const bf *>(dout) + qo, T, H, D))
    return DASH_ERR_CUDA;
  if ((keep_status ? cudaMemsetAsync(w.sem, 0, w.sem_bytes, s)
                   : cudaMemsetAsync(w.status, 0, kStatusBytes + w.sem_bytes, s)) != cudaSuccess ||
      (K == 1 && cudaMemsetAsync(w.dqacc, 0, w.dqacc_bytes, s) != cudaSuccess))
    return DASH_ERR_CUDA;
  if (g.ragged &&
      cudaMemsetAsync(w.lse2, 0, reinterpret_cast<char *>(w.dqacc) - reinterpret_cast<char *>(w.lse2),
                      s) != cudaSuccess)
    return DASH_ERR_CUDA;
  if (dash::launch_varlen_setup(t, seqs, wprefix, s) != cudaSuccess ||
      dash::launch_preprocess_varlen(static_cast<const bf *>(o) + qo,
                                     static_cast<const bf *>(dout) + qo, lse + (size_t)g.tok0 * H,
                                     w.dvec, w.lse2, seqs, n, T, H, D, w.status,
                                     g_wait_ns.load(), s) != cudaSuccess)
    return DASH_ERR_CUDA;
  dash::BwdParams p = base_params(w, static_cast<bf *>(dk) + ko, static_cast<bf *>(dv) + ko,
                                  ordered ? order_log : nullptr, log_stride, H, group, causal,
                                  sc);
  p.seqs = seqs;
  p.seq_wprefix = wprefix;
  p.batch = n;
  p.units = unit;
  p.sched = dash::kShift;
  p.packed = sched == DASH_SCHED_SHIFT_FILL || sched == DASH_SCHED_SHIFT_DUAL;
  const int grid = unit < sms ? unit : sms;
  if (dash::launch_bwd_varlen(D, ordered, causal, K > 1, tq, tk, tv, tdo, p, grid, s) !=
          cudaSuccess ||
      dash::launch_dq_convert_varlen(w.dqacc, static_cast<bf *>(dq) + qo, sc, seqs, n,
                                     (int)g.ntiles, H, D, K, causal, w.status, g_wait_ns.load(),
                                     s) != cudaSuccess)
    return DASH_ERR_CUDA;
  return DASH_OK;
}

static dash_status_t bwd_varlen_impl(const void *q, const void *k, const void *v, const void *o,
                                     const void *dout, const float *lse, void *dq, void *dk,
                                     void *dv, const int *cu_seqlens, int batch, int H,
                                     int group, int D, float scale, dash_mask_t mask,
                                     dash_sched_t sched, void *workspace, size_t workspace_bytes,
                                     dash_stream_t stream, int *order_log) {
  int mx = 0;
  dash_status_t st = check_seqlens(cu_seqlens, batch, &mx);
  if (st != DASH_OK) return st;
  if (H <= 0 || group <= 0 || H % group) return DASH_ERR_INVALID;
  if (mask != DASH_MASK_FULL && mask != DASH_MASK_CAUSAL) return DASH_ERR_INVALID;
  if (!sched_known(sched)) return DASH_ERR_INVALID;
  if (order_log && !aligned4(order_log)) return DASH_ERR_INVALID;
  // refuse before enqueuing anything: every sequence must be runnable with this schedule
  DevInfo dev;
  if ((st = device_info(&dev)) != DASH_OK) return st;
  const int Hkv = H / group, causal = mask == DASH_MASK_CAUSAL;
  const int rs_all = resolve_sched(sched, mask, D, tiles(mx), group);
  const bool packed = mx > 0 && packed_sched(rs_all);
  for (int b = 0; b < batch; ++b) {
    const int S = cu_seqlens[b + 1] - cu_seqlens[b];
    if (S == 0) continue;
    if ((st = check_sizes(1, S, H, group, D)) != DASH_OK) return st;
    if (packed) continue;
    const int N = tiles(S), rs = resolve_sched(sched, mask, D, N, group);
    LaunchPlan plan;
    if (!make_plan(rs, causal, N, Hkv, dev.sms, &plan)) return DASH_ERR_UNSUPPORTED;
  }
  if (mx == 0) return DASH_OK;
  const void *ptrs[] = {q, k, v, o, dout, dq, dk, dv};
  for (const void *ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return DASH_ERR_INVALID;
  if (!lse || !aligned4(lse)) return DASH_ERR_INVALID;
  if (!workspace || !aligned16(workspace)) return DASH_ERR_WORKSPACE;
  // the order log is [tiles of all sequences][longest sequence's tile count]
  const int log_stride = tiles(mx);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (packed) {
    const size_t need = varlen_packed_bytes(cu_seqlens, batch, H, group, D, causal);
    if (need == 0) return DASH_ERR_UNSUPPORTED;
    if (workspace_bytes < need) return DASH_ERR_WORKSPACE;
    const float sc = resolve_scale(scale, D);
    size_t tiles_before = 0;
    for (int b = 0; b < batch;) {
      const VarlenGroup g = next_group(cu_seqlens, batch, b, H, Hkv, causal);
      if (g.nseq > 0) {
        st = bwd_varlen_group(g, cu_seqlens, q, k, v, o, dout, lse, dq, dk, dv, H, group, D, sc,
                              causal, rs_all, dev.sms, workspace, s, b > 0,
                              order_log ? order_log + tiles_before * log_stride : nullptr,
                              log_stride);
        if (st != DASH_OK) return st;
      }
      tiles_before += g.ntiles;
      b = g.b1;
    }
    return DASH_OK;
  }
  if (workspace_bytes < dash_attn_bwd_workspace_bytes(1, mx, H, D)) return DASH_ERR_WORKSPACE;
  bool first = true;
  size_t tiles_before = 0;
  for (int b = 0; b < batch; ++b) {
    const int s0 = cu_seqlens[b], S = cu_seqlens[b + 1] - s0;
    if (S == 0) continue;
    const size_t qo = (size_t)s0 * H * D, ko = (size_t)s0 * Hkv * D;
    st = bwd_impl(static_cast<const __nv_bfloat16 *>(q) + qo,
                  static_cast<const __nv_bfloat16 *>(k) + ko,
                  static_cast<const __nv_bfloat16 *>(v) + ko,
                  static_cast<const __nv_bfloat16 *>(o) + qo,
                  static_cast<const __nv_bfloat16 *>(dout) + qo, lse + (size_t)s0 * H,
                  static_cast<__nv_bfloat16 *>(dq) + qo, static_cast<__nv_bfloat16 *>(dk) + ko,
                  static_cast<__nv_bfloat16 *>(dv) + ko, 1, S, H, group, D, scale, mask, sched,
                  workspace, workspace_bytes, DASH_BWD_ALL, stream, !first,
                  order_log ? order_log + tiles_before * log_stride : nullptr, log_stride);
    if (st != DASH_OK) return st;
    first = false;
    tiles_before += (size_t)H * tiles(S);
  }
  return DASH_OK;
}

dash_status_t dash_attn_bwd_varlen(const void *q, const void *k, const void *v, const void *o,
                                   const void *dout, const float *lse, void *dq, void *dk,
                                   void *dv, const int *cu_seqlens, int batch, int H, int group,
                                   int D, float scale, dash_mask_t mask, dash_sched_t sched,
                                   void *workspace, size_t workspace_bytes,
                                   dash_stream_t stream) {
  return bwd_varlen_impl(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens, batch, H, group, D, scale,
                         mask, sched, workspace, workspace_bytes, stream, nullptr);
}

dash_status_t dash_attn_bwd_varlen_order_log(const void *q, const void *k, const void *v,
                                             const void *o, const void *dout, const float *lse,
                                             void *dq, void *dk, void *dv, const int *cu_seqlens,
                                             int batch, int H, int group, int D, float scale,
                                             dash_mask_t mask, dash_sched_t sched,
                                             void *workspace, size_t workspace_bytes,
                                             int *order_log, dash_stream_t stream) {
  if (!order_log) return DASH_ERR_INVALID;
  return bwd_varlen_impl(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens, batch, H, group, D, scale,
                         mask, sched, workspace, workspace_bytes, stream, order_log);
}

dash_status_t dash_attn_status(void *workspace, dash_stream_t stream) {
  if (!workspace) return DASH_ERR_INVALID;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DASH_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DASH_ERR_CUDA;
  if (word & (dash::kErrMbarTimeout | dash::kErrSemTimeout | dash::kErrAborted))
    return DASH_ERR_TIMEOUT;
  if (word) return DASH_ERR_CUDA;
  return DASH_OK;
}

dash_status_t dash_attn_bwd_status(void *workspace, dash_stream_t stream) {
  return dash_attn_status(workspace, stream);
}

const char *dash_status_string(dash_status_t s) {
  switch (s) {
    case DASH_OK:
      return "ok";
    case DASH_ERR_INVALID:
      return "invalid argument";
    case DASH_ERR_UNSUPPORTED:
      return "unsupported configuration";
    case DASH_ERR_CUDA:
      return "CUDA error";
    case DASH_ERR_TIMEOUT:
      return "device-side wait timed out";
    case DASH_ERR_WORKSPACE:
      return "workspace missing or too small";
  }
  return "unknown status";
}

#ifdef DASH_TRACE_BUILD
// Development trace build only: device buffer of 64 x 32 u64 for the event clocks of CTA
// `cta`.
void dash_debug_set_trace(unsigned long long *buf, int cta) {
  g_trace = buf;
  g_trace_cta = cta;
}
#endif

// ------------------------------------------------------------------ schedule queries
static bool sched_args_ok(int &sched, int mask, int N) {
  if (!sched_known(sched) || (mask != 0 && mask != 1) || N <= 0) return false;
  sched = resolve_sched(sched, mask, 0, N, 1);
  return true;
}

int dash_sched_resolve(int sched, int mask, int D, int N, int group) {
  if (!sched_known(sched) || (mask != 0 && mask != 1) || N <= 0 || group <= 0 ||
      (D != 64 && D != 128))
    return -1;
  return resolve_sched(sched, mask, D, N, group);
}

int dash_sched_grid(int sched, int mask, int N, int heads, int sms) {
  LaunchPlan pl;
  if (!sched_args_ok(sched, mask, N) || heads <= 0 || sms <= 0 ||
      !make_plan(sched, mask, N, heads, sms, &pl))
    return -1;
  return pl.grid;
}

int dash_sched_packed_rank(int mask, int N, int heads, int grid, int head, int q, int kv) {
  int fill = DASH_SCHED_SHIFT_FILL;
  if (!sched_args_ok(fill, mask, N) || heads <= 0 || head < 0 ||
      head >= heads || q < 0 || q >= N || kv < 0 || kv >= N || (mask && kv > q))
    return -1;
  const int W = dash::sched_workers(dash::kShift, mask, N, N & 1);
  if (grid < 1 || grid > heads * W) return -1;
  return dash::packed_rank(mask, N, grid, head, q, kv, N & 1);
}

int dash_sched_workers(int sched, int mask, int N) {
  if (!sched_args_ok(sched, mask, N)) return -1;
  return dash::sched_workers(dash::traversal(sched, mask, N), mask, N, N & 1);
}

int dash_sched_segments(int sched, int mask, int N, int worker) {
  sched = resolve_sched(sched, mask, 0, N, 1);
  const int W = dash_sched_workers(sched, mask, N);
  if (W < 0 || worker < 0 || worker >= W) return -1;
  return dash::sched_segments(dash::traversal(sched, mask, N), mask, N, worker, N & 1);
}

int dash_sched_steps(int sched, int mask, int N, int worker, int segment) {
  sched = resolve_sched(sched, mask, 0, N, 1);
  const int nseg = dash_sched_segments(sched, mask, N, worker);
  if (nseg < 0 || segment < 0 || segment >= nseg) return -1;
  return dash::seg_steps(dash::traversal(sched, mask, N), mask, N, worker, segment, N & 1);
}

int dash_sched_step(int sched, int mask, int N, int worker, int segment, int step, int *kv,
                    int *q, int *rank) {
  sched = resolve_sched(sched, mask, 0, N, 1);
  const int n = dash_sched_steps(sched, mask, N, worker, segment);
  if (n < 0 || step < 0 || step >= n) return -1;
  const int t = dash::traversal(sched, mask, N);
  const int kvb = dash::seg_kv(t, mask, N, worker, segment, N & 1);
  const int qt = dash::step_q(t, mask, N, worker, segment, step, N & 1);
  if (kv) *kv = kvb;
  if (q) *q = qt;
  // ATOMIC adds in no fixed order; report the position the traversal would give
  if (rank) *rank = dash::dq_rank(t, mask, N, qt, kvb, N & 1);
  return 0;
}

}  // extern "C"
