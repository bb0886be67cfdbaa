// noalloc.cu -- dash_attn_bwd_noalloc: the backward pass without a caller-provided
// workspace and without allocating anything.
//
// Some callers cannot hand the library a workspace: a plugin inside a host application
// whose memory pool owns the whole device and gives plugins no allocator, or a code path
// where calling cudaMalloc would implicitly synchronise the device and stall every other
// stream.  For them the workspace lives in a fixed, file-scope device array of
// DASH_NOALLOC_SCRATCH_BYTES.  The array is created when the library's module is loaded on
// a device and stays there, on every device that uses this library, until the process
// exits.
//
// The host cannot use the array's name as a device address (in host code it names a
// host-side shadow), so the first call on each device, with that device current, asks the
// runtime for the array's device address with cudaGetSymbolAddress and caches it; that
// first call should therefore come before any stream capture.  Every call on a device
// shares the one array: two calls whose work may overlap on the GPU (different streams,
// no ordering between them) race on it.  Each call clears what must start at zero (status
// word, dQ accumulator, ordering semaphores) before its kernels run, exactly as
// dash_attn_bwd does with a caller workspace.
#include <mutex>

#include "dash_attn.h"

namespace {

static __device__ __align__(256) unsigned char g_dash_scratch[DASH_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void *g_scratch_ptr[64] = {};

// Device address of the scratch array on the current device (looked up once per device).
dash_status_t scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DASH_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dash_scratch) != cudaSuccess || !p) return DASH_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return DASH_OK;
}

}  // namespace

extern "C" dash_status_t dash_attn_bwd_noalloc(const void *q, const void *k, const void *v,
                                               const void *o, const void *dout,
                                               const float *lse, void *dq, void *dk, void *dv,
                                               int B, int S, int H, int group, int D,
                                               float scale, dash_mask_t mask,
                                               dash_sched_t sched, dash_stream_t stream) {
  const size_t need = dash_attn_bwd_workspace_bytes(B, S, H, D);
  if (need == 0) {  // sizes the backward does not accept: let it report which error
    return dash_attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, S, H, group, D, scale, mask,
                         sched, nullptr, 0, stream);
  }
  if (need > (size_t)DASH_NOALLOC_SCRATCH_BYTES) return DASH_ERR_WORKSPACE;
  void *scratch = nullptr;
  const dash_status_t st = scratch_address(&scratch);
  if (st != DASH_OK) return st;
  return dash_attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, S, H, group, D, scale, mask, sched,
                       scratch, (size_t)DASH_NOALLOC_SCRATCH_BYTES, stream);
}

// The status word sits at the start of the array, where dash_attn_bwd keeps it in any
// workspace.
extern "C" dash_status_t dash_attn_noalloc_status(dash_stream_t stream) {
  void *scratch = nullptr;
  const dash_status_t st = scratch_address(&scratch);
  if (st != DASH_OK) return st;
  return dash_attn_status(scratch, stream);
}
