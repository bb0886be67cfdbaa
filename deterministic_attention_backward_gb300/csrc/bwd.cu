// bwd.cu -- launches of the tile kernel (bwd_kernel.cuh) on uniform batches [B, S, H, D].
#include "bwd_kernel.cuh"

namespace dash {

cudaError_t launch_bwd(int D, bool deterministic, int mode, const CUtensorMap &tq,
                       const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tdo,
                       const BwdParams &p, int grid, cudaStream_t stream) {
  switch (mode) {
    case 6: return launch_bwd_o<6>(D, deterministic, tq, tk, tv, tdo, p, grid, stream);
    case 5: return launch_bwd_o<5>(D, deterministic, tq, tk, tv, tdo, p, grid, stream);
    case 4: return launch_bwd_o<4>(D, deterministic, tq, tk, tv, tdo, p, grid, stream);
    case 2: return launch_bwd_o<2>(D, deterministic, tq, tk, tv, tdo, p, grid, stream);
    case 1: return launch_bwd_o<1>(D, deterministic, tq, tk, tv, tdo, p, grid, stream);
    default: return launch_bwd_o<0>(D, deterministic, tq, tk, tv, tdo, p, grid, stream);
  }
}

}  // namespace dash
