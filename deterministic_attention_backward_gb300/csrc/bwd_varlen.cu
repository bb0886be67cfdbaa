// bwd_varlen.cu -- launches of the tile kernel (bwd_kernel.cuh) on a packed variable-length
// batch [T, H, D]: every sequence's heads are packed onto the persistent grid in one launch
// (the packed shift traversal; the atomic variant visits the same units unordered).
#include "bwd_kernel.cuh"

namespace dash {

cudaError_t launch_bwd_varlen(int D, bool deterministic, bool causal, bool dual,
                              const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                              const CUtensorMap &tdo, const BwdParams &p, int grid,
                              cudaStream_t stream) {
  const int mode = 8 | (causal ? 1 : 0) | (dual ? 4 : 0);
  switch (mode) {
    case 13: return launch_bwd_o<13>(D, deterministic, tq, tk, tv, tdo, p, grid, stream);
    case 12: return launch_bwd_o<12>(D, deterministic, tq, tk, tv, tdo, p, grid, stream);
    case 9: return launch_bwd_o<9>(D, deterministic, tq, tk, tv, tdo, p, grid, stream);
    default: return launch_bwd_o<8>(D, deterministic, tq, tk, tv, tdo, p, grid, stream);
  }
}

}  // namespace dash
