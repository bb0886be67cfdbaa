// aux.cu -- the two memory-bound companions of the backward tile kernel:
//   preprocess:  Dvec[b,h,i] = sum_d dO[b,i,h,d] * O[b,i,h,d]   (fp32)
//                lse2[b,h,i] = LSE[b,h,i] * log2(e)              (exp2-domain LSE)
//                (both [B,H,N*128]: each (b,h) padded to whole tiles; padding stays zero)
//   dq_convert:  dQ[b,i,h,:] = bf16_rne(scale * (acc_0 [+ acc_1]))  (the tile's accumulation
//                strands in ascending order; tile-native -> BSHD, i < S)
// and their forms over a packed variable-length batch [T, H, D], where a sequence table
// {S_b, first token, first tile, N_b} (non-empty sequences, ascending tokens) places each
// token row: sequence b's per-tile arrays are [H, N_b] tiles from its first tile on, and its
// LSE is [H, S_b] from row (first token) * H of the packed LSE.
#include "common.cuh"
#include "ptx.cuh"

namespace dash {
namespace {

// Dot products sum_d o[d] * dout[d] of `rows` consecutive D-element rows.  The rows are
// streamed into shared memory by bulk (TMA) copies, kRows rows of each tensor per chunk,
// two chunks in flight per CTA: the copy engine keeps far more bytes in flight than
// per-thread loads do (measured: 47 us at 37 % of DRAM bandwidth for 16k tokens x 16 heads
// at D = 128 with per-thread loads).  Chunks are dealt round-robin to the CTAs; 256 / kRows
// threads share a row, 16 elements each.  fn(row, dot) runs on the row's first thread.  A
// wait that runs out records kErrMbarTimeout in `status` and stops the CTA.
template <int D>
struct PreCfg {
  static constexpr int kRows = 32 * 128 / D;             // 8 KB of each tensor per chunk
  static constexpr int kChunkBytes = kRows * D * 2;
  static constexpr int kStages = 2;
  static constexpr int kThreadsPerRow = 256 / kRows;     // 8 (D = 128) or 4 (D = 64)
  static constexpr int kElems = D / kThreadsPerRow;      // 16
};
template <int D, typename F>
__device__ __forceinline__ void for_each_row_dot(const __nv_bfloat16 *__restrict__ o,
                                                 const __nv_bfloat16 *__restrict__ dout,
                                                 long long rows, uint32_t *status,
                                                 unsigned long long wait_ns, F fn) {
  using C = PreCfg<D>;
  __shared__ __align__(128) uint8_t buf[C::kStages][2][C::kChunkBytes];
  __shared__ __align__(8) uint64_t bar[C::kStages];
  __shared__ int s_abort;
  const Abort ab{&s_abort, status, wait_ns};
  if (threadIdx.x == 0) {
    for (int st = 0; st < C::kStages; ++st) mbar_init(&bar[st], 1);
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const long long nchunks = (rows + C::kRows - 1) / C::kRows;
  auto issue = [&](long long c, int st) {
    const long long r0 = c * C::kRows;
    const long long left = rows - r0;
    const uint32_t bytes = (uint32_t)(left < C::kRows ? left : C::kRows) * D * 2;
    mbar_arrive_expect_tx(&bar[st], 2 * bytes);
    bulk_load(buf[st][0], o + r0 * D, bytes, &bar[st]);
    bulk_load(buf[st][1], dout + r0 * D, bytes, &bar[st]);
  };
  int issued = 0;  // chunks issued by thread 0 (for the drain on a failed wait)
  if (threadIdx.x == 0)
    for (int st = 0; st < C::kStages; ++st)
      if (blockIdx.x + (long long)st * gridDim.x < nchunks) {
        issue(blockIdx.x + (long long)st * gridDim.x, st);
        ++issued;
      }
  const int rl = threadIdx.x / C::kThreadsPerRow, li = threadIdx.x % C::kThreadsPerRow;
  uint32_t k = 0;
  for (long long c = blockIdx.x; c < nchunks; c += gridDim.x, ++k) {
    const int st = (int)(k % C::kStages);
    const uint32_t ph = (k / C::kStages) & 1;
    const bool ok = mbar_wait(&bar[st], ph, ab);
    if (__syncthreads_or(!ok)) {
      // leave no copy in flight into shared memory
      if (threadIdx.x == 0)
        for (uint32_t kk = k; kk < (uint32_t)issued; ++kk)
          mbar_wait_drain(&bar[kk % C::kStages], (kk / C::kStages) & 1, 100000000ull);
      return;
    }
    const long long r0 = c * C::kRows;
    const long long left = rows - r0;
    const int n = (int)(left < C::kRows ? left : C::kRows);
    float acc = 0.f;
    if (rl < n) {
      const uint8_t *pa = buf[st][0] + (rl * D + li * C::kElems) * 2;
      const uint8_t *pc = buf[st][1] + (rl * D + li * C::kElems) * 2;
#pragma unroll
      for (int q = 0; q < C::kElems / 8; ++q) {
        const uint4 a = *reinterpret_cast<const uint4 *>(pa + 16 * q);
        const uint4 b = *reinterpret_cast<const uint4 *>(pc + 16 * q);
        const __nv_bfloat162 *a2 = reinterpret_cast<const __nv_bfloat162 *>(&a);
        const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&b);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = __bfloat1622float2(a2[e]), y = __bfloat1622float2(b2[e]);
          acc = fmaf(x.x, y.x, acc);
          acc = fmaf(x.y, y.y, acc);
        }
      }
    }
#pragma unroll
    for (int off = C::kThreadsPerRow / 2; off > 0; off >>= 1)
      acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (li == 0 && rl < n) fn(r0 + rl, acc);
    __syncthreads();  // every thread is done with this stage
    if (threadIdx.x == 0) {
      const long long c2 = c + (long long)C::kStages * gridDim.x;
      if (c2 < nchunks) {
        issue(c2, st);
        ++issued;
      }
    }
  }
}

// Rows enumerated in BSHD order, so the O/dO reads of a warp are one contiguous range.
template <int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const __nv_bfloat16 *__restrict__ o,
                                                         const __nv_bfloat16 *__restrict__ dout,
                                                         const float *__restrict__ lse,
                                                         float *__restrict__ dvec,
                                                         float *__restrict__ lse2, int B, int S,
                                                         int H, uint32_t *status,
                                                         unsigned long long wait_ns) {
  const long long rows = (long long)B * S * H;
  for_each_row_dot<D>(o, dout, rows, status, wait_ns, [&](long long row, float acc) {
    const int h = (int)(row % H);
    const long long bi = row / H;
    const int i = (int)(bi % S);
    const int b = (int)(bi / S);
    const size_t Sp = (size_t)(S + kTile - 1) / kTile * kTile;
    const size_t r = ((size_t)b * H + h) * Sp + i;
    dvec[r] = acc;
    lse2[r] = lse[((size_t)b * H + h) * S + i] * kLog2e;
  });
}

// dQ convert, one CTA per dQ tile: the tile's strands are read in their tile-native layout
// ([D/4][128][4] fp32: consecutive threads take consecutive rows, 512 contiguous bytes per
// warp), summed, scaled and rounded to bf16 into a [128][D] shared-memory tile, which is
// then written row by row (D*2 contiguous bytes per row) -- both sides coalesced.
template <int D>
struct ConvTile {
  static constexpr int kRowBytes = D * 2 + 8;  // padded: the 8-byte stores of a warp hit
                                               // at most two rows per bank
  static constexpr int kBytes = kTile * kRowBytes;
};
// Sums `strands` strands of the tile at `tb` into shared memory `st` (bf16, scaled).  Each
// strand is [D/4][128][4] fp32; it is brought in by bulk (TMA) copies of kConvCols
// 4-column groups (16 KB) at a time, two passes in flight, and read back row-fastest
// (conflict-free); `stage` holds 2 x K x 16 KB, `bar` two mbarriers.  A wait that runs out
// records kErrMbarTimeout through `ab` and returns false.
constexpr int kConvCols = 8;                              // 4-column groups per pass
constexpr int kConvChunk = kConvCols * kTile * 16;         // bytes per strand per pass
template <int D, int K>
__device__ __forceinline__ bool conv_tile_load(const float *__restrict__ tb, int strands,
                                               float scale, uint8_t *st, uint8_t *stage,
                                               uint64_t *bar, const Abort &ab) {
  constexpr int C4 = D / 4;
  constexpr int kPasses = C4 / kConvCols;
  constexpr size_t kStrandBytes = (size_t)C4 * kTile * 16;
  auto issue = [&](int pass) {
    uint8_t *dst = stage + (pass & 1) * (K * kConvChunk);
    mbar_arrive_expect_tx(&bar[pass & 1], strands * kConvChunk);
    for (int k = 0; k < strands; ++k)
      bulk_load(dst + k * kConvChunk, reinterpret_cast<const uint8_t *>(tb) + k * kStrandBytes +
                                          (size_t)pass * kConvChunk,
                kConvChunk, &bar[pass & 1]);
  };
  if (threadIdx.x == 0) {
    issue(0);
    if (kPasses > 1) issue(1);
  }
  for (int pass = 0; pass < kPasses; ++pass) {
    const bool ok = mbar_wait(&bar[pass & 1], (pass >> 1) & 1, ab);
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0)  // leave no copy in flight into shared memory
        for (int q = pass; q < kPasses && q < pass + 2; ++q)
          mbar_wait_drain(&bar[q & 1], (q >> 1) & 1, 100000000ull);
      return false;
    }
    const float4 *s0 = reinterpret_cast<const float4 *>(stage + (pass & 1) * (K * kConvChunk));
#pragma unroll
    for (int j = 0; j < kConvCols * kTile / 256; ++j) {
      const int idx = threadIdx.x + 256 * j;  // (4-column group within the pass, row)
      float4 v = s0[idx];
      if constexpr (K == 2) {
        if (strands > 1) {
          const float4 w = s0[kConvChunk / 16 + idx];
          v = make_float4(v.x + w.x, v.y + w.y, v.z + w.z, v.w + w.w);
        }
      }
      const int c4 = pass * kConvCols + idx / kTile, r = idx % kTile;
      __nv_bfloat162 lo = __floats2bfloat162_rn(v.x * scale, v.y * scale);
      __nv_bfloat162 hi = __floats2bfloat162_rn(v.z * scale, v.w * scale);
      uint2 packed;
      packed.x = *reinterpret_cast<uint32_t *>(&lo);
      packed.y = *reinterpret_cast<uint32_t *>(&hi);
      *reinterpret_cast<uint2 *>(st + r * ConvTile<D>::kRowBytes + c4 * 8) = packed;
    }
    __syncthreads();  // every thread is done with this pass's stage
    if (threadIdx.x == 0 && pass + 2 < kPasses) issue(pass + 2);
  }
  return true;
}
// Dynamic shared memory of a convert CTA: two passes of K strands, the bf16 tile, barriers.
template <int D, int K>
constexpr int conv_smem_bytes() {
  return 2 * K * kConvChunk + ConvTile<D>::kBytes + 32;
}
// Writes rows [0, rows) of the shared tile; row r goes to dst + r * row_stride (elements).
template <int D>
__device__ __forceinline__ void conv_tile_store(const uint8_t *st, __nv_bfloat16 *dst,
                                                size_t row_stride, int rows) {
  constexpr int kPer = D / 4;  // 8-byte chunks per row
  for (int idx = threadIdx.x; idx < rows * kPer; idx += blockDim.x) {
    const int r = idx / kPer, c = idx % kPer;
    *reinterpret_cast<uint2 *>(dst + (size_t)r * row_stride + c * 4) =
        *reinterpret_cast<const uint2 *>(st + r * ConvTile<D>::kRowBytes + c * 8);
  }
}

template <int D, int K>
__global__ void __launch_bounds__(256) dq_convert_kernel(const float *__restrict__ acc,
                                                         __nv_bfloat16 *__restrict__ dq,
                                                         float scale, int B, int S, int H,
                                                         int causal, uint32_t *status,
                                                         unsigned long long wait_ns) {
  extern __shared__ __align__(1024) uint8_t sm[];
  uint8_t *st = sm + 2 * K * kConvChunk;
  uint64_t *bar = reinterpret_cast<uint64_t *>(st + ConvTile<D>::kBytes);
  int *s_abort = reinterpret_cast<int *>(bar + 2);
  const Abort ab{s_abort, status, wait_ns};
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int N = (S + kTile - 1) / kTile;
  const long long t = blockIdx.x;  // (b*H + h)*N + i
  const int i = (int)(t % N);
  const long long bh = t / N;
  const int h = (int)(bh % H);
  const int b = (int)(bh / H);
  // a strand that received no partial is not read (tile with a single partial)
  if (!conv_tile_load<D, K>(acc + t * K * (size_t)(kTile * D), (causal ? i + 1 : N) > 1 ? K : 1,
                            scale, st, sm, bar, ab))
    return;
  const int rows = S - i * kTile < kTile ? S - i * kTile : kTile;
  conv_tile_store<D>(st, dq + (((size_t)b * S + (size_t)i * kTile) * H + h) * D,
                     (size_t)H * D, rows);
}

// The sequence holding packed token t: the last table entry whose first token is <= t.
__device__ __forceinline__ int seq_of_token(const int4 *__restrict__ seqs, int batch, int t) {
  int lo = 0, hi = batch;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (seqs[mid].y <= t) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Writes the sequence table (passed by value as the kernel's parameter) into the workspace.
__global__ void varlen_setup_kernel(const VarlenTable t, int4 *__restrict__ seqs,
                                    int *__restrict__ wprefix) {
  for (int i = threadIdx.x; i < t.batch; i += blockDim.x) seqs[i] = t.seqs[i];
  for (int i = threadIdx.x; i <= t.batch; i += blockDim.x) wprefix[i] = t.wprefix[i];
}

// The same over the packed (t, h) rows of a variable-length batch.
template <int D>
__global__ void __launch_bounds__(256) preprocess_varlen_kernel(
    const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
    const float *__restrict__ lse, float *__restrict__ dvec, float *__restrict__ lse2,
    const int4 *__restrict__ seqs, int batch, int T, int H, uint32_t *status,
    unsigned long long wait_ns) {
  const long long rows = (long long)T * H;
  for_each_row_dot<D>(o, dout, rows, status, wait_ns, [&](long long row, float acc) {
    const int h = (int)(row % H);
    const int t = (int)(row / H);
    const int4 sq = seqs[seq_of_token(seqs, batch, t)];
    const int i = t - sq.y;
    const size_t r = ((size_t)sq.z + (size_t)h * sq.w) * kTile + i;
    dvec[r] = acc;
    lse2[r] = lse[(size_t)sq.y * H + (size_t)h * sq.x + i] * kLog2e;
  });
}

// The same per tile of a packed batch: tile t of the group's per-tile arrays belongs to
// the last sequence whose first tile is <= t.
template <int D, int K>
__global__ void __launch_bounds__(256) dq_convert_varlen_kernel(
    const float *__restrict__ acc, __nv_bfloat16 *__restrict__ dq, float scale,
    const int4 *__restrict__ seqs, int batch, int H, int causal, uint32_t *status,
    unsigned long long wait_ns) {
  extern __shared__ __align__(1024) uint8_t sm[];
  uint8_t *st = sm + 2 * K * kConvChunk;
  uint64_t *bar = reinterpret_cast<uint64_t *>(st + ConvTile<D>::kBytes);
  int *s_abort = reinterpret_cast<int *>(bar + 2);
  const Abort ab{s_abort, status, wait_ns};
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int t = blockIdx.x;
  int lo = 0, hi = batch;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (seqs[mid].z <= t) lo = mid;
    else hi = mid;
  }
  const int4 sq = seqs[lo];  // {S_b, first token, first tile, N_b}
  const int local = t - sq.z;
  const int h = local / sq.w, i = local % sq.w;
  if (!conv_tile_load<D, K>(acc + (size_t)t * K * (kTile * D),
                            (causal ? i + 1 : sq.w) > 1 ? K : 1, scale, st, sm, bar, ab))
    return;
  const int rows = sq.x - i * kTile < kTile ? sq.x - i * kTile : kTile;
  conv_tile_store<D>(st, dq + (((size_t)sq.y + (size_t)i * kTile) * H + h) * D, (size_t)H * D,
                     rows);
}

int grid_for(long long work, int per_block, int cap) {
  long long g = (work + per_block - 1) / per_block;
  if (g < 1) g = 1;
  return (int)(g > cap ? cap : g);
}

}  // namespace

// Chunks of PreCfg<D>::kRows rows dealt to at most six CTAs per SM (shared memory: 32 KB
// each), two chunks in flight per CTA.
int pre_grid(long long rows, int D) {
  const long long chunks = (rows + 32 * 128 / D - 1) / (32 * 128 / D);
  return grid_for(chunks, 1, 152 * 6);
}

cudaError_t launch_preprocess(const __nv_bfloat16 *o, const __nv_bfloat16 *dout, const float *lse,
                              float *dvec, float *lse2, int B, int S, int H, int D,
                              uint32_t *status, unsigned long long wait_ns, cudaStream_t stream) {
  const int grid = pre_grid((long long)B * S * H, D);
  if (D == 64)
    preprocess_kernel<64><<<grid, 256, 0, stream>>>(o, dout, lse, dvec, lse2, B, S, H, status,
                                                    wait_ns);
  else
    preprocess_kernel<128><<<grid, 256, 0, stream>>>(o, dout, lse, dvec, lse2, B, S, H, status,
                                                     wait_ns);
  return cudaGetLastError();
}

template <int D, int K>
cudaError_t conv_launch(int grid, cudaStream_t stream, const float *dqacc, __nv_bfloat16 *dq,
                        float scale, int B, int S, int H, int causal, uint32_t *status,
                        unsigned long long wait_ns) {
  constexpr int kSmem = conv_smem_bytes<D, K>();
  cudaError_t e = cudaFuncSetAttribute(dq_convert_kernel<D, K>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  dq_convert_kernel<D, K><<<grid, 256, kSmem, stream>>>(dqacc, dq, scale, B, S, H, causal, status,
                                                        wait_ns);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const float *dqacc, __nv_bfloat16 *dq, float scale, int B, int S,
                              int H, int D, int strands, int causal, uint32_t *status,
                              unsigned long long wait_ns, cudaStream_t stream) {
  const long long tiles = (long long)B * H * ((S + kTile - 1) / kTile);
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int grid = (int)tiles;
  if (D == 64)
    return strands == 2 ? conv_launch<64, 2>(grid, stream, dqacc, dq, scale, B, S, H, causal, status, wait_ns)
                        : conv_launch<64, 1>(grid, stream, dqacc, dq, scale, B, S, H, causal, status, wait_ns);
  return strands == 2 ? conv_launch<128, 2>(grid, stream, dqacc, dq, scale, B, S, H, causal, status, wait_ns)
                      : conv_launch<128, 1>(grid, stream, dqacc, dq, scale, B, S, H, causal, status, wait_ns);
}

cudaError_t launch_varlen_setup(const VarlenTable &t, int4 *seqs, int *wprefix,
                                cudaStream_t stream) {
  varlen_setup_kernel<<<1, 256, 0, stream>>>(t, seqs, wprefix);
  return cudaGetLastError();
}

cudaError_t launch_preprocess_varlen(const __nv_bfloat16 *o, const __nv_bfloat16 *dout,
                                     const float *lse, float *dvec, float *lse2, const int4 *seqs,
                                     int batch, int T, int H, int D, uint32_t *status,
                                     unsigned long long wait_ns, cudaStream_t stream) {
  const int grid = pre_grid((long long)T * H, D);
  if (D == 64)
    preprocess_varlen_kernel<64><<<grid, 256, 0, stream>>>(o, dout, lse, dvec, lse2, seqs, batch,
                                                           T, H, status, wait_ns);
  else
    preprocess_varlen_kernel<128><<<grid, 256, 0, stream>>>(o, dout, lse, dvec, lse2, seqs, batch,
                                                            T, H, status, wait_ns);
  return cudaGetLastError();
}

template <int D, int K>
cudaError_t conv_varlen_launch(int ntiles, cudaStream_t stream, const float *dqacc,
                               __nv_bfloat16 *dq, float scale, const int4 *seqs, int batch, int H,
                               int causal, uint32_t *status, unsigned long long wait_ns) {
  constexpr int kSmem = conv_smem_bytes<D, K>();
  cudaError_t e = cudaFuncSetAttribute(dq_convert_varlen_kernel<D, K>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  dq_convert_varlen_kernel<D, K><<<ntiles, 256, kSmem, stream>>>(dqacc, dq, scale, seqs, batch, H,
                                                                 causal, status, wait_ns);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert_varlen(const float *dqacc, __nv_bfloat16 *dq, float scale,
                                     const int4 *seqs, int batch, int ntiles, int H, int D,
                                     int strands, int causal, uint32_t *status,
                                     unsigned long long wait_ns, cudaStream_t stream) {
  if (ntiles <= 0) return cudaSuccess;
  if (D == 64)
    return strands == 2 ? conv_varlen_launch<64, 2>(ntiles, stream, dqacc, dq, scale, seqs, batch, H, causal, status, wait_ns)
                        : conv_varlen_launch<64, 1>(ntiles, stream, dqacc, dq, scale, seqs, batch, H, causal, status, wait_ns);
  return strands == 2 ? conv_varlen_launch<128, 2>(ntiles, stream, dqacc, dq, scale, seqs, batch, H, causal, status, wait_ns)
                      : conv_varlen_launch<128, 1>(ntiles, stream, dqacc, dq, scale, seqs, batch, H, causal, status, wait_ns);
}

}  // namespace dash
