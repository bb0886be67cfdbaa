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

namespace dash {
namespace {

// sum_d o[d] * dout[d] over one D-element row, by one warp (every lane gets the sum).
template <int D>
__device__ __forceinline__ float row_dot(const __nv_bfloat16 *__restrict__ o,
                                         const __nv_bfloat16 *__restrict__ dout, int lane) {
  constexpr int kPer = D / 32;  // bf16 elements per lane (2 or 4)
  const __nv_bfloat16 *po = o + lane * kPer;
  const __nv_bfloat16 *pd = dout + lane * kPer;
  float acc = 0.f;
  if constexpr (kPer == 4) {
    const uint2 a = *reinterpret_cast<const uint2 *>(po);
    const uint2 c = *reinterpret_cast<const uint2 *>(pd);
    const __nv_bfloat162 *a2 = reinterpret_cast<const __nv_bfloat162 *>(&a);
    const __nv_bfloat162 *c2 = reinterpret_cast<const __nv_bfloat162 *>(&c);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float2 x = __bfloat1622float2(a2[e]), y = __bfloat1622float2(c2[e]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
  } else {
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(po));
    const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(pd));
    acc = fmaf(x.x, y.x, acc);
    acc = fmaf(x.y, y.y, acc);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  return acc;
}

// One warp per (b, i, h) row; rows enumerated in BSHD order so the O/dO reads of a CTA are
// one contiguous range.
template <int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const __nv_bfloat16 *__restrict__ o,
                                                         const __nv_bfloat16 *__restrict__ dout,
                                                         const float *__restrict__ lse,
                                                         float *__restrict__ dvec,
                                                         float *__restrict__ lse2, int B, int S,
                                                         int H) {
  const long long rows = (long long)B * S * H;
  const int lane = threadIdx.x & 31;
  for (long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); row < rows;
       row += (long long)gridDim.x * 8) {
    const float acc = row_dot<D>(o + row * D, dout + row * D, lane);
    if (lane == 0) {
      const int h = (int)(row % H);
      const long long bi = row / H;
      const int i = (int)(bi % S);
      const int b = (int)(bi / S);
      const size_t Sp = (size_t)(S + kTile - 1) / kTile * kTile;
      const size_t r = ((size_t)b * H + h) * Sp + i;
      dvec[r] = acc;
      lse2[r] = lse[((size_t)b * H + h) * S + i] * kLog2e;
    }
  }
}

// One thread per 4 output elements; the 4-column chunk index runs fastest so a warp
// writes contiguous bf16 rows.  dQacc layout: [B,H,N][K][D/4][128][4], K strands.
template <int D, int K>
__global__ void __launch_bounds__(256) dq_convert_kernel(const float *__restrict__ acc,
                                                         __nv_bfloat16 *__restrict__ dq,
                                                         float scale, int B, int S, int H,
                                                         int causal) {
  constexpr int C4 = D / 4;
  const int N = (S + kTile - 1) / kTile;
  const long long total = (long long)B * H * N * kTile * C4;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int c4 = (int)(idx % C4);
    const int r = (int)((idx / C4) % kTile);
    const long long t = idx / ((long long)C4 * kTile);  // (b*H + h)*N + i
    const int i = (int)(t % N);
    const long long bh = t / N;
    const int h = (int)(bh % H);
    const int b = (int)(bh / H);
    if (i * kTile + r >= S) continue;  // padding rows of a partial last tile
    const float *tb = acc + t * K * (C4 * kTile * 4);
    float4 v = *reinterpret_cast<const float4 *>(tb + ((size_t)c4 * kTile + r) * 4);
    if constexpr (K == 2) {  // strand 0 + strand 1 (when the tile has a second partial)
      if ((causal ? i + 1 : N) > 1) {
        const float4 w = *reinterpret_cast<const float4 *>(tb + ((size_t)(C4 + c4) * kTile + r) * 4);
        v = make_float4(v.x + w.x, v.y + w.y, v.z + w.z, v.w + w.w);
      }
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x * scale, v.y * scale);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z * scale, v.w * scale);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t *>(&lo);
    packed.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(dq + (((size_t)b * S + (size_t)i * kTile + r) * H + h) * D +
                               4 * c4) = packed;
  }
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

// One warp per packed (t, h) row, as preprocess_kernel.
template <int D>
__global__ void __launch_bounds__(256) preprocess_varlen_kernel(
    const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
    const float *__restrict__ lse, float *__restrict__ dvec, float *__restrict__ lse2,
    const int4 *__restrict__ seqs, int batch, int T, int H) {
  const long long rows = (long long)T * H;
  const int lane = threadIdx.x & 31;
  for (long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); row < rows;
       row += (long long)gridDim.x * 8) {
    const float acc = row_dot<D>(o + row * D, dout + row * D, lane);
    if (lane == 0) {
      const int h = (int)(row % H);
      const int t = (int)(row / H);
      const int4 sq = seqs[seq_of_token(seqs, batch, t)];
      const int i = t - sq.y;
      const size_t r = ((size_t)sq.z + (size_t)h * sq.w) * kTile + i;
      dvec[r] = acc;
      lse2[r] = lse[(size_t)sq.y * H + (size_t)h * sq.x + i] * kLog2e;
    }
  }
}

// One thread per 4 output elements of a packed (t, h) row, the chunk index fastest.
template <int D, int K>
__global__ void __launch_bounds__(256) dq_convert_varlen_kernel(
    const float *__restrict__ acc, __nv_bfloat16 *__restrict__ dq, float scale,
    const int4 *__restrict__ seqs, int batch, int T, int H, int causal) {
  constexpr int C4 = D / 4;
  const long long total = (long long)T * H * C4;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int c4 = (int)(idx % C4);
    const long long row = idx / C4;
    const int h = (int)(row % H);
    const int t = (int)(row / H);
    const int4 sq = seqs[seq_of_token(seqs, batch, t)];
    const int i = t - sq.y;
    const size_t tile = (size_t)sq.z + (size_t)h * sq.w + i / kTile;
    const int r = i % kTile;
    const float *tb = acc + tile * K * (C4 * kTile * 4);
    float4 v = *reinterpret_cast<const float4 *>(tb + ((size_t)c4 * kTile + r) * 4);
    if constexpr (K == 2) {
      if ((causal ? i / kTile + 1 : sq.w) > 1) {
        const float4 w = *reinterpret_cast<const float4 *>(tb + ((size_t)(C4 + c4) * kTile + r) * 4);
        v = make_float4(v.x + w.x, v.y + w.y, v.z + w.z, v.w + w.w);
      }
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x * scale, v.y * scale);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z * scale, v.w * scale);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t *>(&lo);
    packed.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(dq + row * D + 4 * c4) = packed;
  }
}

int grid_for(long long work, int per_block, int cap) {
  long long g = (work + per_block - 1) / per_block;
  if (g < 1) g = 1;
  return (int)(g > cap ? cap : g);
}

}  // namespace

cudaError_t launch_preprocess(const __nv_bfloat16 *o, const __nv_bfloat16 *dout, const float *lse,
                              float *dvec, float *lse2, int B, int S, int H, int D,
                              cudaStream_t stream) {
  const long long rows = (long long)B * S * H;
  const int grid = grid_for(rows, 8, 152 * 16);
  if (D == 64)
    preprocess_kernel<64><<<grid, 256, 0, stream>>>(o, dout, lse, dvec, lse2, B, S, H);
  else
    preprocess_kernel<128><<<grid, 256, 0, stream>>>(o, dout, lse, dvec, lse2, B, S, H);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const float *dqacc, __nv_bfloat16 *dq, float scale, int B, int S,
                              int H, int D, int strands, int causal, cudaStream_t stream) {
  const long long work = (long long)B * H * ((S + kTile - 1) / kTile) * kTile * (D / 4);
  const int grid = grid_for(work, 256, 152 * 32);
  if (D == 64) {
    if (strands == 2)
      dq_convert_kernel<64, 2><<<grid, 256, 0, stream>>>(dqacc, dq, scale, B, S, H, causal);
    else
      dq_convert_kernel<64, 1><<<grid, 256, 0, stream>>>(dqacc, dq, scale, B, S, H, causal);
  } else {
    if (strands == 2)
      dq_convert_kernel<128, 2><<<grid, 256, 0, stream>>>(dqacc, dq, scale, B, S, H, causal);
    else
      dq_convert_kernel<128, 1><<<grid, 256, 0, stream>>>(dqacc, dq, scale, B, S, H, causal);
  }
  return cudaGetLastError();
}

cudaError_t launch_varlen_setup(const VarlenTable &t, int4 *seqs, int *wprefix,
                                cudaStream_t stream) {
  varlen_setup_kernel<<<1, 256, 0, stream>>>(t, seqs, wprefix);
  return cudaGetLastError();
}

cudaError_t launch_preprocess_varlen(const __nv_bfloat16 *o, const __nv_bfloat16 *dout,
                                     const float *lse, float *dvec, float *lse2, const int4 *seqs,
                                     int batch, int T, int H, int D, cudaStream_t stream) {
  const long long rows = (long long)T * H;
  const int grid = grid_for(rows, 8, 152 * 16);
  if (D == 64)
    preprocess_varlen_kernel<64><<<grid, 256, 0, stream>>>(o, dout, lse, dvec, lse2, seqs, batch,
                                                           T, H);
  else
    preprocess_varlen_kernel<128><<<grid, 256, 0, stream>>>(o, dout, lse, dvec, lse2, seqs, batch,
                                                            T, H);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert_varlen(const float *dqacc, __nv_bfloat16 *dq, float scale,
                                     const int4 *seqs, int batch, int T, int H, int D,
                                     int strands, int causal, cudaStream_t stream) {
  const long long work = (long long)T * H * (D / 4);
  const int grid = grid_for(work, 256, 152 * 32);
  if (D == 64) {
    if (strands == 2)
      dq_convert_varlen_kernel<64, 2><<<grid, 256, 0, stream>>>(dqacc, dq, scale, seqs, batch, T, H, causal);
    else
      dq_convert_varlen_kernel<64, 1><<<grid, 256, 0, stream>>>(dqacc, dq, scale, seqs, batch, T, H, causal);
  } else {
    if (strands == 2)
      dq_convert_varlen_kernel<128, 2><<<grid, 256, 0, stream>>>(dqacc, dq, scale, seqs, batch, T,
                                                                 H, causal);
    else
      dq_convert_varlen_kernel<128, 1><<<grid, 256, 0, stream>>>(dqacc, dq, scale, seqs, batch, T,
                                                                 H, causal);
  }
  return cudaGetLastError();
}

}  // namespace dash
