// fwd.cu -- attention forward producing O (bf16) and LSE (fp32, natural log): the inputs
// the backward consumes.  One CTA per (batch, head, 128-row query tile).
//
// Two passes over the visible KV blocks, both on the tcgen05 tensor cores:
//   pass 1:  S = Q_i K_j^T (TMEM), running row max / row sum of exp2 -> LSE_i
//   pass 2:  S = Q_i K_j^T again, P = exp2(S*scale*log2e - LSE_i*log2e) (exactly
//            normalised, bf16 into TMEM over S), O_i += P V_j with P as the TMEM A operand.
// Recomputing S costs one extra Q K^T product per tile but needs no rescaling of the O
// accumulator.  The forward is support for the backward and is not part of its timing.
//
// Warp roles (256 threads): warp 0 TMA producer, warp 1 MMA issuer, warp 2 TMEM
// allocation, warps 4-7 softmax + epilogue (thread = query row = TMEM lane).
// TMEM columns: S buffers [0,128) and [128,256), O [256, 256+D).
#include "common.cuh"
#include "ptx.cuh"

namespace dash {
namespace {

template <int D>
struct FwdLayout {
  static constexpr int kStages = 2;
  static constexpr int kTileBytes = D * kTile * 2;
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kStageBytes = 2 * kTileBytes;  // K_j then V_j
  static constexpr int offQ = 0;
  static constexpr int offStage = kTileBytes;
  static constexpr int offBar = offStage + kStages * kStageBytes;
  // q_full, kv_full[S], kv_empty[S], s_full[2], s_free[2], o_full, drain
  static constexpr int kNumBars = 1 + 2 * kStages + 4 + 2;
  static constexpr int offMisc = offBar + kNumBars * 8;
  static constexpr int kBytes = offMisc + 16;
  static constexpr uint32_t tS = 0, tO = 256;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kBytes <= 232448, "shared memory budget");
};

template <int D>
struct FBars {
  uint64_t *q_full, *kv_full, *kv_empty, *s_full, *s_free, *o_full, *drain;
  __device__ explicit FBars(uint8_t *smem) {
    using L = FwdLayout<D>;
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + L::offBar);
    q_full = b;
    kv_full = b + 1;
    kv_empty = b + 1 + L::kStages;
    s_full = b + 1 + 2 * L::kStages;
    s_free = s_full + 2;
    o_full = s_free + 2;
    drain = o_full + 1;
  }
};

template <int D>
__global__ void __launch_bounds__(256, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = FwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, kErrSmemAlign);
    return;
  }
  const FBars<D> bar(smem);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + L::offMisc);
  int *s_abort = reinterpret_cast<int *>(smem + L::offMisc + 4);
  const Abort ab{s_abort, p.status, p.wait_ns};
  const int warp = warp_id(), lane = lane_id();

  // heaviest causal tiles first
  const int i = p.N - 1 - (int)(blockIdx.x % p.N);
  const int bh = blockIdx.x / p.N;
  const int h = bh % p.H, b = bh / p.H;
  const int hkv = h / p.G;
  const int nkv = p.causal ? i + 1 : p.N;
  const int T = 2 * nkv;  // pass 1 then pass 2

  if (threadIdx.x == 0) {
    mbar_init(bar.q_full, 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&bar.kv_full[s], 1);
      mbar_init(&bar.kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar.s_full[s], 1);
      mbar_init(&bar.s_free[s], 4);
    }
    mbar_init(bar.o_full, 1);
    mbar_init(bar.drain, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 2) {
    tmem_alloc(s_tmem, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer
    int last[L::kStages];
    for (int s = 0; s < L::kStages; ++s) last[s] = -1;
    bool ok = true;
    mbar_arrive_expect_tx(bar.q_full, L::kTileBytes);
    for (int bx = 0; bx < L::kBoxes; ++bx)
      tma_load_4d(smem + L::offQ + bx * kBoxBytes, &tm_q, bar.q_full, bx * kBoxCols, h,
                  i * kTile, b);
    for (int n = 0; n < T; ++n) {
      const int s = n % L::kStages;
      const uint32_t ph = (n / L::kStages) & 1;
      if (!mbar_wait(&bar.kv_empty[s], ph ^ 1, ab)) {
        ok = false;
        break;
      }
      const bool pass2 = n >= nkv;
      const int j = pass2 ? n - nkv : n;
      mbar_arrive_expect_tx(&bar.kv_full[s], pass2 ? 2 * L::kTileBytes : L::kTileBytes);
      uint8_t *sk = smem + L::offStage + s * L::kStageBytes;
      for (int bx = 0; bx < L::kBoxes; ++bx) {
        tma_load_4d(sk + bx * kBoxBytes, &tm_k, &bar.kv_full[s], bx * kBoxCols, hkv,
                    j * kTile, b);
        if (pass2)
          tma_load_4d(sk + L::kTileBytes + bx * kBoxBytes, &tm_v, &bar.kv_full[s],
                      bx * kBoxCols, hkv, j * kTile, b);
      }
      last[s] = (int)ph;
    }
    if (!ok) {
      mbar_wait_drain(bar.q_full, 0, 100000000ull);
      for (int s = 0; s < L::kStages; ++s)
        if (last[s] >= 0) mbar_wait_drain(&bar.kv_full[s], (uint32_t)last[s], 100000000ull);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdescS = make_idesc_bf16(128, 128, false, false);
    constexpr uint32_t kIdescO = make_idesc_bf16(128, D, false, true);
    const uint32_t sbase = smem_u32(smem);
    bool ok = mbar_wait(bar.q_full, 0, ab);
    tc_fence_after();
    // O += P_m V_m, P_m in S buffer (m & 1), packed bf16x2 in its first 64 columns
    auto issue_pv = [&](int m) -> bool {
      const int bm = m & 1, sm = m % L::kStages;
      if (!mbar_wait(&bar.s_free[bm], (m >> 1) & 1, ab)) return false;
      tc_fence_after();
      const uint32_t aV = sbase + L::offStage + sm * L::kStageBytes + L::kTileBytes;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma_ts(tmem + L::tO, tmem + L::tS + bm * 128 + 8 * k,
               make_sdesc_sw128(aV + k * 2048, kBoxBytes, 1024), kIdescO,
               (m > nkv || k > 0) ? 1u : 0u);
      mma_commit(&bar.kv_empty[sm]);
      return true;
    };
    for (int n = 0; ok && n < T; ++n) {
      const int s = n % L::kStages;
      const int buf = n & 1;
      if (!mbar_wait(&bar.kv_full[s], (n / L::kStages) & 1, ab)) {
        ok = false;
        break;
      }
      if (n >= 2 && !mbar_wait(&bar.s_free[buf], ((n - 2) >> 1) & 1, ab)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t aK = sbase + L::offStage + s * L::kStageBytes;
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t koff = (k >> 2) * kBoxBytes + (k & 3) * 32;
        mma_ss(tmem + L::tS + buf * 128, make_sdesc_sw128(sbase + L::offQ + koff, 16, 1024),
               make_sdesc_sw128(aK + koff, 16, 1024), kIdescS, k > 0);
      }
      mma_commit(&bar.s_full[buf]);
      if (n < nkv) {
        mma_commit(&bar.kv_empty[s]);
      } else if (n > nkv) {
        if (!issue_pv(n - 1)) ok = false;
      }
    }
    if (ok && issue_pv(T - 1)) mma_commit(bar.o_full);
    mma_commit(bar.drain);
    mbar_wait_drain(bar.drain, 0, 100000000ull);
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax + epilogue
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // query row within the tile
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    float m2 = -INFINITY, l = 0.f, lse2 = 0.f;
    bool ok = true;
    for (int n = 0; n < T; ++n) {
      const int buf = n & 1;
      if (!mbar_wait_warp(&bar.s_full[buf], (n >> 1) & 1, ab)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool pass2 = n >= nkv;
      const int j = pass2 ? n - nkv : n;
      const bool diag = p.causal && (j == i);
      const int kv_valid = p.S - j * kTile;  // keys of block j inside S (< 128: last tile)
      const uint32_t tsb = tmem + lane_off + L::tS + buf * 128;
      if (!pass2) {
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t sv[32];
          tmem_ld32(tsb + ch * 32, sv);
          tmem_ld_wait();
          float mx = -INFINITY;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const bool masked = (diag && (ch * 32 + c) > r) || (ch * 32 + c) >= kv_valid;
            const float x = masked ? -INFINITY : __uint_as_float(sv[c]) * p.scale_log2;
            sv[c] = __float_as_uint(x);
            mx = fmaxf(mx, x);
          }
          const float mnew = fmaxf(m2, mx);
          if (mnew != -INFINITY) {
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < 32; ++c) acc += ex2_approx(__uint_as_float(sv[c]) - mnew);
            l = l * ex2_approx(m2 - mnew) + acc;
            m2 = mnew;
          }
        }
      } else {
        if (n == nkv) lse2 = m2 + __log2f(l);
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t sv[32], pk[16];
          tmem_ld32(tsb + ch * 32, sv);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float p0 = ex2_approx(fmaf(__uint_as_float(sv[c]), p.scale_log2, -lse2));
            float p1 = ex2_approx(fmaf(__uint_as_float(sv[c + 1]), p.scale_log2, -lse2));
            if ((diag && (ch * 32 + c) > r) || (ch * 32 + c) >= kv_valid) p0 = 0.f;
            if ((diag && (ch * 32 + c + 1) > r) || (ch * 32 + c + 1) >= kv_valid) p1 = 0.f;
            pk[c / 2] = pack_bf16(p0, p1);
          }
          tmem_st16(tsb + ch * 16, pk);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.s_free[buf]);
    }
    if (ok && mbar_wait_warp(bar.o_full, 0, ab)) {
      tc_fence_after();
      const bool row_ok = i * kTile + r < p.S;  // rows past S (partial last tile): no output
      const size_t orow = ((size_t)(b * p.S + i * kTile + r) * p.H + h) * D;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t ov[32], pk[16];
        tmem_ld32(tmem + lane_off + L::tO + ch * 32, ov);
        tmem_ld_wait();
#pragma unroll
        for (int m = 0; m < 16; ++m)
          pk[m] = pack_bf16(__uint_as_float(ov[2 * m]), __uint_as_float(ov[2 * m + 1]));
        uint4 *dst = reinterpret_cast<uint4 *>(p.o + orow + ch * 32);
        if (row_ok) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            dst[q4] = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
        }
      }
      if (row_ok) p.lse[(size_t)(b * p.H + h) * p.S + i * kTile + r] = lse2 * kLn2;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int D>
cudaError_t launch_fwd_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         const FwdParams &p, cudaStream_t stream) {
  using L = FwdLayout<D>;
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       L::kBytes);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)p.B * p.H * p.N;
  fwd_kernel<D><<<grid, 256, L::kBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

size_t fwd_smem_bytes(int D) {
  return D == 64 ? FwdLayout<64>::kBytes : FwdLayout<128>::kBytes;
}

cudaError_t launch_fwd(int D, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const FwdParams &p, cudaStream_t stream) {
  return D == 64 ? launch_fwd_t<64>(tq, tk, tv, p, stream)
                 : launch_fwd_t<128>(tq, tk, tv, p, stream);
}

}  // namespace dash
