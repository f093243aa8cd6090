// Standard (unfused) attention on sm_103a: the three-step computation that
// the fused forward replaces, kept as the IO-awareness measurement beside it
// ("How FlashAttention got past the O(N^2) memory wall", "The
// standard-attention bottleneck: O(N^2) HBM round trips", Steps 1-4;
// "Before implementing FlashAttention in Triton: FA1, 2 forward pass", "Why
// it is needed": S = Q K^T, P = softmax(S), O = P V, each written to HBM and
// read back by the next step).
//
//   fa_unf_s_kernel        S = scale Q K^T, fp32 [B*H, N, Np] in HBM.  One CTA
//                          per 128-row x 256-key tile: TMA loads of Q and K,
//                          one tcgen05 GEMM (M 128, N 256, K = d) into TMEM,
//                          an epilogue that stages 32-column slices in the
//                          freed operand memory and writes them by TMA stores.
//   fa_unf_softmax_row_kernel  L = max + ln sum exp(S - max) and P = exp(S - L)
//                          in bf16 [B*H, N, Np], one CTA per row with the row
//                          in registers (S read once), for N <= 16384;
//   fa_unf_softmax_kernel  the same for longer rows, one warp per row in two
//                          passes (an online max/sum, then P).
//   fa_unf_pv_kernel       O = P V in bf16.  One CTA per 128-row tile: a
//                          3-stage TMA ring of 64-key blocks of P and V and
//                          tcgen05 GEMMs (M 128, N = d, K 16) accumulating in
//                          TMEM, then the epilogue.
//
// S is kept in fp32 so that L meets its 1e-3 bound (scores rounded to bf16
// would move L by up to half a bf16 ulp of the row maximum); P is bf16, the
// operand type of the P V product.  Under the causal mask S tiles wholly
// right of a query tile's last row are not computed, the softmax reads only
// each row's visible keys and writes zeros for the masked keys of the row's
// 128-row tile, and the P V product covers only those key blocks.  Np = N
// rounded up to 8 (16-byte rows for both matrices); columns >= N are never
// read (the TMA extents are N).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "sm103_ptx.cuh"
#include "tmem_ldst.cuh"

namespace fa {
namespace unf {

constexpr int kRowsS = 128;    // S tile: query rows
constexpr int kKeysS = 256;    // S tile: keys
constexpr int kThreadsS = 128;
constexpr int kRowsPV = 128;   // P V tile: query rows
constexpr int kKeysPV = 64;    // keys per ring stage (one 128-byte row of P)
constexpr int kStagesPV = 3;
constexpr int kThreadsPV = 192;
// Dynamic shared memory of both GEMM kernels is at least this, so that at
// most two CTAs share an SM and their TMEM (256 columns each) always fits.
constexpr int kMinSmem = 100 * 1024;

enum : unsigned { kSiteUS = 301, kSiteUSMma = 302, kSiteUPLoad = 311, kSiteUPMma = 312,
                  kSiteUPEpi = 313 };

template <int D>
struct LayoutS {
  static constexpr int kQ = 0;                    // D/64 boxes of 128 rows x 128 B
  static constexpr int kK = kRowsS * D * 2;       // D/64 boxes of 256 rows x 128 B
  static constexpr int kMisc = kK + kKeysS * D * 2;
  static constexpr int kBarFull = kMisc;
  static constexpr int kBarMma = kMisc + 8;
  static constexpr int kTmemSlot = kMisc + 16;
  static constexpr int kAbort = kMisc + 24;
  static constexpr int kBytes = kMisc + 32;
  static constexpr int kAlloc = kBytes + 1024 > kMinSmem ? kBytes + 1024 : kMinSmem;
};

template <int D>
struct LayoutPV {
  static constexpr int kStage = kRowsPV * 128 + D * 128;  // P block + D/64 boxes of V (8 KB each)
  static constexpr int kMisc = kStagesPV * kStage;
  static constexpr int kBarFull = kMisc;                   // [kStagesPV]
  static constexpr int kBarEmpty = kBarFull + 8 * kStagesPV;
  static constexpr int kBarDone = kBarEmpty + 8 * kStagesPV;
  static constexpr int kTmemSlot = kBarDone + 8;
  static constexpr int kAbort = kTmemSlot + 8;
  static constexpr int kBytes = kAbort + 8;
  static constexpr int kAlloc = kBytes + 1024 > kMinSmem ? kBytes + 1024 : kMinSmem;
};

__device__ __forceinline__ void drain_wait_local(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) return;
  }
}

}  // namespace unf

// S = scale Q K^T for one 128 x 256 tile.  Grid: B*H x ceil(N/128) x
// ceil(N/256) tiles, key tile fastest.  Warp 0 allocates TMEM; thread 0
// issues the loads and the MMAs; all four warps run the epilogue (warp w:
// rows 32w..32w+31 = TMEM lanes).
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(unf::kThreadsS)
    fa_unf_s_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmS, DevError* __restrict__ err, int N,
                    int n_qt, int n_kt, float scale, unsigned long long timeout_ns) {
  using namespace unf;
  using Ly = LayoutS<D>;
  const long long idx = blockIdx.x;
  const int n = static_cast<int>(idx % n_kt);
  const int t = static_cast<int>((idx / n_kt) % n_qt);
  const int bh = static_cast<int>(idx / (static_cast<long long>(n_kt) * n_qt));
  // causal: a tile whose first key lies right of the tile's last row is never read
  if (CAUSAL && n * kKeysS > t * kRowsS + kRowsS - 1) return;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + Ly::kAbort);
  const uint32_t bar_full = base + Ly::kBarFull, bar_mma = base + Ly::kBarMma;
  if (tid == 0) {
    mbar_init(bar_full, 1);
    mbar_init(bar_mma, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(base + Ly::kTmemSlot, 256);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + Ly::kTmemSlot);
  const WaitCtx wc{abort_flag, err, timeout_ns};
  constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;

  if (tid == 0) {
    mbar_arrive_expect_tx(bar_full, (D / 64) * (kRowsS + kKeysS) * 128);
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      tma_load_3d(base + Ly::kQ + c * kRowsS * 128, &tmQ, bar_full, c * 64, t * kRowsS, bh);
      tma_load_3d(base + Ly::kK + c * kKeysS * 128, &tmK, bar_full, c * 64, n * kKeysS, bh);
    }
    if (mbar_wait(bar_full, 0, wc, kSiteUS, static_cast<unsigned>(idx))) {
      tc_fence_after();
      constexpr uint32_t kIdesc = idesc_bf16_f32(kRowsS, kKeysS, false);
      const uint64_t dQ = sw128_desc(base + Ly::kQ, 16, 1024);
      const uint64_t dK = sw128_desc(base + Ly::kK, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t oq = static_cast<uint32_t>(((kk >> 2) * kRowsS * 128 + (kk & 3) * 32) >> 4);
        const uint32_t ok = static_cast<uint32_t>(((kk >> 2) * kKeysS * 128 + (kk & 3) * 32) >> 4);
        mma_ss(tmem, dQ + oq, dK + ok, kIdesc, kk > 0 ? 1u : 0u);
      }
    } else {
      drain_wait_local(bar_full, 0, kDrainNs);  // copies still in flight must land first
    }
    tc_commit(bar_mma);  // also when no MMA was issued: arrives at once
  }
  // ---- epilogue: TMEM -> registers (x scale) -> 128B-swizzled staging in
  // the operand memory the MMA has finished reading -> TMA store
  const bool ok = mbar_wait(bar_mma, 0, wc, kSiteUSMma, static_cast<unsigned>(idx)) && !*abort_flag;
  tc_fence_after();
  const int row0 = t * kRowsS + warp * 32;
  const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  if (__all_sync(0xffffffffu, ok) && row0 < N) {
#pragma unroll 1
    for (int c = 0; c < kKeysS / 32; ++c) {
      const int col0 = n * kKeysS + c * 32;
      if (col0 >= N) break;
      // causal: columns right of every row of this box are never read
      if (CAUSAL && col0 > row0 + 31) break;
      uint32_t r[32];
      tmem_ld32(tl + c * 32, r);
      tmem_ld_wait32(r);
      const uint32_t stage = base + warp * 8192 + (c & 1) * 4096;
      if (c >= 2) {  // the store that last read this buffer has finished reading
        if (lane == 0) bulk_wait_read_le1();
        __syncwarp();
      }
      uint8_t* rowp = gbase + (stage - base) + lane * 128;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        *reinterpret_cast<float4*>(rowp + ((i ^ (lane & 7)) << 4)) =
            make_float4(__uint_as_float(r[4 * i]) * scale, __uint_as_float(r[4 * i + 1]) * scale,
                        __uint_as_float(r[4 * i + 2]) * scale, __uint_as_float(r[4 * i + 3]) * scale);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&tmS, stage, col0, row0, bh);
        bulk_commit_group();
      }
    }
    if (lane == 0) bulk_wait_all();
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// L and P of one row per warp.  S, P: [B*H*N rows][Np]; L: [B*H*N].
template <bool CAUSAL>
__global__ void __launch_bounds__(256)
    fa_unf_softmax_kernel(const float* __restrict__ S, __nv_bfloat16* __restrict__ P,
                          float* __restrict__ Lse, long long rows, int N, int Np) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int q = static_cast<int>(row % N);
  const int kv = CAUSAL ? q + 1 : N;                                           // visible keys
  const int pend = CAUSAL ? min(N, (q / unf::kRowsPV + 1) * unf::kRowsPV) : N;  // P columns written
  const float* s = S + row * Np;
  constexpr float kLog2e = 1.4426950408889634f;
  // pass 1: online maximum and sum (base 2) of this lane's columns
  float m = -INFINITY, l = 0.f;
  for (int c0 = lane * 4; c0 < kv; c0 += 128) {
    float x[4];
    if (c0 + 4 <= kv) {
      const float4 v4 = *reinterpret_cast<const float4*>(s + c0);
      x[0] = v4.x; x[1] = v4.y; x[2] = v4.z; x[3] = v4.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = c0 + i < kv ? s[c0 + i] : -INFINITY;
    }
    const float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])) * kLog2e;
    if (mx > m) {
      l *= ex2(m - mx);
      m = mx;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) l += ex2(fmaf(x[i], kLog2e, -m));
  }
  // merge the lanes' statistics
  float mw = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, o));
  float lw = m == -INFINITY ? 0.f : l * ex2(m - mw);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
  const float L2 = mw + log2f(lw);  // logsumexp in base-2 units
  if (lane == 0) Lse[row] = L2 * 0.693147180559945309f;
  // pass 2: P = 2^(s log2e - L2) on visible keys, 0 on the rest of the row's tile
  __nv_bfloat16* p = P + row * Np;
  for (int c0 = lane * 8; c0 < pend; c0 += 256) {
    float x[8];
    if (c0 + 8 <= kv) {
      const float4 a = *reinterpret_cast<const float4*>(s + c0);
      const float4 b = *reinterpret_cast<const float4*>(s + c0 + 4);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
      x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = c0 + i < kv ? s[c0 + i] : -INFINITY;
    }
    float e[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) e[i] = ex2(fmaf(x[i], kLog2e, -L2));  // 0 at -inf
    *reinterpret_cast<uint4*>(p + c0) = make_uint4(pack_bf16(e[0], e[1]), pack_bf16(e[2], e[3]),
                                                   pack_bf16(e[4], e[5]), pack_bf16(e[6], e[7]));
  }
}

// L and P of one row per CTA of 256 threads, the row held in registers
// (EPT elements per thread, N <= 256 EPT), so that S is read from memory
// once.  Thread t holds columns 4t + 1024c .. 4t + 1024c + 3 for c < EPT/4.
template <bool CAUSAL, int EPT>
__global__ void __launch_bounds__(256)
    fa_unf_softmax_row_kernel(const float* __restrict__ S, __nv_bfloat16* __restrict__ P,
                              float* __restrict__ Lse, int N, int Np) {
  constexpr int kG = EPT / 4;  // float4 groups per thread
  __shared__ float red[2][8];
  const long long row = blockIdx.x;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int q = static_cast<int>(row % N);
  const int kv = CAUSAL ? q + 1 : N;
  const int pend = CAUSAL ? min(N, (q / unf::kRowsPV + 1) * unf::kRowsPV) : N;
  const float* s = S + row * Np;
  constexpr float kLog2e = 1.4426950408889634f;
  float x[kG][4];
  float mx = -INFINITY;
#pragma unroll
  for (int c = 0; c < kG; ++c) {
    const int c0 = 4 * t + 1024 * c;
    if (c0 + 4 <= kv) {
      const float4 v4 = *reinterpret_cast<const float4*>(s + c0);
      x[c][0] = v4.x; x[c][1] = v4.y; x[c][2] = v4.z; x[c][3] = v4.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) x[c][i] = c0 + i < kv ? s[c0 + i] : -INFINITY;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) mx = fmaxf(mx, x[c][i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red[0][warp] = mx;
  __syncthreads();
  float m = red[0][0];
#pragma unroll
  for (int w = 1; w < 8; ++w) m = fmaxf(m, red[0][w]);
  const float m2 = m * kLog2e;  // finite: every row sees at least one key
  float l = 0.f;
#pragma unroll
  for (int c = 0; c < kG; ++c)
#pragma unroll
    for (int i = 0; i < 4; ++i) l += ex2(fmaf(x[c][i], kLog2e, -m2));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  if (lane == 0) red[1][warp] = l;
  __syncthreads();
  float lt = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) lt += red[1][w];
  const float L2 = m2 + log2f(lt);
  if (t == 0) Lse[row] = L2 * 0.693147180559945309f;
  __nv_bfloat16* p = P + row * Np;
#pragma unroll
  for (int c = 0; c < kG; ++c) {
    const int c0 = 4 * t + 1024 * c;
    if (c0 < pend) {
      float e[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) e[i] = ex2(fmaf(x[c][i], kLog2e, -L2));  // 0 at -inf
      *reinterpret_cast<uint2*>(p + c0) = make_uint2(pack_bf16(e[0], e[1]), pack_bf16(e[2], e[3]));
    }
  }
}

// O = P V for one 128-row tile.  Grid: B*H x ceil(N/128).  Warps: 0 TMA
// producer, 1 MMA issuer and TMEM owner, 2-5 epilogue (warp w: TMEM lanes
// 32 (w % 4) ..).
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(unf::kThreadsPV)
    fa_unf_pv_kernel(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmV,
                     __nv_bfloat16* __restrict__ O, DevError* __restrict__ err, int N, int n_qt,
                     unsigned long long timeout_ns) {
  using namespace unf;
  using Ly = LayoutPV<D>;
  constexpr int S = kStagesPV;
  constexpr uint32_t kCols = D < 32 ? 32 : D;  // TMEM columns (power of two)
  const int t = static_cast<int>(blockIdx.x % n_qt);
  const int bh = static_cast<int>(blockIdx.x / n_qt);
  const int kend = CAUSAL ? min(N, (t + 1) * kRowsPV) : N;  // keys this tile's rows may see
  const int nkb = (kend + kKeysPV - 1) / kKeysPV;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + Ly::kAbort);
  const uint32_t bar_full = base + Ly::kBarFull, bar_empty = base + Ly::kBarEmpty;
  const uint32_t bar_done = base + Ly::kBarDone;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(base + Ly::kTmemSlot, kCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + Ly::kTmemSlot);
  const WaitCtx wc{abort_flag, err, timeout_ns};
  constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
  const unsigned unit = blockIdx.x;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------- producer
    int issued = 0;
    for (int j = 0; j < nkb; ++j) {
      const int st = j % S;
      if (!mbar_wait(bar_empty + 8 * st, ((j / S) & 1) ^ 1u, wc, kSiteUPLoad, unit)) break;
      const uint32_t fb = bar_full + 8 * st;
      const uint32_t dst = base + st * Ly::kStage;
      mbar_arrive_expect_tx(fb, Ly::kStage);
      tma_load_3d(dst, &tmP, fb, j * kKeysPV, t * kRowsPV, bh);  // keys >= N read as 0
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(dst + kRowsPV * 128 + c * 8192, &tmV, fb, c * 64, j * kKeysPV, bh);
      ++issued;
    }
    for (int j = issued - S < 0 ? 0 : issued - S; j < issued; ++j)  // every copy has landed
      unf::drain_wait_local(bar_full + 8 * (j % S), (j / S) & 1, kDrainNs);
  } else if (warp == 1 && lane == 0) {
    // ----------------------------------------------------------- MMA issuer
    constexpr uint32_t kIdesc = idesc_bf16_f32(kRowsPV, D, true);  // B = V, MN-major
    for (int j = 0; j < nkb; ++j) {
      const int st = j % S;
      if (!mbar_wait(bar_full + 8 * st, (j / S) & 1, wc, kSiteUPMma, unit)) break;
      tc_fence_after();
      const uint32_t sb = base + st * Ly::kStage;
      const uint64_t dP = sw128_desc(sb, 16, 1024);                   // K-major, 64 keys per row
      const uint64_t dV = sw128_desc(sb + kRowsPV * 128, 8192, 1024);  // 64-column boxes 8 KB apart
#pragma unroll
      for (int kk = 0; kk < kKeysPV / 16; ++kk)
        mma_ss(tmem, dP + static_cast<uint32_t>(kk * 2), dV + static_cast<uint32_t>(kk * 128), kIdesc,
               (j > 0 || kk > 0) ? 1u : 0u);
      tc_commit(bar_empty + 8 * st);
    }
    tc_commit(bar_done);  // every MMA issued above has completed
    unf::drain_wait_local(bar_done, 0, kDrainNs);
  } else if (warp >= 2) {
    // ------------------------------------------------------------- epilogue
    const bool ok = mbar_wait(bar_done, 0, wc, kSiteUPEpi, unit) && !*abort_flag;
    tc_fence_after();
    const int quarter = warp & 3;
    const int row = t * kRowsPV + quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    if (__all_sync(0xffffffffu, ok)) {
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tl + c * 32, r);
        tmem_ld_wait32(r);
        if (row < N) {
          uint4* dst = reinterpret_cast<uint4*>(O + (static_cast<size_t>(bh) * N + row) * D + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pack_bf16(__uint_as_float(r[8 * i]), __uint_as_float(r[8 * i + 1])),
                                pack_bf16(__uint_as_float(r[8 * i + 2]), __uint_as_float(r[8 * i + 3])),
                                pack_bf16(__uint_as_float(r[8 * i + 4]), __uint_as_float(r[8 * i + 5])),
                                pack_bf16(__uint_as_float(r[8 * i + 6]), __uint_as_float(r[8 * i + 7])));
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

}  // namespace fa
