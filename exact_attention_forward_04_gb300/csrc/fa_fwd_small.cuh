// Exact attention forward for short sequences (N <= 128) on sm_103a: one
// CTA of 128 threads per (batch, head), no cluster and no persistence.
//
// The whole row fits one block of keys, so the online-softmax recurrence
// ("Before implementing FlashAttention in Triton: FA1, 2 forward pass", FA2
// section) collapses to its first step: the row maximum m is exact, P~ =
// 2^(s c - m) <= 1 and a single divide by l = sum P~ normalises O.  The
// long-sequence kernel (CTA pairs, 256-row units) would spend most of a
// 128-token head on launching a two-SM cluster and setting it up; this one
// loads Q, K and V once and runs two single-SM tcgen05 products:
//   S = Q K^T      TMEM [0,128)      (M = 128 query rows, N = 128 keys)
//   P~             bf16 pairs over S's columns [0,64), one thread per row
//   O~ = P~ V      TMEM [128,128+d)  (A from TMEM, B = V MN-major)
// then O = O~ / l (bf16) and L = (m + log2 l) ln 2 are stored directly.
// Keys >= N (zero-filled by the TMA) and, under the causal mask, keys right
// of the row are excluded before the maximum.  A negative scale negates the
// S product's A operand (Q), as in the long-sequence kernel.
#pragma once
#include <cuda_bf16.h>

#include "sm103_ptx.cuh"
#include "tmem_ldst.cuh"

namespace fa {
namespace small {

constexpr int kRows = 128;      // query rows and keys of the one block
constexpr int kThreads = 128;   // one thread per row
constexpr uint32_t kColS = 0, kColO = 128;

enum : unsigned { kSiteLoad = 301, kSiteS = 302, kSitePV = 303 };

template <int D>
struct Layout {
  static constexpr int kTile = kRows * D * 2;  // 128 rows x D bf16
  static constexpr int kQ = 0;
  static constexpr int kK = kTile;
  static constexpr int kV = 2 * kTile;
  static constexpr int kMisc = 3 * kTile;
  static constexpr int kBarLoad = kMisc;
  static constexpr int kBarMma = kBarLoad + 8;
  static constexpr int kTmemSlot = kBarMma + 8;
  static constexpr int kAbort = kTmemSlot + 8;
  static constexpr int kBytes = kAbort + 8;
  static constexpr int kAlloc = kBytes + 1024;  // 1024-byte alignment slack
};

// K-major 128B-swizzled 128-row tile: the K step kk within a 64-column atom
// is +32 bytes, the next atom +16 KB.
__device__ __forceinline__ uint32_t kstep(int kk) {
  return static_cast<uint32_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
}

}  // namespace small

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(small::kThreads, 1)
    fa_fwd_small_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O,
                        float* __restrict__ Lse, DevError* __restrict__ err, int N, float c_log2,
                        int negate_s, unsigned long long timeout_ns) {
  using namespace small;
  using Ly = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int bh = static_cast<int>(blockIdx.x);

  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + Ly::kAbort);
  const uint32_t bar_load = base + Ly::kBarLoad, bar_mma = base + Ly::kBarMma;
  if (tid == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(base + Ly::kTmemSlot, 256);
    tmem_relinquish();
  }
  if (tid == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + Ly::kTmemSlot);
  const WaitCtx wc{abort_flag, err, timeout_ns};

  // Q, K and V of the head: rows >= N read as zeros
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_load, 3 * Ly::kTile);
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      tma_load_3d(base + Ly::kQ + c * 16384, &tmQ, bar_load, c * 64, 0, bh);
      tma_load_3d(base + Ly::kK + c * 16384, &tmK, bar_load, c * 64, 0, bh);
      tma_load_3d(base + Ly::kV + c * 16384, &tmV, bar_load, c * 64, 0, bh);
    }
    if (mbar_wait(bar_load, 0, wc, kSiteLoad, bh)) {
      tc_fence_after();
      const uint32_t idS =
          idesc_bf16_f32_ab(kRows, kRows, false, false) | (negate_s ? kIdescNegateA : 0u);
      const uint64_t dQ = sw128_desc(base + Ly::kQ, 16, 1024);
      const uint64_t dK = sw128_desc(base + Ly::kK, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(tmem + kColS, dQ + kstep(kk), dK + kstep(kk), idS, kk > 0 ? 1u : 0u);
    }
    tc_commit(bar_mma);  // also when the wait gave up: the others then stop waiting
  }

  // ---- softmax: thread = query row = TMEM lane
  const int r = tid;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  bool ok = mbar_wait(bar_mma, 0, wc, kSiteS, bh);
  ok = __all_sync(0xffffffffu, ok && *abort_flag == 0);
  float m = 0.f, l = 1.f;
  if (ok) {
    tc_fence_after();
    uint32_t s[4][32];
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_off + kColS + 32 * c, s[c]);
    tmem_ld_wait32(s[0]);
    tmem_ld_dep32(s[1]);
    tmem_ld_dep32(s[2]);
    tmem_ld_dep32(s[3]);
    // visible keys: k < N and, causal, k <= r (row r >= N is never stored)
    const int lim = CAUSAL ? (r < N - 1 ? r : N - 1) : N - 1;
    m = -INFINITY;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float x = 32 * c + e <= lim ? __uint_as_float(s[c][e]) * c_log2 : -INFINITY;
        s[c][e] = __float_as_uint(x);
        m = fmaxf(m, x);
      }
    // key 0 is visible to every row, so m is finite
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t w[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        const float p0 = ex2(__uint_as_float(s[c][e]) - m);
        const float p1 = ex2(__uint_as_float(s[c][e + 1]) - m);
        sum += p0 + p1;
        w[e >> 1] = pack_bf16(p0, p1);
      }
      tmem_st16(tmem + lane_off + kColS + 16 * c, w);  // over S columns already read
    }
    l = sum;
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();  // P~ of every row is in TMEM

  if (tid == 0) {
    if (*abort_flag == 0) {
      tc_fence_after();
      const uint32_t idPV = idesc_bf16_f32_ab(kRows, D, false, true);
      const uint64_t dV = sw128_desc(base + Ly::kV, 16384, 1024);
#pragma unroll
      for (int kk = 0; kk < kRows / 16; ++kk)
        mma_ts(tmem + kColO, tmem + kColS + 8 * kk, dV + static_cast<uint32_t>(kk * 128), idPV,
               kk > 0 ? 1u : 0u);
    }
    tc_commit(bar_mma);
  }
  ok = mbar_wait(bar_mma, 1, wc, kSitePV, bh);
  ok = __all_sync(0xffffffffu, ok && *abort_flag == 0);
  if (ok) {
    tc_fence_after();
    const float inv = 1.0f / l;
    __nv_bfloat16* out = O + (static_cast<size_t>(bh) * N + r) * D;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_off + kColO + 32 * c, v);
      tmem_ld_wait32(v);
      if (r < N) {
        uint4* dst = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
        for (int t = 0; t < 4; ++t)
          dst[t] = make_uint4(
              pack_bf16(__uint_as_float(v[8 * t]) * inv, __uint_as_float(v[8 * t + 1]) * inv),
              pack_bf16(__uint_as_float(v[8 * t + 2]) * inv, __uint_as_float(v[8 * t + 3]) * inv),
              pack_bf16(__uint_as_float(v[8 * t + 4]) * inv, __uint_as_float(v[8 * t + 5]) * inv),
              pack_bf16(__uint_as_float(v[8 * t + 6]) * inv, __uint_as_float(v[8 * t + 7]) * inv));
      }
    }
    if (r < N) Lse[static_cast<size_t>(bh) * N + r] = (m + log2f(l)) * 0.6931471805599453f;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace fa
