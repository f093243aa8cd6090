// Attention backward on sm_103a: dQ, dK, dV from Q, K, V, O, dO and the
// forward's logsumexp L, recomputing P blockwise from S and L
// ("Before implementing FlashAttention in Triton: FA1, 2 forward pass", FA2
// section: L alone gives the normalised P back from S; "How FlashAttention
// got past the O(N^2) memory wall", "v2 and v3": the backward keeps only the
// row statistics and recomputes the blocks it needs).
//
//   P = exp(scale S - L),  D_i = sum_t dO_it O_it,  dP = dO V^T,
//   dS = P * (dP - D),  dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K.
//
// Three kernels:
//   fa_bwd_prep_kernel    D_i per row (fp32) and a zeroed fp32 dQ accumulator
//   fa_bwd_kernel         one CTA per (batch*head, 128-key block j); it walks
//                         the 128-row query blocks i (i >= j under the causal
//                         mask) and keeps dK_j and dV_j in tensor memory
//   fa_bwd_dq_kernel      dQ = bf16(scale * accumulator)
//
// fa_bwd_kernel, per query block (tcgen05, single-SM MMAs, M = 128):
//   S^T  = K_j Q_i^T         TMEM [0,128)     (keys x queries, fp32)
//   dP^T = V_j dO_i^T        TMEM [128,256)
//   compute warps (two groups, queries 0-63 and 64-127): P^T = exp2(S^T c -
//   L log2 e) masked, written back as bf16 over the group's own S^T columns
//   (queries 0-63 at columns 0-31, 64-127 at 64-95); dS^T = P^T (dP^T - D)
//   as bf16 into shared memory (128B-swizzled, keys as rows)
//   dV_j += P^T dO_i         TMEM [256,256+d)  (A from TMEM)
//   dK_j += dS^T Q_i         TMEM [256+d,256+2d)
//   dQ_i  = dS K_j           TMEM [128,128+d)  (A = the dS^T buffer read
//                                              transposed, MN-major)
//   dQ warps stage dQ_i in the Q/dO ring stage the step has finished with
//   (128B-swizzled fp32 boxes) and add it into the fp32 accumulator with TMA
//   bulk reduce-adds; the stage goes back to the producer once the TMA has
//   read it.
// Warps: 0 TMA producer, 1 MMA issuer and TMEM owner, 4-7 and 12-15 compute
// (one key row per thread, one query half per group), 8-11 dQ (one query row
// per thread; at the end dK and dV, one key row per thread), 2-3 idle.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sm103_ptx.cuh"
#include "tmem_ldst.cuh"

namespace fa {
namespace bwd {

constexpr int kBlk = 128;       // keys per CTA, queries per step
constexpr int kThreads = 512;   // 16 warps
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256;

enum : unsigned {
  kSiteBLoad = 211, kSiteBMmaQ = 212, kSiteBMmaFree = 213, kSiteBMmaDS = 214,
  kSiteBSoftS = 221, kSiteBSoftDQ = 222, kSiteBDq = 231, kSiteBKV = 232
};

template <int D>
struct Layout {
  static constexpr int kTile = kBlk * D * 2;                 // 128 rows x D bf16
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  static constexpr int kQ = 2 * kTile;                       // [2] stages
  static constexpr int kDO = 4 * kTile;                      // [2] stages
  static constexpr int kDS = 6 * kTile;                      // 128 x 128 bf16
  static constexpr int kMisc = kDS + kBlk * kBlk * 2;
  static constexpr int kBarKV = kMisc;
  static constexpr int kBarQFull = kBarKV + 8;               // [2]
  static constexpr int kBarQEmpty = kBarQFull + 16;          // [2]
  static constexpr int kBarS = kBarQEmpty + 16;
  static constexpr int kBarDP = kBarS + 8;
  static constexpr int kBarP = kBarDP + 8;
  static constexpr int kBarDS = kBarP + 8;
  static constexpr int kBarDQ = kBarDS + 8;
  static constexpr int kBarDQFree = kBarDQ + 8;
  static constexpr int kBarFin = kBarDQFree + 8;
  static constexpr int kTmemSlot = kBarFin + 8;
  static constexpr int kAbort = kTmemSlot + 8;
  static constexpr int kBytes = kAbort + 8;
  static constexpr int kAlloc = kBytes + 1024;               // 1024-byte alignment slack
};

// K-major 128B-swizzled tile (TMA boxes of 64 columns): the K step kk (16
// elements) within a 64-column atom is +32 bytes, the next atom +16 KB.
__device__ __forceinline__ uint32_t kstep_kmajor(int kk) {
  return static_cast<uint32_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
}

// Bounded wait for the final commit before TMEM is released (CTA scope).
__device__ __forceinline__ void drain_wait_cta(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) return;
  }
}

}  // namespace bwd

// D_i = sum_t dO_it O_it (fp32) for every row, and the dQ accumulator row
// zeroed.  One warp per row.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const __nv_bfloat16* __restrict__ O,
                                                          const __nv_bfloat16* __restrict__ dO,
                                                          float* __restrict__ Dbuf,
                                                          float* __restrict__ dq_acc,
                                                          long long rows) {
  constexpr int kPer = D / 32;  // elements per lane
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const __nv_bfloat16* o = O + row * D + lane * kPer;
  const __nv_bfloat16* g = dO + row * D + lane * kPer;
  float acc = 0.f;
#pragma unroll
  for (int t = 0; t < kPer; t += 2) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(o + t);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(g + t);
    acc = fmaf(__bfloat162float(a.x), __bfloat162float(b.x), acc);
    acc = fmaf(__bfloat162float(a.y), __bfloat162float(b.y), acc);
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (lane == 0) Dbuf[row] = acc;
  float* z = dq_acc + row * D + lane * kPer;
#pragma unroll
  for (int t = 0; t < kPer; ++t) z[t] = 0.f;
}

// dQ = bf16(scale * accumulator), four elements per thread.
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const float* __restrict__ dq_acc,
                                                        __nv_bfloat16* __restrict__ dQ,
                                                        float scale, long long n4) {
  const long long t = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
  if (t >= n4) return;
  const float4 a = reinterpret_cast<const float4*>(dq_acc)[t];
  uint2 pk;
  pk.x = pack_bf16(a.x * scale, a.y * scale);
  pk.y = pack_bf16(a.z * scale, a.w * scale);
  reinterpret_cast<uint2*>(dQ)[t] = pk;
}


// dK_j, dV_j for one (batch*head, 128-key block j) and its share of dQ.
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(bwd::kThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const __grid_constant__ CUtensorMap tmDQ, const float* __restrict__ Lse,
                  const float* __restrict__ Dbuf, __nv_bfloat16* __restrict__ dK,
                  __nv_bfloat16* __restrict__ dV, DevError* __restrict__ err, int N, int BH,
                  float c_log2, float scale, unsigned long long timeout_ns) {
  using namespace bwd;
  using Ly = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int T = (N + kBlk - 1) / kBlk;
  int bh, j;
  if (CAUSAL) {  // blocks with the most query blocks first
    j = static_cast<int>(blockIdx.x) / BH;
    bh = static_cast<int>(blockIdx.x) - j * BH;
  } else {
    bh = static_cast<int>(blockIdx.x) / T;
    j = static_cast<int>(blockIdx.x) - bh * T;
  }
  const int i0 = CAUSAL ? j : 0;  // first query block that sees key block j
  const int n_it = T - i0;

  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + Ly::kAbort);
  const uint32_t bar_kv = base + Ly::kBarKV, bar_qfull = base + Ly::kBarQFull;
  const uint32_t bar_qempty = base + Ly::kBarQEmpty, bar_s = base + Ly::kBarS;
  const uint32_t bar_dp = base + Ly::kBarDP, bar_ds = base + Ly::kBarDS;
  const uint32_t bar_p = base + Ly::kBarP;
  const uint32_t bar_dq = base + Ly::kBarDQ, bar_dqfree = base + Ly::kBarDQFree;
  const uint32_t bar_fin = base + Ly::kBarFin;
  if (tid == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_qfull + 8 * s, 1);
      mbar_init(bar_qempty + 8 * s, 4);  // the dQ warps, after staging dQ there
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    mbar_init(bar_p, 8);       // compute warps: P^T in TMEM
    mbar_init(bar_ds, 8);      // compute warps: dS^T in shared memory
    mbar_init(bar_dq, 1);
    mbar_init(bar_dqfree, 4);  // dQ warps
    mbar_init(bar_fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(base + Ly::kTmemSlot, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + Ly::kTmemSlot);
  const WaitCtx wc{abort_flag, err, timeout_ns};
  const unsigned unit = blockIdx.x;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------- producer
    mbar_arrive_expect_tx(bar_kv, 2 * (D / 64) * 16384);
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      tma_load_3d(base + Ly::kK + c * 16384, &tmK, bar_kv, c * 64, j * kBlk, bh);
      tma_load_3d(base + Ly::kV + c * 16384, &tmV, bar_kv, c * 64, j * kBlk, bh);
    }
    int issued = 0;
    for (int it = 0; it < n_it; ++it) {
      const int st = it & 1;
      if (!mbar_wait(bar_qempty + 8 * st, ((it >> 1) & 1) ^ 1u, wc, kSiteBLoad, unit)) break;
      ++issued;
      const uint32_t fb = bar_qfull + 8 * st;
      mbar_arrive_expect_tx(fb, 2 * (D / 64) * 16384);
      const int row = (i0 + it) * kBlk;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(base + Ly::kQ + st * Ly::kTile + c * 16384, &tmQ, fb, c * 64, row, bh);
        tma_load_3d(base + Ly::kDO + st * Ly::kTile + c * 16384, &tmDO, fb, c * 64, row, bh);
      }
    }
    // every copy must have landed before the CTA may exit (bounded; already
    // true unless a wait above gave up)
    constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
    bwd::drain_wait_cta(bar_kv, 0, kDrainNs);
    for (int b = issued - 2 < 0 ? 0 : issued - 2; b < issued; ++b)
      bwd::drain_wait_cta(bar_qfull + 8 * (b & 1), (b >> 1) & 1, kDrainNs);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_bf16_f32_ab(kBlk, kBlk, false, false);  // S^T, dP^T
    constexpr uint32_t kIdG = idesc_bf16_f32_ab(kBlk, D, false, true);      // dV, dK
    constexpr uint32_t kIdQ = idesc_bf16_f32_ab(kBlk, D, true, true);       // dQ
    const uint64_t dKk = sw128_desc(base + Ly::kK, 16, 1024);       // K_j, K-major
    const uint64_t dVk = sw128_desc(base + Ly::kV, 16, 1024);       // V_j, K-major
    const uint64_t dKmn = sw128_desc(base + Ly::kK, 16384, 1024);   // K_j, MN-major
    const uint64_t dDSk = sw128_desc(base + Ly::kDS, 16, 1024);     // dS^T, K-major
    const uint64_t dDSmn = sw128_desc(base + Ly::kDS, 16384, 1024); // dS, MN-major
    auto qdesc = [&](int st, uint32_t lbo) { return sw128_desc(base + Ly::kQ + st * Ly::kTile, lbo, 1024); };
    auto odesc = [&](int st, uint32_t lbo) { return sw128_desc(base + Ly::kDO + st * Ly::kTile, lbo, 1024); };
    auto issue_s = [&](int it) {  // S^T = K_j Q_i^T
      const uint64_t dQk = qdesc(it & 1, 16);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(tmem + kColS, dKk + kstep_kmajor(kk), dQk + kstep_kmajor(kk), kIdS, kk > 0);
      tc_commit(bar_s);
    };
    auto issue_dp = [&](int it) {  // dP^T = V_j dO_i^T
      const uint64_t dOk = odesc(it & 1, 16);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(tmem + kColDP, dVk + kstep_kmajor(kk), dOk + kstep_kmajor(kk), kIdS, kk > 0);
      tc_commit(bar_dp);
    };
    // Order per step i: dV(i) as soon as P^T(i) is in TMEM, S^T(i+1) right
    // behind it (the pipe reads P^T(i) before S^T(i+1) overwrites those
    // columns), dK(i) and dQ(i) once dS^T(i) is in shared memory, dP^T(i+1)
    // once the dQ warps have read dQ(i) out of its columns.  The tensor pipe
    // then works on the next step while the compute warps work on this one.
    bool ok = mbar_wait(bar_kv, 0, wc, kSiteBKV, unit) &&
              mbar_wait(bar_qfull, 0, wc, kSiteBMmaQ, unit);
    if (ok) {
      tc_fence_after();
      issue_s(0);
      issue_dp(0);
    }
    for (int it = 0; it < n_it && ok; ++it) {
      const int st = it & 1;
      const bool more = it + 1 < n_it;
      if (!mbar_wait(bar_p, it & 1, wc, kSiteBMmaDS, unit)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t acc = it > 0 ? 1u : 0u;
      const uint64_t dOmn = odesc(st, 16384), dQmn = qdesc(st, 16384);
#pragma unroll
      for (int kk = 0; kk < kBlk / 16; ++kk)  // dV_j += P^T dO_i (P^T columns: see the compute warps)
        mma_ts(tmem + kColDV, tmem + kColS + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8),
               dOmn + static_cast<uint32_t>(kk * 128), kIdG, acc | (kk > 0 ? 1u : 0u));
      if (more) {
        if (!mbar_wait(bar_qfull + 8 * ((it + 1) & 1), ((it + 1) >> 1) & 1, wc, kSiteBMmaQ, unit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(it + 1);
      }
      if (!mbar_wait(bar_ds, it & 1, wc, kSiteBMmaDS, unit)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kBlk / 16; ++kk)  // dK_j += dS^T Q_i
        mma_ss(tmem + kColDV + D, dDSk + kstep_kmajor(kk), dQmn + static_cast<uint32_t>(kk * 128),
               kIdG, acc | (kk > 0 ? 1u : 0u));
#pragma unroll
      for (int kk = 0; kk < kBlk / 16; ++kk)  // dQ_i = dS K_j
        mma_ss(tmem + kColDP, dDSmn + static_cast<uint32_t>(kk * 128),
               dKmn + static_cast<uint32_t>(kk * 128), kIdQ, kk > 0 ? 1u : 0u);
      tc_commit(bar_dq);
      if (more) {
        if (!mbar_wait(bar_dqfree, it & 1, wc, kSiteBMmaFree, unit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_dp(it + 1);
      }
    }
    tc_commit(bar_fin);
    bwd::drain_wait_cta(bar_fin, 0, 50ull * 1000 * 1000);
  } else if ((warp >= 4 && warp < 8) || warp >= 12) {
    // -------------------------------------------------------------- compute
    const int qw = warp & 3;
    const int cg = warp >= 12 ? 1 : 0;              // query half of each step
    const int kr = qw * 32 + lane;                  // key row = TMEM lane
    const int kidx = j * kBlk + kr;
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    const float* lse_h = Lse + static_cast<size_t>(bh) * N;
    const float* d_h = Dbuf + static_cast<size_t>(bh) * N;
    uint8_t* ds_row = gbase + Ly::kDS + kr * 128;
    constexpr float kLog2e = 1.4426950408889634f;
    bool ok = true;
    for (int it = 0; it < n_it && ok; ++it) {
      const int qb = (i0 + it) * kBlk;
      // phase 1: P^T from S^T, written back as bf16 over S^T's first 64
      // columns; the packed values stay in registers for phase 2
      ok = mbar_wait(bar_s, it & 1, wc, kSiteBSoftS, unit);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t pk[2][16];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * cg + cc;  // 32-query chunk
        const int q0 = qb + 32 * c;
        const int qq = q0 + lane;  // this lane fetches query qq's logsumexp
        const float nl = qq < N ? -lse_h[qq] * kLog2e : -INFINITY;
        uint32_t sv[32];
        tmem_ld32(tmem + lane_off + kColS + 32 * c, sv);
        tmem_ld_wait32(sv);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float p2[2];
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const float nle = __shfl_sync(0xffffffffu, nl, e + t);
            const bool vis = kidx < N && (!CAUSAL || kidx <= q0 + e + t);
            p2[t] = vis ? ex2(fmaf(__uint_as_float(sv[e + t]), c_log2, nle)) : 0.f;
          }
          pk[cc][e >> 1] = pack_bf16(p2[0], p2[1]);
        }
        // P^T of this group's 64 queries goes inside the group's own S^T
        // columns [64 cg, 64 cg + 64), behind every column of them still to
        // be read: queries 0-63 at columns 0-31, 64-127 at columns 64-95
        tmem_st16(tmem + lane_off + kColS + 64 * cg + 16 * cc, pk[cc]);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p);
      // phase 2: dS^T = P^T (dP^T - D) into shared memory, once dP^T is in
      // and the previous step's dK / dQ products have read the buffer; P is
      // the bf16 value the dV product used
      ok = mbar_wait(bar_dp, it & 1, wc, kSiteBSoftS, unit) &&
           (it == 0 || mbar_wait(bar_dq, (it - 1) & 1, wc, kSiteBSoftDQ, unit));
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * cg + cc;
        const int qq = qb + 32 * c + lane;
        const float dd = qq < N ? d_h[qq] : 0.f;
        uint32_t dp[32];
        tmem_ld32(tmem + lane_off + kColDP + 32 * c, dp);
        tmem_ld_wait32(dp);
        uint32_t dw[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = __uint_as_float(pk[cc][e >> 1] << 16);
          const float p1 = __uint_as_float(pk[cc][e >> 1] & 0xffff0000u);
          const float d0 = __shfl_sync(0xffffffffu, dd, e);
          const float d1 = __shfl_sync(0xffffffffu, dd, e + 1);
          dw[e >> 1] = pack_bf16(p0 * (__uint_as_float(dp[e]) - d0),
                                 p1 * (__uint_as_float(dp[e + 1]) - d1));
        }
        // dS^T row kr, queries [32c, 32c + 32): 128B-swizzled, 64 queries per atom
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int unit16 = 4 * (c & 1) + u;
          uint4* dst = reinterpret_cast<uint4*>(ds_row + (c >> 1) * 16384 +
                                                ((unit16 ^ (kr & 7)) << 4));
          *dst = make_uint4(dw[4 * u], dw[4 * u + 1], dw[4 * u + 2], dw[4 * u + 3]);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();  // dS^T stores -> tensor-core reads
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds);
    }
  } else if (warp >= 8 && warp < 12) {
    // ---------------------------------------------------------- dQ, dK, dV
    const int qw = warp & 3;
    const int r = qw * 32 + lane;                   // TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    bool ok = true;
    for (int it = 0; it < n_it && ok; ++it) {
      ok = mbar_wait(bar_dq, it & 1, wc, kSiteBDq, unit);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // Stage dQ_i (rows 32 qw .. of the query block) in this step's Q/dO
      // ring stage, which every MMA of the step has finished reading: 32
      // rows x 32 fp32 boxes of 4 KB, 128B-swizzled as the TMA expects.  Read
      // in two halves of 64 columns; the columns go back to the MMA thread
      // after the last TMEM read.
      const int st = it & 1;
      const uint32_t region = base + (qw < 2 ? Ly::kQ : Ly::kDO) + st * Ly::kTile +
                              (qw & 1) * (D / 32) * 4096;
      auto stage32 = [&](int c, const uint32_t (&x)[32]) {
        uint8_t* row = gbase + (region - base) + c * 4096 + lane * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4*>(row + ((u ^ (lane & 7)) << 4)) =
              make_uint4(x[4 * u], x[4 * u + 1], x[4 * u + 2], x[4 * u + 3]);
      };
#pragma unroll 1
      for (int half = 0; half < D / 64; ++half) {
        uint32_t g0[32], g1[32];
        tmem_ld32(tmem + lane_off + kColDP + 64 * half, g0);
        tmem_ld32(tmem + lane_off + kColDP + 64 * half + 32, g1);
        tmem_ld_wait32(g0);
        tmem_ld_dep32(g1);
        if (half == D / 64 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_dqfree);
        }
        stage32(2 * half, g0);
        stage32(2 * half + 1, g1);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int y = (i0 + it) * kBlk + qw * 32;
        if (y < N) {  // rows past N are clipped by the TMA; a whole box past N is skipped
#pragma unroll
          for (int c = 0; c < D / 32; ++c) tma_reduce_add_3d(&tmDQ, region + c * 4096, 32 * c, y, bh);
          bulk_commit_group();
          bulk_wait_read_all();
        }
        mbar_arrive(bar_qempty + 8 * st);
      }
    }
    if (lane == 0) bulk_wait_all();
    if (ok) {
      // the last dQ commit covers every earlier MMA: dK_j and dV_j are final
      const int krow = j * kBlk + r;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = kColDV + which * D;
        const float mul = which ? scale : 1.0f;
        __nv_bfloat16* out = (which ? dK : dV) + (static_cast<size_t>(bh) * N + krow) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + col + 32 * c, v);
          tmem_ld_wait32(v);
          if (krow < N) {
            uint4* dst = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
            for (int t = 0; t < 4; ++t)
              dst[t] = make_uint4(
                  pack_bf16(__uint_as_float(v[8 * t]) * mul, __uint_as_float(v[8 * t + 1]) * mul),
                  pack_bf16(__uint_as_float(v[8 * t + 2]) * mul, __uint_as_float(v[8 * t + 3]) * mul),
                  pack_bf16(__uint_as_float(v[8 * t + 4]) * mul, __uint_as_float(v[8 * t + 5]) * mul),
                  pack_bf16(__uint_as_float(v[8 * t + 6]) * mul, __uint_as_float(v[8 * t + 7]) * mul));
          }
        }
      }
    }
  }
  __syncthreads();
  tc_fence_before();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa
