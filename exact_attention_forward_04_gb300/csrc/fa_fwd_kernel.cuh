// Exact attention forward for sm_103a: one CTA per 128-row query tile.
//
// Per tile (FA2 loop order: "Before implementing FlashAttention in Triton:
// FA1, 2 forward pass", FA2 section; "How FlashAttention got past the
// O(N^2) memory wall", tiling loop):
//   TMA loads Q_i once and streams K_j, V_j through a two-stage ring;
//   S = Q_i K_j^T is a tcgen05 MMA into tensor memory (TMEM);
//   each thread owns one row of S: it reads the row from TMEM, masks it,
//   updates the running maximum m and sum l, and writes P~ = exp(S - m)
//   back to TMEM as bf16;
//   O~ (fp32, TMEM) is rescaled by alpha = exp(m_old - m_new) and
//   O~ += P~ V_j is a second tcgen05 MMA with P~ read from TMEM;
//   at the end O = O~ / l (bf16) and L = m + ln l (fp32) go to memory.
// The softmax runs in base 2: with c = scale * log2(e) the row maximum is
// kept as max(s) * c and P~ = 2^(s c - m), so 2^(s c - m) = e^(scale s - m ln 2).
#pragma once
#include <cuda_bf16.h>

#include "sm103_ptx.cuh"
#include "tmem_ldst.cuh"

namespace fa {

constexpr int kBM = 128;               // query rows per tile (MMA M)
constexpr int kBN = 128;               // keys per block (MMA N of S)
constexpr int kBoxBytes = 128 * 128;   // one TMA box: 128 rows x 64 bf16
constexpr uint32_t kTmemCols = 256;    // S (128 columns) + O (up to 128)

// Wait-site ids reported in the device error record.
enum : unsigned { kSiteQ = 1, kSiteKV = 2, kSiteS = 3, kSiteP = 4, kSiteO = 5 };

template <int D>
struct TileLayout {
  static constexpr int kChunks = D / 64;           // 64-column TMA boxes per row
  static constexpr int kTileBytes = kBM * D * 2;   // one 128 x D bf16 tile
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;       // two stages
  static constexpr int kV = kK + 2 * kTileBytes;   // two stages
  static constexpr int kBar = kV + 2 * kTileBytes; // 8 mbarriers
  static constexpr int kTmemSlot = kBar + 8 * 8;
  static constexpr int kAbort = kTmemSlot + 16;
  static constexpr int kBytes = kAbort + 16;
  static constexpr int kAlloc = kBytes + 1024;     // slack to align the base to 1024
};

// Bounded wait used while draining after an abort: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) return;
  }
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(128, 1)
    fa_fwd_tile_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O,
                       float* __restrict__ Lse, DevError* __restrict__ err, int N, int n_qblk,
                       float c_log2, unsigned long long timeout_ns) {
  using Ly = TileLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int tile = blockIdx.x;
  const int bh = tile / n_qblk;
  const int qblk = tile - bh * n_qblk;

  const uint32_t sQ = base + Ly::kQ;
  const uint32_t sK = base + Ly::kK;
  const uint32_t sV = base + Ly::kV;
  const uint32_t bar_q = base + Ly::kBar + 0;
  const uint32_t bar_kv0 = base + Ly::kBar + 8;   // + 8 * stage
  const uint32_t bar_s = base + Ly::kBar + 24;
  const uint32_t bar_p = base + Ly::kBar + 32;
  const uint32_t bar_o = base + Ly::kBar + 40;
  const uint32_t bar_fin = base + Ly::kBar + 48;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + Ly::kAbort);
  const uint32_t* tmem_slot = reinterpret_cast<const uint32_t*>(gbase + Ly::kTmemSlot);

  if (warp == 0) {
    tmem_alloc(base + Ly::kTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 32) {
    mbar_init(bar_q, 1);
    mbar_init(bar_kv0, 1);
    mbar_init(bar_kv0 + 8, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_p, kBM);
    mbar_init(bar_o, 1);
    mbar_init(bar_fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (tid == 64) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;         // S: columns [0, 128); P~ (bf16 pairs) reuses [0, 64)
  const uint32_t tO = tmem + 128;   // O~: columns [128, 128 + D)

  const WaitCtx wc{abort_flag, err, timeout_ns};
  const int n_kblk = (N + kBN - 1) / kBN;
  const int nkv = CAUSAL ? min(qblk + 1, n_kblk) : n_kblk;
  constexpr uint32_t kTxKV = 2u * Ly::kTileBytes;

  auto issue_kv = [&](int stage, int j) {
    const uint32_t bar = bar_kv0 + 8u * stage;
    const uint32_t dK = sK + stage * Ly::kTileBytes;
    const uint32_t dV = sV + stage * Ly::kTileBytes;
    mbar_arrive_expect_tx(bar, kTxKV);
#pragma unroll
    for (int c = 0; c < Ly::kChunks; ++c) {
      tma_load_3d(dK + c * kBoxBytes, &tmK, bar, c * 64, j * kBN, bh);
      tma_load_3d(dV + c * kBoxBytes, &tmV, bar, c * 64, j * kBN, bh);
    }
  };

  // Thread 0 issues every TMA load and every MMA.
  int kv_issued = 0, kv_waited = 0;
  bool q_waited = false;
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_q, Ly::kTileBytes);
#pragma unroll
    for (int c = 0; c < Ly::kChunks; ++c)
      tma_load_3d(sQ + c * kBoxBytes, &tmQ, bar_q, c * 64, qblk * kBM, bh);
    for (; kv_issued < 2 && kv_issued < nkv; ++kv_issued) issue_kv(kv_issued, kv_issued);
  }

  constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false);
  constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, true);
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  const int qrow = qblk * kBM + tid;

  float m_run = -INFINITY;  // running max of s * c (base-2 units)
  float l_run = 0.f;        // running sum of 2^(s c - m_run)
  bool ok = true;

  for (int j = 0; j < nkv; ++j) {
    const int st = j & 1;
    const uint32_t sKs = sK + st * Ly::kTileBytes;
    const uint32_t sVs = sV + st * Ly::kTileBytes;
    if (tid == 0) {
      bool rdy = true;
      if (j == 0) {
        rdy = mbar_wait(bar_q, 0, wc, kSiteQ, tile);
        q_waited = rdy;
      }
      rdy = rdy && mbar_wait(bar_kv0 + 8u * st, (j >> 1) & 1, wc, kSiteKV, tile);
      if (rdy) {
        ++kv_waited;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
          mma_ss(tS, sw128_desc(sQ + off, 16, 1024), sw128_desc(sKs + off, 16, 1024), kIdescS,
                 kk > 0 ? 1u : 0u);
        }
        tc_commit(bar_s);
      }
    }
    ok = mbar_wait(bar_s, j & 1, wc, kSiteS, tile);
    if (!__all_sync(0xffffffffu, ok)) {
      ok = false;
      break;
    }
    tc_fence_after();

    // ---- this thread's row of S
    uint32_t r0[32], r1[32], r2[32], r3[32];
    tmem_ld32(tS + lane_off + 0, r0);
    tmem_ld32(tS + lane_off + 32, r1);
    tmem_ld32(tS + lane_off + 64, r2);
    tmem_ld32(tS + lane_off + 96, r3);
    tmem_ld_wait32(r0);
    tmem_ld_dep32(r1);
    tmem_ld_dep32(r2);
    tmem_ld_dep32(r3);
    float s[128];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      s[i] = __uint_as_float(r0[i]);
      s[32 + i] = __uint_as_float(r1[i]);
      s[64 + i] = __uint_as_float(r2[i]);
      s[96 + i] = __uint_as_float(r3[i]);
    }
    const int kbase = j * kBN;
    if (kbase + kBN > N || (CAUSAL && j == qblk)) {
      const int last = CAUSAL ? min(N - 1, qrow) : N - 1;  // last visible key
#pragma unroll
      for (int c = 0; c < kBN; ++c)
        if (kbase + c > last) s[c] = -INFINITY;
    }
    float mx = s[0];
#pragma unroll
    for (int c = 1; c < kBN; ++c) mx = fmaxf(mx, s[c]);
    const float m_new = fmaxf(m_run, mx * c_log2);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = ex2(m_run - m_use);
    float rsum = 0.f;
    uint32_t p0[32], p1[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const float a = ex2(fmaf(s[2 * c], c_log2, -m_use));
      const float b = ex2(fmaf(s[2 * c + 1], c_log2, -m_use));
      const float e = ex2(fmaf(s[64 + 2 * c], c_log2, -m_use));
      const float f = ex2(fmaf(s[64 + 2 * c + 1], c_log2, -m_use));
      rsum += (a + b) + (e + f);
      p0[c] = pack_bf16(a, b);
      p1[c] = pack_bf16(e, f);
    }
    l_run = l_run * alpha + rsum;
    tmem_st32(tS + lane_off + 0, p0);
    tmem_st32(tS + lane_off + 32, p1);
    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + lane_off + c * 32, o);
        tmem_ld_wait32(o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st32(tO + lane_off + c * 32, o);
      }
    }
    m_run = m_new;
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(bar_p);

    if (tid == 0) {
      if (mbar_wait(bar_p, j & 1, wc, kSiteP, tile)) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          mma_ts(tO, tS + kk * 8, sw128_desc(sVs + kk * 2048, kBoxBytes, 1024), kIdescPV,
                 (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar_o);
      }
    }
    ok = mbar_wait(bar_o, j & 1, wc, kSiteO, tile);
    if (!__all_sync(0xffffffffu, ok)) {
      ok = false;
      break;
    }
    tc_fence_after();
    if (tid == 0 && kv_issued < nkv) {
      issue_kv(st, kv_issued);
      ++kv_issued;
    }
  }

  // ---- epilogue: O = O~ / l in bf16, L = (m + log2 l) ln 2
  if (ok) {
    const float inv_l = 1.0f / l_run;
    const bool row_ok = qrow < N;
    __nv_bfloat16* orow = O + (static_cast<size_t>(bh) * N + qrow) * D;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(tO + lane_off + c * 32, o);
      tmem_ld_wait32(o);
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        w[i] = pack_bf16(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
      if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
        dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
      }
    }
    if (row_ok) Lse[static_cast<size_t>(bh) * N + qrow] = (m_run + log2f(l_run)) * 0.693147180559945309f;
  }

  // ---- teardown: drain whatever this CTA still has in flight, free TMEM
  if (tid == 0) {
    constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
    tc_commit(bar_fin);
    drain_wait(bar_fin, 0, kDrainNs);
    if (!q_waited) drain_wait(bar_q, 0, kDrainNs);
    for (int b = kv_waited; b < kv_issued; ++b) drain_wait(bar_kv0 + 8u * (b & 1), (b >> 1) & 1, kDrainNs);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa
