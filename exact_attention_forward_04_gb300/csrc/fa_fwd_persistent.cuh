// Exact attention forward for sm_103a: persistent, warp-specialised kernel.
//
// Semantics are the FA2 loop order ("Before implementing FlashAttention in
// Triton: FA1, 2 forward pass", FA2 section; "How FlashAttention got past the
// O(N^2) memory wall", tiling loop): each 128-row query tile keeps a running
// maximum m, a running sum l and an unnormalised accumulator O~ that is
// rescaled by alpha = exp(m_old - m_new); one divide at the end, and
// L = m + ln l.  Key blocks entirely right of the diagonal are skipped under
// the causal mask ("v2 and v3").  No score or probability matrix leaves the SM.
//
// GB300 mapping (one CTA per SM, 16 warps):
//   warps 0-3   softmax for query tile 0 (one thread per row of S)
//   warps 4-7   softmax for query tile 1
//   warps 8-11  epilogue (O = O~ / l in bf16, L in fp32)
//   warp 12     TMA producer: Q0/Q1 once per work unit, K_j/V_j through a
//               kStages-deep shared-memory ring
//   warp 13     tcgen05 MMA issuer; owns the TMEM allocation
//   warps 14-15 idle
// A work unit is 256 query rows (two 128-row tiles) of one (batch, head); both
// tiles share every K/V block that is loaded.  TMEM (512 columns):
//   S0 [0,128)  S1 [128,256)  O0 [256,256+D)  O1 [384,384+D)
// and P~ (bf16 pairs) overwrites the first 64 columns of its S tile.  The MMA
// issue order per key block j is  PV0(j), S0(j+1), PV1(j), S1(j+1):
// tcgen05 MMAs of one thread execute in order, so S_t(j+1) never overwrites
// P~_t(j) before PV_t(j) has read it, and the commit that signals S_t(j+1)
// also covers PV_t(j) -- the softmax warps may then rescale O_t in place.
//
// Rescaling is lazy: a row keeps its reference maximum until a block raises
// it by more than kLazyLog2 (in log2 units), so P~ <= 2^kLazyLog2 and O~ is
// rescaled only on such jumps (after the first block they are rare).  The
// final result is the same exact softmax: the reference cancels in O~ / l.
// Two row sums are kept: l over the fp32 P~ (for L) and l_r over the bf16
// values the MMA actually consumed (to normalise O), so that the rounding of a
// dominant P~ cancels between numerator and denominator.
#pragma once
#include <cuda_bf16.h>

#include "sm103_ptx.cuh"
#include "tmem_ldst.cuh"

namespace fa {

namespace pk {

constexpr int kRows = 128;       // rows per query tile = MMA M
constexpr int kKeys = 128;       // keys per block = MMA N of S
constexpr int kBox = 128 * 128;  // bytes of one 128-row x 64-column bf16 TMA box
constexpr int kThreads = 512;
constexpr float kLazyLog2 = 8.0f;

enum : unsigned {
  kSiteLoadQ = 11, kSiteLoadKV = 12, kSiteMmaQ = 21, kSiteMmaKV = 22, kSiteMmaP = 23,
  kSiteMmaFree = 25, kSiteSoftS = 31, kSiteEpiF = 42, kSiteEpiStats = 43
};

template <int D>
struct Layout {
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = kRows * D * 2;              // one 128 x D bf16 tile
  static constexpr int kStages = D == 128 ? 4 : 8;         // K/V ring depth
  static constexpr int kQ = 0;                             // Q0, Q1
  static constexpr int kRing = 2 * kTile;
  static constexpr int kMisc = kRing + kStages * kTile;
  // barriers (8 bytes each)
  static constexpr int kBarQFull = kMisc;
  static constexpr int kBarQEmpty = kBarQFull + 8;
  static constexpr int kBarKVFull = kBarQEmpty + 8;             // [kStages]
  static constexpr int kBarKVEmpty = kBarKVFull + 8 * kStages;  // [kStages]
  static constexpr int kBarS = kBarKVEmpty + 8 * kStages;       // [2]
  static constexpr int kBarP = kBarS + 16;                      // [2]
  static constexpr int kBarOFinal = kBarP + 16;                 // [2]
  static constexpr int kBarStats = kBarOFinal + 16;             // [2]
  static constexpr int kBarOFree = kBarStats + 16;              // [2]
  static constexpr int kBarFin = kBarOFree + 16;
  static constexpr int kTmemSlot = kBarFin + 8;
  static constexpr int kAbort = kTmemSlot + 8;
  static constexpr int kStats = (kAbort + 8 + 15) & ~15;        // float4 [2 units][2][128]
  static constexpr int kBytes = kStats + 4 * kRows * 16;
  static constexpr int kAlloc = kBytes + 1024;
};

// Work-unit schedule: unit u -> (bh, pair p).  Causal: longest rows first
// across all heads, snake order over rounds; non-causal: head-major (a head's
// K/V stays hot in L2).
struct Sched {
  int BH, n_pair, n_units, grid;
  bool causal;
  __device__ __forceinline__ int unit_of(int cta, int k) const {
    const long long base = static_cast<long long>(k) * grid;
    const int pos = (causal && (k & 1)) ? (grid - 1 - cta) : cta;
    const long long u = base + pos;
    return u < n_units ? static_cast<int>(u) : -1;
  }
  __device__ __forceinline__ int rounds() const { return (n_units + grid - 1) / grid; }
  __device__ __forceinline__ void decode(int u, int& bh, int& p) const {
    if (causal) {
      p = n_pair - 1 - u / BH;
      bh = u - (u / BH) * BH;
    } else {
      bh = u / n_pair;
      p = u - bh * n_pair;
    }
  }
};

// Key blocks seen by query tile t of pair p.
__device__ __forceinline__ int kv_blocks(bool causal, int p, int t, int n_kblk) {
  return causal ? min(2 * p + t + 1, n_kblk) : n_kblk;
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) return;
  }
}

__device__ __forceinline__ void setmaxnreg_inc184() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 184;\n" ::: "memory");
}
__device__ __forceinline__ void setmaxnreg_dec64() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 64;\n" ::: "memory");
}
__device__ __forceinline__ void setmaxnreg_dec80() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 80;\n" ::: "memory");
}

// Softmax of one 32-column chunk of a row: P~ = 2^(s c - m) as bf16 pairs
// into w[16]; adds the fp32 values to `sum` and the bf16-rounded values to
// `sum_r` (both packed pairs).
__device__ __forceinline__ void softmax_chunk(const uint32_t (&r)[32], uint64_t c2, uint64_t nm2,
                                              uint64_t& sum, uint64_t& sum_r,
                                              uint32_t (&w)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint64_t arg = f2_fma(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])),
                                c2, nm2);
    float a, b;
    f2_unpack(arg, a, b);
    a = ex2(a);
    b = ex2(b);
    const uint32_t pw = pack_bf16(a, b);
    w[i] = pw;
    sum = f2_add(sum, f2_pack(a, b));
    sum_r = f2_add(sum_r, f2_pack(__uint_as_float(pw << 16), __uint_as_float(pw & 0xffff0000u)));
  }
}

}  // namespace pk

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(pk::kThreads, 1)
    fa_fwd_persistent_kernel(const __grid_constant__ CUtensorMap tmQ,
                             const __grid_constant__ CUtensorMap tmK,
                             const __grid_constant__ CUtensorMap tmV,
                             __nv_bfloat16* __restrict__ O, float* __restrict__ Lse,
                             DevError* __restrict__ err, int N, int BH, float c_log2,
                             unsigned long long timeout_ns) {
  using namespace pk;
  using Ly = Layout<D>;
  constexpr int S = Ly::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + Ly::kAbort);
  float4* s_stats = reinterpret_cast<float4*>(gbase + Ly::kStats);
  const uint32_t bar_qfull = base + Ly::kBarQFull, bar_qempty = base + Ly::kBarQEmpty;
  const uint32_t bar_kvfull = base + Ly::kBarKVFull, bar_kvempty = base + Ly::kBarKVEmpty;
  const uint32_t bar_s = base + Ly::kBarS, bar_p = base + Ly::kBarP;
  const uint32_t bar_ofinal = base + Ly::kBarOFinal, bar_stats = base + Ly::kBarStats;
  const uint32_t bar_ofree = base + Ly::kBarOFree, bar_fin = base + Ly::kBarFin;

  if (warp == 13) {
    tmem_alloc(base + Ly::kTmemSlot, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar_qfull, 1);
    mbar_init(bar_qempty, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_kvfull + 8 * s, 1);
      mbar_init(bar_kvempty + 8 * s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_s + 8 * t, 1);
      mbar_init(bar_p + 8 * t, kRows);
      mbar_init(bar_ofinal + 8 * t, 1);
      mbar_init(bar_stats + 8 * t, kRows);
      mbar_init(bar_ofree + 8 * t, kRows);
    }
    mbar_init(bar_fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (tid == 32 * 12) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<const uint32_t*>(gbase + Ly::kTmemSlot);

  const WaitCtx wc{abort_flag, err, timeout_ns};
  const int n_kblk = (N + kKeys - 1) / kKeys;
  Sched sch;
  sch.BH = BH;
  sch.n_pair = (N + 2 * kRows - 1) / (2 * kRows);
  sch.n_units = BH * sch.n_pair;
  sch.grid = gridDim.x;
  sch.causal = CAUSAL;
  const int n_rounds = sch.rounds();
  const int cta = blockIdx.x;

  // Register split (launch: 512 threads x 128): softmax warpgroups 184,
  // epilogue 64, producer/MMA/idle 80: 2*128*184 + 128*64 + 128*80 = 65536.
  // Each warpgroup executes one setmaxnreg instruction, and its role code is
  // nested under it so the compiler allocates that role within the new limit.
  if (warp >= 12) {
    setmaxnreg_dec80();
    if (warp == 12 && lane == 0) {
      // ---------------------------------------------------------- producer
      int stage = 0;
      uint32_t phase = 0;
      long long n_issued = 0;
      int uidx = 0;
      bool ok = true;
      for (int k = 0; k < n_rounds && ok; ++k) {
        const int u = sch.unit_of(cta, k);
        if (u < 0) continue;
        int bh, p;
        sch.decode(u, bh, p);
        const int nkv = kv_blocks(CAUSAL, p, 1, n_kblk);  // tile 1 sees the most keys
        if (uidx > 0 && !mbar_wait(bar_qempty, (uidx - 1) & 1, wc, kSiteLoadQ, u)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar_qfull, 2 * Ly::kTile);
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int c = 0; c < Ly::kChunks; ++c)
            tma_load_3d(base + Ly::kQ + t * Ly::kTile + c * kBox, &tmQ, bar_qfull, c * 64,
                        (2 * p + t) * kRows, bh);
        ++uidx;
        for (int j = 0; j < nkv && ok; ++j) {
#pragma unroll 1
          for (int which = 0; which < 2; ++which) {  // K_j then V_j
            if (!mbar_wait(bar_kvempty + 8 * stage, phase ^ 1u, wc, kSiteLoadKV, u)) {
              ok = false;
              break;
            }
            const uint32_t fb = bar_kvfull + 8 * stage;
            const uint32_t dst = base + Ly::kRing + stage * Ly::kTile;
            mbar_arrive_expect_tx(fb, Ly::kTile);
            const CUtensorMap* m = which ? &tmV : &tmK;
#pragma unroll
            for (int c = 0; c < Ly::kChunks; ++c)
              tma_load_3d(dst + c * kBox, m, fb, c * 64, j * kKeys, bh);
            ++n_issued;
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // Drain: wait (bounded) until every load this thread started has landed.
      constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
      for (int s = 0; s < S; ++s) {
        const long long cnt = n_issued / S + (s < n_issued % S ? 1 : 0);
        if (cnt > 0) drain_wait(bar_kvfull + 8 * s, static_cast<uint32_t>((cnt - 1) & 1), kDrainNs);
      }
      if (uidx > 0) drain_wait(bar_qfull, (uidx - 1) & 1, kDrainNs);
    } else if (warp == 13 && lane == 0) {
      // -------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdescS = idesc_bf16_f32(kRows, kKeys, false);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(kRows, D, true);
      const uint32_t tS[2] = {tmem, tmem + 128};
      const uint32_t tO[2] = {tmem + 256, tmem + 384};
      const uint32_t sQ[2] = {base + Ly::kQ, base + Ly::kQ + Ly::kTile};
      int stage = 0;
      uint32_t phase = 0;
      uint32_t p_cnt[2] = {0, 0};
      int uidx = 0;
      bool ok = true;

      auto wait_kv = [&](int& st) -> bool {
        if (!mbar_wait(bar_kvfull + 8 * stage, phase, wc, kSiteMmaKV, 0)) return false;
        st = stage;
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
        return true;
      };
      // Descriptors advance by adding (byte offset >> 4) to the start-address
      // field; every operand address stays below 256 KB, so it never carries.
      auto mma_s = [&](int t, int kst) {
        const uint64_t da = sw128_desc(sQ[t], 16, 1024);
        const uint64_t db = sw128_desc(base + Ly::kRing + kst * Ly::kTile, 16, 1024);
#pragma unroll 1
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kBox + (kk & 3) * 32) >> 4;
          mma_ss(tS[t], da + off, db + off, kIdescS, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar_s + 8 * t);
      };
      auto mma_pv = [&](int t, int vst, bool first) {
        const uint64_t db = sw128_desc(base + Ly::kRing + vst * Ly::kTile, kBox, 1024);
#pragma unroll 1
        for (int kk = 0; kk < kKeys / 16; ++kk)
          mma_ts(tO[t], tS[t] + kk * 8, db + static_cast<uint32_t>(kk * (2048 >> 4)), kIdescPV,
                 (!first || kk > 0) ? 1u : 0u);
      };
      // Before PV_t(j): P~_t(j) written (and O_t rescaled if needed), and for
      // j == 0 O_t released by the previous unit's epilogue.
      auto wait_pv_ready = [&](int t, int j) -> bool {
        if (!mbar_wait(bar_p + 8 * t, p_cnt[t] & 1, wc, kSiteMmaP, t)) return false;
        ++p_cnt[t];
        if (j == 0 && uidx > 0) {
          if (!mbar_wait(bar_ofree + 8 * t, (uidx - 1) & 1, wc, kSiteMmaFree, t)) return false;
        }
        tc_fence_after();
        return true;
      };

      for (int k = 0; k < n_rounds && ok; ++k) {
        const int u = sch.unit_of(cta, k);
        if (u < 0) continue;
        int bh, p;
        sch.decode(u, bh, p);
        const int nkv0 = kv_blocks(CAUSAL, p, 0, n_kblk);
        const int nkv1 = kv_blocks(CAUSAL, p, 1, n_kblk);  // nkv1 >= nkv0
        if (!mbar_wait(bar_qfull, uidx & 1, wc, kSiteMmaQ, u)) {
          ok = false;
          break;
        }
        int kst, vst;
        if (!wait_kv(kst)) {
          ok = false;
          break;
        }
        tc_fence_after();
        mma_s(0, kst);
        mma_s(1, kst);
        tc_commit(bar_kvempty + 8 * kst);
        if (nkv1 == 1) tc_commit(bar_qempty);  // last S MMA of the unit issued
        for (int j = 0; j < nkv1; ++j) {
          if (!wait_kv(vst)) {
            ok = false;
            break;
          }
          const bool more = j + 1 < nkv1;
          bool k_next = false;
          if (j < nkv0) {
            if (!wait_pv_ready(0, j)) {
              ok = false;
              break;
            }
            mma_pv(0, vst, j == 0);
            if (j + 1 < nkv0) {
              if (!wait_kv(kst)) {
                ok = false;
                break;
              }
              k_next = true;
              tc_fence_after();
              mma_s(0, kst);
            } else {
              tc_commit(bar_ofinal + 0);
            }
          }
          if (more && !k_next) {
            if (!wait_kv(kst)) {
              ok = false;
              break;
            }
          }
          if (!wait_pv_ready(1, j)) {
            ok = false;
            break;
          }
          mma_pv(1, vst, j == 0);
          tc_commit(bar_kvempty + 8 * vst);
          if (more) {
            mma_s(1, kst);
            tc_commit(bar_kvempty + 8 * kst);
            if (j + 2 == nkv1) tc_commit(bar_qempty);  // last S MMA of the unit issued
          } else {
            tc_commit(bar_ofinal + 8);
          }
        }
        if (!ok) break;
        ++uidx;
      }
      constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
      tc_commit(bar_fin);
      drain_wait(bar_fin, 0, kDrainNs);
    }
    // lanes 1-31 of warps 12-13 and warps 14-15 have no role
  } else if (warp < 8) {
    setmaxnreg_inc184();
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;                 // query tile of this warpgroup
    const int r = tid & 127;                 // row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + t * 128 + lane_off;
    const uint32_t tO = tmem + 256 + t * 128 + lane_off;
    const uint32_t bS = bar_s + 8 * t;
    const uint64_t c2 = f2_pack(c_log2, c_log2);
    uint32_t s_cnt = 0;
    int uidx = 0;
    bool ok = true;
    for (int k = 0; k < n_rounds && ok; ++k) {
      const int u = sch.unit_of(cta, k);
      if (u < 0) continue;
      int bh, p;
      sch.decode(u, bh, p);
      const int nkv = kv_blocks(CAUSAL, p, t, n_kblk);
      const int qrow = (2 * p + t) * kRows + r;
      float m_ref = -INFINITY;  // reference maximum of s * c (base-2 units)
      float l_run = 0.f;        // sum of fp32 2^(s c - m_ref)
      float lr_run = 0.f;       // sum of the bf16-rounded values
      for (int j = 0; j < nkv; ++j) {
        ok = mbar_wait(bS, s_cnt & 1, wc, kSiteSoftS, u);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        ++s_cnt;
        tc_fence_after();
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tmem_ld32(tS + 0, r0);
        tmem_ld32(tS + 32, r1);
        tmem_ld32(tS + 64, r2);
        tmem_ld32(tS + 96, r3);
        tmem_ld_wait32(r0);
        tmem_ld_dep32(r1);
        tmem_ld_dep32(r2);
        tmem_ld_dep32(r3);
        const int kbase = j * kKeys;
        if (kbase + kKeys > N || (CAUSAL && j == 2 * p + t)) {
          const int last = CAUSAL ? min(N - 1, qrow) : N - 1;  // last visible key
          constexpr uint32_t kNegInf = 0xff800000u;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (kbase + c > last) r0[c] = kNegInf;
            if (kbase + 32 + c > last) r1[c] = kNegInf;
            if (kbase + 64 + c > last) r2[c] = kNegInf;
            if (kbase + 96 + c > last) r3[c] = kNegInf;
          }
        }
        float mx0 = __uint_as_float(r0[0]), mx1 = __uint_as_float(r1[0]);
        float mx2 = __uint_as_float(r2[0]), mx3 = __uint_as_float(r3[0]);
#pragma unroll
        for (int c = 1; c < 31; c += 2) {
          mx0 = fmax3(mx0, __uint_as_float(r0[c]), __uint_as_float(r0[c + 1]));
          mx1 = fmax3(mx1, __uint_as_float(r1[c]), __uint_as_float(r1[c + 1]));
          mx2 = fmax3(mx2, __uint_as_float(r2[c]), __uint_as_float(r2[c + 1]));
          mx3 = fmax3(mx3, __uint_as_float(r3[c]), __uint_as_float(r3[c + 1]));
        }
        mx0 = fmax3(mx0, __uint_as_float(r0[31]), __uint_as_float(r1[31]));
        mx2 = fmax3(mx2, __uint_as_float(r2[31]), __uint_as_float(r3[31]));
        const float m_blk = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * c_log2;
        // Lazy reference update: only a jump above kLazyLog2 moves m_ref.
        const bool bump = m_blk > m_ref + kLazyLog2;  // always true at j == 0
        float alpha = 1.0f;
        if (bump) {
          alpha = ex2(m_ref - m_blk);                 // 0 when m_ref == -inf
          m_ref = m_blk;
          l_run *= alpha;
          lr_run *= alpha;
        }
        if (j > 0 && __any_sync(0xffffffffu, bump)) {
          // O~_t(j-1) is complete (the commit behind this S covered PV_t(j-1))
          // and PV_t(j) waits for this warpgroup: rescale this warp's rows.
          const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_ld_wait32(o);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float a, b;
              f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])),
                               a2),
                        a, b);
              o[2 * i] = __float_as_uint(a);
              o[2 * i + 1] = __float_as_uint(b);
            }
            tmem_st32(tO + c * 32, o);
          }
        }
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        const uint64_t nm2 = f2_pack(-m_use, -m_use);
        uint64_t sum = f2_pack(0.f, 0.f), sum_r = f2_pack(0.f, 0.f);
        {
          uint32_t w[16];
          softmax_chunk(r0, c2, nm2, sum, sum_r, w);
          tmem_st16(tS + 0, w);
        }
        {
          uint32_t w[16];
          softmax_chunk(r1, c2, nm2, sum, sum_r, w);
          tmem_st16(tS + 16, w);
        }
        {
          uint32_t w[16];
          softmax_chunk(r2, c2, nm2, sum, sum_r, w);
          tmem_st16(tS + 32, w);
        }
        {
          uint32_t w[16];
          softmax_chunk(r3, c2, nm2, sum, sum_r, w);
          tmem_st16(tS + 48, w);
        }
        float s_lo, s_hi, r_lo, r_hi;
        f2_unpack(sum, s_lo, s_hi);
        f2_unpack(sum_r, r_lo, r_hi);
        l_run += s_lo + s_hi;
        lr_run += r_lo + r_hi;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar_p + 8 * t);
      }
      if (!ok) break;
      // Double-buffered by unit: a unit with a single key block can finish
      // before the epilogue has read the previous unit's statistics.
      s_stats[((uidx & 1) * 2 + t) * kRows + r] = make_float4(m_ref, l_run, lr_run, 0.f);
      mbar_arrive(bar_stats + 8 * t);
      ++uidx;
    }
  } else {
    setmaxnreg_dec64();
    // ----------------------------------------------------------- epilogue
    const int r = tid & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int uidx = 0;
    bool ok = true;
    for (int k = 0; k < n_rounds && ok; ++k) {
      const int u = sch.unit_of(cta, k);
      if (u < 0) continue;
      int bh, p;
      sch.decode(u, bh, p);
#pragma unroll 1
      for (int t = 0; t < 2; ++t) {
        ok = mbar_wait(bar_ofinal + 8 * t, uidx & 1, wc, kSiteEpiF, u) &&
             mbar_wait(bar_stats + 8 * t, uidx & 1, wc, kSiteEpiStats, u);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float4 st = s_stats[((uidx & 1) * 2 + t) * kRows + r];
        const float inv_l = 1.0f / st.z;
        const int qrow = (2 * p + t) * kRows + r;
        const bool row_ok = qrow < N;
        __nv_bfloat16* orow = O + (static_cast<size_t>(bh) * N + qrow) * D;
        const uint32_t tO = tmem + 256 + t * 128 + lane_off;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait32(o);
          if (c == D / 32 - 1) {
            // every TMEM read of O_t is done: the next unit may overwrite it
            tc_fence_before();
            mbar_arrive(bar_ofree + 8 * t);
          }
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16(__uint_as_float(o[2 * i]) * inv_l,
                             __uint_as_float(o[2 * i + 1]) * inv_l);
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
            dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
          }
        }
        if (row_ok)
          Lse[static_cast<size_t>(bh) * N + qrow] = (st.x + log2f(st.y)) * 0.693147180559945309f;
      }
      ++uidx;
    }
  }

  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa
