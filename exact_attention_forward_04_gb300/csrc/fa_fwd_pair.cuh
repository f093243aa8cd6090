// Exact attention forward for sm_103a, head dims 64 and 128: persistent
// kernel on CTA pairs (2-SM tcgen05 MMAs).
//
// Semantics are the FA2 loop order ("Before implementing FlashAttention in
// Triton: FA1, 2 forward pass", FA2 section; "How FlashAttention got past the
// O(N^2) memory wall", tiling loop): a query tile keeps a running maximum m,
// a running sum l and an unnormalised accumulator O~ rescaled by
// alpha = exp(m_old - m_new); one divide at the end and L = m + ln l.  Key
// blocks entirely right of the diagonal are skipped under the causal mask
// ("v2 and v3").  No score or probability matrix leaves the SM.
//
// GB300 mapping.  A cluster of two CTAs (one per SM) owns a work unit of 256
// query rows of one (batch, head): the even CTA rows [0,128), the odd CTA
// rows [128,256).  Keys come in blocks of 256.  Every MMA is a pair MMA
// (M = 256) issued by one thread of the even CTA:
//   S  = Q K_j^T : M 256, N 256 (keys), K = d; each CTA supplies its own
//                  128 query rows and 128 of the 256 keys of K_j
//   O~ += P~ V_j : M 256, N 128, K = 256 (keys); P~ from each CTA's TMEM,
//                  each CTA supplies 64 columns of V_j.  For d = 64 the odd
//                  CTA's 64 columns lie beyond the head and TMA fills them
//                  with zeros: an N = 64 MMA would cost the same, because a
//                  PV instruction is bound by its fixed cost, not its width.
// so each SM loads only half of every K/V block, and each MMA instruction
// carries enough work to keep the tensor pipe streaming.
// Per CTA: TMEM S [0,256) fp32, P~ [256,384) bf16 pairs (8-bit: two buffers
// of 64 columns, block g in buffer g & 1), O~ [384,512) fp32.
// Warps (per CTA, 16):
//   0-3   softmax, keys [0,128) of each block (one thread per row)
//   4-7   softmax, keys [128,256) of each block; the two warpgroups exchange
//         their partial row maxima through shared memory
//   8-11  epilogue (O = O~ / l_r in bf16, L in fp32)
//   12    TMA producer of Q and K (both CTAs; completions land on the even CTA)
//   13    S GEMM issuer (even CTA) and TMEM owner (both CTAs)
//   14    PV GEMM issuer (even CTA)
//   15    TMA producer of V (both CTAs)
// Barrier scopes: the even CTA's MMA thread waits with cluster-scope acquire
// (its barriers receive the odd CTA's arrivals and TMA bytes); every other
// wait is on a barrier fed by this CTA's threads or by the leader's
// multicast commits and uses CTA scope.  The softmax warps' per-block
// arrivals (S read, P~ written) are relaxed cluster-scope arrivals in both
// CTAs: each follows tcgen05.wait::ld/st and tcgen05.fence::before_thread_sync,
// so the TMEM reads or writes it announces are already complete; the other
// arrivals are local in the even CTA and relaxed remote ones in the odd CTA.
// MMA issue order: S(0), then for each block j: S(j+1) as soon as both CTAs
// have read S(j) into registers and every MMA of PV(j-1) has been issued
// (so that the PV product the softmax waits for next is not interleaved
// with S(j+1) in the tensor pipe), PV(j) once P~(j) is written.  The softmax
// of block j+1 writes P~ only after PV(j) has completed (pv_done), and may
// rescale O~ in place at that point.
//
// Rescaling is lazy (a row keeps its reference maximum until a block raises
// it by more than 16 (bf16) or 8 (E4M3 P~) in log2 units).  L uses l, the sum of the fp32
// P~; O is normalised by l plus the bf16 rounding error of each block's
// largest P~ (per key half), so that the rounding of a dominant P~ -- which
// the lazy reference no longer pins to exactly 1 -- cancels between the
// numerator the MMA sees and the denominator.
//
// 8-bit variant (FP8): Q, K and V arrive as E4M3 codes with
// one descale factor per (batch, head) for each; V is laid out keys-last
// ([d][keys]) so that both GEMMs read K-major operands.  The MMAs become
// kind::f8f6f4 (K = 32 per instruction: 4 S and 8 PV instructions per block
// instead of 8 and 16), each CTA loads 16 KB per K or V half-block, P~ is
// written to TMEM as E4M3 (four per column, 64 columns), the descales of Q
// and K fold into the exponent constant and V's into the final divide.  The
// schedule, barriers and softmax are the bf16 kernel's.  Head dim 64 keeps
// the 128-byte rows: the TMA fills bytes 64..127 of each Q and K row with
// zeros and the S product takes only the two K-steps that carry data; V's
// rows 64..127 (the odd CTA's half) read as zeros and pad the PV product as
// in the bf16 kernel.
#pragma once
#include <cuda_bf16.h>

#include "sm103_ptx.cuh"
#include "tmem_ldst.cuh"

namespace fa {

namespace pair {

constexpr int kRows = 128;         // query rows per CTA
constexpr int kKeys = 256;         // keys per block (pair MMA N of S)
constexpr int kHalfKeys = 128;     // keys of a block held by one CTA
constexpr int kPVN = 128;          // N of the PV MMA: O~ columns (head dim 64 pads with zeros)
constexpr int kThreads = 512;
// A row keeps its reference maximum until a block exceeds it by more than
// this (log2 units), so P~ <= 2^threshold: 16 for bf16 P~ (its rounding is
// relative, and fp32 sums of such terms lose nothing that matters), 8 for
// E4M3 P~ (largest finite value 448).
constexpr float kLazyLog2Bf16 = 16.0f;
constexpr float kLazyLog2E4m3 = 8.0f;
constexpr int kTile = 32768;       // one 32 KB operand tile
constexpr int kStages = 4;         // K/V ring depth (tiles)
constexpr uint16_t kBoth = 0x3;    // multicast mask: both CTAs

// TMEM columns
constexpr uint32_t kColS = 0, kColP = 256, kColO = 384;

enum : unsigned {
  kSiteLoadQ = 111, kSiteLoadKV = 112, kSiteMmaQ = 121, kSiteMmaKV = 122, kSiteMmaOFree = 125,
  kSiteSoftS = 131, kSiteSoftPV = 133,
  kSiteEpiF = 141, kSiteEpiStats = 142
};

struct Layout {
  static constexpr int kQ = 0;                                  // 2 buffers of 128 x D bf16
  static constexpr int kRing = 2 * kTile;                       // kStages x 32 KB
  static constexpr int kMisc = kRing + kStages * kTile;
  static constexpr int kBarQFull = kMisc;                       // [2]
  static constexpr int kBarQEmpty = kBarQFull + 16;             // [2]
  static constexpr int kBarKVFull = kBarQEmpty + 16;            // [kStages]
  static constexpr int kBarKVEmpty = kBarKVFull + 8 * kStages;  // [kStages]
  static constexpr int kBarOFinal = kBarKVEmpty + 8 * kStages;
  static constexpr int kBarOFree = kBarOFinal + 8;
  static constexpr int kBarStats = kBarOFree + 8;               // [2] by unit parity
  static constexpr int kBarFin = kBarStats + 16;                // [2] S issuer, PV issuer
  static constexpr int kBarPvIss = kBarFin + 16;                // [2] PV(g) issued, by g parity
  static constexpr int kTmemSlot = kBarPvIss + 16;
  static constexpr int kAbort = kTmemSlot + 8;
  static constexpr int kStats = (kAbort + 8 + 15) & ~15;        // float4 [2 units][2 key halves][128]
  static constexpr int kBytes = kStats + 2 * 2 * kRows * 16;
  static constexpr int kAlloc = kBytes + 1024;
};

// Work-unit schedule over clusters: unit u -> (bh, pair-tile p).  Causal:
// longest rows first across all heads, snake order over rounds; non-causal:
// head-major so that a head's K/V stays hot in L2.
// Work units: (batch*head, 256-row query tile p, key-block range [kb, ke)).
// With `splits` > 1 the visible key blocks of a tile (all of them, or 0..p
// under the causal mask) are cut into min(splits, count) balanced, non-empty
// ranges; each range is a unit of its own and leaves a partial result that a
// combine kernel merges. splits = 1 gives one unit per tile.
// Order: head-major without the mask.  With it, heads go in groups of
// head_group (chosen by the host so that the group's keys and values stay in
// L2 and the static round-robin below stays balanced), longest tiles of the
// group first.
struct Sched {
  int BH, n_tiles, n_units, n_clusters, splits;
  int head_group;  // causal one-pass order: heads scheduled together
  bool causal;
  __host__ __device__ static long long count_units(long long BH, int n_tiles, int splits,
                                                   bool causal) {
    if (!causal) return BH * n_tiles * (splits < n_tiles ? splits : n_tiles);
    const int hi = n_tiles - (splits - 1);  // tiles p >= splits - 1 take all splits
    long long n = hi > 0 ? BH * splits * hi : 0;
    const int lo_top = splits - 2 < n_tiles - 1 ? splits - 2 : n_tiles - 1;  // p + 1 splits each
    if (lo_top >= 0) n += BH * (static_cast<long long>(lo_top) + 1) * (lo_top + 2) / 2;
    return n;
  }
  __device__ __forceinline__ int unit_of(int cl, int k) const {
    const long long base = static_cast<long long>(k) * n_clusters;
    const int pos = (causal && (k & 1)) ? (n_clusters - 1 - cl) : cl;
    const long long u = base + pos;
    return u < n_units ? static_cast<int>(u) : -1;
  }
  __device__ __forceinline__ int rounds() const { return (n_units + n_clusters - 1) / n_clusters; }
  // unit -> (bh, p, split index sp, key blocks [kb, ke)); without SPLIT a
  // unit is a whole tile and the arithmetic stays the one-pass kernel's.
  template <bool SPLIT>
  __device__ __forceinline__ void decode(int u, int& bh, int& p, int& sp, int& kb, int& ke) const {
    if (!SPLIT) {
      if (causal) {
        const int per_group = head_group * n_tiles;
        const int grp = u / per_group;
        const int g0 = grp * head_group;
        const int gs = BH - g0 < head_group ? BH - g0 : head_group;  // last group may be smaller
        const int v = u - grp * per_group;
        p = n_tiles - 1 - v / gs;
        bh = g0 + (v - (v / gs) * gs);
      } else {
        bh = u / n_tiles;
        p = u - bh * n_tiles;
      }
      sp = 0;
      kb = 0;
      ke = causal ? p + 1 : n_tiles;
      return;
    }
    int ns, nkv;
    if (!causal) {
      ns = splits < n_tiles ? splits : n_tiles;
      const int per_head = n_tiles * ns;
      bh = u / per_head;
      const int rem = u - bh * per_head;
      p = rem / ns;
      sp = rem - p * ns;
      nkv = n_tiles;
    } else {
      const int hi = n_tiles - (splits - 1);
      const long long u_hi = hi > 0 ? static_cast<long long>(BH) * splits * hi : 0;
      if (u < u_hi) {
        const int per = BH * splits;
        const int qd = u / per;
        const int rem = u - qd * per;
        p = n_tiles - 1 - qd;
        bh = rem / splits;
        sp = rem - bh * splits;
        ns = splits;
      } else {
        int v = static_cast<int>(u - u_hi);
        p = splits - 2 < n_tiles - 1 ? splits - 2 : n_tiles - 1;
        while (p > 0 && v >= BH * (p + 1)) {
          v -= BH * (p + 1);
          --p;
        }
        ns = p + 1;
        bh = v / ns;
        sp = v - bh * ns;
      }
      nkv = p + 1;
    }
    kb = static_cast<int>(static_cast<long long>(sp) * nkv / ns);
    ke = static_cast<int>(static_cast<long long>(sp + 1) * nkv / ns);
  }
};

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_cl(bar, parity)) {
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

// P~ = 2^(s c - m) for one 32-column chunk of a row, as bf16 pairs into
// w[16]; adds the fp32 values to `sum` (packed pair).
__device__ __forceinline__ void softmax_chunk(const uint32_t (&r)[32], uint64_t c2, uint64_t nm2,
                                              uint64_t& sum, uint32_t (&w)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint64_t arg = f2_fma(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])),
                                c2, nm2);
    float a, b;
    f2_unpack(arg, a, b);
    a = ex2(a);
    b = ex2(b);
    w[i] = pack_bf16(a, b);
    sum = f2_add(sum, f2_pack(a, b));
  }
}

// The same for E4M3 P~: 32 columns -> 8 words of four codes at w[OFF..OFF+8).
template <int OFF>
__device__ __forceinline__ void softmax_chunk_e4m3(const uint32_t (&r)[32], uint64_t c2,
                                                   uint64_t nm2, uint64_t& sum,
                                                   uint32_t (&w)[16]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint64_t a01 = f2_fma(
        f2_pack(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1])), c2, nm2);
    const uint64_t a23 = f2_fma(
        f2_pack(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])), c2, nm2);
    float x0, x1, x2, x3;
    f2_unpack(a01, x0, x1);
    f2_unpack(a23, x2, x3);
    x0 = ex2(x0);
    x1 = ex2(x1);
    x2 = ex2(x2);
    x3 = ex2(x3);
    w[OFF + i] = pack_e4m3x4(x0, x1, x2, x3);
    sum = f2_add(sum, f2_pack(x0, x1));
    sum = f2_add(sum, f2_pack(x2, x3));
  }
}

// bf16(x) - x: the rounding error the P~ V product sees for value x.
__device__ __forceinline__ float bf16_round_err(float x) {
  const uint32_t pw = pack_bf16(x, 0.f);
  return __uint_as_float(pw << 16) - x;
}

// Row maximum of 32 columns (masked entries are -inf).
__device__ __forceinline__ float max32(const uint32_t (&r)[32]) {
  float a = __uint_as_float(r[0]), b = __uint_as_float(r[1]);
#pragma unroll
  for (int c = 2; c < 30; c += 4) {
    a = fmax3(a, __uint_as_float(r[c]), __uint_as_float(r[c + 1]));
    b = fmax3(b, __uint_as_float(r[c + 2]), __uint_as_float(r[c + 3]));
  }
  return fmax3(a, b, fmaxf(__uint_as_float(r[30]), __uint_as_float(r[31])));
}

}  // namespace pair

// SPLIT: units cover key-block ranges (Sched) and the epilogue writes each
// unit's normalised partial O~ (fp32, [splits][BH][N][D]) and partial L
// ([splits][BH][N]) instead of O and L; fa_splitkv_combine_kernel merges them.
// FP8: E4M3 inputs (tmV maps V keys-last), descale_{q,k,v} [BH] fp32.
template <int D, bool CAUSAL, bool SPLIT, bool FP8 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair::kThreads, 1)
    fa_fwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmO, __nv_bfloat16* __restrict__ O,
                       float* __restrict__ Lse, float* __restrict__ part_o,
                       float* __restrict__ part_l, int splits, DevError* __restrict__ err, int N,
                       int BH, float c_log2, unsigned long long timeout_ns, int head_group,
                       int negate_s, const float* __restrict__ descale_q = nullptr,
                       const float* __restrict__ descale_k = nullptr,
                       const float* __restrict__ descale_v = nullptr) {
  static_assert(!FP8 || !SPLIT, "the 8-bit variant is one-pass");
  using namespace pair;
  using Ly = Layout;
  constexpr int S = kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  uint32_t cl, n_cl;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(cl));
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(n_cl));

  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + Ly::kAbort);
  float4* s_stats = reinterpret_cast<float4*>(gbase + Ly::kStats);
  const uint32_t bar_qfull = base + Ly::kBarQFull, bar_qempty = base + Ly::kBarQEmpty;
  const uint32_t bar_kvfull = base + Ly::kBarKVFull, bar_kvempty = base + Ly::kBarKVEmpty;
  const uint32_t bar_ofinal = base + Ly::kBarOFinal, bar_ofree = base + Ly::kBarOFree;
  const uint32_t bar_stats = base + Ly::kBarStats;
  const uint32_t bar_fin = base + Ly::kBarFin;
  const uint32_t bar_pviss = base + Ly::kBarPvIss;

  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_qfull + 8 * b, 1);
      // the unit's last S MMA (commit) and the 4 epilogue warps, which stage
      // the unit's O in the Q buffer for a TMA store
      mbar_init(bar_qempty + 8 * b, 1 + 4);
    }
    // A K stage's full barrier also takes the 16 softmax warps' (both CTAs)
    // "S(b-1) read" arrivals, a V stage's the "P~(b) written" arrivals: one
    // wait then covers everything an S or PV MMA needs. K(0) has no S before
    // it, so its 16 arrivals are made here.
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_kvfull + 8 * s, 1 + 16);
      mbar_init(bar_kvempty + 8 * s, 1);
    }
    mbar_arrive_n(bar_kvfull, 16);
    mbar_init(bar_ofinal, 1);
    mbar_init(bar_ofree, 8);     // 4 epilogue warps x 2 CTAs
    // Two statistics barriers, unit u on barrier u & 1: a unit with one key
    // block can complete before the epilogue has waited for the previous
    // unit's statistics, so one barrier could run two phases ahead of that
    // wait.  Barrier u & 1 completes again only for unit u + 2, whose Q load
    // needs the Q buffer that the epilogue of unit u releases.
    mbar_init(bar_stats, 8);
    mbar_init(bar_stats + 8, 8);
    mbar_init(bar_fin, 1);
    mbar_init(bar_fin + 8, 1);
    mbar_init(bar_pviss, 1);
    mbar_init(bar_pviss + 8, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 13) {
    tmem_alloc_pair(base + Ly::kTmemSlot, 512);
    tmem_relinquish_pair();
  }
  if (tid == 32 * 12) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // both CTAs' barriers and TMEM exist before any remote use
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + Ly::kTmemSlot);

  const WaitCtx wc{abort_flag, err, timeout_ns};
  const int n_kblk = (N + kKeys - 1) / kKeys;
  Sched sch;
  sch.BH = BH;
  sch.n_tiles = n_kblk;
  sch.splits = SPLIT ? splits : 1;
  sch.n_units = static_cast<int>(Sched::count_units(BH, n_kblk, sch.splits, CAUSAL));
  sch.n_clusters = static_cast<int>(n_cl);
  sch.causal = CAUSAL;
  sch.head_group = head_group > 0 ? head_group : BH;
  const int n_rounds = sch.rounds();

  // Register split (launch: 512 threads x 128): softmax warpgroups 184,
  // epilogue 64, producer/MMA/idle 80: 2*128*184 + 128*64 + 128*80 = 65536.
  // Each warpgroup executes one setmaxnreg, with its role nested under it.
  if (warp >= 12) {
    setmaxnreg_dec80();
    if (warp == 12 && lane == 0) {
      // ------------------------------------------------ producer of Q and K
      // K and V never share a ring stage: K(g), ring index 2g, fills stage
      // 2 (g % 2) and V(g) stage 2 (g % 2) + 1, each with phase (g / 2) % 2.
      // Two threads issue them, so that a K load (free once S(g - 2) is
      // done) never queues behind a V load, which waits for PV(g - 2).
      long long n_k = 0;   // K blocks issued (all units)
      int uidx = 0;        // units whose Q has been issued
      bool ok = true;
      // Q is double-buffered: unit uidx uses buffer uidx & 1, free once the
      // last S MMA of unit uidx - 2 has completed (a fresh barrier passes the
      // parity-1 wait at once) and the epilogue has stored that unit's O
      // from it.  The next unit's Q is issued early, from the third K block
      // of the current unit on, as soon as its buffer is free (tested
      // without waiting; waited for only at the unit's last K block), so
      // that it neither queues in front of the next unit's first K block
      // nor holds up the current unit's K loads.
      // Returns 1 once issued, 0 if the buffer is still busy (block false),
      // -1 if the wait gave up.
      auto issue_q = [&](int u_q, bool block) -> int {
        int bh_q, p_q, sp_q, kb_q, ke_q;
        sch.template decode<SPLIT>(u_q, bh_q, p_q, sp_q, kb_q, ke_q);
        const int qb = uidx & 1;
        const uint32_t qf = bar_qfull + 8 * qb;
        const uint32_t qe = bar_qempty + 8 * qb, qpar = ((uidx >> 1) & 1) ^ 1u;
        if (!block && !mbar_test_wait(qe, qpar)) return 0;
        if (block && !mbar_wait(qe, qpar, wc, kSiteLoadQ, u_q)) return -1;
        const uint32_t lq = mapa_shared(qf, 0);
        if constexpr (FP8) {
          // one box: 128 rows x 128 one-byte columns
          if (leader) mbar_arrive_expect_tx(qf, 2 * 16384);
          tma_load_3d_pair(base + Ly::kQ + qb * kTile, &tmQ, lq, 0,
                           p_q * kKeys + static_cast<int>(rank) * kRows, bh_q);
        } else {
          if (leader) mbar_arrive_expect_tx(qf, 2 * (D / 64) * 16384);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d_pair(base + Ly::kQ + qb * kTile + c * 16384, &tmQ, lq, c * 64,
                             p_q * kKeys + static_cast<int>(rank) * kRows, bh_q);
        }
        ++uidx;
        return 1;
      };
      int q_ahead = -1;  // round whose unit's Q was issued ahead
      for (int k = 0; k < n_rounds && ok; ++k) {
        const int u = sch.unit_of(static_cast<int>(cl), k);
        if (u < 0) continue;
        int bh, p, sp, kb, ke;
        sch.template decode<SPLIT>(u, bh, p, sp, kb, ke);
        const int nkv = ke - kb;
        if (q_ahead != k && issue_q(u, true) < 0) {
          ok = false;
          break;
        }
        const int u_next = k + 1 < n_rounds ? sch.unit_of(static_cast<int>(cl), k + 1) : -1;
        const int q_from = nkv > 2 ? 2 : nkv - 1;  // first K block after which the next Q may go
        for (int j = 0; j < nkv && ok; ++j) {
          const int stage = 2 * static_cast<int>(n_k & 1);
          const uint32_t phase = static_cast<uint32_t>((n_k >> 1) & 1);
          if (!mbar_wait(bar_kvempty + 8 * stage, phase ^ 1u, wc, kSiteLoadKV, u)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_kvfull + 8 * stage;
          const uint32_t lfb = mapa_shared(fb, 0);
          const uint32_t dst = base + Ly::kRing + stage * kTile;
          // this CTA's half of K(j): D/64 boxes of 128 keys x 64 columns
          // (8-bit: one box of 128 keys x 128 bytes); keys beyond N read as 0
          if constexpr (FP8) {
            if (leader) mbar_arrive_expect_tx(fb, 2 * 16384);
            tma_load_3d_pair(dst, &tmK, lfb, 0,
                             (kb + j) * kKeys + static_cast<int>(rank) * kHalfKeys, bh);
          } else {
            if (leader) mbar_arrive_expect_tx(fb, 2 * (D / 64) * 16384);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d_pair(dst + c * 16384, &tmK, lfb, c * 64,
                               (kb + j) * kKeys + static_cast<int>(rank) * kHalfKeys, bh);
          }
          ++n_k;
          if (u_next >= 0 && q_ahead != k + 1 && j >= q_from) {
            const int r = issue_q(u_next, j == nkv - 1);
            if (r < 0) {
              ok = false;
              break;
            }
            if (r > 0) q_ahead = k + 1;
          }
        }
      }
      constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
      if (leader) {
        // Every fill completes on the even CTA's barriers (bytes of both
        // CTAs): wait (bounded) until each K stage's last fill has landed.
        for (int s = 0; s < 2; ++s) {  // K(g) with g % 2 == s in stage 2 s
          const long long cnt = (n_k + 1 - s) / 2;
          if (cnt > 0)
            drain_wait(bar_kvfull + 8 * (2 * s), static_cast<uint32_t>((cnt - 1) & 1), kDrainNs);
        }
        for (int b = 1; b <= 2 && b <= uidx; ++b) {  // the last load of each Q buffer
          const int ub = uidx - b;
          drain_wait(bar_qfull + 8 * (ub & 1), static_cast<uint32_t>((ub >> 1) & 1), kDrainNs);
        }
      } else if (!ok) {
        // The odd CTA cannot observe its own fills; after an abort give any
        // copy still in flight time to land before the CTA may exit.
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < kDrainNs) {
        }
      }
    } else if (warp == 15 && lane == 0) {
      // ----------------------------------------------------- producer of V
      long long n_v = 0;  // V blocks issued (all units)
      bool ok = true;
      for (int k = 0; k < n_rounds && ok; ++k) {
        const int u = sch.unit_of(static_cast<int>(cl), k);
        if (u < 0) continue;
        int bh, p, sp, kb, ke;
        sch.template decode<SPLIT>(u, bh, p, sp, kb, ke);
        const int nkv = ke - kb;
        for (int j = 0; j < nkv; ++j) {
          const int stage = 2 * static_cast<int>(n_v & 1) + 1;
          const uint32_t phase = static_cast<uint32_t>((n_v >> 1) & 1);
          if (!mbar_wait(bar_kvempty + 8 * stage, phase ^ 1u, wc, kSiteLoadKV, u)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_kvfull + 8 * stage;
          const uint32_t lfb = mapa_shared(fb, 0);
          const uint32_t dst = base + Ly::kRing + stage * kTile;
          if constexpr (FP8) {
            // this CTA's 64 rows of V^T (head-dim indices 64 rank ..) x 256
            // keys, as two boxes of 128 keys; keys beyond N read as zeros
            if (leader) mbar_arrive_expect_tx(fb, 2 * 16384);
#pragma unroll
            for (int hb = 0; hb < 2; ++hb)
              tma_load_3d_pair(dst + hb * 8192, &tmV, lfb, (kb + j) * kKeys + hb * 128,
                               static_cast<int>(rank) * 64, bh);
          } else {
            // one box of 256 keys x 64 columns (columns 64..127 for the odd
            // CTA; beyond a 64-wide head they read as zeros and only pad the
            // PV MMA)
            if (leader) mbar_arrive_expect_tx(fb, 2 * kTile);
            tma_load_3d_pair(dst, &tmV, lfb, static_cast<int>(rank) * 64, (kb + j) * kKeys, bh);
          }
          ++n_v;
        }
      }
      constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
      if (leader) {
        for (int s = 0; s < 2; ++s) {  // V(g) with g % 2 == s in stage 2 s + 1
          const long long cnt = (n_v + 1 - s) / 2;
          if (cnt > 0)
            drain_wait(bar_kvfull + 8 * (2 * s + 1), static_cast<uint32_t>((cnt - 1) & 1),
                       kDrainNs);
        }
      } else if (!ok) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < kDrainNs) {
        }
      }
    } else if (warp == 13 && lane == 0 && leader) {
      // ------------------------------------------------------ S MMA issuer
      // S and PV GEMMs are issued by two threads: they touch disjoint TMEM
      // columns (S vs P~ and O~) and may interleave in the tensor pipe, and
      // each thread's waits and commits then overlap the other's queued MMAs.
      // negate_s: S' = (-Q) K^T (instruction-descriptor bit 13 negates A), so
      // that a negative scale becomes the positive constant c_log2 on S'
      const uint32_t kIdescS =
          (FP8 ? idesc_e4m3_f32(256, kKeys) : idesc_bf16_f32(256, kKeys, false)) |
          (negate_s ? kIdescNegateA : 0u);
      const uint32_t tS = tmem + kColS;
      long long ring = 0;  // ring index of K(j): 2 per block
      int uidx = 0;
      bool ok = true;
      for (int k = 0; k < n_rounds && ok; ++k) {
        const int u = sch.unit_of(static_cast<int>(cl), k);
        if (u < 0) continue;
        int bh, p, sp, kb, ke;
        sch.template decode<SPLIT>(u, bh, p, sp, kb, ke);
        const int nkv = ke - kb;
        const int qb = uidx & 1;
        const uint64_t dQ = sw128_desc(base + Ly::kQ + qb * kTile, 16, 1024);
        if (!mbar_wait_cl(bar_qfull + 8 * qb, (uidx >> 1) & 1, wc, kSiteMmaQ, u)) {
          ok = false;
          break;
        }
        for (int j = 0; j < nkv; ++j, ring += 2) {
          // K(j) landed and both CTAs have read S(j-1) (one barrier)
          const int kst = static_cast<int>(ring % S);
          if (!mbar_wait_cl(bar_kvfull + 8 * kst, static_cast<uint32_t>((ring / S) & 1), wc,
                            kSiteMmaKV, static_cast<unsigned>(ring))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dK = sw128_desc(base + Ly::kRing + kst * kTile, 16, 1024);
          // S(g) enters the tensor pipe behind every MMA of PV(g - 2): the
          // PV product the softmax waits for next completes first
          {
            const long long gs = ring / 2;
            if (gs >= 2 && !mbar_wait(bar_pviss + 8 * ((gs - 2) & 1),
                                      static_cast<uint32_t>(((gs - 2) >> 1) & 1), wc, kSiteMmaKV,
                                      static_cast<unsigned>(ring))) {
              ok = false;
              break;
            }
          }
          if constexpr (FP8) {
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk)  // 32 bytes of the 128-byte rows each
              mma_pair_ss_f8(tS, dQ + 2 * kk, dK + 2 * kk, kIdescS, kk > 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
              mma_pair_ss(tS, dQ + off, dK + off, kIdescS, kk > 0 ? 1u : 0u);
            }
          }
          // one commit: frees K's stage and tells the softmax that S is ready
          tc_commit_pair(bar_kvempty + 8 * kst, kBoth);
          if (j == nkv - 1) tc_commit_pair(bar_qempty + 8 * qb, kBoth);  // last use of Q
        }
        ++uidx;
      }
      constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
      tc_commit_pair(bar_fin, 0x1);
      drain_wait(bar_fin, 0, kDrainNs);
    } else if (warp == 14 && lane == 0 && leader) {
      // ----------------------------------------------------- PV MMA issuer
      constexpr uint32_t kIdescPV = FP8 ? idesc_e4m3_f32(256, kPVN) : idesc_bf16_f32(256, kPVN, true);
      const uint32_t tP = tmem + kColP, tO = tmem + kColO;
      long long ring = 1;  // ring index of V(j): 2 per block
      int uidx = 0;
      bool ok = true;
      for (int k = 0; k < n_rounds && ok; ++k) {
        const int u = sch.unit_of(static_cast<int>(cl), k);
        if (u < 0) continue;
        int bh, p, sp, kb, ke;
        sch.template decode<SPLIT>(u, bh, p, sp, kb, ke);
        const int nkv = ke - kb;
        for (int j = 0; j < nkv; ++j, ring += 2) {
          // a unit's first PV overwrites O~: the epilogue must have read it
          if (j == 0 && uidx > 0 &&
              !mbar_wait_cl(bar_ofree, (uidx - 1) & 1, wc, kSiteMmaOFree, uidx)) {
            ok = false;
            break;
          }
          // V(j) landed and both CTAs have written P~(j) (one barrier)
          const int vst = static_cast<int>(ring % S);
          if (!mbar_wait_cl(bar_kvfull + 8 * vst, static_cast<uint32_t>((ring / S) & 1), wc,
                            kSiteMmaKV, static_cast<unsigned>(ring))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if constexpr (FP8) {
            // B = V^T K-major (keys contiguous): 32 keys per instruction, 128
            // keys per 8 KB box; A = P~ codes, 4 per TMEM column
            const uint64_t dV = sw128_desc(base + Ly::kRing + vst * kTile, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kKeys / 32; ++kk)
              // P~(g) in buffer g & 1 (two 64-column buffers)
              mma_pair_ts_f8(tO, tP + static_cast<uint32_t>(((ring - 1) / 2) & 1) * 64 + kk * 8,
                             dV + static_cast<uint32_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4),
                             kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
          } else {
            const uint64_t dV = sw128_desc(base + Ly::kRing + vst * kTile, 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk)
              mma_pair_ts(tO, tP + kk * 8, dV + static_cast<uint32_t>(kk * (2048 >> 4)), kIdescPV,
                          (j > 0 || kk > 0) ? 1u : 0u);
          }
          mbar_arrive(bar_pviss + 8 * (((ring - 1) / 2) & 1));  // every MMA of PV(g) issued
          // one commit: frees V's stage and tells the softmax that PV is done
          tc_commit_pair(bar_kvempty + 8 * vst, kBoth);
          if (j == nkv - 1) tc_commit_pair(bar_ofinal, kBoth);
        }
        ++uidx;
      }
      constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
      tc_commit_pair(bar_fin + 8, 0x1);
      drain_wait(bar_fin + 8, 0, kDrainNs);
    }
    // other lanes of warps 12-15 and the odd CTA's warps 13-14 idle
  } else if (warp < 8) {
    setmaxnreg_inc184();
    // ------------------------------------------------------------ softmax
    // Each warp owns 16 rows (TMEM lanes) of its lane quarter and all keys of
    // a block: thread t < 16 holds keys [0, 128) of row t, thread t + 16 keys
    // [128, 256) of the same row (16x32bx2 TMEM accesses), so a row reduction
    // is one shuffle between t and t ^ 16.
    const int h = lane >> 4;                                  // key half
    const int r = (warp & 3) * 32 + (warp >> 2) * 16 + (lane & 15);  // row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32 + (warp >> 2) * 16) << 16;
    const uint32_t tS = tmem + kColS + lane_off;   // + 128 columns for the upper half-warp
    const uint32_t tP = tmem + kColP + lane_off;   // + 64
    const uint32_t tO = tmem + kColO + lane_off;   // + 64
    const uint32_t l_kvfull = mapa_shared(bar_kvfull, 0);  // leader's ring barriers
    uint32_t g = 0;  // blocks processed so far (all units)
    int uidx = 0;
    bool ok = true;
    for (int k = 0; k < n_rounds && ok; ++k) {
      const int u = sch.unit_of(static_cast<int>(cl), k);
      if (u < 0) continue;
      int bh, p, sp, kb, ke;
      sch.template decode<SPLIT>(u, bh, p, sp, kb, ke);
      const int nkv = ke - kb;
      const int qrow = p * kKeys + static_cast<int>(rank) * kRows + r;
      // exponent constant: scale log2(e), times the descales of Q and K for
      // 8-bit codes (kept a normal float so that -inf * c stays -inf)
      float cu = c_log2;
      if constexpr (FP8) cu = fmaxf(c_log2 * __ldg(descale_q + bh) * __ldg(descale_k + bh), 1.17549435e-38f);
      const uint64_t c2 = f2_pack(cu, cu);
      float m_ref = -INFINITY;  // reference maximum of s * c (base-2 units)
      float l_run = 0.f;        // sum of fp32 2^(s c - m_ref), this key half
      float corr_run = 0.f;     // rounding error of each block's largest P~, this key half
      for (int j = 0; j < nkv; ++j) {
        // S(g) done = the completion that frees K(g)'s ring stage (ring index
        // 2g). Its next completion needs this warp's own later arrival, so the
        // parity wait cannot alias.
        ok = mbar_wait(bar_kvempty + 8 * ((2 * g) % S), ((2 * g) / S) & 1, wc, kSiteSoftS, u);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the reducing loads also return each chunk's maximum
        uint32_t r0[32], r1[32], r2[32], r3[32];
        float hm0, hm1, hm2, hm3;
        tmem_ldred16x2_max32<kHalfKeys>(tS + 0, r0, hm0);
        tmem_ldred16x2_max32<kHalfKeys>(tS + 32, r1, hm1);
        tmem_ldred16x2_max32<kHalfKeys>(tS + 64, r2, hm2);
        tmem_ldred16x2_max32<kHalfKeys>(tS + 96, r3, hm3);
        tmem_ldred_wait32(r0, hm0);
        tmem_ldred_dep32(r1, hm1);
        tmem_ldred_dep32(r2, hm2);
        tmem_ldred_dep32(r3, hm3);
        const int jb = kb + j;  // key block index in the head
        const int kbase = jb * kKeys + h * kHalfKeys;
        float mx = fmaxf(fmaxf(hm0, hm1), fmaxf(hm2, hm3));
        if ((CAUSAL && jb == p) || (jb * kKeys + kKeys > N)) {
          const int last = CAUSAL ? min(N - 1, qrow) : N - 1;  // last visible key
          constexpr uint32_t kNegInf = 0xff800000u;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (kbase + c > last) r0[c] = kNegInf;
            if (kbase + 32 + c > last) r1[c] = kNegInf;
            if (kbase + 64 + c > last) r2[c] = kNegInf;
            if (kbase + 96 + c > last) r3[c] = kNegInf;
          }
          // the loads' maxima included masked keys: take the maximum again
          mx = fmaxf(fmaxf(max32(r0), max32(r1)), fmaxf(max32(r2), max32(r3)));
        }
        // row maximum over both key halves: one shuffle with the partner thread
        const float m_blk = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16)) * cu;
        // S(j) is in registers: the leader may compute the next S into TMEM
        // (arrival on the full barrier of the next block's K stage).  Relaxed
        // in both CTAs: tcgen05.wait::ld and the fence below already order
        // the TMEM reads this arrival announces.  Made after the row maximum,
        // whose shuffle would otherwise wait behind it; S(j+1) still enters
        // the tensor pipe before PV(j-1) has finished.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          const uint32_t st = 8u * ((2 * g + 2) % S);
          mbar_arrive_cluster_relaxed(l_kvfull + st);
        }
        // Lazy reference update: only a jump above the threshold moves m_ref.
        const bool bump = m_blk > m_ref + (FP8 ? kLazyLog2E4m3 : kLazyLog2Bf16);  // always at j == 0
        float alpha = 1.0f;
        if (bump) {
          alpha = ex2(m_ref - m_blk);  // 0 when m_ref == -inf
          m_ref = m_blk;
          l_run *= alpha;
          corr_run *= alpha;
        }
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        const uint64_t nm2 = f2_pack(-m_use, -m_use);
        // O is normalised by l plus the rounding error of the largest P~ of
        // this key half: for a row dominated by one key that term cancels the
        // dominant rounding between numerator and denominator.  This and the
        // rescale vote are taken before the exponentials, which hide their
        // latencies.
        {
          const float pmax = ex2(fmaf(mx, cu, -m_use));
          if constexpr (FP8) corr_run += e4m3_round(pmax) - pmax;
          else corr_run += bf16_round_err(pmax);
        }
        const bool resc = j > 0 && __any_sync(0xffffffffu, bump);
        // one accumulator per chunk: four independent add chains
        uint64_t sum0 = f2_pack(0.f, 0.f), sum1 = sum0, sum2 = sum0, sum3 = sum0;
        uint32_t w0[16], w1[16], w2[16], w3[16];  // 8-bit: w0, w1 hold all 32 words
        // 8-bit: keys [0, 128) of the row first (P~ columns [0, 32)); the
        // PV wait below then sits between the two halves, and the first
        // half's TMEM store overlaps the second half's exponentials.
        if constexpr (FP8) {
          softmax_chunk_e4m3<0>(r0, c2, nm2, sum0, w0);
          softmax_chunk_e4m3<8>(r1, c2, nm2, sum1, w0);
        } else {
          softmax_chunk(r0, c2, nm2, sum0, w0);
          softmax_chunk(r1, c2, nm2, sum1, w1);
          softmax_chunk(r2, c2, nm2, sum2, w2);
          softmax_chunk(r3, c2, nm2, sum3, w3);
        }
        // PV of the previous block must be done: it reads the P~ columns and
        // accumulates into O~.  8-bit P~ has two buffers: writing P~(g) then
        // needs only PV(g-2) done, unless O~ is to be rescaled, which needs
        // every earlier PV done.
        const uint32_t pv_back = (!FP8 || resc) ? 1u : 2u;
        if (g >= pv_back) {
          // PV(g-k) done = the completion that frees V(g-k)'s stage (2(g-k) + 1)
          const uint32_t vr = 2 * (g - pv_back) + 1;
          ok = mbar_wait(bar_kvempty + 8 * (vr % S), (vr / S) & 1, wc, kSiteSoftPV, u);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        if (resc) {
          const uint64_t a2 = f2_pack(alpha, alpha);
          // head dim 64: the 64 columns of O~ in one access (threads t and
          // t + 16 take 32 each); 128: two accesses of 32 + 32 columns
          constexpr int kOSplit = D == 64 ? 32 : 64;
#pragma unroll 1
          for (int c = 0; c < D / 64; ++c) {
            uint32_t o[32];
            tmem_ld16x2_32<kOSplit>(tO + c * 32, o);
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
            tmem_st16x2_32<kOSplit>(tO + c * 32, o);
          }
        }
        if constexpr (FP8) {
          // keys [0, 128) of the row at columns [0, 32), [128, 256) at [32, 64)
          const uint32_t tPb = tP + (g & 1) * 64;
          tmem_st16x2_16<32>(tPb + 0, w0);
          softmax_chunk_e4m3<0>(r2, c2, nm2, sum2, w1);
          softmax_chunk_e4m3<8>(r3, c2, nm2, sum3, w1);
          tmem_st16x2_16<32>(tPb + 16, w1);
        } else {
          tmem_st16x2_16<64>(tP + 0, w0);
          tmem_st16x2_16<64>(tP + 16, w1);
          tmem_st16x2_16<64>(tP + 32, w2);
          tmem_st16x2_16<64>(tP + 48, w3);
        }
        const uint64_t sum = f2_add(f2_add(sum0, sum1), f2_add(sum2, sum3));
        float s_lo, s_hi;
        f2_unpack(sum, s_lo, s_hi);
        l_run += s_lo + s_hi;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {  // P~(j) written: arrival on the full barrier of V(j)'s stage
          const uint32_t st = 8u * ((2 * g + 1) % S);
          mbar_arrive_cluster_relaxed(l_kvfull + st);  // after tcgen05.wait::st + fence
        }
        ++g;
      }
      if (!ok) break;
      // Double-buffered by unit: a unit with one key block can finish before
      // the epilogue has read the previous unit's statistics.
      s_stats[((uidx & 1) * 2 + h) * kRows + r] = make_float4(m_ref, l_run, l_run + corr_run, 0.f);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_stats + 8 * (uidx & 1));
      ++uidx;
    }
  } else {
    setmaxnreg_dec64();
    // ----------------------------------------------------------- epilogue
    const int r = tid & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + kColO + lane_off;
    const uint32_t l_ofree = mapa_shared(bar_ofree, 0);
    int uidx = 0;
    bool ok = true;
    for (int k = 0; k < n_rounds && ok; ++k) {
      const int u = sch.unit_of(static_cast<int>(cl), k);
      if (u < 0) continue;
      int bh, p, sp, kb, ke;
      sch.template decode<SPLIT>(u, bh, p, sp, kb, ke);
      ok = mbar_wait(bar_ofinal, uidx & 1, wc, kSiteEpiF, u) &&
           mbar_wait(bar_stats + 8 * (uidx & 1), (uidx >> 1) & 1, wc, kSiteEpiStats, u);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float4 st0 = s_stats[((uidx & 1) * 2 + 0) * kRows + r];
      const float4 st1 = s_stats[((uidx & 1) * 2 + 1) * kRows + r];
      const float l = st0.y + st1.y;
      float inv_l = 1.0f / (st0.z + st1.z);
      if constexpr (FP8) inv_l *= __ldg(descale_v + bh);
      const int qrow = p * kKeys + static_cast<int>(rank) * kRows + r;
      const bool row_ok = qrow < N;
      const size_t prow = (static_cast<size_t>(sp) * BH + bh) * N + qrow;  // partial's row
      // bf16 O is staged in the unit's Q buffer (its last S MMA ran before
      // the PV that completed the unit): this warp's 32 rows as D/64 boxes of
      // 32 rows x 128 bytes, 128-byte swizzled as the O tensor map expects,
      // then written by TMA stores (whole rows per request; rows >= N are
      // clipped).  The TMEM reads of O~ thus end without waiting on global
      // stores.
      const int qw = warp & 3;
      const uint32_t sO = base + Ly::kQ + (uidx & 1) * kTile + qw * (D / 64) * 4096;
      uint8_t* const gO = gbase + (sO - base);
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_ld_wait32(o);
        if (c == D / 32 - 1) {
          // every TMEM read of O~ is done: the next unit may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (leader) mbar_arrive(bar_ofree); else mbar_arrive_cluster_relaxed(l_ofree);
          }
        }
        if (SPLIT) {
          if (row_ok) {
            float4* dst = reinterpret_cast<float4*>(part_o + prow * D + c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                   __uint_as_float(o[4 * i + 2]) * inv_l,
                                   __uint_as_float(o[4 * i + 3]) * inv_l);
          }
        } else {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
          uint8_t* rowp = gO + (c >> 1) * 4096 + lane * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(rowp + (((4 * (c & 1) + i) ^ (lane & 7)) << 4)) =
                make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (!SPLIT) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int row0 = p * kKeys + static_cast<int>(rank) * kRows + qw * 32;
          if (row0 < N) {  // a box wholly past N is skipped
#pragma unroll
            for (int cb = 0; cb < D / 64; ++cb) tma_store_3d(&tmO, sO + cb * 4096, 64 * cb, row0, bh);
            bulk_commit_group();
            bulk_wait_read_all();
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_qempty + 8 * (uidx & 1));  // Q buffer free for the producer
      if (row_ok) {
        const float lse = (st0.x + log2f(l)) * 0.693147180559945309f;
        if (SPLIT) part_l[prow] = lse; else Lse[static_cast<size_t>(bh) * N + qrow] = lse;
      }
      ++uidx;
    }
    if (lane == 0) bulk_wait_all();  // the last TMA stores have completed
  }

  __syncthreads();
  tc_fence_before();
  cluster_sync();  // no pair MMA, commit or remote arrival is still in flight
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}


// Merge of the split units' partial results, row by row (one warp per row):
// L = m + ln sum_s exp(L_s - m) with m = max_s L_s, and
// O = sum_s exp(L_s - L) O_s, O_s being each range's normalised output:
// the block-merge rule of the online softmax applied to whole key ranges.
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(256) fa_splitkv_combine_kernel(
    const float* __restrict__ part_o, const float* __restrict__ part_l,
    __nv_bfloat16* __restrict__ O, float* __restrict__ Lse, int BH, int N, int splits) {
  constexpr int kCols = D / 32;  // columns per lane
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<long long>(BH) * N) return;
  const int bh = static_cast<int>(row / N);
  const int i = static_cast<int>(row - static_cast<long long>(bh) * N);
  const int n_tiles = (N + pair::kKeys - 1) / pair::kKeys;
  const int p = i / pair::kKeys;
  const int avail = CAUSAL ? p + 1 : n_tiles;
  const int ns = splits < avail ? splits : avail;
  const size_t stride = static_cast<size_t>(BH) * N;  // rows per split
  float m = -INFINITY;
  for (int s = 0; s < ns; ++s) m = fmaxf(m, part_l[s * stride + row]);
  float sum = 0.f;
  for (int s = 0; s < ns; ++s) sum += expf(part_l[s * stride + row] - m);
  const float L = m + logf(sum);
  float acc[kCols];
#pragma unroll
  for (int c = 0; c < kCols; ++c) acc[c] = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float w = expf(part_l[s * stride + row] - L);
    const float* src = part_o + (s * stride + row) * D + lane * kCols;
    if (kCols == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      acc[0] += w * v.x;
      acc[1] += w * v.y;
      acc[2] += w * v.z;
      acc[3] += w * v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2*>(src);
      acc[0] += w * v.x;
      acc[1] += w * v.y;
    }
  }
  __nv_bfloat16* dst = O + row * D + lane * kCols;
  if (kCols == 4) {
    uint2 pk;
    pk.x = pack_bf16(acc[0], acc[1]);
    pk.y = pack_bf16(acc[2], acc[3]);
    *reinterpret_cast<uint2*>(dst) = pk;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16(acc[0], acc[1]);
  }
  if (lane == 0) Lse[row] = L;
}

}  // namespace fa
