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
// Three kernels, each product accumulated in tensor memory and written once:
//   fa_bwd_prep_kernel   per row -L log2 e and -D_i (fp32 planes, padded to
//                        whole 128-row blocks); the dK/dV kernel is launched
//                        behind it as a programmatic dependent
//   fa_bwd_dkdv_kernel   key-outer, persistent: a unit is (batch*head,
//                        128-key block j); it walks the 128-row query
//                        blocks i (i >= j under the causal mask) and keeps
//                        dK_j and dV_j in tensor memory
//   fa_bwd_dq_kernel     query-outer, persistent: a unit is (batch*head,
//                        128-row query block i); it walks the key blocks
//                        j (j <= i under the causal mask), recomputes S, P,
//                        dP and dS and keeps dQ_i in tensor memory
// dQ could also come out of the key-outer walk (dQ_i = dS K_j per step), but
// then 64 KB of fp32 partial dQ leave each SM per step and have to be summed
// in L2; recomputing S and dP in a second kernel costs two more products
// per block pair and writes dQ once, in bf16.
//
// fa_bwd_dkdv_kernel, per query block (tcgen05, single-SM MMAs, M = 128):
//   S^T  = K_j Q_i^T         TMEM [0,128)     (keys x queries, fp32)
//   dP^T = V_j dO_i^T        TMEM [128,256)
//   compute warps (two groups, queries 0-63 and 64-127): P^T = exp2(S^T c -
//   L log2 e) masked, written back as bf16 over the group's own S^T columns
//   (queries 0-63 at columns 0-31, 64-127 at 64-95); dS^T = P^T (dP^T - D)
//   as bf16 over dP^T's columns in the same arrangement
//   dV_j += P^T dO_i         TMEM [256,256+d)  (A from TMEM)
//   dK_j += dS^T Q_i         TMEM [256+d,256+2d)  (A from TMEM)
// Warps: 0 TMA producer of K_j, V_j (per unit) and Q_i (ring), 2 TMA producer
// of dO_i (ring), 1 MMA issuer and TMEM owner, 4-7 and 12-15 compute (one key
// row per thread, one query half per group), 8-11 write a unit's dK and dV
// (the next unit's first dV product waits for their read), 3 idle.
//
// fa_bwd_dq_kernel, per key block (single-SM MMAs, M = 128 query rows):
//   S(j)  = Q_i K_j^T        TMEM [0,128) or [128,256) (two buffers, by step
//                            parity, so S(j+1) runs while dS(j) is formed)
//   dP(j) = dO_i V_j^T       TMEM [256,384)
//   compute warps (two groups, keys 0-63 and 64-127 of the block):
//   dS = 2^(S c - L log2 e) (dP - D), masked, written as bf16 pairs over the
//   S columns the group has already read (keys 0-63 at columns 0-31, 64-127
//   at 64-95 of the buffer)
//   dQ_i += dS K_j           TMEM [384,384+d)  (A from TMEM, B = K_j
//                            MN-major)
// Issue order: S(j+1) and dP(j+1) before dQ(j), so the tensor pipe works on
// the next block while the compute warps form dS(j); dP(j+1) waits until
// the compute warps have read dP(j).  At the end of a unit four epilogue
// warps read dQ_i out of TMEM, scale it and store it as bf16; the next
// unit's first dQ product waits for that read.
// Warps: 0 TMA producer of Q_i and dO_i (per unit) and K_j (ring), 2 TMA
// producer of V_j (ring), 1 MMA issuer and TMEM owner, 4-11 compute (one
// query row per thread, one key half per group), 12-15 epilogue, 3 idle.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sm103_ptx.cuh"
#include "tmem_ldst.cuh"

namespace fa {
namespace bwd {

constexpr int kBlk = 128;       // keys per CTA and queries per step; query rows per dQ unit
constexpr int kThreads = 512;   // 16 warps (both kernels)
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256;            // dK/dV kernel
constexpr uint32_t kQColS = 0, kQColDP = 256, kQColAcc = 384;        // dQ kernel
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kUnitSlots = 4;       // ring of unit numbers handed out at run time (see put_unit)
constexpr int kUnitConsumers = 14;  // second producer, MMA thread, 8 compute + 4 output warps

enum : unsigned {
  kSiteBLoad = 211, kSiteBMmaQ = 212, kSiteBMmaDS = 214, kSiteBSoftS = 221, kSiteBKV = 232,
  kSiteBOut = 233,
  kSiteQLoadQ = 241, kSiteQLoadKV = 242, kSiteQMmaQ = 243, kSiteQMmaKV = 244,
  kSiteQMmaDP = 245, kSiteQMmaDS = 246, kSiteQMmaAcc = 247, kSiteQSoft = 251, kSiteQEpi = 252
};

// Compile-time choice between the masked and the unmasked form of a step's
// element loop.  The mask applies to one block of a unit (the diagonal, or
// the keys beyond N), decided at run time; branching to one of two compiled
// forms keeps the compares and selects out of every other block.
template <bool M>
struct MaskTag {
  static constexpr bool value = M;
};

// Shared memory of fa_bwd_dkdv_kernel: K_j and V_j for the whole walk, a ring
// of kQStages Q_i tiles (each with the block's row statistics: 128 values
// of -L log2 e, then 128 of -D) and one of kOStages dO_i tiles.
template <int D>
struct Layout {
  static constexpr int kTile = kBlk * D * 2;                 // 128 rows x D bf16
  static constexpr int kQStages = D == 128 ? 2 : 4;
  static constexpr int kOStages = D == 128 ? 2 : 4;
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  static constexpr int kQRing = 2 * kTile;
  static constexpr int kORing = kQRing + kQStages * kTile;
  static constexpr int kStat = kORing + kOStages * kTile;    // [kQStages] x 1 KB
  static constexpr int kMisc = kStat + kQStages * 1024;
  static constexpr int kBarKVFull = kMisc;
  static constexpr int kBarKVEmpty = kBarKVFull + 8;
  static constexpr int kBarQFull = kBarKVEmpty + 8;          // [kQStages]
  static constexpr int kBarQEmpty = kBarQFull + 8 * kQStages;
  static constexpr int kBarOFull = kBarQEmpty + 8 * kQStages;  // [kOStages]
  static constexpr int kBarOEmpty = kBarOFull + 8 * kOStages;
  static constexpr int kBarS = kBarOEmpty + 8 * kOStages;
  static constexpr int kBarDP = kBarS + 8;
  static constexpr int kBarP = kBarDP + 8;
  static constexpr int kBarDS = kBarP + 8;
  static constexpr int kBarAcc = kBarDS + 8;
  static constexpr int kBarAccFree = kBarAcc + 8;
  static constexpr int kBarFin = kBarAccFree + 8;
  static constexpr int kBarUFull = kBarFin + 8;              // [kUnitSlots]
  static constexpr int kBarUEmpty = kBarUFull + 8 * kUnitSlots;
  static constexpr int kUnits = kBarUEmpty + 8 * kUnitSlots; // int [kUnitSlots]
  static constexpr int kTmemSlot = kUnits + 4 * kUnitSlots;
  static constexpr int kAbort = kTmemSlot + 8;
  static constexpr int kBytes = kAbort + 8;
  static constexpr int kAlloc = kBytes + 1024;               // 1024-byte alignment slack
  static_assert(kAlloc <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");
};

// Shared memory of fa_bwd_dq_kernel: Q_i and dO_i (one buffer each), a ring
// of kKStages K_j tiles and one of kVStages V_j tiles.  K_j is read by S(j)
// and by dQ(j), the last product of a step, V_j only by dP(j): K's ring is
// the deeper one, so that the load of a later K block is under way while
// the compute warps and dQ(j) still hold the tile.
template <int D>
struct DqLayout {
  static constexpr int kTile = kBlk * D * 2;
  static constexpr int kKStages = D == 128 ? 3 : 4;
  static constexpr int kVStages = D == 128 ? 2 : 4;
  static constexpr int kQ = 0;
  static constexpr int kDO = kTile;
  static constexpr int kKRing = 2 * kTile;
  static constexpr int kVRing = kKRing + kKStages * kTile;
  static constexpr int kMisc = kVRing + kVStages * kTile;
  static constexpr int kBarQFull = kMisc;
  static constexpr int kBarQEmpty = kBarQFull + 8;
  static constexpr int kBarKFull = kBarQEmpty + 8;           // [kKStages]
  static constexpr int kBarKEmpty = kBarKFull + 8 * kKStages;
  static constexpr int kBarVFull = kBarKEmpty + 8 * kKStages;  // [kVStages]
  static constexpr int kBarVEmpty = kBarVFull + 8 * kVStages;
  static constexpr int kBarSDP = kBarVEmpty + 8 * kVStages;  // S(j) and dP(j) in TMEM
  static constexpr int kBarDPFree = kBarSDP + 8;             // compute warps have read dP(j)
  static constexpr int kBarDS = kBarDPFree + 8;              // [2] dS(j) in TMEM, by j parity
  static constexpr int kBarAcc = kBarDS + 16;                // the unit's dQ is final
  static constexpr int kBarAccFree = kBarAcc + 8;            // the epilogue has read it
  static constexpr int kBarFin = kBarAccFree + 8;
  static constexpr int kBarUFull = kBarFin + 8;              // [kUnitSlots]
  static constexpr int kBarUEmpty = kBarUFull + 8 * kUnitSlots;
  static constexpr int kUnits = kBarUEmpty + 8 * kUnitSlots; // int [kUnitSlots]
  static constexpr int kTmemSlot = kUnits + 4 * kUnitSlots;
  static constexpr int kAbort = kTmemSlot + 8;
  static constexpr int kBytes = kAbort + 8;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");
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

// Units are handed out at run time: the first producer thread of a CTA
// takes the next unit number from a global counter (atomicAdd) and publishes
// it in a ring of kUnitSlots shared-memory slots, each with a full barrier
// (its arrival) and an empty barrier (one arrival per consuming warp or
// thread); -1 ends the walk.  A CTA thus takes a new unit whenever it is
// about to run out of work, which balances walks of unequal length and lets
// the CTAs of the other backward kernel, launched beside this one, fill SMs
// as they free up.
// Publish unit u (or -1) as the CTA's k-th unit.
__device__ __forceinline__ bool put_unit(uint32_t ufull, uint32_t uempty, volatile int* slots, int k,
                                         int u, const WaitCtx& wc, unsigned site) {
  const int s = k & (kUnitSlots - 1);
  if (!mbar_wait(uempty + 8 * s, static_cast<uint32_t>(((k / kUnitSlots) & 1) ^ 1), wc, site, k))
    return false;
  slots[s] = u;
  mbar_arrive(ufull + 8 * s);
  return true;
}

// The CTA's k-th unit (-1: none left, -2: a wait gave up), read by one thread
// or, with whole_warp, by every lane of a warp (one arrival per warp).
__device__ __forceinline__ int take_unit(uint32_t ufull, uint32_t uempty, const volatile int* slots,
                                         int k, bool whole_warp, const WaitCtx& wc, unsigned site) {
  const int s = k & (kUnitSlots - 1);
  bool ok = mbar_wait(ufull + 8 * s, static_cast<uint32_t>((k / kUnitSlots) & 1), wc, site, k);
  int u = ok ? slots[s] : -2;
  if (whole_warp) {
    ok = __all_sync(0xffffffffu, ok);
    u = ok ? __shfl_sync(0xffffffffu, u, 0) : -2;
    if (ok && (threadIdx.x & 31) == 0) mbar_arrive(uempty + 8 * s);
  } else if (ok) {
    mbar_arrive(uempty + 8 * s);
  }
  return u;
}

// Causal unit order: heads in groups of G (the host picks G so that the
// streamed operands of a group -- Q and dO for the dK/dV walk, K and V for
// the dQ walk -- stay in L2), each group's walks longest first.  Unit u ->
// (head within the group-major order, rank r of the walk by length).  The
// last group may have fewer than G heads.
__device__ __forceinline__ void grouped_unit(int u, int BH, int T, int G, int& bh, int& r) {
  const int full = BH / G;
  const long long in_full = static_cast<long long>(full) * G * T;
  int g0, gs, rr;
  if (u < in_full) {
    const int per = G * T;
    g0 = (u / per) * G;
    gs = G;
    rr = u - (u / per) * per;
  } else {
    g0 = full * G;
    gs = BH - g0;
    rr = static_cast<int>(u - in_full);
  }
  r = rr / gs;
  bh = g0 + (rr - r * gs);
}

// Work unit u of the dK/dV kernel: (batch*head, key block).  Causal: key
// block j walks T - j query blocks, so the smallest j first within a group.
__device__ __forceinline__ void dkdv_unit(int u, int BH, int T, bool causal, int G, int& bh, int& j) {
  if (causal) {
    grouped_unit(u, BH, T, G, bh, j);
  } else {
    bh = u / T;
    j = u - bh * T;
  }
}

// Work unit u of the dQ kernel: (batch*head, query block).  Causal: query
// block i walks i + 1 key blocks, so the largest i first within a group.
__device__ __forceinline__ void dq_unit(int u, int BH, int T, bool causal, int G, int& bh, int& i) {
  if (causal) {
    int r;
    grouped_unit(u, BH, T, G, bh, r);
    i = T - 1 - r;
  } else {
    bh = u / T;
    i = u - bh * T;
  }
}

}  // namespace bwd

// Row statistics in two planes of [B*H][Tp] fp32 (Tp = N rounded up to a
// multiple of 128): NL = -L log2 e and ND = -D with D_i = sum_t dO_it O_it;
// rows N..Tp-1 of a head hold NL = -inf (P = 0) and ND = 0.  D / 16 lanes
// per row, each reading two 16-byte pieces of O and of dO (four loads in
// flight per thread); the blocks stride over groups of 8 * 32 / (D / 16)
// rows, so a grid sized to the SMs covers any size in even passes.  Also
// zeroes the two unit counters of the dK/dV and dQ kernels, and lets the
// dK/dV kernel, launched behind it as a programmatic dependent, start its
// set-up at once (it waits for this grid before it reads anything written
// here).
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const __nv_bfloat16* __restrict__ O,
                                                          const __nv_bfloat16* __restrict__ dO,
                                                          const float* __restrict__ Lse,
                                                          float* __restrict__ NL,
                                                          float* __restrict__ ND, int N, int Tp,
                                                          long long rows_padded,
                                                          int* __restrict__ unit_counters) {
  constexpr int kLanes = D / 16;              // lanes per row
  constexpr int kRowsPerWarp = 32 / kLanes;
  constexpr int kRowsPerBlock = 8 * kRowsPerWarp;
  griddep_launch_dependents();
  if (blockIdx.x == 0 && threadIdx.x < 2) unit_counters[threadIdx.x] = 0;
  const int lane = threadIdx.x & 31, sub = lane % kLanes;
  const int in_block = (threadIdx.x >> 5) * kRowsPerWarp + lane / kLanes;
  for (long long r0 = static_cast<long long>(blockIdx.x) * kRowsPerBlock; r0 < rows_padded;
       r0 += static_cast<long long>(gridDim.x) * kRowsPerBlock) {
    const long long prow = r0 + in_block;
    const bool live = prow < rows_padded;
    const long long bh = live ? prow / Tp : 0;
    const int q = live ? static_cast<int>(prow - bh * Tp) : N;
    const long long row = bh * N + q;
    float acc = 0.f;
    if (q < N) {
      const uint4* po = reinterpret_cast<const uint4*>(O + row * D + sub * 8);
      const uint4* pg = reinterpret_cast<const uint4*>(dO + row * D + sub * 8);
      const uint4 a0 = __ldg(po), a1 = __ldg(po + kLanes);  // elements sub*8.. and sub*8 + D/2..
      const uint4 b0 = __ldg(pg), b1 = __ldg(pg + kLanes);
      const uint32_t aw[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        acc = fmaf(__uint_as_float(aw[t] << 16), __uint_as_float(bw[t] << 16), acc);
        acc = fmaf(__uint_as_float(aw[t] & 0xffff0000u), __uint_as_float(bw[t] & 0xffff0000u), acc);
      }
    }
#pragma unroll
    for (int s = kLanes / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (live && sub == 0) {
      NL[prow] = q < N ? -Lse[row] * bwd::kLog2e : -INFINITY;
      ND[prow] = q < N ? -acc : 0.f;
    }
  }
}

// dK_j, dV_j for every (batch*head, 128-key block j): persistent, units
// taken at run time in the order of bwd::dkdv_unit.
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(bwd::kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const float* __restrict__ NL, const float* __restrict__ ND, int Tp,
                       int* __restrict__ unit_counter,
                       __nv_bfloat16* __restrict__ dK, __nv_bfloat16* __restrict__ dV,
                       DevError* __restrict__ err, int N, int BH, int head_group, float c_log2,
                       float scale, unsigned long long timeout_ns) {
  using namespace bwd;
  using Ly = Layout<D>;
  constexpr int SQ = Ly::kQStages, SO = Ly::kOStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int T = (N + kBlk - 1) / kBlk;
  const int n_units = BH * T;  // the host keeps this below 2^31

  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + Ly::kAbort);
  const uint32_t bar_kvfull = base + Ly::kBarKVFull, bar_kvempty = base + Ly::kBarKVEmpty;
  const uint32_t bar_qfull = base + Ly::kBarQFull, bar_qempty = base + Ly::kBarQEmpty;
  const uint32_t bar_ofull = base + Ly::kBarOFull, bar_oempty = base + Ly::kBarOEmpty;
  const uint32_t bar_s = base + Ly::kBarS, bar_dp = base + Ly::kBarDP;
  const uint32_t bar_p = base + Ly::kBarP, bar_ds = base + Ly::kBarDS;
  const uint32_t bar_acc = base + Ly::kBarAcc, bar_accfree = base + Ly::kBarAccFree;
  const uint32_t bar_fin = base + Ly::kBarFin;
  const uint32_t bar_ufull = base + Ly::kBarUFull, bar_uempty = base + Ly::kBarUEmpty;
  volatile int* unit_slots = reinterpret_cast<volatile int*>(gbase + Ly::kUnits);
  if (tid == 0) {
    mbar_init(bar_kvfull, 1);
    mbar_init(bar_kvempty, 1);  // commit after the unit's last S^T and dP^T
    for (int s = 0; s < SQ; ++s) {
      mbar_init(bar_qfull + 8 * s, 1);
      mbar_init(bar_qempty + 8 * s, 1);  // commit after dK(i)
    }
    for (int s = 0; s < SO; ++s) {
      mbar_init(bar_ofull + 8 * s, 1);
      mbar_init(bar_oempty + 8 * s, 1);  // commit after dV(i)
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    mbar_init(bar_p, 8);       // compute warps: P^T in TMEM
    mbar_init(bar_ds, 8);      // compute warps: dS^T in TMEM
    mbar_init(bar_acc, 1);     // the unit's dK and dV are final
    mbar_init(bar_accfree, 4); // output warps have read them
    mbar_init(bar_fin, 1);
    for (int s = 0; s < kUnitSlots; ++s) {
      mbar_init(bar_ufull + 8 * s, 1);
      mbar_init(bar_uempty + 8 * s, kUnitConsumers);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(base + Ly::kTmemSlot, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    prefetch_tensormap(&tmDO);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + Ly::kTmemSlot);
  const WaitCtx wc{abort_flag, err, timeout_ns};
  constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------- producer of K, V, Q
    // The statistics kernel ahead of this one zeroes the unit counter and
    // writes the planes the bulk copies below read: wait for it (a no-op
    // unless this grid was launched as its programmatic dependent).
    griddep_wait();
    long long g = 0;  // query blocks issued (all units)
    int uidx = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int u = atomicAdd(unit_counter, 1);
      if (u >= n_units) u = -1;
      if (!put_unit(bar_ufull, bar_uempty, unit_slots, k, u, wc, kSiteBLoad) || u < 0) break;
      int bh, j;
      dkdv_unit(u, BH, T, CAUSAL, head_group, bh, j);
      const int i0 = CAUSAL ? j : 0, n_it = T - i0;
      // K_j, V_j: one buffer, free once the previous unit's last S^T and
      // dP^T products have completed
      if (!mbar_wait(bar_kvempty, (uidx & 1) ^ 1u, wc, kSiteBLoad, u)) break;
      mbar_arrive_expect_tx(bar_kvfull, 2 * Ly::kTile);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(base + Ly::kK + c * 16384, &tmK, bar_kvfull, c * 64, j * kBlk, bh);
        tma_load_3d(base + Ly::kV + c * 16384, &tmV, bar_kvfull, c * 64, j * kBlk, bh);
      }
      ++uidx;
      for (int it = 0; it < n_it; ++it, ++g) {
        const int st = static_cast<int>(g % SQ);
        if (!mbar_wait(bar_qempty + 8 * st, static_cast<uint32_t>(((g / SQ) & 1) ^ 1), wc,
                       kSiteBLoad, u)) {
          ok = false;
          break;
        }
        const uint32_t fb = bar_qfull + 8 * st;
        mbar_arrive_expect_tx(fb, Ly::kTile + 1024);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(base + Ly::kQRing + st * Ly::kTile + c * 16384, &tmQ, fb, c * 64,
                      (i0 + it) * kBlk, bh);
        const size_t srow = static_cast<size_t>(bh) * Tp + static_cast<size_t>(i0 + it) * kBlk;
        bulk_load_1d(base + Ly::kStat + st * 1024, NL + srow, 512, fb);
        bulk_load_1d(base + Ly::kStat + st * 1024 + 512, ND + srow, 512, fb);
      }
    }
    // every copy must have landed before the CTA may exit (bounded; already
    // true unless a wait above gave up)
    if (uidx > 0) drain_wait_cta(bar_kvfull, static_cast<uint32_t>((uidx - 1) & 1), kDrainNs);
    for (long long b = g - SQ < 0 ? 0 : g - SQ; b < g; ++b)
      drain_wait_cta(bar_qfull + 8 * static_cast<int>(b % SQ), static_cast<uint32_t>((b / SQ) & 1),
                     kDrainNs);
  } else if (warp == 2 && lane == 0) {
    // ------------------------------------------------------ producer of dO
    long long g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = take_unit(bar_ufull, bar_uempty, unit_slots, k, false, wc, kSiteBLoad);
      if (u < 0) break;
      int bh, j;
      dkdv_unit(u, BH, T, CAUSAL, head_group, bh, j);
      const int i0 = CAUSAL ? j : 0, n_it = T - i0;
      for (int it = 0; it < n_it; ++it, ++g) {
        const int st = static_cast<int>(g % SO);
        if (!mbar_wait(bar_oempty + 8 * st, static_cast<uint32_t>(((g / SO) & 1) ^ 1), wc,
                       kSiteBLoad, u)) {
          ok = false;
          break;
        }
        const uint32_t fb = bar_ofull + 8 * st;
        mbar_arrive_expect_tx(fb, Ly::kTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(base + Ly::kORing + st * Ly::kTile + c * 16384, &tmDO, fb, c * 64,
                      (i0 + it) * kBlk, bh);
      }
    }
    for (long long b = g - SO < 0 ? 0 : g - SO; b < g; ++b)
      drain_wait_cta(bar_ofull + 8 * static_cast<int>(b % SO), static_cast<uint32_t>((b / SO) & 1),
                     kDrainNs);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_bf16_f32_ab(kBlk, kBlk, false, false);  // S^T, dP^T
    constexpr uint32_t kIdG = idesc_bf16_f32_ab(kBlk, D, false, true);      // dV, dK
    const uint64_t dKk = sw128_desc(base + Ly::kK, 16, 1024);       // K_j, K-major
    const uint64_t dVk = sw128_desc(base + Ly::kV, 16, 1024);       // V_j, K-major
    auto qdesc = [&](long long gg, uint32_t lbo) {
      return sw128_desc(base + Ly::kQRing + static_cast<int>(gg % SQ) * Ly::kTile, lbo, 1024);
    };
    auto odesc = [&](long long gg, uint32_t lbo) {
      return sw128_desc(base + Ly::kORing + static_cast<int>(gg % SO) * Ly::kTile, lbo, 1024);
    };
    auto issue_s = [&](long long gg, int u) -> bool {  // S^T = K_j Q_i^T
      if (!mbar_wait(bar_qfull + 8 * static_cast<int>(gg % SQ), static_cast<uint32_t>((gg / SQ) & 1),
                     wc, kSiteBMmaQ, u))
        return false;
      tc_fence_after();
      const uint64_t dQk = qdesc(gg, 16);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(tmem + kColS, dKk + kstep_kmajor(kk), dQk + kstep_kmajor(kk), kIdS, kk > 0);
      tc_commit(bar_s);
      return true;
    };
    auto issue_dp = [&](long long gg, int u) -> bool {  // dP^T = V_j dO_i^T
      if (!mbar_wait(bar_ofull + 8 * static_cast<int>(gg % SO), static_cast<uint32_t>((gg / SO) & 1),
                     wc, kSiteBMmaQ, u))
        return false;
      tc_fence_after();
      const uint64_t dOk = odesc(gg, 16);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(tmem + kColDP, dVk + kstep_kmajor(kk), dOk + kstep_kmajor(kk), kIdS, kk > 0);
      tc_commit(bar_dp);
      return true;
    };
    // Order per step i: dV(i) as soon as P^T(i) is in TMEM, S^T(i+1) right
    // behind it (the pipe reads P^T(i) before S^T(i+1) overwrites those
    // columns), dK(i) once dS^T(i) is in TMEM, then dP^T(i+1) (again behind
    // the product that reads the columns it overwrites).  The tensor pipe
    // then works on the next step while the compute warps work on this one.
    long long g = 0;
    int uidx = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = take_unit(bar_ufull, bar_uempty, unit_slots, k, false, wc, kSiteBKV);
      if (u < 0) break;
      int bh, j;
      dkdv_unit(u, BH, T, CAUSAL, head_group, bh, j);
      const int n_it = T - (CAUSAL ? j : 0);
      if (!mbar_wait(bar_kvfull, static_cast<uint32_t>(uidx & 1), wc, kSiteBKV, u)) break;
      tc_fence_after();
      if (!issue_s(g, u) || !issue_dp(g, u)) break;
      if (n_it == 1) tc_commit(bar_kvempty);
      for (int it = 0; it < n_it; ++it) {
        const long long gg = g + it;
        const bool more = it + 1 < n_it;
        if (!mbar_wait(bar_p, static_cast<uint32_t>(gg & 1), wc, kSiteBMmaDS, u)) {
          ok = false;
          break;
        }
        // the unit's first dV product overwrites the accumulators: the
        // output warps must have read the previous unit's
        if (it == 0 && uidx > 0 &&
            !mbar_wait(bar_accfree, static_cast<uint32_t>((uidx - 1) & 1), wc, kSiteBMmaDS, u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc = it > 0 ? 1u : 0u;
        const uint64_t dOmn = odesc(gg, 16384), dQmn = qdesc(gg, 16384);
#pragma unroll
        for (int kk = 0; kk < kBlk / 16; ++kk)  // dV_j += P^T dO_i (P^T columns: see the compute warps)
          mma_ts(tmem + kColDV, tmem + kColS + 64 * (kk >> 2) + 8 * (kk & 3),
                 dOmn + static_cast<uint32_t>(kk * 128), kIdG, acc | (kk > 0 ? 1u : 0u));
        tc_commit(bar_oempty + 8 * static_cast<int>(gg % SO));  // dO_i has been read
        if (more && !issue_s(gg + 1, u)) {
          ok = false;
          break;
        }
        if (!mbar_wait(bar_ds, static_cast<uint32_t>(gg & 1), wc, kSiteBMmaDS, u)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBlk / 16; ++kk)  // dK_j += dS^T Q_i (dS^T over dP^T's columns)
          mma_ts(tmem + kColDV + D, tmem + kColDP + 64 * (kk >> 2) + 8 * (kk & 3),
                 dQmn + static_cast<uint32_t>(kk * 128), kIdG, acc | (kk > 0 ? 1u : 0u));
        tc_commit(bar_qempty + 8 * static_cast<int>(gg % SQ));  // Q_i has been read
        if (more) {
          if (!issue_dp(gg + 1, u)) {
            ok = false;
            break;
          }
          if (it + 2 == n_it) tc_commit(bar_kvempty);  // the unit's last S^T and dP^T are issued
        } else {
          tc_commit(bar_acc);
        }
      }
      g += n_it;
      ++uidx;
    }
    tc_commit(bar_fin);
    drain_wait_cta(bar_fin, 0, kDrainNs);
  } else if ((warp >= 4 && warp < 8) || warp >= 12) {
    // -------------------------------------------------------------- compute
    const int qw = warp & 3;
    const int cg = warp >= 12 ? 1 : 0;              // query half of each step
    const int kr = qw * 32 + lane;                  // key row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    const uint64_t c2 = f2_pack(c_log2, c_log2);
    long long g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = take_unit(bar_ufull, bar_uempty, unit_slots, k, true, wc, kSiteBSoftS);
      if (u < 0) break;
      int bh, j;
      dkdv_unit(u, BH, T, CAUSAL, head_group, bh, j);
      const int n_it = T - (CAUSAL ? j : 0);
      const bool key_live = j * kBlk + kr < N;
      // the block of keys beyond N (if N is ragged) needs a per-key test, the
      // diagonal query block a per-element one; every other step none
      const bool tail_keys = j == T - 1 && (N % kBlk) != 0;
      for (int it = 0; it < n_it; ++it) {
        const long long gg = g + it;
        const bool diag = CAUSAL && it == 0;
        const bool masked = diag || tail_keys;
        const int qs = static_cast<int>(gg % SQ);
        const float4* s_nl = reinterpret_cast<const float4*>(gbase + Ly::kStat + qs * 1024);
        const float4* s_nd = reinterpret_cast<const float4*>(gbase + Ly::kStat + qs * 1024 + 512);
        // phase 1: P^T from S^T, written back as bf16 over S^T's first 64
        // columns; the packed values stay in registers for phase 2.  The
        // step's row statistics arrived with Q_i.
        ok = mbar_wait(bar_s, static_cast<uint32_t>(gg & 1), wc, kSiteBSoftS, u) &&
             mbar_wait(bar_qfull + 8 * qs, static_cast<uint32_t>((gg / SQ) & 1), wc, kSiteBSoftS, u);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t pk[2][16];
        auto form_p = [&](auto tag) {
          constexpr bool kMasked = decltype(tag)::value;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * cg + cc;  // 32-query chunk
            uint32_t sv[32];
            tmem_ld32(tmem + lane_off + kColS + 32 * c, sv);
            tmem_ld_wait32(sv);
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 nl = s_nl[8 * c + (e >> 2)];
              float x0, x1, x2, x3;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2,
                               f2_pack(nl.x, nl.y)),
                        x0, x1);
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3])), c2,
                               f2_pack(nl.z, nl.w)),
                        x2, x3);
              x0 = ex2(x0);
              x1 = ex2(x1);
              x2 = ex2(x2);
              x3 = ex2(x3);
              if constexpr (kMasked) {  // query 32 c + e + t of the block (local) vs key kr
                if (!key_live || (diag && kr > 32 * c + e)) x0 = 0.f;
                if (!key_live || (diag && kr > 32 * c + e + 1)) x1 = 0.f;
                if (!key_live || (diag && kr > 32 * c + e + 2)) x2 = 0.f;
                if (!key_live || (diag && kr > 32 * c + e + 3)) x3 = 0.f;
              }
              pk[cc][e >> 1] = pack_bf16(x0, x1);
              pk[cc][(e >> 1) + 1] = pack_bf16(x2, x3);
            }
            // P^T of this group's 64 queries goes inside the group's own S^T
            // columns [64 cg, 64 cg + 64), behind every column of them still to
            // be read: queries 0-63 at columns 0-31, 64-127 at columns 64-95
            tmem_st16(tmem + lane_off + kColS + 64 * cg + 16 * cc, pk[cc]);
          }
        };
        if (masked) form_p(MaskTag<true>{}); else form_p(MaskTag<false>{});
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_p);
        // phase 2: dS^T = P^T (dP^T - D), written back as bf16 over dP^T's
        // columns in the same arrangement; P is the bf16 value the dV product
        // used
        ok = mbar_wait(bar_dp, static_cast<uint32_t>(gg & 1), wc, kSiteBSoftS, u);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * cg + cc;
          uint32_t dp[32];
          tmem_ld32(tmem + lane_off + kColDP + 32 * c, dp);
          tmem_ld_wait32(dp);
          uint32_t dw[16];
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 nd = s_nd[8 * c + (e >> 2)];
            const uint32_t w0 = pk[cc][e >> 1], w1 = pk[cc][(e >> 1) + 1];
            float y0, y1, y2, y3;
            f2_unpack(f2_mul(f2_pack(__uint_as_float(w0 << 16), __uint_as_float(w0 & 0xffff0000u)),
                             f2_add(f2_pack(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])),
                                    f2_pack(nd.x, nd.y))),
                      y0, y1);
            f2_unpack(f2_mul(f2_pack(__uint_as_float(w1 << 16), __uint_as_float(w1 & 0xffff0000u)),
                             f2_add(f2_pack(__uint_as_float(dp[e + 2]), __uint_as_float(dp[e + 3])),
                                    f2_pack(nd.z, nd.w))),
                      y2, y3);
            dw[e >> 1] = pack_bf16(y0, y1);
            dw[(e >> 1) + 1] = pack_bf16(y2, y3);
          }
          tmem_st16(tmem + lane_off + kColDP + 64 * cg + 16 * cc, dw);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_ds);
      }
      g += n_it;
    }
  } else if (warp >= 8 && warp < 12) {
    // ------------------------------------------------------------- dK, dV
    const int qw = warp & 3;
    const int r = qw * 32 + lane;                   // TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    for (int uidx = 0;; ++uidx) {
      const int u = take_unit(bar_ufull, bar_uempty, unit_slots, uidx, true, wc, kSiteBOut);
      if (u < 0) break;
      int bh, j;
      dkdv_unit(u, BH, T, CAUSAL, head_group, bh, j);
      bool ok = mbar_wait(bar_acc, static_cast<uint32_t>(uidx & 1), wc, kSiteBOut, u);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
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
          if (which == 1 && c == D / 32 - 1) {  // the accumulators may be overwritten
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_accfree);
          }
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

// dQ for every (batch*head, 128-row query block): persistent, units
// taken at run time in the order of bwd::dq_unit.
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(bwd::kThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                     const float* __restrict__ NL, const float* __restrict__ ND, int Tp,
                     int* __restrict__ unit_counter,
                     __nv_bfloat16* __restrict__ dQ, DevError* __restrict__ err, int N, int BH,
                     int head_group, float c_log2, float scale, unsigned long long timeout_ns) {
  using namespace bwd;
  using Ly = DqLayout<D>;
  constexpr int SK = Ly::kKStages, SV = Ly::kVStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int T = (N + kBlk - 1) / kBlk;
  const int n_units = BH * T;  // the host keeps this below 2^31

  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + Ly::kAbort);
  const uint32_t bar_qfull = base + Ly::kBarQFull, bar_qempty = base + Ly::kBarQEmpty;
  const uint32_t bar_kfull = base + Ly::kBarKFull, bar_kempty = base + Ly::kBarKEmpty;
  const uint32_t bar_vfull = base + Ly::kBarVFull, bar_vempty = base + Ly::kBarVEmpty;
  const uint32_t bar_sdp = base + Ly::kBarSDP, bar_dpfree = base + Ly::kBarDPFree;
  const uint32_t bar_ds = base + Ly::kBarDS, bar_acc = base + Ly::kBarAcc;
  const uint32_t bar_accfree = base + Ly::kBarAccFree, bar_fin = base + Ly::kBarFin;
  const uint32_t bar_ufull = base + Ly::kBarUFull, bar_uempty = base + Ly::kBarUEmpty;
  volatile int* unit_slots = reinterpret_cast<volatile int*>(gbase + Ly::kUnits);
  if (tid == 0) {
    mbar_init(bar_qfull, 1);
    mbar_init(bar_qempty, 1);     // commit after the unit's last S and dP
    for (int s = 0; s < SK; ++s) {
      mbar_init(bar_kfull + 8 * s, 1);
      mbar_init(bar_kempty + 8 * s, 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(bar_vfull + 8 * s, 1);
      mbar_init(bar_vempty + 8 * s, 1);
    }
    mbar_init(bar_sdp, 1);
    mbar_init(bar_dpfree, 8);     // compute warps
    mbar_init(bar_ds, 8);
    mbar_init(bar_ds + 8, 8);
    mbar_init(bar_acc, 1);
    mbar_init(bar_accfree, 4);    // epilogue warps
    mbar_init(bar_fin, 1);
    for (int s = 0; s < kUnitSlots; ++s) {
      mbar_init(bar_ufull + 8 * s, 1);
      mbar_init(bar_uempty + 8 * s, kUnitConsumers);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(base + Ly::kTmemSlot, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    prefetch_tensormap(&tmDO);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + Ly::kTmemSlot);
  const WaitCtx wc{abort_flag, err, timeout_ns};

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ producer of Q, dO, K
    long long g = 0;  // key blocks issued (all units)
    int uidx = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int u = atomicAdd(unit_counter, 1);
      if (u >= n_units) u = -1;
      if (!put_unit(bar_ufull, bar_uempty, unit_slots, k, u, wc, kSiteQLoadQ) || u < 0) break;
      int bh, i;
      dq_unit(u, BH, T, CAUSAL, head_group, bh, i);
      const int nkb = CAUSAL ? i + 1 : T;
      // Q_i, dO_i: one buffer, free once the previous unit's last S and dP
      // products have completed
      if (!mbar_wait(bar_qempty, (uidx & 1) ^ 1u, wc, kSiteQLoadQ, u)) break;
      mbar_arrive_expect_tx(bar_qfull, 2 * Ly::kTile);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(base + Ly::kQ + c * 16384, &tmQ, bar_qfull, c * 64, i * kBlk, bh);
        tma_load_3d(base + Ly::kDO + c * 16384, &tmDO, bar_qfull, c * 64, i * kBlk, bh);
      }
      ++uidx;
      for (int j = 0; j < nkb; ++j, ++g) {
        const int st = static_cast<int>(g % SK);
        if (!mbar_wait(bar_kempty + 8 * st, static_cast<uint32_t>(((g / SK) & 1) ^ 1), wc,
                       kSiteQLoadKV, u)) {
          ok = false;
          break;
        }
        const uint32_t fb = bar_kfull + 8 * st;
        mbar_arrive_expect_tx(fb, Ly::kTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(base + Ly::kKRing + st * Ly::kTile + c * 16384, &tmK, fb, c * 64, j * kBlk, bh);
      }
    }
    // every copy must have landed before the CTA may exit (bounded; already
    // true unless a wait above gave up)
    constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
    if (uidx > 0) drain_wait_cta(bar_qfull, static_cast<uint32_t>((uidx - 1) & 1), kDrainNs);
    for (long long b = g - SK < 0 ? 0 : g - SK; b < g; ++b)
      drain_wait_cta(bar_kfull + 8 * static_cast<int>(b % SK), static_cast<uint32_t>((b / SK) & 1),
                     kDrainNs);
  } else if (warp == 2 && lane == 0) {
    // -------------------------------------------------------- producer of V
    long long g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = take_unit(bar_ufull, bar_uempty, unit_slots, k, false, wc, kSiteQLoadKV);
      if (u < 0) break;
      int bh, i;
      dq_unit(u, BH, T, CAUSAL, head_group, bh, i);
      const int nkb = CAUSAL ? i + 1 : T;
      for (int j = 0; j < nkb; ++j, ++g) {
        const int st = static_cast<int>(g % SV);
        if (!mbar_wait(bar_vempty + 8 * st, static_cast<uint32_t>(((g / SV) & 1) ^ 1), wc,
                       kSiteQLoadKV, u)) {
          ok = false;
          break;
        }
        const uint32_t fb = bar_vfull + 8 * st;
        mbar_arrive_expect_tx(fb, Ly::kTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(base + Ly::kVRing + st * Ly::kTile + c * 16384, &tmV, fb, c * 64, j * kBlk, bh);
      }
    }
    constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
    for (long long b = g - SV < 0 ? 0 : g - SV; b < g; ++b)
      drain_wait_cta(bar_vfull + 8 * static_cast<int>(b % SV), static_cast<uint32_t>((b / SV) & 1),
                     kDrainNs);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdSD = idesc_bf16_f32_ab(kBlk, kBlk, false, false);  // S, dP
    constexpr uint32_t kIdQ = idesc_bf16_f32_ab(kBlk, D, false, true);       // dQ
    const uint64_t dQk = sw128_desc(base + Ly::kQ, 16, 1024);
    const uint64_t dOk = sw128_desc(base + Ly::kDO, 16, 1024);
    // S(gg) into buffer gg & 1 and dP(gg); dP(gg) overwrites dP(gg - 1), so
    // it waits until the compute warps have read that
    auto issue_sdp = [&](long long gg, int u) -> bool {
      const int sk = static_cast<int>(gg % SK), sv = static_cast<int>(gg % SV);
      if (!mbar_wait(bar_kfull + 8 * sk, static_cast<uint32_t>((gg / SK) & 1), wc, kSiteQMmaKV, u))
        return false;
      tc_fence_after();
      const uint64_t dKk = sw128_desc(base + Ly::kKRing + sk * Ly::kTile, 16, 1024);
      const uint64_t dVk = sw128_desc(base + Ly::kVRing + sv * Ly::kTile, 16, 1024);
      const uint32_t sb = tmem + kQColS + static_cast<uint32_t>(gg & 1) * 128;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(sb, dQk + kstep_kmajor(kk), dKk + kstep_kmajor(kk), kIdSD, kk > 0);
      if (!mbar_wait(bar_vfull + 8 * sv, static_cast<uint32_t>((gg / SV) & 1), wc, kSiteQMmaKV, u))
        return false;
      if (gg > 0 &&
          !mbar_wait(bar_dpfree, static_cast<uint32_t>((gg - 1) & 1), wc, kSiteQMmaDP, u))
        return false;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(tmem + kQColDP, dOk + kstep_kmajor(kk), dVk + kstep_kmajor(kk), kIdSD, kk > 0);
      tc_commit(bar_sdp);
      tc_commit(bar_vempty + 8 * sv);  // V_j has been read
      return true;
    };
    long long g = 0;
    int uidx = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = take_unit(bar_ufull, bar_uempty, unit_slots, k, false, wc, kSiteQMmaQ);
      if (u < 0) break;
      int bh, i;
      dq_unit(u, BH, T, CAUSAL, head_group, bh, i);
      const int nkb = CAUSAL ? i + 1 : T;
      if (!mbar_wait(bar_qfull, static_cast<uint32_t>(uidx & 1), wc, kSiteQMmaQ, u)) break;
      tc_fence_after();
      if (!issue_sdp(g, u)) break;
      if (nkb == 1) tc_commit(bar_qempty);
      for (int j = 0; j < nkb; ++j) {
        const long long gg = g + j;
        const int sk = static_cast<int>(gg % SK);
        if (j + 1 < nkb) {
          if (!issue_sdp(gg + 1, u)) {
            ok = false;
            break;
          }
          if (j + 2 == nkb) tc_commit(bar_qempty);  // the unit's last S and dP are issued
        }
        if (!mbar_wait(bar_ds + 8 * static_cast<int>(gg & 1), static_cast<uint32_t>((gg >> 1) & 1),
                       wc, kSiteQMmaDS, u)) {
          ok = false;
          break;
        }
        // the unit's first dQ product overwrites the accumulator: the
        // epilogue must have read the previous unit's
        if (j == 0 && uidx > 0 &&
            !mbar_wait(bar_accfree, static_cast<uint32_t>((uidx - 1) & 1), wc, kSiteQMmaAcc, u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sb = tmem + kQColS + static_cast<uint32_t>(gg & 1) * 128;
        const uint64_t dKmn = sw128_desc(base + Ly::kKRing + sk * Ly::kTile, 16384, 1024);
#pragma unroll
        for (int kk = 0; kk < kBlk / 16; ++kk)  // dQ_i += dS K_j (dS columns: see the compute warps)
          mma_ts(tmem + kQColAcc, sb + 64 * (kk >> 2) + 8 * (kk & 3),
                 dKmn + static_cast<uint32_t>(kk * 128), kIdQ, (j > 0 || kk > 0) ? 1u : 0u);
        tc_commit(bar_kempty + 8 * sk);  // K_j has been read
        if (j == nkb - 1) tc_commit(bar_acc);
      }
      g += nkb;
      ++uidx;
    }
    tc_commit(bar_fin);
    drain_wait_cta(bar_fin, 0, 50ull * 1000 * 1000);
  } else if (warp >= 4 && warp < 12) {
    // -------------------------------------------------------------- compute
    const int grp = (warp - 4) >> 2;                // keys [64 grp, 64 grp + 64) of a block
    const int qw = warp & 3;
    const int rl = qw * 32 + lane;                  // query row in the unit = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    const uint64_t c2 = f2_pack(c_log2, c_log2);
    long long g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = take_unit(bar_ufull, bar_uempty, unit_slots, k, true, wc, kSiteQSoft);
      if (u < 0) break;
      int bh, i;
      dq_unit(u, BH, T, CAUSAL, head_group, bh, i);
      const int nkb = CAUSAL ? i + 1 : T;
      // rows beyond N have NL = -inf: P = 0 and dS = 0 (never stored)
      const size_t srow = static_cast<size_t>(bh) * Tp + static_cast<size_t>(i) * kBlk + rl;
      const float nl = NL[srow], nd = ND[srow];
      const uint64_t nl2 = f2_pack(nl, nl), nd2 = f2_pack(nd, nd);
      for (int j = 0; j < nkb; ++j) {
        const long long gg = g + j;
        ok = mbar_wait(bar_sdp, static_cast<uint32_t>(gg & 1), wc, kSiteQSoft, u);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sb = tmem + lane_off + kQColS + static_cast<uint32_t>(gg & 1) * 128 + 64 * grp;
        const uint32_t dpb = tmem + lane_off + kQColDP + 64 * grp;
        // the last key block holds the diagonal (causal) or the keys >= N;
        // a key of this group at offset t (0..63) is visible iff t <= lim
        const bool masked = CAUSAL ? (j == nkb - 1) : (j == nkb - 1 && (N % kBlk) != 0);
        const int lim = CAUSAL ? rl - 64 * grp : N - 1 - j * kBlk - 64 * grp;
        auto form_ds = [&](auto tag) {
          constexpr bool kMasked = decltype(tag)::value;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t sv[32], dp[32];
            tmem_ld32(sb + 32 * c, sv);
            tmem_ld32(dpb + 32 * c, dp);
            tmem_ld_wait32(sv);
            tmem_ld_dep32(dp);
            if (c == 1) {  // dP(j) is in registers: the next dP product may start
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar_dpfree);
            }
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float a, b;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), c2,
                               nl2),
                        a, b);
              a = ex2(a);
              b = ex2(b);
              if constexpr (kMasked) {
                if (32 * c + 2 * e > lim) a = 0.f;
                if (32 * c + 2 * e + 1 > lim) b = 0.f;
              }
              float x, y;
              f2_unpack(f2_mul(f2_pack(a, b),
                               f2_add(f2_pack(__uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1])),
                                      nd2)),
                        x, y);
              w[e] = pack_bf16(x, y);
            }
            // dS of keys [64 grp + 32 c, +32) as 16 bf16 pairs over S columns
            // this group has already read
            tmem_st16(sb + 16 * c, w);
          }
        };
        if (masked) form_ds(MaskTag<true>{}); else form_ds(MaskTag<false>{});
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_ds + 8 * static_cast<int>(gg & 1));
      }
      g += nkb;
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------- epilogue
    const int qw = warp & 3;
    const int rl = qw * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    for (int uidx = 0;; ++uidx) {
      const int u = take_unit(bar_ufull, bar_uempty, unit_slots, uidx, true, wc, kSiteQEpi);
      if (u < 0) break;
      int bh, i;
      dq_unit(u, BH, T, CAUSAL, head_group, bh, i);
      bool ok = mbar_wait(bar_acc, static_cast<uint32_t>(uidx & 1), wc, kSiteQEpi, u);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int row = i * kBlk + rl;
      __nv_bfloat16* out = dQ + (static_cast<size_t>(bh) * N + row) * D;
#pragma unroll 1
      for (int h = 0; h < D / 64; ++h) {
        uint32_t v0[32], v1[32];
        tmem_ld32(tmem + lane_off + kQColAcc + 64 * h, v0);
        tmem_ld32(tmem + lane_off + kQColAcc + 64 * h + 32, v1);
        tmem_ld_wait32(v0);
        tmem_ld_dep32(v1);
        if (h == D / 64 - 1) {  // the accumulator may be overwritten
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_accfree);
        }
        if (row < N) {
          uint4* dst = reinterpret_cast<uint4*>(out + 64 * h);
#pragma unroll
          for (int t = 0; t < 4; ++t)
            dst[t] = make_uint4(
                pack_bf16(__uint_as_float(v0[8 * t]) * scale, __uint_as_float(v0[8 * t + 1]) * scale),
                pack_bf16(__uint_as_float(v0[8 * t + 2]) * scale, __uint_as_float(v0[8 * t + 3]) * scale),
                pack_bf16(__uint_as_float(v0[8 * t + 4]) * scale, __uint_as_float(v0[8 * t + 5]) * scale),
                pack_bf16(__uint_as_float(v0[8 * t + 6]) * scale, __uint_as_float(v0[8 * t + 7]) * scale));
#pragma unroll
          for (int t = 0; t < 4; ++t)
            dst[4 + t] = make_uint4(
                pack_bf16(__uint_as_float(v1[8 * t]) * scale, __uint_as_float(v1[8 * t + 1]) * scale),
                pack_bf16(__uint_as_float(v1[8 * t + 2]) * scale, __uint_as_float(v1[8 * t + 3]) * scale),
                pack_bf16(__uint_as_float(v1[8 * t + 4]) * scale, __uint_as_float(v1[8 * t + 5]) * scale),
                pack_bf16(__uint_as_float(v1[8 * t + 6]) * scale, __uint_as_float(v1[8 * t + 7]) * scale));
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
