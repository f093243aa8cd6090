// C ABI of the exact attention forward pass (declared in include/fa_fwd.h):
// argument validation, TMA tensor-map encoding and kernel launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa_bwd.cuh"
#include "fa_fwd_small.cuh"
#include "fa_fp8.cuh"
#include "fa_fwd.h"
#include "fa_fwd_pair.cuh"
#include "fa_unfused.cuh"

namespace fa {

__device__ DevError g_dev_error;

// Fixed scratch of the no-allocation split entry point: part of the module
// image, so it exists on every device the library is loaded on and costs no
// allocation call.  Shared by all calls on a device.
constexpr size_t kNoAllocScratchBytes = 64ull << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

thread_local int t_last_cuda_error = 0;
thread_local unsigned int t_last_record[4] = {0, 0, 0, 0};

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return FA_ERR_CUDA;
}

int cuda_fail_drv(CUresult r) {
  t_last_cuda_error = static_cast<int>(r);
  return FA_ERR_CUDA;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Encoded 3-D tensor maps (128-byte swizzle, no interleave, zero fill),
// cached by every argument of the encode call, so that repeated calls on the
// same buffers and shapes skip the encoding.  A map holds only an address
// and a shape: an entry stays correct whatever later happens to the memory
// it names.  4-way set associative, 16 sets, least recently used way
// replaced; thread-safe.
struct TmapKey {
  const void* base;
  cuuint64_t dims[3];
  cuuint64_t strides[2];
  cuuint32_t box[3];
  int dtype;
};

struct TmapCache {
  static constexpr int kSets = 16, kWays = 4;
  std::mutex mu;
  TmapKey key[kSets][kWays];
  CUtensorMap map[kSets][kWays];
  unsigned long long used[kSets][kWays] = {};  // 0 = empty way
  unsigned long long tick = 0;
};
TmapCache g_tmaps;

int encode_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, cuuint64_t d0,
              cuuint64_t d1, cuuint64_t d2, cuuint64_t stride1, cuuint64_t stride2,
              cuuint32_t box0, cuuint32_t box1) {
  TmapKey k;
  std::memset(&k, 0, sizeof(k));  // padding bytes take part in the comparison
  k.base = base;
  k.dims[0] = d0;
  k.dims[1] = d1;
  k.dims[2] = d2;
  k.strides[0] = stride1;
  k.strides[1] = stride2;
  k.box[0] = box0;
  k.box[1] = box1;
  k.box[2] = 1;
  k.dtype = static_cast<int>(dtype);
  unsigned long long h = 1469598103934665603ull;  // FNV-1a over the key's bytes
  const unsigned char* kb = reinterpret_cast<const unsigned char*>(&k);
  for (size_t i = 0; i < sizeof(k); ++i) h = (h ^ kb[i]) * 1099511628211ull;
  const int set = static_cast<int>((h >> 32) % TmapCache::kSets);
  {
    std::lock_guard<std::mutex> lock(g_tmaps.mu);
    for (int w = 0; w < TmapCache::kWays; ++w)
      if (g_tmaps.used[set][w] && std::memcmp(&g_tmaps.key[set][w], &k, sizeof(k)) == 0) {
        *map = g_tmaps.map[set][w];
        g_tmaps.used[set][w] = ++g_tmaps.tick;
        return FA_OK;
      }
  }
  auto fn = encode_tiled();
  if (!fn) return cuda_fail(cudaErrorNotSupported);
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1, stride2};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail_drv(r);
  std::lock_guard<std::mutex> lock(g_tmaps.mu);
  int victim = 0;
  for (int w = 1; w < TmapCache::kWays; ++w)
    if (g_tmaps.used[set][w] < g_tmaps.used[set][victim]) victim = w;
  g_tmaps.key[set][victim] = k;
  g_tmaps.map[set][victim] = *map;
  g_tmaps.used[set][victim] = ++g_tmaps.tick;
  return FA_OK;
}

// [B*H, N, d] bf16 viewed as a 3-D tensor; box = 64 columns x box_rows rows
// x 1 head with 128-byte swizzle.  Rows >= N of a head read as zeros.
int encode_qkv_map(CUtensorMap* map, const void* base, long long BH, long long N, int d,
                   int box_rows = 128) {
  return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, static_cast<cuuint64_t>(d),
                   static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH),
                   static_cast<cuuint64_t>(d) * 2,
                   static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2, 64,
                   static_cast<cuuint32_t>(box_rows));
}

// E4M3 codes [B*H, N, d] (Q, K of the 8-bit forward): box = 128 one-byte
// columns x box_rows rows x 1 head, 128-byte swizzle; rows >= N read as 0,
// and so do columns >= d (d = 64: the upper half of every 128-byte row).
int encode_e4m3_rows_map(CUtensorMap* map, const void* base, long long BH, long long N, int d,
                         int box_rows) {
  return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, static_cast<cuuint64_t>(d),
                   static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH),
                   static_cast<cuuint64_t>(d),
                   static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d), 128,
                   static_cast<cuuint32_t>(box_rows));
}

// E4M3 codes of V keys-last [B*H, d, pitch] (row t = head-dim index t, keys
// contiguous): box = 128 keys x 64 rows x 1 head, 128-byte swizzle.  The
// extent along the keys is N, so keys >= N read as 0 whatever the padding
// holds.
int encode_e4m3_keys_last_map(CUtensorMap* map, const void* base, long long BH, long long N,
                              int d, long long pitch) {
  return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, static_cast<cuuint64_t>(N),
                   static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(BH),
                   static_cast<cuuint64_t>(pitch),
                   static_cast<cuuint64_t>(pitch) * static_cast<cuuint64_t>(d), 128, 64);
}

// Scores S of the unfused path, fp32 [B*H, N, pitch]: box = 32 columns (128
// bytes) x 32 rows x 1 head, for the TMA stores of the S GEMM's epilogue.
int encode_scores_map(CUtensorMap* map, void* base, long long BH, long long N, long long pitch) {
  return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, static_cast<cuuint64_t>(N),
                   static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH),
                   static_cast<cuuint64_t>(pitch) * 4,
                   static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(pitch) * 4, 32, 32);
}

// Probabilities P of the unfused path, bf16 [B*H, N, pitch]: box = 64 keys
// (128 bytes) x 128 rows x 1 head; keys >= N read as zeros.
int encode_probs_map(CUtensorMap* map, const void* base, long long BH, long long N,
                     long long pitch) {
  return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, static_cast<cuuint64_t>(N),
                   static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH),
                   static_cast<cuuint64_t>(pitch) * 2,
                   static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(pitch) * 2, 64, 128);
}

// Row pitch (keys) of the keys-last E4M3 layout: N rounded up to 16 bytes.
long long e4m3_keys_pitch(long long N) { return (N + 15) / 16 * 16; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// negative_scale_ok: the forward kernels take any finite scale (a negative
// one negates the S product's A operand); the backward does not.
int validate(const void* q, const void* k, const void* v, const void* o, const void* lse, int B,
             int H, int N, int d, float scale, int causal, bool negative_scale_ok = true) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || N <= 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (scale < 0.f && !negative_scale_ok) return FA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  const long long n_pair = (static_cast<long long>(N) + 255) / 256;
  if (BH * n_pair > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (BH * N > (1LL << 55)) return FA_ERR_UNSUPPORTED;
  const long long elems = BH * N * d;  // < 2^62 after the check above
  for (const void* p : {q, k, v, o})
    if (reinterpret_cast<uintptr_t>(p) & 15u) return FA_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return FA_ERR_MISALIGNED;
  const size_t nb = static_cast<size_t>(elems) * 2, nl = static_cast<size_t>(BH * N) * 4;
  for (const void* in : {q, k, v})
    if (overlaps(o, nb, in, nb) || overlaps(lse, nl, in, nb)) return FA_ERR_INVALID_ARG;
  if (overlaps(o, nb, lse, nl)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Head-group size of the causal one-pass order (Sched::decode).  Among the
// group sizes whose keys and values (bf16 size) fit in kGroupL2Bytes, the one
// whose static round-robin assignment (Sched::unit_of) gives the smallest
// most-loaded cluster, counting each unit as its key blocks plus a fixed
// cost of 2.5 blocks; ties go to the larger group.  The budget is far below
// the L2's 129 MB: per launch, b1h32n32768d128 causal read 1.68 GB from DRAM
// with 2-head groups (64 MB budget) and 1.14 GB with 1-head groups (16 MB),
// b2h32n8192d128 causal 663 MB with 16-head groups and 405 MB with 1-head
// groups (algorithmic reads 805 MB and 403 MB); the times were equal within
// the +-1% of an interleaved comparison.  Grouping at all (against every
// head at once, whose keys and values stream from DRAM) was 1.11-1.14x on
// b2h32n8192d128.
constexpr long long kGroupL2Bytes = 16ll << 20;

double causal_makespan(long long BH, int n_tiles, int clusters, int g) {
  const long long n = BH * n_tiles;
  const long long rounds = (n + clusters - 1) / clusters;
  double worst = 0.0;
  for (int cl = 0; cl < clusters; ++cl) {
    double tot = 0.0;
    for (long long k = 0; k < rounds; ++k) {
      const long long u = k * clusters + ((k & 1) ? (clusters - 1 - cl) : cl);
      if (u >= n) continue;
      const long long per = static_cast<long long>(g) * n_tiles;
      const long long grp = u / per;
      const long long gs = BH - grp * g < g ? BH - grp * g : g;
      const long long v = u - grp * per;
      tot += static_cast<double>(n_tiles - v / gs) + 2.5;
    }
    worst = tot > worst ? tot : worst;
  }
  return worst;
}

int pick_head_group(long long BH, int n_tiles, int clusters, long long N, int d) {
  const long long kv_head = 4ll * N * d;  // K and V of one head, bf16
  long long gmax = kGroupL2Bytes / (kv_head > 0 ? kv_head : 1);
  if (gmax >= BH) return static_cast<int>(BH);  // every head fits: no grouping
  if (gmax < 1) gmax = 1;
  if (gmax > 64) gmax = 64;
  // The model below costs about BH * n_tiles * gmax steps: bounded to 2^22
  // (a few ms, once per shape); larger shapes take the largest group.
  if (BH * n_tiles * gmax > (1ll << 22)) return static_cast<int>(gmax);
  static std::mutex mu;
  constexpr int kCache = 64;
  static long long key[4][kCache] = {};
  static int val[kCache] = {};
  static int next = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < kCache; ++i)
      if (key[0][i] == BH && key[1][i] == n_tiles && key[2][i] == clusters && key[3][i] == gmax)
        return val[i];
  }
  int best = 1;
  double best_ms = -1.0;
  for (int g = 1; g <= gmax; ++g) {
    const double ms = causal_makespan(BH, n_tiles, clusters, g);
    if (best_ms < 0.0 || ms <= best_ms) {
      best_ms = ms;
      best = g;
    }
  }
  std::lock_guard<std::mutex> lock(mu);
  const int i = next++ % kCache;
  key[0][i] = BH;
  key[1][i] = n_tiles;
  key[2][i] = clusters;
  key[3][i] = gmax;
  val[i] = best;
  return best;
}

struct DeviceInfo {
  bool pair_ready[16] = {};
  int pair_clusters[16] = {};
  bool unf_ready[4] = {};
  DevError* err = nullptr;         // this device's copy of g_dev_error
  void* noalloc_scratch = nullptr;  // this device's copy of g_noalloc_scratch
  int sms = 0;                      // multiprocessors (set by the backward's first launch)
  int prep_per_sm[2] = {};          // resident blocks per SM of the backward's statistics kernel (d 64, 128)
  bool small_ready[4] = {};         // short-sequence forward kernel configured
};

std::mutex g_setup_mu;
DeviceInfo g_dev_info[64];

// The current device, with the addresses of the module's device variables
// on it looked up once (with that device current) and kept.
int current_device(int* dev_out, DeviceInfo** info) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return FA_ERR_UNSUPPORTED;
  DeviceInfo& di = g_dev_info[dev];
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!di.err) {
      DevError* p = nullptr;
      e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_dev_error);
      if (e != cudaSuccess) return cuda_fail(e);
      di.err = p;
    }
  }
  *dev_out = dev;
  *info = &di;
  return FA_OK;
}


// The CTA-pair kernel.  Grid = 2 x (clusters that fit at once).  With SPLIT
// the units cover key-block ranges and write partials to part_o / part_l;
// the caller then launches the combine kernel.  FP8: q, k are E4M3 codes
// [B*H, N, D], v E4M3 codes keys-last [B*H, D, pitch], with descales.
// Forward for N <= 128: one 128-thread CTA per (batch, head) (see
// fa_fwd_small.cuh); launch_pair dispatches here.
template <int D, bool CAUSAL>
int launch_small(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, float scale, cudaStream_t stream) {
  using Ly = small::Layout<D>;
  auto kernel = fa_fwd_small_kernel<D, CAUSAL>;
  int dev = 0;
  DeviceInfo* dip = nullptr;
  int st = current_device(&dev, &dip);
  if (st != FA_OK) return st;
  cudaError_t e = cudaSuccess;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    bool& ready = dip->small_ready[(D == 128 ? 2 : 0) + (CAUSAL ? 1 : 0)];
    if (!ready) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::kAlloc);
      if (e != cudaSuccess) return cuda_fail(e);
      ready = true;
    }
  }
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  CUtensorMap mq, mk, mv;
  if ((st = encode_qkv_map(&mq, q, BH, N, D, small::kRows)) != FA_OK) return st;
  if ((st = encode_qkv_map(&mk, k, BH, N, D, small::kRows)) != FA_OK) return st;
  if ((st = encode_qkv_map(&mv, v, BH, N, D, small::kRows)) != FA_OK) return st;
  // as in launch_pair: a negative scale negates Q in the S product
  const int negate_s = scale < 0.f ? 1 : 0;
  float c_log2 = std::fabs(scale) * 1.4426950408889634f;
  if (!(c_log2 >= 1.17549435e-38f)) c_log2 = 1.17549435e-38f;
  const unsigned long long timeout_ns = 2000ull * 1000 * 1000;
  kernel<<<static_cast<unsigned>(BH), small::kThreads, Ly::kAlloc, stream>>>(
      mq, mk, mv, static_cast<__nv_bfloat16*>(o), lse, dip->err, N, c_log2, negate_s, timeout_ns);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

template <int D, bool CAUSAL, bool SPLIT = false, bool FP8 = false>
int launch_pair(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int N, float scale, cudaStream_t stream, float* part_o = nullptr,
                float* part_l = nullptr, int splits = 1, const float* dsq = nullptr,
                const float* dsk = nullptr, const float* dsv = nullptr) {
  if constexpr (!SPLIT && !FP8) {
    // one block of keys per row: the short-sequence kernel
    if (N <= small::kRows) return launch_small<D, CAUSAL>(q, k, v, o, lse, B, H, N, scale, stream);
  }
  using Ly = pair::Layout;
  auto kernel = fa_fwd_pair_kernel<D, CAUSAL, SPLIT, FP8>;
  const int smem = Ly::kAlloc;
  int dev = 0;
  DeviceInfo* dip = nullptr;
  int st = current_device(&dev, &dip);
  if (st != FA_OK) return st;
  cudaError_t e = cudaSuccess;
  int max_clusters = 0;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    DeviceInfo& di = *dip;
    const int slot = (FP8 ? 8 : 0) + (SPLIT ? 4 : 0) + (D == 128 ? 2 : 0) + (CAUSAL ? 1 : 0);
    if (!di.pair_ready[slot]) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return cuda_fail(e);
      // setmaxnreg split: exactly 512 threads x 128 registers at launch.
      cudaFuncAttributes attr;
      e = cudaFuncGetAttributes(&attr, kernel);
      if (e != cudaSuccess) return cuda_fail(e);
      if (attr.numRegs != 128) return FA_ERR_UNSUPPORTED;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2, 1, 1);
      cfg.blockDim = dim3(pair::kThreads, 1, 1);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 2;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
      if (e != cudaSuccess) return cuda_fail(e);
      if (n < 1) return FA_ERR_UNSUPPORTED;
      di.pair_clusters[slot] = n;
      di.pair_ready[slot] = true;
    }
    max_clusters = di.pair_clusters[slot];
  }
  const long long BH = static_cast<long long>(B) * H;
  CUtensorMap mq, mk, mv, mo;
  // O (bf16 for every variant): TMA stores of 32-row boxes by the epilogue
  if ((st = encode_qkv_map(&mo, o, BH, N, D, 32)) != FA_OK) return st;
  if constexpr (FP8) {
    if ((st = encode_e4m3_rows_map(&mq, q, BH, N, D, pair::kRows)) != FA_OK) return st;
    if ((st = encode_e4m3_rows_map(&mk, k, BH, N, D, pair::kHalfKeys)) != FA_OK) return st;
    if ((st = encode_e4m3_keys_last_map(&mv, v, BH, N, D, e4m3_keys_pitch(N))) != FA_OK)
      return st;
  } else {
    if ((st = encode_qkv_map(&mq, q, BH, N, D, pair::kRows)) != FA_OK) return st;
    if ((st = encode_qkv_map(&mk, k, BH, N, D, pair::kHalfKeys)) != FA_OK) return st;
    if ((st = encode_qkv_map(&mv, v, BH, N, D, pair::kKeys)) != FA_OK) return st;
  }
  DevError* err = dip->err;
  const long long n_units =
      pair::Sched::count_units(BH, (N + pair::kKeys - 1) / pair::kKeys, SPLIT ? splits : 1, CAUSAL);
  if (n_units > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  const int clusters = static_cast<int>(n_units < max_clusters ? n_units : max_clusters);
  // A negative scale negates the S product's A operand (Q) in the MMA, so
  // the kernel sees S' = -S with the positive constant |scale| log2(e).
  const int negate_s = scale < 0.f ? 1 : 0;
  float c_log2 = std::fabs(scale) * 1.4426950408889634f;
  if (!(c_log2 >= 1.17549435e-38f)) c_log2 = 1.17549435e-38f;
  const unsigned long long timeout_ns = 2000ull * 1000 * 1000;
  const int head_group =
      (CAUSAL && !SPLIT) ? pick_head_group(BH, (N + pair::kKeys - 1) / pair::kKeys, clusters, N, D)
                         : static_cast<int>(BH);
  kernel<<<2 * clusters, pair::kThreads, smem, stream>>>(
      mq, mk, mv, mo, static_cast<__nv_bfloat16*>(o), lse, part_o, part_l, SPLIT ? splits : 1, err, N,
      static_cast<int>(BH), c_log2, timeout_ns, head_group, negate_s, dsq, dsk, dsv);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

constexpr int kMaxSplits = 64;

// Bytes of workspace for `splits` partial results: O~ fp32 [splits][B*H][N][d]
// then L fp32 [splits][B*H][N]. 0 if the sizes are out of range.
size_t splitkv_workspace_bytes(int B, int H, int N, int d, int splits) {
  if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128) || splits < 1 || splits > kMaxSplits)
    return 0;
  const unsigned long long rows = static_cast<unsigned long long>(B) * H * N;
  if (rows > (1ull << 40)) return 0;
  return static_cast<size_t>(rows * splits * (static_cast<unsigned long long>(d) + 1) * 4);
}

// Split count for num_splits = 0. Splitting pays only when the one-pass
// units (query tiles) leave SM pairs idle; then the count that minimises
// (waves of units) x (key blocks of the longest unit + a fixed cost of
// about 3 blocks per unit: pipeline fill, the first S and the epilogue) is
// taken, the smaller count on ties.  Timed on b1h1n8192d128 (32 tiles, 76
// SM pairs): 2 splits 1.32x the one-pass kernel, 4 1.22x, 6 1.14x, 8 1.11x,
// 3 1.04x, which is the order this cost gives.
int auto_splits(int B, int H, int N, int causal, int clusters) {
  const long long BH = static_cast<long long>(B) * H;
  const int tiles = (N + pair::kKeys - 1) / pair::kKeys;
  if (clusters < 1 || pair::Sched::count_units(BH, tiles, 1, causal != 0) >= clusters) return 1;
  int best = 1;
  long long best_cost = -1;
  for (int s = 1; s <= 8 && s <= tiles; ++s) {
    const long long units = pair::Sched::count_units(BH, tiles, s, causal != 0);
    const long long waves = (units + clusters - 1) / clusters;
    const long long cost = waves * ((tiles + s - 1) / s + 3);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

template <int D, bool CAUSAL>
int launch_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int N, float scale, int splits, void* ws, cudaStream_t stream) {
  const long long BH = static_cast<long long>(B) * H;
  float* part_o = static_cast<float*>(ws);
  float* part_l = part_o + static_cast<size_t>(splits) * BH * N * D;
  int st = launch_pair<D, CAUSAL, true>(q, k, v, o, lse, B, H, N, scale, stream, part_o, part_l,
                                        splits);
  if (st != FA_OK) return st;
  const long long rows = BH * N;
  const long long blocks = (rows + 7) / 8;
  if (blocks > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  fa_splitkv_combine_kernel<D, CAUSAL><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      part_o, part_l, static_cast<__nv_bfloat16*>(o), lse, static_cast<int>(BH), N, splits);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

int splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
            int d, float scale, int causal, int num_splits, void* ws, size_t ws_bytes,
            cudaStream_t s) {
  const int st0 = validate(q, k, v, o, lse, B, H, N, d, scale, causal);
  if (st0 != FA_OK) return st0;
  if (num_splits < 0 || num_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
  if (num_splits == 0) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    num_splits = auto_splits(B, H, N, causal, sms / 2);
  }
  // No tile has more key blocks than this: more splits would give the same
  // units, so the partials are laid out for the clamped count.
  const int n_tiles = (N + pair::kKeys - 1) / pair::kKeys;
  if (num_splits > n_tiles) num_splits = n_tiles;
  if (num_splits == 1) {
    return d == 128 ? (causal ? launch_pair<128, true>(q, k, v, o, lse, B, H, N, scale, s)
                              : launch_pair<128, false>(q, k, v, o, lse, B, H, N, scale, s))
                    : (causal ? launch_pair<64, true>(q, k, v, o, lse, B, H, N, scale, s)
                              : launch_pair<64, false>(q, k, v, o, lse, B, H, N, scale, s));
  }
  const size_t need = splitkv_workspace_bytes(B, H, N, d, num_splits);
  if (need == 0) return FA_ERR_UNSUPPORTED;
  if (!ws) return FA_ERR_INVALID_ARG;
  if (ws_bytes < need) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ws) & 15u) return FA_ERR_MISALIGNED;
  const size_t nb = static_cast<size_t>(B) * H * N * d * 2, nl = static_cast<size_t>(B) * H * N * 4;
  for (const void* p : {q, k, v, static_cast<const void*>(o)})
    if (overlaps(ws, need, p, nb)) return FA_ERR_INVALID_ARG;
  if (overlaps(ws, need, lse, nl)) return FA_ERR_INVALID_ARG;
  if (d == 128)
    return causal ? launch_splitkv<128, true>(q, k, v, o, lse, B, H, N, scale, num_splits, ws, s)
                  : launch_splitkv<128, false>(q, k, v, o, lse, B, H, N, scale, num_splits, ws, s);
  return causal ? launch_splitkv<64, true>(q, k, v, o, lse, B, H, N, scale, num_splits, ws, s)
                : launch_splitkv<64, false>(q, k, v, o, lse, B, H, N, scale, num_splits, ws, s);
}

// ---------------------------------------------------------------- backward

// Two fp32 planes [B*H][Tp] (Tp = N rounded up to a multiple of 128): the
// rows' -L log2 e and -D; then the two kernels' unit counters (256 bytes).
size_t bwd_workspace_bytes(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128)) return 0;
  const unsigned long long tp = (static_cast<unsigned long long>(N) + bwd::kBlk - 1) / bwd::kBlk * bwd::kBlk;
  const unsigned long long rows = static_cast<unsigned long long>(B) * H * tp;
  if (rows > (1ull << 40)) return 0;
  return static_cast<size_t>(rows * 2 * 4 + 256);
}

// The backward's second stream (the dQ kernel runs on it beside the dK/dV
// kernel) and its fork / join events, per device; g_bwd_mu is held while a
// call enqueues, since they are shared.
struct BwdSide {
  bool ready = false;
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
BwdSide g_bwd_side[64];
std::mutex g_bwd_mu;

bool g_bwd_ready[64][4] = {};
// L2 budget of a causal head group in the backward walks (see launch_bwd).
constexpr long long kBwdGroupL2Bytes = 16ll << 20;

template <int D, bool CAUSAL>
int launch_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
               const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, float scale,
               void* ws, cudaStream_t stream) {
  using Ly = bwd::Layout<D>;
  using LyQ = bwd::DqLayout<D>;
  auto kernel_kv = fa_bwd_dkdv_kernel<D, CAUSAL>;
  auto kernel_q = fa_bwd_dq_kernel<D, CAUSAL>;
  int dev = 0;
  DeviceInfo* dip = nullptr;
  int st = current_device(&dev, &dip);
  if (st != FA_OK) return st;
  cudaError_t e = cudaSuccess;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    bool& ready = g_bwd_ready[dev][(D == 128 ? 2 : 0) + (CAUSAL ? 1 : 0)];
    if (!ready) {
      e = cudaFuncSetAttribute(kernel_kv, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::kAlloc);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel_q, cudaFuncAttributeMaxDynamicSharedMemorySize, LyQ::kAlloc);
      if (e == cudaSuccess && dip->sms == 0)
        e = cudaDeviceGetAttribute(&dip->sms, cudaDevAttrMultiProcessorCount, dev);
      int& per_sm = dip->prep_per_sm[D == 128 ? 1 : 0];
      if (e == cudaSuccess && per_sm == 0)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fa_bwd_prep_kernel<D>, 256, 0);
      if (e != cudaSuccess) return cuda_fail(e);
      if (per_sm < 1) per_sm = 1;
      ready = true;
    }
  }
  const long long BH = static_cast<long long>(B) * H;
  const long long T = (N + bwd::kBlk - 1) / bwd::kBlk;
  if (BH * T > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  const int Tp = static_cast<int>(T * bwd::kBlk);
  const long long rows_padded = BH * Tp;
  constexpr long long kPrepRows = 8 * (32 / (D / 16));  // rows per pass of a 256-thread block
  float* nl = static_cast<float*>(ws);
  float* nd = nl + rows_padded;
  int* counters = reinterpret_cast<int*>(nd + rows_padded);
  CUtensorMap mq, mk, mv, mdo;
  if ((st = encode_qkv_map(&mq, q, BH, N, D, bwd::kBlk)) != FA_OK) return st;
  if ((st = encode_qkv_map(&mk, k, BH, N, D, bwd::kBlk)) != FA_OK) return st;
  if ((st = encode_qkv_map(&mv, v, BH, N, D, bwd::kBlk)) != FA_OK) return st;
  if ((st = encode_qkv_map(&mdo, dout, BH, N, D, bwd::kBlk)) != FA_OK) return st;
  DevError* err = dip->err;
  std::lock_guard<std::mutex> lock(g_bwd_mu);
  BwdSide& side = g_bwd_side[dev];
  if (!side.ready) {
    if ((e = cudaStreamCreateWithFlags(&side.stream, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&side.fork, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&side.join, cudaEventDisableTiming)) != cudaSuccess)
      return cuda_fail(e);
    side.ready = true;
  }
  // one pass of resident blocks over the row groups, in even shares
  const long long prep_groups = (rows_padded + kPrepRows - 1) / kPrepRows;
  const long long prep_slots = static_cast<long long>(dip->sms) * dip->prep_per_sm[D == 128 ? 1 : 0];
  const long long prep_grid = prep_groups < prep_slots ? prep_groups : prep_slots;
  fa_bwd_prep_kernel<D><<<static_cast<unsigned>(prep_grid), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse, nl, nd, N,
      Tp, rows_padded, counters);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  const float c_log2 = scale * 1.4426950408889634f;
  const unsigned long long timeout_ns = 2000ull * 1000 * 1000;
  // One CTA per SM for each kernel (fewer if there are fewer units); each
  // takes units from its counter until none are left.  The dQ kernel goes
  // on the second stream, so that its CTAs start on the SMs the dK/dV
  // kernel's CTAs leave as that kernel runs out of units, and the other way
  // round; the caller's stream then waits for both.
  const long long grid = BH * T < dip->sms ? BH * T : dip->sms;
  // Causal: heads in groups whose streamed operands (two [N, d] bf16
  // tensors per head) fit in kBwdGroupL2Bytes of L2; ungrouped, the CTAs'
  // walks span every head at once and re-read each operand from DRAM
  // about seven times at B=2, H=32, N=8192.
  const long long per_head = 2ll * N * D * 2;
  long long hg = kBwdGroupL2Bytes / per_head;
  hg = hg < 1 ? 1 : (hg > BH ? BH : hg);
  const int head_group = static_cast<int>(hg);
  if ((e = cudaEventRecord(side.fork, stream)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(side.stream, side.fork, 0)) != cudaSuccess)
    return cuda_fail(e);
  {
    // a programmatic dependent of the statistics kernel: its CTAs set up
    // while that kernel finishes, and its producer waits for the grid
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(bwd::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Ly::kAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel_kv, mq, mk, mv, mdo, static_cast<const float*>(nl),
                           static_cast<const float*>(nd), Tp, counters, static_cast<__nv_bfloat16*>(dk),
                           static_cast<__nv_bfloat16*>(dv), err, N, static_cast<int>(BH), head_group,
                           c_log2, scale, timeout_ns);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  kernel_q<<<static_cast<unsigned>(grid), bwd::kThreads, LyQ::kAlloc, side.stream>>>(
      mq, mk, mv, mdo, nl, nd, Tp, counters + 1, static_cast<__nv_bfloat16*>(dq), err, N,
      static_cast<int>(BH), head_group, c_log2, scale, timeout_ns);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  if ((e = cudaEventRecord(side.join, side.stream)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(stream, side.join, 0)) != cudaSuccess)
    return cuda_fail(e);
  return FA_OK;
}

int backward(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
             float scale, int causal, void* ws, size_t ws_bytes, cudaStream_t s) {
  // q, k, v, o, lse: the forward's inputs and outputs, read only here
  const int st0 = validate(q, k, v, o, lse, B, H, N, d, scale, causal, false);
  if (st0 != FA_OK) return st0;
  if (!dout || !dq || !dk || !dv || !ws) return FA_ERR_INVALID_ARG;
  for (const void* p : {dout, static_cast<const void*>(dq), static_cast<const void*>(dk),
                        static_cast<const void*>(dv), static_cast<const void*>(ws)})
    if (reinterpret_cast<uintptr_t>(p) & 15u) return FA_ERR_MISALIGNED;
  const size_t need = bwd_workspace_bytes(B, H, N, d);
  if (need == 0) return FA_ERR_UNSUPPORTED;
  if (ws_bytes < need) return FA_ERR_INVALID_ARG;
  const size_t nb = static_cast<size_t>(B) * H * N * d * 2, nl = static_cast<size_t>(B) * H * N * 4;
  const void* ins[6] = {q, k, v, o, lse, dout};
  const size_t in_sz[6] = {nb, nb, nb, nb, nl, nb};
  const void* outs[4] = {dq, dk, dv, ws};
  const size_t out_sz[4] = {nb, nb, nb, need};
  for (int a = 0; a < 4; ++a) {
    for (int b = 0; b < 6; ++b)
      if (overlaps(outs[a], out_sz[a], ins[b], in_sz[b])) return FA_ERR_INVALID_ARG;
    for (int b = a + 1; b < 4; ++b)
      if (overlaps(outs[a], out_sz[a], outs[b], out_sz[b])) return FA_ERR_INVALID_ARG;
  }
  if (d == 128)
    return causal ? launch_bwd<128, true>(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, scale, ws, s)
                  : launch_bwd<128, false>(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, scale, ws, s);
  return causal ? launch_bwd<64, true>(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, scale, ws, s)
                : launch_bwd<64, false>(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, scale, ws, s);
}

// ------------------------------------------------------- host-buffer path

// Streams and events of the host-buffer path, created once per device.
struct HostPipe {
  static constexpr int kChunks = 8;
  bool ready = false;
  cudaStream_t in = nullptr, run = nullptr, out = nullptr;
  cudaEvent_t fork = nullptr, done = nullptr;
  cudaEvent_t landed[kChunks] = {}, computed[kChunks] = {};
};
HostPipe g_host_pipe[64];
std::mutex g_host_mu;  // held while a call enqueues: the streams and events are shared

// q, k, v host -> device, the forward, O and L device -> host, pipelined
// over up to eight groups of heads: one stream uploads the groups in order
// (the host link is the bottleneck and is best used one transfer at a time),
// a second runs each group's kernel as soon as its inputs have landed, a
// third downloads each group's results as soon as its kernel is done, so
// uploads, kernels and downloads of different groups overlap.  Forked from
// and joined back to the caller's stream.
int host_pipelined(const void* q, const void* k, const void* v, void* o, float* lse, void* dq,
                   void* dk, void* dv, void* do_, float* dlse, int B, int H, int N, int d,
                   float scale, int causal, cudaStream_t caller) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_host_mu);
  HostPipe& hp = g_host_pipe[dev];
  if (!hp.ready) {
    for (cudaStream_t* ps : {&hp.in, &hp.run, &hp.out})
      if ((e = cudaStreamCreateWithFlags(ps, cudaStreamNonBlocking)) != cudaSuccess)
        return cuda_fail(e);
    for (cudaEvent_t* pe : {&hp.fork, &hp.done})
      if ((e = cudaEventCreateWithFlags(pe, cudaEventDisableTiming)) != cudaSuccess)
        return cuda_fail(e);
    for (int c = 0; c < HostPipe::kChunks; ++c) {
      if ((e = cudaEventCreateWithFlags(&hp.landed[c], cudaEventDisableTiming)) != cudaSuccess)
        return cuda_fail(e);
      if ((e = cudaEventCreateWithFlags(&hp.computed[c], cudaEventDisableTiming)) != cudaSuccess)
        return cuda_fail(e);
    }
    hp.ready = true;
  }
  const long long BH = static_cast<long long>(B) * H;
  const int chunks = static_cast<int>(BH < HostPipe::kChunks ? BH : HostPipe::kChunks);
  // Group c holds heads [first_head(c), first_head(c + 1)).  With four or
  // more groups the first and the last carry half the heads of the others:
  // the first upload (before any kernel can start) and the last download
  // (after every kernel) are the parts of the step nothing overlaps.
  auto first_head = [&](int c) -> long long {
    if (chunks < 4) return BH * c / chunks;
    const long long w = 2ll * c - (c > 0 ? 1 : 0) - (c == chunks ? 1 : 0);  // weights 1, 2, ..., 2, 1
    return BH * w / (2ll * chunks - 2);
  };
  const size_t head_b = static_cast<size_t>(N) * d * 2, head_l = static_cast<size_t>(N) * 4;
  auto hb = [](const void* p, size_t off) { return static_cast<const char*>(p) + off; };
  auto db = [](void* p, size_t off) { return static_cast<char*>(p) + off; };
  if ((e = cudaEventRecord(hp.fork, caller)) != cudaSuccess) return cuda_fail(e);
  // Once work is queued on the internal streams, an error return first waits
  // for all of it, so that no copy or kernel of this call still runs on the
  // caller's buffers after the call has returned.
  auto fail_after_fork = [&](int status) {
    for (cudaStream_t s : {hp.in, hp.run, hp.out}) (void)cudaStreamSynchronize(s);
    return status;
  };
  for (cudaStream_t s : {hp.in, hp.run, hp.out})
    if ((e = cudaStreamWaitEvent(s, hp.fork, 0)) != cudaSuccess) return fail_after_fork(cuda_fail(e));
  for (int c = 0; c < chunks; ++c) {
    const long long h0 = first_head(c), h1 = first_head(c + 1);
    if (h1 == h0) continue;  // fewer heads than groups after the halving
    const size_t ob = static_cast<size_t>(h0) * head_b, nb = static_cast<size_t>(h1 - h0) * head_b;
    const size_t ol = static_cast<size_t>(h0) * head_l, nl = static_cast<size_t>(h1 - h0) * head_l;
    const int hn = static_cast<int>(h1 - h0);
    // upload
    if ((e = cudaMemcpyAsync(db(dq, ob), hb(q, ob), nb, cudaMemcpyHostToDevice, hp.in)) != cudaSuccess)
      return fail_after_fork(cuda_fail(e));
    if ((e = cudaMemcpyAsync(db(dk, ob), hb(k, ob), nb, cudaMemcpyHostToDevice, hp.in)) != cudaSuccess)
      return fail_after_fork(cuda_fail(e));
    if ((e = cudaMemcpyAsync(db(dv, ob), hb(v, ob), nb, cudaMemcpyHostToDevice, hp.in)) != cudaSuccess)
      return fail_after_fork(cuda_fail(e));
    if ((e = cudaEventRecord(hp.landed[c], hp.in)) != cudaSuccess) return fail_after_fork(cuda_fail(e));
    // kernel
    if ((e = cudaStreamWaitEvent(hp.run, hp.landed[c], 0)) != cudaSuccess) return fail_after_fork(cuda_fail(e));
    float* lsec = reinterpret_cast<float*>(db(dlse, ol));
    const int st = d == 128
        ? (causal ? launch_pair<128, true>(db(dq, ob), db(dk, ob), db(dv, ob), db(do_, ob), lsec, 1,
                                           hn, N, scale, hp.run)
                  : launch_pair<128, false>(db(dq, ob), db(dk, ob), db(dv, ob), db(do_, ob), lsec, 1,
                                            hn, N, scale, hp.run))
        : (causal ? launch_pair<64, true>(db(dq, ob), db(dk, ob), db(dv, ob), db(do_, ob), lsec, 1,
                                          hn, N, scale, hp.run)
                  : launch_pair<64, false>(db(dq, ob), db(dk, ob), db(dv, ob), db(do_, ob), lsec, 1,
                                           hn, N, scale, hp.run));
    if (st != FA_OK) return fail_after_fork(st);
    if ((e = cudaEventRecord(hp.computed[c], hp.run)) != cudaSuccess) return fail_after_fork(cuda_fail(e));
    // download
    if ((e = cudaStreamWaitEvent(hp.out, hp.computed[c], 0)) != cudaSuccess) return fail_after_fork(cuda_fail(e));
    if ((e = cudaMemcpyAsync(db(o, ob), db(do_, ob), nb, cudaMemcpyDeviceToHost, hp.out)) != cudaSuccess)
      return fail_after_fork(cuda_fail(e));
    if ((e = cudaMemcpyAsync(db(lse, ol), db(dlse, ol), nl, cudaMemcpyDeviceToHost, hp.out)) != cudaSuccess)
      return fail_after_fork(cuda_fail(e));
  }
  // join: the download stream's last work follows every kernel and every
  // upload (through the events), so waiting on it covers the whole call
  if ((e = cudaEventRecord(hp.done, hp.out)) != cudaSuccess) return fail_after_fork(cuda_fail(e));
  if ((e = cudaStreamWaitEvent(caller, hp.done, 0)) != cudaSuccess) return fail_after_fork(cuda_fail(e));
  return FA_OK;
}


// ---------------------------------------------------- unfused attention

// Row pitch (elements) of S and P in the unfused path: N rounded up to 8, so
// that every row of either matrix starts 16-byte aligned.
long long unfused_pitch(long long N) { return (N + 7) / 8 * 8; }

// Bytes of S (fp32, padded to 256 bytes) then P (bf16), [B*H][N][pitch]
// each; 0 if out of range.
size_t unfused_workspace_bytes(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128)) return 0;
  const unsigned long long cells =
      static_cast<unsigned long long>(B) * H * N * static_cast<unsigned long long>(unfused_pitch(N));
  if (cells > (1ull << 44)) return 0;
  return static_cast<size_t>((cells * 4 + 255) / 256 * 256 + cells * 2);
}

template <int D, bool CAUSAL>
int launch_unfused(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int N, float scale, void* ws, cudaStream_t stream) {
  using LyS = unf::LayoutS<D>;
  using LyP = unf::LayoutPV<D>;
  int dev = 0;
  DeviceInfo* dip = nullptr;
  int st = current_device(&dev, &dip);
  if (st != FA_OK) return st;
  cudaError_t e = cudaSuccess;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    bool& ready = dip->unf_ready[(D == 128 ? 2 : 0) + (CAUSAL ? 1 : 0)];
    if (!ready) {
      e = cudaFuncSetAttribute(fa_unf_s_kernel<D, CAUSAL>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, LyS::kAlloc);
      if (e != cudaSuccess) return cuda_fail(e);
      e = cudaFuncSetAttribute(fa_unf_pv_kernel<D, CAUSAL>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, LyP::kAlloc);
      if (e != cudaSuccess) return cuda_fail(e);
      ready = true;
    }
  }
  const long long BH = static_cast<long long>(B) * H;
  const long long pitch = unfused_pitch(N);
  const long long n_qt = (N + unf::kRowsS - 1) / unf::kRowsS;
  const long long n_kt = (N + unf::kKeysS - 1) / unf::kKeysS;
  const long long rows = BH * N;
  // grids: S tiles, softmax rows (one CTA per row up to 16384 keys, else one warp), P V tiles
  if (BH * n_qt * n_kt > 0x7fffffffLL || (rows + 7) / 8 > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (N <= 16384 && rows > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  float* S = static_cast<float*>(ws);
  const size_t s_bytes = (static_cast<size_t>(rows) * pitch * 4 + 255) / 256 * 256;
  __nv_bfloat16* P = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(ws) + s_bytes);
  CUtensorMap mq, mk, ms, mp, mv;
  if ((st = encode_qkv_map(&mq, q, BH, N, D, unf::kRowsS)) != FA_OK) return st;
  if ((st = encode_qkv_map(&mk, k, BH, N, D, unf::kKeysS)) != FA_OK) return st;
  if ((st = encode_qkv_map(&mv, v, BH, N, D, unf::kKeysPV)) != FA_OK) return st;
  if ((st = encode_scores_map(&ms, S, BH, N, pitch)) != FA_OK) return st;
  if ((st = encode_probs_map(&mp, P, BH, N, pitch)) != FA_OK) return st;
  const unsigned long long timeout_ns = 2000ull * 1000 * 1000;
  fa_unf_s_kernel<D, CAUSAL><<<static_cast<unsigned>(BH * n_qt * n_kt), unf::kThreadsS,
                               LyS::kAlloc, stream>>>(mq, mk, ms, dip->err, N,
                                                      static_cast<int>(n_qt),
                                                      static_cast<int>(n_kt), scale, timeout_ns);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  // softmax: the row in registers of one CTA (S read once) up to 16384 keys
  const int np = static_cast<int>(pitch);
  if (N <= 1024)
    fa_unf_softmax_row_kernel<CAUSAL, 4><<<static_cast<unsigned>(rows), 256, 0, stream>>>(S, P, lse, N, np);
  else if (N <= 2048)
    fa_unf_softmax_row_kernel<CAUSAL, 8><<<static_cast<unsigned>(rows), 256, 0, stream>>>(S, P, lse, N, np);
  else if (N <= 4096)
    fa_unf_softmax_row_kernel<CAUSAL, 16><<<static_cast<unsigned>(rows), 256, 0, stream>>>(S, P, lse, N, np);
  else if (N <= 8192)
    fa_unf_softmax_row_kernel<CAUSAL, 32><<<static_cast<unsigned>(rows), 256, 0, stream>>>(S, P, lse, N, np);
  else if (N <= 16384)
    fa_unf_softmax_row_kernel<CAUSAL, 64><<<static_cast<unsigned>(rows), 256, 0, stream>>>(S, P, lse, N, np);
  else
    fa_unf_softmax_kernel<CAUSAL><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
        S, P, lse, rows, N, np);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  fa_unf_pv_kernel<D, CAUSAL><<<static_cast<unsigned>(BH * n_qt), unf::kThreadsPV, LyP::kAlloc,
                                stream>>>(mp, mv, static_cast<__nv_bfloat16*>(o), dip->err, N,
                                          static_cast<int>(n_qt), timeout_ns);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

int unfused(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
            int d, float scale, int causal, void* ws, size_t ws_bytes, cudaStream_t s) {
  const int st0 = validate(q, k, v, o, lse, B, H, N, d, scale, causal);
  if (st0 != FA_OK) return st0;
  const size_t need = unfused_workspace_bytes(B, H, N, d);
  if (need == 0) return FA_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < need) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ws) & 15u) return FA_ERR_MISALIGNED;
  const size_t nb = static_cast<size_t>(B) * H * N * d * 2, nl = static_cast<size_t>(B) * H * N * 4;
  for (const void* p : {q, k, v, static_cast<const void*>(o)})
    if (overlaps(ws, need, p, nb)) return FA_ERR_INVALID_ARG;
  if (overlaps(ws, need, lse, nl)) return FA_ERR_INVALID_ARG;
  if (d == 128)
    return causal ? launch_unfused<128, true>(q, k, v, o, lse, B, H, N, scale, ws, s)
                  : launch_unfused<128, false>(q, k, v, o, lse, B, H, N, scale, ws, s);
  return causal ? launch_unfused<64, true>(q, k, v, o, lse, B, H, N, scale, ws, s)
                : launch_unfused<64, false>(q, k, v, o, lse, B, H, N, scale, ws, s);
}

// ------------------------------------------------------------- self-test

constexpr unsigned kSiteSelfTest = 901;

// One warp waits, through the kernels' own bounded wait, on an mbarrier that
// nothing ever arrives at: the wait must give up after timeout_ns, record
// the site in the device error record and return.
__global__ void fa_selftest_wait_kernel(DevError* err, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wc{&abort_flag, err, timeout_ns};
  (void)mbar_wait(smem_u32(&bar), 0, wc, kSiteSelfTest, 0);
}

int selftest_wait_timeout(unsigned int timeout_us, cudaStream_t s) {
  if (timeout_us == 0 || timeout_us > 1000000u) return FA_ERR_INVALID_ARG;
  int dev = 0;
  DeviceInfo* dip = nullptr;
  const int st = current_device(&dev, &dip);
  if (st != FA_OK) return st;
  fa_selftest_wait_kernel<<<1, 32, 0, s>>>(dip->err, 1000ull * timeout_us);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

// ------------------------------------------------------------- 8-bit path

// Bytes of the E4M3 codes of a [B, H, N, d] tensor in the given layout; 0 if
// out of range.
size_t e4m3_bytes(int B, int H, int N, int d, int keys_last) {
  if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128) || (keys_last != 0 && keys_last != 1))
    return 0;
  const unsigned long long BH = static_cast<unsigned long long>(B) * H;
  const unsigned long long cols = keys_last ? e4m3_keys_pitch(N) : static_cast<unsigned long long>(N);
  if (BH * cols > (1ull << 52)) return 0;
  return static_cast<size_t>(BH * cols * d);
}

int quantize_e4m3(const void* x, void* x8, float* descale, int B, int H, int N, int d,
                  int keys_last, cudaStream_t s) {
  if (!x || !x8 || !descale) return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || N <= 0 || (keys_last != 0 && keys_last != 1)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 65535) return FA_ERR_UNSUPPORTED;  // one grid row per (batch, head)
  const size_t nout = e4m3_bytes(B, H, N, d, keys_last);
  if (nout == 0) return FA_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(x8)) & 15u)
    return FA_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(descale) & 3u) return FA_ERR_MISALIGNED;
  const size_t nx = static_cast<size_t>(BH) * N * d * 2, nd = static_cast<size_t>(BH) * 4;
  if (overlaps(x8, nout, x, nx) || overlaps(descale, nd, x, nx) || overlaps(descale, nd, x8, nout))
    return FA_ERR_INVALID_ARG;
  cudaError_t e = cudaMemsetAsync(descale, 0, nd, s);
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned* bits = reinterpret_cast<unsigned*>(descale);
  const long long slice_vecs = static_cast<long long>(N) * d / fp8::kVec;
  // about 8 CTAs per SM over all slices, at least 1024 vectors per CTA
  long long chunks = (1216 + BH - 1) / BH;
  const long long max_chunks = (slice_vecs + 1023) / 1024;
  if (chunks > max_chunks) chunks = max_chunks;
  if (chunks < 1) chunks = 1;
  const long long per = (slice_vecs + chunks - 1) / chunks;
  const dim3 grid(static_cast<unsigned>(chunks), static_cast<unsigned>(BH));
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  uint8_t* out = static_cast<uint8_t*>(x8);
  fa_amax_kernel<<<grid, fp8::kThreads, 0, s>>>(xb, bits, slice_vecs, per);
  if (keys_last) {
    const dim3 g2(static_cast<unsigned>((N + fp8::kTileKeys - 1) / fp8::kTileKeys),
                  static_cast<unsigned>(BH));
    const int pitch = static_cast<int>(e4m3_keys_pitch(N));
    if (d == 128)
      fa_quant_keys_last_kernel<128><<<g2, fp8::kThreads, 0, s>>>(xb, out, bits, N, pitch);
    else
      fa_quant_keys_last_kernel<64><<<g2, fp8::kThreads, 0, s>>>(xb, out, bits, N, pitch);
  } else {
    fa_quant_rows_kernel<<<grid, fp8::kThreads, 0, s>>>(xb, out, bits, slice_vecs, per);
  }
  fa_descale_kernel<<<static_cast<unsigned>((BH + 255) / 256), 256, 0, s>>>(descale,
                                                                             static_cast<int>(BH));
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

// Q, K, V together (V keys-last): the steps of quantize_e4m3 in four
// launches, each over all three tensors.
int quantize_qkv_e4m3(const void* q, const void* k, const void* v, void* q8, void* k8, void* vt8,
                      float* dsq, float* dsk, float* dsv, int B, int H, int N, int d,
                      cudaStream_t s) {
  const void* ins[3] = {q, k, v};
  void* outs[3] = {q8, k8, vt8};
  float* ds[3] = {dsq, dsk, dsv};
  for (int t = 0; t < 3; ++t)
    if (!ins[t] || !outs[t] || !ds[t]) return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || N <= 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 65535) return FA_ERR_UNSUPPORTED;
  const size_t nrow = e4m3_bytes(B, H, N, d, 0), nkl = e4m3_bytes(B, H, N, d, 1);
  if (nrow == 0 || nkl == 0) return FA_ERR_UNSUPPORTED;
  for (int t = 0; t < 3; ++t) {
    if ((reinterpret_cast<uintptr_t>(ins[t]) | reinterpret_cast<uintptr_t>(outs[t])) & 15u)
      return FA_ERR_MISALIGNED;
    if (reinterpret_cast<uintptr_t>(ds[t]) & 3u) return FA_ERR_MISALIGNED;
  }
  const size_t nx = static_cast<size_t>(BH) * N * d * 2, nd = static_cast<size_t>(BH) * 4;
  const size_t nout[3] = {nrow, nrow, nkl};
  for (int t = 0; t < 3; ++t)
    for (int u = 0; u < 3; ++u) {
      if (overlaps(outs[t], nout[t], ins[u], nx) || overlaps(ds[t], nd, ins[u], nx))
        return FA_ERR_INVALID_ARG;
      if (overlaps(ds[t], nd, outs[u], nout[u])) return FA_ERR_INVALID_ARG;
      if (u != t && (overlaps(outs[t], nout[t], outs[u], nout[u]) || overlaps(ds[t], nd, ds[u], nd)))
        return FA_ERR_INVALID_ARG;
    }
  Qkv3 a;
  for (int t = 0; t < 3; ++t) {
    a.x[t] = static_cast<const __nv_bfloat16*>(ins[t]);
    a.out[t] = static_cast<uint8_t*>(outs[t]);
    a.descale[t] = ds[t];
  }
  const long long slice_vecs = static_cast<long long>(N) * d / fp8::kVec;
  long long chunks = (1216 + 3 * BH - 1) / (3 * BH);
  const long long max_chunks = (slice_vecs + 1023) / 1024;
  if (chunks > max_chunks) chunks = max_chunks;
  if (chunks < 1) chunks = 1;
  const long long per = (slice_vecs + chunks - 1) / chunks;
  const int pitch = static_cast<int>(e4m3_keys_pitch(N));
  const long long tiles = (N + fp8::kTileKeys - 1) / fp8::kTileKeys;
  const unsigned bx = static_cast<unsigned>(BH + 255) / 256;
  fa_zero3_kernel<<<bx, 256, 0, s>>>(a, static_cast<int>(BH));
  fa_amax3_kernel<<<dim3(static_cast<unsigned>(chunks), static_cast<unsigned>(BH), 3), fp8::kThreads, 0,
                    s>>>(a, slice_vecs, per);
  const dim3 gq(static_cast<unsigned>(chunks > tiles ? chunks : tiles), static_cast<unsigned>(BH), 3);
  if (d == 128)
    fa_quant3_kernel<128><<<gq, fp8::kThreads, 0, s>>>(a, N, pitch, slice_vecs, per, static_cast<int>(chunks));
  else
    fa_quant3_kernel<64><<<gq, fp8::kThreads, 0, s>>>(a, N, pitch, slice_vecs, per, static_cast<int>(chunks));
  fa_descale3_kernel<<<dim3(bx, 3), 256, 0, s>>>(a, static_cast<int>(BH));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

int fwd_e4m3(const void* q8, const void* k8, const void* vt8, const float* dsq, const float* dsk,
             const float* dsv, void* o, float* lse, int B, int H, int N, int d, float scale,
             int causal, cudaStream_t s) {
  if (!q8 || !k8 || !vt8 || !dsq || !dsk || !dsv || !o || !lse) return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || N <= 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (scale < 0.f) return FA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (BH * ((static_cast<long long>(N) + 255) / 256) > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (BH * N > (1LL << 45)) return FA_ERR_UNSUPPORTED;
  for (const void* p : {q8, k8, vt8, static_cast<const void*>(o)})
    if (reinterpret_cast<uintptr_t>(p) & 15u) return FA_ERR_MISALIGNED;
  for (const void* p : {static_cast<const void*>(lse), static_cast<const void*>(dsq),
                        static_cast<const void*>(dsk), static_cast<const void*>(dsv)})
    if (reinterpret_cast<uintptr_t>(p) & 3u) return FA_ERR_MISALIGNED;
  const size_t nq = e4m3_bytes(B, H, N, d, 0), nv = e4m3_bytes(B, H, N, d, 1);
  const size_t no = static_cast<size_t>(BH) * N * d * 2, nl = static_cast<size_t>(BH) * N * 4;
  const size_t nd = static_cast<size_t>(BH) * 4;
  const struct { const void* p; size_t n; } ins[6] = {{q8, nq}, {k8, nq}, {vt8, nv},
                                                      {dsq, nd}, {dsk, nd}, {dsv, nd}};
  for (const auto& in : ins)
    if (overlaps(o, no, in.p, in.n) || overlaps(lse, nl, in.p, in.n)) return FA_ERR_INVALID_ARG;
  if (overlaps(o, no, lse, nl)) return FA_ERR_INVALID_ARG;
  if (d == 64)
    return causal ? launch_pair<64, true, false, true>(q8, k8, vt8, o, lse, B, H, N, scale, s,
                                                       nullptr, nullptr, 1, dsq, dsk, dsv)
                  : launch_pair<64, false, false, true>(q8, k8, vt8, o, lse, B, H, N, scale, s,
                                                        nullptr, nullptr, 1, dsq, dsk, dsv);
  return causal ? launch_pair<128, true, false, true>(q8, k8, vt8, o, lse, B, H, N, scale, s,
                                                      nullptr, nullptr, 1, dsq, dsk, dsv)
                : launch_pair<128, false, false, true>(q8, k8, vt8, o, lse, B, H, N, scale, s,
                                                       nullptr, nullptr, 1, dsq, dsk, dsv);
}

}  // namespace
}  // namespace fa

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, float scale, int causal, void* stream) {
  const int st = fa::validate(q, k, v, o, lse, B, H, N, d, scale, causal);
  if (st != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 128)
    return causal ? fa::launch_pair<128, true>(q, k, v, o, lse, B, H, N, scale, s)
                  : fa::launch_pair<128, false>(q, k, v, o, lse, B, H, N, scale, s);
  return causal ? fa::launch_pair<64, true>(q, k, v, o, lse, B, H, N, scale, s)
                : fa::launch_pair<64, false>(q, k, v, o, lse, B, H, N, scale, s);
}

int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, void* dq,
                void* dk, void* dv, void* do_, float* dlse, int B, int H, int N, int d,
                float scale, int causal, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  int st = fa::validate(dq, dk, dv, do_, dlse, B, H, N, d, scale, causal);
  if (st != FA_OK) return st;
  return fa::host_pipelined(q, k, v, o, lse, dq, dk, dv, do_, dlse, B, H, N, d, scale, causal,
                            static_cast<cudaStream_t>(stream));
}

size_t fa_fwd_splitkv_workspace_size(int B, int H, int N, int d, int num_splits) {
  return fa::splitkv_workspace_bytes(B, H, N, d, num_splits);
}

int fa_fwd_splitkv_num_splits(int B, int H, int N, int causal) {
  if (B <= 0 || H <= 0 || N <= 0) return FA_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fa::cuda_fail(e);
  return fa::auto_splits(B, H, N, causal, sms / 2);
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int N, int d, float scale, int causal, int num_splits, void* workspace,
                   size_t workspace_bytes, void* stream) {
  return fa::splitkv(q, k, v, o, lse, B, H, N, d, scale, causal, num_splits, workspace,
                     workspace_bytes, static_cast<cudaStream_t>(stream));
}

int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int N, int d, float scale, int causal, int num_splits,
                           void* stream) {
  const int st = fa::validate(q, k, v, o, lse, B, H, N, d, scale, causal);
  if (st != FA_OK) return st;
  if (num_splits < 0 || num_splits > fa::kMaxSplits) return FA_ERR_INVALID_ARG;
  if (num_splits == 0) {
    const int n = fa_fwd_splitkv_num_splits(B, H, N, causal);
    if (n < 0) return n;
    num_splits = n;
  }
  const int n_tiles = (N + fa::pair::kKeys - 1) / fa::pair::kKeys;  // as fa::splitkv clamps
  if (num_splits > n_tiles) num_splits = n_tiles;
  if (num_splits > 1 &&
      fa::splitkv_workspace_bytes(B, H, N, d, num_splits) > fa::kNoAllocScratchBytes)
    return FA_ERR_UNSUPPORTED;  // the fixed scratch is too small for this call
  int dev = 0;
  fa::DeviceInfo* dip = nullptr;
  int st1 = fa::current_device(&dev, &dip);
  if (st1 != FA_OK) return st1;
  void* scratch = nullptr;  // this device's copy of the module's scratch, looked up once
  {
    std::lock_guard<std::mutex> lock(fa::g_setup_mu);
    if (!dip->noalloc_scratch) {
      const cudaError_t e = cudaGetSymbolAddress(&dip->noalloc_scratch, fa::g_noalloc_scratch);
      if (e != cudaSuccess) {
        dip->noalloc_scratch = nullptr;
        return fa::cuda_fail(e);
      }
    }
    scratch = dip->noalloc_scratch;
  }
  return fa::splitkv(q, k, v, o, lse, B, H, N, d, scale, causal, num_splits, scratch,
                     fa::kNoAllocScratchBytes, static_cast<cudaStream_t>(stream));
}

size_t fa_fwd_splitkv_noalloc_capacity(void) { return fa::kNoAllocScratchBytes; }

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  return fa::bwd_workspace_bytes(B, H, N, d);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
           float scale, int causal, void* workspace, size_t workspace_bytes, void* stream) {
  return fa::backward(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, workspace,
                      workspace_bytes, static_cast<cudaStream_t>(stream));
}

size_t fa_attn_unfused_workspace_size(int B, int H, int N, int d) {
  return fa::unfused_workspace_bytes(B, H, N, d);
}

int fa_attn_unfused(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                    int N, int d, float scale, int causal, void* workspace, size_t workspace_bytes,
                    void* stream) {
  return fa::unfused(q, k, v, o, lse, B, H, N, d, scale, causal, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream));
}

size_t fa_e4m3_bytes(int B, int H, int N, int d, int keys_last) {
  return fa::e4m3_bytes(B, H, N, d, keys_last);
}

int fa_quantize_e4m3(const void* x, void* x8, float* descale, int B, int H, int N, int d,
                     int keys_last, void* stream) {
  return fa::quantize_e4m3(x, x8, descale, B, H, N, d, keys_last,
                           static_cast<cudaStream_t>(stream));
}

int fa_quantize_qkv_e4m3(const void* q, const void* k, const void* v, void* q8, void* k8,
                         void* vt8, float* descale_q, float* descale_k, float* descale_v, int B,
                         int H, int N, int d, void* stream) {
  return fa::quantize_qkv_e4m3(q, k, v, q8, k8, vt8, descale_q, descale_k, descale_v, B, H, N, d,
                               static_cast<cudaStream_t>(stream));
}

int fa_fwd_e4m3(const void* q8, const void* k8, const void* vt8, const float* descale_q,
                const float* descale_k, const float* descale_v, void* o, float* lse, int B,
                int H, int N, int d, float scale, int causal, void* stream) {
  return fa::fwd_e4m3(q8, k8, vt8, descale_q, descale_k, descale_v, o, lse, B, H, N, d, scale,
                      causal, static_cast<cudaStream_t>(stream));
}

int fa_selftest_wait_timeout(unsigned int timeout_us, void* stream) {
  return fa::selftest_wait_timeout(timeout_us, static_cast<cudaStream_t>(stream));
}

int fa_check_errors(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fa::cuda_fail(e);
  fa::DevError rec;
  e = cudaMemcpyFromSymbol(&rec, fa::g_dev_error, sizeof(rec));
  if (e != cudaSuccess) return fa::cuda_fail(e);
  if (rec.code != 0) {
    fa::t_last_record[0] = rec.code;
    fa::t_last_record[1] = rec.site;
    fa::t_last_record[2] = rec.block;
    fa::t_last_record[3] = rec.tile;
    const fa::DevError zero = {0, 0, 0, 0};
    e = cudaMemcpyToSymbol(fa::g_dev_error, &zero, sizeof(zero));
    if (e != cudaSuccess) return fa::cuda_fail(e);
    return FA_ERR_TIMEOUT;
  }
  return FA_OK;
}

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    default: return "FA_ERR_UNKNOWN";
  }
}

int fa_get_last_cuda_error(void) { return fa::t_last_cuda_error; }

int fa_get_last_error_record(unsigned int* out4) {
  if (!out4) return FA_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i) out4[i] = fa::t_last_record[i];
  return FA_OK;
}

int fa_version(void) { return 100; }

}  // extern "C"
