// Per-(batch, head) E4M3 quantisation of a bf16 [B*H, N, d] tensor, the
// input step of the 8-bit forward.
//
// The pages only say that the third FlashAttention version gains about 2x
// over BF16 from FP8 ("How FlashAttention got past the O(N^2) memory wall",
// "v2 and v3"); the scaling is this library's reading: one scale per
// (batch, head) slice, amax = max |x| over the slice, s = 448 / amax (1 when
// amax is 0), code = E4M3(x * s) rounded to nearest even and saturated at
// +-448, descale = amax / 448.  Every step is correctly rounded fp32
// (__fdiv_rn, __fmul_rn), so the codes are a function of the inputs alone.
//
// Three launches on one stream: the slice maxima (atomicMax on the bit
// pattern of |x|, which orders non-negative floats), the codes, and the
// descales written over the maxima.  The caller zeroes the maxima first.
// For Q, K and V together the same steps take four launches (zeroing
// included), each covering all three tensors.
#pragma once
#include <cuda_bf16.h>

#include "sm103_ptx.cuh"

namespace fa {

namespace fp8 {
constexpr int kThreads = 256;
constexpr int kVec = 8;          // bf16 elements per 16-byte load
constexpr int kTileKeys = 64;    // keys per CTA of the keys-last kernel
}  // namespace fp8

// amax_bits[bh] = max over the slice of |x| as float bits.  Grid
// (chunks, BH); each CTA takes a contiguous run of 16-byte vectors.
__global__ void __launch_bounds__(fp8::kThreads) fa_amax_kernel(
    const __nv_bfloat16* __restrict__ x, unsigned* __restrict__ amax_bits,
    long long slice_vecs, long long vecs_per_chunk) {
  const int bh = blockIdx.y;
  const long long lo = static_cast<long long>(blockIdx.x) * vecs_per_chunk;
  const long long hi = min(slice_vecs, lo + vecs_per_chunk);
  const uint4* src = reinterpret_cast<const uint4*>(x) + static_cast<long long>(bh) * slice_vecs;
  uint32_t m = 0;  // max of |bf16| bit patterns (sign cleared): orders like the values
  // four independent 16-byte loads in flight per thread
  for (long long i0 = lo + threadIdx.x; i0 < hi; i0 += 4 * fp8::kThreads) {
    uint4 v[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const long long i = i0 + a * fp8::kThreads;
      v[a] = i < hi ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const uint32_t w[4] = {v[a].x, v[a].y, v[a].z, v[a].w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        m = max(m, w[t] & 0x7fffu);
        m = max(m, (w[t] >> 16) & 0x7fffu);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ uint32_t red[fp8::kThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < fp8::kThreads / 32; ++w) m = max(m, red[w]);
    if (hi > lo) atomicMax(amax_bits + bh, m << 16);  // bf16 bits -> fp32 bits
  }
}

__device__ __forceinline__ float fp8_scale(unsigned amax_bits) {
  const float amax = __uint_as_float(amax_bits);
  return amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
}

// Eight bf16 values (one 16-byte vector) times s -> eight E4M3 codes.
__device__ __forceinline__ uint2 quant8(uint4 v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float f[8];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    f[2 * t] = __fmul_rn(__uint_as_float(w[t] << 16), s);
    f[2 * t + 1] = __fmul_rn(__uint_as_float(w[t] & 0xffff0000u), s);
  }
  return make_uint2(pack_e4m3x4(f[0], f[1], f[2], f[3]), pack_e4m3x4(f[4], f[5], f[6], f[7]));
}

// Codes in the input's own layout [BH, N, d].  Grid (chunks, BH).
__global__ void __launch_bounds__(fp8::kThreads) fa_quant_rows_kernel(
    const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ out,
    const unsigned* __restrict__ amax_bits, long long slice_vecs, long long vecs_per_chunk) {
  const int bh = blockIdx.y;
  const float s = fp8_scale(__ldg(amax_bits + bh));
  const long long lo = static_cast<long long>(blockIdx.x) * vecs_per_chunk;
  const long long hi = min(slice_vecs, lo + vecs_per_chunk);
  const uint4* src = reinterpret_cast<const uint4*>(x) + static_cast<long long>(bh) * slice_vecs;
  uint2* dst = reinterpret_cast<uint2*>(out) + static_cast<long long>(bh) * slice_vecs;
  for (long long i0 = lo + threadIdx.x; i0 < hi; i0 += 4 * fp8::kThreads) {
    uint4 v[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const long long i = i0 + a * fp8::kThreads;
      if (i < hi) v[a] = __ldg(src + i);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const long long i = i0 + a * fp8::kThreads;
      if (i < hi) dst[i] = quant8(v[a], s);
    }
  }
}

// Codes keys-last: out[bh][t][n] for t < D, n < pitch (pitch = N rounded up
// to 16; columns N..pitch-1 are 0).  Grid (ceil(N / 64), BH): a CTA converts
// 64 keys x D into shared memory and writes them back transposed in 16-byte
// runs of 16 keys.
template <int D>
__global__ void __launch_bounds__(fp8::kThreads) fa_quant_keys_last_kernel(
    const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ out,
    const unsigned* __restrict__ amax_bits, int N, int pitch) {
  constexpr int kRow = D + 4;  // padded row: the column reads below spread over the banks
  __shared__ __align__(16) uint8_t tile[fp8::kTileKeys * kRow];
  const int bh = blockIdx.y;
  const int n0 = blockIdx.x * fp8::kTileKeys;
  const float s = fp8_scale(__ldg(amax_bits + bh));
  constexpr int kVecsPerRow = D / fp8::kVec;
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(bh) * N * D);
#pragma unroll
  for (int i = threadIdx.x; i < fp8::kTileKeys * kVecsPerRow; i += fp8::kThreads) {
    const int r = i / kVecsPerRow, c = (i % kVecsPerRow) * fp8::kVec;
    uint2 q = make_uint2(0u, 0u);  // keys >= N: code 0
    if (n0 + r < N) q = quant8(__ldg(src + static_cast<size_t>(n0 + r) * kVecsPerRow + c / fp8::kVec), s);
    *reinterpret_cast<uint32_t*>(tile + r * kRow + c) = q.x;
    *reinterpret_cast<uint32_t*>(tile + r * kRow + c + 4) = q.y;
  }
  __syncthreads();
  uint8_t* dst = out + static_cast<size_t>(bh) * D * pitch;
  constexpr int kRuns = fp8::kTileKeys / 16;
  for (int i = threadIdx.x; i < D * kRuns; i += fp8::kThreads) {
    const int t = i / kRuns, g = i % kRuns;
    const int n = n0 + 16 * g;
    if (n >= pitch) continue;  // pitch is a multiple of 16: a run is all in or all out
    uint32_t w[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      uint32_t b = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) b |= static_cast<uint32_t>(tile[(16 * g + 4 * a + e) * kRow + t]) << (8 * e);
      w[a] = b;
    }
    *reinterpret_cast<uint4*>(dst + static_cast<size_t>(t) * pitch + n) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// descale[bh] = amax / 448, written over the maxima (same buffer).
__global__ void fa_descale_kernel(float* __restrict__ descale, int BH) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < BH) descale[i] = __fdiv_rn(descale[i], 448.f);
}

// ------------------------------------------- Q, K and V in four launches
// The same arithmetic as the kernels above, for three tensors at once
// (blockIdx.z: 0 = Q, 1 = K, 2 = V), V written keys-last.

struct Qkv3 {
  const __nv_bfloat16* x[3];
  uint8_t* out[3];
  float* descale[3];
};

// Selects by a runtime index without indexing the parameter array (which
// would copy it to local memory).
template <typename T>
__device__ __forceinline__ T pick3(const T (&a)[3], int z) {
  return z == 0 ? a[0] : (z == 1 ? a[1] : a[2]);
}

__global__ void fa_zero3_kernel(Qkv3 a, int BH) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < BH) {
    a.descale[0][i] = 0.f;
    a.descale[1][i] = 0.f;
    a.descale[2][i] = 0.f;
  }
}

__global__ void __launch_bounds__(fp8::kThreads) fa_amax3_kernel(Qkv3 a, long long slice_vecs,
                                                                 long long vecs_per_chunk) {
  const int z = blockIdx.z;
  const int bh = blockIdx.y;
  const long long lo = static_cast<long long>(blockIdx.x) * vecs_per_chunk;
  const long long hi = min(slice_vecs, lo + vecs_per_chunk);
  const uint4* src = reinterpret_cast<const uint4*>(pick3(a.x, z)) + static_cast<long long>(bh) * slice_vecs;
  uint32_t m = 0;
  for (long long i0 = lo + threadIdx.x; i0 < hi; i0 += 4 * fp8::kThreads) {
    uint4 v[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const long long i = i0 + t * fp8::kThreads;
      v[t] = i < hi ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t w[4] = {v[t].x, v[t].y, v[t].z, v[t].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        m = max(m, w[e] & 0x7fffu);
        m = max(m, (w[e] >> 16) & 0x7fffu);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ uint32_t red[fp8::kThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < fp8::kThreads / 32; ++w) m = max(m, red[w]);
    if (hi > lo) atomicMax(reinterpret_cast<unsigned*>(pick3(a.descale, z)) + bh, m << 16);
  }
}

// z < 2: codes in rows, chunked as fa_quant_rows_kernel (blockIdx.x <
// chunks); z = 2: keys-last tiles of 64 keys as fa_quant_keys_last_kernel
// (blockIdx.x < ceil(N / 64)).  Blocks past a tensor's own range return.
template <int D>
__global__ void __launch_bounds__(fp8::kThreads) fa_quant3_kernel(Qkv3 a, int N, int pitch,
                                                                  long long slice_vecs,
                                                                  long long vecs_per_chunk,
                                                                  int chunks) {
  const int z = blockIdx.z;
  const int bh = blockIdx.y;
  const float s = fp8_scale(__ldg(reinterpret_cast<const unsigned*>(pick3(a.descale, z)) + bh));
  if (z < 2) {
    if (static_cast<int>(blockIdx.x) >= chunks) return;
    const long long lo = static_cast<long long>(blockIdx.x) * vecs_per_chunk;
    const long long hi = min(slice_vecs, lo + vecs_per_chunk);
    const uint4* src = reinterpret_cast<const uint4*>(z == 0 ? a.x[0] : a.x[1]) + static_cast<long long>(bh) * slice_vecs;
    uint2* dst = reinterpret_cast<uint2*>(z == 0 ? a.out[0] : a.out[1]) + static_cast<long long>(bh) * slice_vecs;
    for (long long i0 = lo + threadIdx.x; i0 < hi; i0 += 4 * fp8::kThreads) {
      uint4 v[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const long long i = i0 + t * fp8::kThreads;
        if (i < hi) v[t] = __ldg(src + i);
      }
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const long long i = i0 + t * fp8::kThreads;
        if (i < hi) dst[i] = quant8(v[t], s);
      }
    }
    return;
  }
  const int n0 = blockIdx.x * fp8::kTileKeys;
  if (n0 >= N) return;
  constexpr int kRow = D + 4;
  __shared__ __align__(16) uint8_t tile[fp8::kTileKeys * kRow];
  constexpr int kVecsPerRow = D / fp8::kVec;
  const uint4* src = reinterpret_cast<const uint4*>(a.x[2] + static_cast<size_t>(bh) * N * D);
#pragma unroll
  for (int i = threadIdx.x; i < fp8::kTileKeys * kVecsPerRow; i += fp8::kThreads) {
    const int r = i / kVecsPerRow, c = (i % kVecsPerRow) * fp8::kVec;
    uint2 q = make_uint2(0u, 0u);
    if (n0 + r < N) q = quant8(__ldg(src + static_cast<size_t>(n0 + r) * kVecsPerRow + c / fp8::kVec), s);
    *reinterpret_cast<uint32_t*>(tile + r * kRow + c) = q.x;
    *reinterpret_cast<uint32_t*>(tile + r * kRow + c + 4) = q.y;
  }
  __syncthreads();
  uint8_t* dst = a.out[2] + static_cast<size_t>(bh) * D * pitch;
  constexpr int kRuns = fp8::kTileKeys / 16;
  for (int i = threadIdx.x; i < D * kRuns; i += fp8::kThreads) {
    const int t = i / kRuns, g = i % kRuns;
    const int n = n0 + 16 * g;
    if (n >= pitch) continue;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t b = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) b |= static_cast<uint32_t>(tile[(16 * g + 4 * q + e) * kRow + t]) << (8 * e);
      w[q] = b;
    }
    *reinterpret_cast<uint4*>(dst + static_cast<size_t>(t) * pitch + n) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

__global__ void fa_descale3_kernel(Qkv3 a, int BH) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < BH) {
    float* ds = pick3(a.descale, static_cast<int>(blockIdx.y));
    ds[i] = __fdiv_rn(ds[i], 448.f);
  }
}

}  // namespace fa
