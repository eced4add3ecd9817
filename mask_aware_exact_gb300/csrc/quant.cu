// FP8 (e4m3) operands for the FP8 forward ("FlashAttention-3", abstract: FP8
// attention with block quantization). Q and K get one scale per 128-row block
// of a head (the block of the attention tiles); V gets one scale per head and
// is stored transposed ([head][d][Npad], keys contiguous) so that it is the
// K-major B operand of O += P V. A value x becomes e4m3(x * (1 / s)) with
// s = absmax / 448 (448 = the largest finite e4m3), rounding to nearest even
// and saturating; a block or head of zeros gets s = 1. The scale, its
// reciprocal and the product are fp32 operations.
//
// Two HBM-bound passes, both over (head, 128-row block) with 256 threads and
// coalesced 16-byte loads (thread t takes the 16-byte chunks t, t + 256, ...
// of the block's 32 KB):
//   quant_qk_kernel  Q and K blocks -> codes and block scales; the V block's
//                    absolute maximum folded into the head's with an atomic max
//   quant_vt_kernel  V block -> codes with the head's scale, transposed through
//                    shared memory as packed 32-bit words
#include <cstdint>

#include <cuda_runtime.h>

#include "internal.h"
#include "ptx_fp8.cuh"

namespace fm {
namespace {

constexpr float kE4m3Max = 448.f;
constexpr int kQThreads = 256;
constexpr int kChunksPerThread = kTile * 128 * 2 / 16 / kQThreads;  // 8 (d = 128)

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float absmax8(const uint4& q) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float a = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) a = fmaxf(a, fmaxf(fabsf(bf16_lo(w[k])), fabsf(bf16_hi(w[k]))));
  return a;
}

// Maximum over the CTA's 256 threads (every thread gets it).
__device__ __forceinline__ float block_max(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int i = 1; i < kQThreads / 32; ++i) m = fmaxf(m, red[i]);
  __syncthreads();  // red is reused by the next call
  return m;
}

__device__ __forceinline__ float scale_of(float absmax) {
  return absmax > 0.f ? absmax / kE4m3Max : 1.f;
}

// 8 bf16 (one 16-byte chunk) times inv -> 8 e4m3 bytes
__device__ __forceinline__ uint2 chunk_to_e4m3(const uint4& q, float inv) {
  uint2 r;
  r.x = pack_e4m3x4(bf16_lo(q.x) * inv, bf16_hi(q.x) * inv, bf16_lo(q.y) * inv,
                    bf16_hi(q.y) * inv);
  r.y = pack_e4m3x4(bf16_lo(q.z) * inv, bf16_hi(q.z) * inv, bf16_lo(q.w) * inv,
                    bf16_hi(q.w) * inv);
  return r;
}

// Loads this thread's chunks of the 128 rows that start at row0 of x
// ([rows][128] bf16); chunk c covers row c / 16, columns 8 (c % 16) .. +8.
// Rows >= live_rows read as zero.
__device__ __forceinline__ void load_block(const uint16_t* __restrict__ x, size_t row0,
                                           int live_rows, uint4 (&v)[kChunksPerThread]) {
  const uint4* src = reinterpret_cast<const uint4*>(x + row0 * 128);
#pragma unroll
  for (int i = 0; i < kChunksPerThread; ++i) {
    const int c = i * kQThreads + threadIdx.x;
    v[i] = (c >> 4) < live_rows ? src[c] : make_uint4(0u, 0u, 0u, 0u);
  }
}

__device__ void quant_rows_block(const uint16_t* __restrict__ x, size_t row0, int live_rows,
                                 uint8_t* __restrict__ x8, float* __restrict__ scale_out,
                                 float* red) {
  uint4 v[kChunksPerThread];
  load_block(x, row0, live_rows, v);
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < kChunksPerThread; ++i) a = fmaxf(a, absmax8(v[i]));
  const float s = scale_of(block_max(a, red));
  const float inv = 1.f / s;
  if (threadIdx.x == 0) *scale_out = s;
  uint2* dst = reinterpret_cast<uint2*>(x8 + row0 * 128);
#pragma unroll
  for (int i = 0; i < kChunksPerThread; ++i) {
    const int c = i * kQThreads + threadIdx.x;
    if ((c >> 4) < live_rows) dst[c] = chunk_to_e4m3(v[i], inv);
  }
}

// One CTA per (head, 128-row block): Q and K blocks quantised, V block's
// absolute maximum into amax[bh] (zeroed by the caller; an integer atomic max
// orders non-negative floats like their bit patterns).
__global__ void __launch_bounds__(kQThreads) quant_qk_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
    const uint16_t* __restrict__ v, int N, int Tr, uint8_t* __restrict__ q8,
    uint8_t* __restrict__ k8, float* __restrict__ qscale, float* __restrict__ kscale,
    unsigned int* __restrict__ vamax) {
  __shared__ float red[kQThreads / 32];
  const int bh = blockIdx.x / Tr, blk = blockIdx.x % Tr;
  const size_t row0 = static_cast<size_t>(bh) * N + static_cast<size_t>(blk) * kTile;
  const int live = min(kTile, N - blk * kTile);
  const size_t si = static_cast<size_t>(bh) * Tr + blk;
  quant_rows_block(q, row0, live, q8, qscale + si, red);
  quant_rows_block(k, row0, live, k8, kscale + si, red);
  uint4 vv[kChunksPerThread];
  load_block(v, row0, live, vv);
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < kChunksPerThread; ++i) a = fmaxf(a, absmax8(vv[i]));
  const float m = block_max(a, red);
  if (threadIdx.x == 0) atomicMax(&vamax[bh], __float_as_uint(m));
}

// V (bf16 [head][N][128]) -> Vt8 (e4m3 [head][128][Npad]) with the head's
// scale; one CTA per (head, 128-key block). Keys >= N are written as 0.
// Thread (key group kg, column group m) converts keys 4kg .. 4kg+3 at
// columns 8m .. 8m+7 (four coalesced 16-byte loads: 16 threads cover one
// 256-byte row) and stores the transposed bytes as eight 32-bit words, one
// per column, each holding its four keys.
__global__ void __launch_bounds__(kQThreads) quant_vt_kernel(
    const uint16_t* __restrict__ v, int N, int Npad, int Tr,
    const unsigned int* __restrict__ amax, uint8_t* __restrict__ vt8,
    float* __restrict__ vscale) {
  constexpr int kRowWords = 128 / 4 + 1;  // 32-bit words per d row of the tile (+1: banks)
  __shared__ uint32_t tile[128 * kRowWords];  // [d][key / 4]
  const int bh = blockIdx.x / Tr, kb = blockIdx.x % Tr;
  const float s = scale_of(__uint_as_float(amax[bh]));
  const float inv = 1.f / s;
  if (kb == 0 && threadIdx.x == 0) vscale[bh] = s;
  const int m = threadIdx.x & 15, d0 = 8 * m;
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int kg = pass * 16 + (threadIdx.x >> 4);  // keys 4kg .. 4kg+3 of the block
    uint2 b[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int n = kb * kTile + 4 * kg + r;
      const uint4 q = n < N ? *reinterpret_cast<const uint4*>(
                                  v + (static_cast<size_t>(bh) * N + n) * 128 + d0)
                            : make_uint4(0u, 0u, 0u, 0u);
      b[r] = chunk_to_e4m3(q, inv);  // zero chunks give zero codes
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      // byte e of each key's 8 codes (column d0 + e) into one word, key order
      const uint32_t x0 = e < 4 ? b[0].x : b[0].y, x1 = e < 4 ? b[1].x : b[1].y;
      const uint32_t x2 = e < 4 ? b[2].x : b[2].y, x3 = e < 4 ? b[3].x : b[3].y;
      const uint32_t sel = static_cast<uint32_t>(e & 3) | (static_cast<uint32_t>((e & 3) + 4) << 4);
      const uint32_t lo = __byte_perm(x0, x1, sel), hi = __byte_perm(x2, x3, sel);
      tile[(d0 + e) * kRowWords + kg] = __byte_perm(lo, hi, 0x5410);
    }
  }
  __syncthreads();
  // thread = (d row, half): 64 keys of that row as 4 x 16 bytes
  const int dr = threadIdx.x >> 1, half = threadIdx.x & 1;
  const uint32_t* srow = tile + dr * kRowWords + half * 16;
  uint4* dst = reinterpret_cast<uint4*>(vt8 + (static_cast<size_t>(bh) * 128 + dr) * Npad +
                                        static_cast<size_t>(kb) * kTile + half * 64);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    dst[i] = make_uint4(srow[4 * i], srow[4 * i + 1], srow[4 * i + 2], srow[4 * i + 3]);
}

}  // namespace

cudaError_t launch_quant_fp8(const uint16_t* q, const uint16_t* k, const uint16_t* v, int BH,
                             int N, const Fp8Operands& f, cudaStream_t s) {
  const int Tr = (N + kTile - 1) / kTile, Npad = Tr * kTile;
  const unsigned grid = static_cast<unsigned>(BH) * static_cast<unsigned>(Tr);
  cudaError_t e = cudaMemsetAsync(f.vamax, 0, static_cast<size_t>(BH) * 4, s);
  if (e != cudaSuccess) return e;
  quant_qk_kernel<<<grid, kQThreads, 0, s>>>(q, k, v, N, Tr, f.q8, f.k8, f.qscale, f.kscale,
                                             f.vamax);
  quant_vt_kernel<<<grid, kQThreads, 0, s>>>(v, N, Npad, Tr, f.vamax, f.vt8, f.vscale);
  return cudaGetLastError();
}

}  // namespace fm
