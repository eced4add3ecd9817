// Per-rank mask localisation for context parallelism ("FlashMask-3: ... Mask-Aware
// Distributed Attention", abstract: under any multi-chunk context-parallel
// assignment, per-rank mask localisation reduces to a zero-communication
// clip-shift-max on the boundary vectors).
//
// A rank that holds the query rows [row0, row0 + rows) and every key gets the
// boundary vectors of its local problem, in local row coordinates [0, rows):
//   clip + shift  every bound b becomes min(max(b - row0, 0), rows); an interval
//                 [s, e) of masked global rows becomes the local interval of the
//                 same rows inside the chunk (empty if they miss it);
//   max           with the causal flag, key j masks the global rows [0, j), i.e.
//                 the local rows [0, c) with c = clip(j - row0); it joins the
//                 upper interval [u0, u1) as [0, max(c, u1)), which is exact when
//                 that interval is empty or starts at a row <= c (the upper
//                 triangle of a causal mask always does). The local mask then
//                 has no causal flag.
// Only the rank's own copy of the O(N) vectors is read: no communication.
#include <cstdint>

#include <cuda_runtime.h>

#include "flashmask.h"

namespace {

__device__ __forceinline__ int clip_shift(int b, int row0, int rows) {
  // b - row0 computed in 64 bits: any int32 bound is safe
  const long long v = static_cast<long long>(b) - row0;
  return static_cast<int>(v < 0 ? 0 : (v > rows ? rows : v));
}

__global__ void __launch_bounds__(256) localize_kernel(fm_mask m, long long n_total, int N,
                                                       int row0, int rows, int32_t* lts,
                                                       int32_t* lte, int32_t* uts, int32_t* ute,
                                                       int32_t* inexact) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= n_total) return;
  const int j = static_cast<int>(idx % N);  // key index
  const int l0 = clip_shift(m.lts[idx], row0, rows), l1 = clip_shift(m.lte[idx], row0, rows);
  int u0 = m.uts ? clip_shift(m.uts[idx], row0, rows) : 0;
  int u1 = m.ute ? clip_shift(m.ute[idx], row0, rows) : 0;
  if (m.causal) {
    const int c = clip_shift(j, row0, rows);  // local rows [0, c) are above the diagonal
    if (c > 0) {
      if (u0 < u1 && u0 > c && inexact) atomicExch(inexact, 1);  // [0, c) and [u0, u1) apart
      u1 = (u0 < u1) ? max(c, u1) : c;
      u0 = 0;
    }
  }
  lts[idx] = l0;
  lte[idx] = l1;
  uts[idx] = u0;
  ute[idx] = u1;
}

}  // namespace

extern "C" {

fm_status flashmask_localize(const fm_mask* mask, int B, int N, int row0, int rows, int32_t* lts,
                             int32_t* lte, int32_t* uts, int32_t* ute, int32_t* inexact,
                             void* stream) {
  if (!mask || !mask->lts || !mask->lte || ((mask->uts == nullptr) != (mask->ute == nullptr)))
    return FM_ERR_INVALID_ARG;
  if (!lts || !lte || !uts || !ute) return FM_ERR_INVALID_ARG;
  if (B <= 0 || N <= 0 || mask->Hm <= 0) return FM_ERR_UNSUPPORTED;
  if (row0 < 0 || rows <= 0 || static_cast<long long>(row0) + rows > N) return FM_ERR_INVALID_ARG;
  const long long n_total = static_cast<long long>(B) * mask->Hm * N;
  const unsigned grid = static_cast<unsigned>((n_total + 255) / 256);
  localize_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      *mask, n_total, N, row0, rows, lts, lte, uts, ute, inexact);
  return cudaGetLastError() == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}

}  // extern "C"
