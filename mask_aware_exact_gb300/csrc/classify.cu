// Tile-classification pre-pass.
//
// "FlashMask: Efficient and Rich Mask Extension of FlashAttention" (abstract):
// the column-wise representation lets the kernels skip computation the mask
// makes unnecessary. Here every (query block, key block) tile of 128 x 128 gets
// its exact three-way label, computed from the boundary vectors without ever
// forming the mask:
//
//  * Column j masks the union of up to three row intervals: [0, j) when causal,
//    [LTS_j, LTE_j) and [UTS_j, UTE_j), each clamped to [0, N]. After sorting
//    and merging, the union is a list of disjoint, non-adjacent intervals.
//  * A merged interval [s, e) fully covers row block r iff ceil(s/128) <= r <
//    floor(e/128), and touches it iff floor(s/128) <= r < ceil(e/128). Both are
//    ranges of r, so the 128 columns of a key block add +1/-1 into two
//    difference arrays over r; a prefix sum gives, per row block, how many
//    columns cover it fully and how many touch it.
//  * FULL iff all columns of the key block cover the block fully; NONE iff no
//    column touches it; otherwise PARTIAL.
//  * N need not be a multiple of 128: the last blocks are short. Only rows and
//    columns < N exist, so the label is exact over the existing entries; an
//    interval that reaches row N covers the short last row block to its end,
//    and columns >= N take no part (the attention kernels mask them).
//
// The same pass writes the per-key-block min/max of each vector, the labels in
// both tile orders, the ascending lists of non-FULL tiles per key block and
// (second kernel) per query block, and (third kernel) each block index ranked
// by descending amount of work, which the attention kernels use as their
// launch order (longest first).
#include <climits>

#include "internal.h"
#include "flashmask.h"

namespace fm {

namespace {

// Inclusive prefix sum over the 128 threads of the block; `total` receives the
// block-wide sum. Every thread of the block must call it.
__device__ __forceinline__ int block_scan128(int v, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[w] = x;
  __syncthreads();
  int pre = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = warp_tot[i];
    pre += (i < w) ? t : 0;
    tot += t;
  }
  __syncthreads();
  total = tot;
  return x + pre;
}

__global__ void __launch_bounds__(128) classify_cols_kernel(MaskDev m, int N, int Tr, int Tc,
                                                            ClassifyTables t) {
  extern __shared__ int sh[];
  int* full_d = sh;             // [Tr + 1]
  int* touch_d = sh + Tr + 1;   // [Tr + 1]
  __shared__ int warp_tot[4];
  __shared__ int red[4][8];
  const int c = blockIdx.x, bm = blockIdx.y, tid = threadIdx.x;
  const int lane = tid & 31, w = tid >> 5;
  for (int i = tid; i < 2 * (Tr + 1); i += 128) sh[i] = 0;

  const size_t base = static_cast<size_t>(bm) * N;
  const int j = c * kTile + tid;
  const bool exists = j < N;                 // the last key block may be short
  const int ncols = min(kTile, N - c * kTile);
  const int Npad = Tr * kTile;
  int v[4] = {0, 0, 0, 0};
  if (exists) {
    v[0] = m.lts[base + j];
    v[1] = m.lte[base + j];
    v[2] = m.uts ? m.uts[base + j] : 0;
    v[3] = m.ute ? m.ute[base + j] : 0;
  }

  // per-key-block min / max of each vector
  int mm[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    mm[2 * k] = exists ? v[k] : INT_MAX;
    mm[2 * k + 1] = exists ? v[k] : INT_MIN;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      mm[2 * k] = min(mm[2 * k], __shfl_xor_sync(0xffffffffu, mm[2 * k], o));
      mm[2 * k + 1] = max(mm[2 * k + 1], __shfl_xor_sync(0xffffffffu, mm[2 * k + 1], o));
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int q = 0; q < 8; ++q) red[w][q] = mm[q];
  }
  __syncthreads();  // also orders the zeroing of the difference arrays
  if (tid < 8) {
    int r = red[0][tid];
    for (int q = 1; q < 4; ++q) r = (tid & 1) ? max(r, red[q][tid]) : min(r, red[q][tid]);
    t.minmax[(static_cast<size_t>(bm) * Tc + c) * 8 + tid] = r;
  }

  // masked row intervals of column j, clamped to [0, N]; an end at N is
  // extended to the padded row count so that it covers the short last block
  int s[3], e[3], n = 0;
  auto add = [&](int a0, int a1) {
    a0 = max(a0, 0);
    a1 = min(a1, N);
    if (a0 < a1) {
      s[n] = a0;
      e[n] = a1 == N ? Npad : a1;
      ++n;
    }
  };
  if (exists) {
    if (m.causal) add(0, j);
    add(v[0], v[1]);
    add(v[2], v[3]);
  }
  // sort by start (at most three)
  for (int a = 0; a < n; ++a)
    for (int b = a + 1; b < n; ++b)
      if (s[b] < s[a]) {
        int ts = s[a]; s[a] = s[b]; s[b] = ts;
        int te = e[a]; e[a] = e[b]; e[b] = te;
      }
  // merge overlapping or adjacent intervals, then mark block ranges
  int cs = 0, ce = -1;
  for (int a = 0; a <= n; ++a) {
    const bool flush = (a == n) || (ce >= 0 && s[a] > ce);
    if (flush && ce >= 0) {
      const int tlo = cs / kTile, thi = (ce + kTile - 1) / kTile;
      atomicAdd(&touch_d[tlo], 1);
      atomicAdd(&touch_d[thi], -1);
      const int flo = (cs + kTile - 1) / kTile, fhi = ce / kTile;
      if (flo < fhi) {
        atomicAdd(&full_d[flo], 1);
        atomicAdd(&full_d[fhi], -1);
      }
      ce = -1;
    }
    if (a == n) break;
    if (ce < 0) {
      cs = s[a];
      ce = e[a];
    } else {
      ce = max(ce, e[a]);
    }
  }
  __syncthreads();

  int carry_full = 0, carry_touch = 0, carry_cnt = 0;
  for (int r0 = 0; r0 < Tr; r0 += kTile) {
    const int r = r0 + tid;
    const int fd = r < Tr ? full_d[r] : 0;
    const int td = r < Tr ? touch_d[r] : 0;
    int tot;
    const int fc = block_scan128(fd, warp_tot, tot) + carry_full;
    carry_full += tot;
    const int tc = block_scan128(td, warp_tot, tot) + carry_touch;
    carry_touch += tot;
    const int lab = (fc == ncols) ? FM_TILE_FULL : (tc == 0 ? FM_TILE_NONE : FM_TILE_PARTIAL);
    const int keep = (r < Tr && lab != FM_TILE_FULL) ? 1 : 0;
    const int pos = block_scan128(keep, warp_tot, tot) - keep + carry_cnt;
    carry_cnt += tot;
    if (r < Tr) {
      t.labels_t[(static_cast<size_t>(bm) * Tc + c) * Tr + r] = static_cast<uint8_t>(lab);
      t.labels[(static_cast<size_t>(bm) * Tr + r) * Tc + c] = static_cast<uint8_t>(lab);
      if (keep) t.col_list[(static_cast<size_t>(bm) * Tc + c) * Tr + pos] = (r << 2) | lab;
    }
  }
  if (tid == 0) t.col_count[static_cast<size_t>(bm) * Tc + c] = carry_cnt;
}

__global__ void __launch_bounds__(128) classify_rows_kernel(int Tr, int Tc, ClassifyTables t) {
  __shared__ int warp_tot[4];
  const int r = blockIdx.x, bm = blockIdx.y, tid = threadIdx.x;
  const uint8_t* lab_row = t.labels + (static_cast<size_t>(bm) * Tr + r) * Tc;
  int32_t* list = t.row_list + (static_cast<size_t>(bm) * Tr + r) * Tc;
  int carry = 0;
  for (int c0 = 0; c0 < Tc; c0 += kTile) {
    const int c = c0 + tid;
    const int lab = c < Tc ? lab_row[c] : FM_TILE_FULL;
    const int keep = lab != FM_TILE_FULL ? 1 : 0;
    int tot;
    const int pos = block_scan128(keep, warp_tot, tot) - keep + carry;
    carry += tot;
    if (keep) list[pos] = (c << 2) | lab;
  }
  if (tid == 0) t.row_count[static_cast<size_t>(bm) * Tr + r] = carry;
}

// Ranks block indices by descending count (ties: ascending index) and writes
// order[rank] = index. blockIdx.y = 0 ranks query blocks, 1 key blocks;
// blockIdx.z takes indices [256 z, 256 z + 256).
__global__ void __launch_bounds__(256) classify_order_kernel(int Tr, int Tc, ClassifyTables t) {
  extern __shared__ int cnt[];
  const int bm = blockIdx.x;
  const int which = blockIdx.y;
  const int i0 = blockIdx.z * blockDim.x;
  const int n = which == 0 ? Tr : Tc;
  const int32_t* src = which == 0 ? t.row_count + static_cast<size_t>(bm) * Tr
                                  : t.col_count + static_cast<size_t>(bm) * Tc;
  int32_t* order = which == 0 ? t.row_order + static_cast<size_t>(bm) * Tr
                              : t.col_order + static_cast<size_t>(bm) * Tc;
  for (int i = threadIdx.x; i < n; i += blockDim.x) cnt[i] = src[i];
  __syncthreads();
  {
    const int i = i0 + threadIdx.x;
    if (i >= n) return;
    const int ci = cnt[i];
    int rank = 0;
    for (int k = 0; k < n; ++k) {
      const int ck = cnt[k];
      rank += (ck > ci) || (ck == ci && k < i);
    }
    order[rank] = i;
  }
}

}  // namespace

cudaError_t launch_classify(const MaskDev& m, int B, int N, const ClassifyTables& t,
                            cudaStream_t s) {
  const int Tr = (N + kTile - 1) / kTile, Tc = Tr;
  const int BHm = B * m.Hm;
  const size_t sh_cols = static_cast<size_t>(2) * (Tr + 1) * sizeof(int);
  const size_t sh_order = static_cast<size_t>(Tr) * sizeof(int);
  cudaError_t e;
  if (sh_cols > 48 * 1024) {
    e = cudaFuncSetAttribute(classify_cols_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sh_cols));
    if (e != cudaSuccess) return e;
  }
  if (sh_order > 48 * 1024) {
    e = cudaFuncSetAttribute(classify_order_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sh_order));
    if (e != cudaSuccess) return e;
  }
  classify_cols_kernel<<<dim3(Tc, BHm), 128, sh_cols, s>>>(m, N, Tr, Tc, t);
  classify_rows_kernel<<<dim3(Tr, BHm), 128, 0, s>>>(Tr, Tc, t);
  classify_order_kernel<<<dim3(BHm, 2, (Tr + 255) / 256), 256, sh_order, s>>>(Tr, Tc, t);
  return cudaGetLastError();
}

}  // namespace fm
