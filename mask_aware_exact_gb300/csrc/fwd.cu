// Forward kernel: exact attention over the non-FULL tiles of one 128-row query
// block ("FlashMask: Efficient and Rich Mask Extension of FlashAttention",
// abstract: skip masked computation, exact result; "FlashAttention-3",
// abstract: warp specialisation overlapping TMA data movement with tensor-core
// work, and block-wise matmul interleaved with softmax).
//
// One CTA = one (batch, head, query block). Warp roles (320 threads):
//   warps 0-7  softmax, two warpgroups. Warpgroup g handles key columns
//              [64g, 64g+64) of every tile; thread (g, r) owns query row r
//              (= TMEM lane r). Each tile: read its half of S from TMEM, apply
//              the element mask on PARTIAL tiles, exchange the half-row maxima
//              through shared memory (one named barrier), keep the running max
//              and partial sum in fp32 (log2 domain), write its half of P as
//              bf16 into TMEM, and rescale its half of the O columns when the
//              max grows by more than 2^8 (lazy rescaling: exact after the
//              final division). Finally O = acc / l and LSE.
//   warp 8     TMA producer: Q once, then K and V tiles of each non-FULL key
//              block into a three-stage ring.
//   warp 9     MMA issuer (one thread): S_t = Q K_t^T (both operands in shared
//              memory, K-major) and O += P_{t-1} V_{t-1} (P from TMEM, V
//              MN-major), so the next S overlaps the current softmax.
//
// TMEM columns (512 allocated): S0 [0,128) S1 [128,256) P0 [256,320)
// P1 [320,384) O [384, 384+d). No region is ever written by one MMA while
// another MMA may still read it: every reuse is ordered by an mbarrier.
#include "internal.h"
#include "ptx.cuh"
#include "flashmask.h"

namespace fm {

namespace {

constexpr int kStages = 3;
constexpr int kThreads = 320;
constexpr uint32_t kColS0 = 0, kColP0 = 256, kColO = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct FwdLayout {
  static constexpr int kTileBytes = kTile * D * 2;  // one 128 x d bf16 tile
  static constexpr int kChunks = D / 64;            // 64-column (128-byte) TMA boxes
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kRed = kV + kStages * kTileBytes;  // fp32 [2 parity][2 group][128]
  static constexpr int kBar = kRed + 2 * 2 * kTile * 4;
  // barriers: q_full, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], p_full[2], o_ready
  static constexpr int kNumBars = 1 + 4 * kStages + 2 + 2 + 1;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kBytes = kTmemSlot + 16;
};

struct FwdBars {
  uint32_t base;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t k_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t k_empty(int s) const { return base + 8 * (1 + kStages + s); }
  __device__ uint32_t v_full(int s) const { return base + 8 * (1 + 2 * kStages + s); }
  __device__ uint32_t v_empty(int s) const { return base + 8 * (1 + 3 * kStages + s); }
  __device__ uint32_t s_full(int b) const { return base + 8 * (1 + 4 * kStages + b); }
  __device__ uint32_t p_full(int b) const { return base + 8 * (3 + 4 * kStages + b); }
  __device__ uint32_t o_ready() const { return base + 8 * (5 + 4 * kStages); }
};

__device__ __forceinline__ void record_failure(int32_t* status, int bit, int site) {
  atomicOr(&status[0], bit);
  atomicCAS(&status[1], 0, site);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The 256 softmax threads (both warpgroups).
__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv, const FwdParams p) {
  using L = FwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // work item: blocks of equal rank (work order) across all heads come together
  const int BH = p.B * p.H;
  const int rank = blockIdx.x / BH, bh = blockIdx.x % BH;
  const int b = bh / p.H, h = bh % p.H;
  const int bm = b * p.mask.Hm + h / (p.H / p.mask.Hm);
  const int r = p.row_order[static_cast<size_t>(bm) * p.Tr + rank];
  const int ntiles = p.row_count[static_cast<size_t>(bm) * p.Tr + r];
  const int32_t* list = p.row_list + (static_cast<size_t>(bm) * p.Tr + r) * p.Tc;
  const int head_row0 = bh * p.N;           // first row of this head in [B*H*N, d]
  const int q_row0 = head_row0 + r * kTile;  // first query row of the block

  if ((smem_u32(smem) & 1023u) != 0) {  // 128-byte swizzle atoms need 1024-byte alignment
    if (tid == 0) record_failure(p.status, kStatusLayout, kSiteFwdSmemAlign);
    return;
  }
  const uint32_t sQ = smem_u32(smem + L::kQ), sK = smem_u32(smem + L::kK),
                 sV = smem_u32(smem + L::kV);
  float* red = reinterpret_cast<float*>(smem + L::kRed);
  const FwdBars bar{smem_u32(smem + L::kBar)};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);

  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar.q_full(), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar.k_full(s), 1);
      mbar_init(bar.k_empty(s), 1);
      mbar_init(bar.v_full(s), 1);
      mbar_init(bar.v_empty(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar.s_full(s), 1);
      mbar_init(bar.p_full(s), 8);
    }
    mbar_init(bar.o_ready(), 1);
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && ntiles > 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mv);
      mbar_arrive_expect_tx(bar.q_full(), L::kTileBytes);
      for (int ch = 0; ch < L::kChunks; ++ch)
        tma_load_2d(sQ + ch * 16384, &mq, ch * 64, q_row0, bar.q_full());
      for (int t = 0; t < ntiles; ++t) {
        const int st = t % kStages, n = t / kStages;
        const int krow = head_row0 + (list[t] >> 2) * kTile;
        if (t >= kStages && !mbar_wait(bar.k_empty(st), (n - 1) & 1, p.status)) {
          record_failure(p.status, kStatusTimeout, kSiteFwdKEmpty);
          break;
        }
        mbar_arrive_expect_tx(bar.k_full(st), L::kTileBytes);
        for (int ch = 0; ch < L::kChunks; ++ch)
          tma_load_2d(sK + st * L::kTileBytes + ch * 16384, &mk, ch * 64, krow, bar.k_full(st));
        if (t >= kStages && !mbar_wait(bar.v_empty(st), (n - 1) & 1, p.status)) {
          record_failure(p.status, kStatusTimeout, kSiteFwdVEmpty);
          break;
        }
        mbar_arrive_expect_tx(bar.v_full(st), L::kTileBytes);
        for (int ch = 0; ch < L::kChunks; ++ch)
          tma_load_2d(sV + st * L::kTileBytes + ch * 16384, &mv, ch * 64, krow, bar.v_full(st));
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16(128, D, 0, 1);
      bool ok = mbar_wait(bar.q_full(), 0, p.status);
      if (!ok) record_failure(p.status, kStatusTimeout, kSiteFwdQ);
      for (int t = 0; ok && t <= ntiles; ++t) {
        if (t < ntiles) {
          const int st = t % kStages, sb = t & 1;
          if (!mbar_wait(bar.k_full(st), (t / kStages) & 1, p.status)) {
            record_failure(p.status, kStatusTimeout, kSiteFwdK);
            break;
          }
          tc_fence_after();
          const uint32_t kb = sK + st * L::kTileBytes;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
            mma_ss(tmem + kColS0 + sb * 128, sdesc_sw128(sQ + off, 16, 1024),
                   sdesc_sw128(kb + off, 16, 1024), idesc_s, k > 0);
          }
          if (t + kStages < ntiles) mma_commit(bar.k_empty(st));
          mma_commit(bar.s_full(sb));
        }
        if (t >= 1) {
          const int u = t - 1, pb = u & 1, st = u % kStages;
          if (!mbar_wait(bar.p_full(pb), (u >> 1) & 1, p.status)) {
            record_failure(p.status, kStatusTimeout, kSiteFwdP);
            break;
          }
          if (!mbar_wait(bar.v_full(st), (u / kStages) & 1, p.status)) {
            record_failure(p.status, kStatusTimeout, kSiteFwdV);
            break;
          }
          tc_fence_after();
          const uint32_t vb = sV + st * L::kTileBytes;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ts(tmem + kColO, tmem + kColP0 + pb * 64 + k * 8,
                   sdesc_sw128(vb + k * 2048, 16384, 1024), idesc_pv, (u > 0 || k > 0));
          if (u + kStages < ntiles) mma_commit(bar.v_empty(st));
          mma_commit(bar.o_ready());
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int g = warp >> 2;                 // warpgroup: key columns [64g, 64g+64)
    const int row = (warp & 3) * 32 + lane;  // query row within the block = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // The tile list and the bounds of a PARTIAL tile's key columns are read one
    // tile ahead so their global-memory latency overlaps the current tile.
    auto load_bounds = [&](int entry, int (&bd)[2][4]) {
      if ((entry & 3) != FM_TILE_PARTIAL) return;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const size_t col = static_cast<size_t>(bm) * p.N + (entry >> 2) * kTile + 64 * g + 32 * k + lane;
        bd[k][0] = p.mask.lts[col];
        bd[k][1] = p.mask.lte[col];
        bd[k][2] = p.mask.uts ? p.mask.uts[col] : 0;
        bd[k][3] = p.mask.ute ? p.mask.ute[col] : 0;
      }
    };
    int next_entry = ntiles > 0 ? list[0] : 0;
    int next_bd[2][4];
    load_bounds(next_entry, next_bd);
    for (int t = 0; t < ntiles; ++t) {
      const int sb = t & 1;
      const int entry = next_entry;
      int bd[2][4];
#pragma unroll
      for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int q = 0; q < 4; ++q) bd[k][q] = next_bd[k][q];
      if (t + 1 < ntiles) {
        next_entry = list[t + 1];
        load_bounds(next_entry, next_bd);
      }
      const int kc = entry >> 2, lab = entry & 3;
      // PARTIAL tile: lane l builds the masked-row bits of key column
      // 64g + 32k + l for this warp's 32 rows; a bit transpose hands each
      // lane its own row's bits over those 32 columns.
      uint32_t mbits[2] = {0u, 0u};
      if (lab == FM_TILE_PARTIAL) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int j = kc * kTile + 64 * g + 32 * k + lane;
          mbits[k] = warp_transpose_bits(column_mask_bits(j, bd[k][0], bd[k][1], bd[k][2],
                                                          bd[k][3], p.mask.causal != 0,
                                                          r * kTile + 32 * (warp & 3)));
        }
      }
      if (!mbar_wait(bar.s_full(sb), (t >> 1) & 1, p.status)) {
        record_failure(p.status, kStatusTimeout, kSiteFwdS);
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[64];
      {
        const uint32_t a = tmem + lane_base + kColS0 + sb * 128 + 64 * g;
        tmem_ld64(a, a + 32, sv);
      }
      if (lab == FM_TILE_PARTIAL) {
#pragma unroll
        for (int jj = 0; jj < 64; ++jj)
          sv[jj] = ((mbits[jj >> 5] >> (jj & 31)) & 1u) ? 0xff800000u : sv[jj];  // -inf
      }
      float mx0 = __uint_as_float(sv[0]), mx1 = __uint_as_float(sv[1]);
      float mx2 = __uint_as_float(sv[2]), mx3 = __uint_as_float(sv[3]);
#pragma unroll
      for (int jj = 4; jj < 64; jj += 4) {
        mx0 = fmaxf(mx0, __uint_as_float(sv[jj]));
        mx1 = fmaxf(mx1, __uint_as_float(sv[jj + 1]));
        mx2 = fmaxf(mx2, __uint_as_float(sv[jj + 2]));
        mx3 = fmaxf(mx3, __uint_as_float(sv[jj + 3]));
      }
      const float pm = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c;
      // exchange half-row maxima (double-buffered by tile parity)
      red[(sb * 2 + g) * kTile + row] = pm;
      softmax_bar();
      const float mx = fmaxf(pm, red[(sb * 2 + (g ^ 1)) * kTile + row]);
      const float m_new = fmaxf(m, mx);
      const bool rescale = m_new > m + kRescaleThreshold;
      float alpha = 1.f;
      if (rescale) {
        alpha = ex2(m - m_new);
        m = m_new;
      }
      const float m_use = (m == -INFINITY) ? 0.f : m;
      float l0 = 0.f, l1 = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float p0 = ex2(fmaf(__uint_as_float(sv[2 * i]), c, -m_use));
        const float p1 = ex2(fmaf(__uint_as_float(sv[2 * i + 1]), c, -m_use));
        l0 += p0;
        l1 += p1;
        pk[i] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + (l0 + l1);
      tmem_st32p(tmem + lane_base + kColP0 + sb * 64 + 32 * g, pk);
      if (t >= 1) {
        // O must hold every earlier P V before it is rescaled (and before the
        // P buffer of tile t+1 is rewritten)
        if (!mbar_wait(bar.o_ready(), (t - 1) & 1, p.status)) {
          record_failure(p.status, kStatusTimeout, kSiteFwdO);
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int ch = 0; ch < D / 64; ++ch) {
            uint32_t v[32];
            const uint32_t addr = tmem + lane_base + kColO + g * (D / 2) + ch * 32;
            tmem_ld32(addr, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st32(addr, v);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.p_full(sb));
    }
    // ------------------------------------------------------------ epilogue
    if (ok && ntiles > 0) {
      if (!mbar_wait(bar.o_ready(), (ntiles - 1) & 1, p.status)) {
        record_failure(p.status, kStatusTimeout, kSiteFwdO);
        ok = false;
      }
      tc_fence_after();
    }
    // row sums through the exchange buffer of the parity the last tile did not
    // use (its previous readers passed the last tile's barrier)
    float* lsum = red + (ntiles & 1) * 2 * kTile;
    lsum[g * kTile + row] = l;
    softmax_bar();
    const float ltot = l + lsum[(g ^ 1) * kTile + row];
    const bool live = ok && ntiles > 0;
    const bool has = live && ltot > 0.f;
    const float inv = has ? 1.f / ltot : 0.f;
    uint16_t* orow = p.o + static_cast<size_t>(q_row0 + row) * D + g * (D / 2);
#pragma unroll
    for (int ch = 0; ch < D / 64; ++ch) {
      uint32_t v[32];
      if (live) {
        tmem_ld32(tmem + lane_base + kColO + g * (D / 2) + ch * 32, v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0u;
      }
      store_row32_bf16(orow + ch * 32, v, inv);
    }
    if (g == 0) {
      const float m_fin = (m == -INFINITY) ? 0.f : m;
      p.lse[q_row0 + row] = has ? (m_fin + __log2f(ltot)) * 0.69314718055994531f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_fwd_t(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const FwdParams& p, cudaStream_t s) {
  using L = FwdLayout<D>;
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       L::kBytes);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(p.B * p.H * p.Tr);
  fwd_kernel<D><<<grid, kThreads, L::kBytes, s>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int d, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       const FwdParams& p, cudaStream_t s) {
  if (d == 64) return launch_fwd_t<64>(mq, mk, mv, p, s);
  return launch_fwd_t<128>(mq, mk, mv, p, s);
}

}  // namespace fm
