// Forward kernel: exact attention over the non-FULL tiles of one 128-row query
// block ("FlashMask: Efficient and Rich Mask Extension of FlashAttention",
// abstract: skip masked computation, exact result; "FlashAttention-3",
// abstract: warp specialisation overlapping TMA data movement with tensor-core
// work, and block-wise matmul interleaved with softmax).
//
// The non-FULL key blocks of the query block are taken two at a time: one step
// computes S = Q [K_a; K_b]^T as a single 128 x 256 product (a tcgen05 MMA with
// N = 256 runs at the tensor core's full rate; N = 128 would run at half), then
// O += P [V_a; V_b] as two K = 128 chains. A list of odd length ends with a
// one-block step.
//
// One CTA = one (batch, head, query block). Warp roles (320 threads):
//   warps 0-7  softmax, two warpgroups. Warpgroup w owns S columns
//              [128w, 128w+128) of every step (key block w of the pair); thread
//              (w, r) owns query row r = TMEM lane r. Per step: read its S
//              slice, apply the element mask on PARTIAL tiles, exchange the two
//              partial row maxima through shared memory, keep the running max
//              and partial sum in fp32 (log2 domain), compute its bf16 P slice
//              in registers while the previous P V product still runs, then
//              write it into TMEM and rescale its half of the O columns when the
//              max grows by more than 2^8 (lazy rescaling: exact after the final
//              division). Finally O = acc / l and LSE.
//   warp 8     TMA producer: Q once; K pairs into a two-slot ring (one step
//              ahead of the V loads); V blocks into a two-slot ring.
//   warp 9     MMA issuer (one thread): S_{u+1} as soon as the softmax has read
//              S_u, then O += P_u V_u.
//
// TMEM columns (512 allocated): S [0,256)  P [256,384)  O [384, 384+d).
// Ordering: S_{u+1} is written after every softmax warp has loaded S_u
// (s_free); P_{u+1} is written after O += P_u V_u has completed (o_ready).
#include "internal.h"
#include "ptx.cuh"
#include "flashmask.h"

namespace fm {

namespace {

constexpr int kThreads = 320;
constexpr uint32_t kColS = 0, kColP = 256, kColO = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct FwdLayout {
  static constexpr int kTileBytes = kTile * D * 2;  // one 128 x d bf16 tile
  static constexpr int kChunks = D / 64;            // 64-column (128-byte) TMA boxes
  static constexpr int kChunkQ = 16384;             // 128 rows x 128 bytes
  static constexpr int kChunkK = 32768;             // 256 rows x 128 bytes (a key pair)
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;          // 2 slots x (2 x kTileBytes)
  static constexpr int kV = kK + 2 * 2 * kTileBytes;  // 2 slots x kTileBytes
  static constexpr int kRed = kV + 2 * kTileBytes;    // fp32 [2 parity][2 groups][128]
  static constexpr int kBar = kRed + 2 * 2 * kTile * 4;
  // q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full, s_free, p_full, o_ready
  static constexpr int kNumBars = 13;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kBytes = kTmemSlot + 16;
};

struct FwdBars {
  uint32_t base;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t k_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t k_empty(int s) const { return base + 8 * (3 + s); }
  __device__ uint32_t v_full(int s) const { return base + 8 * (5 + s); }
  __device__ uint32_t v_empty(int s) const { return base + 8 * (7 + s); }
  __device__ uint32_t s_full() const { return base + 8 * 9; }
  __device__ uint32_t s_free() const { return base + 8 * 10; }
  __device__ uint32_t p_full() const { return base + 8 * 11; }
  __device__ uint32_t o_ready() const { return base + 8 * 12; }
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

// Multiplies kOCols (16 or 32) consecutive TMEM columns of this warp's lanes by f.
template <int n>
__device__ __forceinline__ void tmem_scale_cols(uint32_t taddr, float f) {
  if constexpr (n == 32) {
    uint32_t v[32];
    tmem_ld32(taddr, v);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
    tmem_st32(taddr, v);
  } else {
    uint32_t v[16];
    tmem_ld16(taddr, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
    tmem_st16(taddr, v);
  }
}

// Writes kOCols (16 or 32) TMEM columns of this lane's row, times f, as bf16.
template <int n>
__device__ __forceinline__ void tmem_cols_to_bf16(uint32_t taddr, bool live, float f,
                                                  uint16_t* dst) {
  uint32_t v[n];
  if (live) {
    if constexpr (n == 32) {
      tmem_ld32(taddr, v);
    } else {
      tmem_ld16(taddr, v);
    }
  } else {
#pragma unroll
    for (int i = 0; i < n; ++i) v[i] = 0u;
  }
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < n / 8; ++i) {
    uint4 q4;
    q4.x = pack_bf16x2(__uint_as_float(v[8 * i + 0]) * f, __uint_as_float(v[8 * i + 1]) * f);
    q4.y = pack_bf16x2(__uint_as_float(v[8 * i + 2]) * f, __uint_as_float(v[8 * i + 3]) * f);
    q4.z = pack_bf16x2(__uint_as_float(v[8 * i + 4]) * f, __uint_as_float(v[8 * i + 5]) * f);
    q4.w = pack_bf16x2(__uint_as_float(v[8 * i + 6]) * f, __uint_as_float(v[8 * i + 7]) * f);
    d4[i] = q4;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv, const FwdParams p) {
  using L = FwdLayout<D>;
  constexpr int kOCols = D / 2;  // O columns per softmax warpgroup
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Work item: head-major, longest query blocks of each head first, so the
  // CTAs that run together share one head's K and V in L2.
  const int bh = blockIdx.x / p.Tr, rank = blockIdx.x % p.Tr;
  const int b = bh / p.H, h = bh % p.H;
  const int bm = b * p.mask.Hm + h / (p.H / p.mask.Hm);
  const int r = p.row_order[static_cast<size_t>(bm) * p.Tr + rank];
  const int ntiles = p.row_count[static_cast<size_t>(bm) * p.Tr + r];
  const int nsteps = (ntiles + 1) >> 1;
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
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar.k_full(s), 1);
      mbar_init(bar.k_empty(s), 1);
      mbar_init(bar.v_full(s), 1);
      mbar_init(bar.v_empty(s), 1);
    }
    mbar_init(bar.s_full(), 1);
    mbar_init(bar.s_free(), 8);
    mbar_init(bar.p_full(), 8);
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
        tma_load_2d(sQ + ch * L::kChunkQ, &mq, ch * 64, q_row0, bar.q_full());
      // K pair of step u into slot u & 1 (rows 0-127: first block, 128-255: second)
      auto load_k = [&](int u) -> bool {
        const int slot = u & 1;
        if (u >= 2 && !mbar_wait(bar.k_empty(slot), ((u >> 1) - 1) & 1, p.status)) {
          record_failure(p.status, kStatusTimeout, kSiteFwdKEmpty);
          return false;
        }
        const int nb = min(2, ntiles - 2 * u);
        mbar_arrive_expect_tx(bar.k_full(slot), nb * L::kTileBytes);
        for (int bb = 0; bb < nb; ++bb) {
          const int krow = head_row0 + (list[2 * u + bb] >> 2) * kTile;
          for (int ch = 0; ch < L::kChunks; ++ch)
            tma_load_2d(sK + slot * 2 * L::kTileBytes + ch * L::kChunkK + bb * L::kChunkQ, &mk,
                        ch * 64, krow, bar.k_full(slot));
        }
        return true;
      };
      bool ok = load_k(0);
      if (ok && nsteps > 1) ok = load_k(1);
      for (int u = 0; ok && u < nsteps; ++u) {
        const int nb = min(2, ntiles - 2 * u);
        for (int bb = 0; bb < nb; ++bb) {
          const int vi = 2 * u + bb, slot = vi & 1;
          if (vi >= 2 && !mbar_wait(bar.v_empty(slot), ((vi >> 1) - 1) & 1, p.status)) {
            record_failure(p.status, kStatusTimeout, kSiteFwdVEmpty);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar.v_full(slot), L::kTileBytes);
          const int vrow = head_row0 + (list[vi] >> 2) * kTile;
          for (int ch = 0; ch < L::kChunks; ++ch)
            tma_load_2d(sV + slot * L::kTileBytes + ch * L::kChunkQ, &mv, ch * 64, vrow,
                        bar.v_full(slot));
        }
        if (ok && u + 2 < nsteps) ok = load_k(u + 2);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t idesc_pv = idesc_bf16(128, D, 0, 1);
      auto issue_s = [&](int u) -> bool {
        const int slot = u & 1;
        if (!mbar_wait(bar.k_full(slot), (u >> 1) & 1, p.status)) {
          record_failure(p.status, kStatusTimeout, kSiteFwdK);
          return false;
        }
        tc_fence_after();
        const int nb = min(2, ntiles - 2 * u);
        const uint32_t idesc_s = nb == 2 ? idesc_bf16(128, 256, 0, 0) : idesc_bf16(128, 128, 0, 0);
        const uint32_t kb = sK + slot * 2 * L::kTileBytes;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          mma_ss(tmem + kColS, sdesc_sw128(sQ + (k >> 2) * L::kChunkQ + (k & 3) * 32, 16, 1024),
                 sdesc_sw128(kb + (k >> 2) * L::kChunkK + (k & 3) * 32, 16, 1024), idesc_s, k > 0);
        }
        if (u + 2 < nsteps) mma_commit(bar.k_empty(slot));
        mma_commit(bar.s_full());
        return true;
      };
      bool ok = mbar_wait(bar.q_full(), 0, p.status);
      if (!ok) record_failure(p.status, kStatusTimeout, kSiteFwdQ);
      if (ok) ok = issue_s(0);
      for (int u = 0; ok && u < nsteps; ++u) {
        if (u + 1 < nsteps) {
          // S_{u+1} overwrites S_u: wait until every softmax warp has loaded it
          if (!mbar_wait(bar.s_free(), u & 1, p.status)) {
            record_failure(p.status, kStatusTimeout, kSiteFwdS);
            break;
          }
          if (!issue_s(u + 1)) break;
        }
        if (!mbar_wait(bar.p_full(), u & 1, p.status)) {
          record_failure(p.status, kStatusTimeout, kSiteFwdP);
          break;
        }
        const int nb = min(2, ntiles - 2 * u);
        for (int bb = 0; bb < nb; ++bb) {
          const int vi = 2 * u + bb, slot = vi & 1;
          if (!mbar_wait(bar.v_full(slot), (vi >> 1) & 1, p.status)) {
            record_failure(p.status, kStatusTimeout, kSiteFwdV);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t vb = sV + slot * L::kTileBytes;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ts(tmem + kColO, tmem + kColP + 64 * bb + 8 * k,
                   sdesc_sw128(vb + k * 2048, 16384, 1024), idesc_pv, (vi > 0 || k > 0));
          if (vi + 2 < ntiles) mma_commit(bar.v_empty(slot));
        }
        if (!ok) break;
        mma_commit(bar.o_ready());
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int w = warp >> 2;                 // warpgroup: key block w of each pair
    const int row = (warp & 3) * 32 + lane;  // query row within the block = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // This warpgroup's list entry of each step, read one step ahead.
    auto entry_of = [&](int u) { return (2 * u + w < ntiles) ? list[2 * u + w] : -1; };
    int next_entry = nsteps > 0 ? entry_of(0) : -1;
    for (int u = 0; u < nsteps; ++u) {
      const int entry = next_entry;
      if (u + 1 < nsteps) next_entry = entry_of(u + 1);
      const bool active = entry >= 0;  // a one-block last step leaves warpgroup 1 idle
      // PARTIAL tile: lane l builds the masked-row bits of key column 32k + l
      // for this warp's 32 rows; a bit transpose hands each lane its own row's
      // bits over those 32 columns. The bound loads overlap the wait for S.
      uint32_t mbits[4] = {0u, 0u, 0u, 0u};
      if (active && (entry & 3) == FM_TILE_PARTIAL) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j = (entry >> 2) * kTile + 32 * k + lane;
          const size_t col = static_cast<size_t>(bm) * p.N + j;
          const int lts = p.mask.lts[col], lte = p.mask.lte[col];
          const int uts = p.mask.uts ? p.mask.uts[col] : 0, ute = p.mask.ute ? p.mask.ute[col] : 0;
          mbits[k] = warp_transpose_bits(column_mask_bits(j, lts, lte, uts, ute,
                                                          p.mask.causal != 0,
                                                          r * kTile + 32 * (warp & 3)));
        }
      }
      if (!mbar_wait(bar.s_full(), u & 1, p.status)) {
        record_failure(p.status, kStatusTimeout, kSiteFwdS);
        ok = false;
        break;
      }
      tc_fence_after();
      // pass 1: the row maximum of this warpgroup's 128 columns
      float pm = -INFINITY;
      const bool partial = (entry & 3) == FM_TILE_PARTIAL;
      const uint32_t s_addr = tmem + lane_base + kColS + 128 * w;
      if (active) {
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t sv[64];
          tmem_ld64(s_addr + 64 * hh, s_addr + 64 * hh + 32, sv);
          if (partial) {
#pragma unroll
            for (int jj = 0; jj < 64; ++jj)
              sv[jj] = ((mbits[2 * hh + (jj >> 5)] >> (jj & 31)) & 1u) ? 0xff800000u : sv[jj];
          }
#pragma unroll
          for (int jj = 0; jj < 64; jj += 4) {
            mx0 = fmaxf(mx0, __uint_as_float(sv[jj]));
            mx1 = fmaxf(mx1, __uint_as_float(sv[jj + 1]));
            mx2 = fmaxf(mx2, __uint_as_float(sv[jj + 2]));
            mx3 = fmaxf(mx3, __uint_as_float(sv[jj + 3]));
          }
        }
        pm = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c;
      }
      // exchange the two partial row maxima (double-buffered by step parity)
      red[((u & 1) * 2 + w) * kTile + row] = pm;
      softmax_bar();
      const float mx = fmaxf(pm, red[((u & 1) * 2 + (w ^ 1)) * kTile + row]);
      const float m_new = fmaxf(m, mx);
      const bool rescale = m_new > m + kRescaleThreshold;
      float alpha = 1.f;
      if (rescale) {
        alpha = ex2(m - m_new);
        m = m_new;
      }
      const float m_use = (m == -INFINITY) ? 0.f : m;
      // pass 2: P in registers (64 columns at a time) while O += P_{u-1} V_{u-1}
      // may still run
      float l0 = 0.f, l1 = 0.f;
      uint32_t pk[64];
      if (active) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t sv[64];
          tmem_ld64(s_addr + 64 * hh, s_addr + 64 * hh + 32, sv);
          if (partial) {
#pragma unroll
            for (int jj = 0; jj < 64; ++jj)
              sv[jj] = ((mbits[2 * hh + (jj >> 5)] >> (jj & 31)) & 1u) ? 0xff800000u : sv[jj];
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float p0 = ex2(fmaf(__uint_as_float(sv[2 * i]), c, -m_use));
            const float p1 = ex2(fmaf(__uint_as_float(sv[2 * i + 1]), c, -m_use));
            l0 += p0;
            l1 += p1;
            pk[32 * hh + i] = pack_bf16x2(p0, p1);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.s_free());  // S may be overwritten by the next step
      l = l * alpha + (l0 + l1);
      if (u >= 1) {
        // the P region and O are free once O += P_{u-1} V_{u-1} has completed
        if (!mbar_wait(bar.o_ready(), (u - 1) & 1, p.status)) {
          record_failure(p.status, kStatusTimeout, kSiteFwdO);
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if (active) {
        tmem_st32p(tmem + lane_base + kColP + 64 * w, &pk[0]);
        tmem_st32p(tmem + lane_base + kColP + 64 * w + 32, &pk[32]);
      }
      if (u >= 1 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int ch = 0; ch < kOCols / 32; ++ch)
          tmem_scale_cols<32>(tmem + lane_base + kColO + w * kOCols + 32 * ch, alpha);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.p_full());
    }
    // ------------------------------------------------------------ epilogue
    if (ok && nsteps > 0) {
      if (!mbar_wait(bar.o_ready(), (nsteps - 1) & 1, p.status)) {
        record_failure(p.status, kStatusTimeout, kSiteFwdO);
        ok = false;
      }
      tc_fence_after();
    }
    // row sums through the exchange buffer of the parity the last step did not
    // use (its previous readers passed the last step's barrier)
    float* lsum = red + (nsteps & 1) * 2 * kTile;
    lsum[w * kTile + row] = l;
    softmax_bar();
    const float ltot = l + lsum[(w ^ 1) * kTile + row];
    const bool live = ok && nsteps > 0;
    const bool has = live && ltot > 0.f;
    const float inv = has ? 1.f / ltot : 0.f;
    uint16_t* orow = p.o + static_cast<size_t>(q_row0 + row) * D + w * kOCols;
#pragma unroll
    for (int ch = 0; ch < kOCols / 32; ++ch)
      tmem_cols_to_bf16<32>(tmem + lane_base + kColO + w * kOCols + 32 * ch, live, inv,
                            orow + 32 * ch);
    if (w == 0) {
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
