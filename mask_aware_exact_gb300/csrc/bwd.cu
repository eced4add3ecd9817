// Backward kernels ("FlashMask: Efficient and Rich Mask Extension of
// FlashAttention", abstract: exact forward and backward that skip masked
// work; the gradient recomputes P from Q, K and the saved LSE as in the
// FlashAttention family):
//
//   bwd_pre     D_i = <dO_i, O_i> (fp32), lse2_i = LSE_i * log2(e) (+inf for a
//               fully masked row, so its P is exactly 0), dQ accumulator = 0
//               (skipped when the forward of the same shape and workspace
//               already zeroed it and left its tag in the status word).
//   bwd_kernel  one CTA per (batch, head, key block of 128 keys), looping over
//               the non-FULL query blocks of that key block:
//                 S^T  = K Q^T              (tcgen05, TMEM)
//                 dP^T = V dO^T             (tcgen05, TMEM)
//                 P^T  = exp2(S^T c - lse2) masked on PARTIAL tiles -> bf16 in TMEM
//                 dV  += P^T dO             (A from TMEM)
//                 dS^T = P^T (dP^T - D)     -> bf16 in shared memory
//                 dK  += dS^T Q             (dS^T K-major)
//                 dQ_t = dS K               -> TMEM -> the tile's own Q/dO stage
//                                              buffers -> TMA bulk reduce-add into
//                                              the fp32 global accumulator
//               (Reductions issued as red.global from the drain warps were
//               measured to slow the compute warps' exponentials and TMEM loads
//               about 2.4x on GB300; the bulk reduce leaves that traffic to the
//               TMA engine. Either way one SM adds at most about 25 bytes per
//               clock into L2, so a tile's 64 KB of dQ takes >= 2600 cycles.)
//   dq_convert  dQ = bf16(scale * accumulator).
//
// Warp roles of bwd_kernel (448 threads): warps 0-7 compute, two warpgroups;
// warpgroup g handles queries [64g, 64g+64) of every tile and thread (g, t)
// owns key t (= TMEM lane t). Warps 8-11 drain dQ_t (thread t = query t),
// warp 12 is the TMA producer, warp 13 the MMA issuer.
//
// TMEM columns (512): S^T / P^T [0,128)  dP^T / dQ_t [128,256)
//                     dV [256, 256+d)    dK [384, 384+d)
// Warpgroup g writes its bf16 P^T half into S^T columns [64g, 64g+32), which
// only it has read, so the two warpgroups never race on TMEM.
#include "internal.h"
#include "ptx.cuh"
#include "flashmask.h"

namespace fm {

namespace {

constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;
constexpr int kThreads = 448;

// TMEM column of the P^T operand for queries [16k, 16k+16) (A of the dV MMA).
__device__ __forceinline__ uint32_t pt_col(int k) { return kColS + 8 * k + (k >= 4 ? 32 : 0); }

template <int D>
struct BwdLayout {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kChunks = D / 64;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kDS = kV + kTileBytes;           // 128 keys x 128 queries bf16
  static constexpr int kQ = kDS + kTile * kTile * 2;    // 2 stages
  static constexpr int kDO = kQ + 2 * kTileBytes;       // 2 stages
  static constexpr int kLse = kDO + 2 * kTileBytes;     // fp32[2][128]
  static constexpr int kDelta = kLse + 2 * kTile * 4;   // fp32[2][128]
  static constexpr int kBar = kDelta + 2 * kTile * 4;
  // kv_full, q_full[2], q_empty[2], s_full, dp_full, pt_ready, ds_ready, dv_done,
  // tile_done, dq_drained, do_full[2], do_empty[2]
  static constexpr int kNumBars = 16;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kBytes = kTmemSlot + 16;
};

struct BwdBars {
  uint32_t base;
  __device__ uint32_t kv_full() const { return base; }
  __device__ uint32_t q_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t q_empty(int s) const { return base + 8 * (3 + s); }
  __device__ uint32_t s_full() const { return base + 8 * 5; }
  __device__ uint32_t dp_full() const { return base + 8 * 6; }
  __device__ uint32_t pt_ready() const { return base + 8 * 7; }
  __device__ uint32_t ds_ready() const { return base + 8 * 8; }
  __device__ uint32_t dv_done() const { return base + 8 * 9; }
  __device__ uint32_t tile_done() const { return base + 8 * 10; }
  __device__ uint32_t dq_drained() const { return base + 8 * 11; }
  __device__ uint32_t do_full(int s) const { return base + 8 * (12 + s); }
  __device__ uint32_t do_empty(int s) const { return base + 8 * (14 + s); }
};


__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Adds a shared-memory box into global memory through a tensor map (fp32 add).
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t src, int x,
                                                  int y) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::
          "l"(reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(src)
      : "memory");
}
// Prefetch of `bytes` (a multiple of 16) of global memory into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void drain_bar() { asm volatile("bar.sync 2, 128;" ::: "memory"); }
// the 256 compute threads (warps 0-7)
__device__ __forceinline__ void compute_bar() { asm volatile("bar.sync 3, 256;" ::: "memory"); }


// ---------------------------------------------------------------- preprocess
// One padded row (bh, n) per D/8 threads, n < Npad: rows n >= N (the short last
// block) get D = 0 and lse2 = +inf, so that their P is exactly 0. The dQ
// accumulator row is zeroed too, unless the status word holds the tag that
// the forward leaves after zeroing the accumulator of this same workspace
// and problem shape itself.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const uint16_t* __restrict__ o,
                                                      const uint16_t* __restrict__ dout,
                                                      const float* __restrict__ lse,
                                                      float* __restrict__ delta,
                                                      float* __restrict__ lse2,
                                                      float* __restrict__ dq_accum,
                                                      long long rows_pad, int N, int Npad,
                                                      const int32_t* zero_tag_word,
                                                      int32_t zero_tag, int32_t* kv_sync,
                                                      long long nsync) {
  constexpr int kThreadsPerRow = D / 8;  // 8 bf16 (16 bytes) per thread and row
  constexpr int kRows = 4;               // rows per thread, their loads all in flight
  const long long gt = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gt < nsync) kv_sync[gt] = 0;  // split key blocks' arrivals and flags
  const int part = static_cast<int>(gt % kThreadsPerRow);
  const long long prow0 = (gt / kThreadsPerRow / 2) * (2 * kRows) + (gt / kThreadsPerRow) % 2;
  const bool zero_acc = *zero_tag_word != zero_tag;
  // rows prow0 + 2r (r < kRows): a warp's two row groups interleave, so each
  // load instruction reads two whole 2d-byte rows
  uint4 a[kRows], g[kRows];
  float L[kRows];
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const long long prow = prow0 + 2 * r;
    const long long bh = prow / Npad;
    const int n = static_cast<int>(prow - bh * Npad);
    const bool live = prow < rows_pad && n < N;
    const long long row = bh * N + n;  // row of O, dO and LSE
    a[r] = g[r] = make_uint4(0u, 0u, 0u, 0u);
    L[r] = -INFINITY;
    if (live) {
      a[r] = *reinterpret_cast<const uint4*>(o + row * D + part * 8);
      g[r] = *reinterpret_cast<const uint4*>(dout + row * D + part * 8);
      if (part == 0) L[r] = lse[row];
    }
  }
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const long long prow = prow0 + 2 * r;
    float acc = 0.f;
    const uint32_t* ap = reinterpret_cast<const uint32_t*>(&a[r]);
    const uint32_t* gp = reinterpret_cast<const uint32_t*>(&g[r]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(__uint_as_float(ap[i] << 16), __uint_as_float(gp[i] << 16), acc);
      acc = fmaf(__uint_as_float(ap[i] & 0xffff0000u), __uint_as_float(gp[i] & 0xffff0000u), acc);
    }
    if (prow < rows_pad && zero_acc) {
      float4* z = reinterpret_cast<float4*>(dq_accum + prow * D + part * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int off = kThreadsPerRow / 2; off > 0; off >>= 1)
      acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (prow < rows_pad && part == 0) {
      delta[prow] = acc;
      lse2[prow] = (L[r] == -INFINITY) ? INFINITY : L[r] * 1.4426950408889634f;
    }
  }
}

// ---------------------------------------------------------------- main
// kSplit: the grid has the split CTAs described below (p.split_e > 0); the
// instantiation without them keeps the plain one-CTA-per-key-block code.
template <int D, bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
               const __grid_constant__ CUtensorMap mdq, const BwdParams p) {
  using L = BwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Work item: head-major, longest key blocks of each head first, so the CTAs
  // that run together reduce into one head's dQ accumulator, which then stays
  // in L2 (fp32 reductions into L2-resident lines run at about twice the rate
  // of reductions that reach DRAM).
  // Each head has Tc + E (kSplitParts - 1) CTAs: the first E kSplitParts
  // take the E longest key blocks, kSplitParts slots each: a block seen by
  // n query blocks is split into nparts = min(kSplitParts, n / kPartTiles)
  // consecutive parts of its tile list when that is at least two (slots past
  // nparts leave at once); the rest take the other key blocks whole. So a key
  // block that every query block sees (a global prefix) does not keep one SM
  // busy long after the others have finished.
  const int E = kSplit ? p.split_e : 0;
  const int per_head = p.Tc + E * (kSplitParts - 1);
  // head, mask head, rank and part of CTA `idx`
  auto decode = [&](int idx, int& bh_, int& bm_, int& rank_, int& part_, bool& cand_) {
    bh_ = idx / per_head;
    const int slot = idx % per_head;
    const int b_ = bh_ / p.H, h_ = bh_ % p.H;
    bm_ = b_ * p.mask.Hm + h_ / (p.H / p.mask.Hm);
    cand_ = kSplit && slot < E * kSplitParts;
    rank_ = cand_ ? slot / kSplitParts : slot - E * (kSplitParts - 1);
    part_ = cand_ ? slot % kSplitParts : 0;
  };
  int bh, bm, rank, part;
  bool cand;
  decode(blockIdx.x, bh, bm, rank, part, cand);
  const int kb = p.col_order[static_cast<size_t>(bm) * p.Tc + rank];
  const int count = p.col_count[static_cast<size_t>(bm) * p.Tc + kb];
  const int nparts = cand ? min(kSplitParts, max(1, count / kPartTiles)) : 1;
  if (kSplit && part >= nparts) return;  // this block needs fewer parts
  const bool split = kSplit && nparts > 1;
  const int t0 = part * count / nparts;
  const int ntiles = (part + 1) * count / nparts - t0;
  const int32_t* list = p.col_list + (static_cast<size_t>(bm) * p.Tc + kb) * p.Tr + t0;
  // the accumulator is about to receive this backward's sums: a later
  // preprocess must zero it again
  if (blockIdx.x == 0 && tid == 0) p.status[3] = 0;

  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) record_failure(p.status, kStatusLayout, kSiteBwdSmemAlign);
    return;
  }
  const uint32_t sK = smem_u32(smem + L::kK), sV = smem_u32(smem + L::kV),
                 sDS = smem_u32(smem + L::kDS), sQ = smem_u32(smem + L::kQ),
                 sDO = smem_u32(smem + L::kDO);
  const float* lse_s = reinterpret_cast<const float*>(smem + L::kLse);
  const float* delta_s = reinterpret_cast<const float*>(smem + L::kDelta);
  const BwdBars bar{smem_u32(smem + L::kBar)};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);

  // Q and lse2 (which = 0) or dO and D (which = 1) of tile t into stage t % 2;
  // lse2 and D live in the padded [B*H, Npad] workspace arrays
  auto load_tile = [&](int t, int which) {
    const int st = t & 1;
    const int qb = list[t] >> 2;
    const size_t prow = static_cast<size_t>(bh) * p.Npad + qb * kTile;
    const uint32_t fb = which == 0 ? bar.q_full(st) : bar.do_full(st);
    const uint32_t dst = (which == 0 ? sQ : sDO) + st * L::kTileBytes;
    mbar_arrive_expect_tx(fb, L::kTileBytes + kTile * 4);
    for (int ch = 0; ch < L::kChunks; ++ch)
      tma_load_3d(dst + ch * 16384, which == 0 ? &mq : &mdo, ch * 64, qb * kTile, bh, fb);
    bulk_load(smem_u32((which == 0 ? lse_s : delta_s) + st * kTile),
              (which == 0 ? p.lse2 : p.delta) + prow, kTile * 4, fb);
  };
  if (warp == 12 && lane == 0) {
    // The producer sets up the barriers its loads complete and issues K, V
    // and the first two tiles before the block-wide sync, so that the loads
    // overlap the TMEM allocation and the other set-up.
    mbar_init(bar.kv_full(), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar.q_full(s), 1);
      mbar_init(bar.do_full(s), 1);
    }
    fence_barrier_init();
    if (ntiles > 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mv);
      tma_prefetch_desc(&mdo);
      mbar_arrive_expect_tx(bar.kv_full(), 2 * L::kTileBytes);
      for (int ch = 0; ch < L::kChunks; ++ch) {
        tma_load_3d(sK + ch * 16384, &mk, ch * 64, kb * kTile, bh, bar.kv_full());
        tma_load_3d(sV + ch * 16384, &mv, ch * 64, kb * kTile, bh, bar.kv_full());
      }
      for (int t = 0; t < 2 && t < ntiles; ++t) {
        load_tile(t, 0);
        load_tile(t, 1);
      }
    }
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar.q_empty(s), 1);
      mbar_init(bar.do_empty(s), 1);
    }
    mbar_init(bar.s_full(), 1);
    mbar_init(bar.dp_full(), 1);
    mbar_init(bar.pt_ready(), 8);
    mbar_init(bar.ds_ready(), 8);
    mbar_init(bar.dv_done(), 1);
    mbar_init(bar.tile_done(), 1);
    mbar_init(bar.dq_drained(), 4);
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 12) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && ntiles > 0) {
      // K and V of the CTA that will start about one CTA duration from now
      // (CTAs start in index order, one per SM) go to L2 ahead of its own
      // loads, which then do not wait for DRAM
      const int fut = blockIdx.x + p.num_sms;
      if (fut < static_cast<int>(gridDim.x)) {
        int fbh, fbm, frank, fpart;
        bool fcand;
        decode(fut, fbh, fbm, frank, fpart, fcand);
        const int fkb = p.col_order[static_cast<size_t>(fbm) * p.Tc + frank];
        const int rows = min(kTile, p.N - fkb * kTile);
        const size_t off = (static_cast<size_t>(fbh) * p.N + fkb * kTile) * D;
        bulk_prefetch_l2(p.k + off, rows * D * 2);
        bulk_prefetch_l2(p.v + off, rows * D * 2);
      }
      for (int t = 2; t < ntiles; ++t) {
        const int st = t & 1;
        // the Q (then dO) buffer of stage st is free once the dQ boxes staged
        // in it two tiles earlier have been read by the bulk reduce; Q goes
        // first, so that S and P of a tile can start before its dO lands
        if (!mbar_wait(bar.q_empty(st), ((t >> 1) - 1) & 1, p.status)) {
          record_failure(p.status, kStatusTimeout, kSiteBwdQEmpty);
          break;
        }
        load_tile(t, 0);
        if (!mbar_wait(bar.do_empty(st), ((t >> 1) - 1) & 1, p.status)) {
          record_failure(p.status, kStatusTimeout, kSiteBwdQEmpty);
          break;
        }
        load_tile(t, 1);
      }
    }
  } else if (warp == 13) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t id_st = idesc_bf16(128, 128, 0, 0);  // S^T, dP^T
      constexpr uint32_t id_kd = idesc_bf16(128, D, 0, 1);    // dV, dK
      constexpr uint32_t id_dq = idesc_bf16(128, D, 1, 1);    // dQ (M = queries)
      // Shared-memory descriptors are built once: every operand address here
      // keeps the descriptor's 14-bit address field (16-byte units) below
      // 2^14, so the descriptor of base + off is the base's plus off / 16.
      const uint64_t kK = sdesc_sw128(sK, 16, 1024), kV = sdesc_sw128(sV, 16, 1024);
      const uint64_t kQ = sdesc_sw128(sQ, 16, 1024), kDO = sdesc_sw128(sDO, 16, 1024);
      const uint64_t kDS = sdesc_sw128(sDS, 16, 1024);
      const uint64_t mDO = sdesc_sw128(sDO, 16384, 1024), mQ = sdesc_sw128(sQ, 16384, 1024);
      const uint64_t mDS = sdesc_sw128(sDS, 16384, 1024), mK = sdesc_sw128(sK, 16384, 1024);
      auto d16 = [](uint32_t bytes) { return static_cast<uint64_t>(bytes >> 4); };
      bool ok = mbar_wait(bar.kv_full(), 0, p.status);
      if (!ok) record_failure(p.status, kStatusTimeout, kSiteBwdKV);
      for (int t = 0; ok && t < ntiles; ++t) {
        const int st = t & 1;
        const uint64_t stage = d16(st * L::kTileBytes);
        if (!mbar_wait(bar.q_full(st), (t >> 1) & 1, p.status)) {
          record_failure(p.status, kStatusTimeout, kSiteBwdQ);
          break;
        }
        if (t >= 1 && !mbar_wait(bar.dv_done(), (t - 1) & 1, p.status)) {  // P^T_{t-1} consumed
          record_failure(p.status, kStatusTimeout, kSiteBwdDV);
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t off = d16((k >> 2) * 16384 + (k & 3) * 32);
          mma_ss(tmem + kColS, kK + off, kQ + stage + off, id_st, k > 0);
        }
        mma_commit(bar.s_full());
        if (t >= 1 && !mbar_wait(bar.dq_drained(), (t - 1) & 1, p.status)) {  // dQ_{t-1} read out
          record_failure(p.status, kStatusTimeout, kSiteBwdDrained);
          break;
        }
        if (!mbar_wait(bar.do_full(st), (t >> 1) & 1, p.status)) {  // dO_t landed
          record_failure(p.status, kStatusTimeout, kSiteBwdQ);
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t off = d16((k >> 2) * 16384 + (k & 3) * 32);
          mma_ss(tmem + kColDP, kV + off, kDO + stage + off, id_st, k > 0);
        }
        mma_commit(bar.dp_full());
        if (!mbar_wait(bar.pt_ready(), t & 1, p.status)) {
          record_failure(p.status, kStatusTimeout, kSiteBwdPT);
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ts(tmem + kColDV, tmem + pt_col(k), mDO + stage + d16(k * 2048), id_kd,
                 (t > 0 || k > 0));
        mma_commit(bar.dv_done());
        if (!mbar_wait(bar.ds_ready(), t & 1, p.status)) {
          record_failure(p.status, kStatusTimeout, kSiteBwdDS);
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t off = d16((k >> 2) * 16384 + (k & 3) * 32);
          mma_ss(tmem + kColDK, kDS + off, mQ + stage + d16(k * 2048), id_kd, (t > 0 || k > 0));
        }
        // dQ_t = dS K: A = dS^T read MN-major (M = queries), B = K read MN-major
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ss(tmem + kColDP, mDS + d16(k * 2048), mK + d16(k * 2048), id_dq, k > 0);
        mma_commit(bar.tile_done());
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ compute (thread = key)
    const int g = warp >> 2;               // queries [64g, 64g+64) of each tile
    const int j = (warp & 3) * 32 + lane;  // key within the block = TMEM lane
    const int key = kb * kTile + j;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    // keys >= N (the short last block of a sequence) do not exist: their P^T
    // row is forced to 0 and their dK, dV rows are not stored
    const bool key_exists = key < p.N;
    const size_t col = static_cast<size_t>(bm) * p.N + (key_exists ? key : 0);
    const int lts = key_exists ? p.mask.lts[col] : 0, lte = key_exists ? p.mask.lte[col] : 0;
    const int uts = (key_exists && p.mask.uts) ? p.mask.uts[col] : 0;
    const int ute = (key_exists && p.mask.ute) ? p.mask.ute[col] : 0;
    const bool causal = p.mask.causal != 0;
    const float c = p.scale_log2;
    bool ok = true;
    int next_entry = ntiles > 0 ? list[0] : 0;  // read one tile ahead
    for (int t = 0; t < ntiles; ++t) {
      const int st = t & 1;
      const int entry = next_entry;
      if (t + 1 < ntiles) next_entry = list[t + 1];
      const int qb = entry >> 2, lab = entry & 3;
      if (!mbar_wait(bar.q_full(st), (t >> 1) & 1, p.status) ||
          !mbar_wait(bar.s_full(), t & 1, p.status)) {
        record_failure(p.status, kStatusTimeout, kSiteBwdS);
        ok = false;
        break;
      }
      tc_fence_after();
      const float* ls = lse_s + st * kTile + 64 * g;
      uint32_t pk[32];  // P^T half-row as bf16 pairs (the dV operand and the dS input)
      {
        uint32_t v[64];
        const uint32_t a = tmem + lane_base + kColS + 64 * g;
        tmem_ld64(a, a + 32, v);
        // masked-query bits of this thread's key column for queries 64g + [32h, 32h+32)
        uint32_t mb[2] = {0u, 0u};
        if (!key_exists) {
          mb[0] = mb[1] = 0xffffffffu;
        } else if (lab == FM_TILE_PARTIAL) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
            mb[hh] = column_mask_bits(key, lts, lte, uts, ute, causal,
                                      qb * kTile + 64 * g + 32 * hh);
        }
        const uint64_t c2 = f2_make(c, c);
#pragma unroll
        for (int i4 = 0; i4 < 16; ++i4) {
          const float4 l4 = reinterpret_cast<const float4*>(ls)[i4];  // broadcast
          const uint64_t nl2[2] = {f2_make(-l4.x, -l4.y), f2_make(-l4.z, -l4.w)};
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int q0 = 4 * i4 + 2 * u;
            // s * c - lse2 for a pair of queries in one paired fp32 instruction
            float x0, x1;
            f2_split(f2_fma(f2_make(__uint_as_float(v[q0]), __uint_as_float(v[q0 + 1])), c2,
                            nl2[u]),
                     x0, x1);
            float p0 = ex2(x0), p1 = ex2(x1);
            p0 = ((mb[q0 >> 5] >> (q0 & 31)) & 1u) ? 0.f : p0;
            p1 = ((mb[q0 >> 5] >> ((q0 + 1) & 31)) & 1u) ? 0.f : p1;
            pk[2 * i4 + u] = pack_bf16x2(p0, p1);
          }
        }
      }
      tmem_st32p(tmem + lane_base + kColS + 64 * g, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.pt_ready());

      if (!mbar_wait(bar.dp_full(), t & 1, p.status)) {
        record_failure(p.status, kStatusTimeout, kSiteBwdDP);
        ok = false;
        break;
      }
      if (t >= 1 && !mbar_wait(bar.tile_done(), (t - 1) & 1, p.status)) {  // dS_{t-1} consumed
        record_failure(p.status, kStatusTimeout, kSiteBwdDone);
        ok = false;
        break;
      }
      if (!mbar_wait(bar.do_full(st), (t >> 1) & 1, p.status)) {  // D of this tile landed
        record_failure(p.status, kStatusTimeout, kSiteBwdDP);
        ok = false;
        break;
      }
      tc_fence_after();
      const float* dl = delta_s + st * kTile + 64 * g;
      // row j of dS^T, queries [64g, 64g+64): the 128-byte row of chunk g, in
      // two 32-query halves
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kColDP + 64 * g + 32 * hh, v);
        uint32_t dk[16];
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const float4 d4 = reinterpret_cast<const float4*>(dl + 32 * hh)[i4];  // broadcast
          const uint64_t nd2[2] = {f2_make(-d4.x, -d4.y), f2_make(-d4.z, -d4.w)};
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int i = 2 * i4 + u;
            const uint32_t pw = pk[16 * hh + i];
            // P (dP - D) for a pair of queries in two paired fp32 instructions
            const uint64_t dd = f2_add(f2_make(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                                       nd2[u]);
            float d0, d1;
            f2_split(f2_mul(f2_make(__uint_as_float(pw << 16), __uint_as_float(pw & 0xffff0000u)), dd),
                     d0, d1);
            dk[i] = pack_bf16x2(d0, d1);
          }
        }
        const uint32_t base = sDS + g * 16384;
#pragma unroll
        for (int pc = 0; pc < 4; ++pc)
          st_shared_v4(base + sw128_offset(j, 4 * hh + pc), dk[4 * pc], dk[4 * pc + 1],
                       dk[4 * pc + 2], dk[4 * pc + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.ds_ready());
    }
    // ------------------------------------------------------------ epilogue: dV, dK
    if (ok && ntiles > 0) {
      if (!mbar_wait(bar.tile_done(), (ntiles - 1) & 1, p.status)) {
        record_failure(p.status, kStatusTimeout, kSiteBwdDone);
        ok = false;
      }
      tc_fence_after();
    }
    const bool live = ok && ntiles > 0;
    // a split key block: each part but the last to finish leaves its fp32
    // dV, dK in the workspace slot of its arrival order; the last adds them
    // to its own and writes the block
    int add_parts = 0;
    bool write_out = true;
    float* part_base = nullptr;
    if (split) {
      int32_t* sync = p.kv_sync + (static_cast<size_t>(bh) * E + rank) * kSyncWords;
      part_base = p.kv_part + (static_cast<size_t>(bh) * E + rank) * (kSplitParts - 1) * 2 * kTile * D;
      volatile int* arrival_s = reinterpret_cast<volatile int*>(tmem_slot + 1);
      if (tid == 0) *arrival_s = atomicAdd(sync, 1);
      compute_bar();
      const int arrival = *arrival_s;
      if (arrival < nparts - 1) {
        float* part = part_base + static_cast<size_t>(arrival) * 2 * kTile * D;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const uint32_t colbase = (which == 0 ? kColDV : kColDK) + g * (D / 2);
#pragma unroll
          for (int ch = 0; ch < D / 64; ++ch) {
            uint32_t v[32];
            if (live) {
              tmem_ld32(tmem + lane_base + colbase + ch * 32, v);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = 0u;
            }
            float4* dst = reinterpret_cast<float4*>(part + (which * kTile + j) * D + g * (D / 2) +
                                                    ch * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                   __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
          }
        }
        __threadfence();
        compute_bar();
        if (tid == 0) atomicExch(sync + 1 + arrival, 1);  // this partial is complete
        write_out = false;
      } else {
        // the other parts' partials: each has been counted, so it is being
        // written by a CTA that waits for nothing; the waits are bounded all
        // the same
        if (tid == 0) {
          const uint64_t w0 = global_timer_ns();
          for (int i = 0; i < nparts - 1; ++i) {
            while (*reinterpret_cast<volatile int32_t*>(sync + 1 + i) == 0) {
              if (global_timer_ns() - w0 > FM_WAIT_LIMIT_NS) {
                record_failure(p.status, kStatusTimeout, kSiteBwdSplit);
                break;
              }
            }
          }
        }
        compute_bar();
        __threadfence();
        add_parts = nparts - 1;
      }
    }
    // dV, then dK (scaled), as bf16 through the dS^T buffer (free once the
    // last tile's products have completed): thread (g, j) writes row j,
    // columns [g D/2, g D/2 + D/2), into the buffer (128-byte swizzled rows:
    // half g for d = 128, 16-byte units [4g, 4g + 4) of a single half for
    // d = 64); then the 256 threads copy the tile out in 16-byte pieces, a
    // warp covering whole consecutive rows, so that every store is
    // coalesced. Keys >= N of a short last key block are not written.
    constexpr int kRowPieces = D / 8;  // 16-byte pieces per row
    for (int which = 0; which < 2 && write_out; ++which) {
      const uint32_t colbase = (which == 0 ? kColDV : kColDK) + g * (D / 2);
      const float f = which == 0 ? 1.f : p.scale;
      if (which == 1) compute_bar();  // the dV tile has been copied out
#pragma unroll
      for (int ch = 0; ch < D / 64; ++ch) {
        uint32_t v[32];
        if (live) {
          tmem_ld32(tmem + lane_base + colbase + ch * 32, v);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        for (int q = 0; q < add_parts; ++q) {
          const float4* src = reinterpret_cast<const float4*>(
              part_base + static_cast<size_t>(q) * 2 * kTile * D + (which * kTile + j) * D +
              g * (D / 2) + ch * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 a = __ldcg(src + i);
            v[4 * i] = __float_as_uint(__uint_as_float(v[4 * i]) + a.x);
            v[4 * i + 1] = __float_as_uint(__uint_as_float(v[4 * i + 1]) + a.y);
            v[4 * i + 2] = __float_as_uint(__uint_as_float(v[4 * i + 2]) + a.z);
            v[4 * i + 3] = __float_as_uint(__uint_as_float(v[4 * i + 3]) + a.w);
          }
        }
        uint32_t w16[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w16[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * f, __uint_as_float(v[2 * i + 1]) * f);
        const uint32_t half = D == 128 ? sDS + g * 16384 : sDS;
        const int unit0 = D == 128 ? 4 * ch : 4 * g;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          st_shared_v4(half + sw128_offset(j, unit0 + u), w16[4 * u], w16[4 * u + 1],
                       w16[4 * u + 2], w16[4 * u + 3]);
      }
      compute_bar();
      uint16_t* out = (which == 0 ? p.dv : p.dk) + (static_cast<size_t>(bh) * p.N + kb * kTile) * D;
#pragma unroll
      for (int i = 0; i < kTile * kRowPieces / 256; ++i) {
        const int c = tid + 256 * i;  // piece c: row c / kRowPieces, piece c % kRowPieces
        const int row = c / kRowPieces, pc = c % kRowPieces;
        const uint32_t src = D == 128 ? sDS + (pc >> 3) * 16384 + sw128_offset(row, pc & 7)
                                      : sDS + sw128_offset(row, pc);
        uint32_t a0, a1, a2, a3;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                     : "r"(src)
                     : "memory");
        if (kb * kTile + row < p.N)
          *reinterpret_cast<uint4*>(out + static_cast<size_t>(row) * D + pc * 8) =
              make_uint4(a0, a1, a2, a3);
      }
    }
  } else {
    // ------------------------------------------------------------ dQ drain
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int ln = tid - 256;  // TMEM lane this thread reads
    int next_qb = ntiles > 0 ? (list[0] >> 2) : 0;  // read one tile ahead
    // lane = query: dQ_t (fp32, 128 queries x d) goes to the stage buffers of
    // tile t in 32-column boxes of 128 rows x 128 bytes, 128-byte swizzled,
    // then one thread adds the boxes into the accumulator with TMA
    const bool leader = tid == 256;
    for (int t = 0; t < ntiles; ++t) {
      const int st = t & 1;
      const int qb = next_qb;
      if (t + 1 < ntiles) next_qb = list[t + 1] >> 2;
      if (!mbar_wait(bar.tile_done(), t & 1, p.status)) {
        record_failure(p.status, kStatusTimeout, kSiteBwdDQ);
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kColDP + ch * 32, v);
        const uint32_t box = (ch * 16384 < L::kTileBytes)
                                 ? sQ + st * L::kTileBytes + ch * 16384
                                 : sDO + st * L::kTileBytes + ch * 16384 - L::kTileBytes;
#pragma unroll
        for (int c16 = 0; c16 < 8; ++c16)
          st_shared_v4(box + sw128_offset(ln, c16), v[4 * c16], v[4 * c16 + 1], v[4 * c16 + 2],
                       v[4 * c16 + 3]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.dq_drained());
      fence_proxy_async_smem();
      drain_bar();
      if (leader) {
        // the boxes staged in the Q buffer form one bulk group and those in
        // the dO buffer a second, so that the Q buffer returns to the
        // producer as soon as the first group has been read
        constexpr int kQBoxes = L::kTileBytes / 16384;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          const uint32_t box = (ch < kQBoxes)
                                   ? sQ + st * L::kTileBytes + ch * 16384
                                   : sDO + st * L::kTileBytes + (ch - kQBoxes) * 16384;
          tma_reduce_add_2d(&mdq, box, ch * 32, bh * p.Npad + qb * kTile);
          if (ch == kQBoxes - 1) bulk_commit_group();
        }
        bulk_commit_group();
        bulk_wait_read_1();  // the Q-buffer group has been read
        if (t + 2 < ntiles) mbar_arrive(bar.q_empty(st));
        bulk_wait_read_all();
        if (t + 2 < ntiles) mbar_arrive(bar.do_empty(st));
      }
    }
    // the last reductions must have read their boxes before the CTA's
    // shared memory goes; their adds complete before the kernel does
    if (leader) bulk_wait_read_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// dQ = bf16(scale * accumulator); 8 elements per thread of the unpadded
// [heads, N, d] output, read from the padded [heads, Npad, d] accumulator.
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc, float scale,
                                                         uint16_t* __restrict__ dq, long long n8,
                                                         int N, int Npad, int d) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const long long e = i * 8;
  const long long row = e / d;  // (bh, n) with n < N
  const long long bh = row / N;
  const long long src = (bh * Npad + (row - bh * N)) * d + (e - row * d);
  const float4 a = *reinterpret_cast<const float4*>(acc + src);
  const float4 b = *reinterpret_cast<const float4*>(acc + src + 4);
  uint4 o;
  o.x = pack_bf16x2(a.x * scale, a.y * scale);
  o.y = pack_bf16x2(a.z * scale, a.w * scale);
  o.z = pack_bf16x2(b.x * scale, b.y * scale);
  o.w = pack_bf16x2(b.z * scale, b.w * scale);
  reinterpret_cast<uint4*>(dq)[i] = o;
}

template <int D, bool kSplit>
cudaError_t launch_bwd_t(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const CUtensorMap& mdo, const CUtensorMap& mdq, const BwdParams& p,
                         cudaStream_t s) {
  using L = BwdLayout<D>;
  cudaError_t e = cudaFuncSetAttribute(bwd_kernel<D, kSplit>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  const int per_head = p.Tc + (kSplit ? p.split_e * (kSplitParts - 1) : 0);
  const unsigned grid = static_cast<unsigned>(p.B * p.H * per_head);
  bwd_kernel<D, kSplit><<<grid, kThreads, L::kBytes, s>>>(mq, mk, mv, mdo, mdq, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_pre(int d, const uint16_t* o, const uint16_t* dout, const float* lse,
                           float* delta, float* lse2, float* dq_accum, long long heads, int N,
                           int Npad, const int32_t* zero_tag_word, int32_t zero_tag,
                           int32_t* kv_sync, int split_e, cudaStream_t s) {
  const long long rows_pad = heads * Npad;
  const long long threads = rows_pad * (d / 8) / 4;  // four rows per thread
  const unsigned grid = static_cast<unsigned>((threads + 255) / 256);
  const long long nsync = heads * split_e * kSyncWords;
  if (d == 64)
    bwd_pre_kernel<64><<<grid, 256, 0, s>>>(o, dout, lse, delta, lse2, dq_accum, rows_pad, N, Npad,
                                            zero_tag_word, zero_tag, kv_sync, nsync);
  else
    bwd_pre_kernel<128><<<grid, 256, 0, s>>>(o, dout, lse, delta, lse2, dq_accum, rows_pad, N,
                                             Npad, zero_tag_word, zero_tag, kv_sync, nsync);
  return cudaGetLastError();
}

cudaError_t launch_bwd(int d, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       const CUtensorMap& mdo, const CUtensorMap& mdq, const BwdParams& p,
                       cudaStream_t s) {
  const bool split = p.split_e > 0;
  if (d == 64)
    return split ? launch_bwd_t<64, true>(mq, mk, mv, mdo, mdq, p, s)
                 : launch_bwd_t<64, false>(mq, mk, mv, mdo, mdq, p, s);
  return split ? launch_bwd_t<128, true>(mq, mk, mv, mdo, mdq, p, s)
               : launch_bwd_t<128, false>(mq, mk, mv, mdo, mdq, p, s);
}

cudaError_t launch_dq_convert(int d, const float* dq_accum, float scale, uint16_t* dq,
                              long long heads, int N, int Npad, cudaStream_t s) {
  const long long n8 = heads * N * d / 8;
  const unsigned grid = static_cast<unsigned>((n8 + 255) / 256);
  dq_convert_kernel<<<grid, 256, 0, s>>>(dq_accum, scale, dq, n8, N, Npad, d);
  return cudaGetLastError();
}

}  // namespace fm
