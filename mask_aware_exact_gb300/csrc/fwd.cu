// Forward kernel: exact attention over the non-FULL tiles of a pair of 128-row
// query blocks ("FlashMask: Efficient and Rich Mask Extension of
// FlashAttention", abstract: skip masked computation, exact result;
// "FlashAttention-3", abstract: warp specialisation overlapping TMA data
// movement with tensor-core work, and block-wise matmul interleaved with
// softmax).
//
// A work item is one head's pair of adjacent query blocks (r0, r1) = (2p,
// 2p + 1). Both tiles walk the merged list of key blocks that are non-FULL for
// either of them; each K and V block is loaded once and serves both. Each tile
// t has one chain through the tensor cores and TMEM,
//
//     S_t = Q_t K_j^T -> softmax_t (P_t over S_t) -> O_t += P_t V_j -> S_t of the next block,
//
// and one softmax warpgroup. A single thread issues both tiles' products in the
// order S_0(j), O_1 += P_1 V (tile 1's previous step), S_1(j), O_0 += P_0 V
// (step j), so that while one tile's softmax works the tensor pipe holds the
// other tile's products and the two softmax warpgroups take turns. P stays in
// TMEM (the A operand of P V), which keeps the shared-memory traffic of a step
// to the Q K^T operands and V: with both operands of an M = N = 128 product in
// shared memory the tensor cores' shared-memory reads (about 128 bytes per
// clock) are already the limit. A tile skips the key blocks that are FULL for
// it.
//
// Persistent CTAs (one per SM) take items from a work counter in the
// workspace, head-major (a head's K and V stay in L2 while its pairs run) and
// longest pair first within a head. Warp roles (384 threads):
//   warps 0-3   softmax of tile 0: thread = query row = TMEM lane, the whole
//               128-key row of S in registers: element mask on PARTIAL tiles,
//               row maximum, exponentials (log2 domain), row sum, P as bf16 (or
//               e4m3) over S_t. O_t is rescaled only when the maximum grows by
//               more than 2^8 (lazy rescaling, exact after the final division).
//               Epilogue: O_t / l, LSE.
//   warps 4-7   softmax of tile 1.
//   warp 8      work scheduler; TMA producer of Q_0, Q_1 (once per item) and
//               of the K ring.
//   warp 9      MMA issuer of both tiles (one thread).
//   warp 10     TMA producer of the V ring.
//   warp 11     idle (completes the register-split warpgroup).
//
// TMEM columns (512): S_0/P_0 [0,128), S_1/P_1 [128,256), O_0 [256,256+d),
// O_1 [384,384+d). S_t of the next block is issued only after O_t += P_t V
// has completed (the product reads P_t from S_t's columns), so by the time the
// softmax sees S_t complete, O_t is quiescent and may be rescaled in place.
#include "internal.h"
#include "ptx.cuh"
#include "ptx_fp8.cuh"
#include "flashmask.h"

namespace fm {

namespace {

constexpr int kThreads = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// FP8: P is stored as e4m3(p * kFp8PScale). With the running maximum lagging
// by at most kRescaleThresholdFp8 (log2 units), p < 2^threshold and
// p * kFp8PScale stays below 448, the largest finite e4m3 value.
constexpr float kRescaleThresholdFp8 = 4.0f;
constexpr float kFp8PScale = 28.0f;
// Roles that read each published work item: the MMA warp, the V producer and
// the first warp of each softmax warpgroup (which shares it with the other
// three through shared memory).
constexpr int kSchedReaders = 4;
// Per-thread register limits after the split (setmaxnreg): softmax warpgroups,
// producer / MMA warpgroup. Their sum over the 384 threads must not exceed the
// pool the CTA is launched with (threads x registers of the compiled kernel).
constexpr int kRegsSoftmax = 208, kRegsOther = 88;
constexpr int kRegPool = 256 * kRegsSoftmax + 128 * kRegsOther;

__device__ __forceinline__ uint32_t col_s(int t) { return 128u * static_cast<uint32_t>(t); }
__device__ __forceinline__ uint32_t col_o(int t) { return 256u + 128u * static_cast<uint32_t>(t); }

template <int D, bool kFp8>
struct FwdLayout {
  static constexpr int kTileBytes = kTile * D * (kFp8 ? 1 : 2);  // one 128 x d tile
  static constexpr int kChunks = kFp8 ? 1 : D / 64;  // 128-byte-wide TMA boxes per tile
  static constexpr int kChunk = 16384;              // 128 rows x 128 bytes
  static constexpr int kKSlots = kTileBytes >= 32768 ? 3 : 4;
  static constexpr int kVSlots = kTileBytes >= 32768 ? 2 : 4;
  static constexpr int kQ = 0;                            // Q_0, Q_1
  static constexpr int kK = kQ + 2 * kTileBytes;          // kKSlots x kTileBytes
  static constexpr int kV = kK + kKSlots * kTileBytes;    // kVSlots x kTileBytes
  static constexpr int kBar = kV + kVSlots * kTileBytes;
  static constexpr int kNumBars = 4 + 2 * kKSlots + 2 * kVSlots + 12;
  static constexpr int kSched = kBar + kNumBars * 8;  // int[6]: ring[2], share[2][2]
  static constexpr int kTmemSlot = kSched + 32;
  static constexpr int kBytes = kTmemSlot + 16;
};

// q_full[2] q_empty[2] k_full[KS] k_empty[KS] v_full[VS] v_empty[VS] s_full[2]
// p_full[2] pv_done[2] o_free[2] sched_full[2] sched_empty[2]
template <int KS, int VS>
struct FwdBars {
  uint32_t b;
  static constexpr int kT = 4 + 2 * KS + 2 * VS;
  __device__ uint32_t q_full(int t) const { return b + 8 * t; }
  __device__ uint32_t q_empty(int t) const { return b + 8 * (2 + t); }
  __device__ uint32_t k_full(int s) const { return b + 8 * (4 + s); }
  __device__ uint32_t k_empty(int s) const { return b + 8 * (4 + KS + s); }
  __device__ uint32_t v_full(int s) const { return b + 8 * (4 + 2 * KS + s); }
  __device__ uint32_t v_empty(int s) const { return b + 8 * (4 + 2 * KS + VS + s); }
  __device__ uint32_t s_full(int t) const { return b + 8 * (kT + t); }
  __device__ uint32_t p_full(int t) const { return b + 8 * (kT + 2 + t); }
  __device__ uint32_t pv_done(int t) const { return b + 8 * (kT + 4 + t); }
  __device__ uint32_t o_free(int t) const { return b + 8 * (kT + 6 + t); }
  __device__ uint32_t sched_full(int s) const { return b + 8 * (kT + 8 + s); }
  __device__ uint32_t sched_empty(int s) const { return b + 8 * (kT + 10 + s); }
};

// The 128 threads of softmax warpgroup t.
__device__ __forceinline__ void group_bar(int t) {
  asm volatile("bar.sync %0, 128;" ::"r"(1 + t) : "memory");
}

// Multiplies 32 consecutive TMEM columns of this warp's lanes by f.
__device__ __forceinline__ void tmem_scale32(uint32_t taddr, float f) {
  uint32_t v[32];
  tmem_ld32(taddr, v);
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
  tmem_st32(taddr, v);
}

// Writes 32 TMEM columns of this lane's row, times f, as bf16 (the TMEM load
// runs on every lane of the warp; only lanes with `store` write).
__device__ __forceinline__ void tmem_cols_to_bf16(uint32_t taddr, bool live, float f,
                                                  uint16_t* dst, bool store) {
  uint32_t v[32];
  if (live) {
    tmem_ld32(taddr, v);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0u;
  }
  if (!store) return;  // after the (warp-collective) TMEM load
  store_row32_bf16(dst, v, f);
}

// kShortLast: N is not a multiple of 128. kFp8 (d = 128 only): e4m3 Q, K and
// transposed V with block scales, kind::f8f6f4 MMAs (K = 32 per instruction),
// P stored as e4m3(p * kFp8PScale).
template <int D, bool kShortLast, bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv, const FwdParams p) {
  using L = FwdLayout<D, kFp8>;
  constexpr int KS = L::kKSlots, VS = L::kVSlots;
  static_assert(!kFp8 || D == 128, "the FP8 forward is for d = 128");
  static_assert(L::kBytes <= 232448, "shared memory");
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = p.B * p.H * p.Tp;

  if ((smem_u32(smem) & 1023u) != 0) {  // 128-byte swizzle atoms need 1024-byte alignment
    if (tid == 0) record_failure(p.status, kStatusLayout, kSiteFwdSmemAlign);
    return;
  }
  const uint32_t sQ = smem_u32(smem + L::kQ), sK = smem_u32(smem + L::kK),
                 sV = smem_u32(smem + L::kV);
  // [0, 2): the item ring; [2 + 2t, 4 + 2t): the item as warpgroup t shares it
  volatile int* sched = reinterpret_cast<volatile int*>(smem + L::kSched);
  const FwdBars<KS, VS> bar{smem_u32(smem + L::kBar)};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);

  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar.q_full(t), 1);
      mbar_init(bar.q_empty(t), 1);
      mbar_init(bar.s_full(t), 1);
      mbar_init(bar.p_full(t), 4);
      mbar_init(bar.pv_done(t), 1);
      mbar_init(bar.o_free(t), 4);
      mbar_init(bar.sched_full(t), 1);
      mbar_init(bar.sched_empty(t), kSchedReaders);
    }
    for (int s = 0; s < KS; ++s) {
      mbar_init(bar.k_full(s), 1);
      mbar_init(bar.k_empty(s), 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(bar.v_full(s), 1);
      mbar_init(bar.v_empty(s), 1);
    }
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Work item n: head-major, longest pairs of each head first.
  struct Item {
    int bh, bm, r0, r1, count;
    const int32_t* list;
  };
  auto decode = [&](int n) -> Item {
    Item it;
    it.bh = n / p.Tp;
    const int rank = n % p.Tp;
    const int b = it.bh / p.H, h = it.bh % p.H;
    it.bm = b * p.mask.Hm + h / (p.H / p.mask.Hm);
    const size_t base = static_cast<size_t>(it.bm) * p.Tp;
    const int pair = p.pair_order[base + rank];
    it.count = p.pair_count[base + pair];
    it.list = p.pair_list + (base + pair) * p.Tc;
    it.r0 = 2 * pair;
    it.r1 = 2 * pair + 1;  // may be Tr: a missing block whose entries are all FULL
    return it;
  };
  // Label of tile t in a merged-list entry (FM_TILE_FULL: not visited).
  auto label = [](int entry, int t) -> int { return t == 0 ? (entry >> 2) & 3 : entry & 3; };
  // The k-th item of this CTA (k = 0, 1, ...) from the ring, or -1 when no
  // item is left or the wait gave up (then `ok` is false).
  auto read_item = [&](int k, bool& ok) -> int {
    const int s = k & 1;
    if (!mbar_wait(bar.sched_full(s), (k >> 1) & 1, p.status)) {
      record_failure(p.status, kStatusTimeout, kSiteFwdSched);
      ok = false;
      return -1;
    }
    const int n = sched[s];
    mbar_arrive(bar.sched_empty(s));
    return n;
  };

  // Registers: the two softmax warpgroups hold a 128-key row of S each; the
  // producer / MMA warpgroup (warps 8-11) needs few. Each warpgroup changes its
  // own limit at the top of its branch. The split fits the launch's pool of
  // 384 x 168: 256 x 208 + 128 x 88 = 64512 (the host checks the kernel's
  // register count before launching).
  if (warp >= 8) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther) : "memory");
  if (warp == 8) {
    // ------------------------------------------------------------ scheduler, TMA producer of Q, K
    if (lane == 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      auto claim = [&]() -> int {
        const int n = atomicAdd(p.sched, 1);
        return n < n_items ? n : -1;
      };
      int cur = claim();
      sched[0] = cur;
      mbar_arrive(bar.sched_full(0));
      bool ok = true;
      int J = 0;  // running step over the merged lists of this CTA's items
      for (int k = 0; ok && cur >= 0; ++k) {
        const Item it = decode(cur);
        // Q_t of the item once the previous item's S_t products have completed;
        // a missing second block reloads the first (its products are never issued)
        for (int t = 0; t < 2 && ok; ++t) {
          if (k >= 1 && !mbar_wait(bar.q_empty(t), (k - 1) & 1, p.status)) {
            record_failure(p.status, kStatusTimeout, kSiteFwdKEmpty);
            ok = false;
            break;
          }
          const int qb = (t == 1 && it.r1 < p.Tr) ? it.r1 : it.r0;
          mbar_arrive_expect_tx(bar.q_full(t), L::kTileBytes);
          for (int ch = 0; ch < L::kChunks; ++ch)
            tma_load_3d(sQ + t * L::kTileBytes + ch * L::kChunk, &mq, ch * 64, qb * kTile, it.bh,
                        bar.q_full(t));
        }
        for (int j = 0; ok && j < it.count; ++j, ++J) {
          const int slot = J % KS;
          if (J >= KS && !mbar_wait(bar.k_empty(slot), ((J / KS) - 1) & 1, p.status)) {
            record_failure(p.status, kStatusTimeout, kSiteFwdKEmpty);
            ok = false;
            break;
          }
          const int kb = it.list[j] >> 4;
          mbar_arrive_expect_tx(bar.k_full(slot), L::kTileBytes);
          for (int ch = 0; ch < L::kChunks; ++ch)
            tma_load_3d(sK + slot * L::kTileBytes + ch * L::kChunk, &mk, ch * 64, kb * kTile,
                        it.bh, bar.k_full(slot));
        }
        if (!ok) break;
        // claim the next item once this one's loads are issued; its ring
        // entry was last used by item k - 1, which every reader has taken
        const int nxt = claim();
        const int s = (k + 1) & 1;
        if (k >= 1 && !mbar_wait(bar.sched_empty(s), ((k - 1) >> 1) & 1, p.status)) {
          record_failure(p.status, kStatusTimeout, kSiteFwdSched);
          break;
        }
        sched[s] = nxt;
        mbar_arrive(bar.sched_full(s));
        cur = nxt;
      }
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ TMA producer of V
    if (lane == 0) {
      tma_prefetch_desc(&mv);
      bool ok = true;
      int J = 0;
      for (int k = 0; ok; ++k) {
        const int n = read_item(k, ok);
        if (n < 0) break;
        const Item it = decode(n);
        for (int j = 0; ok && j < it.count; ++j, ++J) {
          const int slot = J % VS;
          if (J >= VS && !mbar_wait(bar.v_empty(slot), ((J / VS) - 1) & 1, p.status)) {
            record_failure(p.status, kStatusTimeout, kSiteFwdVEmpty);
            ok = false;
            break;
          }
          const int kb = it.list[j] >> 4;
          mbar_arrive_expect_tx(bar.v_full(slot), L::kTileBytes);
          if constexpr (kFp8) {
            // V^T tile: the head's 128 rows of d, the block's 128 keys
            tma_load_2d(sV + slot * L::kTileBytes, &mv, kb * kTile, it.bh * 128, bar.v_full(slot));
          } else {
            for (int ch = 0; ch < L::kChunks; ++ch)
              tma_load_3d(sV + slot * L::kTileBytes + ch * L::kChunk, &mv, ch * 64, kb * kTile,
                          it.bh, bar.v_full(slot));
          }
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer (both tiles)
    // One thread issues every product in the order, per step j of the merged
    // list, S_0(j), O_1 += P_1 V (previous step of tile 1), S_1(j),
    // O_0 += P_0 V (step j): while one tile's softmax runs, the tensor pipe
    // holds the other tile's products, so the two softmax warpgroups
    // alternate. S_t(j) overwrites the TMEM columns the previous P_t V read, so
    // it waits for that product to complete.
    if (lane == 0) {
      constexpr uint32_t idesc_s = kFp8 ? idesc_e4m3(128, 128) : idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idesc_pv = kFp8 ? idesc_e4m3(128, D) : idesc_bf16(128, D, 0, 1);
      constexpr int kSSteps = kFp8 ? D / 32 : D / 16;  // K steps of S = Q K^T
      constexpr int kPvSteps = kFp8 ? 4 : 8;           // K steps (keys) of O += P V
      // Shared-memory descriptors are built once: the address field (bits
      // 0-13, in 16-byte units) of every operand stays below 2^14 here, so a
      // descriptor for base + off is the base descriptor plus off / 16.
      const uint64_t dq0 = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dq1 = sdesc_sw128(sQ + L::kTileBytes, 16, 1024);
      const uint64_t dk_base = sdesc_sw128(sK, 16, 1024);
      // V is MN-major [keys][d] in bf16, K-major [d][keys] as e4m3 V^T
      const uint64_t dv_base = kFp8 ? sdesc_sw128(sV, 16, 1024) : sdesc_sw128(sV, 16384, 1024);
      bool ok = true;
      int J0 = 0;                // running step of the item's first entry
      int nv[2] = {0, 0};        // P V products per tile so far
      // S_t of step J into TMEM (K of step J has landed); the previous P_t V
      // must have completed
      auto issue_s = [&](int t, int J) -> bool {
        if (nv[t] > 0 && !mbar_wait(bar.pv_done(t), (nv[t] - 1) & 1, p.status)) return false;
        tc_fence_after();
        const uint64_t dq = t == 0 ? dq0 : dq1;
        const uint64_t kd = dk_base + static_cast<uint64_t>(((J % KS) * L::kTileBytes) >> 4);
        const uint32_t ts = tmem + col_s(t);
#pragma unroll
        for (int kk = 0; kk < kSSteps; ++kk) {
          // 32 bytes of each 128-byte row per K step (16 bf16 or 32 e4m3)
          const uint64_t off16 = static_cast<uint64_t>(((kk >> 2) * L::kChunk + (kk & 3) * 32) >> 4);
          if constexpr (kFp8)
            mma_ss_f8(ts, dq + off16, kd + off16, idesc_s, kk > 0);
          else
            mma_ss(ts, dq + off16, kd + off16, idesc_s, kk > 0);
        }
        mma_commit(bar.s_full(t));
        return true;
      };
      // O_t += P_t V of step J once P_t is in TMEM and V has landed; the item's
      // first product overwrites O_t after the previous item's O_t was read out
      auto issue_pv = [&](int t, int J, bool first, int k) -> bool {
        const int vs = J % VS;
        if (!mbar_wait(bar.p_full(t), nv[t] & 1, p.status) ||
            !mbar_wait(bar.v_full(vs), (J / VS) & 1, p.status) ||
            (first && k > 0 && !mbar_wait(bar.o_free(t), (k - 1) & 1, p.status)))
          return false;
        tc_fence_after();
        const uint64_t vd = dv_base + static_cast<uint64_t>((vs * L::kTileBytes) >> 4);
        const uint32_t ts = tmem + col_s(t), to = tmem + col_o(t);
#pragma unroll
        for (int kk = 0; kk < kPvSteps; ++kk) {
          // A: P, 8 TMEM columns per K step; B: the next 16 key rows of V
          // (bf16) or the next 32 key bytes of each row of V^T (e4m3)
          if constexpr (kFp8)
            mma_ts_f8(to, ts + 8 * kk, vd + static_cast<uint64_t>((kk * 32) >> 4), idesc_pv,
                      (!first || kk > 0));
          else
            mma_ts(to, ts + 8 * kk, vd + static_cast<uint64_t>((kk * 2048) >> 4), idesc_pv,
                   (!first || kk > 0));
        }
        mma_commit(bar.pv_done(t));
        ++nv[t];
        return true;
      };
      for (int k = 0; ok; ++k) {
        const int n = read_item(k, ok);
        if (n < 0) break;
        const Item it = decode(n);
        if (!mbar_wait(bar.q_full(0), k & 1, p.status) ||
            !mbar_wait(bar.q_full(1), k & 1, p.status)) {
          ok = false;
          break;
        }
        // the last step each tile visits: Q_t is free for the next item once
        // that step's S_t has completed (usually found at once: the list's
        // last entry, or the one before it)
        int last[2];
        for (int t = 0; t < 2; ++t) {
          last[t] = it.count - 1;
          while (last[t] >= 0 && label(it.list[last[t]], t) == FM_TILE_FULL) --last[t];
          if (last[t] < 0) mma_commit(bar.q_empty(t));
        }
        bool first[2] = {true, true};
        int pend1 = -1;  // step of tile 1 whose P V is still to be issued
        for (int j = 0; ok && j < it.count; ++j) {
          const int J = J0 + j, entry = it.list[j];
          const bool a0 = label(entry, 0) != FM_TILE_FULL, a1 = label(entry, 1) != FM_TILE_FULL;
          ok = mbar_wait(bar.k_full(J % KS), (J / KS) & 1, p.status);
          if (ok && a0) {
            ok = issue_s(0, J);
            if (ok && j == last[0]) mma_commit(bar.q_empty(0));
          }
          if (ok && pend1 >= 0) {
            // tile 1's previous step: its V slot is released after this product
            ok = issue_pv(1, pend1, first[1], k);
            if (ok) mma_commit(bar.v_empty(pend1 % VS));
            first[1] = false;
            pend1 = -1;
          }
          if (ok && a1) {
            ok = issue_s(1, J);
            if (ok && j == last[1]) mma_commit(bar.q_empty(1));
            pend1 = J;
          }
          if (ok) mma_commit(bar.k_empty(J % KS));  // both tiles' S of this step issued
          if (ok && a0) {
            ok = issue_pv(0, J, first[0], k);
            first[0] = false;
          }
          // V of this step is released now unless tile 1 still needs it
          if (ok && !a1) {
            ok = mbar_wait(bar.v_full(J % VS), (J / VS) & 1, p.status);
            if (ok) mma_commit(bar.v_empty(J % VS));
          }
        }
        if (ok && pend1 >= 0) {
          ok = issue_pv(1, pend1, first[1], k);
          if (ok) mma_commit(bar.v_empty(pend1 % VS));
        }
        if (!ok) {
          record_failure(p.status, kStatusTimeout, kSiteFwdP);
          break;
        }
        J0 += it.count;
      }
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax) : "memory");
    // ------------------------------------------------------------ softmax of tile t
    const int t = warp >> 2;
    const int row = (warp & 3) * 32 + lane;  // query row within the block = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t ts = tmem + lane_base + col_s(t), to = tmem + lane_base + col_o(t);
    constexpr float kThresh = kFp8 ? kRescaleThresholdFp8 : kRescaleThreshold;
    volatile int* share = sched + 2 + 2 * t;
    // After a failed wait the warp keeps stepping through its items without
    // touching TMEM, so that the four warps pass the same named barriers and
    // the CTA can still reach its exit; `ok` is kept uniform across the warp.
    bool ok = true;
    int ns = 0;  // products of this tile so far
    for (int k = 0;; ++k) {
      if ((warp & 3) == 0 && lane == 0) {
        bool okr = true;
        share[k & 1] = read_item(k, okr);
      }
      group_bar(t);
      const int n = share[k & 1];
      if (n < 0) break;
      const Item it = decode(n);
      const int r = t == 0 ? it.r0 : it.r1;
      const bool tile_exists = r < p.Tr;
      const int bh = it.bh, bm = it.bm;
      // FP8: the true score is S times scale_Q(query block) * scale_K(key
      // block); the product folds into each tile's exponent scale c
      const float c_row = (kFp8 && tile_exists)
                              ? p.scale_log2 * p.qscale[static_cast<size_t>(bh) * p.Tr + r]
                              : p.scale_log2;
      float m = -INFINITY, l = 0.f;
      bool first = true;  // no product of this tile in the item yet
      for (int j = 0; j < it.count; ++j) {
        const int entry = it.list[j];
        const int lab = label(entry, t);
        if (lab == FM_TILE_FULL) continue;
        const int kb = entry >> 4;
        const float c =
            kFp8 ? c_row * p.kscale[static_cast<size_t>(bh) * p.Tc + kb] : c_row;
        // The element mask applies on PARTIAL tiles and on every tile of a short
        // last key block (its keys >= N do not exist and are masked).
        const bool short_keys = kShortLast && kb == p.Tc - 1;
        const bool partial = lab == FM_TILE_PARTIAL || short_keys;
        // lane l builds the masked-row bits of key column 32q + l for this
        // warp's 32 rows; a bit transpose hands each lane its own row's bits
        // over those 32 columns. The bound loads overlap the wait for S.
        uint32_t mbits[4] = {0u, 0u, 0u, 0u};
        if (partial) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int jc = kb * kTile + 32 * q + lane;
            uint32_t colbits = 0xffffffffu;  // a key >= N masks every row
            if (!kShortLast || jc < p.N) {
              const size_t col = static_cast<size_t>(bm) * p.N + jc;
              const int lts = p.mask.lts[col], lte = p.mask.lte[col];
              const int uts = p.mask.uts ? p.mask.uts[col] : 0;
              const int ute = p.mask.ute ? p.mask.ute[col] : 0;
              colbits = column_mask_bits(jc, lts, lte, uts, ute, p.mask.causal != 0,
                                         r * kTile + 32 * (warp & 3));
            }
            mbits[q] = warp_transpose_bits(colbits);
          }
        }
        if (ok) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar.s_full(t), ns & 1, p.status));
          if (!ok && lane == 0) record_failure(p.status, kStatusTimeout, kSiteFwdS);
        }
        if (ok) {
          tc_fence_after();
          uint32_t sv[128];
          tmem_ld64(ts, ts + 32, *reinterpret_cast<uint32_t(*)[64]>(sv));
          tmem_ld64(ts + 64, ts + 96, *reinterpret_cast<uint32_t(*)[64]>(sv + 64));
          if (partial) {
#pragma unroll
            for (int jj = 0; jj < 128; ++jj)
              sv[jj] = ((mbits[jj >> 5] >> (jj & 31)) & 1u) ? 0xff800000u : sv[jj];
          }
          float mx[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) mx[u] = __uint_as_float(sv[u]);
#pragma unroll
          for (int jj = 8; jj < 128; jj += 8) {
#pragma unroll
            for (int u = 0; u < 8; ++u) mx[u] = fmaxf(mx[u], __uint_as_float(sv[jj + u]));
          }
          const float pm =
              fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                    fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * c;
          const float m_new = fmaxf(m, pm);
          const bool rescale = m_new > m + kThresh;
          float alpha = 1.f;
          if (rescale) {
            alpha = ex2(m - m_new);
            m = m_new;
          }
          const float m_use = (m == -INFINITY) ? 0.f : m;
          // pairs of columns through the paired fp32 instructions: s * c - m
          // and the running pairs of partial sums take one issue slot per pair
          const uint64_t c2 = f2_make(c, c), nm2 = f2_make(-m_use, -m_use);
          uint64_t la = f2_make(0.f, 0.f), lb = f2_make(0.f, 0.f);
          // P is packed in place over the S registers already consumed: bf16
          // pairs in sv[0..63], or e4m3 quads in sv[0..31]
          float pq0 = 0.f, pq1 = 0.f;
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            float x0, x1;
            f2_split(f2_fma(f2_make(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])),
                            c2, nm2),
                     x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            if (i & 1)
              lb = f2_add(lb, f2_make(p0, p1));
            else
              la = f2_add(la, f2_make(p0, p1));
            if constexpr (kFp8) {
              // the scale keeps small probabilities above e4m3's subnormal range
              if (i & 1)
                sv[i >> 1] = pack_e4m3x4(pq0, pq1, p0 * kFp8PScale, p1 * kFp8PScale);
              else
                pq0 = p0 * kFp8PScale, pq1 = p1 * kFp8PScale;
            } else {
              sv[i] = pack_bf16x2(p0, p1);
            }
          }
          float l0, l1, l2, l3;
          f2_split(la, l0, l1);
          f2_split(lb, l2, l3);
          l = l * alpha + ((l0 + l1) + (l2 + l3));
          // P over S_t's own columns: keys [0, 128) as bf16 pairs in columns
          // [0, 64) (the A operand of P V), or as e4m3 quads in columns [0, 32)
          tmem_st32p(ts, sv);
          if constexpr (!kFp8) tmem_st32p(ts + 32, sv + 32);
          // O_t is quiescent here (its last product completed before S_t was
          // issued); the item's first product overwrites it, so no rescale then
          if (!first && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) tmem_scale32(to + 32 * ch, alpha);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.p_full(t));
        first = false;
        ++ns;
      }
      // ---------------------------------------------------------- epilogue of the item
      const bool live = ok && !first;
      if (live) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar.pv_done(t), (ns - 1) & 1, p.status));
        if (!ok && lane == 0) record_failure(p.status, kStatusTimeout, kSiteFwdO);
        tc_fence_after();
      }
      const bool has = live && ok && l > 0.f;
      // FP8: O accumulated (kFp8PScale P) (V / scale_V)
      const float inv = has ? (kFp8 ? p.vscale[bh] * (1.f / kFp8PScale) : 1.f) / l : 0.f;
      // rows >= N of a short last query block, and a missing second block, do
      // not exist: nothing is stored for them
      const bool row_exists = tile_exists && (!kShortLast || r * kTile + row < p.N);
      const size_t orow0 = static_cast<size_t>(bh) * p.N + static_cast<size_t>(r) * kTile + row;
      uint16_t* orow = p.o + (row_exists ? orow0 : 0) * D;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch)
        tmem_cols_to_bf16(to + 32 * ch, live && ok, inv, orow + 32 * ch, row_exists);
      // O_t has been read (the loads above completed): the next item's first
      // product may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.o_free(t));
      if (row_exists) {
        const float m_fin = (m == -INFINITY) ? 0.f : m;
        p.lse[orow0] = has ? (m_fin + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool kShortLast, bool kFp8 = false>
cudaError_t launch_fwd_t(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const FwdParams& p, cudaStream_t s) {
  using L = FwdLayout<D, kFp8>;
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D, kShortLast, kFp8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  // the register split inside the kernel needs the full pool at launch; a
  // build that allocated fewer registers per thread is refused, not run
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, fwd_kernel<D, kShortLast, kFp8>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * kThreads < kRegPool) return cudaErrorInvalidConfiguration;
  // persistent: one CTA per SM (at most one per work item); the item counter
  // starts at zero
  const int items = p.B * p.H * p.Tp;
  const unsigned grid = static_cast<unsigned>(items < p.num_sms ? items : p.num_sms);
  e = cudaMemsetAsync(p.sched, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  fwd_kernel<D, kShortLast, kFp8><<<grid, kThreads, L::kBytes, s>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int d, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       const FwdParams& p, cudaStream_t s) {
  const bool short_last = p.N % kTile != 0;
  if (d == 64)
    return short_last ? launch_fwd_t<64, true>(mq, mk, mv, p, s)
                      : launch_fwd_t<64, false>(mq, mk, mv, p, s);
  return short_last ? launch_fwd_t<128, true>(mq, mk, mv, p, s)
                    : launch_fwd_t<128, false>(mq, mk, mv, p, s);
}

cudaError_t launch_fwd_fp8(const CUtensorMap& mq8, const CUtensorMap& mk8,
                           const CUtensorMap& mvt8, const FwdParams& p, cudaStream_t s) {
  return p.N % kTile != 0 ? launch_fwd_t<128, true, true>(mq8, mk8, mvt8, p, s)
                          : launch_fwd_t<128, false, true>(mq8, mk8, mvt8, p, s);
}

}  // namespace fm
