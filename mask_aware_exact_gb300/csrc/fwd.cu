// Forward kernel: exact attention over the non-FULL tiles of one 128-row query
// block ("FlashMask: Efficient and Rich Mask Extension of FlashAttention",
// abstract: skip masked computation, exact result; "FlashAttention-3",
// abstract: warp specialisation overlapping TMA data movement with tensor-core
// work, and block-wise matmul interleaved with softmax).
//
// The non-FULL key blocks of the query block are visited one per step. The
// tensor cores run ahead of the softmax: S_{j+2} = Q K_{j+2}^T is issued as
// soon as O += P_j V_j (the last reader of its TMEM region) has completed, so
// the S products stay off the chain softmax_j -> O += P_j V_j, and the
// softmax warps find S_{j+1} ready when they finish step j. P_j is written
// over S_j's own region.
//
// The two softmax warpgroups split every key block in halves and keep
// separate online-softmax states: warpgroup w owns keys [64w, 64w+64) of every
// block, its own running maximum and sum per row and its own accumulator O_w
// = sum over its keys of P V. So the warpgroups never wait for each other
// inside a step (no exchange of row maxima); the two states are merged once,
// in the epilogue: with m = max(m_0, m_1) and f_w = 2^(m_w - m),
// O = (f_0 O_0 + f_1 O_1) / (f_0 l_0 + f_1 l_1), the exact result.
//
// Given a workspace sized for the backward, the scheduler thread also zeroes
// each query block's rows of the backward's fp32 dQ accumulator with bulk
// copies from a zeroed shared-memory buffer, using HBM bandwidth the forward
// leaves idle, and the backward preprocess then skips that pass.
//
// Persistent CTAs (one per SM) take query blocks from a work counter; see the
// kernel's comment. Warp roles (384 threads):
//   warps 0-7  softmax, two warpgroups. Thread (w, r) owns query row r (= TMEM
//              lane r) and key columns [64w, 64w+64) of every block: it loads
//              its 64 S values into registers, applies the element mask on
//              PARTIAL tiles, keeps its running max and partial sum in fp32
//              (log2 domain), and writes its P slice into TMEM. O_w is
//              rescaled only when that max grows by more than 2^8 (lazy
//              rescaling: exact after the final division). Epilogue: merge of
//              the two halves, O (staged, stored by TMA) and LSE, run one
//              item late, inside the next item's first step.
//   warp 8     work scheduler and TMA producer of Q (once per item) and K
//              blocks (two-slot ring).
//   warp 9     S issuer (one thread): S_j once K_j has landed and the P V
//              products of step j-2 (the last readers of its TMEM region)
//              have completed.
//   warp 10    TMA producer of V blocks (two-slot ring).
//   warp 11    P V issuer (one thread): for step j waits until V_j has landed
//              and both halves of P_j are written (and, at an item's first
//              step, the previous item's O_0 and O_1 have been read out), then
//              issues O_w += P_{j,w} V_{j,w} for both halves.
//   S and P V come from two threads so that neither waits behind the other:
//   one thread issuing both spends each step issuing P V, waiting for those
//   products to complete (the next S overwrites the columns they read) and
//   issuing S, about 2000 cycles per step in a clock64 trace, during which
//   the softmax warps waited for S.
//
// TMEM columns (512 allocated): S regions [0,128) [128,256), O_0 [256, 256+d),
// O_1 [384, 384+d). Ordering: S_{j+2} reuses the region of S_j / P_j once the
// products of step j have completed; warpgroup w rescales O_w at step j only
// after the products of step j-1 have completed.
#include "internal.h"
#include "ptx.cuh"
#include "ptx_fp8.cuh"
#include "flashmask.h"

namespace fm {

namespace {

constexpr int kThreads = 384;
constexpr int kSRegions = 2;  // TMEM S/P regions of 128 columns
constexpr int kKSlots = 2, kVSlots = 2;
// O accumulator of softmax warpgroup w (its half of the keys of every block)
__device__ __forceinline__ uint32_t col_o(int w) { return 256u + 128u * static_cast<uint32_t>(w); }
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// FP8: P is stored as e4m3(p * kFp8PScale). With the running maximum lagging
// by at most kRescaleThresholdFp8 (log2 units), p < 2^threshold and
// p * kFp8PScale stays below 448, the largest finite e4m3 value.
constexpr float kRescaleThresholdFp8 = 4.0f;
constexpr float kFp8PScale = 28.0f;

template <int D, bool kFp8>
struct FwdLayout {
  static constexpr int kTileBytes = kTile * D * (kFp8 ? 1 : 2);  // one 128 x d tile
  static constexpr int kChunks = kFp8 ? 1 : D / 64;  // 128-byte-wide TMA boxes per tile
  static constexpr int kChunk = 16384;              // 128 rows x 128 bytes
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;             // kKSlots x kTileBytes
  static constexpr int kV = kK + kKSlots * kTileBytes;   // kVSlots x kTileBytes
  // bf16 O staging for the TMA stores: 128 rows x D, as 128-byte swizzled
  // 64-column halves of 16 KB
  static constexpr int kOStage = kV + kVSlots * kTileBytes;
  static constexpr int kRed = kOStage + kTile * D * 2;  // fp32 [m, l][2 groups][128]
  static constexpr int kBar = kRed + 2 * 2 * kTile * 4;
  // q_full, k_full[2], v_full[2], s_full[2], p_full[2], pv_done[2],
  // sched_full[2], sched_empty[2], o_free. K slot, V slot and S region of step
  // J are all J % 2, so "S_J done" also frees K slot J % 2 and "P_J V_J done"
  // also frees V slot J % 2.
  static_assert(kKSlots == kSRegions && kVSlots == kSRegions, "slots follow the S regions");
  static constexpr int kNumBars = 1 + kKSlots + kVSlots + 3 * kSRegions + 5;
  // int[8] x 4: the item ring (two entries), then the item as softmax warp 0
  // shares it (two entries)
  static constexpr int kSched = (kBar + kNumBars * 8 + 31) / 32 * 32;
  static constexpr int kTmemSlot = kSched + 128;
  // 16 KB of zeros, the source of the bulk copies that clear the dQ
  // accumulator rows of each query block (bf16 forward only)
  static constexpr int kZero = kTmemSlot + 16;
  static constexpr int kZeroBytes = kFp8 ? 0 : 16384;
  static constexpr int kBytes = kZero + kZeroBytes;
};

static_assert(FwdLayout<128, false>::kOStage % 1024 == 0 &&
                  FwdLayout<64, false>::kOStage % 1024 == 0 &&
                  FwdLayout<128, true>::kOStage % 1024 == 0,
              "the 128-byte swizzle of the O staging buffer needs 1024-byte alignment");
static_assert(FwdLayout<128, false>::kBytes <= 227 * 1024, "shared memory per CTA");
static_assert(FwdLayout<128, false>::kSched % 32 == 0 && FwdLayout<64, false>::kSched % 32 == 0 &&
                  FwdLayout<128, true>::kSched % 32 == 0,
              "the item ring is read and written with 16-byte shared-memory accesses");
static_assert(FwdLayout<128, false>::kZero % 16 == 0, "bulk copies read 16-byte aligned sources");

struct FwdBars {
  uint32_t base;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t k_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t v_full(int s) const { return base + 8 * (1 + kKSlots + s); }
  __device__ uint32_t s_full(int r) const { return base + 8 * (1 + kKSlots + kVSlots + r); }
  __device__ uint32_t p_full(int r) const {
    return base + 8 * (1 + kKSlots + kVSlots + kSRegions + r);
  }
  __device__ uint32_t pv_done(int r) const {
    return base + 8 * (1 + kKSlots + kVSlots + 2 * kSRegions + r);
  }
  __device__ uint32_t sched_full(int s) const {
    return base + 8 * (1 + kKSlots + kVSlots + 3 * kSRegions + s);
  }
  __device__ uint32_t sched_empty(int s) const {
    return base + 8 * (3 + kKSlots + kVSlots + 3 * kSRegions + s);
  }
  __device__ uint32_t o_free() const { return base + 8 * (5 + kKSlots + kVSlots + 3 * kSRegions); }
};

// Roles that read each published work item: the S issuer, the P V issuer, the
// V producer and softmax warp 0 (which shares it with the other seven).
constexpr int kSchedReaders = 4;


__device__ __forceinline__ void ld_shared_v4i(uint32_t addr, int& a, int& b, int& c, int& d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void st_shared_v4i(uint32_t addr, int a, int b, int c, int d) {
  st_shared_v4(addr, static_cast<uint32_t>(a), static_cast<uint32_t>(b), static_cast<uint32_t>(c),
               static_cast<uint32_t>(d));
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

// 3-D tiled store of one box from shared memory (x, y, z = column, row within
// the head, head), in the current bulk async-group; rows outside the tensor
// map (beyond the head's length) are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(z), "r"(src)
      : "memory");
}

// Merges 32 TMEM columns of this lane's row from two accumulators, f0 * A +
// f1 * B (the TMEM loads run on every lane of the warp), and writes them as
// bf16 to 64 bytes of the row's 128-byte swizzled staging row, 16-byte units
// [unit0, unit0 + 4).
__device__ __forceinline__ void tmem_merge_to_stage(uint32_t ta, uint32_t tb, bool live, float f0,
                                                    float f1, uint32_t stage_half, int row,
                                                    int unit0) {
  uint32_t a[32], b[32];
  if (live) {
    tmem_ld32(ta, a);
    tmem_ld32(tb, b);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) a[i] = b[i] = 0u;
  }
  uint32_t w16[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    w16[i] = pack_bf16x2(__uint_as_float(a[2 * i]) * f0 + __uint_as_float(b[2 * i]) * f1,
                         __uint_as_float(a[2 * i + 1]) * f0 + __uint_as_float(b[2 * i + 1]) * f1);
#pragma unroll
  for (int u = 0; u < 4; ++u)
    st_shared_v4(stage_half + sw128_offset(row, unit0 + u), w16[4 * u], w16[4 * u + 1],
                 w16[4 * u + 2], w16[4 * u + 3]);
}

// kShortLast: N is not a multiple of 128. kFp8 (d = 128 only): e4m3 Q, K and
// transposed V with block scales, kind::f8f6f4 MMAs (K = 32 per instruction),
// P stored as e4m3(p * kFp8PScale).
//
// Persistent: one CTA per SM takes work items (one query block of one head)
// from a global counter until none is left. The Q/K producer claims the items
// and publishes them to the other roles through a two-entry ring in shared
// memory. Every role numbers the key blocks it handles with one running step
// index J across items, so the K, V and S rings, their barriers and the
// tensor pipe run on from one item into the next: the next item's Q, first K
// blocks and first S products are loaded and computed while the softmax warps
// finish the current item. Two hand-offs cross an item boundary: Q is
// reloaded once the last S of the previous item has completed, and the first
// O += P V of an item (which overwrites O) waits until the softmax warps have
// read the previous item's O out of TMEM (o_free).
template <int D, bool kShortLast, bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mo,
               const FwdParams p) {
  using L = FwdLayout<D, kFp8>;
  static_assert(!kFp8 || D == 128, "the FP8 forward is for d = 128");
  constexpr int kOCols = D / 2;  // O columns per softmax warpgroup
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = p.B * p.H * p.Tr;

  if ((smem_u32(smem) & 1023u) != 0) {  // 128-byte swizzle atoms need 1024-byte alignment
    if (tid == 0) record_failure(p.status, kStatusLayout, kSiteFwdSmemAlign);
    return;
  }
  const uint32_t sQ = smem_u32(smem + L::kQ), sK = smem_u32(smem + L::kK),
                 sV = smem_u32(smem + L::kV), sO = smem_u32(smem + L::kOStage);
  float* red = reinterpret_cast<float*>(smem + L::kRed);
  // int[8] entries: [0, 2) the item ring, [2, 4) the item as softmax warp 0
  // shares it with the other seven
  const uint32_t ring = smem_u32(smem + L::kSched), share = ring + 64;
  const FwdBars bar{smem_u32(smem + L::kBar)};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);

  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if constexpr (!kFp8) {
    if (p.dq_zero != nullptr) {
      uint4* z = reinterpret_cast<uint4*>(smem + L::kZero);
      for (int i = tid; i < L::kZeroBytes / 16; i += blockDim.x) z[i] = make_uint4(0u, 0u, 0u, 0u);
      fence_proxy_async_smem();  // the zeros are read by the bulk-copy engine
    }
  }
  if (blockIdx.x == 0 && tid == 0) p.status[3] = p.dq_zero != nullptr ? p.dq_tag : 0;
  if (tid == 0) {
    mbar_init(bar.q_full(), 1);
    for (int s = 0; s < kKSlots; ++s) mbar_init(bar.k_full(s), 1);
    for (int s = 0; s < kVSlots; ++s) mbar_init(bar.v_full(s), 1);
    for (int g = 0; g < kSRegions; ++g) {
      mbar_init(bar.s_full(g), 1);
      mbar_init(bar.p_full(g), 8);
      mbar_init(bar.pv_done(g), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar.sched_full(s), 1);
      mbar_init(bar.sched_empty(s), kSchedReaders);
    }
    mbar_init(bar.o_free(), 8);
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Work item n: head-major, longest query blocks of each head first, so the
  // CTAs working at the same time share one head's K and V in L2.
  // The scheduler looks up everything an item needs once and publishes it:
  // {n, r (query block), ntiles, first list entry, bh (head), bm (mask
  // head), -, -}, n = -1 when no item is left. The other roles then start an
  // item without global loads or integer divisions on their paths.
  struct Item {
    int n, bh, bm, r, ntiles, first, head_row0, q_row0;
    const int32_t* list;
  };
  auto make_item = [&](const int (&v)[8]) -> Item {
    Item it;
    it.n = v[0];
    it.r = v[1];
    it.ntiles = v[2];
    it.first = v[3];
    it.bh = v[4];
    it.bm = v[5];
    it.list = p.row_list + (static_cast<size_t>(it.bm) * p.Tr + it.r) * p.Tc;
    it.head_row0 = it.bh * p.N;               // first row of this head in [B*H*N, d]
    it.q_row0 = it.head_row0 + it.r * kTile;  // first query row of the block
    return it;
  };
  // The k-th item of this CTA (k = 0, 1, ...) from the ring into v (n = -1
  // when no item is left or the wait gave up; then `ok` is false).
  auto read_item = [&](int k, int (&v)[8], bool& ok) {
    const int s = k & 1;
    v[0] = -1;
    v[1] = v[2] = v[3] = v[4] = v[5] = v[6] = v[7] = 0;
    if (!mbar_wait(bar.sched_full(s), (k >> 1) & 1, p.status)) {
      record_failure(p.status, kStatusTimeout, kSiteFwdSched);
      ok = false;
      return;
    }
    ld_shared_v4i(ring + 32 * s, v[0], v[1], v[2], v[3]);
    ld_shared_v4i(ring + 32 * s + 16, v[4], v[5], v[6], v[7]);
    mbar_arrive(bar.sched_empty(s));
  };
  auto take_item = [&](int k, bool& ok) -> Item {
    int v[8];
    read_item(k, v, ok);
    return make_item(v);
  };

  if (warp == 8) {
    // ------------------------------------------------------------ scheduler, TMA producer of Q, K
    if (lane == 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      // claims an item and looks up its ring entry
      auto claim = [&](int (&v)[8]) {
        v[0] = -1;
        v[1] = v[2] = v[3] = v[4] = v[5] = v[6] = v[7] = 0;
        const int n = atomicAdd(p.sched, 1);
        if (n >= n_items) return;
        const int bh = n / p.Tr, rank = n % p.Tr;
        const int b = bh / p.H, h = bh % p.H;
        const int bm = b * p.mask.Hm + h / (p.H / p.mask.Hm);
        const size_t mr = static_cast<size_t>(bm) * p.Tr;
        const int r = p.row_order[mr + rank];
        const int nt = p.row_count[mr + r];
        v[0] = n;
        v[1] = r;
        v[2] = nt;
        v[3] = nt > 0 ? p.row_list[(mr + r) * p.Tc] : 0;
        v[4] = bh;
        v[5] = bm;
      };
      auto publish = [&](int s, const int (&v)[8]) {
        st_shared_v4i(ring + 32 * s, v[0], v[1], v[2], v[3]);
        st_shared_v4i(ring + 32 * s + 16, v[4], v[5], v[6], v[7]);
        mbar_arrive(bar.sched_full(s));
      };
      // K of step J into slot J % 2 once S_{J-2} has completed; kb is the
      // key block, bh the head (3-D map: rows past the head's end read zeros)
      auto load_k = [&](int J, int kb, int bh) -> bool {
        const int slot = J % kKSlots;
        if (J >= kKSlots &&
            !mbar_wait(bar.s_full(slot), ((J / kKSlots) - 1) & 1, p.status)) {
          record_failure(p.status, kStatusTimeout, kSiteFwdKEmpty);
          return false;
        }
        mbar_arrive_expect_tx(bar.k_full(slot), L::kTileBytes);
        for (int ch = 0; ch < L::kChunks; ++ch)
          tma_load_3d(sK + slot * L::kTileBytes + ch * L::kChunk, &mk, ch * 64, kb * kTile, bh,
                      bar.k_full(slot));
        return true;
      };
      int cur[8];
      claim(cur);
      publish(0, cur);
      bool ok = true;
      int J = 0, J_last = -1;  // running step; last step of the previous item with tiles
      for (int k = 0; ok && cur[0] >= 0; ++k) {
        const Item it = make_item(cur);
        if (it.ntiles > 0) {
          // the Q buffer is free once the last S of the previous item is done
          if (J_last >= 0 && !mbar_wait(bar.s_full(J_last % kSRegions),
                                        (J_last / kSRegions) & 1, p.status)) {
            record_failure(p.status, kStatusTimeout, kSiteFwdKEmpty);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar.q_full(), L::kTileBytes);
          for (int ch = 0; ch < L::kChunks; ++ch)
            tma_load_3d(sQ + ch * L::kChunk, &mq, ch * 64, it.r * kTile, it.bh, bar.q_full());
          int e_next = it.first;  // list entries read one step ahead
          for (int j = 0; ok && j < it.ntiles; ++j, ++J) {
            const int e = e_next;
            if (j + 1 < it.ntiles) e_next = it.list[j + 1];
            ok = load_k(J, e >> 2, it.bh);
          }
          J_last = J - 1;
        }
        if constexpr (!kFp8) {
          // zero this query block's rows of the backward's dQ accumulator
          // (contiguous: 128 rows of D fp32) while the forward runs, which
          // leaves HBM mostly idle, instead of in the backward preprocess;
          // issued after the item's Q and K loads so as not to delay them
          if (p.dq_zero != nullptr) {
            char* dst = reinterpret_cast<char*>(
                p.dq_zero + (static_cast<size_t>(it.bh) * p.Tr + it.r) * kTile * D);
#pragma unroll
            for (int c = 0; c < kTile * D * 4 / L::kZeroBytes; ++c)
              bulk_store(dst + c * L::kZeroBytes, smem_u32(smem + L::kZero), L::kZeroBytes);
            bulk_commit_group();
            bulk_wait_read_8();
          }
        }
        // claim the next item once this one's loads are issued; its ring
        // entry was last used by item k - 1, which every reader has taken
        int nxt[8];
        claim(nxt);
        const int s = (k + 1) & 1;
        if (k >= 1 && !mbar_wait(bar.sched_empty(s), ((k - 1) >> 1) & 1, p.status)) {
          record_failure(p.status, kStatusTimeout, kSiteFwdSched);
          ok = false;
          break;
        }
        publish(s, nxt);
#pragma unroll
        for (int i = 0; i < 8; ++i) cur[i] = nxt[i];
      }
      if constexpr (!kFp8) bulk_wait_all();  // the zeroing copies, before the CTA exits
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ TMA producer of V
    if (lane == 0) {
      tma_prefetch_desc(&mv);
      bool ok = true;
      int J = 0;
      for (int k = 0; ok; ++k) {
        const Item it = take_item(k, ok);
        if (it.n < 0) break;
        int e_next = it.first;  // list entries read one step ahead
        for (int j = 0; ok && j < it.ntiles; ++j, ++J) {
          const int slot = J % kVSlots;
          const int kb = e_next >> 2;
          if (j + 1 < it.ntiles) e_next = it.list[j + 1];
          if (J >= kVSlots &&
              !mbar_wait(bar.pv_done(slot), ((J / kVSlots) - 1) & 1, p.status)) {
            record_failure(p.status, kStatusTimeout, kSiteFwdVEmpty);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar.v_full(slot), L::kTileBytes);
          if constexpr (kFp8) {
            // V^T tile: the head's 128 rows of d, the block's 128 keys
            tma_load_2d(sV + slot * L::kTileBytes, &mv, kb * kTile, it.bh * 128,
                        bar.v_full(slot));
          } else {
            for (int ch = 0; ch < L::kChunks; ++ch)
              tma_load_3d(sV + slot * L::kTileBytes + ch * L::kChunk, &mv, ch * 64, kb * kTile,
                          it.bh, bar.v_full(slot));
          }
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ S issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = kFp8 ? idesc_e4m3(128, 128) : idesc_bf16(128, 128, 0, 0);
      constexpr int kSSteps = kFp8 ? D / 32 : D / 16;  // K steps of S = Q K^T
      // Shared-memory descriptors are built once: the address field (bits
      // 0-13, in 16-byte units) of every operand stays below 2^14 here, so a
      // descriptor for base + off is the base descriptor plus off / 16. This
      // keeps the per-MMA instruction stream of this thread short.
      const uint64_t dq_base = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dk_base = sdesc_sw128(sK, 16, 1024);
      bool ok = true;
      int J = 0, ti = 0;  // running step; items with tiles so far
      for (int k = 0; ok; ++k) {
        const Item it = take_item(k, ok);
        if (it.n < 0) break;
        const int ntiles = it.ntiles;
        if (ntiles == 0) continue;
        if (!mbar_wait(bar.q_full(), ti & 1, p.status)) {
          record_failure(p.status, kStatusTimeout, kSiteFwdQ);
          break;
        }
        // S of step J into region J % 2 once K_J has landed and the P V
        // products of step J - 2 (the last readers of that region) have
        // completed; this thread waits only for those, never for the
        // softmax, so S runs up to two steps ahead of the P V products
        for (int j = 0; ok && j < ntiles; ++j, ++J) {
          const int slot = J % kKSlots, g = J % kSRegions;
          if (J >= kSRegions &&
              !mbar_wait(bar.pv_done(g), ((J / kSRegions) - 1) & 1, p.status)) {
            record_failure(p.status, kStatusTimeout, kSiteFwdO);
            ok = false;
            break;
          }
          if (!mbar_wait(bar.k_full(slot), (J / kKSlots) & 1, p.status)) {
            record_failure(p.status, kStatusTimeout, kSiteFwdK);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t kd = dk_base + static_cast<uint64_t>((slot * L::kTileBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kSSteps; ++kk) {
            // 32 bytes of each 128-byte row per K step (16 bf16 or 32 e4m3)
            const uint64_t off16 =
                static_cast<uint64_t>(((kk >> 2) * L::kChunk + (kk & 3) * 32) >> 4);
            if constexpr (kFp8)
              mma_ss_f8(tmem + 128 * g, dq_base + off16, kd + off16, idesc_s, kk > 0);
            else
              mma_ss(tmem + 128 * g, dq_base + off16, kd + off16, idesc_s, kk > 0);
          }
          mma_commit(bar.s_full(g));  // also frees K slot J % 2
        }
        ++ti;
      }
    }
  } else if (warp == 11) {
    // ------------------------------------------------------------ P V issuer
    // For step j: waits until V_j has landed, both halves of P_j are written
    // (and, at an item's first step, the previous item's O_0 and O_1 have been
    // read out), then issues O_w += P_{j,w} V_{j,w} for both halves.
    if (lane == 0) {
      constexpr uint32_t idesc_pv = kFp8 ? idesc_e4m3(128, D) : idesc_bf16(128, D, 0, 1);
      constexpr int kPvSteps = kFp8 ? 4 : 8;  // K steps (keys) of O += P V
      // V is MN-major [keys][d] in bf16, K-major [d][keys] as e4m3 V^T
      const uint64_t dv_base = kFp8 ? sdesc_sw128(sV, 16, 1024) : sdesc_sw128(sV, 16384, 1024);
      bool ok = true;
      int J = 0, ti = 0;
      for (int k = 0; ok; ++k) {
        const Item it = take_item(k, ok);
        if (it.n < 0) break;
        const int ntiles = it.ntiles;
        if (ntiles == 0) continue;
        for (int j = 0; j < ntiles; ++j, ++J) {
          const int g = J % kSRegions, vs = J % kVSlots;
          ok = mbar_wait(bar.v_full(vs), (J / kVSlots) & 1, p.status);
          // the item's first products overwrite O_0 and O_1: the previous
          // item's accumulators must have been read out
          if (j == 0 && ti > 0) ok = ok && mbar_wait(bar.o_free(), (ti - 1) & 1, p.status);
          ok = ok && mbar_wait(bar.p_full(g), (J / kSRegions) & 1, p.status);
          if (!ok) {
            record_failure(p.status, kStatusTimeout, kSiteFwdP);
            break;
          }
          tc_fence_after();
          const uint64_t vd = dv_base + static_cast<uint64_t>((vs * L::kTileBytes) >> 4);
#pragma unroll
          for (int w = 0; w < 2; ++w) {
#pragma unroll
            for (int kk = 0; kk < kPvSteps / 2; ++kk) {
              // O_w += P_w V_w over keys [64w, 64w+64): A = P_w, 8 TMEM
              // columns per K step from column 64w (bf16 pairs or e4m3
              // quads); B = the next 16 key rows of V (bf16) or the next 32
              // key bytes of each row of V^T (e4m3)
              if constexpr (kFp8)
                mma_ts_f8(tmem + col_o(w), tmem + 128 * g + 64 * w + 8 * kk,
                          vd + static_cast<uint64_t>((64 * w + kk * 32) >> 4), idesc_pv,
                          (j > 0 || kk > 0));
              else
                mma_ts(tmem + col_o(w), tmem + 128 * g + 64 * w + 8 * kk,
                       vd + static_cast<uint64_t>(((4 * w + kk) * 2048) >> 4), idesc_pv,
                       (j > 0 || kk > 0));
            }
          }
          mma_commit(bar.pv_done(g));  // also frees V slot J % 2
        }
        ++ti;
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int w = warp >> 2;                 // warpgroup: key columns [64w, 64w+64)
    const int row = (warp & 3) * 32 + lane;  // query row within the block = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    constexpr float kThresh = kFp8 ? kRescaleThresholdFp8 : kRescaleThreshold;
    // After a failed wait the warp keeps stepping through its items without
    // touching TMEM, so that all eight warps pass the same named barriers and
    // the CTA can still reach its exit; `ok` is kept uniform across the warp.
    bool ok = true;
    int J = 0;  // running step
    // The epilogue of an item (query block r of head bh whose last step was
    // jl; has_tiles = 0 for an item no key sees): the two halves' states are
    // merged, O = (f_0 O_0 + f_1 O_1) / (f_0 l_0 + f_1 l_1), staged as bf16
    // and stored by TMA, and LSE written. It runs one item late, inside the
    // next item's first step once that step's P has been written, so that the
    // last P V products of the item have completed by then and the next
    // item's first S and softmax step overlap them instead of waiting.
    auto finish = [&](float m_, float l_, int r_, int bh_, int has_tiles, int jl) {
      if (ok && has_tiles) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar.pv_done(jl % kSRegions),
                                               (jl / kSRegions) & 1, p.status));
        if (!ok && lane == 0) record_failure(p.status, kStatusTimeout, kSiteFwdO);
        tc_fence_after();
      }
      // each warpgroup publishes its row maximum and sum
      red[w * kTile + row] = m_;
      red[(2 + w) * kTile + row] = l_;
      // the O staging buffer is free once the previous item's stores have
      // read it (long done: a whole item ago)
      if (tid == 0) bulk_wait_read_all();
      softmax_bar();
      const float m_o = red[(w ^ 1) * kTile + row], l_o = red[(2 + (w ^ 1)) * kTile + row];
      const float m_all = fmaxf(m_, m_o);
      const float f_self = (m_ == -INFINITY) ? 0.f : ex2(m_ - m_all);
      const float f_oth = (m_o == -INFINITY) ? 0.f : ex2(m_o - m_all);
      const float ltot = l_ * f_self + l_o * f_oth;
      const bool live = ok && has_tiles;
      const bool has = live && ltot > 0.f;
      // FP8: O accumulated (kFp8PScale P) (V / scale_V)
      const float inv = has ? (kFp8 ? p.vscale[bh_] * (1.f / kFp8PScale) : 1.f) / ltot : 0.f;
      const float f0 = (w == 0 ? f_self : f_oth) * inv, f1 = (w == 0 ? f_oth : f_self) * inv;
      // rows >= N of a short last query block do not exist: no LSE for them
      // (their O rows lie outside the tensor map and are not stored)
      const bool row_exists = !kShortLast || r_ * kTile + row < p.N;
      // this warpgroup's columns [w D/2, w D/2 + D/2) of the row go to the
      // staging buffer: half w for d = 128, units [4w, 4w + 4) of the single
      // half for d = 64; one thread then stores the tile with TMA, so the
      // softmax warps issue no global stores of O
#pragma unroll
      for (int ch = 0; ch < kOCols / 32; ++ch)
        tmem_merge_to_stage(tmem + lane_base + col_o(0) + w * kOCols + 32 * ch,
                            tmem + lane_base + col_o(1) + w * kOCols + 32 * ch, live, f0, f1,
                            sO + (D == 128 ? w * 16384 : 0), row, D == 128 ? 4 * ch : 4 * w);
      if (has_tiles) {
        // O_0 and O_1 have been read (the loads above completed): the next
        // item's first products may overwrite them
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.o_free());
      }
      fence_proxy_async_smem();  // the staged rows are read by the TMA engine
      if (w == 0 && row_exists) {
        const float m_fin = (m_all == -INFINITY) ? 0.f : m_all;
        p.lse[static_cast<size_t>(bh_) * p.N + r_ * kTile + row] =
            has ? (m_fin + __log2f(ltot)) * 0.69314718055994531f : -INFINITY;
      }
      // every warp has read the exchange buffer before the next epilogue
      // writes it, and has staged its O rows
      softmax_bar();
      if (tid == 0) {
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf)
          tma_store_3d(&mo, sO + hf * 16384, 64 * hf, r_ * kTile, bh_);
        bulk_commit_group();
      }
    };
    bool pend = false;  // an item whose epilogue is still to run
    float pend_m = 0.f, pend_l = 0.f;
    int pend_r = 0, pend_bh = 0, pend_jl = 0;
    for (int k = 0;; ++k) {
      // warp 0 takes the item from the ring and shares it through shared
      // memory, so that the eight warps agree on it even after a failure
      if (warp == 0 && lane == 0) {
        bool okr = true;
        int v[8];
        read_item(k, v, okr);
        st_shared_v4i(share + 32 * (k & 1), v[0], v[1], v[2], v[3]);
        st_shared_v4i(share + 32 * (k & 1) + 16, v[4], v[5], v[6], v[7]);
      }
      softmax_bar();
      int v[8];
      ld_shared_v4i(share + 32 * (k & 1), v[0], v[1], v[2], v[3]);
      ld_shared_v4i(share + 32 * (k & 1) + 16, v[4], v[5], v[6], v[7]);
      if (v[0] < 0) break;
      const Item it = make_item(v);
      const int ntiles = it.ntiles, r = it.r, bh = it.bh, bm = it.bm;
      // FP8: the true score is S times scale_Q(query block) * scale_K(key
      // block); the product folds into each tile's exponent scale c
      const float c_row = kFp8 ? p.scale_log2 * p.qscale[static_cast<size_t>(bh) * p.Tr + r]
                               : p.scale_log2;
      float m = -INFINITY, l = 0.f;
      // The element mask applies on PARTIAL tiles and on every tile of a short
      // last key block (its keys >= N do not exist and are masked). Lane l
      // needs the bounds of key columns 64w + l and 64w + 32 + l of a masked
      // step's block; they are loaded one step ahead (and the list entries
      // two steps ahead), so that their latency hides behind a step.
      auto masked_step = [&](int e) {
        return (e & 3) == FM_TILE_PARTIAL || (kShortLast && (e >> 2) == p.Tc - 1);
      };
      auto load_bounds = [&](int e, int (&bd)[8]) {
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int jc = (e >> 2) * kTile + 64 * w + 32 * kk + lane;
          bd[4 * kk] = bd[4 * kk + 1] = bd[4 * kk + 2] = bd[4 * kk + 3] = 0;
          if (!kShortLast || jc < p.N) {
            const size_t col = static_cast<size_t>(bm) * p.N + jc;
            bd[4 * kk] = p.mask.lts[col];
            bd[4 * kk + 1] = p.mask.lte[col];
            bd[4 * kk + 2] = p.mask.uts ? p.mask.uts[col] : 0;
            bd[4 * kk + 3] = p.mask.ute ? p.mask.ute[col] : 0;
          }
        }
      };
      int ent_nxt = ntiles > 1 ? it.list[1] : 0;  // the entry of step j + 1
      int bnd[8] = {0, 0, 0, 0, 0, 0, 0, 0};       // bounds of step j
      if (ntiles > 0 && masked_step(it.first)) load_bounds(it.first, bnd);
      int entry_cur = it.first;
      for (int j = 0; j < ntiles; ++j) {
        const int Jj = J + j;
        const int entry = entry_cur;
        int bnd_nxt[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (j + 1 < ntiles && masked_step(ent_nxt)) load_bounds(ent_nxt, bnd_nxt);
        const int ent_nn = j + 2 < ntiles ? it.list[j + 2] : 0;
        const int g = Jj % kSRegions;
        const float c =
            kFp8 ? c_row * p.kscale[static_cast<size_t>(bh) * p.Tc + (entry >> 2)] : c_row;
        const bool partial = masked_step(entry);
        // lane l builds the masked-row bits of key column 64w + 32k + l for this
        // warp's 32 rows; a bit transpose hands each lane its own row's bits
        // over those 32 columns
        uint32_t mbits[2] = {0u, 0u};
        if (partial) {
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const int jc = (entry >> 2) * kTile + 64 * w + 32 * kk + lane;
            uint32_t colbits = 0xffffffffu;  // a key >= N masks every row
            if (!kShortLast || jc < p.N)
              colbits = column_mask_bits(jc, bnd[4 * kk], bnd[4 * kk + 1], bnd[4 * kk + 2],
                                         bnd[4 * kk + 3], p.mask.causal != 0,
                                         r * kTile + 32 * (warp & 3));
            mbits[kk] = warp_transpose_bits(colbits);
          }
        }
        entry_cur = ent_nxt;
        ent_nxt = ent_nn;
#pragma unroll
        for (int i = 0; i < 8; ++i) bnd[i] = bnd_nxt[i];
        if (ok) {
          ok = __all_sync(0xffffffffu,
                          mbar_wait(bar.s_full(g), (Jj / kSRegions) & 1, p.status));
          if (!ok && lane == 0) record_failure(p.status, kStatusTimeout, kSiteFwdS);
        }
        uint32_t sv[64];
        float pm = -INFINITY;
        if (ok) {
          tc_fence_after();
          const uint32_t s_addr = tmem + lane_base + 128 * g + 64 * w;
          tmem_ld64(s_addr, s_addr + 32, sv);
          if (partial) {
#pragma unroll
            for (int jj = 0; jj < 64; ++jj)
              sv[jj] = ((mbits[jj >> 5] >> (jj & 31)) & 1u) ? 0xff800000u : sv[jj];
          }
          // four independent chains of three-input maxima over the 64 columns
          float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
          for (int jj = 0; jj < 64; jj += 8) {
            mx0 = fmax3(mx0, __uint_as_float(sv[jj]), __uint_as_float(sv[jj + 1]));
            mx1 = fmax3(mx1, __uint_as_float(sv[jj + 2]), __uint_as_float(sv[jj + 3]));
            mx2 = fmax3(mx2, __uint_as_float(sv[jj + 4]), __uint_as_float(sv[jj + 5]));
            mx3 = fmax3(mx3, __uint_as_float(sv[jj + 6]), __uint_as_float(sv[jj + 7]));
          }
          pm = fmax3(fmaxf(mx0, mx1), mx2, mx3) * c;
        }
        if (ok) {
          // this warpgroup's own running maximum over its half of the keys
          const float m_new = fmaxf(m, pm);
          const bool rescale = m_new > m + kThresh;
          float alpha = 1.f;
          if (rescale) {
            alpha = ex2(m - m_new);
            m = m_new;
          }
          const float m_use = (m == -INFINITY) ? 0.f : m;
          // pairs of columns through the paired fp32 instructions: s * c - m
          // and the running pair of partial sums take one issue slot per pair
          const uint64_t c2 = f2_make(c, c), nm2 = f2_make(-m_use, -m_use);
          uint64_t l2 = f2_make(0.f, 0.f);
          uint32_t pk[32];  // bf16 pairs; FP8: e4m3 quads in pk[0..15]
          float pq0 = 0.f, pq1 = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float x0, x1;
            f2_split(f2_fma(f2_make(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])),
                            c2, nm2),
                     x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            l2 = f2_add(l2, f2_make(p0, p1));
            if constexpr (kFp8) {
              // the scale keeps small probabilities above e4m3's subnormal range
              if (i & 1)
                pk[i >> 1] = pack_e4m3x4(pq0, pq1, p0 * kFp8PScale, p1 * kFp8PScale);
              else
                pq0 = p0 * kFp8PScale, pq1 = p1 * kFp8PScale;
            } else {
              pk[i] = pack_bf16x2(p0, p1);
            }
          }
          float l0, l1;
          f2_split(l2, l0, l1);
          l = l * alpha + (l0 + l1);
          // P_j over the S columns this warpgroup has just read (the other
          // warpgroup may still be reading its own): keys [64w, 64w+64) as
          // bf16 pairs in columns [64w, 64w+32) (the A operand of P V)
          if constexpr (kFp8) {
            // ... or as e4m3 quads in columns [64w, 64w+16)
            tmem_st16(tmem + lane_base + 128 * g + 64 * w,
                      *reinterpret_cast<const uint32_t(*)[16]>(pk));
          } else {
            tmem_st32p(tmem + lane_base + 128 * g + 64 * w, pk);
          }
          if (j >= 1 && __any_sync(0xffffffffu, rescale)) {
            // O_w is rescaled once the products of step j-1 have completed
            ok = __all_sync(0xffffffffu, mbar_wait(bar.pv_done((Jj - 1) % kSRegions),
                                                   ((Jj - 1) / kSRegions) & 1, p.status));
            if (ok) {
              tc_fence_after();
#pragma unroll
              for (int ch = 0; ch < D / 32; ++ch)
                tmem_scale_cols<32>(tmem + lane_base + col_o(w) + 32 * ch, alpha);
            } else if (lane == 0) {
              record_failure(p.status, kStatusTimeout, kSiteFwdO);
            }
          }
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.p_full(g));
        if (j == 0 && pend) {
          finish(pend_m, pend_l, pend_r, pend_bh, 1, pend_jl);
          pend = false;
        }
      }
      if (ntiles > 0) {
        // this item's epilogue runs inside the next item's first step
        pend = true;
        pend_m = m;
        pend_l = l;
        pend_r = r;
        pend_bh = bh;
        pend_jl = J + ntiles - 1;
      } else {
        finish(-INFINITY, 0.f, r, bh, 0, 0);  // no key: O = 0, LSE = -inf
      }
      J += ntiles;
    }
    if (pend) finish(pend_m, pend_l, pend_r, pend_bh, 1, pend_jl);
    if (tid == 0) bulk_wait_read_all();  // the last O stores, before the CTA exits
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
                         const CUtensorMap& mo, const FwdParams& p, cudaStream_t s) {
  using L = FwdLayout<D, kFp8>;
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D, kShortLast, kFp8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (at most one per work item); the item counter
  // starts at zero
  const int items = p.B * p.H * p.Tr;
  const unsigned grid = static_cast<unsigned>(items < p.num_sms ? items : p.num_sms);
  e = cudaMemsetAsync(p.sched, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  fwd_kernel<D, kShortLast, kFp8><<<grid, kThreads, L::kBytes, s>>>(mq, mk, mv, mo, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int d, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       const CUtensorMap& mo, const FwdParams& p, cudaStream_t s) {
  const bool short_last = p.N % kTile != 0;
  if (d == 64)
    return short_last ? launch_fwd_t<64, true>(mq, mk, mv, mo, p, s)
                      : launch_fwd_t<64, false>(mq, mk, mv, mo, p, s);
  return short_last ? launch_fwd_t<128, true>(mq, mk, mv, mo, p, s)
                    : launch_fwd_t<128, false>(mq, mk, mv, mo, p, s);
}

cudaError_t launch_fwd_fp8(const CUtensorMap& mq8, const CUtensorMap& mk8,
                           const CUtensorMap& mvt8, const CUtensorMap& mo, const FwdParams& p,
                           cudaStream_t s) {
  return p.N % kTile != 0 ? launch_fwd_t<128, true, true>(mq8, mk8, mvt8, mo, p, s)
                          : launch_fwd_t<128, false, true>(mq8, mk8, mvt8, mo, p, s);
}

}  // namespace fm
