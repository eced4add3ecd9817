// Host side of the C ABI declared in include/flashmask.h: argument checks,
// workspace layout, TMA descriptors and kernel launches. Nothing here
// allocates device memory.
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "flashmask.h"

namespace {

using fm::kTile;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Blocks per sequence and the per-head row count of the padded workspace arrays
// (the last block of a sequence whose length is not a multiple of 128 is short).
int blocks_of(int N) { return (N + kTile - 1) / kTile; }
int padded(int N) { return blocks_of(N) * kTile; }

bool shape_ok(int B, int H, int Hm, int N, int d) {
  if (B <= 0 || H <= 0 || Hm <= 0 || N <= 0) return false;
  // the classification keeps per-query-block arrays of one key block in shared
  // memory (2 * 4 * (Tr + 1) bytes)
  if (N > FM_MAX_SEQLEN) return false;
  if (d != 64 && d != 128) return false;
  if (H % Hm != 0) return false;
  const long long rows = static_cast<long long>(B) * H * padded(N);
  if (rows >= (1LL << 31)) return false;
  return true;
}

fm_ws_layout make_layout(int B, int H, int Hm, int N, int d, int for_bwd) {
  fm_ws_layout L;
  std::memset(&L, 0, sizeof(L));
  const size_t Tr = blocks_of(N), Tc = Tr, BHm = static_cast<size_t>(B) * Hm;
  const size_t BHN = static_cast<size_t>(B) * H * padded(N);  // padded rows per head
  size_t off = 0;
  L.status = off;
  off = align_up(off + 16, 256);
  L.minmax = off;
  off = align_up(off + BHm * Tc * 8 * 4, 256);
  L.labels = off;
  off = align_up(off + BHm * Tr * Tc, 256);
  L.labels_t = off;
  off = align_up(off + BHm * Tc * Tr, 256);
  L.row_count = off;
  off = align_up(off + BHm * Tr * 4, 256);
  L.row_list = off;
  off = align_up(off + BHm * Tr * Tc * 4, 256);
  L.row_order = off;
  off = align_up(off + BHm * Tr * 4, 256);
  L.col_count = off;
  off = align_up(off + BHm * Tc * 4, 256);
  L.col_list = off;
  off = align_up(off + BHm * Tc * Tr * 4, 256);
  L.col_order = off;
  off = align_up(off + BHm * Tc * 4, 256);
  if (for_bwd) {
    L.lse2 = off;
    off = align_up(off + BHN * 4, 256);
    L.delta = off;
    off = align_up(off + BHN * 4, 256);
    L.dq_accum = off;
    off = align_up(off + BHN * d * 4, 256);
    const size_t E = fm::split_blocks(static_cast<int>(Tc));
    L.kv_part = off;
    off = align_up(off + static_cast<size_t>(B) * H * E * (fm::kSplitParts - 1) * 2 * kTile * d * 4,
                   256);
    L.kv_sync = off;
    off = align_up(off + static_cast<size_t>(B) * H * E * fm::kSyncWords * 4, 256);
  }
  L.total = off;
  return L;
}

// Nonzero tag of a backward workspace layout, left in the fourth status word by
// a forward that zeroed the dQ accumulator of a workspace with this layout
// (FNV-1a over the shape; bit 0 set so it is never 0).
int32_t dq_zero_tag(int B, int H, int Hm, int N, int d) {
  uint32_t h = 2166136261u;
  for (int v : {B, H, Hm, N, d}) h = (h ^ static_cast<uint32_t>(v)) * 16777619u;
  return static_cast<int32_t>(h | 1u);
}

// The backward adds split CTAs only from this many key blocks per head on:
// they cost an SM slot each even when no key block needs them (about 1% of
// the backward at 256 key blocks), and only long sequences make key blocks
// long enough to be worth splitting. FM_BWD_SPLIT_MIN_BLOCKS overrides it.
int split_min_blocks() {
  const char* e = std::getenv("FM_BWD_SPLIT_MIN_BLOCKS");
  return e != nullptr ? std::atoi(e) : 512;
}

fm::ClassifyTables tables(const fm_ws_layout& L, void* ws) {
  char* w = static_cast<char*>(ws);
  fm::ClassifyTables t;
  t.minmax = reinterpret_cast<int32_t*>(w + L.minmax);
  t.labels = reinterpret_cast<uint8_t*>(w + L.labels);
  t.labels_t = reinterpret_cast<uint8_t*>(w + L.labels_t);
  t.row_count = reinterpret_cast<int32_t*>(w + L.row_count);
  t.row_list = reinterpret_cast<int32_t*>(w + L.row_list);
  t.row_order = reinterpret_cast<int32_t*>(w + L.row_order);
  t.col_count = reinterpret_cast<int32_t*>(w + L.col_count);
  t.col_list = reinterpret_cast<int32_t*>(w + L.col_list);
  t.col_order = reinterpret_cast<int32_t*>(w + L.col_order);
  return t;
}

bool mask_ok(const fm_mask* m) {
  if (!m || !m->lts || !m->lte) return false;
  if ((m->uts == nullptr) != (m->ute == nullptr)) return false;
  return true;
}

fm::MaskDev mask_dev(const fm_mask* m) {
  fm::MaskDev d;
  d.lts = m->lts;
  d.lte = m->lte;
  d.uts = m->uts;
  d.ute = m->ute;
  d.Hm = m->Hm;
  d.causal = m->causal ? 1 : 0;
  return d;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SMs of the current device (the persistent forward's grid), looked up once
// per device; threads that race on the first lookup store the same value.
int sm_count() {
  constexpr int kMaxDev = 256;
  static std::atomic<int> cached[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Tensor map over the [rows, d] fp32 dQ accumulator with 128-row x 32-column
// boxes (128 bytes wide) and 128-byte swizzle, used for TMA reduce-add.
bool make_map_f32(CUtensorMap* m, const void* base, long long rows, int d) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 4};
  cuuint32_t box[2] = {32, static_cast<cuuint32_t>(kTile)};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map over [heads, N, cols] (elements of `esize` bytes: bf16 or e4m3)
// with boxes of one head, 128 rows and 128 bytes per row, 128-byte swizzle.
// Each head is its own 2-D slab: a box that runs past row N of a head reads
// zeros, never the next head's rows.
bool make_map3(CUtensorMap* m, const void* base, long long heads, int N, int cols, int esize) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * esize,
                           static_cast<cuuint64_t>(N) * cols * esize};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esize), static_cast<cuuint32_t>(kTile), 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
            const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map over a [rows, cols] byte matrix (e4m3) with 128 x 128-byte boxes
// and 128-byte swizzle.
bool make_map_u8(CUtensorMap* m, const void* base, long long rows, long long cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
  cuuint32_t box[2] = {128, static_cast<cuuint32_t>(kTile)};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Workspace of the FP8 forward: the forward's classification layout, then the
// e4m3 operands and their scales.
struct Fp8Layout {
  fm_ws_layout base;
  size_t q8, k8, vt8, qscale, kscale, vscale, vamax, total;
};

Fp8Layout make_fp8_layout(int B, int H, int Hm, int N) {
  Fp8Layout F;
  F.base = make_layout(B, H, Hm, N, 128, 0);
  const size_t BH = static_cast<size_t>(B) * H, Tr = blocks_of(N);
  size_t off = F.base.total;
  F.q8 = off;
  off = align_up(off + BH * N * 128, 256);
  F.k8 = off;
  off = align_up(off + BH * N * 128, 256);
  F.vt8 = off;
  off = align_up(off + BH * 128 * padded(N), 256);
  F.qscale = off;
  off = align_up(off + BH * Tr * 4, 256);
  F.kscale = off;
  off = align_up(off + BH * Tr * 4, 256);
  F.vscale = off;
  off = align_up(off + BH * 4, 256);
  F.vamax = off;
  off = align_up(off + BH * 4, 256);
  F.total = off;
  return F;
}

fm_status check_ws(void* ws, size_t ws_bytes, const fm_ws_layout& L) {
  if (!ws) return FM_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return FM_ERR_WORKSPACE;
  if (ws_bytes < L.total) return FM_ERR_WORKSPACE;
  return FM_OK;
}

}  // namespace

extern "C" {

size_t flashmask_workspace_bytes(int B, int H, int Hm, int N, int d, int for_bwd) {
  if (!shape_ok(B, H, Hm, N, d)) return 0;
  return make_layout(B, H, Hm, N, d, for_bwd).total;
}

fm_status flashmask_workspace_layout(int B, int H, int Hm, int N, int d, int for_bwd,
                                     fm_ws_layout* out) {
  if (!out) return FM_ERR_INVALID_ARG;
  if (!shape_ok(B, H, Hm, N, d)) return FM_ERR_UNSUPPORTED;
  *out = make_layout(B, H, Hm, N, d, for_bwd);
  return FM_OK;
}

fm_status flashmask_classify(const fm_mask* mask, int B, int N, void* ws, size_t ws_bytes,
                             void* stream) {
  if (!mask_ok(mask)) return FM_ERR_INVALID_ARG;
  const int Hm = mask->Hm;
  // the classification part of the layout depends on (B, Hm, N) only
  if (!shape_ok(B, Hm, Hm, N, 64)) return FM_ERR_UNSUPPORTED;
  const fm_ws_layout L = make_layout(B, Hm, Hm, N, 64, 0);
  const fm_status ws_st = check_ws(ws, ws_bytes, L);
  if (ws_st != FM_OK) return ws_st;
  cudaError_t e = fm::launch_classify(mask_dev(mask), B, N, tables(L, ws),
                                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}

fm_status flashmask_fwd(const void* q, const void* k, const void* v, const fm_mask* mask, int B,
                        int H, int N, int d, float scale, void* o, float* lse, void* ws,
                        size_t ws_bytes, int ws_classified, void* stream) {
  if (!q || !k || !v || !o || !lse || !mask_ok(mask)) return FM_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FM_ERR_INVALID_ARG;
  if (!shape_ok(B, H, mask->Hm, N, d)) return FM_ERR_UNSUPPORTED;
  const fm_ws_layout L = make_layout(B, H, mask->Hm, N, d, 0);
  const fm_status ws_st = check_ws(ws, ws_bytes, L);
  if (ws_st != FM_OK) return ws_st;
  const long long heads = static_cast<long long>(B) * H;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map3(&mq, q, heads, N, d, 2) || !make_map3(&mk, k, heads, N, d, 2) ||
      !make_map3(&mv, v, heads, N, d, 2) || !make_map3(&mo, o, heads, N, d, 2))
    return FM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const fm::ClassifyTables t = tables(L, ws);
  if (!ws_classified) {
    if (fm::launch_classify(mask_dev(mask), B, N, t, s) != cudaSuccess) return FM_ERR_CUDA;
  }
  fm::FwdParams p;
  p.mask = mask_dev(mask);
  p.B = B;
  p.H = H;
  p.N = N;
  p.Tr = blocks_of(N);
  p.Tc = blocks_of(N);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.qscale = p.kscale = p.vscale = nullptr;
  p.row_count = t.row_count;
  p.row_list = t.row_list;
  p.row_order = t.row_order;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.status = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + L.status);
  p.sched = p.status + 2;  // third word of the 16-byte status region
  p.num_sms = sm_count();
  if (p.num_sms <= 0) return FM_ERR_CUDA;
  // a workspace large enough for the backward gets its dQ accumulator zeroed
  // here, where HBM is mostly idle, instead of in the backward preprocess
  const fm_ws_layout Lb = make_layout(B, H, mask->Hm, N, d, 1);
  p.dq_zero = ws_bytes >= Lb.total
                  ? reinterpret_cast<float*>(static_cast<char*>(ws) + Lb.dq_accum)
                  : nullptr;
  p.dq_tag = dq_zero_tag(B, H, mask->Hm, N, d);
  return fm::launch_fwd(d, mq, mk, mv, mo, p, s) == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}

size_t flashmask_fwd_fp8_workspace_bytes(int B, int H, int Hm, int N) {
  if (!shape_ok(B, H, Hm, N, 128)) return 0;
  return make_fp8_layout(B, H, Hm, N).total;
}

fm_status flashmask_fwd_fp8_layout(int B, int H, int Hm, int N, fm_fp8_layout* out) {
  if (!out) return FM_ERR_INVALID_ARG;
  if (!shape_ok(B, H, Hm, N, 128)) return FM_ERR_UNSUPPORTED;
  const Fp8Layout F = make_fp8_layout(B, H, Hm, N);
  out->fwd_total = F.base.total;
  out->q8 = F.q8;
  out->k8 = F.k8;
  out->vt8 = F.vt8;
  out->qscale = F.qscale;
  out->kscale = F.kscale;
  out->vscale = F.vscale;
  out->total = F.total;
  return FM_OK;
}

fm_status flashmask_fwd_fp8(const void* q, const void* k, const void* v, const fm_mask* mask,
                            int B, int H, int N, int d, float scale, void* o, float* lse, void* ws,
                            size_t ws_bytes, int ws_classified, void* stream) {
  if (!q || !k || !v || !o || !lse || !mask_ok(mask)) return FM_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FM_ERR_INVALID_ARG;
  if (d != 128 || !shape_ok(B, H, mask->Hm, N, d)) return FM_ERR_UNSUPPORTED;
  const Fp8Layout F = make_fp8_layout(B, H, mask->Hm, N);
  fm_ws_layout whole = F.base;
  whole.total = F.total;
  const fm_status ws_st = check_ws(ws, ws_bytes, whole);
  if (ws_st != FM_OK) return ws_st;
  char* w = static_cast<char*>(ws);
  fm::Fp8Operands f;
  f.q8 = reinterpret_cast<uint8_t*>(w + F.q8);
  f.k8 = reinterpret_cast<uint8_t*>(w + F.k8);
  f.vt8 = reinterpret_cast<uint8_t*>(w + F.vt8);
  f.qscale = reinterpret_cast<float*>(w + F.qscale);
  f.kscale = reinterpret_cast<float*>(w + F.kscale);
  f.vscale = reinterpret_cast<float*>(w + F.vscale);
  f.vamax = reinterpret_cast<unsigned int*>(w + F.vamax);
  const int BH = B * H;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map3(&mq, f.q8, BH, N, 128, 1) || !make_map3(&mk, f.k8, BH, N, 128, 1) ||
      !make_map_u8(&mv, f.vt8, static_cast<long long>(BH) * 128, padded(N)) ||
      !make_map3(&mo, o, BH, N, 128, 2))
    return FM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const fm::ClassifyTables t = tables(F.base, ws);
  if (!ws_classified) {
    if (fm::launch_classify(mask_dev(mask), B, N, t, s) != cudaSuccess) return FM_ERR_CUDA;
  }
  if (fm::launch_quant_fp8(static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k),
                           static_cast<const uint16_t*>(v), BH, N, f, s) != cudaSuccess)
    return FM_ERR_CUDA;
  fm::FwdParams p;
  p.mask = mask_dev(mask);
  p.B = B;
  p.H = H;
  p.N = N;
  p.Tr = blocks_of(N);
  p.Tc = blocks_of(N);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.qscale = f.qscale;
  p.kscale = f.kscale;
  p.vscale = f.vscale;
  p.row_count = t.row_count;
  p.row_list = t.row_list;
  p.row_order = t.row_order;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.status = reinterpret_cast<int32_t*>(w + F.base.status);
  p.sched = p.status + 2;
  p.num_sms = sm_count();
  if (p.num_sms <= 0) return FM_ERR_CUDA;
  // the FP8 operands overlap a backward layout's dQ accumulator: the kernel
  // clears the tag, so a later backward preprocess zeroes it again
  p.dq_zero = nullptr;
  p.dq_tag = 0;
  return fm::launch_fwd_fp8(mq, mk, mv, mo, p, s) == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}

fm_status flashmask_bwd_preprocess(const void* o, const float* lse, const void* dout, int B, int H,
                                   int Hm, int N, int d, void* ws, size_t ws_bytes, void* stream) {
  if (!o || !lse || !dout) return FM_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(dout) || !aligned16(lse)) return FM_ERR_INVALID_ARG;
  if (!shape_ok(B, H, Hm, N, d)) return FM_ERR_UNSUPPORTED;
  const fm_ws_layout L = make_layout(B, H, Hm, N, d, 1);
  const fm_status ws_st = check_ws(ws, ws_bytes, L);
  if (ws_st != FM_OK) return ws_st;
  char* w = static_cast<char*>(ws);
  return fm::launch_bwd_pre(d, static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout),
                            lse, reinterpret_cast<float*>(w + L.delta),
                            reinterpret_cast<float*>(w + L.lse2),
                            reinterpret_cast<float*>(w + L.dq_accum),
                            static_cast<long long>(B) * H, N, padded(N),
                            reinterpret_cast<const int32_t*>(w + L.status) + 3,
                            dq_zero_tag(B, H, Hm, N, d), reinterpret_cast<int32_t*>(w + L.kv_sync),
                            fm::split_blocks(blocks_of(N)), static_cast<cudaStream_t>(stream)) ==
                     cudaSuccess
             ? FM_OK
             : FM_ERR_CUDA;
}

fm_status flashmask_bwd_main(const void* q, const void* k, const void* v, const void* dout,
                             const fm_mask* mask, int B, int H, int N, int d, float scale,
                             void* dk, void* dv, void* ws, size_t ws_bytes, void* stream) {
  if (!q || !k || !v || !dout || !dk || !dv || !mask_ok(mask)) return FM_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(dk) ||
      !aligned16(dv))
    return FM_ERR_INVALID_ARG;
  if (!shape_ok(B, H, mask->Hm, N, d)) return FM_ERR_UNSUPPORTED;
  const fm_ws_layout L = make_layout(B, H, mask->Hm, N, d, 1);
  const fm_status ws_st = check_ws(ws, ws_bytes, L);
  if (ws_st != FM_OK) return ws_st;
  const long long heads = static_cast<long long>(B) * H;
  const long long rows_pad = heads * padded(N);
  char* w = static_cast<char*>(ws);
  float* dq_accum = reinterpret_cast<float*>(w + L.dq_accum);
  CUtensorMap mq, mk, mv, mdo, mdq;
  if (!make_map3(&mq, q, heads, N, d, 2) || !make_map3(&mk, k, heads, N, d, 2) ||
      !make_map3(&mv, v, heads, N, d, 2) || !make_map3(&mdo, dout, heads, N, d, 2) ||
      !make_map_f32(&mdq, dq_accum, rows_pad, d))
    return FM_ERR_CUDA;
  const fm::ClassifyTables t = tables(L, ws);
  fm::BwdParams p;
  p.mask = mask_dev(mask);
  p.B = B;
  p.H = H;
  p.N = N;
  p.Npad = padded(N);
  p.Tr = blocks_of(N);
  p.Tc = blocks_of(N);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.col_count = t.col_count;
  p.col_list = t.col_list;
  p.col_order = t.col_order;
  p.lse2 = reinterpret_cast<float*>(w + L.lse2);
  p.delta = reinterpret_cast<float*>(w + L.delta);
  p.dq_accum = dq_accum;
  p.split_e = p.Tc >= split_min_blocks() ? fm::split_blocks(p.Tc) : 0;
  p.kv_part = reinterpret_cast<float*>(w + L.kv_part);
  p.kv_sync = reinterpret_cast<int32_t*>(w + L.kv_sync);
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.num_sms = sm_count();
  if (p.num_sms <= 0) return FM_ERR_CUDA;
  p.dk = static_cast<uint16_t*>(dk);
  p.dv = static_cast<uint16_t*>(dv);
  p.status = reinterpret_cast<int32_t*>(w + L.status);
  return fm::launch_bwd(d, mq, mk, mv, mdo, mdq, p, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? FM_OK
             : FM_ERR_CUDA;
}

fm_status flashmask_bwd_finalize(int B, int H, int Hm, int N, int d, float scale, void* dq,
                                 void* ws, size_t ws_bytes, void* stream) {
  if (!dq || !aligned16(dq)) return FM_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FM_ERR_INVALID_ARG;
  if (!shape_ok(B, H, Hm, N, d)) return FM_ERR_UNSUPPORTED;
  const fm_ws_layout L = make_layout(B, H, Hm, N, d, 1);
  const fm_status ws_st = check_ws(ws, ws_bytes, L);
  if (ws_st != FM_OK) return ws_st;
  return fm::launch_dq_convert(d, reinterpret_cast<const float*>(static_cast<char*>(ws) + L.dq_accum),
                               scale, static_cast<uint16_t*>(dq), static_cast<long long>(B) * H, N,
                               padded(N), static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FM_OK
             : FM_ERR_CUDA;
}

fm_status flashmask_bwd(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dout, const fm_mask* mask, int B, int H,
                        int N, int d, float scale, void* dq, void* dk, void* dv, void* ws,
                        size_t ws_bytes, int ws_classified, void* stream) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !mask_ok(mask))
    return FM_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(lse))
    return FM_ERR_INVALID_ARG;
  if (!shape_ok(B, H, mask->Hm, N, d)) return FM_ERR_UNSUPPORTED;
  const fm_ws_layout L = make_layout(B, H, mask->Hm, N, d, 1);
  const fm_status ws_st = check_ws(ws, ws_bytes, L);
  if (ws_st != FM_OK) return ws_st;
  if (!ws_classified) {
    if (fm::launch_classify(mask_dev(mask), B, N, tables(L, ws), static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
      return FM_ERR_CUDA;
  }
  fm_status st = flashmask_bwd_preprocess(o, lse, dout, B, H, mask->Hm, N, d, ws, ws_bytes, stream);
  if (st != FM_OK) return st;
  st = flashmask_bwd_main(q, k, v, dout, mask, B, H, N, d, scale, dk, dv, ws, ws_bytes, stream);
  if (st != FM_OK) return st;
  return flashmask_bwd_finalize(B, H, mask->Hm, N, d, scale, dq, ws, ws_bytes, stream);
}

// ---------------------------------------------------------------- no-allocation forward
// Some callers cannot allocate device memory at all: code running inside a
// pre-reserved memory pool or an allocator callback, embedded runtimes that
// forbid cudaMalloc after start-up, or plug-ins handed only their input and
// output buffers. flashmask_fwd_noalloc serves them with a fixed scratch area
// that lives in the library itself instead of a caller-provided workspace.
}  // extern "C"

namespace {

// The scratch area (classification tables and the status word). Every GPU that
// loads the library holds it until the process exits. In host code the name
// only stands for the array; its device address comes from
// cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[kMaxDevices] = {};

fm_status noalloc_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return FM_ERR_CUDA;
    g_noalloc_addr[dev] = ptr;
  }
  *out = g_noalloc_addr[dev];
  return FM_OK;
}

}  // namespace

extern "C" {

fm_status flashmask_fwd_noalloc(const void* q, const void* k, const void* v, const fm_mask* mask,
                                int B, int H, int N, int d, float scale, void* o, float* lse,
                                void* stream) {
  if (!q || !k || !v || !o || !lse || !mask_ok(mask)) return FM_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FM_ERR_INVALID_ARG;
  if (!shape_ok(B, H, mask->Hm, N, d)) return FM_ERR_UNSUPPORTED;
  const fm_ws_layout L = make_layout(B, H, mask->Hm, N, d, 0);
  if (L.total > FM_NOALLOC_SCRATCH_BYTES) return FM_ERR_WORKSPACE;  // beyond the fixed scratch
  void* scratch = nullptr;
  const fm_status st = noalloc_scratch_address(&scratch);
  if (st != FM_OK) return st;
  // the status word must start at zero; the tables are rewritten by the classification
  if (cudaMemsetAsync(static_cast<char*>(scratch) + L.status, 0, 16,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FM_ERR_CUDA;
  return flashmask_fwd(q, k, v, mask, B, H, N, d, scale, o, lse, scratch,
                       FM_NOALLOC_SCRATCH_BYTES, 0, stream);
}

fm_status flashmask_check_status(void* ws, void* stream, int* detail) {
  if (detail) *detail = 0;
  if (!ws) return FM_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return FM_ERR_CUDA;
  int32_t h[2] = {0, 0};
  if (cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FM_ERR_CUDA;
  if (h[0] == 0) return FM_OK;
  if (detail) *detail = h[1];
  if (cudaMemset(ws, 0, sizeof(h)) != cudaSuccess) return FM_ERR_CUDA;
  return FM_ERR_TIMEOUT;
}

const char* flashmask_status_string(fm_status s) {
  switch (s) {
    case FM_OK: return "ok";
    case FM_ERR_INVALID_ARG: return "invalid argument";
    case FM_ERR_UNSUPPORTED: return "unsupported shape";
    case FM_ERR_CUDA: return "CUDA error";
    case FM_ERR_TIMEOUT: return "a kernel wait timed out";
    case FM_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
  }
  return "unknown status";
}

}  // extern "C"
