/*
 * flashmask.h: C ABI of the column-wise-masked exact attention library
 * (libflashmask.so, sm_103a).
 *
 * What it computes ("FlashMask: Efficient and Rich Mask Extension of
 * FlashAttention", abstract; "FlashMask-3: ... Mask-Aware Distributed
 * Attention", abstract): exact scaled-dot-product attention, forward and
 * backward, under a mask stored column-wise as four int32 query-axis boundary
 * vectors per key column. For key column j, query row i is MASKED when
 *
 *     (causal && j > i) || (LTS[j] <= i < LTE[j]) || (UTS[j] <= i < UTE[j])
 *
 * Intervals are half-open; an interval whose start >= end masks nothing, and
 * bounds outside [0, N] act as if clamped to [0, N]. Over visible entries:
 *
 *     S = scale * Q K^T,  P = softmax_rows(S),  O = P V,  LSE = rowwise ln sum exp(S)
 *
 * A query row with no visible key gets O = 0 and LSE = -inf; it contributes
 * nothing to any gradient. The backward returns dQ, dK, dV for an upstream
 * gradient dO (the FlashAttention recomputation scheme: P is rebuilt from Q, K
 * and LSE; D = rowsum(dO * O)).
 *
 * Layouts (all row-major, contiguous, device memory owned by the caller):
 *   Q, K, V, O, dO, dQ, dK, dV : bf16  [B, H, N, d]
 *   LSE                        : fp32  [B, H, N]     (natural log)
 *   LTS, LTE, UTS, UTE         : int32 [B, Hm, N]    (head h reads mask head h / (H / Hm))
 * Supported shapes: d in {64, 128}; 1 <= N <= FM_MAX_SEQLEN (the last 128-row
 * block of a sequence whose length is not a multiple of 128 is short; its
 * missing rows and keys take no part); H % Hm == 0; B * H * Npad < 2^31 with
 * Npad = N rounded up to a multiple of 128. Other shapes return
 * FM_ERR_UNSUPPORTED.
 *
 * Workspace: the library never allocates. The caller passes one device buffer
 * of at least flashmask_workspace_bytes(...) bytes, aligned to 256 bytes. It
 * holds the tile classification (written by flashmask_classify), the backward's
 * fp32 scratch and a device status word. One workspace must not be used by two
 * calls that may run at the same time.
 *
 * The status word (the first 16 bytes of the workspace) must be zero before
 * the workspace is first passed to a call that launches kernels: allocate the
 * workspace zeroed (cudaMemset, torch.zeros) or call flashmask_check_status()
 * on it once, which reads the word and clears it. The calls themselves do not
 * clear it (a failure recorded by one call stays visible until it is checked),
 * and a kernel that finds it nonzero gives up every wait that is not already
 * satisfied, leaving its outputs undefined; flashmask_check_status() then
 * reports FM_ERR_TIMEOUT.
 *
 * Streams and errors: every call validates its arguments on the host and
 * returns an error WITHOUT launching anything if they are bad. Otherwise it
 * enqueues kernels on `stream` (a cudaStream_t, NULL for the legacy default
 * stream) and returns FM_OK without synchronising. Every wait inside a kernel
 * is bounded in time; a kernel whose wait gives up records the failure in the
 * workspace status word and exits. flashmask_check_status() reads and clears
 * that word.
 */
#ifndef FLASHMASK_H
#define FLASHMASK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FM_OK = 0,
  FM_ERR_INVALID_ARG = 1,  /* null pointer, negative size, scale not finite, ...   */
  FM_ERR_UNSUPPORTED = 2,  /* d not in {64,128}, N < 1, H % Hm != 0, ...           */
  FM_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed          */
  FM_ERR_TIMEOUT = 4,      /* a kernel wait gave up (see flashmask_check_status)   */
  FM_ERR_WORKSPACE = 5     /* workspace null, misaligned or smaller than required  */
} fm_status;

/* Tile edge (rows and columns) of the classification. */
#define FM_TILE 128

/* Longest supported sequence (2^21 tokens, 16384 blocks of 128). */
#define FM_MAX_SEQLEN 2097152

/* Three-way tile label ("FlashMask" abstract: skip the computation that the
 * mask makes unnecessary). */
#define FM_TILE_NONE 0    /* no entry of the tile is masked: no mask work        */
#define FM_TILE_PARTIAL 1 /* some entries masked: mask applied element by element */
#define FM_TILE_FULL 2    /* every entry masked: the tile is skipped             */

/* The column-wise mask: device pointers to int32 [B, Hm, N] vectors.
 * uts and ute may both be NULL (no upper interval). */
typedef struct {
  const int32_t* lts;
  const int32_t* lte;
  const int32_t* uts;
  const int32_t* ute;
  int Hm;     /* number of mask heads, 1 <= Hm <= H, H % Hm == 0 */
  int causal; /* nonzero: also mask j > i                         */
} fm_mask;

/* Byte offsets of the workspace regions (from the workspace base), for callers
 * that want to read the classification. Regions marked [bwd] exist only when
 * the workspace was sized with for_bwd != 0 (otherwise their offsets are 0).
 *   status    int32[4]                   device status word (0 = OK; must be zero
 *                                        before first use, see above), detail, the
 *                                        forward's work-item counter (reset by each
 *                                        call) and the dQ-zeroed tag (see flashmask_fwd)
 *   minmax    int32  [B,Hm,Tc,8]         per key block: min/max of LTS, LTE, UTS, UTE
 *   labels    uint8  [B,Hm,Tr,Tc]        tile label, query-block major
 *   labels_t  uint8  [B,Hm,Tc,Tr]        tile label, key-block major
 *   row_count int32  [B,Hm,Tr]           non-FULL tiles per query block
 *   row_list  int32  [B,Hm,Tr,Tc]        (key block << 2) | label, ascending
 *   row_order int32  [B,Hm,Tr]           query blocks by descending row_count
 *   col_count int32  [B,Hm,Tc]           non-FULL tiles per key block
 *   col_list  int32  [B,Hm,Tc,Tr]        (query block << 2) | label, ascending
 *   col_order int32  [B,Hm,Tc]           key blocks by descending col_count
 *   lse2      fp32   [B,H,Npad]   [bwd]  LSE * log2(e) (+inf for a fully masked
 *                                       row and for the padding rows n >= N)
 *   delta     fp32   [B,H,Npad]   [bwd]  rowsum(dO * O) (0 on padding rows)
 *   dq_accum  fp32   [B,H,Npad,d] [bwd]  dQ accumulator
 *   kv_part   fp32   [B,H,E,3,2,128,d] [bwd] dV, dK of the parts of a split key
 *                                        block that finish first (see flashmask_bwd)
 *   kv_sync   int32  [B,H,E,8]    [bwd]  arrivals and ready flags per split block
 * with Tr = Tc = ceil(N / 128), Npad = 128 * Tr and E = min(Tc, 16). */
typedef struct {
  size_t status, minmax, labels, labels_t, row_count, row_list, row_order, col_count, col_list,
      col_order, lse2, delta, dq_accum, kv_part, kv_sync, total;
} fm_ws_layout;

/* Workspace size in bytes for the given problem; 0 for an unsupported shape. */
size_t flashmask_workspace_bytes(int B, int H, int Hm, int N, int d, int for_bwd);

/* Fills *out with the region offsets described above. */
fm_status flashmask_workspace_layout(int B, int H, int Hm, int N, int d, int for_bwd,
                                     fm_ws_layout* out);

/* Tile classification pre-pass ("FlashMask" abstract: the column-wise
 * representation lets whole masked blocks be skipped; "FlashMask-3" abstract:
 * the four boundary vectors): reduces the boundary vectors to the
 * per-key-block min/max table, the exact three-way label of every (query
 * block, key block) tile, the compacted non-FULL lists and the
 * descending-work orders, all in the workspace. Reads 16*B*Hm*N bytes.
 * Asynchronous on `stream`. */
fm_status flashmask_classify(const fm_mask* mask, int B, int N, void* ws, size_t ws_bytes,
                             void* stream);

/* Forward ("FlashMask" abstract: exact attention under the column-wise mask,
 * masked tiles skipped; "FlashAttention-3" abstract: the block-wise matmuls
 * overlapped with the softmax): O [B,H,N,d] bf16 and LSE [B,H,N] fp32 from
 * Q, K, V, as defined at the top of this file. `scale`
 * multiplies Q K^T (pass 1/sqrt(d) for standard attention). If
 * ws_classified == 0 the call runs flashmask_classify first; pass 1 to reuse a
 * classification of the same mask already in `ws`. Asynchronous on `stream`.
 * When ws_bytes is at least flashmask_workspace_bytes(..., for_bwd = 1), the
 * forward also zeroes that layout's dQ accumulator (bulk copies issued while
 * the attention runs) and leaves a tag of the shape in the fourth status word;
 * the backward preprocess of the same shape on this workspace then skips its
 * own zeroing pass, and the backward main kernel clears the tag again. */
fm_status flashmask_fwd(const void* q, const void* k, const void* v, const fm_mask* mask, int B,
                        int H, int N, int d, float scale, void* o, float* lse, void* ws,
                        size_t ws_bytes, int ws_classified, void* stream);

/* Backward ("FlashMask" abstract: exact gradients under the same mask, masked
 * tiles skipped; the FlashAttention README's memory savings, read here as P
 * recomputed from Q, K and the saved LSE rather than stored): dQ, dK, dV
 * [B,H,N,d] bf16 from Q, K, V, the forward's O and LSE, and the upstream
 * gradient dO. The workspace must be sized with for_bwd != 0.
 * ws_classified as in flashmask_fwd. Asynchronous on `stream`. The main
 * kernel gives each (head, key block) one CTA, except that with Tc >= 512 key
 * blocks (the environment variable FM_BWD_SPLIT_MIN_BLOCKS changes 512), among
 * the E = min(Tc, 16) longest key blocks of each head one seen by n query
 * blocks is split over min(4, n / 64) CTAs when that is at least two (a
 * global prefix would otherwise keep one SM busy long after the rest); the
 * parts' fp32 dK, dV are added through the workspace. */
fm_status flashmask_bwd(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dout, const fm_mask* mask, int B, int H,
                        int N, int d, float scale, void* dq, void* dk, void* dv, void* ws,
                        size_t ws_bytes, int ws_classified, void* stream);

/* The three stages flashmask_bwd runs after the (optional) classification,
 * exposed so that a caller can schedule or time them separately. They must run
 * in this order on one stream with one workspace:
 *   preprocess: D = rowsum(dO * O), lse2 = LSE * log2(e), dQ accumulator = 0
 *               (HBM-bound; reads O and dO, writes 4*(2+d)*B*H*N bytes; the
 *               accumulator's 4*d*B*H*N bytes are skipped when the preceding
 *               flashmask_fwd on this workspace, of this shape, zeroed it).
 *   main:       dK, dV and the fp32 dQ accumulator over every non-FULL tile
 *               (needs a classification of `mask` and the preprocess output).
 *   finalize:   dQ = bf16(scale * accumulator).
 * Hm is the mask's number of heads (it fixes the workspace layout). */
fm_status flashmask_bwd_preprocess(const void* o, const float* lse, const void* dout, int B, int H,
                                   int Hm, int N, int d, void* ws, size_t ws_bytes, void* stream);
fm_status flashmask_bwd_main(const void* q, const void* k, const void* v, const void* dout,
                             const fm_mask* mask, int B, int H, int N, int d, float scale,
                             void* dk, void* dv, void* ws, size_t ws_bytes, void* stream);
fm_status flashmask_bwd_finalize(int B, int H, int Hm, int N, int d, float scale, void* dq,
                                 void* ws, size_t ws_bytes, void* stream);

/* Forward without any allocation or caller workspace: the paper has no
 * counterpart; this exists for callers that cannot allocate device memory
 * (inside a memory-pool or allocator callback, in runtimes that forbid
 * cudaMalloc once started, or in plug-ins that are handed only their inputs and
 * outputs). Same arguments and results as flashmask_fwd (with ws_classified =
 * 0), but the classification tables live in a fixed scratch array of
 * FM_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads the
 * library holds until the process exits. Shapes whose tables would not fit
 * (about B*Hm*(N/128)^2*10 bytes; N = 131072 with B*Hm = 1 fits) return
 * FM_ERR_WORKSPACE before anything is launched. The call allocates nothing:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 *   - The first call on each device looks up the scratch array's device
 *     address (cudaGetSymbolAddress) with that device current; make that first
 *     call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents; each
 *     call clears the status word it needs at zero and rewrites the tables.
 *     Calls that may overlap on the GPU (other streams, other threads) race
 *     on the array and must be serialised by the caller.
 *   - A device-side wait failure is recorded in the scratch status word, which
 *     callers cannot read; callers that need that report use flashmask_fwd. */
#define FM_NOALLOC_SCRATCH_BYTES (16u << 20)
fm_status flashmask_fwd_noalloc(const void* q, const void* k, const void* v, const fm_mask* mask,
                                int B, int H, int N, int d, float scale, void* o, float* lse,
                                void* stream);

/* FP8 forward ("FlashAttention-3", abstract: block quantization for FP8
 * attention): the same inputs, mask and outputs as flashmask_fwd (bf16 Q, K, V
 * [B,H,N,d], bf16 O and fp32 LSE), with the two products of each tile taken in
 * e4m3 on the tensor cores. d must be 128 (FM_ERR_UNSUPPORTED otherwise).
 * Each call quantises into the workspace: Q and K with one scale per head and
 * 128-row block (scale = absmax / 448, values rounded to nearest even and
 * saturated), V transposed with one scale per head; P is rounded to e4m3 as
 * 28 * P before P V (the running maximum is allowed to lag the true one by
 * at most 4 in log2 units, so 28 * P <= 448). The row sums, the running
 * maximum, LSE and every
 * accumulation stay fp32, so LSE carries only the error of the quantised
 * scores. Results differ from flashmask_fwd by the e4m3 rounding (3 mantissa
 * bits, relative step 2^-4): on random data O's relative Frobenius error is a
 * few percent, not the bf16 path's 1e-3.
 *   Workspace: flashmask_fwd_fp8_workspace_bytes(B, H, Hm, N) bytes, 256-byte
 *   aligned; its first part is the forward workspace layout (for_bwd = 0) of
 *   flashmask_workspace_layout with d = 128, so ws_classified works as in
 *   flashmask_fwd and flashmask_check_status reads its status word. The rest,
 *   at the byte offsets flashmask_fwd_fp8_layout gives, holds what the call
 *   wrote last (the caller may read it back):
 *     q8, k8   e4m3   [B,H,N,128]     Q / scale_Q, K / scale_K
 *     vt8      e4m3   [B,H,128,Npad]  (V / scale_V)^T, keys >= N zero
 *     qscale   fp32   [B,H,Tr]        scale_Q of each 128-row block
 *     kscale   fp32   [B,H,Tr]        scale_K of each 128-row block
 *     vscale   fp32   [B,H]           scale_V of each head
 *   A scale is absmax / 448 computed in fp32 (1 for an all-zero block) and a
 *   value is e4m3(x * (1 / scale)), both products rounded in fp32. The size
 *   function returns 0, the layout function FM_ERR_UNSUPPORTED, for an
 *   unsupported shape. Asynchronous on `stream`. */
typedef struct {
  size_t fwd_total, q8, k8, vt8, qscale, kscale, vscale, total;
} fm_fp8_layout;
size_t flashmask_fwd_fp8_workspace_bytes(int B, int H, int Hm, int N);
fm_status flashmask_fwd_fp8_layout(int B, int H, int Hm, int N, fm_fp8_layout* out);
fm_status flashmask_fwd_fp8(const void* q, const void* k, const void* v, const fm_mask* mask,
                            int B, int H, int N, int d, float scale, void* o, float* lse, void* ws,
                            size_t ws_bytes, int ws_classified, void* stream);

/* Forward and backward between HOST buffers, for callers whose tensors live in
 * host memory (the pages have no counterpart; the computation is exactly
 * flashmask_classify + flashmask_fwd + flashmask_bwd). The heads are cut into
 * chunks of `chunk_heads` consecutive heads of one batch entry (heads are
 * independent) and three streams overlap the copy of chunk c+1 to the device,
 * the kernels of chunk c and the copy of chunk c-1 back to the host, in three
 * slots carved from the device workspace `dev_ws` (>= the size
 * flashmask_host_workspace_bytes() returns for the same shape and chunk, 256-byte
 * aligned; the function returns 0 for an unsupported shape or chunk).
 *   Host pointers: q, k, v, dout [B,H,N,d] bf16; mask->lts/lte/uts/ute
 *   [B,Hm,N] int32; outputs o, dq, dk, dv [B,H,N,d] bf16 and lse [B,H,N] fp32.
 *   Page-locked host memory (cudaHostAlloc, torch pin_memory) lets the copies
 *   run concurrently with the kernels; pageable memory works but serialises.
 *   chunk_heads must divide H and either divide H / Hm or be a multiple of it
 *   (a chunk reads whole mask heads); otherwise FM_ERR_UNSUPPORTED.
 *   The call orders its work after what is already queued on `stream` and
 *   returns only when every output is in host memory (or with the first error;
 *   a kernel wait that gave up gives FM_ERR_TIMEOUT). It allocates no device
 *   memory; three streams and a few events are created once per device and
 *   kept, and calls on one device are serialised by a lock. */
size_t flashmask_host_workspace_bytes(int B, int H, int Hm, int N, int d, int chunk_heads);
fm_status flashmask_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dout,
                                 const fm_mask* mask, int B, int H, int N, int d, float scale,
                                 void* o, float* lse, void* dq, void* dk, void* dv, void* dev_ws,
                                 size_t ws_bytes, int chunk_heads, void* stream);

/* Per-rank mask localisation for context parallelism ("FlashMask-3: ... Mask-Aware
 * Distributed Attention", abstract: under any multi-chunk context-parallel
 * assignment, per-rank localisation reduces to a zero-communication
 * clip-shift-max on the boundary vectors). For a rank that holds the query rows
 * [row0, row0 + rows) of each sequence and every key, writes the boundary
 * vectors of its local problem: int32 [B, Hm, N] device arrays lts, lte, uts,
 * ute (all four written; caller-owned) in local row coordinates [0, rows),
 * with no causal flag (the local mask is non-causal):
 *   every bound b -> min(max(b - row0, 0), rows)               (clip, shift)
 *   causal: key j's masked rows [0, j) become [0, c), c = clip(j - row0), and
 *   join the upper interval as [0, max(c, end))                 (max)
 * Column j of the local mask then marks exactly the chunk's rows that the
 * global mask marks, whenever that upper interval is empty or starts at a row
 * <= c (true for every causal mask whose upper interval lies above the
 * diagonal). Otherwise the column masks more than it should and *inexact
 * (device int32, may be NULL; set to 1, never cleared) records it. A rank with
 * several chunks calls this once per chunk. Keys are not localised (the local
 * problem is rows x N). Bad arguments (row0 < 0, rows < 1, row0 + rows > N,
 * null pointers) return before any launch. Asynchronous on `stream`. */
fm_status flashmask_localize(const fm_mask* mask, int B, int N, int row0, int rows, int32_t* lts,
                             int32_t* lte, int32_t* uts, int32_t* ute, int32_t* inexact,
                             void* stream);

/* Self-test of the failure path (no counterpart in the pages). Launches `ctas`
 * (1..1024) one-warp CTAs whose mbarrier wait can never complete, bounded the
 * way every wait of the library is: CTA 0 gives up after `limit_ns` (1e6..2e9)
 * of wall time and records site 301 in the workspace status word; the other
 * CTAs use the library's own limit but leave as soon as they see that status,
 * as the CTAs of an attention kernel do when one of their waits fails. No
 * fault, no hang; the context stays usable. Returns FM_OK once queued on
 * `stream`; flashmask_check_status() then returns FM_ERR_TIMEOUT with detail
 * 301. ws: any workspace of >= 16 bytes, 256-byte aligned (only the status
 * word is used). */
fm_status flashmask_selftest_timeout(void* ws, size_t ws_bytes, long long limit_ns, int ctas,
                                     void* stream);

/* Synchronises `stream`, then reads and clears the workspace status word.
 * Returns FM_ERR_TIMEOUT if a kernel wait gave up since the last check,
 * FM_ERR_CUDA if the stream reports an error, FM_OK otherwise. If detail is
 * not NULL it receives the recorded failure site (0 if none). */
fm_status flashmask_check_status(void* ws, void* stream, int* detail);

/* Static description of a status code. */
const char* flashmask_status_string(fm_status s);

#ifdef __cplusplus
}
#endif
#endif /* FLASHMASK_H */
