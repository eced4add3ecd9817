// Host-side launch interface shared by the C ABI and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fm {

constexpr int kTile = 128;

// Device status word layout (int32[4] at the start of the workspace):
//   [0] bit mask of failures (kStatusTimeout, kStatusLayout)
//   [1] first failure site (one of the Site codes below), 0 if none
enum : int { kStatusTimeout = 1, kStatusLayout = 2 };
enum Site : int {
  kSiteNone = 0,
  kSiteFwdQ = 101, kSiteFwdK, kSiteFwdV, kSiteFwdS, kSiteFwdP, kSiteFwdO, kSiteFwdKEmpty,
  kSiteFwdVEmpty, kSiteFwdSmemAlign, kSiteFwdSched,
  kSiteBwdKV = 201, kSiteBwdQ, kSiteBwdQEmpty, kSiteBwdS, kSiteBwdDP, kSiteBwdPT, kSiteBwdDS,
  kSiteBwdDV, kSiteBwdDQ, kSiteBwdDrained, kSiteBwdDone, kSiteBwdSmemAlign, kSiteBwdSplit,
  kSiteSelftest = 301,
};

// Backward load balance: among the split_blocks(Tc) longest key blocks of
// each head, one seen by n query blocks is processed by min(kSplitParts,
// n / kPartTiles) CTAs (consecutive parts of its tile list) when that is at
// least two; the parts add their dK, dV through kv_part.
constexpr int kSplitParts = 4;
constexpr int kPartTiles = 64;
constexpr int kSyncWords = 8;  // per split block: arrivals, ready flags of the parts
__host__ __device__ constexpr int split_blocks(int Tc) { return Tc < 16 ? Tc : 16; }

struct MaskDev {
  const int32_t* lts;
  const int32_t* lte;
  const int32_t* uts;  // may be null (then ute is null too)
  const int32_t* ute;
  int Hm;
  int causal;
};

struct ClassifyTables {
  int32_t* minmax;     // [B,Hm,Tc,8]
  uint8_t* labels;     // [B,Hm,Tr,Tc]
  uint8_t* labels_t;   // [B,Hm,Tc,Tr]
  int32_t* row_count;  // [B,Hm,Tr]
  int32_t* row_list;   // [B,Hm,Tr,Tc]
  int32_t* row_order;  // [B,Hm,Tr]
  int32_t* col_count;  // [B,Hm,Tc]
  int32_t* col_list;   // [B,Hm,Tc,Tr]
  int32_t* col_order;  // [B,Hm,Tc]
};

// FP8 operands of the FP8 forward (in the workspace): Q and K e4m3 [B*H, N, 128]
// with one scale per (head, 128-row block); V transposed, e4m3 [B*H, 128, Npad],
// with one scale per head.
struct Fp8Operands {
  uint8_t* q8;
  uint8_t* k8;
  uint8_t* vt8;
  float* qscale;        // [B*H, Tr]
  float* kscale;        // [B*H, Tr]
  float* vscale;        // [B*H]
  unsigned int* vamax;  // [B*H] scratch
};

struct FwdParams {
  MaskDev mask;
  int B, H, N, Tr, Tc;
  float scale_log2;  // scale * log2(e)
  const float* qscale;  // FP8 forward only: per-block scales of Q, K and per-head scale of V
  const float* kscale;
  const float* vscale;
  const int32_t* row_count;
  const int32_t* row_list;
  const int32_t* row_order;
  uint16_t* o;  // bf16 [B,H,N,d]
  float* lse;   // [B,H,N]
  int32_t* status;
  int32_t* sched;  // work-item counter (zeroed by the launch)
  int num_sms;     // persistent grid size
  // Backward workspace only (else null): the fp32 dQ accumulator [B,H,Tr*128,d],
  // whose rows of each query block the forward zeroes, and the tag it leaves in
  // the fourth status word so that the backward preprocess can skip that pass.
  float* dq_zero;
  int32_t dq_tag;
};

struct BwdParams {
  MaskDev mask;
  int B, H, N, Tr, Tc;
  int Npad;          // rows per head of lse2, delta and dq_accum (Tr * 128)
  float scale;       // applied to dK here and to dQ in the conversion kernel
  float scale_log2;  // scale * log2(e)
  const int32_t* col_count;
  const int32_t* col_list;
  const int32_t* col_order;
  const float* lse2;   // [B,H,Npad]
  const float* delta;  // [B,H,Npad]
  float* dq_accum;     // [B,H,Npad,d]
  // The E = split_blocks(Tc) longest key blocks of each head may be split
  // over up to kSplitParts CTAs; all parts but the last to finish leave their
  // fp32 dV, dK in kv_part (slot = arrival order), the last adds them.
  int split_e;
  float* kv_part;      // [B,H,E,kSplitParts-1,2,128,d]
  int32_t* kv_sync;    // [B,H,E,kSyncWords]: arrivals, then one ready flag per slot
  uint16_t* dk;
  uint16_t* dv;
  const uint16_t* k;  // K and V, for the L2 prefetch of a later CTA's blocks
  const uint16_t* v;
  int num_sms;        // CTAs resident at once (one per SM)
  int32_t* status;
};

cudaError_t launch_classify(const MaskDev& m, int B, int N, const ClassifyTables& t,
                            cudaStream_t s);
cudaError_t launch_fwd(int d, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       const CUtensorMap& mo, const FwdParams& p, cudaStream_t s);
cudaError_t launch_fwd_fp8(const CUtensorMap& mq8, const CUtensorMap& mk8,
                           const CUtensorMap& mvt8, const CUtensorMap& mo, const FwdParams& p,
                           cudaStream_t s);
cudaError_t launch_quant_fp8(const uint16_t* q, const uint16_t* k, const uint16_t* v, int BH,
                             int N, const Fp8Operands& f, cudaStream_t s);
cudaError_t launch_bwd_pre(int d, const uint16_t* o, const uint16_t* dout, const float* lse,
                           float* delta, float* lse2, float* dq_accum, long long heads, int N,
                           int Npad, const int32_t* zero_tag_word, int32_t zero_tag,
                           int32_t* kv_sync, int split_e, cudaStream_t s);
cudaError_t launch_bwd(int d, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       const CUtensorMap& mdo, const CUtensorMap& mdq, const BwdParams& p,
                       cudaStream_t s);
cudaError_t launch_dq_convert(int d, const float* dq_accum, float scale, uint16_t* dq,
                              long long heads, int N, int Npad, cudaStream_t s);

}  // namespace fm
