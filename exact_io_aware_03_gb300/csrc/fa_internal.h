// Internal launch interface between the C ABI (fa_api.cu) and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa.h"

namespace fa {

// Problem description shared by all kernels. q, o, dO, dq are [B][H][Nq][d];
// k, v, dk, dv are [B][Hkv][Nk][d] with H a multiple of Hkv: query head h
// attends key/value head h / (H / Hkv) (Hkv == H: plain multi-head).
//
// Packed variable-length batches (cu_q != nullptr): q, o, dO, dq are
// [H][total_q][d], k, v, dk, dv are [Hkv][total_k][d], LSE is [H][total_q];
// sequence b occupies rows [cu_q[b], cu_q[b+1]) of the queries and
// [cu_k[b], cu_k[b+1]) of the keys, and Nq, Nk hold the largest lengths.
struct Problem {
  int B, H, Nq, Nk, d;
  float scale;   // multiplies Q K^T
  int causal;    // bottom-right causal mask when non-zero
  int Hkv;       // key/value heads
  const int* cu_q = nullptr;   // device int32 [B+1], or nullptr (dense)
  const int* cu_k = nullptr;
  int total_q = 0, total_k = 0;
};

// Where the rows of sequence b, query head h live (see Problem).
struct SeqView {
  int q_off, len_q, k_off, len_k;   // row offsets inside the head's rows, lengths
  int hq, hk;                       // head coordinate of q/o/lse and of k/v rows
  long qrows, krows;                // rows per head coordinate
  bool bad;                         // a length outside [0, Nq] x [0, Nk]
};

__device__ __forceinline__ SeqView seq_view(const Problem& p, int b, int h) {
  SeqView v;
  const int hkv = h / (p.H / p.Hkv);
  if (p.cu_q == nullptr) {
    v.q_off = 0; v.len_q = p.Nq; v.k_off = 0; v.len_k = p.Nk;
    v.hq = b * p.H + h; v.hk = b * p.Hkv + hkv;
    v.qrows = p.Nq; v.krows = p.Nk;
    v.bad = false;
    return v;
  }
  v.q_off = p.cu_q[b];
  v.len_q = p.cu_q[b + 1] - v.q_off;
  v.k_off = p.cu_k[b];
  v.len_k = p.cu_k[b + 1] - v.k_off;
  v.hq = h; v.hk = hkv;
  v.qrows = p.total_q; v.krows = p.total_k;
  v.bad = v.len_q < 0 || v.len_q > p.Nq || v.len_k < 0 || v.len_k > p.Nk || v.q_off < 0 ||
          v.k_off < 0 || (long)v.q_off + v.len_q > p.total_q ||
          (long)v.k_off + v.len_k > p.total_k;
  if (v.bad) { v.len_q = 0; v.len_k = 0; v.q_off = 0; v.k_off = 0; }
  return v;
}

struct FwdF32Args {
  Problem p;
  const float* q;
  const float* k;
  const float* v;
  const float* bias;   // [B][Nk] or nullptr
  float* o;
  float* lse;          // may be nullptr
};

// bf16 tensor-core forward. Tensor maps view each tensor as 3-D
// (d, N, B*H) with a (64, 128, 1) box and 128-byte swizzle.
struct FwdBf16Args {
  Problem p;
  CUtensorMap tm_q, tm_k, tm_v;
  CUtensorMap tm_o;    // output, same view as tm_q (TMA stores)
  const float* bias;   // [B][Nk] or nullptr
  uint16_t* o;         // bf16 [B][H][Nq][d]
  float* lse;
  uint32_t* err;       // device error word
  int head_group;      // heads per CTA-ordering group (set by the launcher)
  int n_split;         // split-KV: number of key ranges (1 = off)
  float* part_o;       // split-KV workspace: fp32 O [n_split][B*H][Nq][d]
  float* part_lse;     // split-KV workspace: LSE [n_split][B*H][Nq]
  // e4m3 forward: per-head max |x| of q [B*H], k and v [B*Hkv] (tm_q, tm_k
  // then view the e4m3 q, k and tm_v the transposed e4m3 v [B*Hkv][d][Nk16])
  const float* amax_q;
  const float* amax_k;
  const float* amax_v;
  // persistent form: the unit counter (set to 0xFFFFFFFF on the launch's
  // stream; it lives in the LSE word of the last unit's first row) and the
  // number of units; nullptr: one unit per CTA
  uint32_t* sched;
  int n_units;
};

// Per-head e4m3 scale: x ~= scale * e4m3(x / scale), scale = max|x| / 448
// (448 = the largest finite e4m3 value), 1 for an all-zero head.
__host__ __device__ inline float fp8_scale(float amax) { return amax > 0.f ? amax / 448.f : 1.f; }

struct BwdBf16Args {
  Problem p;
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  CUtensorMap tm_dqacc;   // fp32 dQ accumulator as (d, Nq, B*H), box (32, 32, 1), 128B swizzle
  CUtensorMap tm_dk, tm_dv, tm_dq;   // outputs, same views as tm_k / tm_q (TMA stores)
  const uint16_t* o;
  const uint16_t* dO;
  const float* lse;
  const float* bias;
  float* D;            // workspace: -scale * rowsum(dO o O), [B*H][nq_pad] (0 in the padding)
  float* lse2;         // workspace: -LSE * log2(e), [B*H][nq_pad] (-inf for fully
                       // masked rows and in the padding)
  float* dq_acc;       // workspace: fp32 dQ accumulator [B][H][Nq][d]
  int* sched;          // workspace: work-item counter of the persistent main kernel
                       // (zeroed by the launcher before each launch)
  uint16_t* dq;
  uint16_t* dk;
  uint16_t* dv;
  uint32_t* err;
  int num_sms;
  int nq_pad;          // Nq rounded up to a multiple of 128
  int head_group;      // dQ kernel: heads per CTA-ordering group (set by its launcher)
};

// Id of the current device's context (unique for the life of the process);
// device-variable addresses cached per device are valid only for this id.
fa_status current_context_id(unsigned long long* id);

cudaError_t launch_fwd_f32(const FwdF32Args& a, cudaStream_t s);
cudaError_t launch_fwd_bf16(const FwdBf16Args& a, cudaStream_t s);
// e4m3 forward (d = 128, dense, no split): amax_* and the e4m3 tensor maps set.
cudaError_t launch_fwd_fp8(const FwdBf16Args& a, cudaStream_t s);
// Per-head max |x| of q [B*H rows_q d], k, v [B*Hkv rows_k d] into amax (zeroed
// by the caller), then q, k -> e4m3 (same layout) and v -> e4m3 transposed
// [B*Hkv][d][nk16] (keys past Nk zero).
struct QuantFp8Args {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  uint8_t* q8;
  uint8_t* k8;
  uint8_t* vt8;
  float* amax_q;   // [B*H]
  float* amax_k;   // [B*Hkv]
  float* amax_v;   // [B*Hkv]
  int heads_q, heads_kv, Nq, Nk, nk16, d;
};
cudaError_t launch_quant_fp8(const QuantFp8Args& a, cudaStream_t s);
// Backward stages (bit mask): D / base-2 LSE / zeroed dQ accumulator; the
// tensor-core main loop; the dQ conversion. BWD_DET selects the deterministic
// variant of the main loop (dK, dV only; no accumulator is zeroed when dq_acc
// is null) and BWD_DQ the query-outer dQ kernel that completes it.
enum : unsigned { BWD_PRE = 1u, BWD_MAIN = 2u, BWD_POST = 4u, BWD_DET = 8u, BWD_DQ = 16u };
cudaError_t launch_bwd_bf16(const BwdBf16Args& a, cudaStream_t s, unsigned stages);
cudaError_t launch_bwd_dq(const BwdBf16Args& a, cudaStream_t s);

}  // namespace fa
