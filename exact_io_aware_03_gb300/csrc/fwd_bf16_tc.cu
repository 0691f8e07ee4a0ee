// bf16 forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Dataflow (query-tile outer, key/value tiles streamed: the order of
// "FlashAttention, Explained", §20, with the online-softmax merge of
// "Understanding FlashAttention Pt 1", §2.4):
//
//   one CTA = two 128-row query tiles Q0, Q1 of one (b, h), kept in shared
//   memory; K_j / V_j tiles of 128 keys stream through an NS-stage ring.
//   For each key tile j and each query tile t:
//     S_t   = Q_t K_j^T              tcgen05.mma, fp32 accumulator in TMEM
//     P_t   = exp2(S_t*c - m_t)      softmax warps: TMEM -> registers -> TMEM
//                                    (P overwrites S in place as packed bf16)
//     O_t  += P_t V_j                tcgen05.mma with A read from TMEM
//   and after the last tile O = O_t / l_t, LSE = ln 2 * (m_t + log2 l_t).
//
// Warp roles (320 threads, one CTA per SM):
//   warps 0-3   softmax for Q0 (thread = query row = TMEM lane)
//   warps 4-7   softmax for Q1
//   warp  8     TMA producer (one lane)
//   warp  9     TMEM allocator + MMA issuer (one lane)
// The MMA order S0(j) S1(j) | PV0(j) S0(j+1) | PV1(j) S1(j+1) | ... lets the
// tensor core work on one query tile while the softmax warps of the other
// tile exponentiate (two tiles in ping-pong).
//
// TMEM (512 columns): S0/P0 [0,128), S1/P1 [128,256), O0 [256,256+D),
// O1 [256+D, 256+2D).
//
// Softmax details:
//  - exponentials in base 2 with scale*log2(e) folded in ("flash-attention",
//    Part VI);
//  - the running max is only moved when the new tile's max exceeds it by more
//    than kRescaleLog2 (8, i.e. a factor 256): otherwise P is formed against the
//    stale max, which keeps every p <= 2^8 and the result exact, and saves the
//    rescale of O in TMEM. The rescale of O, when needed, is done by the
//    softmax warps themselves after the previous PV product has completed;
//  - causal tiles wholly above the bottom-right diagonal are skipped, only
//    tiles that cross it (or the ragged last key tile) are masked element by
//    element ("Understanding FlashAttention Pt 1", §3.5);
//  - key tiles outside the first/last key with a finite bias are skipped
//    (they contribute exactly zero);
//  - a row with no visible key keeps m = -inf and l = 0 and is written as
//    O = 0, LSE = -inf.
#include <algorithm>
#include <cmath>
#include <cstdint>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kBM = 128;       // rows per query tile (= TMEM lanes)
constexpr int kBN = 128;       // keys per key tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;

// FP8: q, k are e4m3 [rows][d] and v is e4m3 transposed, [d][keys] (every
// operand K-major), with per-head scales; d = 128 only (one 128-byte row).
template <int D, bool FP8>
struct FwdCfg {
  static constexpr int EB = FP8 ? 1 : 2;                   // element bytes of q, k, v
  static constexpr int NS = FP8 ? 3 : ((D == 128) ? 2 : 4);   // K/V ring stages
  static constexpr int TILE = kBM * D * EB;                // bytes of one q/k/v tile
  static constexpr int SUB = kBM * 128;                    // bytes of one 128-byte-wide box
  static constexpr int NBOX = D * EB / 128;                // boxes per tile
  static constexpr int OTILE = kBM * D * 2;                // bf16 O tile (epilogue staging)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = 2 * TILE;
  static constexpr int OFF_V = OFF_K + NS * TILE;
  // O staging: the Q buffers (bf16), or a buffer of its own (FP8 tiles are smaller)
  static constexpr int OFF_OST = FP8 ? OFF_V + NS * TILE : OFF_Q;
  static constexpr int OFF_MISC = FP8 ? OFF_OST + 2 * OTILE : OFF_V + NS * TILE;
  // warp roles: softmax warps 0-7, then the TMA producer and the MMA issuer
  static constexpr int W_TMA = 8, W_MMA = 9;
  static constexpr int NT = 320;
  // misc: bias buffers [2 tiles][2 bufs][128] floats, then barriers
  static constexpr int OFF_BIAS = OFF_MISC;
  static constexpr int OFF_BAR = OFF_BIAS + 2 * 2 * kBN * 4;
  static constexpr int NBAR = 2 /*q_full*/ + 2 * NS /*kv full/empty*/ + 2 /*k0*/ + 2 /*s_full*/ +
                              2 /*p_full*/ + 2 /*o_done*/ + 4 /*bias*/ + 1 /*drain*/;
  static constexpr int OFF_SCALARS = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_SCALARS + 64;
  static constexpr int SMEM_ALLOC = BYTES + 1024;          // slack for 1024-B alignment
};

// Step i of the key loop reads V_i and K_{i+1} (PV of key tile i, S of tile
// i+1): one barrier covers both loads and one commit releases both stages.
// K of the first tile has its own pair.
struct Bars {
  uint64_t* q_full;    // [2]
  uint64_t* kv_full;   // [NS] V_i in V stage i%NS and K_{i+1} in K stage (i+1)%NS landed
  uint64_t* kv_empty;  // [NS] step i's products done: V stage i%NS, K stage (i+1)%NS free
  uint64_t* k0_full;   // K of the first key tile (K stage 0)
  uint64_t* k0_empty;  // its S products done
  uint64_t* s_full;    // [2]
  uint64_t* p_full;    // [2]
  uint64_t* o_done;    // [2]
  uint64_t* bias_rdy;  // [2 tiles][2 bufs]
  uint64_t* drain;     // [1]
};

template <int D, bool FP8>
__device__ __forceinline__ Bars carve_bars(uint8_t* smem) {
  using C = FwdCfg<D, FP8>;
  uint64_t* b = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  Bars r;
  r.q_full = b; b += 2;
  r.kv_full = b; b += C::NS;
  r.kv_empty = b; b += C::NS;
  r.k0_full = b; b += 1;
  r.k0_empty = b; b += 1;
  r.s_full = b; b += 2;
  r.p_full = b; b += 2;
  r.o_done = b; b += 2;
  r.bias_rdy = b; b += 4;
  r.drain = b;
  return r;
}

template <int D, bool CAUSAL, bool BIAS, bool FP8>
__device__ __forceinline__ void fwd_body(const FwdBf16Args& a) {
  using C = FwdCfg<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const Problem& p = a.p;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;

  Bars bars = carve_bars<D, FP8>(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_SCALARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_SCALARS + 4);
  int* key_lo_s = reinterpret_cast<int*>(smem + C::OFF_SCALARS + 8);
  int* key_hi_s = reinterpret_cast<int*>(smem + C::OFF_SCALARS + 12);
  int* nfin_s = reinterpret_cast<int*>(smem + C::OFF_SCALARS + 16);   // keys with a finite bias
  int* nzf_s = reinterpret_cast<int*>(smem + C::OFF_SCALARS + 20);    // a finite bias != 0 seen
  float* bias_buf = reinterpret_cast<float*>(smem + C::OFF_BIAS);
  const WaitCtx wc{abort_flag, a.err};

  // ---- which (query-tile pair, head). Heads are taken in groups of
  // a.head_group whose K/V fit comfortably in L2; within a group the CTAs go
  // heaviest first (last query tiles, the most key tiles under a causal mask),
  // cycling over the group's heads, so that both L2 reuse of K/V and the load
  // balance of the causal triangle are kept.
  const int n_pairs = (p.Nq + 2 * kBM - 1) / (2 * kBM);
  const int BH = p.B * p.H;
  const int G = a.head_group;
  const int grp = (int)(blockIdx.x / (G * n_pairs));
  const int g0 = grp * G;
  const int gsz = min(G, BH - g0);
  const int rr = (int)(blockIdx.x - (long)g0 * n_pairs);
  const int bh = g0 + rr % gsz;
  const int pair = n_pairs - 1 - rr / gsz;
  const int b = bh / p.H;
  // rows, lengths and head coordinates of this (sequence, head); query rows
  // and keys are numbered from 0 inside the sequence below
  const SeqView sv = seq_view(p, b, bh % p.H);
  const int Nq = sv.len_q, Nk = sv.len_k;
  const int q_base = pair * 2 * kBM;
  const float* bias_row = BIAS ? a.bias + (size_t)b * Nk : nullptr;

  // ---- key-tile ranges [lo, hi_t) of the two query tiles, from the keys
  // [klo, khi] that can be visible: the whole sequence, or (with a bias) the
  // first to the last key with a finite bias, known after the scan below
  const int n_kv = (Nk + kBN - 1) / kBN;
  int lo = 0, hi = 0;
  int hi_t[2] = {0, 0};
  bool any = false;
  auto set_ranges = [&](int klo, int khi) {
    int hi_all;
    if (khi < 0) {
      lo = hi_all = 0;
    } else {
      lo = klo / kBN;
      hi_all = khi / kBN + 1;
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int r0 = q_base + t * kBM;
      int h = hi_all;
      if (r0 >= Nq) {
        h = lo;   // tile past the last query row: inactive
      } else if (CAUSAL) {
        const long last_row = min(r0 + kBM - 1, Nq - 1);
        const long lim = last_row + (long)Nk - Nq;
        h = lim < 0 ? 0 : (int)min((long)hi_all, lim / kBN + 1);
      }
      hi_t[t] = max(h, lo);
    }
    if (a.n_split > 1) {
      // split-KV: this CTA covers key tiles [s_lo, s_hi) of its query tiles only
      const int per = (n_kv + a.n_split - 1) / a.n_split;
      const int s_lo = (int)blockIdx.y * per, s_hi = min(n_kv, s_lo + per);
      lo = max(lo, s_lo);
#pragma unroll
      for (int t = 0; t < 2; ++t) hi_t[t] = max(lo, min(hi_t[t], s_hi));
    }
    hi = max(hi_t[0], hi_t[1]);
    any = hi > lo;
  };
  if (!BIAS) set_ranges(0, Nk - 1);
  // the producer thread's first loads, in the order the first products use
  // them: Q of tile 0, K of the first key tile, Q of tile 1
  auto first_loads = [&]() {
    for (int t = 0; t < 2; ++t) {
      if (hi_t[t] > lo) {
        mbar_arrive_expect_tx(&bars.q_full[t], C::TILE);
        for (int c = 0; c < C::NBOX; ++c)
          tma_load_3d(smem + C::OFF_Q + t * C::TILE + c * C::SUB, &a.tm_q, c * (128 / C::EB),
                      sv.q_off + q_base + t * kBM, sv.hq, &bars.q_full[t]);
      }
      if (t == 0) {
        mbar_arrive_expect_tx(bars.k0_full, C::TILE);
        for (int c = 0; c < C::NBOX; ++c)
          tma_load_3d(smem + C::OFF_K + c * C::SUB, &a.tm_k, c * (128 / C::EB), sv.k_off + lo * kBN,
                      sv.hk, bars.k0_full);
      }
    }
  };

  // ---- set-up: barriers, TMEM, optional scan of the bias row. Without a
  // bias the producer thread issues the first loads right after initialising
  // the barriers, under the rest of the set-up.
  if (warp == C::W_TMA && lane == 0) {
    mbar_init(&bars.q_full[0], 1);
    mbar_init(&bars.q_full[1], 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);
    }
    mbar_init(bars.k0_full, 1);
    mbar_init(bars.k0_empty, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars.s_full[t], 1);
      mbar_init(&bars.p_full[t], kBM / 32);   // one arrival per softmax warp
      mbar_init(&bars.o_done[t], 1);
      mbar_init(&bars.bias_rdy[2 * t + 0], kBM / 32);
      mbar_init(&bars.bias_rdy[2 * t + 1], kBM / 32);
    }
    mbar_init(bars.drain, 1);
    *abort_flag = 0;
    *key_lo_s = Nk;
    if (sv.bad && pair == n_pairs - 1) atomicOr(a.err, ERR_BAD_SEQLEN);
    *key_hi_s = -1;
    *nfin_s = 0;
    *nzf_s = 0;
    fence_mbar_init();
    tma_prefetch_desc(&a.tm_q);
    tma_prefetch_desc(&a.tm_k);
    tma_prefetch_desc(&a.tm_v);
    if (!BIAS && any) first_loads();
  }
  if (warp == C::W_MMA) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  __syncthreads();
  if (BIAS) {
    // first and last key with a finite bias (tiles outside are skipped), how
    // many keys have one, and whether any of those is not 0
    int klo = Nk, khi = -1, cnt = 0;
    bool nz = false;
    for (int j = threadIdx.x; j < Nk; j += C::NT) {
      const float bj = bias_row[j];
      if (bj != -INFINITY) {
        klo = min(klo, j);
        khi = max(khi, j);
        ++cnt;
        nz |= (bj != 0.f);
      }
    }
    if (klo < Nk) atomicMin(key_lo_s, klo);
    if (khi >= 0) atomicMax(key_hi_s, khi);
    if (cnt) atomicAdd(nfin_s, cnt);
    if (nz) atomicOr(nzf_s, 1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (BIAS) set_ranges(*key_lo_s, *key_hi_s);
  // A bias that is 0 on keys [0, khi] and -inf past them is a key-padding
  // mask: adding it is the same as hiding the keys past khi, which the
  // softmax warps then do like the ragged tail of a key range, without the
  // per-tile bias values.
  const bool pad_only = BIAS && *nzf_s == 0 && *nfin_s == *key_hi_s + 1;
  const bool use_bias = BIAS && !pad_only;
  const long key_last = pad_only ? (long)*key_hi_s : (long)Nk - 1;

  if (warp == C::W_TMA) {
    // ================================================================ TMA producer
    if (lane == 0 && any) {
      if (BIAS) first_loads();
      auto load_k = [&](int j, int stage, uint64_t* bar) {
        for (int c = 0; c < C::NBOX; ++c)
          tma_load_3d(smem + C::OFF_K + stage * C::TILE + c * C::SUB, &a.tm_k, c * (128 / C::EB),
                      sv.k_off + j * kBN, sv.hk, bar);
      };
      auto load_v = [&](int j, int stage, uint64_t* bar) {
        if constexpr (FP8) {
          // V^T tile: 128 keys (bytes) x D rows
          tma_load_3d(smem + C::OFF_V + stage * C::TILE, &a.tm_v, j * kBN, 0, sv.hk, bar);
        } else {
          for (int c = 0; c < C::NBOX; ++c)
            tma_load_3d(smem + C::OFF_V + stage * C::TILE + c * C::SUB, &a.tm_v, c * 64,
                        sv.k_off + j * kBN, sv.hk, bar);
        }
      };
      int nkv = 0;   // steps whose loads were issued
      for (int j = lo; j < hi; ++j) {
        const int i = j - lo, s = i % C::NS, u = i / C::NS, s1 = (i + 1) % C::NS;
        const bool next_k = j + 1 < hi;
        // V stage s held V_{i-NS} and K stage s1 held K_{i+1-NS}: both free once
        // step i-NS is done (for i = NS-1, K stage 0 held the first tile's K)
        if (u > 0 && !wait1(&bars.kv_empty[s], (u - 1) & 1, wc, ERR_WAIT_LOAD)) break;
        if (next_k && i + 1 == C::NS && !wait1(bars.k0_empty, 0, wc, ERR_WAIT_LOAD)) break;
        mbar_arrive_expect_tx(&bars.kv_full[s], (next_k ? 2 : 1) * C::TILE);
        load_v(j, s, &bars.kv_full[s]);
        if (next_k) load_k(j + 1, s1, &bars.kv_full[s]);
        ++nkv;
      }
      // Drain: wait (bounded, ignoring the abort flag) for the last fill of
      // every stage, so that no copy is still landing when the CTA exits.
      // In a normal run every fill has already been consumed and these
      // return at once.
      const WaitCtx wd{abort_flag, a.err, true};
      wait1(bars.k0_full, 0, wd, ERR_WAIT_DRAIN);
      for (int i = max(0, nkv - C::NS); i < nkv; ++i)
        wait1(&bars.kv_full[i % C::NS], (i / C::NS) & 1, wd, ERR_WAIT_DRAIN);
      for (int t = 0; t < 2; ++t)
        if (hi_t[t] > lo) wait1(&bars.q_full[t], 0, wd, ERR_WAIT_DRAIN);
    }
  } else if (warp == C::W_MMA) {
    // ================================================================ MMA issuer
    // (the whole warp, converged; one elected lane issues each instruction)
    if (any) {
      constexpr uint32_t idesc_s =
          FP8 ? idesc_e4m3_f32(kBM, kBN, false, false) : idesc_bf16_f32(kBM, kBN, false, false);
      // PV: B = V (MN-major, d contiguous) or, FP8, V^T (K-major, keys contiguous)
      constexpr uint32_t idesc_pv =
          FP8 ? idesc_e4m3_f32(kBM, D, false, false) : idesc_bf16_f32(kBM, D, false, true);
      const uint32_t q_addr = smem_u32(smem + C::OFF_Q);
      const uint32_t k_addr = smem_u32(smem + C::OFF_K);
      const uint32_t v_addr = smem_u32(smem + C::OFF_V);
      auto active = [&](int t, int j) { return j >= lo && j < hi_t[t]; };
      // operand descriptors of each stage, built once; an instruction's
      // descriptor is the stage's plus its byte offset
      const uint64_t qd0 = sdesc_sw128(q_addr, 16, 1024);
      const uint64_t kd0 = sdesc_sw128(k_addr, 16, 1024);
      const uint64_t vd0 = FP8 ? sdesc_sw128(v_addr, 16, 1024) : sdesc_sw128(v_addr, C::SUB, 1024);
      auto issue_s = [&](int t, int s) {
        const uint64_t qd = sdesc_offset(qd0, t * C::TILE), kd = sdesc_offset(kd0, s * C::TILE);
        // K steps of 32 bytes (16 bf16 or 32 e4m3) along the 128-byte rows
#pragma unroll
        for (int kk = 0; kk < D * C::EB / 32; ++kk) {
          const uint32_t off = (kk / 4) * C::SUB + (kk % 4) * 32;
          if constexpr (FP8)
            mma_ss_f8_w(tmem + t * 128, sdesc_offset(qd, off), sdesc_offset(kd, off), idesc_s, kk > 0);
          else
            mma_ss_w(tmem + t * 128, sdesc_offset(qd, off), sdesc_offset(kd, off), idesc_s, kk > 0);
        }
      };
      auto issue_pv = [&](int t, int s, bool acc) {
        const uint64_t vd = sdesc_offset(vd0, s * C::TILE);
        if constexpr (FP8) {
          // P as packed e4m3 (4 keys per TMEM column): 32 keys per K step
#pragma unroll
          for (int kk = 0; kk < kBN / 32; ++kk)
            mma_ts_f8_w(tmem + 256 + t * D, tmem + t * 128 + kk * 8, sdesc_offset(vd, kk * 32), idesc_pv,
                      (acc || kk > 0) ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts_w(tmem + 256 + t * D, tmem + t * 128 + kk * 8, sdesc_offset(vd, kk * 2048), idesc_pv,
                   (acc || kk > 0) ? 1u : 0u);
        }
      };
      // S of the first key tile for each query tile as soon as that tile's
      // Q has landed (the loads go out Q0, K of the first key tile, Q1)
      bool ok = wait_warp(bars.k0_full, 0, wc, ERR_WAIT_MMA);
      for (int t = 0; t < 2 && ok; ++t) {
        if (!active(t, lo)) continue;
        if (!(ok = wait_warp(&bars.q_full[t], 0, wc, ERR_WAIT_MMA))) break;
        tc_fence_after();
        issue_s(t, 0);
        mma_commit_w(&bars.s_full[t]);
      }
      if (ok) mma_commit_w(bars.k0_empty);
      for (int j = lo; j < hi && ok; ++j) {
        const int i = j - lo, s = i % C::NS, s1 = (i + 1) % C::NS;
        // V_i and K_{i+1}
        if (!wait_warp(&bars.kv_full[s], (i / C::NS) & 1, wc, ERR_WAIT_MMA)) { ok = false; break; }
        tc_fence_after();
        for (int t = 0; t < 2 && ok; ++t) {
          if (active(t, j)) {
            if (!wait_warp(&bars.p_full[t], i & 1, wc, ERR_WAIT_MMA)) { ok = false; break; }
            tc_fence_after();
            issue_pv(t, s, i > 0);
            mma_commit_w(&bars.o_done[t]);
          }
          if (j + 1 < hi && active(t, j + 1)) {
            issue_s(t, s1);
            mma_commit_w(&bars.s_full[t]);
          }
        }
        if (!ok) break;
        mma_commit_w(&bars.kv_empty[s]);
      }
      // drain every MMA issued so far before TMEM is released
      mma_commit_w(bars.drain);
      wait_warp(bars.drain, 0, WaitCtx{abort_flag, a.err, true}, ERR_WAIT_DRAIN);
    }
  } else {
    // ================================================================ softmax
    const int t = warp / 4;                 // query tile of this warpgroup
    const int r = (warp % 4) * 32 + lane;   // row within the tile = TMEM lane
    const int row_g = q_base + t * kBM + r;
    const uint32_t lane_base = tmem + ((uint32_t)((warp % 4) * 32) << 16);
    const uint32_t s_col = t * 128, o_col = 256 + t * D;
    // FP8: S = sq * sk * (q8 k8^T), folded into the exponent's scale
    const float sqk = FP8 ? fp8_scale(a.amax_q[bh]) * fp8_scale(a.amax_k[sv.hk]) : 1.f;
    const float sl2 = p.scale * sqk * kLog2e;
    const long off = (long)Nk - Nq;
    // last visible key of this row / of the tile's first row (tile-uniform)
    const long lim_row = CAUSAL ? min((long)row_g + off, key_last) : key_last;
    const long lim_tile = CAUSAL ? min((long)(q_base + t * kBM) + off, key_last) : key_last;
    float m = -INFINITY, l = 0.f;
    const int n_t = hi_t[t] - lo;
    int i = 0;
    for (; i < n_t; ++i) {
      const int j = lo + i;
      const int key0 = j * kBN;
      if (use_bias) {
        float* bb = bias_buf + (t * 2 + (i & 1)) * kBN;
        const int kj = key0 + r;
        bb[r] = kj < Nk ? bias_row[kj] * kLog2e : -INFINITY;
        mbar_arrive_warp(&bars.bias_rdy[t * 2 + (i & 1)]);
        if (!wait_warp(&bars.bias_rdy[t * 2 + (i & 1)], (i >> 1) & 1, wc, ERR_WAIT_SOFTMAX)) break;
      }
      if (!wait_warp(&bars.s_full[t], i & 1, wc, ERR_WAIT_SOFTMAX)) break;
      tc_fence_after();
      float s[kBN];
      uint32_t* su = reinterpret_cast<uint32_t*>(s);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + s_col + c * 32, su + c * 32);
      tmem_ld_wait();

      const bool need_mask = (long)key0 + kBN - 1 > lim_tile;
      const bool scaled = use_bias || need_mask;
      // Scores are handled in pairs with the packed f32x2 instructions, and
      // the row max with the three-input max: about three instructions per
      // score in total.
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (scaled) {
        const float* bb = bias_buf + (t * 2 + (i & 1)) * kBN;
        const long lim_rel = lim_row - key0;
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
        for (int c = 0; c < kBN; c += 4) {
          // four bias values per shared-memory load (the same address in
          // every lane: a broadcast)
          float4 b4 = make_float4(0.f, 0.f, 0.f, 0.f);
          if (use_bias) b4 = *reinterpret_cast<const float4*>(bb + c);
          float v[4];
          f2_unpack(fma2(f2_pack(s[c], s[c + 1]), sl2x2, f2_pack(b4.x, b4.y)), v[0], v[1]);
          f2_unpack(fma2(f2_pack(s[c + 2], s[c + 3]), sl2x2, f2_pack(b4.z, b4.w)), v[2], v[3]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (need_mask && c + e > lim_rel) v[e] = -INFINITY;
            s[c + e] = v[e];
          }
          m4[(c / 2) & 3] = fmax3(m4[(c / 2) & 3], v[0], v[1]);
          m4[(c / 2 + 1) & 3] = fmax3(m4[(c / 2 + 1) & 3], v[2], v[3]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kBN; c += 2) m4[(c / 2) & 3] = fmax3(m4[(c / 2) & 3], s[c], s[c + 1]);
      }
      float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      if (!scaled) mx *= sl2;
      // conditional move of the running max
      float alpha = 1.f;
      bool moved = false;
      if (mx > m + kRescaleLog2 || (m == -INFINITY && mx > -INFINITY)) {
        alpha = ex2(m - mx);   // m = -inf -> 0
        moved = (m != -INFINITY);
        m = mx;
      }
      const float mu = (m == -INFINITY) ? 0.f : m;
      // p = exp2(s * scale*log2e - mu) (or exp2(s - mu) for scores already in
      // the base-2 domain), as one packed FMA per pair
      const uint64_t mul2 = scaled ? f2_pack(1.f, 1.f) : f2_pack(sl2, sl2);
      const uint64_t nmu2 = f2_pack(-mu, -mu);
      uint64_t ps2[4] = {0ull, 0ull, 0ull, 0ull};   // row sum as 4 packed partial sums
      if constexpr (FP8) {
        // P as e4m3, 4 keys per TMEM column (p <= 2^8 fits the e4m3 range)
#pragma unroll
        for (int c0 = 0; c0 < kBN; c0 += 32) {
          uint32_t pk[8];
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            float x0, x1, x2, x3;
            f2_unpack(fma2(f2_pack(s[c0 + c], s[c0 + c + 1]), mul2, nmu2), x0, x1);
            f2_unpack(fma2(f2_pack(s[c0 + c + 2], s[c0 + c + 3]), mul2, nmu2), x2, x3);
            const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
            ps2[(c / 2) & 3] = add2(ps2[(c / 2) & 3], f2_pack(p0, p1));
            ps2[(c / 2 + 1) & 3] = add2(ps2[(c / 2 + 1) & 3], f2_pack(p2, p3));
            pk[c / 4] = pack_e4m3x4(p0, p1, p2, p3);
          }
          tmem_st8(lane_base + s_col + c0 / 4, pk);
        }
      } else {
#pragma unroll
        for (int c0 = 0; c0 < kBN; c0 += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float x0, x1;
            f2_unpack(fma2(f2_pack(s[c0 + c], s[c0 + c + 1]), mul2, nmu2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            ps2[(c / 2) & 3] = add2(ps2[(c / 2) & 3], f2_pack(p0, p1));
            pk[c / 2] = pack_bf16x2(p0, p1);
          }
          tmem_st16(lane_base + s_col + c0 / 2, pk);
        }
      }
      float ps[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) f2_unpack(ps2[k], ps[2 * k], ps[2 * k + 1]);
      const float psum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      l = l * alpha + psum;
      // rescale O if any row of this warp moved its max and O already holds data
      if (__any_sync(0xffffffffu, moved) && i > 0) {
        if (!wait_warp(&bars.o_done[t], (i - 1) & 1, wc, ERR_WAIT_SOFTMAX)) break;
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t ov[32];
          tmem_ld32(lane_base + o_col + c0, ov);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
          tmem_st32(lane_base + o_col + c0, ov);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(&bars.p_full[t]);
    }
    // ---- epilogue: O = O_acc / l (bf16), LSE = ln2 * (m + log2 l)
    const bool completed = (i == n_t);
    bool have_o = completed && n_t > 0;
    if (have_o) {
      if (!wait_warp(&bars.o_done[t], (n_t - 1) & 1, wc, ERR_WAIT_SOFTMAX)) have_o = false;
      tc_fence_after();
    }
    if (completed && a.n_split > 1) {
      // partial result of this key range: normalised O in fp32 and its LSE,
      // merged by the combine kernel
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const size_t prow = ((size_t)blockIdx.y * p.B * p.H + bh) * p.Nq + row_g;
      float* orow = a.part_o + prow * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t ov[32];
        if (have_o) {
          tmem_ld32(lane_base + o_col + c0, ov);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) ov[c] = 0u;
        }
        if (row_g < Nq) {
          float4* dst = reinterpret_cast<float4*>(orow + c0);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            dst[v4] = make_float4(__uint_as_float(ov[4 * v4]) * inv, __uint_as_float(ov[4 * v4 + 1]) * inv,
                                  __uint_as_float(ov[4 * v4 + 2]) * inv,
                                  __uint_as_float(ov[4 * v4 + 3]) * inv);
        }
      }
      if (row_g < Nq) a.part_lse[prow] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
    if (a.n_split <= 1) {
      // O = O_acc / l in bf16, staged in this tile's Q buffer (free: every
      // S product of the tile is done) as the 128-byte-swizzled 64-column
      // boxes TMA uses, then stored with TMA by one thread of the
      // warpgroup; the CTA waits only until TMA has read the buffer. A
      // packed sequence's ragged last tile gets plain coalesced stores (a
      // 128-row box would run into the next sequence).
      const int r0 = q_base + t * kBM;
      const bool do_epi = completed && r0 < Nq;
      uint8_t* stage = smem + C::OFF_OST + t * C::OTILE;
      if (do_epi) {
        // FP8: O = sv * (P8 v8) / l
        const float sv_ = FP8 ? fp8_scale(a.amax_v[sv.hk]) : 1.f;
        const float inv = l > 0.f ? sv_ / l : 0.f;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t ov[32];
          if (have_o) {
            tmem_ld32(lane_base + o_col + c0, ov);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = 0u;
          }
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2)
            pk[c / 2] = pack_bf16x2(__uint_as_float(ov[c]) * inv, __uint_as_float(ov[c + 1]) * inv);
          uint8_t* rowp = stage + (c0 / 64) * C::SUB + r * 128;
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            const int j = (c0 % 64) / 8 + v4;
            *reinterpret_cast<uint4*>(rowp + ((j ^ (r & 7)) * 16)) =
                make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
        }
        if (row_g < Nq)
          a.lse[(size_t)sv.hq * sv.qrows + sv.q_off + row_g] =
              l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        fence_proxy_async_smem();   // generic-proxy writes, before TMA reads them
      }
      // all 128 threads of the warpgroup arrive; the tile is written only if
      // every warp staged its rows
      if (named_bar_and(1 + t, kBM, do_epi)) {
        if (p.cu_q == nullptr || r0 + kBM <= Nq) {
          if (r == 0) {
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_store_3d(&a.tm_o, stage + c * C::SUB, c * 64, sv.q_off + r0, sv.hq);
            bulk_commit_group();
            bulk_wait_group_read0();   // shared memory may be released
          }
        } else {
          constexpr int CPR = D / 8;   // 16-byte pieces per row
          for (int idx = r; idx < kBM * CPR; idx += kBM) {
            const int row = idx / CPR, c = idx % CPR;
            if (r0 + row < Nq) {
              const uint4 v = *reinterpret_cast<const uint4*>(
                  stage + (c / 8) * C::SUB + row * 128 + (((c % 8) ^ (row & 7)) * 16));
              *reinterpret_cast<uint4*>(a.o + ((size_t)sv.hq * sv.qrows + sv.q_off + r0 + row) * D +
                                        c * 8) = v;
            }
          }
        }
      }
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == C::W_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL, bool BIAS>
__global__ void __launch_bounds__(FwdCfg<D, false>::NT, 1) fwd_bf16_kernel(const __grid_constant__ FwdBf16Args a) {
  fwd_body<D, CAUSAL, BIAS, false>(a);
}

// The same forward on e4m3 operands (kind::f8f6f4 MMAs at twice the bf16
// rate): S from e4m3 Q, K with per-head scales, P rounded to e4m3 for PV.
template <int D, bool CAUSAL, bool BIAS>
__global__ void __launch_bounds__(FwdCfg<D, true>::NT, 1) fwd_fp8_kernel(const __grid_constant__ FwdBf16Args a) {
  fwd_body<D, CAUSAL, BIAS, true>(a);
}

// Split-KV combine (the merge of partial softmax states over disjoint key
// ranges: "flash-attention", Part VI; "FlashAttention: Mathematical
// Foundations...", Flash-Decoding): with partial (O_s, LSE_s),
//   LSE = log sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s.
// One warp per query row; a row whose every partial is empty stays O = 0,
// LSE = -inf.
template <int D>
__global__ void __launch_bounds__(256) splitkv_combine_kernel(const float* __restrict__ part_o,
                                                              const float* __restrict__ part_lse,
                                                              uint16_t* __restrict__ o,
                                                              float* __restrict__ lse, long rows,
                                                              int n_split) {
  const long row = ((long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float mx = -INFINITY;
  for (int s = 0; s < n_split; ++s) mx = fmaxf(mx, part_lse[(long)s * rows + row]);
  constexpr int PER = D / 32;   // columns per lane
  float acc[PER];
#pragma unroll
  for (int c = 0; c < PER; ++c) acc[c] = 0.f;
  float sum = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < n_split; ++s) {
      const float ls = part_lse[(long)s * rows + row];
      if (ls == -INFINITY) continue;
      const float w = __expf(ls - mx);
      sum += w;
      const float* src = part_o + ((long)s * rows + row) * D + lane * PER;
#pragma unroll
      for (int c = 0; c < PER; ++c) acc[c] = fmaf(w, src[c], acc[c]);
    }
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  uint16_t* dst = o + row * D + lane * PER;
#pragma unroll
  for (int c = 0; c < PER; c += 2)
    *reinterpret_cast<uint32_t*>(dst + c) = pack_bf16x2(acc[c] * inv, acc[c + 1] * inv);
  if (lane == 0) lse[row] = sum > 0.f ? mx + __logf(sum) : -INFINITY;
}

template <int D, bool CAUSAL, bool BIAS>
cudaError_t launch_one(const FwdBf16Args& a, cudaStream_t s) {
  using C = FwdCfg<D, false>;
  auto kern = fwd_bf16_kernel<D, CAUSAL, BIAS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  const long BH = (long)a.p.B * a.p.H;
  const long n_pairs = (a.p.Nq + 2 * kBM - 1) / (2 * kBM);
  // heads per ordering group: K and V of a group within ~48 MiB of L2
  const long kv_bytes = 2L * a.p.Nk * D * 2;
  FwdBf16Args b = a;
  b.head_group = (int)std::max(1L, std::min(BH, (48L << 20) / std::max(kv_bytes, 1L)));
  const dim3 grid((unsigned)(BH * n_pairs), (unsigned)std::max(1, a.n_split));
  kern<<<grid, C::NT, C::SMEM_ALLOC, s>>>(b);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.n_split <= 1) return e;
  const long rows = BH * a.p.Nq;
  splitkv_combine_kernel<D><<<(unsigned)((rows * 32 + 255) / 256), 256, 0, s>>>(
      a.part_o, a.part_lse, a.o, a.lse, rows, a.n_split);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const FwdBf16Args& a, cudaStream_t s) {
  const bool bias = a.bias != nullptr;
  if (a.p.causal)
    return bias ? launch_one<D, true, true>(a, s) : launch_one<D, true, false>(a, s);
  return bias ? launch_one<D, false, true>(a, s) : launch_one<D, false, false>(a, s);
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdBf16Args& a, cudaStream_t s) {
  return a.p.d == 64 ? launch_d<64>(a, s) : launch_d<128>(a, s);
}

namespace {
template <bool CAUSAL, bool BIAS>
cudaError_t launch_fp8_one(const FwdBf16Args& a, cudaStream_t s) {
  using C = FwdCfg<128, true>;
  static_assert(C::SMEM_ALLOC <= 232448, "shared memory per CTA");
  auto kern = fwd_fp8_kernel<128, CAUSAL, BIAS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  const long BH = (long)a.p.B * a.p.H;
  const long n_pairs = (a.p.Nq + 2 * kBM - 1) / (2 * kBM);
  const long kv_bytes = 2L * a.p.Nk * 128;   // e4m3 K and V of a head
  FwdBf16Args b = a;
  b.head_group = (int)std::max(1L, std::min(BH, (48L << 20) / std::max(kv_bytes, 1L)));
  b.n_split = 1;
  kern<<<(unsigned)(BH * n_pairs), C::NT, C::SMEM_ALLOC, s>>>(b);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_fwd_fp8(const FwdBf16Args& a, cudaStream_t s) {
  const bool bias = a.bias != nullptr;
  if (a.p.causal) return bias ? launch_fp8_one<true, true>(a, s) : launch_fp8_one<true, false>(a, s);
  return bias ? launch_fp8_one<false, true>(a, s) : launch_fp8_one<false, false>(a, s);
}

}  // namespace fa
