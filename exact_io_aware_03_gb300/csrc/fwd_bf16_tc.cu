// bf16 forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Dataflow (query-tile outer, key/value tiles streamed: the order of
// "FlashAttention, Explained", §20, with the online-softmax merge of
// "Understanding FlashAttention Pt 1", §2.4):
//
//   one work unit = two 128-row query tiles Q0, Q1 of one (b, h), kept in
//   shared memory; K_j / V_j tiles of 128 keys stream through an NS-stage
//   ring. For each key tile j and each query tile t:
//     S_t   = Q_t K_j^T              tcgen05.mma, fp32 accumulator in TMEM
//     P_t   = exp2(S_t*c - m_t)      softmax warps: TMEM -> registers -> TMEM
//                                    (P overwrites S in place as packed bf16)
//     O_t  += P_t V_j                tcgen05.mma with A read from TMEM
//   and after the last tile O = O_t / l_t, LSE = ln 2 * (m_t + log2 l_t).
//
// Scheduling: a CTA takes the unit with its own index first. In the
// persistent form (grid = one CTA per SM) it then claims further units from
// a counter, one at a time, until none is left; the pipeline runs on across
// units: the K/V ring and every barrier phase continue, the next unit is
// claimed a few key steps before the current one ends and its Q tiles are
// prefetched into L2, its first K tile is loaded with the current unit's last
// V tile, its Q tiles as soon as the current unit's last S product of that
// tile is done, and its first S products are issued right after the current
// unit's last PV products, under the softmax warps' epilogue of the current
// unit. Otherwise (key bias, packed sequences, split-KV, FP8, or no more units
// than SMs) each CTA computes one unit.
//
// The counter needs memory that no other launch touches: it is the LSE word
// of the last unit's first row (row 0 of the last head), which the launcher
// sets to 0xFFFFFFFF with a memset on the launch's stream. A claim is one
// atomic decrement: the unit is 0xFFFFFFFF - (value before it), valid below
// the number of claimable units; a claim past the end adds its 1 back at once.
// The last unit is claimed last; its epilogue stores the row's LSE with a
// compare-and-swap from the exhausted value, which succeeds once every
// overshooting claim has been undone, and later overshoots only dip the word
// and restore it. The LSE values the kernel writes stay clear of the counter
// range even after such a dip: they are never negative NaNs (arithmetic NaNs
// are positive), and a +0 or positive subnormal LSE on that row is stored as
// -0.
//
// Warp roles (320 threads, one CTA per SM):
//   warps 0-3   softmax for Q0 (thread = query row = TMEM lane)
//   warps 4-7   softmax for Q1
//   warp  8     TMA producer and unit claims (one lane)
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
constexpr int kClaimAhead = 2;   // key steps between claiming the next unit and the last step's loads

// FP8: q, k are e4m3 [rows][d] and v is e4m3 transposed, [d][keys] (every
// operand K-major), with per-head scales; d = 128 only (one 128-byte row).
template <int D, bool FP8, bool PERSIST>
struct FwdCfg {
  static constexpr int EB = FP8 ? 1 : 2;                   // element bytes of q, k, v
  static constexpr int NS = FP8 ? 3 : ((D == 128) ? 2 : 4);   // K/V ring stages
  static constexpr int TILE = kBM * D * EB;                // bytes of one q/k/v tile
  static constexpr int SUB = kBM * 128;                    // bytes of one 128-byte-wide box
  static constexpr int NBOX = D * EB / 128;                // boxes per tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = 2 * TILE;
  static constexpr int OFF_V = OFF_K + NS * TILE;
  static constexpr int OTILE = kBM * D * 2;                // bf16 O tile
  // O staging. One unit per CTA: the tile's Q buffer (bf16; free once the
  // tile's last S product is done) or, FP8, a buffer of its own, read by TMA
  // stores. Persistent: the next unit's Q is already in the Q buffers, so
  // each softmax warpgroup has one 64-column box of its own (a 4 KiB slice
  // per warp).
  static constexpr int OFF_OST = PERSIST ? OFF_V + NS * TILE : (FP8 ? OFF_V + NS * TILE : OFF_Q);
  static constexpr int OST_BYTES = PERSIST ? 2 * kBM * 128 : (FP8 ? 2 * OTILE : 0);
  // warp roles: softmax warps 0-7, then the TMA producer and the MMA issuer
  static constexpr int W_TMA = 8, W_MMA = 9;
  static constexpr int NT = 320;
  // key bias: [2 tiles][2 buffers][128] floats (the persistent form has no bias)
  static constexpr int OFF_BIAS = OFF_V + NS * TILE + OST_BYTES;
  static constexpr int OFF_BAR = OFF_BIAS + (PERSIST ? 0 : 2 * 2 * kBN * 4);
  static constexpr int NBAR = 2 /*q_full*/ + 2 /*q_empty*/ + 2 * NS /*kv full/empty*/ + 2 /*k0*/ +
                              2 /*s_full*/ + 2 /*p_full*/ + 2 /*o_done*/ + 4 /*bias*/ +
                              4 /*unit ring*/ + 1 /*drain*/;
  // scalars: abort flag, TMEM base, bias scan results (4 words); then the
  // unit ring of the persistent form: 2 entries of 32 bytes
  static constexpr int OFF_SCALARS = OFF_BAR + NBAR * 8;
  static constexpr int OFF_RING = (OFF_SCALARS + 24 + 31) / 32 * 32;
  static constexpr int BYTES = OFF_RING + 2 * 32;
  static constexpr int SMEM_ALLOC = BYTES + 1024;          // slack for 1024-B alignment
  static_assert(SMEM_ALLOC <= 232448, "shared memory per CTA");
};

// Step g of the key loop (counted over all units of the CTA) reads V_g and
// K_{g+1} (PV of its key tile, S of the next one, which is the next unit's
// first key tile at a unit's last step): one barrier covers both loads and
// one commit releases both stages. K of the CTA's first key tile has its own
// pair.
struct Bars {
  uint64_t* q_full;      // [2] Q of tile t landed
  uint64_t* q_empty;     // [2] the last S product of tile t in a unit done (Q stage free)
  uint64_t* kv_full;     // [NS] V_g in V stage g%NS and K_{g+1} in K stage (g+1)%NS landed
  uint64_t* kv_empty;    // [NS] step g's products done: V stage g%NS, K stage (g+1)%NS free
  uint64_t* k0_full;     // K of the first key tile (K stage 0)
  uint64_t* k0_empty;    // its S products done
  uint64_t* s_full;      // [2]
  uint64_t* p_full;      // [2]
  uint64_t* o_done;      // [2]
  uint64_t* bias_rdy;    // [2 tiles][2 bufs]
  uint64_t* unit_full;   // [2] unit ring entry written by the producer
  uint64_t* unit_empty;  // [2] entry read by the MMA warp and every softmax warp
  uint64_t* drain;       // [1]
};

template <int D, bool FP8, bool PERSIST>
__device__ __forceinline__ Bars carve_bars(uint8_t* smem) {
  using C = FwdCfg<D, FP8, PERSIST>;
  uint64_t* b = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  Bars r;
  r.q_full = b; b += 2;
  r.q_empty = b; b += 2;
  r.kv_full = b; b += C::NS;
  r.kv_empty = b; b += C::NS;
  r.k0_full = b; b += 1;
  r.k0_empty = b; b += 1;
  r.s_full = b; b += 2;
  r.p_full = b; b += 2;
  r.o_done = b; b += 2;
  r.bias_rdy = b; b += 4;
  r.unit_full = b; b += 2;
  r.unit_empty = b; b += 2;
  r.drain = b;
  return r;
}

// One unit per CTA (key bias, causal mask, packed sequences, split-KV, FP8):
// the CTA computes the unit with its own index.
template <int D, bool CAUSAL, bool BIAS, bool FP8>
__device__ __forceinline__ void fwd_body_one(const FwdBf16Args& a) {
  using C = FwdCfg<D, FP8, false>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const Problem& p = a.p;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;

  Bars bars = carve_bars<D, FP8, false>(smem);
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
  // packed sequences: the grid is sized by the longest one, and a CTA whose
  // query-tile pair starts past its sequence's end has no rows; it leaves
  // before any set-up (the sequence's last CTA reports a bad length first)
  if (p.cu_q != nullptr && q_base >= Nq) {
    if (sv.bad && pair == n_pairs - 1 && threadIdx.x == 0) atomicOr(a.err, ERR_BAD_SEQLEN);
    return;
  }

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

// One work unit of the persistent form: a pair of 128-row query tiles of one
// (batch, head) of a dense problem, and the key tiles [0, hi0) and [0, hi1)
// its two tiles read (0: tile inactive).
struct PUnit {
  int bh;       // query head coordinate (b * H + h) of q, o, lse
  int hk;       // key/value head coordinate of k, v
  int q_base;   // first query row of the pair
  int hi0, hi1;
};

// Units are numbered in this order: heads in groups of a.head_group whose K/V
// fit comfortably in L2; within a group heaviest first (last query tiles, the
// most key tiles under a causal mask), cycling over the group's heads, so
// that both L2 reuse of K/V and the load balance of the causal triangle are
// kept.
template <bool CAUSAL>
__device__ __forceinline__ PUnit punit(const FwdBf16Args& a, int id) {
  const Problem& p = a.p;
  const int n_pairs = (p.Nq + 2 * kBM - 1) / (2 * kBM);
  const int BH = p.B * p.H;
  const int G = a.head_group;
  const int g0 = id / (G * n_pairs) * G;
  const int gsz = min(G, BH - g0);
  const int rr = id - g0 * n_pairs;
  PUnit u;
  u.bh = g0 + rr % gsz;
  const int b = u.bh / p.H, h = u.bh - b * p.H;
  u.hk = b * p.Hkv + h / (p.H / p.Hkv);
  u.q_base = (n_pairs - 1 - rr / gsz) * 2 * kBM;
  const int n_kv = (p.Nk + kBN - 1) / kBN;
  int hi[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int r0 = u.q_base + t * kBM;
    int h2 = n_kv;
    if (r0 >= p.Nq) {
      h2 = 0;   // tile past the last query row: inactive
    } else if (CAUSAL) {
      const long last_row = min(r0 + kBM - 1, p.Nq - 1);
      const long lim = last_row + (long)p.Nk - p.Nq;
      h2 = lim < 0 ? 0 : (int)min((long)n_kv, lim / kBN + 1);
    }
    hi[t] = h2;
  }
  u.hi0 = hi[0];
  u.hi1 = hi[1];
  return u;
}

// Claim the next unit from the counter (one thread): units [gridDim.x,
// n_units) are handed out in order; -1 once none is left. A claim that finds
// the counter exhausted changes nothing; one that overshoots (it raced the
// last claims) adds its decrement back.
__device__ __forceinline__ int claim_unit(const FwdBf16Args& a) {
  const uint32_t n_dyn = (uint32_t)(a.n_units - (int)gridDim.x);
  if (0xFFFFFFFFu - *reinterpret_cast<volatile uint32_t*>(a.sched) >= n_dyn) return -1;
  const uint32_t k = 0xFFFFFFFFu - atomicSub(a.sched, 1u);
  if (k < n_dyn) return (int)gridDim.x + (int)k;
  atomicAdd(a.sched, 1u);
  return -1;
}

// Store the LSE of the row whose word held the counter (the last unit's, so
// every claim but overshoots is done): swap it in once the counter reads
// exhausted, i.e. no overshooting claim is still to be undone. Bounded: on
// time-out the error word records it and the value is stored plainly.
__device__ __forceinline__ void store_counter_lse(const FwdBf16Args& a, float v, const WaitCtx& w) {
  // +0 and positive subnormals as -0: after a dip by an overshooting claim
  // their bit pattern would wrap into the counter's range
  if (__float_as_uint(v) < 0x00800000u) v = -0.f;
  const uint32_t done = 0xFFFFFFFFu - (uint32_t)(a.n_units - (int)gridDim.x);
  const uint64_t t0 = globaltimer();
  while (atomicCAS(a.sched, done, __float_as_uint(v)) != done) {
    if (globaltimer() - t0 > FA_WAIT_TIMEOUT_NS) {
      raise_abort(w, ERR_WAIT_EPILOGUE);
      *reinterpret_cast<volatile float*>(a.sched) = v;
      return;
    }
  }
}

// Persistent form (dense bf16 q, k, v; no key bias; no split): grid = one CTA
// per SM. A CTA takes the unit with its own index first, then claims further
// units from the counter, one at a time, until none is left. The pipeline runs
// on across units: the K/V ring and every barrier phase continue; the next
// unit is claimed kClaimAhead key steps before the current unit's last step
// and its Q tiles are prefetched into L2; its first K tile is loaded with the
// current unit's last V tile, its Q tiles as soon as the current unit's last
// S product of that tile is done, and its first S products are issued right
// after the current unit's last PV products, under the softmax warps'
// epilogue of the current unit. The per-unit values the hot loops use are
// kept in plain scalars (the unit ring carries them precomputed).
template <int D, bool CAUSAL>
__device__ __forceinline__ void fwd_body_persistent(const FwdBf16Args& a) {
  using C = FwdCfg<D, false, true>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const Problem& p = a.p;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  const int Nq = p.Nq, Nk = p.Nk;

  Bars bars = carve_bars<D, false, true>(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_SCALARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_SCALARS + 4);
  // unit ring: [2] entries of 32 bytes (the unit, its id at +28)
  uint8_t* ring = smem + C::OFF_RING;
  const WaitCtx wc{abort_flag, a.err};

  const PUnit u0 = punit<CAUSAL>(a, (int)blockIdx.x);

  // ---- loads (producer thread). Q fills per tile, for the q_empty phases.
  int nq0 = 0, nq1 = 0;
  auto load_q = [&](const PUnit& u, int t) {
    mbar_arrive_expect_tx(&bars.q_full[t], C::TILE);
    for (int c = 0; c < C::NBOX; ++c)
      tma_load_3d(smem + C::OFF_Q + t * C::TILE + c * C::SUB, &a.tm_q, c * 64, u.q_base + t * kBM, u.bh,
                  &bars.q_full[t]);
    if (t == 0) ++nq0; else ++nq1;
  };
  auto load_k = [&](int hk, int j, int stage, uint64_t* bar) {
    for (int c = 0; c < C::NBOX; ++c)
      tma_load_3d(smem + C::OFF_K + stage * C::TILE + c * C::SUB, &a.tm_k, c * 64, j * kBN, hk, bar);
  };
  auto load_v = [&](int hk, int j, int stage, uint64_t* bar) {
    for (int c = 0; c < C::NBOX; ++c)
      tma_load_3d(smem + C::OFF_V + stage * C::TILE + c * C::SUB, &a.tm_v, c * 64, j * kBN, hk, bar);
  };

  // ---- set-up: barriers, then (producer) the first unit's loads in the
  // order its first products use them: Q of tile 0, K of the first key tile,
  // Q of tile 1; TMEM
  const bool any0 = max(u0.hi0, u0.hi1) > 0;
  if (warp == C::W_TMA && lane == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars.q_full[t], 1);
      mbar_init(&bars.q_empty[t], 1);
      mbar_init(&bars.s_full[t], 1);
      mbar_init(&bars.p_full[t], kBM / 32);   // one arrival per softmax warp
      mbar_init(&bars.o_done[t], 1);
      mbar_init(&bars.unit_full[t], 1);
      mbar_init(&bars.unit_empty[t], 2 * kBM / 32 + 1);   // softmax warps + MMA warp
    }
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);
    }
    mbar_init(bars.k0_full, 1);
    mbar_init(bars.k0_empty, 1);
    mbar_init(bars.drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&a.tm_q);
    tma_prefetch_desc(&a.tm_k);
    tma_prefetch_desc(&a.tm_v);
    if (any0) {
      if (u0.hi0 > 0) load_q(u0, 0);
      mbar_arrive_expect_tx(bars.k0_full, C::TILE);
      load_k(u0.hk, 0, 0, bars.k0_full);
      if (u0.hi1 > 0) load_q(u0, 1);
    }
  }
  if (warp == C::W_MMA) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::W_TMA) {
    // ================================================================ TMA producer
    if (lane == 0) {
      int e = 0;   // unit ring entries written
      // publish the CTA's next unit (-1: none) once the ring slot's previous
      // entry has been read by every consumer warp
      auto publish = [&](int id, const PUnit& u) -> bool {
        const int sl = e & 1;
        if (e >= 2 && !wait1(&bars.unit_empty[sl], ((e - 2) >> 1) & 1, wc, ERR_WAIT_LOAD)) return false;
        if (id >= 0) *reinterpret_cast<PUnit*>(ring + sl * 32) = u;
        *reinterpret_cast<volatile int*>(ring + sl * 32 + 28) = id;
        mbar_arrive(&bars.unit_full[sl]);
        ++e;
        return true;
      };
      PUnit cur = u0, nxt = u0;
      int nkv = 0;   // steps whose loads were issued (steps are counted over all units)
      bool ok = true;
      while (ok) {
        const int n = max(cur.hi0, cur.hi1);
        int nid = -1;
        // a unit without key tiles ends the CTA's claims (its first K could not
        // come with a previous step); the remaining units go to other CTAs
        if (n == 0) ok = publish(-1, nxt);
        for (int i = 0; i < n && ok; ++i) {
          if (i == max(0, n - 1 - kClaimAhead)) {
            // claim the next unit and prefetch its Q tiles into L2
            nid = claim_unit(a);
            if (nid >= 0) {
              nxt = punit<CAUSAL>(a, nid);
              for (int c = 0; c < C::NBOX; ++c) {
                if (nxt.hi0 > 0) tma_prefetch_l2_3d(&a.tm_q, c * 64, nxt.q_base, nxt.bh);
                if (nxt.hi1 > 0) tma_prefetch_l2_3d(&a.tm_q, c * 64, nxt.q_base + kBM, nxt.bh);
              }
            }
          }
          // the next unit is published before the last step's loads (they
          // include its first K)
          if (i == n - 1 && !(ok = publish(nid, nxt))) break;
          const int g = nkv, s = g % C::NS, u = g / C::NS, s1 = (g + 1) % C::NS;
          const bool k_cur = i + 1 < n;
          const bool k_nxt = !k_cur && nid >= 0 && max(nxt.hi0, nxt.hi1) > 0;
          // V stage s held V_{g-NS} and K stage s1 held K_{g+1-NS}: both free once
          // step g-NS is done (for g = NS-1, K stage 0 held the first key tile's K)
          if (u > 0 && !(ok = wait1(&bars.kv_empty[s], (u - 1) & 1, wc, ERR_WAIT_LOAD))) break;
          if ((k_cur || k_nxt) && g + 1 == C::NS && !(ok = wait1(bars.k0_empty, 0, wc, ERR_WAIT_LOAD))) break;
          mbar_arrive_expect_tx(&bars.kv_full[s], ((k_cur || k_nxt) ? 2 : 1) * C::TILE);
          load_v(cur.hk, i, s, &bars.kv_full[s]);
          if (k_cur) load_k(cur.hk, i + 1, s1, &bars.kv_full[s]);
          if (k_nxt) load_k(nxt.hk, 0, s1, &bars.kv_full[s]);
          ++nkv;
        }
        if (!ok || nid < 0) break;
        // Q of the next unit, each tile once the current unit's last S
        // product of that tile is done
        if (nxt.hi0 > 0) {
          if (nq0 > 0 && !(ok = wait1(&bars.q_empty[0], (nq0 - 1) & 1, wc, ERR_WAIT_LOAD))) break;
          load_q(nxt, 0);
        }
        if (nxt.hi1 > 0) {
          if (nq1 > 0 && !(ok = wait1(&bars.q_empty[1], (nq1 - 1) & 1, wc, ERR_WAIT_LOAD))) break;
          load_q(nxt, 1);
        }
        cur = nxt;
      }
      // Drain: wait (bounded, ignoring the abort flag) for the last fill of
      // every stage, so that no copy is still landing when the CTA exits.
      const WaitCtx wd{abort_flag, a.err, true};
      if (any0) wait1(bars.k0_full, 0, wd, ERR_WAIT_DRAIN);
      for (int i = max(0, nkv - C::NS); i < nkv; ++i)
        wait1(&bars.kv_full[i % C::NS], (i / C::NS) & 1, wd, ERR_WAIT_DRAIN);
      if (nq0 > 0) wait1(&bars.q_full[0], (nq0 - 1) & 1, wd, ERR_WAIT_DRAIN);
      if (nq1 > 0) wait1(&bars.q_full[1], (nq1 - 1) & 1, wd, ERR_WAIT_DRAIN);
    }
  } else if (warp == C::W_MMA) {
    // ================================================================ MMA issuer
    // (the whole warp, converged; one elected lane issues each instruction)
    constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, false, false);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, D, false, true);   // B = V, MN-major
    const uint64_t qd0 = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
    const uint64_t kd0 = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);
    const uint64_t vd0 = sdesc_sw128(smem_u32(smem + C::OFF_V), C::SUB, 1024);
    auto issue_s = [&](int t, int s) {
      const uint64_t qd = sdesc_offset(qd0, t * C::TILE), kd = sdesc_offset(kd0, s * C::TILE);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk / 4) * C::SUB + (kk % 4) * 32;
        mma_ss_w(tmem + t * 128, sdesc_offset(qd, off), sdesc_offset(kd, off), idesc_s, kk > 0);
      }
    };
    auto issue_pv = [&](int t, int s, bool acc) {
      const uint64_t vd = sdesc_offset(vd0, s * C::TILE);
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk)
        mma_ts_w(tmem + 256 + t * D, tmem + t * 128 + kk * 8, sdesc_offset(vd, kk * 2048), idesc_pv,
                 (acc || kk > 0) ? 1u : 0u);
    };
    int e = 0;   // unit ring entries read
    int nqw0 = 0, nqw1 = 0;   // Q fills waited for, per tile
    int npv0 = 0, npv1 = 0;   // PV products issued, per tile
    int hi0 = u0.hi0, hi1 = u0.hi1;
    bool ok = true;
    // S of the first key tile for each query tile as soon as that tile's Q
    // has landed (the loads go out Q0, K of the first key tile, Q1)
    if (any0) {
      ok = wait_warp(bars.k0_full, 0, wc, ERR_WAIT_MMA);
      if (ok && hi0 > 0 && (ok = wait_warp(&bars.q_full[0], 0, wc, ERR_WAIT_MMA))) {
        ++nqw0;
        tc_fence_after();
        issue_s(0, 0);
        mma_commit_w(&bars.s_full[0]);
        if (hi0 == 1) mma_commit_w(&bars.q_empty[0]);
      }
      if (ok && hi1 > 0 && (ok = wait_warp(&bars.q_full[1], 0, wc, ERR_WAIT_MMA))) {
        ++nqw1;
        tc_fence_after();
        issue_s(1, 0);
        mma_commit_w(&bars.s_full[1]);
        if (hi1 == 1) mma_commit_w(&bars.q_empty[1]);
      }
      if (ok) mma_commit_w(bars.k0_empty);
    }
    int G = 0;   // first step of the current unit
    while (ok) {
      const int n = max(hi0, hi1);
      int nid = -1, nhi0 = 0, nhi1 = 0;
      auto next_unit = [&]() -> bool {
        const int sl = e & 1;
        if (!wait_warp(&bars.unit_full[sl], (e >> 1) & 1, wc, ERR_WAIT_MMA)) return false;
        nid = *reinterpret_cast<volatile int*>(ring + sl * 32 + 28);
        if (nid >= 0) {
          const PUnit nu = *reinterpret_cast<const PUnit*>(ring + sl * 32);
          nhi0 = nu.hi0;
          nhi1 = nu.hi1;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.unit_empty[sl]);
        ++e;
        return true;
      };
      if (n == 0) ok = next_unit();
      for (int i = 0; i < n && ok; ++i) {
        const int g = G + i, s = g % C::NS, s1 = (g + 1) % C::NS;
        // V_g and K_{g+1}
        if (!(ok = wait_warp(&bars.kv_full[s], (g / C::NS) & 1, wc, ERR_WAIT_MMA))) break;
        if (i == n - 1 && !(ok = next_unit())) break;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int hit = t ? hi1 : hi0;
          if (i < hit) {
            // (the first PV of a unit overwrites O: its softmax warps arrive on
            // P of the unit's first key tile only after their epilogue of the
            // previous unit has read O out of TMEM)
            if (!(ok = wait_warp(&bars.p_full[t], (t ? npv1 : npv0) & 1, wc, ERR_WAIT_MMA))) break;
            tc_fence_after();
            issue_pv(t, s, i > 0);
            if (t) ++npv1; else ++npv0;
            mma_commit_w(&bars.o_done[t]);
          }
          if (i + 1 < n) {
            if (i + 1 < hit) {
              issue_s(t, s1);
              mma_commit_w(&bars.s_full[t]);
              if (i + 2 == hit) mma_commit_w(&bars.q_empty[t]);   // the tile's last S
            }
          } else if (nid >= 0 && (t ? nhi1 : nhi0) > 0) {
            // S of the next unit's first key tile (its K came with this step's V)
            if (!(ok = wait_warp(&bars.q_full[t], (t ? nqw1 : nqw0) & 1, wc, ERR_WAIT_MMA))) break;
            if (t) ++nqw1; else ++nqw0;
            tc_fence_after();
            issue_s(t, s1);
            mma_commit_w(&bars.s_full[t]);
            if ((t ? nhi1 : nhi0) == 1) mma_commit_w(&bars.q_empty[t]);
          }
        }
        if (!ok) break;
        mma_commit_w(&bars.kv_empty[s]);
      }
      G += n;
      if (!ok || nid < 0) break;
      hi0 = nhi0;
      hi1 = nhi1;
    }
    // drain every MMA issued so far before TMEM is released
    if (any0 || G > 0) {
      mma_commit_w(bars.drain);
      wait_warp(bars.drain, 0, WaitCtx{abort_flag, a.err, true}, ERR_WAIT_DRAIN);
    }
  } else {
    // ================================================================ softmax
    const int t = warp / 4;                 // query tile of this warpgroup
    const int r = (warp % 4) * 32 + lane;   // row within the tile = TMEM lane
    const int wq = warp & 3;                // TMEM lane quarter of this warp
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t s_col = t * 128, o_col = 256 + t * D;
    const float sl2 = p.scale * kLog2e;
    const long off = (long)Nk - Nq;
    uint8_t* wst = smem + C::OFF_OST + t * (kBM * 128) + wq * 4096;   // this warp's staging slice
    int e = 0;   // unit ring entries read
    int c = 0;   // S tiles of this warpgroup so far (over all units)
    int bh = u0.bh, q_base = u0.q_base, n_t = t ? u0.hi1 : u0.hi0;
    for (;;) {
      const int r0 = q_base + t * kBM;
      const int row_g = r0 + r;
      // last visible key of this row / of the tile's first row (tile-uniform)
      const long lim_row = CAUSAL ? min((long)row_g + off, (long)Nk - 1) : (long)Nk - 1;
      const long lim_tile = CAUSAL ? min((long)r0 + off, (long)Nk - 1) : (long)Nk - 1;
      float m = -INFINITY, l = 0.f;
      int i = 0;
      for (; i < n_t; ++i) {
        const int ci = c + i;   // this S tile's count, for the barrier phases
        const int key0 = i * kBN;
        if (!wait_warp(&bars.s_full[t], ci & 1, wc, ERR_WAIT_SOFTMAX)) break;
        tc_fence_after();
        float s[kBN];
        uint32_t* su = reinterpret_cast<uint32_t*>(s);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(lane_base + s_col + cc * 32, su + cc * 32);
        tmem_ld_wait();

        const bool need_mask = (long)key0 + kBN - 1 > lim_tile;
        // Scores in pairs with the packed f32x2 instructions, the row max with
        // the three-input max: about three instructions per score in total.
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (need_mask) {
          const long lim_rel = lim_row - key0;
          const uint64_t sl2x2 = f2_pack(sl2, sl2), z2 = f2_pack(0.f, 0.f);
#pragma unroll
          for (int cc = 0; cc < kBN; cc += 2) {
            float v0, v1;
            f2_unpack(fma2(f2_pack(s[cc], s[cc + 1]), sl2x2, z2), v0, v1);
            if (cc > lim_rel) v0 = -INFINITY;
            if (cc + 1 > lim_rel) v1 = -INFINITY;
            s[cc] = v0;
            s[cc + 1] = v1;
            m4[(cc / 2) & 3] = fmax3(m4[(cc / 2) & 3], v0, v1);
          }
        } else {
#pragma unroll
          for (int cc = 0; cc < kBN; cc += 2) m4[(cc / 2) & 3] = fmax3(m4[(cc / 2) & 3], s[cc], s[cc + 1]);
        }
        float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        if (!need_mask) mx *= sl2;
        // conditional move of the running max
        float alpha = 1.f;
        bool moved = false;
        if (mx > m + kRescaleLog2 || (m == -INFINITY && mx > -INFINITY)) {
          alpha = ex2(m - mx);   // m = -inf -> 0
          moved = (m != -INFINITY);
          m = mx;
        }
        const float mu = (m == -INFINITY) ? 0.f : m;
        // p = exp2(s * scale*log2e - mu) (or exp2(s - mu) for masked tiles,
        // already in the base-2 domain), as one packed FMA per pair
        const uint64_t mul2 = need_mask ? f2_pack(1.f, 1.f) : f2_pack(sl2, sl2);
        const uint64_t nmu2 = f2_pack(-mu, -mu);
        uint64_t ps2[4] = {0ull, 0ull, 0ull, 0ull};   // row sum as 4 packed partial sums
#pragma unroll
        for (int c0 = 0; c0 < kBN; c0 += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int cc = 0; cc < 32; cc += 2) {
            float x0, x1;
            f2_unpack(fma2(f2_pack(s[c0 + cc], s[c0 + cc + 1]), mul2, nmu2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            ps2[(cc / 2) & 3] = add2(ps2[(cc / 2) & 3], f2_pack(p0, p1));
            pk[cc / 2] = pack_bf16x2(p0, p1);
          }
          tmem_st16(lane_base + s_col + c0 / 2, pk);
        }
        float ps[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) f2_unpack(ps2[q], ps[2 * q], ps[2 * q + 1]);
        const float psum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
        l = l * alpha + psum;
        // rescale O if any row of this warp moved its max and O already holds data
        if (__any_sync(0xffffffffu, moved) && i > 0) {
          if (!wait_warp(&bars.o_done[t], (ci - 1) & 1, wc, ERR_WAIT_SOFTMAX)) break;
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t ov[32];
            tmem_ld32(lane_base + o_col + c0, ov);
            tmem_ld_wait();
#pragma unroll
            for (int cc = 0; cc < 32; ++cc) ov[cc] = __float_as_uint(__uint_as_float(ov[cc]) * alpha);
            tmem_st32(lane_base + o_col + c0, ov);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(&bars.p_full[t]);
      }
      // ---- epilogue: O = O_acc / l (bf16), LSE = ln2 * (m + log2 l)
      const bool completed = (i == n_t);   // warp-uniform
      bool have_o = completed && n_t > 0;
      if (have_o) {
        if (!wait_warp(&bars.o_done[t], (c + n_t - 1) & 1, wc, ERR_WAIT_SOFTMAX)) have_o = false;
        tc_fence_after();
      }
      const bool do_epi = completed && r0 < Nq;   // warp-uniform
      const float inv = l > 0.f ? 1.f / l : 0.f;
      // Each warp its own 32 rows (its TMEM lane quarter), one 64-column box
      // at a time: out of TMEM (O stays there until this warp arrives on P of
      // the next unit's first key tile), staged in the warp's 4 KiB slice
      // (16-byte pieces XOR-swizzled by row against bank conflicts), then
      // written with coalesced 16-byte stores, eight lanes per 128-byte row
      // segment. No barrier beyond the warp: the epilogue is on the path to
      // the next unit's first P.
      uint16_t* orow0 = a.o + ((size_t)bh * Nq + r0 + wq * 32) * D;
      const int rows_left = Nq - (r0 + wq * 32);   // rows of this warp inside the problem
#pragma unroll
      for (int cb = 0; cb < D / 64; ++cb) {
        uint32_t ov[64];
        if (have_o) {
          tmem_ld32(lane_base + o_col + cb * 64, ov);
          tmem_ld32(lane_base + o_col + cb * 64 + 32, ov + 32);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int cc = 0; cc < 64; ++cc) ov[cc] = 0u;
        }
        __syncwarp();   // every lane is done with the previous box
        if (do_epi) {
          uint8_t* rowp = wst + lane * 128;
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4) {
            const uint32_t* x = ov + v4 * 8;
            const uint4 w = make_uint4(
                pack_bf16x2(__uint_as_float(x[0]) * inv, __uint_as_float(x[1]) * inv),
                pack_bf16x2(__uint_as_float(x[2]) * inv, __uint_as_float(x[3]) * inv),
                pack_bf16x2(__uint_as_float(x[4]) * inv, __uint_as_float(x[5]) * inv),
                pack_bf16x2(__uint_as_float(x[6]) * inv, __uint_as_float(x[7]) * inv));
            *reinterpret_cast<uint4*>(rowp + ((v4 ^ (lane & 7)) * 16)) = w;
          }
        }
        __syncwarp();   // the box is staged
        if (do_epi) {
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int row = it * 4 + lane / 8, q16 = lane % 8;
            if (row < rows_left) {
              const uint4 v = *reinterpret_cast<const uint4*>(wst + row * 128 + ((q16 ^ (row & 7)) * 16));
              *reinterpret_cast<uint4*>(orow0 + (size_t)row * D + cb * 64 + q16 * 8) = v;
            }
          }
        }
      }
      if (do_epi && row_g < Nq) {
        const float lse_v = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        float* dst = a.lse + (size_t)bh * Nq + row_g;
        if (dst == reinterpret_cast<float*>(a.sched))
          store_counter_lse(a, lse_v, wc);
        else
          *dst = lse_v;
      }
      if (!completed) break;
      c += n_t;
      // the CTA's next unit
      const int sl = e & 1;
      if (!wait_warp(&bars.unit_full[sl], (e >> 1) & 1, wc, ERR_WAIT_SOFTMAX)) break;
      const int nid = *reinterpret_cast<volatile int*>(ring + sl * 32 + 28);
      if (nid >= 0) {
        const PUnit nu = *reinterpret_cast<const PUnit*>(ring + sl * 32);
        bh = nu.bh;
        q_base = nu.q_base;
        n_t = t ? nu.hi1 : nu.hi0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.unit_empty[sl]);
      ++e;
      if (nid < 0) break;
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

template <int D, bool CAUSAL, bool BIAS, bool PERSIST>
__global__ void __launch_bounds__(FwdCfg<D, false, PERSIST>::NT, 1) fwd_bf16_kernel(const __grid_constant__ FwdBf16Args a) {
  if constexpr (PERSIST)
    fwd_body_persistent<D, CAUSAL>(a);
  else
    fwd_body_one<D, CAUSAL, BIAS, false>(a);
}

// The same forward on e4m3 operands (kind::f8f6f4 MMAs at twice the bf16
// rate): S from e4m3 Q, K with per-head scales, P rounded to e4m3 for PV.
template <int D, bool CAUSAL, bool BIAS>
__global__ void __launch_bounds__(FwdCfg<D, true, false>::NT, 1) fwd_fp8_kernel(const __grid_constant__ FwdBf16Args a) {
  fwd_body_one<D, CAUSAL, BIAS, true>(a);
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

// SMs of the current device (cached per device).
int sm_count() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

// The persistent form (one CTA per SM, further units claimed from a counter in
// the LSE word of the last unit's first row) is used for dense bf16 problems
// without a key bias or split, with more units (query-tile pairs x heads)
// than SMs and key tiles in every unit (so that each unit's first K tile can
// be loaded with the previous unit's last step). Measured against one unit
// per CTA on a GB300: non-causal B=2 H=32 N=8192 d=128 1.36 -> 1.27 ms,
// B=4 H=16 N=2048 d=64 100 -> 91 us; causal B=4 H=16 N=4096 d=128
// 203 -> 200 us, B=4 H=16 N=2048 d=64 61 -> 59 us, but B=2 H=32 N=8192
// d=128 (13.5 units per SM) 707 -> 713 us, hence the causal limit below.
bool use_persistent(const FwdBf16Args& b, long units, int sms) {
  const Problem& p = b.p;
  const bool steps_everywhere =   // the first query-tile pair sees a key
      p.Nk >= 1 && (!p.causal || (long)std::min(2 * kBM - 1, p.Nq - 1) + p.Nk - p.Nq >= 0);
  // causal: up to 8 units per SM (the per-unit transition then costs less
  // than one CTA per unit; at 13.5 per SM it cost 1% more)
  const bool few = !p.causal || units <= 8L * sms;
  return sms > 0 && units > sms && units - sms < (1L << 22) && b.bias == nullptr &&
         p.cu_q == nullptr && b.n_split <= 1 && b.lse != nullptr && steps_everywhere && few;
}

template <int D, bool CAUSAL, bool BIAS, bool PERSIST>
cudaError_t launch_kernel(const FwdBf16Args& b, dim3 grid, cudaStream_t s) {
  using C = FwdCfg<D, false, PERSIST>;
  auto kern = fwd_bf16_kernel<D, CAUSAL, BIAS, PERSIST>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  kern<<<grid, C::NT, C::SMEM_ALLOC, s>>>(b);
  return cudaGetLastError();
}

template <int D, bool CAUSAL, bool BIAS>
cudaError_t launch_one(const FwdBf16Args& a, cudaStream_t s) {
  const long BH = (long)a.p.B * a.p.H;
  const long n_pairs = (a.p.Nq + 2 * kBM - 1) / (2 * kBM);
  const long units = BH * n_pairs;
  // heads per ordering group: K and V of a group within ~48 MiB of L2
  const long kv_bytes = 2L * a.p.Nk * D * 2;
  FwdBf16Args b = a;
  b.head_group = (int)std::max(1L, std::min(BH, (48L << 20) / std::max(kv_bytes, 1L)));
  b.sched = nullptr;
  b.n_units = (int)units;
  cudaError_t e;
  if constexpr (!BIAS) {
    const int sms = sm_count();
    if (use_persistent(b, units, sms)) {
      b.sched = reinterpret_cast<uint32_t*>(b.lse + (size_t)(BH - 1) * a.p.Nq);
      if ((e = cudaMemsetAsync(b.sched, 0xFF, sizeof(uint32_t), s)) != cudaSuccess) return e;
      return launch_kernel<D, CAUSAL, false, true>(b, dim3((unsigned)sms), s);
    }
  }
  e = launch_kernel<D, CAUSAL, BIAS, false>(b, dim3((unsigned)units, (unsigned)std::max(1, a.n_split)), s);
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
  using C = FwdCfg<128, true, false>;
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
  b.sched = nullptr;   // one unit per CTA
  b.n_units = (int)(BH * n_pairs);
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
