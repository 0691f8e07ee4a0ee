// bf16 backward on the 5th-generation tensor cores.
//
// Three launches on the caller's stream ("flash-attention", Part VII;
// "FlashAttention, Explained", §17; "Understanding FlashAttention Pt 1", §3.6):
//
//  1. bwd_pre: D_i = rowsum(dO_i o O_i) in fp32, LSE converted to the base-2
//     domain (a fully masked row's -inf becomes +inf so that its recomputed
//     probabilities are exactly 0), and the fp32 dQ accumulator zeroed.
//  2. bwd_main: one work item per (128-key tile j, key/value head), taken by
//     a persistent CTA (one per SM); the key/value tile stays resident in
//     shared memory while the item walks the 128-row query tiles i that see j
//     (causal: only i at or below the bottom-right diagonal) and per tile
//       S^T  = K_j Q_i^T                      tcgen05 -> TMEM (lane = key)
//       P^T  = exp2(S^T*c + bias - LSE_i)     recomputed from the saved LSE
//       dP^T = V_j dO_i^T                      tcgen05 -> TMEM
//       dV_j += P^T dO_i                       A = P^T read from TMEM
//       dS^T = P^T o (dP^T - D_i)              -> shared memory (bf16)
//       dK_j += dS^T Q_i                       A = dS^T from shared memory
//       dQ_i  = dS K_j                         A = dS from shared memory
//     dQ_i is reduce-added (TMA bulk tensor reductions) into the accumulator, because
//     several key tiles contribute to the same query rows; dK_j and dV_j stay
//     in TMEM until the last query tile and are written once, scaled.
//  3. bwd_post: dQ = bf16(accumulator).
//
// Deterministic variant (DET): bwd_main runs without the dQ product; dS^T
// goes to TMEM as packed bf16 (next to P^T's place, in the dP^T columns) and
// dK += dS^T Q reads it from there like dV reads P^T. dQ is then formed by
// the query-outer kernel of bwd_dq_tc.cu, which sums the key tiles in a fixed
// order; there is no accumulator to zero and no bwd_post. dO is double-buffered
// in the shared memory the dS and staging buffers used.
//
// Warp roles of bwd_main (512 threads): warps 0-7 are two warpgroups that
// split the query columns of every tile; they compute P^T (kept in fp32
// registers) and dS^T (thread = key = TMEM lane) and write dK/dV at the end
// of an item; warps 8-11 read dQ_i out of TMEM (thread = query row), stage it
// in shared memory and reduce-add it into global memory; warp 12 fetches work
// items and issues TMA loads; warp 13 allocates TMEM and issues the MMAs.
// The deterministic form has no dQ warps (320 threads: TMA warp 8, MMA 9).
// TMEM (512 columns): S^T [0,128), then per half h of the query columns the
// packed bf16 P^T in [64h, 64h+32) (each warpgroup overwrites only scores it
// has already read); dP^T then dQ [128,256); dV [256,256+D); dK [256+D,256+2D).
// dS^T goes to shared memory only: it is the A operand of both dK (K-major
// view) and dQ (MN-major view), so the S^T columns are free as soon as dV has
// read P^T, and S^T of the next tile overlaps dK and dQ of this one.
#include <algorithm>
#include <cmath>
#include <cstdint>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kT = 128;   // keys per key tile = rows per query tile
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ preprocess
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const uint16_t* __restrict__ o,
                                                      const uint16_t* __restrict__ dO,
                                                      const float* __restrict__ lse,
                                                      float* __restrict__ Dv,
                                                      float* __restrict__ lse2,
                                                      float* __restrict__ dq_acc,
                                                      const Problem p, int nq_pad,
                                                      uint32_t* err) {
  // Statistics are laid out per (sequence, head) with nq_pad (a multiple of
  // 128) rows, so that every 128-row tile of them is one aligned 512-byte
  // block. They are stored in the form the main loops use them: -scale * D
  // (dS = P o (scale * dP - scale * D) is then one fused multiply-add and a
  // multiply, and comes out already scaled for dK and dQ) and -LSE * log2(e)
  // (added to the base-2 score). Padding rows and rows that see no key get 0
  // and -inf: their recomputed P is exactly 0.
  constexpr int LPR = D / 8;          // lanes per row, 8 bf16 (16 B) per lane
  constexpr int RPW = 32 / LPR;       // rows per warp and unrolled step
  constexpr int U = 4;                // unrolled steps: U rows' loads in flight per lane
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, li = lane % LPR;
  const long warp_g = ((long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const long nwarps = ((long)gridDim.x * blockDim.x) / 32;
  const long prows = (long)p.B * p.H * nq_pad;
  for (long r0 = warp_g * RPW * U; r0 < prows; r0 += nwarps * RPW * U) {
    uint4 av[U], gv[U];
    float L[U];
    long row[U];
    bool valid[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long pr = r0 + u * RPW + sub;   // padded statistics row
      const bool in = pr < prows;
      const int bh = (int)(min(pr, prows - 1) / nq_pad);
      const int i = (int)(pr - (long)bh * nq_pad);
      const SeqView sv = seq_view(p, bh / p.H, bh % p.H);
      if (in && i == 0 && sv.bad) atomicOr(err, ERR_BAD_SEQLEN);
      valid[u] = in && i < sv.len_q;
      row[u] = (long)sv.hq * sv.qrows + sv.q_off + i;   // row of O, dO, LSE, dQ accumulator
      av[u] = gv[u] = make_uint4(0u, 0u, 0u, 0u);
      L[u] = -INFINITY;
      if (valid[u]) {
        av[u] = reinterpret_cast<const uint4*>(o + row[u] * D)[li];
        gv[u] = reinterpret_cast<const uint4*>(dO + row[u] * D)[li];
        if (li == 0) L[u] = lse[row[u]];
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long pr = r0 + u * RPW + sub;
      const uint32_t a4[4] = {av[u].x, av[u].y, av[u].z, av[u].w};
      const uint32_t g4[4] = {gv[u].x, gv[u].y, gv[u].z, gv[u].w};
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(__uint_as_float(a4[e] << 16), __uint_as_float(g4[e] << 16), acc);
        acc = fmaf(__uint_as_float(a4[e] & 0xffff0000u), __uint_as_float(g4[e] & 0xffff0000u),
                   acc);
      }
      if (valid[u] && dq_acc) {
        float4* z = reinterpret_cast<float4*>(dq_acc + row[u] * D);
        z[2 * li] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[2 * li + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int w = LPR / 2; w >= 1; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
      if (pr < prows && li == 0) {
        Dv[pr] = valid[u] ? -p.scale * acc : 0.f;
        lse2[pr] = (L[u] == -INFINITY) ? -INFINITY : -L[u] * kLog2e;
      }
    }
  }
}

// ------------------------------------------------------------------ post
__global__ void __launch_bounds__(256) bwd_post_kernel(const float* __restrict__ acc,
                                                       uint16_t* __restrict__ dq, long n8) {
  // groups of eight values (two float4 loads, one 16-byte store), four
  // groups (eight loads) in flight per thread
  constexpr int U = 4;
  const long stride = (long)gridDim.x * blockDim.x;
  const float4* a4 = reinterpret_cast<const float4*>(acc);
  for (long i0 = (long)blockIdx.x * blockDim.x + threadIdx.x; i0 < n8; i0 += stride * U) {
    float4 v[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long i = i0 + u * stride;
      if (i < n8) {
        v[u][0] = a4[2 * i];
        v[u][1] = a4[2 * i + 1];
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long i = i0 + u * stride;
      if (i < n8)
        reinterpret_cast<uint4*>(dq)[i] =
            make_uint4(pack_bf16x2(v[u][0].x, v[u][0].y), pack_bf16x2(v[u][0].z, v[u][0].w),
                       pack_bf16x2(v[u][1].x, v[u][1].y), pack_bf16x2(v[u][1].z, v[u][1].w));
    }
  }
}

// ------------------------------------------------------------------ main
template <int D, bool DET>
struct BwdCfg {
  static constexpr int TILE = kT * D * 2;     // bf16 [128][D]
  static constexpr int SUB = kT * 128;        // one 64-column box
  static constexpr int ND = DET ? 2 : 1;      // dO stages
  // reduction form at d = 64: dQ issued before dK, and the next step's Q and
  // dO prefetched into L2 (measured faster together; each alone, and both
  // at d = 128, slower)
  static constexpr bool DQ_FIRST = !DET && D == 64;
  // Threads and roles. Reduction form: warps 0-7 P and dS, 8-11 the dQ
  // read-out (one per TMEM lane quarter), 12 TMA, 13 MMA, 14-15 idle (they
  // complete the last warpgroup for the register split); deterministic
  // form (no dQ): warps 0-7 P and dS, 8 TMA, 9 MMA.
  static constexpr int NT = DET ? 320 : 512;
  static constexpr int W_PROD = DET ? 8 : 12, W_MMA = DET ? 9 : 13;
  // register split of the reduction form: the launch gives 512 x 128;
  // warpgroups 0-2 take 144 each, warpgroup 3 (TMA, MMA, idle) gives up to 80
  static constexpr int REG_HI = 144, REG_LO = 80;
  static_assert(DET || 3 * 128 * REG_HI + 128 * REG_LO == 512 * 128, "register split");
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_Q = OFF_V + TILE;         // [2 stages]
  static constexpr int OFF_DO = OFF_Q + 2 * TILE;    // [ND stages]
  static constexpr int OFF_DQST = OFF_DO + ND * TILE;               // 32 KiB: second dQ staging slice
  static constexpr int OFF_DS = OFF_DQST + (DET ? 0 : 32768);       // dS^T boxes
  // per Q stage: base-2 LSE [128] then D [128] of the tile's rows (TMA)
  static constexpr int OFF_STAT = OFF_DS + (DET ? 0 : kT * kT * 2);
  static constexpr int OFF_BAR = OFF_STAT + 2 * 2 * kT * 4;
  static constexpr int NBAR = 20 + 2 * ND;   // see BwdBars
  // dK/dV write-out of an item: both tiles staged at once, dV in the dS
  // buffer and (reduction form, d = 128) dK in the Q stage of the item's last
  // tile, which the item no longer reads; at d = 64 both fit the dS buffer;
  // the deterministic form stages them in the Q stages (one item per CTA)
  static constexpr bool DK_IN_Q = !DET && 2 * TILE > 32768;
  static constexpr int OFF_SCALARS = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_SCALARS + 16 + 2 * 64;   // flags, then the work-item ring
  static_assert(BYTES <= 232448, "shared memory per CTA");
};

// The kernel's mbarriers: one array in shared memory, each barrier at a fixed
// index (addresses computed at each use from the one base, rather than kept
// as separate pointers across the whole kernel).
template <int ND>
struct BwdBars {
  uint64_t* b;
  // K, V of the current item landed / every MMA of an item done (its K/V
  // free, dK and dV final)
  __device__ __forceinline__ uint64_t* kv_full() const { return b; }
  __device__ __forceinline__ uint64_t* kv_empty() const { return b + 1; }
  // [2] Q_i with its statistics in a stage / the stage free
  __device__ __forceinline__ uint64_t* q_full() const { return b + 2; }
  __device__ __forceinline__ uint64_t* q_empty() const { return b + 4; }
  // [ND] dO_i landed / free
  __device__ __forceinline__ uint64_t* do_full() const { return b + 6; }
  __device__ __forceinline__ uint64_t* do_empty() const { return b + 6 + ND; }
  // S^T done; dP^T done; P^T in TMEM, dS^T written (one arrival per P/dS
  // warp); dQ_i done; dQ_i read out of TMEM (one arrival per dQ warp);
  // every MMA of the CTA done
  __device__ __forceinline__ uint64_t* s_full() const { return b + 6 + 2 * ND; }
  __device__ __forceinline__ uint64_t* dp_full() const { return b + 7 + 2 * ND; }
  __device__ __forceinline__ uint64_t* p_full() const { return b + 8 + 2 * ND; }
  __device__ __forceinline__ uint64_t* ds_full() const { return b + 9 + 2 * ND; }
  __device__ __forceinline__ uint64_t* dq_full() const { return b + 10 + 2 * ND; }
  __device__ __forceinline__ uint64_t* dq_empty() const { return b + 11 + 2 * ND; }
  __device__ __forceinline__ uint64_t* drain() const { return b + 12 + 2 * ND; }
  // [2] work-item ring: item written / read by every consumer warp
  __device__ __forceinline__ uint64_t* sched_full() const { return b + 13 + 2 * ND; }
  __device__ __forceinline__ uint64_t* sched_empty() const { return b + 15 + 2 * ND; }
  // barrier of the P/dS warps (one arrival per warp)
  __device__ __forceinline__ uint64_t* cw() const { return b + 17 + 2 * ND; }
  // reduction form, once per item: its dK/dV staged by the P/dS warps (one
  // arrival per warp); the staging read by the TMA stores (one arrival, from
  // the TMA warp)
  __device__ __forceinline__ uint64_t* epi_staged() const { return b + 18 + 2 * ND; }
  __device__ __forceinline__ uint64_t* epi_read() const { return b + 19 + 2 * ND; }
};


// ------------------------------------------------------------------ work items
// A work item is one (key/value head, key tile). Items are numbered in this
// order: heads in groups of a.head_group whose Q, dO (and dQ accumulator)
// stay in L2 together; within a group, key tile by key tile over the group's
// heads, low key tiles (the most query tiles under a causal mask) first, so
// that the last items to start are the short ones.
struct BwdItem {
  int b, h_q0, grp, key0, Nq, Nk, i0, nqh;
  int rot;    // the query tiles are walked from i0 + rot, wrapping around
  int n;      // query-tile steps: every query head of the group x query tiles [i0, n_qt)
  long off;   // Nk - Nq: bottom-right causal alignment
  SeqView sv;
};

template <bool CAUSAL>
__device__ __forceinline__ BwdItem bwd_item(const BwdBf16Args& a, int w) {
  const Problem& p = a.p;
  BwdItem t;
  const int n_kt = (p.Nk + kT - 1) / kT;
  const int BHkv = p.B * p.Hkv;
  const int G = a.head_group;
  const int g0 = (int)(w / ((long)G * n_kt)) * G;
  const int gsz = min(G, BHkv - g0);
  const int rr = (int)(w - (long)g0 * n_kt);
  const int bh_kv = g0 + rr % gsz;
  t.b = bh_kv / p.Hkv;
  t.grp = p.H / p.Hkv;
  t.h_q0 = (bh_kv % p.Hkv) * t.grp;   // first query head of the group
  // rows and lengths of this sequence (keys and queries numbered from 0 in it)
  t.sv = seq_view(p, t.b, t.h_q0);
  t.Nq = t.sv.len_q;
  t.Nk = t.sv.len_k;
  t.key0 = (rr / gsz) * kT;
  t.off = (long)t.Nk - t.Nq;
  // query tiles [i0, n_qt) can see this key tile
  const int n_qt = (t.Nq + kT - 1) / kT;
  t.i0 = 0;
  if (CAUSAL) {
    // smallest i with i*128 + 127 + off >= key0
    const long need = (long)t.key0 - t.off - (kT - 1);
    t.i0 = need <= 0 ? 0 : (int)min((long)n_qt, (need + kT - 1) / kT);
  }
  t.nqh = n_qt - t.i0;
  // Without a causal mask every key tile of a head walks the same query
  // tiles; starting each at a different one keeps the items of a head that
  // run at the same time from reduce-adding into the same dQ rows at once.
  // (Under a causal mask the items start at their diagonal tiles already.)
  t.rot = CAUSAL ? 0 : (t.key0 / kT) % max(t.nqh, 1);
  t.n = t.key0 < t.Nk ? max(0, t.nqh) * t.grp : 0;
  return t;
}

// A slot of the work-item ring in shared memory: the item and what the loops
// of the MMA and P/dS warps need of it, decoded once by the TMA warp.
struct BwdSlot {
  int w;          // item index; -1: no more items
  int n;          // query-tile steps (0: nothing to compute, dK = dV = 0)
  int i0, nqh;    // query tiles [i0, i0 + nqh) of each query head (nqh >= 1)
  int rot;        // first query tile walked: i0 + rot (then wrapping around)
  int off;        // Nk - Nq of the sequence
  int key0;       // first key of the tile
  int qc0;        // coordinate of the group's first query head in q / dO / dq
  int q_off;      // first row of the sequence
  int nk;         // keys of the sequence
  int bias_row;   // b * Nk: the sequence's row of the key bias
  int g0;         // global index of the item's first query-tile step
  int kph;        // ordinal of the item among the CTA's items with n > 0
};
static_assert(sizeof(BwdSlot) <= 64, "two ring slots fit the 128 bytes after the flags");

// Warp-collective: whether any key of the item's tile has a finite bias (a
// tile whose keys are all masked out contributes nothing: dK = dV = 0).
__device__ __forceinline__ bool bwd_item_any_key(const BwdBf16Args& a, const BwdItem& t) {
  bool any = false;
#pragma unroll
  for (int m = 0; m < kT / 32; ++m) {
    const int key = t.key0 + m * 32 + (int)lane_id();
    if (key < t.Nk && a.bias[(size_t)t.b * t.Nk + key] * kLog2e != -INFINITY) any = true;
  }
  return __any_sync(0xffffffffu, any);
}

// The main backward kernel. The non-deterministic form is persistent: one
// CTA per SM takes work items in order from a counter in the workspace
// (the TMA warp fetches them and passes them to the MMA warp and the P/dS
// warps through a two-slot ring in shared memory), and every barrier phase
// and ring stage runs on across items. So the next item's K/V and first Q,
// dO tiles load, and its first S^T and dP^T products run, while the P/dS
// warps write out the previous item's dK and dV. The deterministic form
// (dS^T through TMEM, no dQ) takes one item per CTA, the CTA's index.
template <int D, bool CAUSAL, bool BIAS, bool DET>
__global__ void __launch_bounds__(BwdCfg<D, DET>::NT, 1) bwd_main_kernel(const __grid_constant__ BwdBf16Args a) {
  using C = BwdCfg<D, DET>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const Problem& p = a.p;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;

  const BwdBars<C::ND> bars{reinterpret_cast<uint64_t*>(smem + C::OFF_BAR)};
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_SCALARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_SCALARS + 4);
  volatile BwdSlot* slots = reinterpret_cast<volatile BwdSlot*>(smem + C::OFF_SCALARS + 16);   // [2]
  const WaitCtx wc{abort_flag, a.err};
  const int n_items = p.B * p.Hkv * ((p.Nk + kT - 1) / kT);

  if (threadIdx.x == 0) {
    if ((smem_u32(smem) & 1023u) != 0) atomicOr(a.err, ERR_WAIT_DRAIN);   // layout invariant
    mbar_init(bars.kv_full(), 1);
    mbar_init(bars.kv_empty(), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.q_full()[s], 1);
      mbar_init(&bars.q_empty()[s], 1);
      mbar_init(&bars.sched_full()[s], 1);
      // the MMA warp, each P/dS warp and each dQ warp
      mbar_init(&bars.sched_empty()[s], 1 + 2 * kT / 32 + (DET ? 0 : 4));
    }
    for (int s = 0; s < C::ND; ++s) {
      mbar_init(&bars.do_full()[s], 1);
      mbar_init(&bars.do_empty()[s], 1);
    }
    mbar_init(bars.s_full(), 1);
    mbar_init(bars.dp_full(), 1);
    mbar_init(bars.p_full(), 2 * kT / 32);    // one arrival per compute warp
    mbar_init(bars.ds_full(), 2 * kT / 32);
    mbar_init(bars.dq_full(), 1);
    mbar_init(bars.dq_empty(), 4);            // one arrival per dQ warp
    mbar_init(bars.drain(), 1);
    mbar_init(bars.cw(), 2 * kT / 32);
    mbar_init(bars.epi_staged(), 2 * kT / 32);
    mbar_init(bars.epi_read(), 1);
    *abort_flag = (smem_u32(smem) & 1023u) != 0;
    fence_mbar_init();
  }
  if (warp == C::W_MMA) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // query head (within the batch) and first row of step `lt` of item t, and
  // the head's coordinate in q/dO/dq
  auto q_head = [&](const BwdItem& t, int lt) { return t.h_q0 + lt / max(t.nqh, 1); };
  auto q_coord = [&](const BwdItem& t, int h) { return p.cu_q ? h : t.b * p.H + h; };
  auto q_row0 = [&](const BwdItem& t, int lt) {
    const int nqh = max(t.nqh, 1);
    return (t.i0 + (lt % nqh + t.rot) % nqh) * kT;
  };

  if (warp >= C::W_PROD) {
  if constexpr (!DET) setmaxnreg_dec<C::REG_LO>();
  if (warp == C::W_PROD) {
    // ================================================================ TMA producer + scheduler
    int g = 0, kph = 0;     // query-tile steps / non-empty items so far
    int nq = 0, nd = 0, nkv = 0;   // Q / dO / K,V fills issued
    bool ok = true;
    // the previous item's dK/dV stores (reduction form): ragged tile (written
    // by the P/dS warps themselves), first key row, key/value head, Q stage
    // holding dK
    bool pv_ragged = false;
    int pv_row = 0, pv_hk = 0, pv_sk = 0;
    for (int u = 0; ok; ++u) {
      int w;
      if (DET) {
        w = u == 0 ? (int)blockIdx.x : -1;
      } else {
        w = lane == 0 ? atomicAdd(a.sched, 1) : 0;
        w = __shfl_sync(0xffffffffu, w, 0);
        if (w >= n_items) w = -1;
      }
      BwdItem t;
      int n = 0;
      if (w >= 0) {
        t = bwd_item<CAUSAL>(a, w);
        n = (!BIAS || bwd_item_any_key(a, t)) ? t.n : 0;
      }
      if (lane == 0) {
        // slot u & 1 is free once item u - 2 is done with it
        if (u >= 2 && !wait1(&bars.sched_empty()[u & 1], ((u >> 1) - 1) & 1, wc, ERR_WAIT_LOAD)) ok = false;
        if (ok) {
          volatile BwdSlot* sl = slots + (u & 1);
          sl->w = w;
          if (w >= 0) {
            sl->n = n;
            sl->i0 = t.i0;
            sl->nqh = max(t.nqh, 1);
            sl->rot = t.rot;
            sl->off = (int)t.off;
            sl->key0 = t.key0;
            sl->qc0 = p.cu_q ? t.h_q0 : t.b * p.H + t.h_q0;
            sl->q_off = t.sv.q_off;
            sl->nk = t.Nk;
            sl->bias_row = t.b * t.Nk;
            sl->g0 = g;
            sl->kph = kph;
          }
          mbar_arrive(&bars.sched_full()[u & 1]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      // step lt's Q (with its statistics) and dO
      auto load_step = [&](int lt) -> bool {
        const int gi = g + lt, s = gi & 1, uq = gi >> 1;
        const int q0 = q_row0(t, lt), hq = q_head(t, lt);
        if (C::DQ_FIRST && lt + 1 < n) {
          // the next step's Q and dO into L2 (d = 64; at d = 128 the extra
          // requests measured slower)
          const int q1 = q_row0(t, lt + 1), h1 = q_coord(t, q_head(t, lt + 1));
          for (int c = 0; c < D / 64; ++c) {
            tma_prefetch_l2_3d(&a.tm_q, c * 64, t.sv.q_off + q1, h1);
            tma_prefetch_l2_3d(&a.tm_do, c * 64, t.sv.q_off + q1, h1);
          }
        }
        if (uq > 0 && !wait1(&bars.q_empty()[s], (uq - 1) & 1, wc, ERR_WAIT_LOAD)) return false;
        mbar_arrive_expect_tx(&bars.q_full()[s], C::TILE + 2 * kT * 4);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + C::OFF_Q + s * C::TILE + c * C::SUB, &a.tm_q, c * 64, t.sv.q_off + q0,
                      q_coord(t, hq), &bars.q_full()[s]);
        float* st = reinterpret_cast<float*>(smem + C::OFF_STAT) + s * 2 * kT;
        const size_t srow = ((size_t)t.b * p.H + hq) * a.nq_pad + q0;
        bulk_load_1d(st, a.lse2 + srow, kT * 4, &bars.q_full()[s]);
        bulk_load_1d(st + kT, a.D + srow, kT * 4, &bars.q_full()[s]);
        ++nq;
        // dO stage sd may be refilled once dV of its previous tile is done
        const int sd = gi % C::ND, ud = gi / C::ND;
        if (ud > 0 && !wait1(&bars.do_empty()[sd], (ud - 1) & 1, wc, ERR_WAIT_LOAD)) return false;
        mbar_arrive_expect_tx(&bars.do_full()[sd], C::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + C::OFF_DO + sd * C::TILE + c * C::SUB, &a.tm_do, c * 64, t.sv.q_off + q0,
                      q_coord(t, hq), &bars.do_full()[sd]);
        ++nd;
        return true;
      };
      // Reduction form: the TMA stores of the previous item's dK and dV, once
      // the P/dS warps have staged them; then the staging buffers are handed
      // back (the dS buffer to the P/dS warps, the Q stage that held dK to
      // the loads below: it is refilled at the second tile of this item at
      // the earliest, so every load into it follows this).
      auto store_prev = [&]() -> bool {
        if (!wait1(bars.epi_staged(), (u - 1) & 1, wc, ERR_WAIT_LOAD)) return false;
        if (!pv_ragged) {
          uint8_t* st_dk = C::DK_IN_Q ? smem + C::OFF_Q + pv_sk * C::TILE : smem + C::OFF_DS + C::TILE;
          for (int c = 0; c < D / 64; ++c) {
            tma_store_3d(&a.tm_dv, smem + C::OFF_DS + c * C::SUB, c * 64, pv_row, pv_hk);
            tma_store_3d(&a.tm_dk, st_dk + c * C::SUB, c * 64, pv_row, pv_hk);
          }
          bulk_commit_group();
          bulk_wait_group_read0();
        }
        mbar_arrive(bars.epi_read());
        return true;
      };
      if (w < 0) {
        if (!DET && u > 0 && lane == 0 && !*abort_flag) store_prev();
        break;
      }
      if (lane == 0 && !*abort_flag) {
        // the first tile's Q and dO go out before K and V, which wait for
        // the previous item's last product
        if (n > 0) ok = load_step(0);
        if (n > 0 && ok) {
          // K and V of the previous item are free once all of its MMAs are done
          if (kph > 0 && !wait1(bars.kv_empty(), (kph - 1) & 1, wc, ERR_WAIT_LOAD)) ok = false;
          if (ok) {
            mbar_arrive_expect_tx(bars.kv_full(), 2 * C::TILE);
            for (int c = 0; c < D / 64; ++c) {
              tma_load_3d(smem + C::OFF_K + c * C::SUB, &a.tm_k, c * 64, t.sv.k_off + t.key0, t.sv.hk,
                          bars.kv_full());
              tma_load_3d(smem + C::OFF_V + c * C::SUB, &a.tm_v, c * 64, t.sv.k_off + t.key0, t.sv.hk,
                          bars.kv_full());
            }
            ++nkv;
          }
        }
        if (!DET && u > 0 && ok) ok = store_prev();
        for (int lt = 1; lt < n && ok; ++lt) ok = load_step(lt);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if constexpr (!DET) {
        // where this item's dK/dV go and where dK is staged
        pv_ragged = p.cu_k != nullptr && t.key0 + kT > t.Nk;
        pv_row = t.sv.k_off + t.key0;
        pv_hk = t.sv.hk;
        pv_sk = (g + n + 1) & 1;   // the Q stage of the item's last tile
      }
      g += n;
      if (n > 0) ++kph;
    }
    if (lane == 0) {
      // Drain: wait (bounded, ignoring the abort flag) for the last fill of
      // every buffer, so that no copy is still landing when the CTA exits.
      const WaitCtx wd{abort_flag, a.err, true};
      if (nkv > 0) wait1(bars.kv_full(), (nkv - 1) & 1, wd, ERR_WAIT_DRAIN);
      for (int i = max(0, nq - 2); i < nq; ++i) wait1(&bars.q_full()[i & 1], (i >> 1) & 1, wd, ERR_WAIT_DRAIN);
      for (int i = max(0, nd - C::ND); i < nd; ++i)
        wait1(&bars.do_full()[i % C::ND], (i / C::ND) & 1, wd, ERR_WAIT_DRAIN);
      if (!DET) bulk_wait_group0();   // the dK/dV stores are complete
    }
  } else if (warp == C::W_MMA) {
    // ================================================================ MMA issuer
    constexpr uint32_t id_s = idesc_bf16_f32(kT, kT, false, false);    // S^T, dP^T
    constexpr uint32_t id_acc = idesc_bf16_f32(kT, D, false, true);    // dV, dK (A K-major)
    constexpr uint32_t id_dq = idesc_bf16_f32(kT, D, true, true);      // dQ (A = dS, MN-major)
    const uint32_t t_s = tmem, t_dp = tmem + 128, t_dv = tmem + 256, t_dk = tmem + 256 + D;
    // operand descriptors, built once for the start of shared memory: an
    // operand's is this plus its byte offset (K-major boxes read along K:
    // LBO 16; along the 128-row direction: LBO = one box)
    const uint32_t sbase = smem_u32(smem);
    const uint64_t dk16c = sdesc_sw128(sbase, 16, 1024), dsubc = sdesc_sw128(sbase, C::SUB, 1024);
    // the bases passed through an opaque move inside each step, so that the
    // forty descriptors of a step are one add each right where they are
    // used, not values kept in registers across the loop
    auto opaque = [](uint64_t x) {
      asm volatile("" : "+l"(x));
      return x;
    };
    // S^T = K Q^T for global step gi (both K-major, 128-byte rows per box)
    auto issue_s = [&](int gi) {
      const uint32_t q_o = C::OFF_Q + (gi & 1) * C::TILE;
      const uint64_t dk16 = opaque(dk16c);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t o = (kk / 4) * C::SUB + (kk % 4) * 32;
        mma_ss_w(t_s, sdesc_offset(dk16, C::OFF_K + o), sdesc_offset(dk16, q_o + o), id_s, kk > 0);
      }
      mma_commit_w(bars.s_full());
    };
    int g = 0, kph = 0;
    bool ok = true, issued = false;
    for (int u = 0; ok; ++u) {
      if (!wait_warp(&bars.sched_full()[u & 1], (u >> 1) & 1, wc, ERR_WAIT_LOAD)) break;
      const int w = slots[u & 1].w, n = slots[u & 1].n;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.sched_empty()[u & 1]);
      if (w < 0) break;
      if (n == 0) continue;
      {
        // (the whole warp, converged; lane 0 issues each instruction)
        // Issue order per query tile i:  dP(i) [after dQ(i-1) left TMEM],
        // dV(i) [after P(i)], S(i+1) [after Q(i+1) landed; the S columns are
        // free once dV(i) has read P(i)], dK(i) and dQ(i) [after dS(i)].
        // S(i+1) and the softmax of tile i+1 thus overlap dK(i) and dQ(i).
        // dK(i), the last reader of Q(i), goes before dQ(i) so that the load
        // of Q(i+2) into its stage starts a product earlier. The first dV and
        // dK of an item start from zero: the P/dS warps arrive on P of the
        // item's first tile only after they have read the previous item's
        // dK, dV.
        ok = !__any_sync(0xffffffffu, *abort_flag) && wait_warp(bars.kv_full(), kph & 1, wc, ERR_WAIT_MMA) &&
             wait_warp(&bars.q_full()[g & 1], (g >> 1) & 1, wc, ERR_WAIT_MMA);
        if (ok) {
          tc_fence_after();
          issue_s(g);
          issued = true;
        }
        for (int lt = 0; lt < n && ok; ++lt) {
          const int gi = g + lt, s = gi & 1, sd = gi % C::ND;
          const uint32_t q_o = C::OFF_Q + s * C::TILE, do_o = C::OFF_DO + sd * C::TILE;
          const uint64_t dk16 = opaque(dk16c), dsub = opaque(dsubc);
          // dP^T = V dO^T, once dQ of the previous tile has left TMEM (DET: the
          // dS^T of the previous tile in these columns was read by dK, an
          // earlier MMA). dO(i) has usually landed long before: its wait
          // goes first, off the path from dQ(i-1) to dP(i).
          if (!(ok = wait_warp(&bars.do_full()[sd], (gi / C::ND) & 1, wc, ERR_WAIT_MMA))) break;
          if (!DET && gi > 0 && !(ok = wait_warp(bars.dq_empty(), (gi - 1) & 1, wc, ERR_WAIT_MMA))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = (kk / 4) * C::SUB + (kk % 4) * 32;
            mma_ss_w(t_dp, sdesc_offset(dk16, C::OFF_V + o), sdesc_offset(dk16, do_o + o), id_s, kk > 0);
          }
          mma_commit_w(bars.dp_full());
          // dV(i) as soon as P(i) is in TMEM; the wait for Q(i+1), which
          // often lands later than P(i), then runs while dV(i) computes
          if (!(ok = wait_warp(bars.p_full(), gi & 1, wc, ERR_WAIT_MMA))) break;
          tc_fence_after();
          // dV += P^T dO  (P^T packed bf16: query columns [0,64) in TMEM columns
          // [0,32), [64,128) in [64,96))
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_ts_w(t_dv, t_s + (kk / 4) * 64 + (kk % 4) * 8, sdesc_offset(dsub, do_o + kk * 2048), id_acc,
                   (lt > 0 || kk > 0) ? 1u : 0u);
          mma_commit_w(&bars.do_empty()[sd]);   // dV is the last reader of dO(i)
          if (lt + 1 < n) {
            if (!(ok = wait_warp(&bars.q_full()[(gi + 1) & 1], ((gi + 1) >> 1) & 1, wc, ERR_WAIT_MMA))) break;
            tc_fence_after();
            issue_s(gi + 1);
          }
          if (!(ok = wait_warp(bars.ds_full(), gi & 1, wc, ERR_WAIT_MMA))) break;
          tc_fence_after();
          if constexpr (DET) {
            // dK += dS^T Q with dS^T packed in TMEM like P^T (in the dP^T columns)
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk)
              mma_ts_w(t_dk, t_dp + (kk / 4) * 64 + (kk % 4) * 8, sdesc_offset(dsub, q_o + kk * 2048),
                     id_acc, (lt > 0 || kk > 0) ? 1u : 0u);
            mma_commit_w(&bars.q_empty()[s]);
          } else {
            // dK += dS^T Q (A = dS^T: K-major view of the dS boxes), which
            // frees the Q stage, and dQ = dS K. d = 128: dK first, so that
            // the load of Q(i+2) into the stage starts a product earlier;
            // d = 64 (with the next step's Q and dO prefetched into L2, so
            // that their loads land sooner): dQ first, so that its read-out
            // and the next dP start a product earlier.
            auto issue_dk = [&]() {
#pragma unroll
              for (int kk = 0; kk < kT / 16; ++kk)
                mma_ss_w(t_dk, sdesc_offset(dk16, C::OFF_DS + (kk / 4) * C::SUB + (kk % 4) * 32),
                       sdesc_offset(dsub, q_o + kk * 2048), id_acc, (lt > 0 || kk > 0) ? 1u : 0u);
              mma_commit_w(&bars.q_empty()[s]);
            };
            auto issue_dq = [&]() {
#pragma unroll
              for (int kk = 0; kk < kT / 16; ++kk)
                mma_ss_w(t_dp, sdesc_offset(dsub, C::OFF_DS + kk * 2048),
                       sdesc_offset(dsub, C::OFF_K + kk * 2048), id_dq, kk > 0 ? 1u : 0u);
              mma_commit_w(bars.dq_full());
            };
            if constexpr (C::DQ_FIRST) {
              issue_dq();
              issue_dk();
            } else {
              issue_dk();
              issue_dq();
            }
          }
        }
        // every MMA of this item: its K/V buffers are free, dK and dV final
        mma_commit_w(bars.kv_empty());
      }
      g += n;
      ++kph;
    }
    if (issued) {
      mma_commit_w(bars.drain());
      wait_warp(bars.drain(), 0, WaitCtx{abort_flag, a.err, true}, ERR_WAIT_DRAIN);
    }
  }
  } else if (!DET && warp >= 8) {
    // ================================================================ dQ warps 8-11
    setmaxnreg_inc<C::REG_HI>();
    // dQ of every query-tile step (TMEM lane = query row): each warp reads its
    // 32 rows, all D columns, out of TMEM at once (the columns go back to the
    // MMA warp for the next dP), then reduce-adds them into the fp32
    // accumulator with TMA in boxes of 32 rows x 32 columns (4 KiB, 128-byte
    // swizzled) through its 8 KiB slot of the staging buffer (two boxes per
    // bulk group at d = 128, one at d = 64).
    const int qw = warp - 8;   // TMEM lane quarter
    const uint32_t lane_base = tmem + ((uint32_t)(qw * 32) << 16);
    uint8_t* slot = smem + C::OFF_DQST + qw * 8192;
    constexpr int NB = D / 32;   // boxes per row block
    for (int u = 0;; ++u) {
      if (!wait_warp(&bars.sched_full()[u & 1], (u >> 1) & 1, wc, ERR_WAIT_LOAD)) break;
      volatile BwdSlot* cur = slots + (u & 1);
      if (cur->w < 0) break;
      const int n = cur->n, g = cur->g0;
      bool ok = true;
      for (int lt = 0; lt < n && ok; ++lt) {
        const int gi = g + lt;
        if (!(ok = wait_warp(bars.dq_full(), gi & 1, wc, ERR_WAIT_EPILOGUE))) break;
        tc_fence_after();
        uint32_t x[D];
#pragma unroll
        for (int c = 0; c < D; c += 64) tmem_ld64(lane_base + 128 + c, x + c);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive_warp(bars.dq_empty());
        const int nqh = cur->nqh;
        const int row0 = cur->q_off + (cur->i0 + (lt % nqh + cur->rot) % nqh) * kT + qw * 32;
        const int qc = cur->qc0 + lt / nqh;
        if constexpr (D == 64) {
          // one bulk group per box; a box waits only for the box two back
          // (in its half of the slot) to have been read. (At d = 128 this
          // measured slower than the pairs below.)
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            if (lane == 0) bulk_wait_group_read1();
            __syncwarp();
            uint8_t* bx = slot + (b & 1) * 4096;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t* v = x + b * 32 + 4 * k;
              *reinterpret_cast<uint4*>(bx + lane * 128 + ((k ^ (lane & 7)) * 16)) =
                  make_uint4(v[0], v[1], v[2], v[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_3d(&a.tm_dqacc, bx, b * 32, row0, qc);
              bulk_commit_group();
            }
          }
        } else {
#pragma unroll
          for (int b2 = 0; b2 < NB; b2 += 2) {
            if (lane == 0) bulk_wait_group_read0();   // the slot's previous boxes have been read
            __syncwarp();
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const uint32_t* v = x + (b2 + bb) * 32 + 4 * k;
                *reinterpret_cast<uint4*>(slot + bb * 4096 + lane * 128 + ((k ^ (lane & 7)) * 16)) =
                    make_uint4(v[0], v[1], v[2], v[3]);
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
              for (int bb = 0; bb < 2; ++bb)
                tma_reduce_add_3d(&a.tm_dqacc, slot + bb * 4096, (b2 + bb) * 32, row0, qc);
              bulk_commit_group();
            }
          }
        }
      }
      mbar_arrive_warp(&bars.sched_empty()[u & 1]);   // done with the slot
      if (!ok) break;
    }
    // reductions complete before the CTA exits
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  } else {
    // ================================================================ warps 0-7
    if constexpr (!DET) setmaxnreg_inc<C::REG_HI>();
    // Two warpgroups share the 128 keys (thread = key = TMEM lane) and split the
    // 128 query columns of each tile: warpgroup h handles columns [64h, 64h+64)
    // of S^T / P^T / dP^T / dS^T, and columns [h*D/2, (h+1)*D/2) of dK, dV.
    const int h = warp / 4;
    const int r = (warp % 4) * 32 + lane;            // key within the tile = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp % 4) * 32) << 16);
    const float sl2 = p.scale * kLog2e;
    float* stat = reinterpret_cast<float*>(smem + C::OFF_STAT);
    uint8_t* ds_s = smem + C::OFF_DS;
    constexpr int HD = D / 2;      // dK / dV columns per warpgroup
    // the current item: its ring slot (read from shared memory where needed,
    // to keep the tile loop's registers few) and first global step
    volatile BwdSlot* cur = slots;

    // P^T of global step gi = exp2(S^T * scale*log2e + bias - LSE2), masked
    // -> 0, kept in fp32 registers for dS; packed bf16 copy to TMEM for dV.
    float P[64];
    auto compute_p = [&](int gi) -> bool {
      const int q0 = (cur->i0 + ((gi - cur->g0) % cur->nqh + cur->rot) % cur->nqh) * kT;
      const int off = cur->off, key = cur->key0 + r;
      // this tile's base-2 LSE (staged by TMA with Q) for this warpgroup's columns
      if (!wait_warp(&bars.q_full()[gi & 1], (gi >> 1) & 1, wc, ERR_WAIT_SOFTMAX)) return false;
      const float* stl = stat + (gi & 1) * 2 * kT + h * 64;
      if (!wait_warp(bars.s_full(), gi & 1, wc, ERR_WAIT_SOFTMAX)) return false;
      tc_fence_after();
      const bool need_mask = CAUSAL && (q0 + off < key - r + kT - 1);
      // the key's term: its bias (log2 domain), -inf past the end of a ragged tile
      const float kb =
          key < cur->nk ? (BIAS ? a.bias[(size_t)cur->bias_row + key] * kLog2e : 0.f) : -INFINITY;
      const int thr = key - off - q0 - h * 64;   // local column < thr -> masked
      // the second 32 scores load while the first 32 are exponentiated
      uint32_t* sv = reinterpret_cast<uint32_t*>(P);
      tmem_ld32(lane_base + h * 64, sv);
      tmem_ld_wait();
      tmem_ld32(lane_base + h * 64 + 32, sv + 32);
      const uint64_t sl2x2 = f2_pack(sl2, sl2), kb2 = f2_pack(kb, kb);
      // x = S * scale * log2(e) + key bias - LSE * log2(e) (the key term is
      // -inf for a key past the end of a ragged tile)
#pragma unroll
      for (int e = 0; e < 64; e += 4) {
        if (e == 32) tmem_ld_wait_regs32(sv + 32);
        const float4 L4 = *reinterpret_cast<const float4*>(stl + e);   // -LSE * log2(e)
        float x[4];
        f2_unpack(add2(fma2(f2_pack(P[e], P[e + 1]), sl2x2, kb2), f2_pack(L4.x, L4.y)), x[0], x[1]);
        f2_unpack(add2(fma2(f2_pack(P[e + 2], P[e + 3]), sl2x2, kb2), f2_pack(L4.z, L4.w)), x[2],
                  x[3]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (need_mask && e + j < thr) x[j] = -INFINITY;
          P[e + j] = ex2(x[j]);
        }
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          pk[e / 2] = pack_bf16x2(P[half * 32 + e], P[half * 32 + e + 1]);
        tmem_st16(lane_base + h * 64 + half * 16, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(bars.p_full());
      return true;
    };
    // dS^T = scale * P^T o (dP^T - D) of global step gi, into the dS boxes
    // in shared memory (A operand of dK += dS^T Q and of dQ = dS K).
    auto compute_ds = [&](int gi) -> bool {
      const float* std_ = stat + (gi & 1) * 2 * kT + kT + h * 64;   // -scale * D
      const uint64_t sc2 = f2_pack(p.scale, p.scale);
      if (!wait_warp(bars.dp_full(), gi & 1, wc, ERR_WAIT_SOFTMAX)) return false;
      tc_fence_after();
      // two chunks of 32 query columns; at d = 128 the second loads while the
      // first is processed (at d = 64 that measured slower)
      constexpr bool kPipe = D == 128;
      uint32_t dpa[64];
      tmem_ld32(lane_base + 128 + h * 64, dpa);
      tmem_ld_wait();
      if (kPipe) tmem_ld32(lane_base + 128 + h * 64 + 32, dpa + 32);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t* dpv = dpa + half * 32;
        if (half == 1) {
          if (kPipe) {
            tmem_ld_wait_regs32(dpa + 32);
          } else {
            tmem_ld32(lane_base + 128 + h * 64 + 32, dpa + 32);
            tmem_ld_wait();
          }
        }
        uint32_t dsk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 D4 = *reinterpret_cast<const float4*>(std_ + half * 32 + e);
          const float* Pp = P + half * 32 + e;
          float d[4];
          f2_unpack(mul2(fma2(f2_pack(__uint_as_float(dpv[e]), __uint_as_float(dpv[e + 1])), sc2,
                              f2_pack(D4.x, D4.y)),
                         f2_pack(Pp[0], Pp[1])),
                    d[0], d[1]);
          f2_unpack(mul2(fma2(f2_pack(__uint_as_float(dpv[e + 2]), __uint_as_float(dpv[e + 3])),
                              sc2, f2_pack(D4.z, D4.w)),
                         f2_pack(Pp[2], Pp[3])),
                    d[2], d[3]);
          dsk[e / 2] = pack_bf16x2(d[0], d[1]);
          dsk[e / 2 + 1] = pack_bf16x2(d[2], d[3]);
        }
        if (DET) {
          // packed into this warpgroup's own dP^T columns, over scores it has
          // already read (chunk 0 -> columns [0,16), chunk 1 -> [16,32))
          tmem_st16(lane_base + 128 + h * 64 + half * 16, dsk);
        } else {
          // row = key of the 128-byte-swizzled box holding query columns
          // [64h, 64h+64); this chunk is its 16-byte pieces 4*half .. 4*half+3
          uint8_t* rowp = ds_s + h * C::SUB + r * 128;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int chunk = (half * 4 + k) ^ (r & 7);
            *reinterpret_cast<uint4*>(rowp + chunk * 16) =
                make_uint4(dsk[4 * k], dsk[4 * k + 1], dsk[4 * k + 2], dsk[4 * k + 3]);
          }
        }
      }
      if (DET) {
        tmem_st_wait();
      } else {
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive_warp(bars.ds_full());
      return true;
    };

    // The staging of dK and dV, one tile each, as the 128-byte-swizzled
    // 64-column boxes TMA uses. Deterministic form (one item per CTA): in the
    // Q stages, stored by one of these threads. Reduction form: dV in the dS
    // buffer and dK in the Q stage of the item's last tile (d = 64: both in
    // the dS buffer), stored by the TMA warp, which hands the dS buffer back
    // once TMA has read it (epi_read) and refills that Q stage only after
    // the read; so the write-out costs the P/dS warps one pass, and the next
    // item's loads and first products go on meanwhile.
    // Barrier of the eight compute warps, on an mbarrier so that a warp that
    // has stopped makes the others' wait run out instead of hang.
    // Used once per ragged item in the reduction form, once in the
    // deterministic form (one item per CTA).
    int ncw = 0;   // uses so far (the same count in every compute warp)
    auto cw_sync = [&]() -> bool {
      mbar_arrive_warp(bars.cw());
      return wait_warp(bars.cw(), DET ? 0u : (uint32_t)(ncw++ & 1), wc, ERR_WAIT_EPILOGUE);
    };
    for (int u = 0;; ++u) {
      if (!wait_warp(&bars.sched_full()[u & 1], (u >> 1) & 1, wc, ERR_WAIT_LOAD)) break;
      cur = slots + (u & 1);   // held until this item's epilogue is done with it
      if (cur->w < 0) break;
      const int n = cur->n;

      // Order per tile i: dS(i), then P(i+1) (its S^T was issued right after
      // dV(i)); P of the item's first tile first.
      bool ok = true;
      int lt = 0;
      const int g = cur->g0;
      if (n > 0) ok = compute_p(g);
      // the previous item's staging has been read by TMA before the dS buffer
      // is written again (every compute warp waits once per item, even after
      // a failed wait, so that the phases stay in step)
      if (!DET && u > 0 && !wait_warp(bars.epi_read(), (u - 1) & 1, wc, ERR_WAIT_EPILOGUE)) ok = false;
      if (n > 0) {
        for (; ok && lt < n; ++lt) {
          const int gi = g + lt;
          if (!(ok = compute_ds(gi))) break;
          if (lt + 1 < n && !(ok = compute_p(gi + 1))) break;
        }
        if (ok) {
          // every MMA of the item is done (committed after its last product)
          ok = wait_warp(bars.kv_empty(), cur->kph & 1, wc, ERR_WAIT_EPILOGUE);
          tc_fence_after();
        }
      }
      // ---- dK, dV of this key tile. Each thread reads its key row (this
      // warpgroup's half of the columns) out of TMEM and stages it. A packed
      // sequence's ragged last tile is written with plain coalesced stores
      // instead of TMA (a 128-row box would run into the next sequence's
      // rows).
      const BwdItem t = bwd_item<CAUSAL>(a, cur->w);
      const bool ragged = p.cu_k != nullptr && t.key0 + kT > t.Nk;
      // staging of dV (which = 0) and dK (which = 1)
      const int sk = (g + n + 1) & 1;
      auto stg = [&](int which) -> uint8_t* {
        if (DET) return smem + C::OFF_Q + which * C::TILE;
        if (which == 0) return smem + C::OFF_DS;
        return C::DK_IN_Q ? smem + C::OFF_Q + sk * C::TILE : smem + C::OFF_DS + C::TILE;
      };
      if (ok) {
        const bool have = n > 0;
#pragma unroll
        for (int which = 0; which < 2; ++which) {   // 0: dV, 1: dK
#pragma unroll
          for (int c0 = 0; c0 < HD; c0 += 32) {
            uint32_t x[32];
            if (have) {
              tmem_ld32(lane_base + 256 + which * D + h * HD + c0, x);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) x[e] = 0u;
            }
            uint32_t pkd[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2)
              pkd[e / 2] = pack_bf16x2(__uint_as_float(x[e]), __uint_as_float(x[e + 1]));
            const int col = h * HD + c0;   // first column of these 32
            uint8_t* rowp = stg(which) + (col / 64) * C::SUB + r * 128;
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              const int j = (col % 64) / 8 + v4;
              *reinterpret_cast<uint4*>(rowp + ((j ^ (r & 7)) * 16)) =
                  make_uint4(pkd[4 * v4], pkd[4 * v4 + 1], pkd[4 * v4 + 2], pkd[4 * v4 + 3]);
            }
          }
        }
        fence_proxy_async_smem();   // the generic-proxy writes, before TMA reads them
      }
      // (the abort flag is read once for the warp, so its lanes leave together)
      bool stop = !ok || __any_sync(0xffffffffu, *abort_flag);
      if (DET || ragged) {
        // every warp's rows staged; a warp whose wait failed has raised the
        // abort flag before arriving
        if (!cw_sync() || __any_sync(0xffffffffu, *abort_flag)) stop = true;
        if (!stop && !ragged) {
          if (threadIdx.x == 0) {
#pragma unroll
            for (int which = 0; which < 2; ++which)
#pragma unroll
              for (int c = 0; c < D / 64; ++c)
                tma_store_3d(which ? &a.tm_dk : &a.tm_dv, stg(which) + c * C::SUB, c * 64,
                             t.sv.k_off + t.key0, t.sv.hk);
            bulk_commit_group();
          }
        } else if (!stop) {
          constexpr int CPR = D / 8;   // 16-byte pieces per row
          for (int idx = threadIdx.x; idx < 2 * kT * CPR; idx += 2 * kT) {
            const int which = idx / (kT * CPR), rem = idx % (kT * CPR);
            const int row = rem / CPR, c = rem % CPR;
            if (t.key0 + row < t.Nk) {
              const uint4 v = *reinterpret_cast<const uint4*>(
                  stg(which) + (c / 8) * C::SUB + row * 128 + (((c % 8) ^ (row & 7)) * 16));
              uint16_t* dst = (which ? a.dk : a.dv) +
                              ((size_t)t.sv.hk * t.sv.krows + t.sv.k_off + t.key0 + row) * D + c * 8;
              *reinterpret_cast<uint4*>(dst) = v;
            }
          }
        }
      }
      if (stop) break;
      // reduction form: staged (a ragged tile: already stored) -> the TMA warp
      if (!DET) mbar_arrive_warp(bars.epi_staged());
      mbar_arrive_warp(&bars.sched_empty()[u & 1]);   // done with the slot
    }
    // (deterministic form) the stores are complete before the CTA exits
    if (DET && lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::W_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL, bool BIAS, bool DET>
cudaError_t launch_main(const BwdBf16Args& a, cudaStream_t s) {
  using C = BwdCfg<D, DET>;
  auto kern = bwd_main_kernel<D, CAUSAL, BIAS, DET>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::BYTES);
  if (e != cudaSuccess) return e;
  const long BHkv = (long)a.p.B * a.p.Hkv;
  const long n_items = BHkv * ((a.p.Nk + kT - 1) / kT);
  // Heads per ordering group. Every item of a key/value head streams the Q
  // and dO tiles of its query heads and reduce-adds into their dQ rows, while
  // each item's K/V tile is read once and passes through L2. A group of
  // about 1024 items (several waves of CTAs) keeps enough heads in flight
  // that few items reduce into the same dQ rows at once, and its Q, dO and
  // fp32 dQ accumulator are kept within 64 MiB so that the streaming K/V
  // does not evict them.
  const long n_kt = (a.p.Nk + kT - 1) / kT;
  const long head_bytes = (long)(a.p.H / a.p.Hkv) * a.p.Nq * D * (2 + 2 + 4);
  const long g_items = (1024 + n_kt - 1) / n_kt;
  const long g_l2 = (64L << 20) / std::max(head_bytes, 1L);
  BwdBf16Args b = a;
  b.head_group = (int)std::max(1L, std::min(BHkv, std::min(g_items, g_l2)));
  long grid = n_items;
  if (!DET) {
    // persistent: one CTA per SM, items from the counter
    grid = std::min(n_items, (long)std::max(a.num_sms, 1));
    if ((e = cudaMemsetAsync(a.sched, 0, sizeof(int), s)) != cudaSuccess) return e;
  }
  kern<<<(unsigned)grid, C::NT, C::BYTES, s>>>(b);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const BwdBf16Args& a, cudaStream_t s, unsigned stages) {
  // rows of O, dO and the dQ accumulator
  const long rows = a.p.cu_q ? (long)a.p.H * a.p.total_q : (long)a.p.B * a.p.H * a.p.Nq;
  cudaError_t e = cudaSuccess;
  if (stages & BWD_PRE) {
    constexpr int kRowsPerBlock = 8 * (32 / (D / 8));
    const long BH = (long)a.p.B * a.p.H;
    const long prows = BH * a.nq_pad;
    const long blocks = min((prows + kRowsPerBlock - 1) / kRowsPerBlock, (long)a.num_sms * 8);
    bwd_pre_kernel<D><<<(unsigned)blocks, 256, 0, s>>>(a.o, a.dO, a.lse, a.D, a.lse2, a.dq_acc,
                                                      a.p, a.nq_pad, a.err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (stages & BWD_MAIN) {
    const BwdBf16Args& m = a;
    const bool bias = a.bias != nullptr;
    if (stages & BWD_DET) {
      if (a.p.causal)
        e = bias ? launch_main<D, true, true, true>(m, s) : launch_main<D, true, false, true>(m, s);
      else
        e = bias ? launch_main<D, false, true, true>(m, s) : launch_main<D, false, false, true>(m, s);
    } else {
      if (a.p.causal)
        e = bias ? launch_main<D, true, true, false>(m, s) : launch_main<D, true, false, false>(m, s);
      else
        e = bias ? launch_main<D, false, true, false>(m, s)
                 : launch_main<D, false, false, false>(m, s);
    }
    if (e != cudaSuccess) return e;
  }
  if (stages & BWD_DQ) {
    if ((e = launch_bwd_dq(a, s)) != cudaSuccess) return e;
  }
  if (stages & BWD_POST) {
    const long n8 = rows * D / 8;
    const long blocks = min((n8 + 255) / 256, (long)a.num_sms * 8);
    bwd_post_kernel<<<(unsigned)blocks, 256, 0, s>>>(a.dq_acc, a.dq, n8);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return e;
}

}  // namespace

cudaError_t launch_bwd_bf16(const BwdBf16Args& a, cudaStream_t s, unsigned stages) {
  return a.p.d == 64 ? launch_d<64>(a, s, stages) : launch_d<128>(a, s, stages);
}

}  // namespace fa
