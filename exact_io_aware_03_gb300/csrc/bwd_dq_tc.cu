// dQ of the bf16 backward without cross-CTA accumulation (the deterministic
// backward's second kernel).
//
// The key-tile-outer backward ("flash-attention", Part VII) makes every key
// tile add its share of dQ_i into a shared accumulator, so the order of the
// floating-point additions depends on CTA timing. Here dQ is instead formed
// query-tile outer, the loop order of the forward ("FlashAttention,
// Explained", §20): one CTA owns a 128-row query tile of one head, keeps
// Q_i and dO_i in shared memory, streams the key/value tiles it can see
// through a TMA ring, and per key tile j
//   S    = Q_i K_j^T                    tcgen05 -> TMEM (lane = query row)
//   P    = exp2(S*c + bias - LSE2_i)    recomputed from the saved LSE
//   dP   = dO_i V_j^T                   tcgen05 -> TMEM
//   dS   = P o (dP - D_i)               -> TMEM as packed bf16
//   dQ_i += dS K_j                      A = dS read from TMEM, fp32 in TMEM
// ("Understanding FlashAttention Pt 1", §3.6). dQ_i is written once, scaled,
// in bf16, and the key tiles are always added in the same order, so the
// result is bitwise reproducible. dK and dV come from the key-outer kernel
// run without its dQ product.
//
// Warp roles (320 threads, one CTA per SM): warps 0-7 are two warpgroups that
// split the 128 keys of every tile (thread = query row = TMEM lane, warpgroup
// h takes keys [64h, 64h+64)); warp 8 issues the TMA loads; warp 9 owns TMEM
// and issues the MMAs. Q_i and dO_i are copied once from shared memory into
// TMEM, so that all three products read their A operand from TMEM (the
// shared-memory operand path is the slower one: it has to stream both
// operands). TMEM (512 columns): S [0,128), dP then packed dS [128,256),
// dQ [256,256+D), Q_i [256+D, 256+3D/2), dO_i [256+3D/2, 256+2D) (bf16 pairs).
// MMA order per key tile j: dP(j), S(j+1) (once the warpgroups have read
// S(j)), then dQ(j) once dS(j) is in TMEM.
#include <algorithm>
#include <cmath>
#include <cstdint>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 320;
constexpr int kT = 128;   // query rows per tile = keys per key tile
constexpr float kLog2e = 1.4426950408889634f;

// K_j is read twice, by S(j) and, a tile later, by dQ(j), so the K ring has
// one stage more than the V ring (V_j is read by dP(j) only): the load of
// K_{j+1} then starts a whole tile before S(j+1) needs it instead of when
// dQ(j-1) completes, which left the tensor core waiting for the copy.
template <int D>
struct DqCfg {
  static constexpr int NSK = (D == 128) ? 3 : 4;  // K ring stages
  static constexpr int NSV = (D == 128) ? 2 : 4;  // V ring stages
  static constexpr int TILE = kT * D * 2;         // bf16 [128][D]
  static constexpr int SUB = kT * 128;            // one 64-column box
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = TILE;
  static constexpr int OFF_K = 2 * TILE;
  static constexpr int OFF_V = OFF_K + NSK * TILE;
  static constexpr int OFF_BIAS = OFF_V + NSV * TILE;   // [2 warpgroups][2 bufs][128] floats
  static constexpr int OFF_BAR = OFF_BIAS + 2 * 2 * kT * 4;
  static constexpr int NBAR = 1 /*q_full*/ + 2 * NSK + 2 * NSV /*k/v full/empty*/ +
                              1 /*s_full*/ + 1 /*s_free*/ + 1 /*dp_full*/ + 1 /*ds_full*/ +
                              1 /*dq_full*/ + 1 /*qt_ready*/ + 4 /*bias*/ + 1 /*drain*/;
  static constexpr int OFF_SCALARS = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_SCALARS + 64;
};

template <int D, bool CAUSAL, bool BIAS>
__global__ void __launch_bounds__(kThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdBf16Args a) {
  using C = DqCfg<D>;
  // 128-byte-swizzled TMA boxes need 1024-byte alignment; the dynamic
  // shared memory of a kernel without static shared memory starts there
  // (checked below: a misaligned base aborts the CTA with an error)
  extern __shared__ __align__(1024) uint8_t smem[];
  const Problem& p = a.p;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;

  uint64_t* bb = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bb;   bb += 1;   // Q_i and dO_i
  uint64_t* k_full = bb;   bb += C::NSK;
  uint64_t* k_empty = bb;  bb += C::NSK;
  uint64_t* v_full = bb;   bb += C::NSV;
  uint64_t* v_empty = bb;  bb += C::NSV;
  uint64_t* s_full = bb;   bb += 1;   // S done
  uint64_t* s_free = bb;   bb += 1;   // S read by both warpgroups (one arrival per warp)
  uint64_t* qt_ready = bb; bb += 1;   // Q_i, dO_i copied into TMEM (one arrival per warp)
  uint64_t* dp_full = bb;  bb += 1;
  uint64_t* ds_full = bb;  bb += 1;   // dS in TMEM (one arrival per warp)
  uint64_t* dq_full = bb;  bb += 1;   // every dQ product done
  uint64_t* bias_rdy = bb; bb += 4;   // [warpgroup][buffer], one arrival per warp
  uint64_t* drain = bb;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_SCALARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_SCALARS + 4);
  int* key_lo_s = reinterpret_cast<int*>(smem + C::OFF_SCALARS + 8);
  int* key_hi_s = reinterpret_cast<int*>(smem + C::OFF_SCALARS + 12);
  float* bias_buf = reinterpret_cast<float*>(smem + C::OFF_BIAS);
  const WaitCtx wc{abort_flag, a.err};

  // ---- which (query tile, head): heads in groups of a.head_group whose K/V
  // fit in L2; within a group the heaviest tiles (the last query tiles under
  // a causal mask) first, cycling over the group's heads.
  const int n_qt = (p.Nq + kT - 1) / kT;
  const int BH = p.B * p.H;
  const int G = a.head_group;
  const int grp = (int)(blockIdx.x / ((long)G * n_qt));
  const int g0 = grp * G;
  const int gsz = min(G, BH - g0);
  const int rr = (int)(blockIdx.x - (long)g0 * n_qt);
  const int bh = g0 + rr % gsz;
  const int qt = n_qt - 1 - rr / gsz;
  const int b = bh / p.H;
  const SeqView sv = seq_view(p, b, bh % p.H);
  const int Nq = sv.len_q, Nk = sv.len_k;
  const int q0 = qt * kT;
  const float* bias_row = BIAS ? a.bias + (size_t)b * Nk : nullptr;

  if (threadIdx.x == 0) {
    if ((smem_u32(smem) & 1023u) != 0) atomicOr(a.err, ERR_WAIT_DRAIN);   // layout invariant
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NSK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < C::NSV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 2 * kT / 32);   // one arrival per compute warp
    mbar_init(qt_ready, 2 * kT / 32);
    mbar_init(dp_full, 1);
    mbar_init(ds_full, 2 * kT / 32);
    mbar_init(dq_full, 1);
    for (int t = 0; t < 4; ++t) mbar_init(&bias_rdy[t], kT / 32);
    mbar_init(drain, 1);
    *abort_flag = (smem_u32(smem) & 1023u) != 0;
    *key_lo_s = Nk;
    *key_hi_s = -1;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&a.tm_q);
    tma_prefetch_desc(&a.tm_do);
    tma_prefetch_desc(&a.tm_k);
    tma_prefetch_desc(&a.tm_v);
  }
  __syncthreads();
  if (BIAS && q0 < Nq) {
    // first and last key with a finite bias; key tiles outside are skipped
    int lo = Nk, hi = -1;
    for (int j = threadIdx.x; j < Nk; j += kThreads) {
      if (bias_row[j] != -INFINITY) {
        lo = min(lo, j);
        hi = max(hi, j);
      }
    }
    if (lo < Nk) atomicMin(key_lo_s, lo);
    if (hi >= 0) atomicMax(key_hi_s, hi);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- key tiles [lo, hi) seen by this query tile
  const int n_kv = (Nk + kT - 1) / kT;
  const long off = (long)Nk - Nq;   // bottom-right causal offset
  int lo = 0, hi = n_kv;
  if (BIAS) {
    const int klo = *key_lo_s, khi = *key_hi_s;
    if (khi < 0) {
      hi = 0;
    } else {
      lo = klo / kT;
      hi = khi / kT + 1;
    }
  }
  if (q0 >= Nq) {
    hi = lo;
  } else if (CAUSAL) {
    const long lim = (long)min(q0 + kT - 1, Nq - 1) + off;
    hi = lim < 0 ? 0 : (int)min((long)hi, lim / kT + 1);
  }
  hi = max(hi, lo);
  const int n = *abort_flag ? 0 : hi - lo;

  if (warp == 8) {
    // ================================================================ TMA producer
    if (lane == 0 && n > 0) {
      mbar_arrive_expect_tx(q_full, 2 * C::TILE);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(smem + C::OFF_Q + c * C::SUB, &a.tm_q, c * 64, sv.q_off + q0, sv.hq, q_full);
        tma_load_3d(smem + C::OFF_DO + c * C::SUB, &a.tm_do, c * 64, sv.q_off + q0, sv.hq, q_full);
      }
      int nk = 0, nv = 0;
      for (int j = lo; j < hi; ++j) {
        const int i = j - lo;
        const int sk = i % C::NSK, uk = i / C::NSK, sv_ = i % C::NSV, uv = i / C::NSV;
        if (uk > 0 && !wait1(&k_empty[sk], (uk - 1) & 1, wc, ERR_WAIT_LOAD)) break;
        mbar_arrive_expect_tx(&k_full[sk], C::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + C::OFF_K + sk * C::TILE + c * C::SUB, &a.tm_k, c * 64,
                      sv.k_off + j * kT, sv.hk, &k_full[sk]);
        ++nk;
        if (uv > 0 && !wait1(&v_empty[sv_], (uv - 1) & 1, wc, ERR_WAIT_LOAD)) break;
        mbar_arrive_expect_tx(&v_full[sv_], C::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + C::OFF_V + sv_ * C::TILE + c * C::SUB, &a.tm_v, c * 64,
                      sv.k_off + j * kT, sv.hk, &v_full[sv_]);
        ++nv;
      }
      // no copy may still be landing when the CTA exits (bounded, ignores abort)
      const WaitCtx wd{abort_flag, a.err, true};
      wait1(q_full, 0, wd, ERR_WAIT_DRAIN);
      for (int i = max(0, nk - C::NSK); i < nk; ++i)
        wait1(&k_full[i % C::NSK], (i / C::NSK) & 1, wd, ERR_WAIT_DRAIN);
      for (int i = max(0, nv - C::NSV); i < nv; ++i)
        wait1(&v_full[i % C::NSV], (i / C::NSV) & 1, wd, ERR_WAIT_DRAIN);
    }
  } else if (warp == 9) {
    // ================================================================ MMA issuer
    // (the whole warp, converged; lane 0 issues each instruction)
    if (n > 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(kT, kT, false, false);   // S, dP (K-major)
      constexpr uint32_t id_dq = idesc_bf16_f32(kT, D, false, true);    // dQ: B = K, MN-major
      const uint32_t t_s = tmem, t_dp = tmem + 128, t_dq = tmem + 256;
      const uint32_t t_q = tmem + 256 + D, t_do = tmem + 256 + D + D / 2;
      // operand descriptors, built once for the start of shared memory: an
      // operand's is this plus its byte offset
      const uint32_t sbase = smem_u32(smem);
      const uint64_t dk16 = sdesc_sw128(sbase, 16, 1024), dsub = sdesc_sw128(sbase, C::SUB, 1024);
      // D = A B^T over the head dimension: A (Q or dO) in TMEM, B (K or V) a
      // K-major tile of 64-column boxes at byte offset b_o
      auto issue_nt = [&](uint32_t d, uint32_t a_t, uint32_t b_o) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = (kk / 4) * C::SUB + (kk % 4) * 32;
          mma_ts_w(d, a_t + kk * 8, sdesc_offset(dk16, b_o + o), id_s, kk > 0 ? 1u : 0u);
        }
      };
      bool ok = wait_warp(qt_ready, 0, wc, ERR_WAIT_MMA) && wait_warp(&k_full[0], 0, wc, ERR_WAIT_MMA);
      if (ok) {
        tc_fence_after();
        issue_nt(t_s, t_q, C::OFF_K);
        mma_commit_w(s_full);
      }
      // Every wait of an iteration but the one for dS(i) comes first, while
      // dQ(i-1) is still executing, and dP(i), S(i+1) are then issued back to
      // back: the issuing thread stalls while the MMA queue is full, so a wait
      // between two products would leave the tensor core idle.
      for (int i = 0; i < n && ok; ++i) {
        const int s = i % C::NSK, sv_ = i % C::NSV, s1 = (i + 1) % C::NSK;
        const bool next = i + 1 < n;
        if (!(ok = wait_warp(&v_full[sv_], (i / C::NSV) & 1, wc, ERR_WAIT_MMA))) break;
        // S(i+1) needs K_{i+1} and both warpgroups done reading S(i)
        if (next && !(ok = wait_warp(&k_full[s1], ((i + 1) / C::NSK) & 1, wc, ERR_WAIT_MMA))) break;
        if (next && !(ok = wait_warp(s_free, i & 1, wc, ERR_WAIT_MMA))) break;
        tc_fence_after();
        // dP = dO V^T (the dP columns are free: dQ(i-1), which read dS(i-1)
        // there, was issued before and MMAs complete in order)
        issue_nt(t_dp, t_do, C::OFF_V + sv_ * C::TILE);
        mma_commit_w(dp_full);
        mma_commit_w(&v_empty[sv_]);
        if (next) {
          issue_nt(t_s, t_q, C::OFF_K + s1 * C::TILE);
          mma_commit_w(s_full);
        }
        // dQ += dS K_j: dS packed bf16, keys [0,64) in TMEM columns [128,160),
        // keys [64,128) in [192,224)
        if (!(ok = wait_warp(ds_full, i & 1, wc, ERR_WAIT_MMA))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          mma_ts_w(t_dq, t_dp + (kk / 4) * 64 + (kk % 4) * 8,
                 sdesc_offset(dsub, C::OFF_K + s * C::TILE + kk * 2048), id_dq,
                 (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit_w(&k_empty[s]);
      }
      if (ok) mma_commit_w(dq_full);
      mma_commit_w(drain);
      wait_warp(drain, 0, WaitCtx{abort_flag, a.err, true}, ERR_WAIT_DRAIN);
    }
  } else {
    // ================================================================ warps 0-7
    const int h = warp / 4;                  // key half of every tile
    const int r = (warp % 4) * 32 + lane;    // query row within the tile = TMEM lane
    const int row = q0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)((warp % 4) * 32) << 16);
    const float sl2 = p.scale * kLog2e;
    constexpr int HD = D / 2;                // dQ columns per warpgroup
    // statistics of this row, -LSE * log2(e) and -scale * D (padding rows:
    // -inf and 0, so P = 0)
    const size_t srow = (size_t)bh * a.nq_pad + min(q0 + r, a.nq_pad - 1);
    const float nlse2 = a.lse2[srow], nDrow = a.D[srow];
    // last visible key of this row / of the tile's first row
    const long lim_row = CAUSAL ? min((long)row + off, (long)Nk - 1) : (long)Nk - 1;
    const long lim_tile = CAUSAL ? min((long)q0 + off, (long)Nk - 1) : (long)Nk - 1;
    // Q_i and dO_i into TMEM: this thread's row, the warpgroup's half of the
    // head dimension, read from the 128-byte-swizzled boxes
    auto copy_q_do = [&]() -> bool {
      if (!wait_warp(q_full, 0, wc, ERR_WAIT_SOFTMAX)) return false;
      constexpr int NC = D / 16;                   // 16-byte chunks per half row
      const int col0 = h * (D / 2);
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint8_t* rowp = smem + (which ? C::OFF_DO : C::OFF_Q) + (col0 / 64) * C::SUB + r * 128;
        uint32_t x[D / 4];
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          const int chunk = ((col0 % 64) / 8 + j) ^ (r & 7);
          const uint4 u = *reinterpret_cast<const uint4*>(rowp + chunk * 16);
          x[4 * j] = u.x; x[4 * j + 1] = u.y; x[4 * j + 2] = u.z; x[4 * j + 3] = u.w;
        }
        const uint32_t dst = lane_base + 256 + D + which * (D / 2) + h * (D / 4);
        if constexpr (D == 128) tmem_st32(dst, x);
        else tmem_st16(dst, x);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(qt_ready);
      return true;
    };
    float P[64];
    auto compute_p = [&](int i) -> bool {
      const int key0 = (lo + i) * kT;
      const float* bbuf = bias_buf + (h * 2 + (i & 1)) * kT;
      if (BIAS) {
        float* w = bias_buf + (h * 2 + (i & 1)) * kT;
        w[r] = key0 + r < Nk ? bias_row[key0 + r] * kLog2e : -INFINITY;
        mbar_arrive_warp(&bias_rdy[h * 2 + (i & 1)]);
        if (!wait_warp(&bias_rdy[h * 2 + (i & 1)], (i >> 1) & 1, wc, ERR_WAIT_SOFTMAX))
          return false;
      }
      if (!wait_warp(s_full, i & 1, wc, ERR_WAIT_SOFTMAX)) return false;
      tc_fence_after();
      uint32_t* su = reinterpret_cast<uint32_t*>(P);
      tmem_ld32(lane_base + h * 64, su);
      tmem_ld32(lane_base + h * 64 + 32, su + 32);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive_warp(s_free);   // the S columns may take the next tile's scores
      const bool need_mask = (long)key0 + kT - 1 > lim_tile;
      const long lim_rel = lim_row - key0 - h * 64;   // local column > lim_rel -> masked
      const uint64_t sl2x2 = f2_pack(sl2, sl2), nl2 = f2_pack(nlse2, nlse2);
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        float x0, x1;
        if (BIAS) {
          const uint64_t b2 = *reinterpret_cast<const uint64_t*>(bbuf + h * 64 + c);
          f2_unpack(add2(fma2(f2_pack(P[c], P[c + 1]), sl2x2, b2), nl2), x0, x1);
        } else {
          f2_unpack(fma2(f2_pack(P[c], P[c + 1]), sl2x2, nl2), x0, x1);
        }
        if (need_mask && c > lim_rel) x0 = -INFINITY;
        if (need_mask && c + 1 > lim_rel) x1 = -INFINITY;
        P[c] = ex2(x0);
        P[c + 1] = ex2(x1);
      }
      return true;
    };
    auto compute_ds = [&](int i) -> bool {
      if (!wait_warp(dp_full, i & 1, wc, ERR_WAIT_SOFTMAX)) return false;
      tc_fence_after();
      const uint64_t nD2 = f2_pack(nDrow, nDrow), sc2 = f2_pack(p.scale, p.scale);
      // two chunks of 32 keys; the packed dS of chunk c goes to columns
      // [16c, 16c+16) of this warpgroup's own dP columns, already read
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t dpv[32];
        tmem_ld32(lane_base + 128 + h * 64 + half * 32, dpv);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float d0, d1;
          // dS = scale * P o (dP - D)
          f2_unpack(mul2(fma2(f2_pack(__uint_as_float(dpv[c]), __uint_as_float(dpv[c + 1])), sc2,
                              nD2),
                         f2_pack(P[half * 32 + c], P[half * 32 + c + 1])),
                    d0, d1);
          pk[c / 2] = pack_bf16x2(d0, d1);
        }
        tmem_st16(lane_base + 128 + h * 64 + half * 16, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(ds_full);
      return true;
    };
    bool ok = n == 0 || (copy_q_do() && compute_p(0));
    int i = 0;
    for (; ok && i < n; ++i) {
      if (!(ok = compute_ds(i))) break;
      if (i + 1 < n && !(ok = compute_p(i + 1))) break;
    }
    // ---- dQ = dS K summed over the key tiles (dS carries the scale), bf16; rows that see
    // no key get 0. Staged in the Q buffer (Q_i lives in TMEM, so the
    // buffer is free) as the 128-byte-swizzled boxes TMA uses and stored by
    // one thread with TMA; a packed sequence's ragged last tile gets plain
    // coalesced stores. (Warp-uniform control flow: the TMEM loads and the
    // named barrier are collective.)
    bool do_epi = ok && i == n && q0 < Nq;
    uint8_t* stage = smem + C::OFF_Q;   // [D/64 boxes][128 rows][128 B]
    if (do_epi) {
      const bool have = n > 0;
      if (have) {
        do_epi = wait_warp(dq_full, 0, wc, ERR_WAIT_EPILOGUE);
        tc_fence_after();
      }
      if (do_epi) {
#pragma unroll
        for (int c0 = 0; c0 < HD; c0 += 32) {
          uint32_t x[32];
          if (have) {
            tmem_ld32(lane_base + 256 + h * HD + c0, x);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] = 0u;
          }
          uint32_t pkd[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            pkd[e / 2] = pack_bf16x2(__uint_as_float(x[e]), __uint_as_float(x[e + 1]));
          const int col = h * HD + c0;
          uint8_t* rowp = stage + (col / 64) * C::SUB + r * 128;
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            const int j = (col % 64) / 8 + v4;
            *reinterpret_cast<uint4*>(rowp + ((j ^ (r & 7)) * 16)) =
                make_uint4(pkd[4 * v4], pkd[4 * v4 + 1], pkd[4 * v4 + 2], pkd[4 * v4 + 3]);
          }
        }
        fence_proxy_async_smem();
      }
    }
    if (named_bar_and(1, 2 * kT, do_epi)) {
      if (p.cu_q == nullptr || q0 + kT <= Nq) {
        if (threadIdx.x == 0) {
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_store_3d(&a.tm_dq, stage + c * C::SUB, c * 64, sv.q_off + q0, sv.hq);
          bulk_commit_group();
          bulk_wait_group_read0();   // shared memory may be released
        }
      } else {
        constexpr int CPR = D / 8;
        for (int idx = threadIdx.x; idx < kT * CPR; idx += 2 * kT) {
          const int rw = idx / CPR, c = idx % CPR;
          if (q0 + rw < Nq) {
            const uint4 v = *reinterpret_cast<const uint4*>(
                stage + (c / 8) * C::SUB + rw * 128 + (((c % 8) ^ (rw & 7)) * 16));
            *reinterpret_cast<uint4*>(a.dq + ((size_t)sv.hq * sv.qrows + sv.q_off + q0 + rw) * D +
                                      c * 8) = v;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL, bool BIAS>
cudaError_t launch_one(const BwdBf16Args& a, cudaStream_t s) {
  using C = DqCfg<D>;
  static_assert(C::BYTES <= 232448, "shared memory per CTA");
  auto kern = bwd_dq_kernel<D, CAUSAL, BIAS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::BYTES);
  if (e != cudaSuccess) return e;
  const long BH = (long)a.p.B * a.p.H;
  const long n_qt = (a.p.Nq + kT - 1) / kT;
  // heads per ordering group: K and V of a group within ~48 MiB of L2 (with
  // grouped heads, query heads that share K/V are adjacent)
  const long kv_bytes = 2L * a.p.Nk * D * 2;
  BwdBf16Args b = a;
  b.head_group = (int)std::max(1L, std::min(BH, (48L << 20) / std::max(kv_bytes, 1L)));
  kern<<<(unsigned)(BH * n_qt), kThreads, C::BYTES, s>>>(b);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const BwdBf16Args& a, cudaStream_t s) {
  const bool bias = a.bias != nullptr;
  if (a.p.causal)
    return bias ? launch_one<D, true, true>(a, s) : launch_one<D, true, false>(a, s);
  return bias ? launch_one<D, false, true>(a, s) : launch_one<D, false, false>(a, s);
}

}  // namespace

cudaError_t launch_bwd_dq(const BwdBf16Args& a, cudaStream_t s) {
  return a.p.d == 64 ? launch_d<64>(a, s) : launch_d<128>(a, s);
}

}  // namespace fa
