// fp32 forward on the CUDA cores (FFMA), for fp32 inputs.
//
// fp32 results must stay within 1e-5 of the exact answer, which rules out the
// TF32 tensor path; the work here is tiny next to the bf16 path, so a plain
// query-outer SIMT kernel is enough. Each query row is owned by a group of
// TPR = d/32 adjacent lanes, each holding 32 of the row's d elements
// (interleaved: element e*TPR + t belongs to lane t of the group, so the
// group's shared-memory reads fall in distinct banks). Keys stream through
// shared memory 32 at a time and are folded into the row state with the
// blockwise online-softmax recurrence (running max m, denominator l,
// unnormalised accumulator a; one division at the end) of "Understanding
// FlashAttention Pt 1", §2.4, in base 2 with scale*log2(e) folded into q
// ("flash-attention", Part VI).
#include <cmath>
#include <cstdint>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kThreads = 128;
constexpr int kKeys = 32;   // keys per shared-memory tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
__global__ void __launch_bounds__(kThreads) fwd_f32_kernel(FwdF32Args a) {
  constexpr int TPR = D / 32;              // lanes per query row
  constexpr int ROWS = kThreads / TPR;     // query rows per CTA
  __shared__ float sk[kKeys][D];
  __shared__ float sv[kKeys][D];
  __shared__ float sb[kKeys];

  const Problem& p = a.p;
  const int n_qt = (p.Nq + ROWS - 1) / ROWS;
  const long bh = blockIdx.x / n_qt;
  const int qt = blockIdx.x % n_qt;
  const int b = (int)(bh / p.H);
  const int tq = threadIdx.x % TPR;
  const int row = qt * ROWS + threadIdx.x / TPR;
  const bool row_ok = row < p.Nq;

  const float* qh = a.q + (size_t)bh * p.Nq * D;
  const long bh_kv = (long)b * p.Hkv + (bh % p.H) / (p.H / p.Hkv);   // shared key/value head
  const float* kh = a.k + (size_t)bh_kv * p.Nk * D;
  const float* vh = a.v + (size_t)bh_kv * p.Nk * D;
  const float* bias = a.bias ? a.bias + (size_t)b * p.Nk : nullptr;

  const float sl2 = p.scale * kLog2e;
  float q[32], acc[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    q[e] = row_ok ? qh[(size_t)row * D + e * TPR + tq] * sl2 : 0.f;
    acc[e] = 0.f;
  }
  // last key visible to this row (bottom-right causal) and to the CTA
  const long off = (long)p.Nk - p.Nq;
  const long lim = p.causal ? (long)row + off : (long)p.Nk - 1;
  long cta_last = p.Nk - 1;
  if (p.causal) {
    long last_row = (long)min(qt * ROWS + ROWS - 1, p.Nq - 1);
    cta_last = min(cta_last, last_row + off);
  }
  float m = -INFINITY, l = 0.f;

  for (long k0 = 0; k0 <= cta_last; k0 += kKeys) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kKeys * D; idx += kThreads) {
      const int r = idx / D, c = idx % D;
      const long kj = k0 + r;
      const bool in = kj < p.Nk;
      sk[r][c] = in ? kh[kj * D + c] : 0.f;
      sv[r][c] = in ? vh[kj * D + c] : 0.f;
    }
    if (threadIdx.x < kKeys) {
      const long kj = k0 + threadIdx.x;
      sb[threadIdx.x] = (kj < p.Nk) ? (bias ? bias[kj] * kLog2e : 0.f) : -INFINITY;
    }
    __syncthreads();

    float s[kKeys];
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < kKeys; ++c) {
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) dot = fmaf(q[e], sk[c][e * TPR + tq], dot);
#pragma unroll
      for (int w = 1; w < TPR; w <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, w);
      float v = dot + sb[c];
      if (k0 + c > lim) v = -INFINITY;
      s[c] = v;
      mx = fmaxf(mx, v);
    }
    const float m_new = fmaxf(m, mx);
    if (m_new == -INFINITY) continue;   // nothing visible yet: state stays (−inf, 0, 0)
    const float alpha = exp2f(m - m_new);   // m = −inf -> 0
    float psum = 0.f;
#pragma unroll
    for (int c = 0; c < kKeys; ++c) {
      s[c] = exp2f(s[c] - m_new);
      psum += s[c];
    }
    l = l * alpha + psum;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      float o = acc[e] * alpha;
#pragma unroll
      for (int c = 0; c < kKeys; ++c) o = fmaf(s[c], sv[c][e * TPR + tq], o);
      acc[e] = o;
    }
    m = m_new;
  }

  if (!row_ok) return;
  float* oh = a.o + (size_t)bh * p.Nq * D + (size_t)row * D;
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int e = 0; e < 32; ++e) oh[e * TPR + tq] = acc[e] * inv;
  if (a.lse && tq == 0)
    a.lse[(size_t)bh * p.Nq + row] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_fwd_f32(const FwdF32Args& a, cudaStream_t s) {
  const Problem& p = a.p;
  const long BH = (long)p.B * p.H;
  if (p.d == 64) {
    const int rows = kThreads / 2;
    const long grid = BH * ((p.Nq + rows - 1) / rows);
    fwd_f32_kernel<64><<<(unsigned)grid, kThreads, 0, s>>>(a);
  } else {
    const int rows = kThreads / 4;
    const long grid = BH * ((p.Nq + rows - 1) / rows);
    fwd_f32_kernel<128><<<(unsigned)grid, kThreads, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace fa
