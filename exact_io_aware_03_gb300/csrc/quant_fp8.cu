// bf16 -> e4m3 quantization for the FP8 forward ("FlashAttention, Explained",
// §21 and "FlashAttention: Mathematical Foundations...", the FA-3 FP8 path:
// low-precision operands with scaling factors).
//
// One scale per (batch, head) and tensor: scale = max|x| / 448 (448 = the
// largest finite e4m3 value), x8 = e4m3(x / scale) rounded to nearest even
// (`cvt.rn.satfinite`), so x ~= scale * x8. Q and K keep their [rows][d]
// layout; V is written transposed, [d][keys] with the key count padded to a
// multiple of 16 (TMA rows start on 16-byte boundaries; the padding is 0), so
// that it is a K-major operand of O += P V.
//
// Three launches: the per-head max |x| of q, k, v (atomicMax on the float's
// bits, exact for non-negative floats; the caller zeroes the maxima), then
// q and k row-wise, then v through a shared-memory transpose.
#include <cstdint>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// grid (chunks, heads, 3 tensors); each thread folds 8 bf16 per step
__global__ void __launch_bounds__(256) amax_kernel(QuantFp8Args a) {
  const int which = blockIdx.z;   // 0: q, 1: k, 2: v
  const int head = blockIdx.y;
  const int heads = which == 0 ? a.heads_q : a.heads_kv;
  if (head >= heads) return;
  const long rows = which == 0 ? a.Nq : a.Nk;
  const long n8 = rows * a.d / 8;   // 16-byte groups of this head
  const uint16_t* x = (which == 0 ? a.q : which == 1 ? a.k : a.v) + (size_t)head * rows * a.d;
  float m = 0.f;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (long)gridDim.x * blockDim.x) {
    const uint4 u = reinterpret_cast<const uint4*>(x)[i];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[e])), fabsf(bf16_hi(w[e]))));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float wm[8];
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x / 32] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < 8; ++i) m = fmaxf(m, wm[i]);
    float* out = (which == 0 ? a.amax_q : which == 1 ? a.amax_k : a.amax_v) + head;
    atomicMax(reinterpret_cast<unsigned int*>(out), __float_as_uint(m));
  }
}

// q and k, row layout kept: grid (chunks, heads, 2); 16 elements per thread step
__global__ void __launch_bounds__(256) quant_rows_kernel(QuantFp8Args a) {
  const int which = blockIdx.z;
  const int head = blockIdx.y;
  const int heads = which == 0 ? a.heads_q : a.heads_kv;
  if (head >= heads) return;
  const long rows = which == 0 ? a.Nq : a.Nk;
  const long n16 = rows * a.d / 16;
  const size_t base = (size_t)head * rows * a.d;
  const uint16_t* x = (which == 0 ? a.q : a.k) + base;
  uint8_t* y = (which == 0 ? a.q8 : a.k8) + base;
  const float sc = fp8_scale((which == 0 ? a.amax_q : a.amax_k)[head]);
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (long)gridDim.x * blockDim.x) {
    const uint4 u0 = reinterpret_cast<const uint4*>(x)[2 * i];
    const uint4 u1 = reinterpret_cast<const uint4*>(x)[2 * i + 1];
    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      o[e] = pack_e4m3x4(bf16_lo(w[2 * e]) / sc, bf16_hi(w[2 * e]) / sc, bf16_lo(w[2 * e + 1]) / sc,
                         bf16_hi(w[2 * e + 1]) / sc);
    reinterpret_cast<uint4*>(y)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// v -> v^T: one block per (64-key tile, head); d = 128
constexpr int kVK = 64;
__global__ void __launch_bounds__(256) quant_vt_kernel(QuantFp8Args a) {
  __shared__ float t[kVK][129];   // +1 column: the transposed reads hit distinct banks
  const int head = blockIdx.y;
  const int k0 = blockIdx.x * kVK;
  const uint16_t* x = a.v + (size_t)head * a.Nk * 128;
  const float sc = fp8_scale(a.amax_v[head]);
  // load 64 keys x 128 columns (8 bf16 per thread step)
  for (int i = threadIdx.x; i < kVK * 16; i += 256) {
    const int kr = i / 16, c8 = (i % 16) * 8;
    float v8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (k0 + kr < a.Nk) {
      const uint4 u = *reinterpret_cast<const uint4*>(x + (size_t)(k0 + kr) * 128 + c8);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v8[2 * e] = bf16_lo(w[e]);
        v8[2 * e + 1] = bf16_hi(w[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) t[kr][c8 + e] = v8[e];
  }
  __syncthreads();
  // write row c (one of 128) of v^T: this block's 64 keys, 16 per thread step
  uint8_t* y = a.vt8 + (size_t)head * 128 * a.nk16;
  for (int i = threadIdx.x; i < 128 * (kVK / 16); i += 256) {
    const int c = i / (kVK / 16), kq = (i % (kVK / 16)) * 16;
    if (k0 + kq >= a.nk16) continue;   // nk16 is a multiple of 16
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      o[e] = pack_e4m3x4(t[kq + 4 * e][c] / sc, t[kq + 4 * e + 1][c] / sc, t[kq + 4 * e + 2][c] / sc,
                         t[kq + 4 * e + 3][c] / sc);
    *reinterpret_cast<uint4*>(y + (size_t)c * a.nk16 + k0 + kq) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

cudaError_t launch_quant_fp8(const QuantFp8Args& a, cudaStream_t s) {
  const int heads = a.heads_q > a.heads_kv ? a.heads_q : a.heads_kv;
  const long rows = a.Nq > a.Nk ? a.Nq : a.Nk;
  const unsigned chunks = (unsigned)((rows * a.d / 8 + 256 * 8 - 1) / (256 * 8));
  amax_kernel<<<dim3(chunks, heads, 3), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  quant_rows_kernel<<<dim3(chunks, heads, 2), 256, 0, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  quant_vt_kernel<<<dim3((unsigned)((a.nk16 + kVK - 1) / kVK), a.heads_kv, 1), 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace fa
