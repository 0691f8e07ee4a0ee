// C ABI of the library (declared in include/fa.h): argument validation,
// TMA tensor-map encoding and dispatch to the kernels. Allocates no device
// memory: the only device state is a per-device error word (a __device__
// variable) whose address is looked up once per device.
#include <cmath>
#include <cstdint>
#include <algorithm>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

// The current device's context id, unique for the life of the process (a
// context created after cudaDeviceReset gets a new one). The driver entry
// point is looked up once; the device's primary context is made current
// first if the runtime has not done so yet.
fa_status current_context_id(unsigned long long* id) {
  using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static std::mutex mu;
  static CtxGetIdFn fn = nullptr;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!fn) {
      void* f = nullptr;
      cudaDriverEntryPointQueryResult q{};
      const cudaError_t e =
          cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f) return FA_ERR_CUDA;
      fn = reinterpret_cast<CtxGetIdFn>(f);
    }
  }
  if (fn(nullptr, id) == CUDA_SUCCESS) return FA_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return FA_ERR_CUDA;
  return fn(nullptr, id) == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

}  // namespace fa

namespace {

__device__ uint32_t g_fa_err_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t* g_err_ptr[kMaxDevices];
unsigned long long g_err_ctx[kMaxDevices];   // context id each address belongs to

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

fa_status get_encode(EncodeTiledFn* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return FA_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  *out = g_encode;
  return FA_OK;
}

fa_status get_err_ptr(uint32_t** out) {
  int dev = 0;
  unsigned long long ctx = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  if (fa::current_context_id(&ctx) != FA_OK) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  // looked up again when the device's context is not the one the cached
  // address belongs to (after cudaDeviceReset the module is reloaded)
  if (!g_err_ptr[dev] || g_err_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_err_word) != cudaSuccess || !p) return FA_ERR_CUDA;
    g_err_ptr[dev] = static_cast<uint32_t*>(p);
    g_err_ctx[dev] = ctx;
  }
  *out = g_err_ptr[dev];
  return FA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shared size/shape checks. Returns FA_OK or the error.
fa_status check_problem(int B, int H, int Nq, int Nk, int d, float scale, fa_dtype dtype,
                        int Hkv) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if (Hkv < 1 || Hkv > H || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP32) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long BH = (long long)B * H;
  if (BH >= (1LL << 31)) return FA_ERR_INVALID_ARG;
  if ((long long)Nq * d >= (1LL << 31) || (long long)Nk * d >= (1LL << 31))
    return FA_ERR_INVALID_ARG;
  // one CTA per (query-tile pair, head) must fit a 1-D grid
  if (BH * ((Nq + 255) / 256) >= (1LL << 31)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// 3-D view (d, N, B*H) of a bf16 [B][H][N][d] tensor, box (64, 128, 1),
// 128-byte swizzle, zero fill outside the tensor.
fa_status make_map(CUtensorMap* m, const void* base, int BH, int N, int d) {
  EncodeTiledFn enc = nullptr;
  fa_status st = get_encode(&enc);
  if (st != FA_OK) return st;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// 3-D view (d, N, B*H) of the fp32 dQ accumulator for TMA reduce-add:
// box (32, 32, 1) = one 128-byte-swizzled 4 KiB tile.
fa_status make_map_f32_acc(CUtensorMap* m, const void* base, int BH, int N, int d) {
  EncodeTiledFn enc = nullptr;
  fa_status st = get_encode(&enc);
  if (st != FA_OK) return st;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)N * d * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// 3-D view (dim0, dim1, dim2) of a byte tensor with rows of dim0 bytes, box
// (128, 128, 1), 128-byte swizzle, zero fill outside (the e4m3 operands).
fa_status make_map_u8(CUtensorMap* m, const void* base, long dim0, long dim1, long dim2) {
  EncodeTiledFn enc = nullptr;
  fa_status st = get_encode(&enc);
  if (st != FA_OK) return st;
  cuuint64_t dims[3] = {(cuuint64_t)dim0, (cuuint64_t)dim1, (cuuint64_t)dim2};
  cuuint64_t strides[2] = {(cuuint64_t)dim0, (cuuint64_t)(dim0 * dim1)};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// Workspace of the e4m3 forward: per-head max |x| (q, k, v), e4m3 q, k, and
// the transposed e4m3 v with keys padded to a multiple of 16; each part on a
// 256-byte boundary.
struct Fp8Ws {
  size_t amax, q8, k8, vt8, total;
};
Fp8Ws fp8_ws_layout(int B, int H, int Hkv, int Nq, int Nk, int d) {
  Fp8Ws w;
  const size_t nk16 = ((size_t)Nk + 15) / 16 * 16;
  w.amax = 0;
  w.q8 = round256(4 * ((size_t)B * H + 2 * (size_t)B * Hkv));
  w.k8 = w.q8 + round256((size_t)B * H * Nq * d);
  w.vt8 = w.k8 + round256((size_t)B * Hkv * Nk * d);
  w.total = w.vt8 + round256((size_t)B * Hkv * d * nk16);
  return w;
}

// Workspace of the backward: padded statistics for B*H (sequence, head)
// pairs of nq_max rows, then the fp32 dQ accumulator of `dq_rows` rows and,
// with it, the main kernel's work-item counter.
size_t bwd_ws_bytes(int B, int H, int nq_max, size_t dq_rows, int d) {
  const size_t prow = (size_t)B * H * (((size_t)nq_max + 127) / 128 * 128);
  return 2 * round256(prow * 4) + (dq_rows ? round256(dq_rows * (size_t)d * 4) + 256 : 0);
}


// One thread waits (bounded) on an mbarrier that nothing ever arrives at, so
// the wait runs out: it records FA_ERR_DEVICE's code in the error word and
// returns, exactly as a stalled pipeline stage in the real kernels would.
__global__ void selftest_timeout_kernel(uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  fa::mbar_init(&bar, 1);
  abort_flag = 0;
  fa::fence_mbar_init();
  const fa::WaitCtx w{&abort_flag, err};
  fa::wait1(&bar, 0, w, fa::ERR_WAIT_SOFTMAX);
}

// Shape checks of a packed variable-length batch (host side; the kernels
// check every sequence's offsets and lengths against these bounds).
fa_status check_varlen(int total_q, int total_k, int max_q, int max_k, int d, const int* cu_q,
                       const int* cu_k) {
  if (!cu_q || !cu_k || !aligned(cu_q, 4) || !aligned(cu_k, 4)) return FA_ERR_INVALID_ARG;
  if (total_q < 1 || total_k < 1 || max_q > total_q || max_k > total_k) return FA_ERR_INVALID_ARG;
  if ((long long)total_q * d >= (1LL << 31) || (long long)total_k * d >= (1LL << 31))
    return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Tensor maps and pointers of the bf16 forward (everything but the split).
fa_status fwd_bf16_setup(fa::FwdBf16Args* a, const fa::Problem& p, const void* q, const void* k,
                         const void* v, const float* key_bias, void* o, float* lse) {
  *a = fa::FwdBf16Args{};
  a->p = p;
  const int BH = p.B * p.H;
  fa_status st;
  if ((st = make_map(&a->tm_q, q, BH, p.Nq, p.d)) != FA_OK) return st;
  if ((st = make_map(&a->tm_k, k, p.B * p.Hkv, p.Nk, p.d)) != FA_OK) return st;
  if ((st = make_map(&a->tm_v, v, p.B * p.Hkv, p.Nk, p.d)) != FA_OK) return st;
  if ((st = make_map(&a->tm_o, o, BH, p.Nq, p.d)) != FA_OK) return st;
  a->bias = key_bias;
  a->o = static_cast<uint16_t*>(o);
  a->lse = lse;
  a->n_split = 1;
  return get_err_ptr(&a->err);
}

}  // namespace

extern "C" {

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported head dim or dtype";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call failed";
    case FA_ERR_DEVICE: return "FA_ERR_DEVICE: a kernel timed out on a device-side wait";
  }
  return "unknown fa_status";
}

fa_status fa_fwd(const void* q, const void* k, const void* v, const float* key_bias, void* o,
                 float* lse, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                 fa_dtype dtype, void* stream) {
  return fa_fwd_gqa(q, k, v, key_bias, o, lse, B, H, H, Nq, Nk, d, scale, causal, dtype, stream);
}

fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, const float* key_bias, void* o,
                     float* lse, int B, int H, int H_kv, int Nq, int Nk, int d, float scale,
                     int causal, fa_dtype dtype, void* stream) {
  fa_status st = check_problem(B, H, Nq, Nk, d, scale, dtype, H_kv);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return FA_ERR_INVALID_ARG;
  if ((key_bias && !aligned(key_bias, 4)) || (lse && !aligned(lse, 4))) return FA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  fa::Problem p{B, H, Nq, Nk, d, scale, causal ? 1 : 0, H_kv};

  if (dtype == FA_DTYPE_FP32) {
    fa::FwdF32Args a{p, static_cast<const float*>(q), static_cast<const float*>(k),
                     static_cast<const float*>(v), key_bias, static_cast<float*>(o), lse};
    return fa::launch_fwd_f32(a, s) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  }
  if (!lse) return FA_ERR_INVALID_ARG;
  fa::FwdBf16Args a;
  st = fwd_bf16_setup(&a, p, q, k, v, key_bias, o, lse);
  if (st != FA_OK) return st;
  return fa::launch_fwd_bf16(a, s) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H, int H_kv,
                        int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                        float scale, int causal, void* stream) {
  fa_status st = check_problem(B, H, max_seqlen_q, max_seqlen_k, d, scale, FA_DTYPE_BF16, H_kv);
  if (st != FA_OK) return st;
  st = check_varlen(total_q, total_k, max_seqlen_q, max_seqlen_k, d, cu_seqlens_q, cu_seqlens_k);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  fa::Problem p{B, H, max_seqlen_q, max_seqlen_k, d, scale, causal ? 1 : 0, H_kv};
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.total_q = total_q;
  p.total_k = total_k;
  fa::FwdBf16Args a{};
  a.p = p;
  if ((st = make_map(&a.tm_q, q, H, total_q, d)) != FA_OK) return st;
  if ((st = make_map(&a.tm_k, k, H_kv, total_k, d)) != FA_OK) return st;
  if ((st = make_map(&a.tm_v, v, H_kv, total_k, d)) != FA_OK) return st;
  if ((st = make_map(&a.tm_o, o, H, total_q, d)) != FA_OK) return st;
  a.o = static_cast<uint16_t*>(o);
  a.lse = lse;
  a.n_split = 1;
  if ((st = get_err_ptr(&a.err)) != FA_OK) return st;
  return fa::launch_fwd_bf16(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                   : FA_ERR_CUDA;
}

size_t fa_fwd_splitkv_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1 || num_splits < 1) return 0;
  const size_t rows = (size_t)num_splits * B * H * Nq;
  return round256(rows * (size_t)d * 4) + round256(rows * 4);
}

int fa_fwd_splitkv_default_splits(int B, int H, int Nq, int Nk, int d) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1) return 0;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 148;
  const long ctas = (long)B * H * ((Nq + 255) / 256);
  const long n_kv = (Nk + 127) / 128;
  // One CTA per (head, query-tile pair, split), in waves of one CTA per SM:
  // the split count whose grid wastes least of its last wave, i.e. the least
  // waves(s) * (key tiles per split + ~3 tiles of fixed cost per CTA), with
  // at least 4 key tiles per split and at most 128 splits.
  const long max_s = std::max(1L, std::min(128L, n_kv / 4));
  long best = 1;
  double best_t = 0.0;
  for (long s = 1; s <= max_s; ++s) {
    const double waves = (double)((ctas * s + sms - 1) / sms);
    const double t = waves * (double)((n_kv + s - 1) / s + 3);
    if (s == 1 || t < best_t) {
      best = s;
      best_t = t;
    }
  }
  return (int)best;
}

fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, const float* key_bias,
                         void* o, float* lse, int B, int H, int H_kv, int Nq, int Nk, int d,
                         float scale, int causal, int num_splits, void* workspace,
                         size_t workspace_bytes, void* stream) {
  fa_status st = check_problem(B, H, Nq, Nk, d, scale, FA_DTYPE_BF16, H_kv);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(workspace, 256) || !aligned(lse, 4) || (key_bias && !aligned(key_bias, 4)))
    return FA_ERR_INVALID_ARG;
  if (num_splits < 1 || num_splits > 1024) return FA_ERR_INVALID_ARG;
  if (workspace_bytes < fa_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, num_splits))
    return FA_ERR_INVALID_ARG;
  fa::Problem p{B, H, Nq, Nk, d, scale, causal ? 1 : 0, H_kv};
  fa::FwdBf16Args a;
  st = fwd_bf16_setup(&a, p, q, k, v, key_bias, o, lse);
  if (st != FA_OK) return st;
  if (num_splits > 1) {
    const size_t rows = (size_t)num_splits * B * H * Nq;
    a.n_split = num_splits;
    a.part_o = static_cast<float*>(workspace);
    a.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + round256(rows * d * 4));
  }
  return fa::launch_fwd_bf16(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                   : FA_ERR_CUDA;
}

size_t fa_bwd_workspace_size(int B, int H, int Nq, int Nk, int d) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1) return 0;
  return bwd_ws_bytes(B, H, Nq, (size_t)B * H * Nq, d);
}

size_t fa_bwd_varlen_workspace_size(int B, int H, int total_q, int max_seqlen_q, int d) {
  if (B < 1 || H < 1 || total_q < 1 || max_seqlen_q < 1 || d < 1) return 0;
  return bwd_ws_bytes(B, H, max_seqlen_q, (size_t)H * total_q, d);
}

size_t fa_bwd_deterministic_workspace_size(int B, int H, int Nq, int d) {
  if (B < 1 || H < 1 || Nq < 1 || d < 1) return 0;
  return bwd_ws_bytes(B, H, Nq, 0, d);
}

}  // extern "C"

namespace {

// Validation and argument set-up shared by fa_bwd and its three stages.
fa_status bwd_common(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dO, void* dq, void* dk, void* dv,
                     const float* key_bias, int B, int H, int Hkv, int Nq, int Nk, int d,
                     float scale, int causal, fa_dtype dtype, void* workspace,
                     size_t workspace_bytes, void* stream, unsigned stages,
                     const int* cu_q = nullptr, const int* cu_k = nullptr, int total_q = 0,
                     int total_k = 0) {
  fa_status st = check_problem(B, H, Nq, Nk, d, scale, dtype, Hkv);
  if (st != FA_OK) return st;
  const bool varlen = cu_q != nullptr;
  if (varlen && ((st = check_varlen(total_q, total_k, Nq, Nk, d, cu_q, cu_k)) != FA_OK)) return st;
  if (varlen && key_bias) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16) return FA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !workspace)
    return FA_ERR_INVALID_ARG;
  const void* p16[] = {q, k, v, o, dO, dq, dk, dv};
  for (const void* ptr : p16)
    if (!aligned(ptr, 16)) return FA_ERR_INVALID_ARG;
  if (!aligned(lse, 4) || (key_bias && !aligned(key_bias, 4)) || !aligned(workspace, 256))
    return FA_ERR_INVALID_ARG;
  const bool det = (stages & fa::BWD_DET) != 0;   // no dQ accumulator
  const size_t dq_rows = det ? 0 : varlen ? (size_t)H * total_q : (size_t)B * H * Nq;
  if (workspace_bytes < bwd_ws_bytes(B, H, Nq, dq_rows, d)) return FA_ERR_INVALID_ARG;

  fa::BwdBf16Args a{};
  a.p = fa::Problem{B, H, Nq, Nk, d, scale, causal ? 1 : 0, Hkv};
  a.p.cu_q = cu_q;
  a.p.cu_k = cu_k;
  a.p.total_q = total_q;
  a.p.total_k = total_k;
  // tensor-map views: (d, rows per head coordinate, head coordinates)
  const int qh = varlen ? H : B * H, kh = varlen ? Hkv : B * Hkv;
  const int qn = varlen ? total_q : Nq, kn = varlen ? total_k : Nk;
  if (stages & (fa::BWD_MAIN | fa::BWD_DQ)) {
    if ((st = make_map(&a.tm_q, q, qh, qn, d)) != FA_OK) return st;
    if ((st = make_map(&a.tm_k, k, kh, kn, d)) != FA_OK) return st;
    if ((st = make_map(&a.tm_v, v, kh, kn, d)) != FA_OK) return st;
    if ((st = make_map(&a.tm_do, dO, qh, qn, d)) != FA_OK) return st;
    if ((st = make_map(&a.tm_dk, dk, kh, kn, d)) != FA_OK) return st;
    if ((st = make_map(&a.tm_dv, dv, kh, kn, d)) != FA_OK) return st;
    if ((st = make_map(&a.tm_dq, dq, qh, qn, d)) != FA_OK) return st;
  }
  a.o = static_cast<const uint16_t*>(o);
  a.dO = static_cast<const uint16_t*>(dO);
  a.lse = lse;
  a.bias = key_bias;
  a.nq_pad = (Nq + 127) / 128 * 128;
  const size_t prow = (size_t)B * H * a.nq_pad;
  char* ws = static_cast<char*>(workspace);
  a.D = reinterpret_cast<float*>(ws);
  a.lse2 = reinterpret_cast<float*>(ws + round256(prow * 4));
  a.dq_acc = det ? nullptr : reinterpret_cast<float*>(ws + 2 * round256(prow * 4));
  a.sched = det ? nullptr
                : reinterpret_cast<int*>(ws + 2 * round256(prow * 4) +
                                         round256(dq_rows * (size_t)d * 4));
  if (!det && (stages & fa::BWD_MAIN) &&
      (st = make_map_f32_acc(&a.tm_dqacc, a.dq_acc, qh, qn, d)) != FA_OK)
    return st;
  a.dq = static_cast<uint16_t*>(dq);
  a.dk = static_cast<uint16_t*>(dk);
  a.dv = static_cast<uint16_t*>(dv);
  if ((st = get_err_ptr(&a.err)) != FA_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&a.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  cudaError_t e = fa::launch_bwd_bf16(a, static_cast<cudaStream_t>(stream), stages);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

#define FA_BWD_ARGS                                                                          \
  q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, H, Nq, Nk, d, scale, causal, dtype, workspace, \
      workspace_bytes, stream

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dO, void* dq, void* dk, void* dv, const float* key_bias, int B,
                 int H, int Nq, int Nk, int d, float scale, int causal, fa_dtype dtype,
                 void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_common(FA_BWD_ARGS, fa::BWD_PRE | fa::BWD_MAIN | fa::BWD_POST);
}

fa_status fa_bwd_preprocess(const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dO, void* dq, void* dk, void* dv,
                            const float* key_bias, int B, int H, int Nq, int Nk, int d,
                            float scale, int causal, fa_dtype dtype, void* workspace,
                            size_t workspace_bytes, void* stream) {
  return bwd_common(FA_BWD_ARGS, fa::BWD_PRE);
}

fa_status fa_bwd_main(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dO, void* dq, void* dk, void* dv,
                      const float* key_bias, int B, int H, int Nq, int Nk, int d, float scale,
                      int causal, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                      void* stream) {
  return bwd_common(FA_BWD_ARGS, fa::BWD_MAIN);
}

fa_status fa_bwd_postprocess(const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* dO, void* dq, void* dk, void* dv,
                             const float* key_bias, int B, int H, int Nq, int Nk, int d,
                             float scale, int causal, fa_dtype dtype, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return bwd_common(FA_BWD_ARGS, fa::BWD_POST);
}

#undef FA_BWD_ARGS

fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dO, void* dq, void* dk, void* dv,
                        const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H, int H_kv,
                        int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                        float scale, int causal, void* workspace, size_t workspace_bytes,
                        void* stream) {
  if (!cu_seqlens_q) return FA_ERR_INVALID_ARG;
  return bwd_common(q, k, v, o, lse, dO, dq, dk, dv, nullptr, B, H, H_kv, max_seqlen_q,
                    max_seqlen_k, d, scale, causal, FA_DTYPE_BF16, workspace, workspace_bytes,
                    stream, fa::BWD_PRE | fa::BWD_MAIN | fa::BWD_POST, cu_seqlens_q, cu_seqlens_k,
                    total_q, total_k);
}

fa_status fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dO, void* dq, void* dk, void* dv,
                     const float* key_bias, int B, int H, int H_kv, int Nq, int Nk, int d,
                     float scale, int causal, fa_dtype dtype, void* workspace,
                     size_t workspace_bytes, void* stream) {
  return bwd_common(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, H_kv, Nq, Nk, d, scale,
                    causal, dtype, workspace, workspace_bytes, stream,
                    fa::BWD_PRE | fa::BWD_MAIN | fa::BWD_POST);
}

fa_status fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dO, void* dq, void* dk, void* dv,
                               const float* key_bias, int B, int H, int H_kv, int Nq, int Nk,
                               int d, float scale, int causal, fa_dtype dtype, void* workspace,
                               size_t workspace_bytes, void* stream) {
  return bwd_common(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, H_kv, Nq, Nk, d, scale,
                    causal, dtype, workspace, workspace_bytes, stream,
                    fa::BWD_PRE | fa::BWD_MAIN | fa::BWD_DQ | fa::BWD_DET);
}

fa_status fa_bwd_deterministic_stage(const void* q, const void* k, const void* v, const void* o,
                                     const float* lse, const void* dO, void* dq, void* dk,
                                     void* dv, const float* key_bias, int B, int H, int H_kv,
                                     int Nq, int Nk, int d, float scale, int causal,
                                     fa_dtype dtype, void* workspace, size_t workspace_bytes,
                                     void* stream, int stage) {
  static const unsigned kStages[3] = {fa::BWD_PRE, fa::BWD_MAIN, fa::BWD_DQ};
  if (stage < 1 || stage > 3) return FA_ERR_INVALID_ARG;
  return bwd_common(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, H_kv, Nq, Nk, d, scale,
                    causal, dtype, workspace, workspace_bytes, stream,
                    kStages[stage - 1] | fa::BWD_DET);
}

fa_status fa_bwd_varlen_deterministic(const void* q, const void* k, const void* v,
                                      const void* o, const float* lse, const void* dO, void* dq,
                                      void* dk, void* dv, const int* cu_seqlens_q,
                                      const int* cu_seqlens_k, int B, int H, int H_kv,
                                      int total_q, int total_k, int max_seqlen_q,
                                      int max_seqlen_k, int d, float scale, int causal,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  if (!cu_seqlens_q) return FA_ERR_INVALID_ARG;
  return bwd_common(q, k, v, o, lse, dO, dq, dk, dv, nullptr, B, H, H_kv, max_seqlen_q,
                    max_seqlen_k, d, scale, causal, FA_DTYPE_BF16, workspace, workspace_bytes,
                    stream, fa::BWD_PRE | fa::BWD_MAIN | fa::BWD_DQ | fa::BWD_DET, cu_seqlens_q,
                    cu_seqlens_k, total_q, total_k);
}

size_t fa_fwd_fp8_workspace_size(int B, int H, int H_kv, int Nq, int Nk, int d) {
  if (B < 1 || H < 1 || H_kv < 1 || Nq < 1 || Nk < 1 || d < 1) return 0;
  return fp8_ws_layout(B, H, H_kv, Nq, Nk, d).total;
}

fa_status fa_fwd_fp8_stage(const void* q, const void* k, const void* v, const float* key_bias,
                           void* o, float* lse, int B, int H, int H_kv, int Nq, int Nk, int d,
                           float scale, int causal, void* workspace, size_t workspace_bytes,
                           void* stream, int stage) {
  if (stage < 0 || stage > 2) return FA_ERR_INVALID_ARG;
  fa_status st = check_problem(B, H, Nq, Nk, d, scale, FA_DTYPE_BF16, H_kv);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || (key_bias && !aligned(key_bias, 4)) || !aligned(workspace, 256))
    return FA_ERR_INVALID_ARG;
  const Fp8Ws w = fp8_ws_layout(B, H, H_kv, Nq, Nk, d);
  if (workspace_bytes < w.total) return FA_ERR_INVALID_ARG;
  char* ws = static_cast<char*>(workspace);
  float* amax = reinterpret_cast<float*>(ws + w.amax);
  const int nk16 = (Nk + 15) / 16 * 16;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (stage == 0 || stage == 1) {
    fa::QuantFp8Args qa;
    qa.q = static_cast<const uint16_t*>(q);
    qa.k = static_cast<const uint16_t*>(k);
    qa.v = static_cast<const uint16_t*>(v);
    qa.q8 = reinterpret_cast<uint8_t*>(ws + w.q8);
    qa.k8 = reinterpret_cast<uint8_t*>(ws + w.k8);
    qa.vt8 = reinterpret_cast<uint8_t*>(ws + w.vt8);
    qa.amax_q = amax;
    qa.amax_k = amax + (size_t)B * H;
    qa.amax_v = amax + (size_t)B * H + (size_t)B * H_kv;
    qa.heads_q = B * H;
    qa.heads_kv = B * H_kv;
    qa.Nq = Nq;
    qa.Nk = Nk;
    qa.nk16 = nk16;
    qa.d = d;
    if (cudaMemsetAsync(amax, 0, w.q8, s) != cudaSuccess) return FA_ERR_CUDA;
    if (fa::launch_quant_fp8(qa, s) != cudaSuccess) return FA_ERR_CUDA;
  }
  if (stage == 0 || stage == 2) {
    fa::FwdBf16Args a{};
    a.p = fa::Problem{B, H, Nq, Nk, d, scale, causal ? 1 : 0, H_kv};
    if ((st = make_map_u8(&a.tm_q, ws + w.q8, d, Nq, (long)B * H)) != FA_OK) return st;
    if ((st = make_map_u8(&a.tm_k, ws + w.k8, d, Nk, (long)B * H_kv)) != FA_OK) return st;
    if ((st = make_map_u8(&a.tm_v, ws + w.vt8, nk16, d, (long)B * H_kv)) != FA_OK) return st;
    if ((st = make_map(&a.tm_o, o, B * H, Nq, d)) != FA_OK) return st;
    a.bias = key_bias;
    a.o = static_cast<uint16_t*>(o);
    a.lse = lse;
    a.n_split = 1;
    a.amax_q = amax;
    a.amax_k = amax + (size_t)B * H;
    a.amax_v = amax + (size_t)B * H + (size_t)B * H_kv;
    if ((st = get_err_ptr(&a.err)) != FA_OK) return st;
    if (fa::launch_fwd_fp8(a, s) != cudaSuccess) return FA_ERR_CUDA;
  }
  return FA_OK;
}

fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, const float* key_bias, void* o,
                     float* lse, int B, int H, int H_kv, int Nq, int Nk, int d, float scale,
                     int causal, void* workspace, size_t workspace_bytes, void* stream) {
  return fa_fwd_fp8_stage(q, k, v, key_bias, o, lse, B, H, H_kv, Nq, Nk, d, scale, causal,
                          workspace, workspace_bytes, stream, 0);
}

fa_status fa_selftest_device_timeout(void* stream) {
  uint32_t* err = nullptr;
  fa_status st = get_err_ptr(&err);
  if (st != FA_OK) return st;
  selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_get_last_device_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  uint32_t w = 0;
  if (cudaMemcpyFromSymbol(&w, g_fa_err_word, sizeof(w)) != cudaSuccess) return FA_ERR_CUDA;
  if (w) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_fa_err_word, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
    return FA_ERR_DEVICE;
  }
  return FA_OK;
}

}  // extern "C"
