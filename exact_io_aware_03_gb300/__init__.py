"""Python binding of the GB300 exact-attention C ABI (include/fa.h).

The functions ``fa_fwd``, ``fa_bwd``, ``fa_bwd_workspace_size``,
``fa_status_string`` and ``fa_get_last_device_error`` have the C names and
arguments (integers for pointers and the stream). ``fwd`` and ``bwd`` are thin
conveniences over them for torch CUDA tensors: they only allocate the output
tensors with torch and marshal pointers; every step of the computation runs
in the library's CUDA kernels. There is no CPU or PyTorch fallback: if the
library is not built, every call raises.
"""
import ctypes
import os

from . import build as _build

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_DEVICE = range(5)
FA_DTYPE_BF16, FA_DTYPE_FP32 = 0, 1

_lib = None


class FaError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        msg = fa_status_string(status) if _lib is not None else "status %d" % status
        super().__init__("%s%s" % (where + ": " if where else "", msg))


def library_path():
    return _build.LIB


def load(path=None):
    """Load libfa_gb300.so (built by ``build.build()``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise ImportError("libfa_gb300.so not found at %s: run "
                          "exact_io_aware_03_gb300.build.build() first" % path)
    lib = ctypes.CDLL(path)
    vp, cint, cf, csz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, vp, cint, cint, cint, cint, cint, cf, cint,
                           cint, vp]
    lib.fa_fwd.restype = cint
    lib.fa_bwd_workspace_size.argtypes = [cint] * 5
    lib.fa_bwd_workspace_size.restype = csz
    lib.fa_fwd_splitkv_workspace_size.argtypes = [cint] * 6
    lib.fa_fwd_splitkv_workspace_size.restype = csz
    lib.fa_fwd_splitkv_default_splits.argtypes = [cint] * 5
    lib.fa_fwd_splitkv_default_splits.restype = cint
    lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, vp, cint, cint, cint, cint, cint, cint, cf,
                                   cint, cint, vp, csz, vp]
    lib.fa_fwd_varlen.argtypes = [vp] * 7 + [cint] * 8 + [cf, cint, vp]
    lib.fa_fwd_varlen.restype = cint
    lib.fa_bwd_varlen.argtypes = [vp] * 11 + [cint] * 8 + [cf, cint, vp, csz, vp]
    lib.fa_bwd_varlen.restype = cint
    lib.fa_bwd_varlen_workspace_size.argtypes = [cint] * 5
    lib.fa_bwd_varlen_workspace_size.restype = csz
    lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, cint, cint, cint, cint, cint, cint, cf,
                               cint, cint, vp]
    lib.fa_fwd_gqa.restype = cint
    lib.fa_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, cint, cint, cint, cint,
                               cint, cint, cf, cint, cint, vp, csz, vp]
    lib.fa_bwd_gqa.restype = cint
    lib.fa_fwd_splitkv.restype = cint
    lib.fa_fwd_fp8_workspace_size.argtypes = [cint] * 6
    lib.fa_fwd_fp8_workspace_size.restype = csz
    lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, cint, cint, cint, cint, cint, cint, cf,
                               cint, vp, csz, vp]
    lib.fa_fwd_fp8.restype = cint
    lib.fa_fwd_fp8_stage.argtypes = list(lib.fa_fwd_fp8.argtypes) + [cint]
    lib.fa_fwd_fp8_stage.restype = cint
    lib.fa_bwd_deterministic_workspace_size.argtypes = [cint] * 4
    lib.fa_bwd_deterministic_workspace_size.restype = csz
    lib.fa_bwd_deterministic.argtypes = list(lib.fa_bwd_gqa.argtypes)
    lib.fa_bwd_deterministic.restype = cint
    lib.fa_bwd_deterministic_stage.argtypes = list(lib.fa_bwd_gqa.argtypes) + [cint]
    lib.fa_bwd_deterministic_stage.restype = cint
    lib.fa_bwd_varlen_deterministic.argtypes = list(lib.fa_bwd_varlen.argtypes)
    lib.fa_bwd_varlen_deterministic.restype = cint
    for name in ("fa_bwd", "fa_bwd_preprocess", "fa_bwd_main", "fa_bwd_postprocess"):
        f = getattr(lib, name)
        f.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, cint, cint, cint, cint, cint,
                      cf, cint, cint, vp, csz, vp]
        f.restype = cint
    lib.fa_status_string.argtypes = [cint]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_get_last_device_error.argtypes = [vp]
    lib.fa_get_last_device_error.restype = cint
    lib.fa_selftest_device_timeout.argtypes = [vp]
    lib.fa_selftest_device_timeout.restype = cint
    _lib = lib
    return lib


# ------------------------------------------------------------------ C names

def fa_fwd(q, k, v, key_bias, o, lse, B, H, Nq, Nk, d, scale, causal, dtype, stream):
    return load().fa_fwd(q, k, v, key_bias, o, lse, B, H, Nq, Nk, d, scale, causal, dtype,
                         stream)


def fa_fwd_splitkv(q, k, v, key_bias, o, lse, B, H, H_kv, Nq, Nk, d, scale, causal, num_splits,
                   workspace, workspace_bytes, stream):
    return load().fa_fwd_splitkv(q, k, v, key_bias, o, lse, B, H, H_kv, Nq, Nk, d, scale, causal,
                                 num_splits, workspace, workspace_bytes, stream)


def fa_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, H, H_kv, total_q, total_k,
                  max_seqlen_q, max_seqlen_k, d, scale, causal, stream):
    return load().fa_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, H, H_kv, total_q,
                                total_k, max_seqlen_q, max_seqlen_k, d, scale, causal, stream)


def fa_bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, B, H, H_kv,
                  total_q, total_k, max_seqlen_q, max_seqlen_k, d, scale, causal, workspace,
                  workspace_bytes, stream):
    return load().fa_bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, B, H,
                                H_kv, total_q, total_k, max_seqlen_q, max_seqlen_k, d, scale,
                                causal, workspace, workspace_bytes, stream)


def fa_bwd_varlen_workspace_size(B, H, total_q, max_seqlen_q, d):
    return load().fa_bwd_varlen_workspace_size(B, H, total_q, max_seqlen_q, d)


def fa_fwd_gqa(q, k, v, key_bias, o, lse, B, H, H_kv, Nq, Nk, d, scale, causal, dtype, stream):
    return load().fa_fwd_gqa(q, k, v, key_bias, o, lse, B, H, H_kv, Nq, Nk, d, scale, causal,
                             dtype, stream)


def fa_bwd_gqa(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, H_kv, Nq, Nk, d, scale, causal,
               dtype, workspace, workspace_bytes, stream):
    return load().fa_bwd_gqa(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, H_kv, Nq, Nk, d,
                             scale, causal, dtype, workspace, workspace_bytes, stream)


def fa_fwd_fp8_workspace_size(B, H, H_kv, Nq, Nk, d):
    return load().fa_fwd_fp8_workspace_size(B, H, H_kv, Nq, Nk, d)


def fa_fwd_fp8(q, k, v, key_bias, o, lse, B, H, H_kv, Nq, Nk, d, scale, causal, workspace,
               workspace_bytes, stream):
    return load().fa_fwd_fp8(q, k, v, key_bias, o, lse, B, H, H_kv, Nq, Nk, d, scale, causal,
                             workspace, workspace_bytes, stream)


def fa_fwd_fp8_stage(q, k, v, key_bias, o, lse, B, H, H_kv, Nq, Nk, d, scale, causal, workspace,
                     workspace_bytes, stream, stage):
    return load().fa_fwd_fp8_stage(q, k, v, key_bias, o, lse, B, H, H_kv, Nq, Nk, d, scale, causal,
                                   workspace, workspace_bytes, stream, stage)


def fa_bwd_deterministic_workspace_size(B, H, Nq, d):
    return load().fa_bwd_deterministic_workspace_size(B, H, Nq, d)


def fa_bwd_deterministic(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, H_kv, Nq, Nk, d, scale,
                         causal, dtype, workspace, workspace_bytes, stream):
    return load().fa_bwd_deterministic(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, H_kv, Nq,
                                       Nk, d, scale, causal, dtype, workspace, workspace_bytes,
                                       stream)


def fa_bwd_deterministic_stage(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, H_kv, Nq, Nk, d,
                               scale, causal, dtype, workspace, workspace_bytes, stream, stage):
    return load().fa_bwd_deterministic_stage(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H,
                                             H_kv, Nq, Nk, d, scale, causal, dtype, workspace,
                                             workspace_bytes, stream, stage)


def fa_bwd_varlen_deterministic(q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, B, H,
                                H_kv, total_q, total_k, max_seqlen_q, max_seqlen_k, d, scale,
                                causal, workspace, workspace_bytes, stream):
    return load().fa_bwd_varlen_deterministic(q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens_q,
                                              cu_seqlens_k, B, H, H_kv, total_q, total_k,
                                              max_seqlen_q, max_seqlen_k, d, scale, causal,
                                              workspace, workspace_bytes, stream)


def fa_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, num_splits):
    return load().fa_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, num_splits)


def fa_fwd_splitkv_default_splits(B, H, Nq, Nk, d):
    return load().fa_fwd_splitkv_default_splits(B, H, Nq, Nk, d)


def fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, Nq, Nk, d, scale, causal, dtype,
           workspace, workspace_bytes, stream):
    return load().fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, Nq, Nk, d, scale,
                         causal, dtype, workspace, workspace_bytes, stream)


def fa_bwd_preprocess(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, Nq, Nk, d, scale, causal,
                      dtype, workspace, workspace_bytes, stream):
    return load().fa_bwd_preprocess(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, Nq, Nk, d,
                                    scale, causal, dtype, workspace, workspace_bytes, stream)


def fa_bwd_main(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, Nq, Nk, d, scale, causal,
                dtype, workspace, workspace_bytes, stream):
    return load().fa_bwd_main(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, Nq, Nk, d, scale,
                              causal, dtype, workspace, workspace_bytes, stream)


def fa_bwd_postprocess(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, Nq, Nk, d, scale, causal,
                       dtype, workspace, workspace_bytes, stream):
    return load().fa_bwd_postprocess(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, Nq, Nk, d,
                                     scale, causal, dtype, workspace, workspace_bytes, stream)


def fa_bwd_workspace_size(B, H, Nq, Nk, d):
    return load().fa_bwd_workspace_size(B, H, Nq, Nk, d)


def fa_status_string(status):
    return load().fa_status_string(status).decode()


def fa_get_last_device_error(stream):
    return load().fa_get_last_device_error(stream)


def fa_selftest_device_timeout(stream):
    return load().fa_selftest_device_timeout(stream)


FA_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def fa_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, Nq, Nk, d, scale, causal,
                   dtype, stream):
    """fa_bwd without a workspace argument: the library's own fixed device
    array (FA_NOALLOC_SCRATCH_BYTES) serves as the workspace, for callers that
    cannot allocate device memory. Calls that overlap on the GPU race."""
    lib = load()
    f = lib.fa_bwd_noalloc
    if f.restype is not ctypes.c_int or not f.argtypes:
        vp, cint, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        f.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, cint, cint, cint, cint, cint, cf,
                      cint, cint, vp]
        f.restype = cint
    return f(q, k, v, o, lse, dO, dq, dk, dv, key_bias, B, H, Nq, Nk, d, scale, causal, dtype,
             stream)


# ------------------------------------------------------------------ torch conveniences

def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return FA_DTYPE_BF16
    if t.dtype == torch.float32:
        return FA_DTYPE_FP32
    raise TypeError("q/k/v must be bfloat16 or float32, got %s" % t.dtype)


def _check(t, name):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous [B, H, N, d]" % name)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(t):
    import torch
    return torch.cuda.current_stream(t.device).cuda_stream


def fwd(q, k, v, key_bias=None, causal=False, scale=None, out=None, lse=None):
    """O [B,H,Nq,d] (q's dtype) and LSE [B,H,Nq] (fp32) for CUDA tensors [B,H,N,d].

    Calls fa_fwd (fa_fwd_gqa when k, v have fewer heads than q)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    if key_bias is not None:
        _check(key_bias, "key_bias")
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        if Hkv == H:
            name = "fa_fwd"
            st = fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(key_bias), _ptr(out), _ptr(lse),
                        B, H, Nq, Nk, d, float(scale), int(bool(causal)), _dtype_code(q),
                        _stream(q))
        else:
            name = "fa_fwd_gqa"
            st = fa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(key_bias), _ptr(out), _ptr(lse),
                            B, H, Hkv, Nq, Nk, d, float(scale), int(bool(causal)),
                            _dtype_code(q), _stream(q))
    if st != FA_OK:
        raise FaError(st, name)
    return out, lse


def fwd_fp8(q, k, v, key_bias=None, causal=False, scale=None, out=None, lse=None, workspace=None,
            stage=0):
    """FP8 forward (fa_fwd_fp8): bf16 q, k, v quantized to e4m3 per head into
    ``workspace``, attention on the tensor cores' fp8 path; bf16 O, fp32 LSE.
    stage: 0 both, 1 quantization only, 2 attention only (from the workspace)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = d ** -0.5
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    if workspace is None:
        workspace = torch.empty(fa_fwd_fp8_workspace_size(B, H, Hkv, Nq, Nk, d), dtype=torch.uint8,
                                device=q.device)
    with torch.cuda.device(q.device):
        st = fa_fwd_fp8_stage(_ptr(q), _ptr(k), _ptr(v), _ptr(key_bias), _ptr(out), _ptr(lse), B, H,
                              Hkv, Nq, Nk, d, float(scale), int(bool(causal)), _ptr(workspace),
                              workspace.numel(), _stream(q), int(stage))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_fp8")
    return out, lse


def fwd_splitkv(q, k, v, key_bias=None, causal=False, scale=None, num_splits=None, out=None,
                lse=None, workspace=None):
    """Split-KV forward (bf16): same results as ``fwd``; num_splits=None picks a
    split count that fills the device."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = d ** -0.5
    if num_splits is None:
        with torch.cuda.device(q.device):
            num_splits = fa_fwd_splitkv_default_splits(B, H, Nq, Nk, d)
    out = torch.empty_like(q) if out is None else out
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(max(1, fa_fwd_splitkv_workspace_size(B, H, Nq, Nk, d,
                                                                     num_splits)),
                                dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        st = fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(key_bias), _ptr(out), _ptr(lse),
                            B, H, Hkv, Nq, Nk, d, float(scale), int(bool(causal)), int(num_splits),
                            _ptr(workspace), workspace.numel(), _stream(q))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_splitkv")
    return out, lse


def _varlen_meta(cu_q, cu_k):
    """B, total and max lengths of int32 offset tensors (read once on the host)."""
    cq, ck = cu_q.detach().cpu().tolist(), cu_k.detach().cpu().tolist()
    B = len(cq) - 1
    return (B, cq[-1], ck[-1], max(cq[i + 1] - cq[i] for i in range(B)),
            max(ck[i + 1] - ck[i] for i in range(B)))


def fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, causal=False, scale=None, out=None,
               lse=None, max_seqlen_q=None, max_seqlen_k=None):
    """Packed sequences: q [H, total_q, d], k/v [H_kv, total_k, d] bf16 CUDA tensors,
    cu_seqlens int32 CUDA tensors [B+1]. Returns O [H, total_q, d], LSE [H, total_q]."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (cu_seqlens_q, "cu_seqlens_q"),
                 (cu_seqlens_k, "cu_seqlens_k")):
        _check(t, n)
    H, total_q, d = q.shape
    Hkv, total_k = k.shape[0], k.shape[1]
    B, tq, tk, mq, mk = _varlen_meta(cu_seqlens_q, cu_seqlens_k)
    max_seqlen_q = max(1, mq) if max_seqlen_q is None else max_seqlen_q
    max_seqlen_k = max(1, mk) if max_seqlen_k is None else max_seqlen_k
    if scale is None:
        scale = d ** -0.5
    out = torch.empty_like(q) if out is None else out
    if lse is None:
        lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        st = fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q),
                           _ptr(cu_seqlens_k), B, H, Hkv, total_q, total_k, max_seqlen_q,
                           max_seqlen_k, d, float(scale), int(bool(causal)), _stream(q))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_varlen")
    return out, lse


def bwd_varlen(q, k, v, o, lse, dO, cu_seqlens_q, cu_seqlens_k, causal=False, scale=None,
               workspace=None, dq=None, dk=None, dv=None, max_seqlen_q=None, max_seqlen_k=None,
               deterministic=False):
    """Backward of ``fwd_varlen`` (packed [H, total, d] tensors).

    deterministic: use fa_bwd_varlen_deterministic (bitwise reproducible dq).
    """
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (lse, "lse"), (dO, "dO")):
        _check(t, n)
    H, total_q, d = q.shape
    Hkv, total_k = k.shape[0], k.shape[1]
    B, tq, tk, mq, mk = _varlen_meta(cu_seqlens_q, cu_seqlens_k)
    max_seqlen_q = max(1, mq) if max_seqlen_q is None else max_seqlen_q
    max_seqlen_k = max(1, mk) if max_seqlen_k is None else max_seqlen_k
    if scale is None:
        scale = d ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        nbytes = (fa_bwd_deterministic_workspace_size(B, H, max_seqlen_q, d) if deterministic
                  else fa_bwd_varlen_workspace_size(B, H, total_q, max_seqlen_q, d))
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    fn = fa_bwd_varlen_deterministic if deterministic else fa_bwd_varlen
    with torch.cuda.device(q.device):
        st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                           _ptr(dk), _ptr(dv), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B, H, Hkv,
                           total_q, total_k, max_seqlen_q, max_seqlen_k, d, float(scale),
                           int(bool(causal)), _ptr(workspace), workspace.numel(), _stream(q))
    if st != FA_OK:
        raise FaError(st, fn.__name__)
    return dq, dk, dv


def bwd(q, k, v, o, lse, dO, key_bias=None, causal=False, scale=None, workspace=None,
        dq=None, dk=None, dv=None, stage=None, deterministic=False):
    """dQ, dK, dV (q's dtype) for CUDA tensors; o and lse from ``fwd`` on the same inputs.

    Calls fa_bwd (fa_bwd_gqa when k, v have fewer heads than q).

    stage: None runs the whole backward (fa_bwd); "preprocess", "main" or
    "postprocess" runs only that launch (the three in order equal fa_bwd).
    deterministic: use fa_bwd_deterministic (bitwise reproducible dq); its
    stages are "preprocess", "dkdv" and "dq".
    """
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (lse, "lse"), (dO, "dO")):
        _check(t, n)
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = d ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = (fa_bwd_deterministic_workspace_size(B, H, Nq, d) if deterministic
                else fa_bwd_workspace_size(B, H, Nq, Nk, d))
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    if deterministic:
        extra = ()
        if stage is None:
            fn = fa_bwd_deterministic
        else:
            fn = fa_bwd_deterministic_stage
            extra = ({"preprocess": 1, "dkdv": 2, "dq": 3}[stage],)
        with torch.cuda.device(q.device):
            st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                    _ptr(dk), _ptr(dv), _ptr(key_bias), B, H, Hkv, Nq, Nk, d, float(scale),
                    int(bool(causal)), _dtype_code(q), _ptr(workspace), workspace.numel(),
                    _stream(q), *extra)
        if st != FA_OK:
            raise FaError(st, fn.__name__)
        return dq, dk, dv
    if stage is None and Hkv == H:
        fn = fa_bwd
        heads = (B, H)
    elif stage is None:
        fn = fa_bwd_gqa
        heads = (B, H, Hkv)
    else:
        if Hkv != H:
            raise ValueError("the single-stage backward calls take H_kv == H")
        fn = {"preprocess": fa_bwd_preprocess, "main": fa_bwd_main,
              "postprocess": fa_bwd_postprocess}[stage]
        heads = (B, H)
    with torch.cuda.device(q.device):
        st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                _ptr(dk), _ptr(dv), _ptr(key_bias), *heads, Nq, Nk, d, float(scale),
                int(bool(causal)), _dtype_code(q), _ptr(workspace), workspace.numel(),
                _stream(q))
    if st != FA_OK:
        raise FaError(st, fn.__name__)
    return dq, dk, dv


def check_device_error(device=None):
    """Synchronise the current stream and raise if a kernel reported a device-side timeout."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        st = fa_get_last_device_error(torch.cuda.current_stream(dev).cuda_stream)
    if st != FA_OK:
        raise FaError(st, "device")
