"""Helpers shared by the GPU parity tests: tolerances, comparisons against the
fp64 oracle, and guard bands around outputs.

Tolerances (bf16 I/O): max-abs <= 1e-2 + floor and relative L2 <= 5e-3 on O
and on the gradients; |LSE error| <= 1e-3. `floor` is max |bf16(ref) - ref|,
the error that rounding the exact answer to bf16 alone already makes; it is
added because a correctly rounded bf16 output of magnitude >= 2 already
differs from the exact value by up to 2^-8 * |x| / 2. fp32 I/O: max-abs <= 1e-5.
"""
import numpy as np
import torch

BF16_ATOL = 1e-2
BF16_REL_L2 = 5e-3
LSE_ATOL = 1e-3
F32_ATOL = 1e-5


def bf16_floor(ref):
    r = torch.from_numpy(np.ascontiguousarray(ref))
    return float((r.to(torch.bfloat16).double() - r).abs().max()) if r.numel() else 0.0


def compare(name, got, ref, dtype="bf16", extra=""):
    """got: torch tensor (any device/dtype); ref: float64 numpy array of the same shape."""
    g = got.detach().double().cpu().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (name, g.shape, ref.shape)
    assert np.all(np.isfinite(g)), "%s: non-finite output %s" % (name, extra)
    err = np.abs(g - ref)
    max_abs = float(err.max()) if err.size else 0.0
    if dtype == "fp32":
        assert max_abs <= F32_ATOL, "%s: max-abs %.3e > %.1e %s" % (name, max_abs, F32_ATOL, extra)
        return {"max_abs": max_abs}
    floor = bf16_floor(ref)
    nrm = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(g - ref)) / nrm if nrm > 0 else float(np.linalg.norm(g))
    assert max_abs <= BF16_ATOL + floor, "%s: max-abs %.3e > %.1e + floor %.3e %s" % (
        name, max_abs, BF16_ATOL, floor, extra)
    assert rel <= BF16_REL_L2, "%s: rel-L2 %.3e > %.1e %s" % (name, rel, BF16_REL_L2, extra)
    return {"max_abs": max_abs, "rel_l2": rel, "floor": floor}


def compare_lse(got, ref, atol=LSE_ATOL, extra=""):
    g = got.detach().double().cpu().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape
    ninf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(g), ninf), "LSE: -inf pattern differs %s" % extra
    fin = ~ninf
    if fin.any():
        err = float(np.abs(g[fin] - ref[fin]).max())
        assert err <= atol, "LSE: max-abs %.3e > %.1e %s" % (err, atol, extra)
        return err
    return 0.0


class Guarded:
    """A contiguous CUDA tensor of `shape` carved from the middle of a larger
    buffer whose head and tail are filled with a sentinel, so that writes past
    either end are detected by `check()`."""

    PAD = 4096   # elements on each side (multiple of 16 bytes for every dtype used)

    def __init__(self, shape, dtype, device="cuda", fill=None):
        n = int(np.prod(shape))
        self.n = n
        self.buf = torch.empty(n + 2 * self.PAD, dtype=dtype, device=device)
        self.sentinel = torch.tensor(0xA5 if not dtype.is_floating_point else -12345.0,
                                     dtype=dtype)
        self.buf.fill_(self.sentinel.item())
        self.t = self.buf[self.PAD:self.PAD + n].view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def check(self, name=""):
        head = self.buf[:self.PAD]
        tail = self.buf[self.PAD + self.n:]
        s = self.sentinel.item()
        assert bool((head == s).all()) and bool((tail == s).all()), \
            "%s: write outside the output tensor" % name
