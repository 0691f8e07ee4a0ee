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


# Every comparison made in this process, in order: the achieved errors next to
# the gates (tests/conftest.py writes them out when FA_PARITY_REPORT is set).
REPORT = []


def compare(name, got, ref, dtype="bf16", extra=""):
    """got: torch tensor (any device/dtype); ref: float64 numpy array of the same shape."""
    g = got.detach().double().cpu().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (name, g.shape, ref.shape)
    finite = bool(np.all(np.isfinite(g)))
    err = np.abs(g - ref)
    max_abs = float(err.max()) if err.size else 0.0
    if dtype == "fp32":
        REPORT.append({"case": extra, "tensor": name, "dtype": dtype, "n": int(ref.size),
                       "max_abs": max_abs, "gate_max_abs": F32_ATOL, "finite": finite})
        assert finite, "%s: non-finite output %s" % (name, extra)
        assert max_abs <= F32_ATOL, "%s: max-abs %.3e > %.1e %s" % (name, max_abs, F32_ATOL, extra)
        return {"max_abs": max_abs}
    floor = bf16_floor(ref)
    nrm = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(g - ref)) / nrm if nrm > 0 else float(np.linalg.norm(g))
    REPORT.append({"case": extra, "tensor": name, "dtype": dtype, "n": int(ref.size),
                   "max_abs": max_abs, "floor": floor, "gate_max_abs": BF16_ATOL + floor,
                   "needs_floor": max_abs > BF16_ATOL, "max_abs_ref": float(np.abs(ref).max())
                   if ref.size else 0.0, "rel_l2": rel, "gate_rel_l2": BF16_REL_L2,
                   "finite": finite})
    assert finite, "%s: non-finite output %s" % (name, extra)
    assert max_abs <= BF16_ATOL + floor, "%s: max-abs %.3e > %.1e + floor %.3e %s" % (
        name, max_abs, BF16_ATOL, floor, extra)
    assert rel <= BF16_REL_L2, "%s: rel-L2 %.3e > %.1e %s" % (name, rel, BF16_REL_L2, extra)
    return {"max_abs": max_abs, "rel_l2": rel, "floor": floor}


def compare_lse(got, ref, atol=LSE_ATOL, extra=""):
    g = got.detach().double().cpu().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape
    ninf = np.isneginf(ref)
    same_inf = bool(np.array_equal(np.isneginf(g), ninf))
    fin = ~ninf
    err = float(np.abs(g[fin] - ref[fin]).max()) if fin.any() and same_inf else 0.0
    REPORT.append({"case": extra, "tensor": "LSE", "dtype": "fp32", "n": int(ref.size),
                   "max_abs": err, "gate_max_abs": atol, "neg_inf_rows": int(ninf.sum()),
                   "neg_inf_pattern_equal": same_inf})
    assert same_inf, "LSE: -inf pattern differs %s" % extra
    assert err <= atol, "LSE: max-abs %.3e > %.1e %s" % (err, atol, extra)
    return err


def write_report(path):
    """The comparisons of this process as a markdown table (and JSON beside it)."""
    import json
    with open(path + ".json", "w") as f:
        json.dump(REPORT, f, indent=1)
    lines = ["| case | tensor | n | max-abs | bf16 floor | max-abs gate | needs floor | "
             "rel-L2 (gate 5e-3) |", "|---|---|---|---|---|---|---|---|"]
    for r in REPORT:
        lines.append("| %s | %s | %d | %.2e | %s | %.2e | %s | %s |" % (
            r["case"], r["tensor"], r["n"], r["max_abs"],
            "%.2e" % r["floor"] if "floor" in r else "-", r["gate_max_abs"],
            ("yes" if r.get("needs_floor") else "no") if "floor" in r else "-",
            "%.2e" % r["rel_l2"] if "rel_l2" in r else "-"))
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")


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
