"""Run the library's kernels on a named workload a few times, for profilers.

    python -m exact_io_aware_03_gb300.profile_case --workload NAME [--pass fwd|bwd|both]
                                                   [--iters N] [--causal 0|1]
                                                   [--deterministic] [--fp8]
                                                   [--splitkv] [--nk N]

Inputs are the seeded synthetic tensors of `workloads.py`. Each iteration runs
fa_fwd (or fa_fwd_fp8, or fa_fwd_splitkv with its default split count) and/or
fa_bwd (or fa_bwd_deterministic) once on the current stream; the script synchronises and
checks the device error word at the end. Nothing is timed or compared: this
is the small, self-contained command to put under `ncu`.
"""
import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None):
    import torch

    import exact_io_aware_03_gb300 as fa
    import workloads
    from exact_io_aware_03_gb300 import build

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="bf16_b4h16_n4096_d128_causal_bwd",
                    choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--pass", dest="which", choices=["fwd", "bwd", "both"], default="both")
    ap.add_argument("--iters", type=int, default=2)
    ap.add_argument("--causal", type=int, choices=[0, 1], default=None,
                    help="override the workload's causal flag")
    ap.add_argument("--deterministic", action="store_true",
                    help="run fa_bwd_deterministic instead of fa_bwd")
    ap.add_argument("--fp8", action="store_true",
                    help="forward: run fa_fwd_fp8 (e4m3) instead of fa_fwd")
    ap.add_argument("--splitkv", action="store_true",
                    help="forward: run fa_fwd_splitkv with its default split count")
    ap.add_argument("--nk", type=int, default=None, help="override the workload's key count")
    args = ap.parse_args(argv)

    w = workloads.WORKLOADS[args.workload]
    if args.causal is not None:
        w = w.with_(causal=bool(args.causal))
    if args.nk is not None:
        w = w.with_(Nk=args.nk)
    build.build()
    fa.load()
    dev = torch.device("cuda", 0)
    x = workloads.make_inputs(w, with_dO=True)
    q, k, v, dO = (x[n].to(dev) for n in ("q", "k", "v", "dO"))
    bias = None if x["bias"] is None else x["bias"].to(dev)
    kw = dict(key_bias=bias, causal=w.causal, scale=w.scale)
    o, lse = fa.fwd(q, k, v, **kw)
    if w.dtype == "bf16":
        ws_bytes = (fa.fa_bwd_deterministic_workspace_size(w.B, w.H, w.Nq, w.d)
                    if args.deterministic else fa.fa_bwd_workspace_size(w.B, w.H, w.Nq, w.Nk, w.d))
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if args.splitkv:
        with torch.cuda.device(dev):
            ns = fa.fa_fwd_splitkv_default_splits(w.B, w.H, w.Nq, w.Nk, w.d)
        wsk = torch.empty(max(1, fa.fa_fwd_splitkv_workspace_size(w.B, w.H, w.Nq, w.Nk, w.d, ns)),
                          dtype=torch.uint8, device=dev)
    for _ in range(args.iters):
        if args.which in ("fwd", "both"):
            if args.splitkv:
                fa.fwd_splitkv(q, k, v, num_splits=ns, out=o, lse=lse, workspace=wsk, **kw)
            elif args.fp8:
                fa.fwd_fp8(q, k, v, out=o, lse=lse, **kw)
            else:
                fa.fwd(q, k, v, out=o, lse=lse, **kw)
        if args.which in ("bwd", "both") and w.dtype == "bf16":
            fa.bwd(q, k, v, o, lse, dO, workspace=ws, dq=dq, dk=dk, dv=dv,
                   deterministic=args.deterministic, **kw)
    torch.cuda.synchronize(dev)
    fa.check_device_error(dev)
    print("ok: %s %s x%d" % (w.name, args.which, args.iters))
    return 0


if __name__ == "__main__":
    sys.exit(main())
