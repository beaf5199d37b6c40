"""Run a few forwards of a seeded synthetic layer, for profilers (ncu) and phase traces.

    python -m quantized_moe_noaux_b300.profile_run --layer glm52 --tokens 1 --iters 5
    python -m quantized_moe_noaux_b300.profile_run --layer glm52_skewed --tokens 2048 --path grouped
    python -m quantized_moe_noaux_b300.profile_run --layer glm52 --tokens 1 --trace trace.npy

Each iteration is one ``moe_layer_forward`` on fresh seeded activations. ``--copies`` layer
copies are used in turn so consecutive forwards read different weights (as in the
benchmark). ``--trace`` records the last iteration's per-CTA trace (``moe_layer_set_trace``: the decode
kernel's phase timestamps in ns, the grouped GEMMs' per-role wait cycles) and saves it as a
numpy array [CTAs, 64].
No comparison against a reference is made here: the tests do that.
"""

from __future__ import annotations

import argparse
import os
import sys

import numpy as np

PHASES = ["start", "activation panel", "router rows", "all router rows seen", "shared gate/up",
          "shared gate/up seen", "shared down", "routing seen", "routed gate/up",
          "first routed gate/up seen", "routed down", "all down seen", "output written",
          "producer: shared issued", "producer: routing seen"]

GEMM_SLOTS = ["kernel", "mma_wait_operands", "mma_wait_accumulator", "dq_wait_weights",
              "dq_wait_stage", "act_producer_wait", "w_producer_wait", "epi_wait", "epi_busy",
              "tiles", "dq_loop"]

_PATHS = {"auto": 0, "gemv": 1, "grouped": 2, "generic": 3}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--layer", default="glm52")
    ap.add_argument("--tokens", type=int, default=1)
    ap.add_argument("--iters", type=int, default=5)
    ap.add_argument("--copies", type=int, default=1)
    ap.add_argument("--path", default="auto", choices=sorted(_PATHS))
    ap.add_argument("--trace", default=None, help="save decode phase timestamps here (.npy)")
    ap.add_argument("--warm-ms", type=float, default=0.0,
                    help="run forwards for this long first, so the traced ones see loaded clocks")
    args = ap.parse_args(argv)

    import torch

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import quantized_moe_noaux_b300 as moe
    from synth import LAYERS, make_layer, make_x

    spec = LAYERS[args.layer]
    arrays = make_layer(spec)
    T = args.tokens
    layers = [moe.MoeLayer.from_spec(spec, arrays, max_tokens=T) for _ in range(max(1, args.copies))]
    for L in layers:
        L.set_path(_PATHS[args.path])
    dt = torch.bfloat16 if spec.act_dtype == "bf16" else torch.float32

    def dev(x):
        if spec.act_dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(np.ascontiguousarray(x)).cuda()

    xs = [dev(make_x(spec, T, s)) for s in range(args.iters)]
    out = torch.empty((T, spec.hidden), dtype=dt, device="cuda")
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    buf = torch.zeros((nsm, 64), dtype=torch.int64, device="cuda") if args.trace else None
    if args.warm_ms > 0:
        import time
        t_end = time.time() + args.warm_ms / 1e3
        s = 0
        while time.time() < t_end:
            for _ in range(20):
                layers[s % len(layers)].forward(xs[s % len(xs)], out)
                s += 1
            torch.cuda.synchronize()
    for s in range(args.iters):
        L = layers[s % len(layers)]
        if buf is not None and s == args.iters - 1:
            torch.cuda.synchronize()
            L.set_trace(buf, nsm)
        L.forward(xs[s], out)
    torch.cuda.synchronize()
    for L in layers:
        if L.status() != 0:
            raise SystemExit("device status word set")
    if buf is not None:
        t = buf.cpu().numpy()
        np.save(args.trace, t)
        t0 = t[:, 0][t[:, 0] > 0].min() if (t[:, 0] > 0).any() else 0
        for i, name in enumerate(PHASES):
            v = t[:, i][t[:, i] > 0] - t0
            if v.size:
                print(f"{i:2d} {name:26s} CTAs={v.size:3d}  min {v.min() / 1e3:8.2f}  "
                      f"median {np.median(v) / 1e3:8.2f}  max {v.max() / 1e3:8.2f} us")
        for i, name in ((15, "selection done"), (23, "grouping done")):
            v = t[:, i][t[:, i] > 0] - t0
            if v.size and (t[:, 20] > 0).any():
                print(f"{i:2d} {name:26s} CTAs={v.size:3d}  min {v.min() / 1e3:8.2f}  "
                      f"median {np.median(v) / 1e3:8.2f}  max {v.max() / 1e3:8.2f} us")
        ok = (t[:, 25] > t[:, 24]) & (t[:, 12] > t[:, 0])
        if ok.any():
            mhz = (t[ok, 25] - t[ok, 24]) / (t[ok, 12] - t[ok, 0]) * 1e3
            print(f"decode kernel SM clock (consumer thread 0, cycles / ns): median {np.median(mhz):.0f} MHz, "
                  f"min {mhz.min():.0f}, max {mhz.max():.0f}")
        if (t[:, 0] > 0).any() and (t[:, 20] > 0).any():
            blk = t[:, 16:23].astype(np.float64)
            med = np.median(blk, axis=0)
            names = ["consumer_wait_data", "consumer_compute", "consumer_epilogue", "consumer_transition",
                     "items", "producer_wait_slot", "items_issued"]
            print("decode kernel, median per CTA (cycles): " +
                  ", ".join(f"{n}={v:.0f}" for n, v in zip(names, med)))
            t = t.copy()
            t[:, 16:23] = 0
        for base, label in ((16, "gate/up GEMM"), (32, "down GEMM"), (48, "shared gate/up GEMM")):
            blk = t[:, base:base + 11].astype(np.float64)
            used = blk[:, 0] > 0
            if not used.any():
                continue
            med = np.median(blk[used], axis=0)
            print(f"{label}: CTAs={int(used.sum())} median cycles: " +
                  ", ".join(f"{n}={v:.0f}" for n, v in zip(GEMM_SLOTS, med)))
    print(f"ok: {args.iters} forwards of {spec.name} at T={T} (path {args.path})")


if __name__ == "__main__":
    main()
