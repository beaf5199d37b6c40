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

PHASES = ["start", "-", "router rows written", "all router rows seen",
          "epilogue: shared gate/up done", "epilogue: routed gate/up done", "epilogue: shared down done",
          "selection done", "-", "-", "-", "-",
          "epilogue: all units done", "producer: all issued", "mma: all issued", "routing done"]
DECODE_SLOTS = ["dec wait data (cycles)", "dec wait A slot", "dec busy", "dec items (wg0)",
                "mma wait A", "mma wait accumulator", "mma h staging", "units",
                "epi wait accumulator", "epi busy", "epi last-arriver work", "prod wait slot",
                "prod items issued"]

GEMM_SLOTS = ["kernel", "mma_wait_operands", "mma_wait_accumulator", "dq_wait_weights",
              "dq_wait_stage", "act_producer_wait", "w_producer_wait", "epi_wait", "epi_busy",
              "tiles", "dq_loop"]

_PATHS = {"auto": 0, "gemv": 1, "grouped": 2, "generic": 3}


def parser() -> argparse.ArgumentParser:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--layer", default="glm52")
    ap.add_argument("--tokens", type=int, default=1)
    ap.add_argument("--iters", type=int, default=5)
    ap.add_argument("--copies", type=int, default=1)
    ap.add_argument("--path", default="auto", choices=sorted(_PATHS))
    ap.add_argument("--trace", default=None, help="save decode phase timestamps here (.npy)")
    ap.add_argument("--warm-ms", type=float, default=0.0,
                    help="run forwards for this long first, so the traced ones see loaded clocks")
    return ap


def main(argv=None):
    args = parser().parse_args(argv)

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
        decode = (t[:, 29] > 0).any()
        if decode:
            for i, name in enumerate(PHASES):
                v = t[:, i][t[:, i] > 0] - t0
                if v.size:
                    print(f"{i:2d} {name:28s} CTAs={v.size:3d}  min {v.min() / 1e3:8.2f}  "
                          f"median {np.median(v) / 1e3:8.2f}  max {v.max() / 1e3:8.2f} us")
            print("CTA 0 stamps (us): " + ", ".join(f"{i}:{(t[0, i] - t0) / 1e3:.2f}" for i in (0, 2, 3, 6, 7, 15)
                                                      if t[0, i] > 0))
            ok = (t[:, 30] > t[:, 29]) & (t[:, 12] > t[:, 0])
            if ok.any():
                mhz = (t[ok, 30] - t[ok, 29]) / (t[ok, 12] - t[ok, 0]) * 1e3
                print(f"decode kernel SM clock (epilogue thread 0, cycles / ns): median {np.median(mhz):.0f} MHz")
            blk = t[:, 16:29].astype(np.float64)
            med = np.median(blk, axis=0)
            mx = blk.max(axis=0)
            for n, v, m in zip(DECODE_SLOTS, med, mx):
                print(f"   {n:28s} median {v:12.0f}  max {m:12.0f}")
            for i, n in ((32, "stager wait"), (33, "mma issue blocks"), (34, "mma loop total"),
                         (35, "dec wait routing"), (36, "dec wait h ready"), (37, "dec loop total"),
                         (38, "dec phase 0 start"), (39, "dec phase 1 start"), (40, "dec phase 2 start"),
                         (41, "dec phase 3 start")):
                print(f"   {n:28s} median {np.median(t[:, i]):12.0f}  max {t[:, i].max():12.0f}")
            t = t.copy()
            t[:, 16:48] = 0
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
