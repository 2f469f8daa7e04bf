"""Phase timelines of the batch-1 tensor-core engine and of the batched
engine (tracing).

Builds the timeline variant of the library (libq4_tl.so: the engines stamp
the GPU's global timer at six points of every phase of every CTA), runs one
token of a fused decoder stack on it and summarises, per phase, when the CTAs
reached it, when their input was staged, when their last unit was handed to
the epilogue and stored, and when the producer issued its last copy; per
layer, how the time splits into unit loops, boundaries and the spread between
CTAs.  With --batch B (2..8) the stack runs on the batched engine, whose six
events are: reached, first weights issued (RMSNorm: previous phase seen),
first stage landed (RMSNorm: rows formed), last unit handed over, phase
published, first input chunk issued.

    python -m weight_streaming_q4_gb300.timeline [--config 8b|70b] [--layers 3] [--batch 8]

Memory plumbing only (torch allocations and the seeded filler); every
arithmetic step runs in the library.
"""
from __future__ import annotations

import argparse

import numpy as np

from . import _lib, build, model, synth

KINDS = ("q|k|v", "o", "gate|up", "down")
EVENTS = ("reached", "barrier", "staged", "last unit", "last store", "last copy")
BT_KINDS = ("q|k|v", "o", "norm", "gate|up", "down", "norm")
BT_EVENTS = ("reached", "weights/seen", "landed/formed", "last unit", "published", "input")


def summarise(tl: np.ndarray, n_phases: int, grid: int) -> dict:
    """tl [CTA][phase][event] ns (0 = no such event) -> per-phase medians and
    maxima (us from the first stamp) and per-layer splits."""
    t = tl[:grid, :n_phases].astype(np.int64)
    t0 = t[t > 0].min()
    rel = np.where(t > 0, (t - t0) / 1e3, np.nan)
    phases = []
    for p in range(n_phases):
        row = {"phase": p, "kind": KINDS[p % 4] if p < n_phases - 1 else "closing"}
        for e, name in enumerate(EVENTS):
            v = rel[:, p, e]
            v = v[~np.isnan(v)]
            row[name] = (round(float(np.median(v)), 2), round(float(v.max()), 2)) if v.size else None
        phases.append(row)
    layers = []
    for first in range(0, n_phases - 1 - 3, 4):
        nxt = first + 4
        if nxt >= n_phases or not phases[nxt]["staged"]:
            break
        span = phases[nxt]["staged"][0] - phases[first]["staged"][0]   # staged input to staged input
        loops = boundaries = spread = 0.0
        for p in range(first, first + 4):
            staged, last = phases[p]["staged"], phases[p]["last unit"]
            following = phases[p + 1]["staged"]
            if not (staged and last and following):
                continue
            loops += last[0] - staged[0]                      # median CTA's unit loop
            spread += last[1] - last[0]                       # slowest CTA's extra
            boundaries += following[0] - phases[p]["last store"][1]   # last store -> next input staged
        layers.append({"layer": first // 4, "us": round(span, 2), "unit_loops_us": round(loops, 2),
                       "spread_us": round(spread, 2), "boundaries_us": round(boundaries, 2),
                       "unit_loop_frac": round(loops / span, 3) if span > 0 else None})
    return {"phases": phases, "layers": layers}


def summarise_batched(tl: np.ndarray, n_layers: int, grid: int) -> dict:
    """The batched engine's timeline (phase 0 the first RMSNorm, then six
    phases per layer) -> per-phase medians and maxima and, per layer (the
    previous layer's last RMSNorm published to this layer's), the median
    CTA's product loops (first stage landed -> last unit) and the rest
    (flag barriers, RMSNorms, tails)."""
    n_phases = 6 * n_layers + 1
    t = tl[:grid, :n_phases].astype(np.int64)
    t0 = t[t > 0].min()
    rel = np.where(t > 0, (t - t0) / 1e3, np.nan)
    phases = []
    for p in range(n_phases):
        row = {"phase": p, "kind": "norm" if p == 0 else BT_KINDS[(p - 1) % 6]}
        for e, name in enumerate(BT_EVENTS):
            v = rel[:, p, e]
            v = v[~np.isnan(v)]
            row[name] = (round(float(np.median(v)), 2), round(float(v.max()), 2)) if v.size else None
        phases.append(row)
    layers = []
    for l in range(1, n_layers):
        first, last = 6 * l + 1, 6 * l + 6
        span = phases[last]["published"][1] - phases[first - 1]["published"][1]
        loops = sum(phases[p]["last unit"][0] - phases[p]["landed/formed"][0]
                    for p in range(first, last + 1) if BT_KINDS[(p - 1) % 6] != "norm")
        layers.append({"layer": l, "us": round(span, 2), "unit_loops_us": round(loops, 2),
                       "rest_us": round(span - loops, 2)})
    return {"phases": phases, "layers": layers}


def run(config: str = "8b", n_layers: int = 3, seed: int = 0, batch: int = 1) -> dict:
    """One token of a fused stack on the timeline build (the previous binding
    of the library is restored afterwards)."""
    prev = _lib._lib
    _lib.use_library(build.build_timeline())
    try:
        return _run(config, n_layers, seed, batch)
    finally:
        _lib._lib = prev


def _run(config: str, n_layers: int, seed: int, batch: int) -> dict:
    import torch
    cfg = dict(synth.LLAMA_8B if config == "8b" else synth.LLAMA_70B)
    cfg.pop("n_layers")
    shape = _lib.LayerShape.of(**cfg)
    wbuf, ptrs = model.resident_layers(shape, n_layers, seed)
    ws, offs, nb = model.workspace(shape, n_layers, batch)
    mode = _lib.Q4_DEC_FUSED | (_lib.Q4_DEC_BATCH_ENGINE if batch > 1 else 0)
    dec = _lib.q4_decoder_create(shape, ptrs, batch, ws, nb, mode)
    h = torch.from_numpy(synth.activations(batch, cfg["hidden"], seed).reshape(-1).view("int16").copy()).cuda()
    for _ in range(5):
        _lib.q4_layer_decode(dec, h)
    torch.cuda.synchronize()
    _lib.q4_timeline_read(clear=True)
    _lib.q4_layer_decode(dec, h)
    torch.cuda.synchronize()
    status = _lib.q4_decoder_status(dec)
    tl = _lib.q4_timeline_read(clear=True)
    _lib.q4_decoder_destroy(dec)
    grid = min(torch.cuda.get_device_properties(0).multi_processor_count, _lib.TIMELINE_CTAS)
    out = summarise(tl, 4 * n_layers + 1, grid) if batch == 1 else summarise_batched(tl, n_layers, grid)
    out.update(config=config, n_layers=n_layers, status=status, batch=batch)
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="8b", choices=["8b", "70b"])
    ap.add_argument("--layers", type=int, default=3)
    ap.add_argument("--batch", type=int, default=1, help="2..8: the batched engine")
    args = ap.parse_args()
    r = run(args.config, args.layers, batch=args.batch)
    events = EVENTS if args.batch == 1 else BT_EVENTS
    print(f"{args.config}-shaped stack, {args.layers} layers, batch {args.batch}, one token; status {r['status']}")
    print("phase kind      " + " | ".join(f"{e:>16s}" for e in events) + "   [us from the first stamp, median/max]")
    for p in r["phases"]:
        cells = [f"{v[0]:7.2f}/{v[1]:7.2f}" if v else f"{'-':>15s}" for v in (p[e] for e in events)]
        print(f"{p['phase']:5d} {p['kind']:8s}  " + " | ".join(cells))
    if args.batch > 1:
        for layer in r["layers"]:
            print(f"layer {layer['layer']}: {layer['us']} us; product loops {layer['unit_loops_us']} us, "
                  f"barriers, RMSNorms and tails {layer['rest_us']} us")
        return
    for layer in r["layers"]:
        print(f"layer {layer['layer']}: {layer['us']} us; unit loops {layer['unit_loops_us']} us "
              f"({layer['unit_loop_frac']}), slowest-CTA spread {layer['spread_us']} us, "
              f"boundaries (last store -> next input staged) {layer['boundaries_us']} us")


if __name__ == "__main__":
    main()
