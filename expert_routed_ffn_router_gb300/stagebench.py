"""Per-stage timing of the layer's entry points on synthetic inputs (CUDA events).

    python -m expert_routed_ffn_router_gb300.stagebench --stage router --workload prefill

Stages: router (moe_router_topk), dispatch (moe_dispatch on the router's output), combine
(moe_combine on seeded expert outputs Yp and the router's routing), layer
(moe_layer_forward; with --fp8 the FP8 layer on E4M3 experts).  The router, dispatch and
combine stages allocate only their own inputs, so they run at full token counts without the
22.5 GB of expert weights -- small enough for profiler captures.  Prints one JSON line with
the mean milliseconds per call and the call's status word (for the layer also the number of
activated experts).
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import torch

from . import binding as B
from . import synth


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--stage", choices=("router", "dispatch", "combine", "layer"),
                    default="router")
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--T", type=int, default=0, help="override the token count")
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--fp8", action="store_true", help="layer stage: E4M3 expert weights")
    args = ap.parse_args(argv)

    dev = torch.device("cuda", 0)
    w = synth.workload(args.workload, **({"T": args.T} if args.T else {}))
    r = synth.routing_inputs(w)
    to = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    X, Wg, bias = to(r["X"]), to(r["W_gate"]), torch.from_numpy(r["bias"]).to(dev)
    T, H, E, K = w.T, w.H, w.E, w.K
    ws = torch.zeros(B.moe_workspace_bytes(T, H, E, K, w.I, w.Is), dtype=torch.uint8, device=dev)
    idx = torch.empty(T, K, dtype=torch.int32, device=dev)
    wt = torch.empty(T, K, dtype=torch.float32, device=dev)

    if args.stage == "router":
        def run():
            B.moe_router_topk(X, Wg, bias, K, idx, wt, ws)
    elif args.stage == "dispatch":
        B.moe_router_topk(X, Wg, bias, K, idx, wt, ws)
        counts = torch.empty(E, dtype=torch.int32, device=dev)
        offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(T * K, dtype=torch.int32, device=dev)
        slot = torch.empty(T, K, dtype=torch.int32, device=dev)
        Xp = torch.empty(T * K, H, dtype=torch.bfloat16, device=dev)
        aff = torch.empty(E, E, dtype=torch.int32, device=dev)

        def run():
            B.moe_dispatch(X, idx, E, counts, offsets, perm, slot, Xp, aff, ws)
    elif args.stage == "combine":
        B.moe_router_topk(X, Wg, bias, K, idx, wt, ws)
        counts = torch.empty(E, dtype=torch.int32, device=dev)
        offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(T * K, dtype=torch.int32, device=dev)
        slot = torch.empty(T, K, dtype=torch.int32, device=dev)
        Xp = torch.empty(T * K, H, dtype=torch.bfloat16, device=dev)
        B.moe_dispatch(X, idx, E, counts, offsets, perm, slot, Xp, None, ws)
        g = torch.Generator(device=dev)
        g.manual_seed(12345)
        Yp = torch.randn(T * K, H, generator=g, device=dev).to(torch.bfloat16)
        Ysh = torch.randn(T, H, generator=g, device=dev)
        Y = torch.empty(T, H, dtype=torch.float32, device=dev)

        def run():
            B.moe_combine(Yp, slot, wt, Ysh, Y)
    else:
        weights = synth.expert_weights_device(w, dev)
        weights["W_gate"], weights["bias"] = Wg, bias
        layer = B.MoELayer(weights, T, K, fp8=args.fp8)

        def run():
            layer.forward(X)

    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.iters):
        run()
    e1.record()
    torch.cuda.synchronize()
    out = {"stage": args.stage, "workload": w.name, "T": T,
           "ms": round(e0.elapsed_time(e1) / args.iters, 4)}
    if args.stage == "layer":
        # the layer's own workspace and by-products: status word, activated experts
        out.update(fp8=args.fp8, status=layer.status(),
                   n_active=int((layer.counts > 0).sum().item()))
    else:
        out["status"] = B.moe_read_status(ws)
    print(json.dumps(out))


if __name__ == "__main__":
    main()
