"""A small case of the hot path for kernel profiling (ncu) and quick timing.

Runs `--layers` sender layers of a workload through mf_compress and the same
number of receiver layers through mf_retrieve, at the workload's real
per-layer sizes (so one launch moves exactly the bytes of one bench launch),
while keeping the device footprint to a few GB.  Prints per-kernel launch
counts and mean device times from the library's event profiler, and the kept
fraction, retrieval GB/s and compressor tokens/s for each top-p value given.

    python -m cross_model_attention_gb300.profile_case --workload 1 --layers 2
    python -m cross_model_attention_gb300.profile_case --workload 3 --layers 1 \
        --heads 16 --seqlen 16512 --exact --p 0.8      # B = 128 kernels, ~4 GB
    python -m cross_model_attention_gb300.profile_case --workload 1 --layers 2 \
        --kv-heads 4                                   # the non-team retrieval
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", type=int, default=1)
    ap.add_argument("--layers", type=int, default=2)
    ap.add_argument("--repeat", type=int, default=2)
    ap.add_argument("--p", type=str, default=None,
                    help="top-p, or a comma-separated list: one report per value")
    ap.add_argument("--heads", type=int, default=None,
                    help="sender heads (and KV heads), to shrink the device footprint")
    ap.add_argument("--seqlen", type=int, default=None,
                    help="one sequence of this length instead of the workload's")
    ap.add_argument("--exact", action="store_true",
                    help="size each layer's tiles exactly (one sync) instead of at the bound")
    ap.add_argument("--kv-heads", type=int, default=None,
                    help="receiver KV heads (other than 8: the non-team retrieval kernel)")
    args = ap.parse_args()

    from cross_model_attention_gb300 import accounting, synth, workloads
    w = workloads.get(args.workload)
    kw = {}
    if args.heads:
        kw.update(sender_heads=args.heads, sender_kv_heads=args.heads)
    if args.seqlen or kw:
        w = workloads.scaled(w, [args.seqlen] if args.seqlen else w.seqlens, **kw)
    rcv = w.receivers[0]
    if args.kv_heads:
        import dataclasses
        rcv = dataclasses.replace(rcv, kv_heads=args.kv_heads)
    lm = rcv.layer_map(w.sender_layers)[:args.layers]
    ps = [w.p[0]] if args.p is None else [float(x) for x in args.p.split(",")]
    qk = [synth.sender_qk(w, m) for _, m in lm]
    vs = np.stack([synth.receiver_v(w, rcv, j)["v"] for j, _ in lm])
    Ws = np.stack([synth.head_map_weights(w, rcv, j) for j, _ in lm])

    import torch
    import __graft_entry__
    from cross_model_attention_gb300 import mapflow
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    conv = (lambda a: torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)) \
        if w.dtype == "bf16" else (lambda a: torch.from_numpy(a).to(dev))
    q = [conv(x["q"]) for x in qk]
    k = [conv(x["k"]) for x in qk]
    v = conv(vs)
    W = torch.from_numpy(Ws).to(dev)
    o = torch.empty((len(lm), w.T, rcv.heads, w.d), dtype=v.dtype, device=dev)
    for p in ps:
        bsr = mapflow.BSR(len(lm), w.T, w.sender_heads, w.B, w.cu_seqlens)
        bsr.set_exact(args.exact)
        bsr.profile(True)
        for _ in range(args.repeat):
            for l in range(len(lm)):
                bsr.compress(l, q[l], k[l], p)
            bsr.retrieve(W, v, o, list(range(len(lm))))
        bsr.device_status()
        prof = bsr.profile_read()
        out = {name: {"launches": n, "ms_per_launch": (ms / n if n else None)}
               for name, (n, ms) in prof.items()}
        nnz = [bsr.info(l)[0] for l in range(len(lm))]
        ms = {name: v["ms_per_launch"] or 0.0 for name, v in out.items()}
        t_comp = (ms["stats"] + ms["select"] + ms["scan"] + ms["pack"] + ms["union"]) / 1e3
        t_ret = ms["retrieve"] / 1e3
        out.update({
            "p": p, "nnz": nnz,
            "kept_fraction": float(np.mean(nnz)) / (w.sender_heads * accounting.candidate_blocks(w)),
            "retrieval_gbs": (accounting.retrieval_bytes(w, rcv, int(np.mean(nnz))) / t_ret / 1e9
                              if t_ret > 0 else None),
            "compressor_tokens_per_s": w.T / t_comp if t_comp > 0 else None,
            "stats_tflops": (accounting.qk_flops(w) / (ms["stats"] / 1e3) / 1e12
                             if ms["stats"] > 0 else None),
        })
        print(json.dumps(out), flush=True)
        bsr.close()


if __name__ == "__main__":
    main()
