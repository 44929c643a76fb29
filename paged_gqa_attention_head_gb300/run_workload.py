"""Run one named workload through the library a few times (for profilers).

  python -m paged_gqa_attention_head_gb300.run_workload <workload> [--iters N] [--op auto|append]
                                                         [--first N]

Workloads are the seeded shapes in `inputs.WORKLOADS` (a prefill marked causal=False runs
through the non-causal entry point).  `--first N` (decode workloads) keeps
the first N sequences of the batch, with the same lengths, in a pool of their own pages (a
cut-down case whose device footprint suits a profiler capture).  Prints the mean time of
the timed iterations (CUDA events) and the KV bytes one call reads; every launch goes
through the C ABI.
"""
from __future__ import annotations

import argparse

import torch

from . import inputs, sinkattn as sa


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("workload", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--op", choices=["auto", "append"], default="auto")
    ap.add_argument("--first", type=int, default=0)
    args = ap.parse_args()
    dev = torch.device("cuda:0")
    w = inputs.make_workload(args.workload, seed=0)
    if args.first and isinstance(w, inputs.DecodeInputs):
        spec = inputs.WORKLOADS[args.workload]
        lens = [int(x) for x in w.cache.lens[:args.first]]
        w = inputs.make_decode(lens, len(lens), w.num_qo_heads, w.num_kv_heads, w.head_dim, seed=0,
                               sinks=w.sinks is not None, kv_dtype=spec.get("kv_dtype", "bf16"))
    if args.op == "append":
        lens = w.new_lens
        a = inputs.make_append(lens, [0] * len(lens), w.num_kv_heads, w.head_dim, seed=0)
        c = a.cache
        t = (a.k.to(dev), a.v.to(dev), a.cu_seqlens.to(dev), c.block_table.to(dev),
             a.start_pos.to(dev), c.k_pages.to(dev), c.v_pages.to(dev))
        fn = lambda: sa.append_kv(*t)  # noqa: E731
    elif isinstance(w, inputs.DecodeInputs):
        c = w.cache
        t = (w.q.to(dev), c.k_pages.to(dev), c.v_pages.to(dev), c.block_table.to(dev),
             c.lens.to(dev), None if w.sinks is None else w.sinks.to(dev), w.scale)
        fn = lambda: sa.decode(*t)  # noqa: E731
    else:
        kw = {}
        if w.prefix is not None:
            kw = dict(k_pages=w.prefix.k_pages.to(dev), v_pages=w.prefix.v_pages.to(dev),
                      prefix_block_table=w.prefix.block_table.to(dev),
                      prefix_lens=w.prefix.lens.to(dev))
        t = (w.q.to(dev), w.k.to(dev), w.v.to(dev), w.cu_seqlens.to(dev),
             None if w.sinks is None else w.sinks.to(dev), w.scale)
        if inputs.WORKLOADS[args.workload].get("causal", True):
            fn = lambda: sa.prefill(*t, **kw)  # noqa: E731
        else:
            fn = lambda: sa.prefill_noncausal(*t)  # noqa: E731
    fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.iters):
        fn()
    e1.record()
    torch.cuda.synchronize()
    extra = f", {w.kv_bytes()} KV bytes per call" if isinstance(w, inputs.DecodeInputs) else ""
    print(f"{args.workload}: {e0.elapsed_time(e1) / args.iters:.4f} ms per call{extra}")


if __name__ == "__main__":
    main()
