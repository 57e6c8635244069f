"""Run the route-sort path a fixed number of times on one synthetic workload.

A small driver for external profilers: it builds nothing, allocates the inputs and
outputs of one workload once, issues ``--calls`` back-to-back ``route_sort`` calls on the
current stream and synchronizes.  Example::

    python -m moe_expert_routing_sort_gb300.profile_calls --workload wide_T16384_E4096 --calls 4
    python -m moe_expert_routing_sort_gb300.profile_calls --gate-hidden 7168 --calls 4
"""
from __future__ import annotations

import argparse

import numpy as np


def main(argv=None) -> int:
    from . import datagen

    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--workload", default="decode_T1_E896_G8", choices=list(datagen.WORKLOADS))
    p.add_argument("--calls", type=int, default=8)
    p.add_argument("--tokens", type=int, default=None, help="override the workload's T")
    p.add_argument("--gate-hidden", type=int, default=None,
                   help="run moe_gate_route_sort with this hidden size (gate GEMV ahead)")
    args = p.parse_args(argv)

    import torch

    from . import binding

    kw = {} if args.tokens is None else {"T": args.tokens}
    w = datagen.workload(args.workload, **kw)
    inp = datagen.make_inputs(w)
    logits = torch.from_numpy(inp.logits_bf16.view(np.int16)).view(torch.bfloat16).cuda()
    bias = torch.from_numpy(inp.bias).cuda()
    out = binding.RouteSortBuffers.allocate(w.T, w.E, w.topk, w.block_m, device="cuda")
    if args.gate_hidden is not None:
        g = datagen.make_gate_inputs(w.T, w.E, args.gate_hidden, seed=w.seed)
        hid = torch.from_numpy(g.hidden_bf16.view(np.int16)).view(torch.bfloat16).cuda()
        wg = torch.from_numpy(g.w_gate_bf16.view(np.int16)).view(torch.bfloat16).cuda()
        gb = torch.from_numpy(g.bias).cuda()
        for _ in range(args.calls):
            binding.gate_route_sort(hid, wg, gb, w.n_group, w.topk_group, w.topk,
                                    w.routed_scale, w.block_m, out=out, logits=logits)
        torch.cuda.synchronize()
        print(f"{w.name} with gate H={args.gate_hidden}: {args.calls} calls, "
              f"status={out.status_word()}")
        return 0
    for _ in range(args.calls):
        binding.route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                           w.block_m, out=out)
    torch.cuda.synchronize()
    print(f"{w.name}: {args.calls} calls, T={w.T}, npp={int(out.num_tokens_post_pad.item())}, "
          f"status={out.status_word()}")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
