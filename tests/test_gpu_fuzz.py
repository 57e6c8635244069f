"""Seeded random shapes through moe_route_sort, against the CPU oracle element by element.

Each case draws a group layout (G groups of g experts, E = G * g <= 4096), Kg kept groups, K
routes per token (at most the experts of the kept groups), block_m, a token count T spread
log-uniformly from 1 to 3000 (so that every dispatch, from the one-token kernel through the
grid paths to the three-kernel path, is reached), the logit spread, the bias range and the
routed scale, with the library's default dispatch.  Tokens whose selection hinges on a gap
below 1e-6 are redrawn, as in every parity test (the bias range is never zero: with equal
biases, experts with equal bf16 logits tie exactly and no redraw separates them).
"""
import numpy as np
import pytest
import torch

import oracle
import moe_expert_routing_sort_gb300 as mrs
from _support import WEIGHT_ATOL, check_sort_invariants, redraw_callback
from moe_expert_routing_sort_gb300 import datagen

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
N_CASES = 48
MAX_LOGITS = 3_000_000  # T * E per case (the oracle's time)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mrs.build()
    oracle.build()
    mrs.load()


def _draw_case(seed):
    rng = np.random.default_rng(1000 + seed)
    G = int(rng.choice([1, 2, 3, 4, 5, 6, 8, 12, 16, 32, 64]))
    g_max = 4096 // G
    # mostly multiples of 4 (segment-shaped layouts), sometimes any size
    g = int(rng.integers(1, g_max + 1))
    if rng.random() < 0.7 and g >= 4:
        g -= g % 4
    E = G * g
    Kg = int(rng.integers(1, G + 1))
    K = int(rng.integers(1, min(32, Kg * g) + 1))
    B = int(2 ** rng.integers(0, 11))
    t_max = max(1, min(3000, MAX_LOGITS // E))
    T = int(np.exp(rng.uniform(0.0, np.log(t_max + 1))))
    T = max(1, min(T, t_max))
    return dict(T=T, E=E, n_group=G, topk_group=Kg, topk=K, block_m=B,
                routed_scale=float(rng.choice([1.0, 2.5, rng.uniform(0.5, 2.5)])),
                logit_std=float(rng.choice([0.5, 1.0, 1.5, 3.0])),
                bias_half_range=float(rng.choice([0.01, 0.05, 0.1, 0.5])),
                skewed=bool(rng.random() < 0.25), seed=seed)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_shape(seed):
    c = _draw_case(seed)
    w = datagen.workload("prefill_T512_E896", **c)
    inp = datagen.make_inputs(w, needs_redraw=redraw_callback(oracle, w))
    ref = oracle.route_sort(inp.logits_bf16, inp.bias, w.n_group, w.topk_group, w.topk,
                            w.routed_scale, w.block_m)
    logits = torch.from_numpy(inp.logits_bf16.view(np.int16)).view(torch.bfloat16).to(DEV)
    bias = torch.from_numpy(inp.bias).to(DEV)
    out = mrs.RouteSortBuffers.allocate(w.T, w.E, w.topk, w.block_m, device=DEV)
    out.sorted_token_ids.fill_(-7)
    out.expert_ids.fill_(-7)
    mrs.route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale, w.block_m,
                   out=out)
    torch.cuda.synchronize()
    npp = int(out.num_tokens_post_pad.item())
    assert out.status_word() == 0, c
    assert npp == ref.num_tokens_post_pad, c
    assert np.array_equal(out.topk_ids.cpu().numpy(), ref.topk_ids), c
    assert np.max(np.abs(out.topk_weights.cpu().numpy() - ref.topk_weights),
                  initial=0.0) <= WEIGHT_ATOL, c
    sid = out.sorted_token_ids.cpu().numpy()
    assert np.array_equal(sid[:npp], ref.sorted_token_ids), c
    assert np.array_equal(out.expert_ids[: npp // w.block_m].cpu().numpy(), ref.expert_ids), c
    sw = out.sorted_weights[:npp].cpu().numpy()
    real = sid[:npp] != w.T * w.topk
    assert np.array_equal(sw[real], out.topk_weights.cpu().numpy().reshape(-1)[sid[:npp][real]])
    assert np.all(sw[~real] == 0.0), c
    check_sort_invariants(ref.topk_ids, w.E, w.block_m, sid, out.expert_ids.cpu().numpy(),
                          ref.num_tokens_post_pad)
