"""moe_route_sort_noalloc: the allocation-free entry point, for callers that cannot provide
or allocate scratch memory (a runtime plugin handed only its input and output pointers, a
serving path that must not call cudaMalloc, a fully pre-reserved memory budget).

Its results must equal those of moe_route_sort with a caller workspace, on two calls in a
row (different inputs, and different shapes, so whatever the first call left in the shared
static scratch cannot leak into the second).  The file runs last (its name sorts last) and
needs nothing from the other test files, so it passes alone in a fresh process too.
"""
import numpy as np
import pytest
import torch

import moe_expert_routing_sort_gb300 as mrs
from moe_expert_routing_sort_gb300 import datagen

pytestmark = pytest.mark.gpu

WEIGHT_ATOL = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mrs.build()
    mrs.load()


def _inputs(name, seed, T=None):
    kw = {"seed": seed}
    if T is not None:
        kw["T"] = T
    w = datagen.workload(name, **kw)
    inp = datagen.make_inputs(w)
    logits = torch.from_numpy(inp.logits_bf16.view(np.int16)).view(torch.bfloat16).cuda()
    bias = torch.from_numpy(inp.bias).cuda()
    return w, logits, bias


def _with_workspace(w, logits, bias):
    out = mrs.route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                         w.block_m)
    torch.cuda.synchronize()
    return out


def _no_alloc(w, logits, bias):
    out = mrs.RouteSortBuffers.allocate(w.T, w.E, w.topk, w.block_m, device="cuda")
    for t in (out.topk_ids, out.sorted_token_ids, out.expert_ids, out.num_tokens_post_pad):
        t.fill_(-9)
    mrs.moe_route_sort_noalloc(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                               w.block_m, out.topk_ids, out.topk_weights,
                               out.sorted_token_ids, out.sorted_weights, out.expert_ids,
                               out.num_tokens_post_pad)
    torch.cuda.synchronize()
    return out


def _same(a, b, w):
    npp = int(a.num_tokens_post_pad.item())
    assert npp == int(b.num_tokens_post_pad.item())
    assert torch.equal(a.topk_ids, b.topk_ids)
    assert torch.max(torch.abs(a.topk_weights - b.topk_weights)).item() <= WEIGHT_ATOL
    assert torch.equal(a.sorted_token_ids[:npp], b.sorted_token_ids[:npp])
    assert torch.max(torch.abs(a.sorted_weights[:npp] - b.sorted_weights[:npp]),
                     ).item() <= WEIGHT_ATOL
    assert torch.equal(a.expert_ids[: npp // w.block_m], b.expert_ids[: npp // w.block_m])


@pytest.mark.parametrize("first,second", [
    (("skewed_T8192_E896", None), ("prefill_T512_E896", None)),
    (("decode_T1_E896_G8", None), ("wide_T16384_E4096", None)),
    (("prefill_T512_E896", 40), ("skewed_T8192_E896", 3000)),
])
def test_no_alloc_matches_workspace_entry_point_twice(first, second):
    for k, (name, T) in enumerate((first, second)):
        w, logits, bias = _inputs(name, seed=10 + k, T=T)
        _same(_no_alloc(w, logits, bias), _with_workspace(w, logits, bias), w)


def test_no_alloc_rejects_shapes_beyond_its_scratch():
    # the size check runs before anything touches the (fake) pointers
    lib = mrs.load()
    base = 0x7F0000000000
    T, E, K, B = 600000, 4096, 8, 128
    assert mrs.moe_route_sort_workspace_bytes(T, E, K, B) > 32 * 1024 * 1024
    rc = lib.moe_route_sort_noalloc(base, base + 0x100000, T, E, 16, 4, K, 1.0, B,
                                    base + 0x200000, base + 0x300000, base + 0x400000,
                                    base + 0x500000, base + 0x600000, base + 0x700000, None)
    assert rc == -13
    assert "static" in mrs.strerror(rc)
