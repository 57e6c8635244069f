"""The one-launch paths of moe_route_sort and moe_sort.  Calls of 129 to 2048 tokens run on a
cooperative grid with one warp per token (up to 16 tokens per CTA); calls of 5 to 128 tokens
(2 to 320 with the test hook) on a cooperative grid with one CTA per token (up to four per CTA
past the SM count); both exchange the selected ids through the workspace around one grid-wide
barrier.  For mid-sized calls (by default up to 256 tokens
and at most 512 KiB of logits, segment-shaped groups; the grid paths are switched off in those
tests) one cluster of 16 CTAs runs the route step and both sort phases in a single launch,
exchanging per-expert counts through distributed shared memory.  Every case is compared with the CPU oracle bit for
bit (weights within 1e-6) and with the three-kernel multi-CTA path on the same inputs; the
library's test hooks force the paths on (any size) or off.  moe_sort does the same from given
routes on one cluster (by default 128 to 8192 routes).  The cluster paths touch no workspace
byte beyond the status word; the tests use that to check which path ran.
"""
import numpy as np
import pytest
import torch

import oracle
import moe_expert_routing_sort_gb300 as mrs
from _support import WEIGHT_ATOL, check_sort_invariants, ids_for, redraw_callback
from moe_expert_routing_sort_gb300 import datagen

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
POISON = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mrs.build()
    oracle.build()
    mrs.load()
    yield
    mrs.moe_route_sort_debug_set(mrs.DEBUG_CLUSTER_TOKENS, -1)
    mrs.moe_route_sort_debug_set(mrs.DEBUG_GRID_TOKENS, -1)
    mrs.moe_route_sort_debug_set(mrs.DEBUG_WARP_GRID_TOKENS, -1)


def _case(name, T, seed=0, **over):
    w = datagen.workload(name, T=T, seed=seed, **over)
    inp = datagen.make_inputs(w, needs_redraw=redraw_callback(oracle, w))
    ref = oracle.route_sort(inp.logits_bf16, inp.bias, w.n_group, w.topk_group, w.topk,
                            w.routed_scale, w.block_m)
    return w, inp, ref


NEVER = 1 << 30  # the warp-grid hook's limit that keeps it off (it takes T > limit)


def _run(w, inp, cluster_tokens, grid=0, warp=NEVER):
    """One call with the cluster paths limited to T <= cluster_tokens, the per-token grid path
    to T <= grid and the warp-per-token grid path to T > warp (both off unless given); returns
    the buffers and whether any workspace byte past the status word changed."""
    logits = torch.from_numpy(inp.logits_bf16.view(np.int16)).view(torch.bfloat16).to(DEV)
    bias = torch.from_numpy(inp.bias).to(DEV)
    out = mrs.RouteSortBuffers.allocate(w.T, w.E, w.topk, w.block_m, device=DEV)
    out.workspace.fill_(POISON)
    out.sorted_token_ids.fill_(-7)
    out.expert_ids.fill_(-7)
    mrs.moe_route_sort_debug_set(mrs.DEBUG_CLUSTER_TOKENS, cluster_tokens)
    mrs.moe_route_sort_debug_set(mrs.DEBUG_GRID_TOKENS, grid)
    mrs.moe_route_sort_debug_set(mrs.DEBUG_WARP_GRID_TOKENS, warp)
    try:
        mrs.route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                       w.block_m, out=out)
        torch.cuda.synchronize()
    finally:
        mrs.moe_route_sort_debug_set(mrs.DEBUG_CLUSTER_TOKENS, -1)
        mrs.moe_route_sort_debug_set(mrs.DEBUG_GRID_TOKENS, -1)
        mrs.moe_route_sort_debug_set(mrs.DEBUG_WARP_GRID_TOKENS, -1)
    touched = bool(torch.any(out.workspace[16:] != POISON).item())
    return out, touched


def _path(out):
    """Which kind of path the last call on `out` took, from its workspace (poisoned before the
    call): the three-kernel path's route kernel writes every unit's flag word (bytes 16..),
    the grid paths only the exchanged ids further on, the cluster and single-CTA paths
    nothing past the status word."""
    ws = out.workspace
    if bool(torch.any(ws[16:20] != POISON).item()):
        return "three"
    return "grid" if bool(torch.any(ws[16:] != POISON).item()) else "one-launch"


def _assert_matches(out, ref, w):
    npp = int(out.num_tokens_post_pad.item())
    assert npp == ref.num_tokens_post_pad
    ids = out.topk_ids.cpu().numpy()
    wt = out.topk_weights.cpu().numpy()
    assert np.array_equal(ids, ref.topk_ids)
    assert np.max(np.abs(wt - ref.topk_weights), initial=0.0) <= WEIGHT_ATOL
    sid = out.sorted_token_ids[:npp].cpu().numpy()
    sw = out.sorted_weights[:npp].cpu().numpy()
    assert np.array_equal(sid, ref.sorted_token_ids)
    assert np.array_equal(out.expert_ids[: npp // w.block_m].cpu().numpy(), ref.expert_ids)
    real = sid != w.T * w.topk
    assert np.all(sw[~real] == 0.0)
    assert np.array_equal(sw[real], wt.reshape(-1)[sid[real]])
    assert out.status_word() == 0
    check_sort_invariants(ref.topk_ids, w.E, w.block_m, out.sorted_token_ids.cpu().numpy(),
                          out.expert_ids.cpu().numpy(), ref.num_tokens_post_pad)


FORCE = 1 << 20  # the hook's token limit that puts every call of these tests on the cluster


def _both_paths(w, inp, ref, cluster=True):
    a, touched_a = _run(w, inp, FORCE)
    if cluster:
        assert not touched_a, "the cluster path wrote into the workspace (did it run?)"
    else:
        assert touched_a, "a shape without a segment layout took the cluster path"
    _assert_matches(a, ref, w)
    b, touched_b = _run(w, inp, 0)
    assert touched_b, "the three-kernel path left the workspace alone (did it run?)"
    _assert_matches(b, ref, w)
    npp = int(a.num_tokens_post_pad.item())
    assert torch.equal(a.sorted_token_ids[:npp], b.sorted_token_ids[:npp])
    assert torch.equal(a.sorted_weights[:npp], b.sorted_weights[:npp])
    assert torch.equal(a.topk_weights, b.topk_weights)


# T spans one token per CTA-warp, ragged CTA ranges (T not a multiple of 16) and sizes past
# the default reach.
@pytest.mark.parametrize("T", [65, 100, 256, 257, 511, 512, 777, 1024])
def test_prefill_shape(T):
    w, inp, ref = _case("prefill_T512_E896", T)
    _both_paths(w, inp, ref)


@pytest.mark.parametrize("T", [65, 300, 1000])
def test_skewed_distribution(T):
    # a few hot experts: most CTAs hold routes of the same experts, so `before` sums matter
    w, inp, ref = _case("skewed_T8192_E896", T)
    _both_paths(w, inp, ref)


@pytest.mark.parametrize("T", [70, 600])
def test_wide_experts(T):
    w, inp, ref = _case("wide_T16384_E4096", T)
    _both_paths(w, inp, ref)


# cluster: whether the shape has a segment layout (a group splits into equal lane segments
# of a multiple of 4 experts), which the cluster path needs; the other shapes keep the
# three-kernel path whatever the limit.
@pytest.mark.parametrize("E,G,Kg,K,B,T,cluster", [(256, 8, 4, 8, 16, 130, True),
                                                   (64, 8, 4, 6, 16, 200, False),
                                                   (128, 4, 2, 4, 64, 99, True),
                                                   (512, 16, 16, 10, 8, 515, True),
                                                   (120, 8, 4, 8, 16, 333, False),
                                                   (96, 3, 2, 8, 16, 333, True),
                                                   (4096, 16, 16, 32, 1024, 150, True)])
def test_other_shapes(E, G, Kg, K, B, T, cluster):
    w, inp, ref = _case("prefill_T512_E896", T, E=E, n_group=G, topk_group=Kg, topk=K,
                        block_m=B)
    _both_paths(w, inp, ref, cluster)


def test_widened_limit_runs_larger_calls_in_one_cluster():
    w, inp, ref = _case("prefill_T512_E896", 2048)
    out, touched = _run(w, inp, 4096)
    assert not touched
    _assert_matches(out, ref, w)


@pytest.mark.parametrize("name,T,cluster", [("prefill_T512_E896", 65, True),
                                             ("prefill_T512_E896", 256, True),
                                             ("prefill_T512_E896", 257, False),
                                             ("prefill_T512_E896", 512, False),
                                             ("skewed_T8192_E896", 200, True),
                                             ("wide_T16384_E4096", 65, False)])
def test_default_reach(name, T, cluster):
    # by default: T <= 256 and at most 512 KiB of logits
    w, inp, ref = _case(name, T)
    out, touched = _run(w, inp, -1)
    assert touched != cluster
    _assert_matches(out, ref, w)


def test_softmax_scoring_on_the_cluster_path():
    w = datagen.workload("prefill_T512_E896", T=300, n_group=1, topk_group=1, topk=8)
    inp = datagen.make_inputs(w)
    ref = oracle.route_sort_softmax(inp.logits_bf16, w.topk, w.routed_scale, w.block_m)
    logits = torch.from_numpy(inp.logits_bf16.view(np.int16)).view(torch.bfloat16).to(DEV)
    outs = []
    for limit in (FORCE, 0):
        out = mrs.RouteSortBuffers.allocate(w.T, w.E, w.topk, w.block_m, device=DEV)
        out.workspace.fill_(POISON)
        mrs.moe_route_sort_debug_set(mrs.DEBUG_CLUSTER_TOKENS, limit)
        mrs.moe_route_sort_debug_set(mrs.DEBUG_GRID_TOKENS, 0)
        mrs.moe_route_sort_debug_set(mrs.DEBUG_WARP_GRID_TOKENS, NEVER)
        try:
            mrs.route_sort_softmax(logits, w.topk, w.routed_scale, w.block_m, out=out)
            torch.cuda.synchronize()
        finally:
            mrs.moe_route_sort_debug_set(mrs.DEBUG_CLUSTER_TOKENS, -1)
            mrs.moe_route_sort_debug_set(mrs.DEBUG_GRID_TOKENS, -1)
            mrs.moe_route_sort_debug_set(mrs.DEBUG_WARP_GRID_TOKENS, -1)
        assert bool(torch.any(out.workspace[16:] != POISON).item()) == (limit == 0)
        npp = int(out.num_tokens_post_pad.item())
        assert npp == ref["num_tokens_post_pad"]
        assert np.array_equal(out.topk_ids.cpu().numpy(), ref["topk_ids"])
        assert np.max(np.abs(out.topk_weights.cpu().numpy() - ref["topk_weights"]),
                      initial=0.0) <= WEIGHT_ATOL
        assert np.array_equal(out.sorted_token_ids[:npp].cpu().numpy(), ref["sorted_token_ids"])
        assert np.array_equal(out.expert_ids[: npp // w.block_m].cpu().numpy(),
                              ref["expert_ids"])
        assert out.status_word() == 0
        outs.append(out)
    assert torch.equal(outs[0].topk_weights, outs[1].topk_weights)


# ------------------------------------------------------------------ moe_sort
def _sort(ids, wts, E, B, limit):
    T, K = ids.shape
    out = mrs.RouteSortBuffers.allocate(T, E, K, B, device=DEV)
    out.workspace.fill_(POISON)
    out.sorted_token_ids.fill_(-7)
    mrs.moe_route_sort_debug_set(mrs.DEBUG_CLUSTER_TOKENS, limit)
    try:
        mrs.moe_sort(torch.from_numpy(ids).to(DEV), torch.from_numpy(wts).to(DEV), E, B,
                     out.sorted_token_ids, out.sorted_weights, out.expert_ids,
                     out.num_tokens_post_pad, out.workspace)
        torch.cuda.synchronize()
    finally:
        mrs.moe_route_sort_debug_set(mrs.DEBUG_CLUSTER_TOKENS, -1)
    touched = bool(torch.any(out.workspace[16:] != POISON).item())
    return out, touched


@pytest.mark.parametrize("dist", ["uniform", "shared", "one_expert", "every_third_dropped",
                                  "all_dropped", "dup_in_token"])
@pytest.mark.parametrize("T,K,E,B", [(129, 16, 896, 32), (500, 16, 896, 64), (1000, 8, 4096, 128),
                                     (3001, 8, 256, 64)])
def test_moe_sort_on_one_cluster(dist, T, K, E, B):
    rng = np.random.default_rng(T + K + E + B)
    ids = ids_for(dist, T, K, E, rng)
    wts = rng.uniform(0.01, 1.0, (T, K)).astype(np.float32)
    ref = oracle.sort(ids, wts, E, B)
    outs = []
    for limit, cluster in ((FORCE, True), (0, False)):
        out, touched = _sort(ids, wts, E, B, limit)
        assert touched != cluster
        npp = int(out.num_tokens_post_pad.item())
        assert npp == ref.num_tokens_post_pad
        assert np.array_equal(out.sorted_token_ids[:npp].cpu().numpy(), ref.sorted_token_ids)
        assert np.array_equal(out.sorted_weights[:npp].cpu().numpy(), ref.sorted_weights)
        assert np.array_equal(out.expert_ids[: npp // B].cpu().numpy(), ref.expert_ids)
        assert out.status_word() == ref.flags == 0
        outs.append(out)
    npp = ref.num_tokens_post_pad
    assert torch.equal(outs[0].sorted_token_ids[:npp], outs[1].sorted_token_ids[:npp])


def test_moe_sort_cluster_flags_out_of_range_ids():
    rng = np.random.default_rng(5)
    T, E, K, B = 700, 64, 4, 16
    ids = rng.integers(0, E, (T, K)).astype(np.int32)
    ids[T // 3, 2] = E
    ids[T - 1, 0] = E + 100
    wts = np.ones((T, K), np.float32)
    ref = oracle.sort(ids, wts, E, B)
    out, touched = _sort(ids, wts, E, B, FORCE)
    assert not touched
    npp = int(out.num_tokens_post_pad.item())
    assert npp == ref.num_tokens_post_pad
    assert np.array_equal(out.sorted_token_ids[:npp].cpu().numpy(), ref.sorted_token_ids)
    assert out.status_word() == mrs.DEVICE_BAD_EXPERT_ID


@pytest.mark.parametrize("T,K,cluster", [(129, 16, True), (512, 16, True), (513, 16, False),
                                         (2000, 4, True), (1025, 8, False)])
def test_moe_sort_default_reach(T, K, cluster):
    # by default up to 8192 routes (T * K); the smallest calls (up to 128 routes) take the
    # single-CTA kernel, which leaves the workspace alone too
    E, B = 896, 32
    rng = np.random.default_rng(T)
    ids = ids_for("uniform", T, K, E, rng)
    wts = rng.uniform(0.01, 1.0, (T, K)).astype(np.float32)
    ref = oracle.sort(ids, wts, E, B)
    out, touched = _sort(ids, wts, E, B, -1)
    assert touched != cluster
    npp = int(out.num_tokens_post_pad.item())
    assert np.array_equal(out.sorted_token_ids[:npp].cpu().numpy(), ref.sorted_token_ids)


# ----------------------------------------- a few tokens: one CTA each, a cooperative grid
@pytest.mark.parametrize("T", [2, 3, 5, 8, 9, 15, 16, 33, 64, 127, 128, 153, 304, 320])
@pytest.mark.parametrize("E,G,Kg,K,B", [(896, 8, 4, 16, 32), (896, 1, 1, 16, 32),
                                         (4096, 16, 4, 8, 128), (64, 8, 4, 6, 16),
                                         (129, 3, 2, 5, 16), (4000, 5, 2, 8, 32)])
def test_few_tokens_on_one_cluster(T, E, G, Kg, K, B):
    w, inp, ref = _case("decode_T1_E896_G8", T, E=E, n_group=G, topk_group=Kg, topk=K,
                        block_m=B, seed=E + T)
    a, _ = _run(w, inp, -1, grid=FORCE)  # one CTA per token on a cooperative grid
    _assert_matches(a, ref, w)
    b, _ = _run(w, inp, 0)            # single-CTA kernel (T <= 8) or the three-kernel path
    _assert_matches(b, ref, w)
    npp = int(a.num_tokens_post_pad.item())
    assert torch.equal(a.sorted_token_ids[:npp], b.sorted_token_ids[:npp])


@pytest.mark.parametrize("T", [2, 7, 16])
def test_few_tokens_exact_ties(T):
    # every logit equal: many survivors per token (the kernel's fallback ranking)
    w = datagen.workload("decode_T1_E896_G8", T=T)
    logits = np.full((T, 896), datagen.float32_to_bf16_bits(np.float32([0.75]))[0], np.uint16)
    bias = np.zeros(896, np.float32)
    bias[::7] = 0.03125
    inp = datagen.RouterInputs(w, logits, bias)
    ref = oracle.route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                            w.block_m)
    out, _ = _run(w, inp, -1, grid=FORCE)
    _assert_matches(out, ref, w)


@pytest.mark.parametrize("T", [2, 9, 100])
def test_few_tokens_softmax(T):
    w = datagen.workload("prefill_T512_E896", T=T, n_group=1, topk_group=1, topk=8)
    inp = datagen.make_inputs(w)
    ref = oracle.route_sort_softmax(inp.logits_bf16, w.topk, w.routed_scale, w.block_m)
    logits = torch.from_numpy(inp.logits_bf16.view(np.int16)).view(torch.bfloat16).to(DEV)
    out = mrs.RouteSortBuffers.allocate(w.T, w.E, w.topk, w.block_m, device=DEV)
    mrs.route_sort_softmax(logits, w.topk, w.routed_scale, w.block_m, out=out)
    torch.cuda.synchronize()
    npp = int(out.num_tokens_post_pad.item())
    assert npp == ref["num_tokens_post_pad"]
    assert np.array_equal(out.topk_ids.cpu().numpy(), ref["topk_ids"])
    assert np.max(np.abs(out.topk_weights.cpu().numpy() - ref["topk_weights"]),
                  initial=0.0) <= WEIGHT_ATOL
    assert np.array_equal(out.sorted_token_ids[:npp].cpu().numpy(), ref["sorted_token_ids"])
    assert np.array_equal(out.expert_ids[: npp // w.block_m].cpu().numpy(), ref["expert_ids"])
    assert out.status_word() == 0


# ------------------------------- a few hundred tokens: one warp per token, a cooperative grid
# T spans one token per CTA (the hook forces the path below the SM count), ragged CTA ranges
# and the default reach's ends; shapes include ones without a segment layout (the generic warp
# routine) and a single group.
@pytest.mark.parametrize("T", [2, 3, 17, 152, 153, 200, 305, 512, 777, 1024, 2048])
@pytest.mark.parametrize("E,G,Kg,K,B", [(896, 8, 4, 16, 32), (896, 1, 1, 16, 32),
                                         (4096, 16, 4, 8, 128), (64, 8, 4, 6, 16),
                                         (129, 3, 2, 5, 16), (4000, 5, 2, 8, 32)])
def test_warp_grid(T, E, G, Kg, K, B):
    if E >= 4000 and T > 600:
        pytest.skip("the keys of ceil(T / #SMs) tokens of 4096 experts exceed shared memory")
    w, inp, ref = _case("prefill_T512_E896", T, E=E, n_group=G, topk_group=Kg, topk=K,
                        block_m=B, seed=7 * E + T)
    a, _ = _run(w, inp, -1, warp=1)
    assert _path(a) == "grid"
    _assert_matches(a, ref, w)
    b, _ = _run(w, inp, 0)  # single-CTA kernel (T <= 8) or the three-kernel path
    _assert_matches(b, ref, w)
    npp = int(a.num_tokens_post_pad.item())
    assert torch.equal(a.sorted_token_ids[:npp], b.sorted_token_ids[:npp])
    assert torch.equal(a.sorted_weights[:npp], b.sorted_weights[:npp])
    assert torch.equal(a.topk_weights, b.topk_weights)


@pytest.mark.parametrize("T", [300, 1000])
def test_warp_grid_skewed(T):
    # a few hot experts: most CTAs hold routes of the same experts (earlier-CTA counts matter)
    w, inp, ref = _case("skewed_T8192_E896", T)
    a, _ = _run(w, inp, -1, warp=1)
    assert _path(a) == "grid"
    _assert_matches(a, ref, w)


@pytest.mark.parametrize("T", [200, 600])
def test_warp_grid_exact_ties(T):
    # every logit equal: many survivors per token, every CTA routes to the same experts
    w = datagen.workload("prefill_T512_E896", T=T)
    logits = np.full((T, 896), datagen.float32_to_bf16_bits(np.float32([0.75]))[0], np.uint16)
    bias = np.zeros(896, np.float32)
    bias[::7] = 0.03125
    inp = datagen.RouterInputs(w, logits, bias)
    ref = oracle.route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                            w.block_m)
    out, _ = _run(w, inp, -1, warp=1)
    assert _path(out) == "grid"
    _assert_matches(out, ref, w)


@pytest.mark.parametrize("T", [5, 300, 1000])
def test_warp_grid_softmax(T):
    w = datagen.workload("prefill_T512_E896", T=T, n_group=1, topk_group=1, topk=8)
    inp = datagen.make_inputs(w)
    ref = oracle.route_sort_softmax(inp.logits_bf16, w.topk, w.routed_scale, w.block_m)
    logits = torch.from_numpy(inp.logits_bf16.view(np.int16)).view(torch.bfloat16).to(DEV)
    out = mrs.RouteSortBuffers.allocate(w.T, w.E, w.topk, w.block_m, device=DEV)
    out.workspace.fill_(POISON)
    mrs.moe_route_sort_debug_set(mrs.DEBUG_WARP_GRID_TOKENS, 1)
    try:
        mrs.route_sort_softmax(logits, w.topk, w.routed_scale, w.block_m, out=out)
        torch.cuda.synchronize()
    finally:
        mrs.moe_route_sort_debug_set(mrs.DEBUG_WARP_GRID_TOKENS, -1)
    assert _path(out) == "grid"
    npp = int(out.num_tokens_post_pad.item())
    assert npp == ref["num_tokens_post_pad"]
    assert np.array_equal(out.topk_ids.cpu().numpy(), ref["topk_ids"])
    assert np.max(np.abs(out.topk_weights.cpu().numpy() - ref["topk_weights"]),
                  initial=0.0) <= WEIGHT_ATOL
    assert np.array_equal(out.sorted_token_ids[:npp].cpu().numpy(), ref["sorted_token_ids"])
    assert np.array_equal(out.expert_ids[: npp // w.block_m].cpu().numpy(), ref["expert_ids"])
    assert out.status_word() == 0


@pytest.mark.parametrize("name,T,path", [("prefill_T512_E896", 4, "one-launch"),
                                          ("prefill_T512_E896", 5, "grid"),
                                          ("prefill_T512_E896", 64, "grid"),
                                          ("prefill_T512_E896", 129, "grid"),
                                          ("prefill_T512_E896", 512, "grid"),
                                          ("prefill_T512_E896", 2048, "grid"),
                                          ("prefill_T512_E896", 2049, "three"),
                                          ("wide_T16384_E4096", 600, "grid"),
                                          ("skewed_T8192_E896", 8192, "three")])
def test_default_dispatch(name, T, path):
    w, inp, ref = _case(name, T)
    out, _ = _run(w, inp, -1, grid=-1, warp=-1)
    assert _path(out) == path
    _assert_matches(out, ref, w)


@pytest.mark.parametrize("T", [3, 300])
def test_bias_not_16_byte_aligned(T):
    # the exact-key step reads 16-byte bias vectors only from a 16-byte aligned bias; a bias one
    # float into a buffer takes the 4-byte loads
    w, inp, ref = _case("prefill_T512_E896", T)
    logits = torch.from_numpy(inp.logits_bf16.view(np.int16)).view(torch.bfloat16).to(DEV)
    store = torch.zeros(w.E + 1, dtype=torch.float32, device=DEV)
    store[1:] = torch.from_numpy(inp.bias).to(DEV)
    bias = store[1:]
    assert bias.data_ptr() % 16 != 0
    out = mrs.RouteSortBuffers.allocate(w.T, w.E, w.topk, w.block_m, device=DEV)
    mrs.route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale, w.block_m,
                   out=out)
    torch.cuda.synchronize()
    _assert_matches(out, ref, w)
