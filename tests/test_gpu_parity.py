"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on a GB300.

Bit-exact: topk_ids, sorted_token_ids[0:npp), expert_ids[0:npp/B), num_tokens_post_pad.
Weights: within 1e-6 absolute (IEEE expf on both sides, no fast-math), sentinel rows exactly
0, and sorted_weights exact copies of the GPU's own topk_weights.  Inputs are redrawn where
the oracle's selection margin is below 1e-6, so ulp-level differences between two correct
sigmoid evaluations cannot change an id.  The full-size workloads are compared on every
token, in the launch configuration the benchmark times.
"""
import ctypes
import functools
import hashlib

import numpy as np
import pytest
import torch

import oracle
import moe_expert_routing_sort_gb300 as mrs
from _support import WEIGHT_ATOL, check_sort_invariants, ids_for, redraw_callback
from moe_expert_routing_sort_gb300 import datagen

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mrs.build()
    oracle.build()
    mrs.load()


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


@functools.lru_cache(maxsize=None)
def inputs_for(name: str, T=None, seed=0):
    kw = {}
    if T is not None:
        kw["T"] = T
    if seed:
        kw["seed"] = seed
    w = datagen.workload(name, **kw)
    inp = datagen.make_inputs(w, needs_redraw=redraw_callback(oracle, w))
    ref = oracle.route_sort(inp.logits_bf16, inp.bias, w.n_group, w.topk_group, w.topk,
                            w.routed_scale, w.block_m)
    return w, inp, ref


def run_gpu(w, inp, poison=False):
    logits = to_dev_bf16(inp.logits_bf16)
    bias = torch.from_numpy(inp.bias).to(DEV)
    out = mrs.RouteSortBuffers.allocate(w.T, w.E, w.topk, w.block_m, device=DEV)
    if poison:
        for t in (out.topk_ids, out.sorted_token_ids, out.expert_ids, out.num_tokens_post_pad):
            t.fill_(-7)
        for t in (out.topk_weights, out.sorted_weights):
            t.fill_(float("nan"))
        out.workspace.fill_(0xA5)
    mrs.route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale, w.block_m,
                   out=out)
    torch.cuda.synchronize()
    return out


def assert_matches(out, ref, w):
    npp = int(out.num_tokens_post_pad.item())
    assert npp == ref.num_tokens_post_pad
    ids = out.topk_ids.cpu().numpy()
    wt = out.topk_weights.cpu().numpy()
    bad = np.nonzero(np.any(ids != ref.topk_ids, axis=1))[0]
    assert bad.size == 0, f"topk_ids differ on tokens {bad[:10]}"
    assert np.max(np.abs(wt - ref.topk_weights), initial=0.0) <= WEIGHT_ATOL
    sid = out.sorted_token_ids[:npp].cpu().numpy()
    sw = out.sorted_weights[:npp].cpu().numpy()
    eid = out.expert_ids[: npp // w.block_m].cpu().numpy()
    assert np.array_equal(sid, ref.sorted_token_ids)
    assert np.array_equal(eid, ref.expert_ids)
    assert np.max(np.abs(sw - ref.sorted_weights), initial=0.0) <= WEIGHT_ATOL
    N = w.T * w.topk
    real = sid != N
    assert np.all(sw[~real] == 0.0)
    assert np.array_equal(sw[real], wt.reshape(-1)[sid[real]])
    assert out.status_word() == 0


# ------------------------------------------------------------ the five workloads
@pytest.mark.parametrize("name", list(datagen.WORKLOADS))
def test_workload_full_size(name):
    w, inp, ref = inputs_for(name)
    out = run_gpu(w, inp)
    assert_matches(out, ref, w)
    check_sort_invariants(ref.topk_ids, w.E, w.block_m, out.sorted_token_ids.cpu().numpy(),
                          out.expert_ids.cpu().numpy(), ref.num_tokens_post_pad)


@pytest.mark.parametrize("name", ["decode_T1_E896_G8", "prefill_T512_E896"])
def test_poisoned_buffers_do_not_matter(name):
    w, inp, ref = inputs_for(name)
    assert_matches(run_gpu(w, inp, poison=True), ref, w)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_other_seeds(seed):
    w, inp, ref = inputs_for("skewed_T8192_E896", T=3000, seed=seed)
    assert_matches(run_gpu(w, inp), ref, w)


# ------------------------------------------------------ ragged sizes, both paths
@pytest.mark.parametrize("T", [1, 2, 3, 4, 8, 9, 31, 32, 33, 63, 64, 65, 100, 151, 152, 153, 997])
def test_ragged_token_counts(T):
    w, inp, ref = inputs_for("prefill_T512_E896", T=T)
    assert_matches(run_gpu(w, inp), ref, w)


SHAPES = [
    # E, G, Kg, K, B, std
    (129, 3, 2, 5, 16, 1.0),      # E not a multiple of 8 (unaligned rows)
    (129, 1, 1, 7, 1, 1.0),
    (64, 64, 8, 8, 4, 1.0),       # one expert per group, 64 groups
    (256, 8, 4, 8, 64, 1.0),      # DeepSeek-V3-like
    (384, 1, 1, 8, 128, 1.0),     # Kimi-K2-like
    (4096, 16, 16, 32, 1024, 1.0),  # every group kept, K = 32, B = 1024
    (1, 1, 1, 1, 8, 1.0),         # one expert
    (96, 6, 6, 1, 2, 2.0),
    (2048, 32, 5, 12, 32, 1.0),
    (4000, 5, 2, 8, 32, 1.0),     # 800 experts per group: the one-token kernel's widest rows
]


@pytest.mark.parametrize("T", [1, 8, 17, 64, 65, 700])
@pytest.mark.parametrize("E,G,Kg,K,B,std", SHAPES)
def test_shapes(E, G, Kg, K, B, std, T):
    w = datagen.Workload("shape", T=T, E=E, n_group=G, topk_group=Kg, topk=K,
                         routed_scale=1.5, block_m=B, logit_std=std)
    inp = datagen.make_inputs(w, needs_redraw=redraw_callback(oracle, w))
    ref = oracle.route_sort(inp.logits_bf16, inp.bias, G, Kg, K, 1.5, B)
    assert_matches(run_gpu(w, inp), ref, w)


def test_exact_ties_go_to_lower_index():
    for T in (1, 40, 300):
        w = datagen.Workload("ties", T=T, E=896, n_group=8, topk_group=4, topk=16,
                             routed_scale=2.5, block_m=32)
        logits = np.full((T, 896), datagen.float32_to_bf16_bits(np.float32([0.75]))[0],
                         np.uint16)
        bias = np.zeros(896, np.float32)
        bias[::7] = 0.03125  # a few exact ties at a higher key
        inp = datagen.RouterInputs(w, logits, bias)
        ref = oracle.route_sort(logits, bias, 8, 4, 16, 2.5, 32)
        assert_matches(run_gpu(w, inp), ref, w)


def test_proxy_bound_holds_for_every_bf16_input():
    out = torch.zeros(2, dtype=torch.float32, device=DEV)
    mrs.moe_route_sort_proxy_selftest(out)
    torch.cuda.synchronize()
    max_err, bound = out.cpu().tolist()
    assert 0.0 < max_err <= bound, (max_err, bound)


@pytest.mark.parametrize("T", [300, 2000])
def test_huge_bias_takes_the_exact_route(T):
    # |bias| above the proxy's rounding limit makes every step exact.  Keys near 1100 are
    # spaced 1.2e-4 apart, so tokens are redrawn at a correspondingly wider margin.
    w = datagen.Workload("bigbias", T=T, E=896, n_group=8, topk_group=4, topk=16,
                         routed_scale=2.5, block_m=32)
    bias = datagen.make_inputs(datagen.workload("prefill_T512_E896", T=1)).bias.copy()
    bias[::45] += np.float32(1100.0)

    def needs(logits, _):
        m = oracle.margins(logits, bias, 8, 4, 16)
        return np.nonzero(m < 5e-4)[0]

    logits = datagen.make_inputs(w, needs_redraw=needs).logits_bf16
    inp = datagen.RouterInputs(w, logits, bias)
    ref = oracle.route_sort(logits, bias, 8, 4, 16, 2.5, 32)
    assert_matches(run_gpu(w, inp), ref, w)


def test_empty_call():
    w = datagen.workload("prefill_T512_E896", T=0)
    out = mrs.RouteSortBuffers.allocate(0, w.E, w.topk, w.block_m, device=DEV)
    out.num_tokens_post_pad.fill_(123)
    out.workspace.fill_(0xFF)
    logits = torch.empty((0, w.E), dtype=torch.bfloat16, device=DEV)
    bias = torch.zeros(w.E, dtype=torch.float32, device=DEV)
    mrs.route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale, w.block_m,
                   out=out)
    torch.cuda.synchronize()
    assert int(out.num_tokens_post_pad.item()) == 0
    assert out.status_word() == 0


def test_inputs_unchanged():
    w, inp, ref = inputs_for("skewed_T8192_E896")
    logits = to_dev_bf16(inp.logits_bf16)
    bias = torch.from_numpy(inp.bias).to(DEV)
    h0 = hashlib.sha256(logits.view(torch.int16).cpu().numpy().tobytes() +
                        bias.cpu().numpy().tobytes()).hexdigest()
    mrs.route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale, w.block_m)
    torch.cuda.synchronize()
    h1 = hashlib.sha256(logits.view(torch.int16).cpu().numpy().tobytes() +
                        bias.cpu().numpy().tobytes()).hexdigest()
    assert h0 == h1


# ------------------------------------------------------------------ split entry points
@pytest.mark.parametrize("name", ["decode_T1_E896_G8", "skewed_T8192_E896",
                                  "wide_T16384_E4096"])
def test_moe_topk(name):
    w, inp, ref = inputs_for(name)
    logits = to_dev_bf16(inp.logits_bf16)
    bias = torch.from_numpy(inp.bias).to(DEV)
    ids = torch.full((w.T, w.topk), -5, dtype=torch.int32, device=DEV)
    wt = torch.full((w.T, w.topk), float("nan"), dtype=torch.float32, device=DEV)
    mrs.moe_topk(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale, ids, wt)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ref.topk_ids)
    assert np.max(np.abs(wt.cpu().numpy() - ref.topk_weights)) <= WEIGHT_ATOL


@pytest.mark.parametrize("dist", ["uniform", "shared", "one_expert", "every_third_dropped",
                                  "all_dropped", "dup_in_token"])
@pytest.mark.parametrize("T,K,E,B", [(5, 4, 33, 8), (64, 16, 896, 32), (3001, 8, 256, 64),
                                     (16384, 8, 4096, 128)])
def test_moe_sort_distributions(dist, T, K, E, B):
    rng = np.random.default_rng(T + K + E + B)
    ids = ids_for(dist, T, K, E, rng)
    wts = rng.uniform(0.01, 1.0, (T, K)).astype(np.float32)
    ref = oracle.sort(ids, wts, E, B)
    out = mrs.RouteSortBuffers.allocate(T, E, K, B, device=DEV)
    out.sorted_token_ids.fill_(-3)
    out.workspace.fill_(0x5A)
    d_ids = torch.from_numpy(ids).to(DEV)
    d_w = torch.from_numpy(wts).to(DEV)
    mrs.moe_sort(d_ids, d_w, E, B, out.sorted_token_ids, out.sorted_weights, out.expert_ids,
                 out.num_tokens_post_pad, out.workspace)
    torch.cuda.synchronize()
    npp = int(out.num_tokens_post_pad.item())
    assert npp == ref.num_tokens_post_pad
    assert np.array_equal(out.sorted_token_ids[:npp].cpu().numpy(), ref.sorted_token_ids)
    assert np.array_equal(out.sorted_weights[:npp].cpu().numpy(), ref.sorted_weights)
    assert np.array_equal(out.expert_ids[: npp // B].cpu().numpy(), ref.expert_ids)
    assert out.status_word() == ref.flags == 0


@pytest.mark.parametrize("dist", ["uniform", "shared", "one_expert", "every_third_dropped",
                                  "all_dropped", "dup_in_token"])
@pytest.mark.parametrize("T,K,E,B", [(5, 4, 33, 8), (3001, 8, 256, 64), (16384, 8, 4096, 128)])
def test_moe_sort_atomic_places_the_same_routes(dist, T, K, E, B):
    # order inside an expert's segment is unspecified: compare each segment as a set, and
    # everything else exactly
    rng = np.random.default_rng(T + K + E + B)
    ids = ids_for(dist, T, K, E, rng)
    wts = rng.uniform(0.01, 1.0, (T, K)).astype(np.float32)
    ref = oracle.sort(ids, wts, E, B)
    out = mrs.RouteSortBuffers.allocate(T, E, K, B, device=DEV)
    out.sorted_token_ids.fill_(-3)
    out.workspace.fill_(0x5A)
    mrs.moe_sort(torch.from_numpy(ids).to(DEV), torch.from_numpy(wts).to(DEV), E, B,
                 out.sorted_token_ids, out.sorted_weights, out.expert_ids,
                 out.num_tokens_post_pad, out.workspace, atomic=True)
    torch.cuda.synchronize()
    npp = int(out.num_tokens_post_pad.item())
    assert npp == ref.num_tokens_post_pad
    eids = out.expert_ids[: npp // B].cpu().numpy()
    assert np.array_equal(eids, ref.expert_ids)
    sid = out.sorted_token_ids[:npp].cpu().numpy()
    sw = out.sorted_weights[:npp].cpu().numpy()
    flat_w = wts.reshape(-1)
    # padding rows exactly where the oracle has them (each segment's tail)
    assert np.array_equal(sid == T * K, ref.sorted_token_ids == T * K)
    # per expert segment: same set of flat indices, weights travel with their route
    starts = np.flatnonzero(np.r_[True, eids[1:] != eids[:-1]]) * B
    ends = np.r_[starts[1:], npp]
    for s0, s1 in zip(starts, ends):
        assert np.array_equal(np.sort(sid[s0:s1]), np.sort(ref.sorted_token_ids[s0:s1]))
    real = sid < T * K
    assert np.array_equal(sw[real], flat_w[sid[real]])
    assert np.all(sw[~real] == 0.0)
    assert out.status_word() == ref.flags == 0


@pytest.mark.parametrize("T", [3, 2000])
def test_moe_sort_flags_out_of_range_ids(T):
    rng = np.random.default_rng(T)
    E, K, B = 64, 4, 16
    ids = rng.integers(0, E, (T, K)).astype(np.int32)
    ids[T // 2, 1] = E + 3
    wts = np.ones((T, K), np.float32)
    ref = oracle.sort(ids, wts, E, B)
    assert ref.flags == oracle.FLAG_BAD_EXPERT_ID
    out = mrs.RouteSortBuffers.allocate(T, E, K, B, device=DEV)
    mrs.moe_sort(torch.from_numpy(ids).to(DEV), torch.from_numpy(wts).to(DEV), E, B,
                 out.sorted_token_ids, out.sorted_weights, out.expert_ids,
                 out.num_tokens_post_pad, out.workspace)
    torch.cuda.synchronize()
    npp = int(out.num_tokens_post_pad.item())
    assert npp == ref.num_tokens_post_pad
    assert np.array_equal(out.sorted_token_ids[:npp].cpu().numpy(), ref.sorted_token_ids)
    assert out.status_word() == mrs.DEVICE_BAD_EXPERT_ID


# ------------------------------------------------------------------ CUDA graphs
# every dispatch: one token, the single-CTA kernel, the per-token grid, the warp-per-token grid,
# the 16-CTA cluster (with the warp grid switched off, as it would take T = 200) and the
# three-kernel path
@pytest.mark.parametrize("name,T,warp_grid", [("decode_T1_E896_G8", None, True),
                                              ("prefill_T512_E896", 3, True),
                                              ("prefill_T512_E896", 40, True),
                                              ("prefill_T512_E896", None, True),
                                              ("prefill_T512_E896", 200, False),
                                              ("skewed_T8192_E896", 3000, True)])
def test_graph_replay_with_changed_inputs(name, T, warp_grid):
    w, inp, _ = inputs_for(name, T=T)
    logits = to_dev_bf16(inp.logits_bf16)
    bias = torch.from_numpy(inp.bias).to(DEV)
    out = mrs.RouteSortBuffers.allocate(w.T, w.E, w.topk, w.block_m, device=DEV)
    s = torch.cuda.Stream()
    # the hook is read when a call is enqueued: captured calls keep the path they took
    mrs.moe_route_sort_debug_set(mrs.DEBUG_WARP_GRID_TOKENS, -1 if warp_grid else 1 << 30)
    try:
        with torch.cuda.stream(s):
            mrs.route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                           w.block_m, out=out)  # first call outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            mrs.route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                           w.block_m, out=out)
    finally:
        mrs.moe_route_sort_debug_set(mrs.DEBUG_WARP_GRID_TOKENS, -1)
    for seed in range(1, 9):
        ws = datagen.workload(name, T=w.T, seed=seed)
        new = datagen.make_inputs(ws, needs_redraw=redraw_callback(oracle, ws))
        logits.copy_(to_dev_bf16(new.logits_bf16))
        bias.copy_(torch.from_numpy(new.bias).to(DEV))
        out.sorted_token_ids.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.route_sort(new.logits_bf16, new.bias, w.n_group, w.topk_group, w.topk,
                                w.routed_scale, w.block_m)
        assert_matches(out, ref, w)


@pytest.mark.parametrize("name", ["decode_T1_E896_G8", "prefill_T512_E896"])
def test_from_host_matches_device_call(name):
    # copy in, route-sort, copy the whole output block back: same bytes as the device call
    w, inp, ref = inputs_for(name)
    h_logits = torch.from_numpy(inp.logits_bf16.view(np.int16)).view(torch.bfloat16).pin_memory()
    d_logits = torch.empty_like(h_logits, device=DEV)
    bias = torch.from_numpy(inp.bias).to(DEV)
    out = mrs.RouteSortBuffers.allocate(w.T, w.E, w.topk, w.block_m, device=DEV)
    out.outputs.fill_(0)
    h_res = torch.empty(out.outputs.numel(), dtype=torch.uint8).pin_memory()
    mrs.route_sort_from_host(h_logits, d_logits, bias, w.n_group, w.topk_group, w.topk,
                             w.routed_scale, w.block_m, out, h_res)
    torch.cuda.synchronize()
    dev = run_gpu(w, inp)
    npp = int(dev.num_tokens_post_pad.item())
    assert torch.equal(h_res, out.outputs.cpu())  # the copy-out is the device block
    assert torch.equal(out.topk_ids.cpu(), dev.topk_ids.cpu())
    assert torch.equal(out.num_tokens_post_pad.cpu(), dev.num_tokens_post_pad.cpu())
    assert torch.equal(out.sorted_token_ids[:npp].cpu(), dev.sorted_token_ids[:npp].cpu())
    assert torch.equal(out.expert_ids[: npp // w.block_m].cpu(),
                       dev.expert_ids[: npp // w.block_m].cpu())
    assert torch.equal(out.topk_weights.cpu(), dev.topk_weights.cpu())


# ---------------------------------------------- the metadata drives a grouped GEMM
@pytest.mark.parametrize("name", ["prefill_T512_E896", "skewed_T8192_E896"])
def test_metadata_drives_a_block_grouped_gemm(name):
    # A consumer in the shape of GEMM1: for each block_m block, the rows named by
    # sorted_token_ids (token = row // K, sentinel rows skipped) times the block's expert
    # weight, scaled by sorted_weights, summed back per token.  It must equal the dense
    # per-token sum over the token's top-k experts.  Synthetic activations and weights.
    w, inp, _ = inputs_for(name, T=1024 if name.startswith("skewed") else None)
    out = run_gpu(w, inp)
    T, K, B, E = w.T, w.topk, w.block_m, w.E
    H, N = 64, 32
    g = torch.Generator(device=DEV).manual_seed(7)
    X = torch.randn(T, H, device=DEV, generator=g)
    W = torch.randn(E, H, N, device=DEV, generator=g) / H ** 0.5
    npp = int(out.num_tokens_post_pad.item())
    nb = npp // B
    rows = out.sorted_token_ids[:npp].long().view(nb, B)
    valid = rows < T * K
    tok = torch.where(valid, rows // K, torch.zeros_like(rows))
    rw = torch.where(valid, out.sorted_weights[:npp].view(nb, B), torch.zeros(nb, B, device=DEV))
    Y = torch.bmm(X[tok], W[out.expert_ids[:nb].long()]) * rw.unsqueeze(-1)  # [nb, B, N]
    got = torch.zeros(T, N, device=DEV).index_add_(0, tok.view(-1), Y.view(-1, N))
    ids = out.topk_ids.long()
    ref = torch.einsum("th,tkhn,tk->tn", X, W[ids], out.topk_weights)
    assert torch.allclose(got, ref, rtol=1e-4, atol=1e-4), (got - ref).abs().max().item()


@pytest.mark.parametrize("name,T", [("decode_T1_E896_G8", None), ("prefill_T512_E896", None),
                                    ("skewed_T8192_E896", 3000)])
def test_zero_copy_host_buffers(name, T):
    # logits read from, and every output written to, pinned host memory mapped into the
    # device's address space: the same results as the device buffers, with no copies
    w, inp, ref = inputs_for(name, T=T)
    h_logits = torch.from_numpy(inp.logits_bf16.view(np.int16)).view(torch.bfloat16).pin_memory()
    bias = torch.from_numpy(inp.bias).to(DEV)
    out = mrs.RouteSortBuffers.allocate_pinned(w.T, w.E, w.topk, w.block_m)
    out.outputs.fill_(0xA5)
    mrs.route_sort_mapped(mrs.map_host(h_logits), w.T, w.E, bias, w.n_group, w.topk_group,
                          w.topk, w.routed_scale, w.block_m, out)
    torch.cuda.synchronize()
    assert not out.topk_ids.is_cuda
    assert_matches(out, ref, w)


def test_map_host_address():
    t = torch.arange(1024, dtype=torch.int32).pin_memory()
    addr = mrs.map_host(t)
    assert addr != 0  # usable by the kernels: see test_zero_copy_host_buffers
    with pytest.raises(ValueError):
        mrs.map_host(torch.zeros(4))  # pageable: not accepted by the binding
