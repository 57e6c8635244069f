"""Failure paths of the CUDA path, exercised on a healthy GPU (nothing here faults or hangs).

* Bounded device waits: the library's test hook lowers the limit of every bounded wait to
  zero, so the multi-CTA path gives up on its row copies and its look-back at once.  The call
  must still return, report MOE_RS_DEVICE_WAIT_TIMEOUT in its status word, keep every write
  inside the caller's buffers, and leave the context usable for the next, correct call.
* Guard regions: every output and the workspace sit between canary bytes, at exactly the
  lengths the header documents; no workload, distribution or odd shape may touch a canary.
  This stands in for a memory checker ("Summary -- general gfx1250 ordinary-TP route
  optimization", Correctness and testing: poisoned and reused buffers).
* Proxy check: with the in-library check forced to fail, the route kernels must evaluate
  every expert exactly and still match the oracle bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import moe_expert_routing_sort_gb300 as mrs
from _support import WEIGHT_ATOL, redraw_callback
from moe_expert_routing_sort_gb300 import datagen

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
CANARY = 0x5A
PAD = 4096  # canary bytes on each side of a buffer


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mrs.build()
    oracle.build()
    mrs.load()
    yield
    mrs.moe_route_sort_debug_set(mrs.DEBUG_WAIT_LIMIT_NS, -1)
    mrs.moe_route_sort_debug_set(mrs.DEBUG_FORCE_PROXY_FAIL, 0)


def _inputs(name, T=None, seed=0):
    kw = {"seed": seed}
    if T is not None:
        kw["T"] = T
    w = datagen.workload(name, **kw)
    inp = datagen.make_inputs(w, needs_redraw=redraw_callback(oracle, w))
    logits = torch.from_numpy(inp.logits_bf16.view(np.int16)).view(torch.bfloat16).to(DEV)
    bias = torch.from_numpy(inp.bias).to(DEV)
    return w, inp, logits, bias


class Guarded:
    """A device buffer of exactly `n` elements between PAD canary bytes on each side."""

    def __init__(self, n, dtype):
        self.nbytes = n * torch.empty(0, dtype=dtype).element_size()
        self.raw = torch.full((2 * PAD + self.nbytes,), CANARY, dtype=torch.uint8, device=DEV)
        self.t = self.raw[PAD:PAD + self.nbytes].view(dtype)
        self.t.view(torch.uint8).fill_(0xA7)  # poisoned contents

    def intact(self):
        lo = self.raw[:PAD]
        hi = self.raw[PAD + self.nbytes:]
        return bool(torch.all(lo == CANARY).item()) and bool(torch.all(hi == CANARY).item())


def _guarded_outputs(T, E, K, B):
    P = mrs.moe_sort_max_padded(T, E, K, B)
    NB = mrs.moe_sort_max_blocks(T, E, K, B)
    return {
        "topk_ids": Guarded(T * K, torch.int32),
        "topk_weights": Guarded(T * K, torch.float32),
        "sorted_token_ids": Guarded(P, torch.int32),
        "sorted_weights": Guarded(P, torch.float32),
        "expert_ids": Guarded(NB, torch.int32),
        "num_tokens_post_pad": Guarded(1, torch.int32),
        "workspace": Guarded(mrs.moe_route_sort_workspace_bytes(T, E, K, B), torch.uint8),
    }


def _assert_intact(bufs, what):
    bad = [n for n, g in bufs.items() if not g.intact()]
    assert not bad, f"{what}: writes outside {bad}"


def _status(ws):
    return int(ws[:4].view(torch.int32).item())


# ------------------------------------------------------------------ bounded waits
# T = 512 runs on the warp-per-token grid and T = 40 on the per-token grid (their grid barriers
# give up), T = 200 with the warp grid off as one cluster (route step and both sort phases in
# one launch; its row copies give up); the others take the three-kernel path
@pytest.mark.parametrize("name,T,warp_grid", [("prefill_T512_E896", None, True),
                                              ("prefill_T512_E896", 40, True),
                                              ("prefill_T512_E896", 200, False),
                                              ("skewed_T8192_E896", 3000, True),
                                              ("wide_T16384_E4096", 2000, True)])
def test_wait_timeout_is_reported_and_the_context_survives(name, T, warp_grid):
    w, inp, logits, bias = _inputs(name, T=T)
    bufs = _guarded_outputs(w.T, w.E, w.topk, w.block_m)
    v = {k: g.t for k, g in bufs.items()}
    mrs.moe_route_sort_debug_set(mrs.DEBUG_WAIT_LIMIT_NS, 0)
    if not warp_grid:
        mrs.moe_route_sort_debug_set(mrs.DEBUG_WARP_GRID_TOKENS, 1 << 30)
    try:
        mrs.moe_route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                           w.block_m, **v)
        torch.cuda.synchronize()
    finally:
        mrs.moe_route_sort_debug_set(mrs.DEBUG_WAIT_LIMIT_NS, -1)
        mrs.moe_route_sort_debug_set(mrs.DEBUG_WARP_GRID_TOKENS, -1)
    assert _status(v["workspace"]) & 0x2, "the timed-out waits were not reported"
    _assert_intact(bufs, "timed-out call")
    # the next call on the same stream, with the default limit, is correct
    ref = oracle.route_sort(inp.logits_bf16, inp.bias, w.n_group, w.topk_group, w.topk,
                            w.routed_scale, w.block_m)
    mrs.moe_route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                       w.block_m, **v)
    torch.cuda.synchronize()
    assert _status(v["workspace"]) == 0
    npp = int(v["num_tokens_post_pad"].item())
    assert npp == ref.num_tokens_post_pad
    assert np.array_equal(v["topk_ids"].view(w.T, w.topk).cpu().numpy(), ref.topk_ids)
    assert np.array_equal(v["sorted_token_ids"][:npp].cpu().numpy(), ref.sorted_token_ids)
    assert np.array_equal(v["expert_ids"][: npp // w.block_m].cpu().numpy(), ref.expert_ids)
    _assert_intact(bufs, "call after the timeout")


def test_wait_timeout_in_the_sort_step_alone():
    w, inp, logits, bias = _inputs("skewed_T8192_E896", T=3000)
    routed = mrs.route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                            w.block_m)
    bufs = _guarded_outputs(w.T, w.E, w.topk, w.block_m)
    v = {k: g.t for k, g in bufs.items()}
    mrs.moe_route_sort_debug_set(mrs.DEBUG_WAIT_LIMIT_NS, 0)
    try:
        mrs.moe_sort(routed.topk_ids, routed.topk_weights, w.E, w.block_m,
                     v["sorted_token_ids"], v["sorted_weights"], v["expert_ids"],
                     v["num_tokens_post_pad"], v["workspace"])
        torch.cuda.synchronize()
    finally:
        mrs.moe_route_sort_debug_set(mrs.DEBUG_WAIT_LIMIT_NS, -1)
    assert _status(v["workspace"]) & 0x2
    _assert_intact(bufs, "timed-out moe_sort")


# ------------------------------------------------------------------ guard regions
@pytest.mark.parametrize("name,T", [(n, None) for n in datagen.WORKLOADS] +
                         [("prefill_T512_E896", 1), ("prefill_T512_E896", 65),
                          ("prefill_T512_E896", 997), ("skewed_T8192_E896", 153)])
def test_route_sort_writes_stay_inside_the_documented_lengths(name, T):
    w, inp, logits, bias = _inputs(name, T=T)
    bufs = _guarded_outputs(w.T, w.E, w.topk, w.block_m)
    v = {k: g.t for k, g in bufs.items()}
    mrs.moe_route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                       w.block_m, **v)
    torch.cuda.synchronize()
    _assert_intact(bufs, name)
    mrs.moe_route_sort_softmax(logits, w.topk, w.routed_scale, w.block_m, **v)
    torch.cuda.synchronize()
    _assert_intact(bufs, name + " softmax")


@pytest.mark.parametrize("E,G,Kg,K,B,T", [(129, 1, 1, 7, 8, 300), (4096, 64, 8, 32, 1024, 70),
                                          (1, 1, 1, 1, 1, 100), (256, 16, 4, 8, 1, 2000),
                                          (4096, 1, 1, 32, 64, 33)])
def test_odd_shapes_write_inside(E, G, Kg, K, B, T):
    rng = np.random.default_rng(E + T)
    x = rng.standard_normal((T, E)).astype(np.float32)
    bits = (x.view(np.uint32) + 0x7FFF + ((x.view(np.uint32) >> 16) & 1)) >> 16
    logits = torch.from_numpy(bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16).to(DEV)
    bias = torch.from_numpy(rng.uniform(-0.1, 0.1, E).astype(np.float32)).to(DEV)
    bufs = _guarded_outputs(T, E, K, B)
    v = {k: g.t for k, g in bufs.items()}
    mrs.moe_route_sort(logits, bias, G, Kg, K, 2.5, B, **v)
    torch.cuda.synchronize()
    _assert_intact(bufs, f"E={E} G={G} K={K} B={B} T={T}")


@pytest.mark.parametrize("dist", ["uniform", "one_expert", "third_dropped", "all_dropped",
                                  "out_of_range", "duplicates"])
@pytest.mark.parametrize("T,K,E,B", [(40, 6, 64, 16), (3000, 16, 896, 64),
                                     (2000, 8, 4096, 128)])
def test_moe_sort_writes_stay_inside(dist, T, K, E, B):
    rng = np.random.default_rng(T + K)
    ids = rng.integers(0, E, (T, K)).astype(np.int32)
    if dist == "one_expert":
        ids[:] = 3 % E
    elif dist == "third_dropped":
        ids.reshape(-1)[::3] = -1
    elif dist == "all_dropped":
        ids[:] = -5
    elif dist == "out_of_range":
        ids.reshape(-1)[::7] = E + 2
    elif dist == "duplicates":
        ids[:, 1] = ids[:, 0]
    w = rng.random((T, K)).astype(np.float32)
    ids_d = torch.from_numpy(ids).to(DEV)
    w_d = torch.from_numpy(w).to(DEV)
    bufs = _guarded_outputs(T, E, K, B)
    v = {k: g.t for k, g in bufs.items()}
    for atomic in (False, True):
        mrs.moe_sort(ids_d, w_d, E, B, v["sorted_token_ids"], v["sorted_weights"],
                     v["expert_ids"], v["num_tokens_post_pad"], v["workspace"], atomic=atomic)
        torch.cuda.synchronize()
        _assert_intact(bufs, f"moe_sort {dist} atomic={atomic}")


def test_moe_topk_and_gate_write_inside():
    w, inp, logits, bias = _inputs("skewed_T8192_E896", T=700)
    ids = Guarded(w.T * w.topk, torch.int32)
    wt = Guarded(w.T * w.topk, torch.float32)
    mrs.moe_topk(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                 ids.t.view(w.T, w.topk), wt.t.view(w.T, w.topk))
    torch.cuda.synchronize()
    assert ids.intact() and wt.intact()
    T, E, H = 5, 896, 1024
    g = datagen.make_gate_inputs(T, E, H, seed=3)
    hid = torch.from_numpy(g.hidden_bf16.view(np.int16)).view(torch.bfloat16).to(DEV)
    wg = torch.from_numpy(g.w_gate_bf16.view(np.int16)).view(torch.bfloat16).to(DEV)
    gb = torch.from_numpy(g.bias).to(DEV)
    lg = Guarded(T * E, torch.bfloat16)
    bufs = _guarded_outputs(T, E, 16, 32)
    v = {k: b.t for k, b in bufs.items()}
    mrs.moe_gate_route_sort(hid, wg, gb, 8, 4, 16, 2.5, 32, lg.t.view(T, E), **v)
    torch.cuda.synchronize()
    assert lg.intact()
    _assert_intact(bufs, "gate")


# ------------------------------------------------------------------ proxy check
# sizes that take the pruning three-kernel path (the grid paths below them use exact keys)
@pytest.mark.parametrize("name,T", [("skewed_T8192_E896", 3000), ("wide_T16384_E4096", 2100)])
def test_failed_proxy_check_takes_exact_keys(name, T):
    w, inp, logits, bias = _inputs(name, T=T)
    ref = oracle.route_sort(inp.logits_bf16, inp.bias, w.n_group, w.topk_group, w.topk,
                            w.routed_scale, w.block_m)
    state = torch.full((1,), -1, dtype=torch.int32, device=DEV)

    def run_and_compare():
        out = mrs.route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                             w.block_m)
        mrs.moe_route_sort_proxy_state(state)
        torch.cuda.synchronize()
        npp = int(out.num_tokens_post_pad.item())
        assert npp == ref.num_tokens_post_pad
        assert np.array_equal(out.topk_ids.cpu().numpy(), ref.topk_ids)
        assert np.max(np.abs(out.topk_weights.cpu().numpy() - ref.topk_weights)) <= WEIGHT_ATOL
        assert np.array_equal(out.sorted_token_ids[:npp].cpu().numpy(), ref.sorted_token_ids)
        assert out.status_word() == 0
        return int(state.item())

    mrs.moe_route_sort_debug_set(mrs.DEBUG_FORCE_PROXY_FAIL, 1)
    try:
        assert run_and_compare() == 2  # check failed: no pruning, same results
    finally:
        mrs.moe_route_sort_debug_set(mrs.DEBUG_FORCE_PROXY_FAIL, 0)
    assert run_and_compare() == 1  # the real check runs again and passes on this GPU
