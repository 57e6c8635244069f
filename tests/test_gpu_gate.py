"""Parity of the gate projection fused ahead of the path (moe_gate_route_sort, through the C
ABI) with the CPU oracle, on a GB300.

Inputs are on the coarse grids of datagen.make_gate_inputs, where every fp32 partial sum of a
dot product is exact: the GPU's logits must then equal the oracle's (one nearest-even
rounding of the exact dot product) bit for bit, and everything downstream is compared as in
the route-sort parity tests (hidden rows whose oracle selection margin is below 1e-6 are
redrawn).  On general bf16 inputs the fp32 sum is rounded, so there each logit is checked
against the oracle's within one bf16 step plus the worst-case error of an fp32 sum of H terms
(H * 2^-24 * the sum of the terms' magnitudes: cancellation makes a small logit's bf16 step
smaller than that), nearly all of them must be equal, and they are identical from call to
call; every token
whose logits row equals the oracle's routes bit for bit like the oracle's (the oracle only
ever routes its own logits: no expected value comes from the GPU), and the sort metadata is
compared exactly when every row matches, else through the sort invariants.
"""
import numpy as np
import pytest
import torch

import oracle
import moe_expert_routing_sort_gb300 as mrs
from _support import WEIGHT_ATOL, check_sort_invariants, gate_redraw_callback
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


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def _logit_bound(hb, wb):
    """Per logit: one bf16 step at the oracle's value plus the worst-case rounding error of an
    fp32 sum of the H products (H * 2^-24 * sum |h * w|)."""
    hx = (hb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    wx = (wb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    H = hx.shape[1]
    return H * 2.0 ** -24 * (np.abs(hx) @ np.abs(wx).T)


def _bf16_step(bits):
    v = np.abs((bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    return 2.0 ** (np.floor(np.log2(np.maximum(v, 2.0 ** -126))) - 7)


def _run(inp, G, Kg, K, R, B, poison=False):
    hidden = _bf16_dev(inp.hidden_bf16)
    w = _bf16_dev(inp.w_gate_bf16)
    bias = torch.from_numpy(inp.bias).to(DEV)
    T, E = hidden.shape[0], w.shape[0]
    out = mrs.RouteSortBuffers.allocate(T, E, K, B, device=DEV)
    logits = torch.empty(T, E, dtype=torch.bfloat16, device=DEV)
    if poison:
        logits.view(torch.int16).fill_(0x7FC0)
        for t in (out.topk_ids, out.sorted_token_ids, out.expert_ids, out.num_tokens_post_pad):
            t.fill_(-7)
        for t in (out.topk_weights, out.sorted_weights):
            t.fill_(float("nan"))
        out.workspace.fill_(0xA5)
    mrs.gate_route_sort(hidden, w, bias, G, Kg, K, R, B, out=out, logits=logits)
    torch.cuda.synchronize()
    return logits.view(torch.int16).cpu().numpy().view(np.uint16), out


SHAPES = [
    # E, G, Kg, K, B, H
    (896, 8, 4, 16, 32, 7168),   # Kimi-K3-shaped decode, model hidden size
    (896, 8, 4, 16, 32, 3584),   # the routed (latent) size of the same model
    (896, 1, 1, 16, 32, 7168),
    (256, 8, 4, 8, 64, 4096),
    (4096, 16, 4, 8, 128, 7168),
    (129, 3, 2, 5, 16, 1000),    # ragged rows per CTA and a ragged last chunk
    (64, 8, 4, 6, 16, 8),        # one vector per row
    (1, 1, 1, 1, 8, 8192),
]


@pytest.mark.parametrize("T", [1, 2, 5, 8])
@pytest.mark.parametrize("E,G,Kg,K,B,H", SHAPES)
def test_exact_grid(E, G, Kg, K, B, H, T):
    R = 2.5
    inp = datagen.make_gate_inputs(T, E, H, seed=E + H + T,
                                   needs_redraw=gate_redraw_callback(oracle, G, Kg, K))
    logits, out = _run(inp, G, Kg, K, R, B, poison=(T == 5))
    ref = oracle.gate_route_sort(inp.hidden_bf16, inp.w_gate_bf16, inp.bias, G, Kg, K, R, B)
    assert np.array_equal(logits, ref["logits"])
    npp = int(out.num_tokens_post_pad.item())
    assert npp == ref["num_tokens_post_pad"]
    assert np.array_equal(out.topk_ids.cpu().numpy(), ref["topk_ids"])
    wt = out.topk_weights.cpu().numpy()
    assert np.max(np.abs(wt - ref["topk_weights"]), initial=0.0) <= WEIGHT_ATOL
    sid = out.sorted_token_ids[:npp].cpu().numpy()
    assert np.array_equal(sid, ref["sorted_token_ids"])
    assert np.array_equal(out.expert_ids[: npp // B].cpu().numpy(), ref["expert_ids"])
    sw = out.sorted_weights[:npp].cpu().numpy()
    real = sid != T * K
    assert np.all(sw[~real] == 0.0)
    assert np.array_equal(sw[real], wt.reshape(-1)[sid[real]])
    assert out.status_word() == 0
    check_sort_invariants(ref["topk_ids"], E, B, out.sorted_token_ids.cpu().numpy(),
                          out.expert_ids.cpu().numpy(), ref["num_tokens_post_pad"])


@pytest.mark.parametrize("T,E,H", [(1, 896, 7168), (8, 896, 3584), (3, 4096, 7168)])
def test_general_inputs_within_one_bf16_step(T, E, H):
    rng = np.random.default_rng(T * E)
    hb = datagen.float32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wb = datagen.float32_to_bf16_bits((rng.standard_normal((E, H)) / H ** 0.5).astype(np.float32))
    inp = datagen.GateInputs(hb, wb, np.zeros(E, np.float32))
    a, _ = _run(inp, 8 if E % 8 == 0 else 1, 4 if E % 8 == 0 else 1, 8, 1.0, 32)
    b, _ = _run(inp, 8 if E % 8 == 0 else 1, 4 if E % 8 == 0 else 1, 8, 1.0, 32)
    assert np.array_equal(a, b)  # fixed summation order: the same bits every call
    ref = oracle.gate_logits(hb, wb)
    ga = (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    gr = (ref.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.all(np.abs(ga - gr) <= _bf16_step(ref) + _logit_bound(hb, wb))
    assert np.mean(a == ref) > 0.99  # fp32 accumulation rarely moves the rounding


@pytest.mark.parametrize("T,E,G,Kg,K,B,H", [(1, 896, 8, 4, 16, 32, 7168),
                                             (8, 896, 8, 4, 16, 32, 3584),
                                             (5, 896, 1, 1, 16, 32, 7168),
                                             (3, 4096, 16, 4, 8, 128, 7168),
                                             (8, 256, 8, 4, 8, 64, 4096)])
def test_general_inputs_route_like_the_oracle(T, E, G, Kg, K, B, H):
    R = 2.5
    inp = datagen.make_gate_inputs(T, E, H, seed=7 * T + E + H, grid="general",
                                   needs_redraw=gate_redraw_callback(oracle, G, Kg, K))
    logits, out = _run(inp, G, Kg, K, R, B)
    ref = oracle.gate_route_sort(inp.hidden_bf16, inp.w_gate_bf16, inp.bias, G, Kg, K, R, B)
    # logits: one bf16 step plus the fp32 accumulation bound; the fraction that differs at
    # all is reported
    ga = (logits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    gr = (ref["logits"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    bound = _bf16_step(ref["logits"]) + _logit_bound(inp.hidden_bf16, inp.w_gate_bf16)
    assert np.all(np.abs(ga - gr) <= bound)
    diff = logits != ref["logits"]
    print(f"general gate inputs T={T} E={E} H={H}: {int(diff.sum())} of {diff.size} logits "
          f"({100.0 * diff.mean():.3f}%) one bf16 step from the oracle's")
    assert diff.mean() < 0.01
    # rows with the oracle's exact logits route exactly like the oracle
    same = ~np.any(diff, axis=1)
    ids = out.topk_ids.cpu().numpy()
    wt = out.topk_weights.cpu().numpy()
    assert np.array_equal(ids[same], ref["topk_ids"][same])
    assert np.max(np.abs(wt[same] - ref["topk_weights"][same]), initial=0.0) <= WEIGHT_ATOL
    npp = int(out.num_tokens_post_pad.item())
    sid = out.sorted_token_ids[:npp].cpu().numpy()
    eid = out.expert_ids[: npp // B].cpu().numpy()
    sw = out.sorted_weights[:npp].cpu().numpy()
    if same.all():
        assert npp == ref["num_tokens_post_pad"]
        assert np.array_equal(sid, ref["sorted_token_ids"])
        assert np.array_equal(eid, ref["expert_ids"])
        assert np.max(np.abs(sw - ref["sorted_weights"]), initial=0.0) <= WEIGHT_ATOL
    check_sort_invariants(ids, E, B, out.sorted_token_ids.cpu().numpy(),
                          out.expert_ids.cpu().numpy(), npp, sorted_weights=sw,
                          topk_weights=wt)
    assert out.status_word() == 0


def test_empty_call():
    hidden = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(64, 64, dtype=torch.bfloat16, device=DEV)
    bias = torch.zeros(64, dtype=torch.float32, device=DEV)
    logits, out = mrs.gate_route_sort(hidden, w, bias, 8, 4, 6, 1.0, 16)
    torch.cuda.synchronize()
    assert int(out.num_tokens_post_pad.item()) == 0
