"""Parity of the softmax-scored path (moe_route_sort_softmax, through the C ABI) with the
CPU oracle, on a GB300.

Selection runs on the bf16 logits themselves, which both sides hold exactly, so ids and all
sort metadata are compared bit for bit with no redrawing of inputs.  Weights are held to the
path's 1e-6 absolute tolerance: both sides evaluate expf on the same float differences (each
within 2 ulp); slot 0's term is exactly 1 and every other term is at most 1, so the sum is
at least 1 and a term's error reaches a weight scaled by R / sum, which keeps the difference
at a few ulp of R / 2 (about 5e-7 at R = 2.5).  A stress case with near-equal top logits (the
worst case: sums near 2) checks that margin on many tokens.  The shapes cover the
four kernels the call dispatches to (one-token, single-CTA, segment, generic), ragged token
counts, exact ties, signed zeros and logits outside the fp16 range of the unit bounds.
"""
import numpy as np
import pytest
import torch

import oracle
import moe_expert_routing_sort_gb300 as mrs
from _support import WEIGHT_ATOL, check_sort_invariants
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


def _logits(T, E, std, seed):
    w = datagen.Workload("softmax", T=T, E=E, n_group=1, topk_group=1, topk=1,
                         routed_scale=1.0, block_m=1, logit_std=std, seed=seed)
    return datagen.make_inputs(w).logits_bf16


def _run(logits_bits, K, R, B, poison=False):
    T, E = logits_bits.shape
    x = torch.from_numpy(np.ascontiguousarray(logits_bits).view(np.int16)).view(torch.bfloat16)
    out = mrs.RouteSortBuffers.allocate(T, E, K, B, device=DEV)
    if poison:
        for t in (out.topk_ids, out.sorted_token_ids, out.expert_ids, out.num_tokens_post_pad):
            t.fill_(-7)
        for t in (out.topk_weights, out.sorted_weights):
            t.fill_(float("nan"))
        out.workspace.fill_(0xA5)
    mrs.route_sort_softmax(x.to(DEV), K, R, B, out=out)
    torch.cuda.synchronize()
    return out


def _check(logits_bits, K, R, B, poison=False):
    T, E = logits_bits.shape
    out = _run(logits_bits, K, R, B, poison)
    ref = oracle.route_sort_softmax(logits_bits, K, R, B)
    atol = WEIGHT_ATOL
    npp = int(out.num_tokens_post_pad.item())
    assert npp == ref["num_tokens_post_pad"]
    ids = out.topk_ids.cpu().numpy()
    wt = out.topk_weights.cpu().numpy()
    bad = np.nonzero(np.any(ids != ref["topk_ids"], axis=1))[0]
    assert bad.size == 0, f"topk_ids differ on tokens {bad[:10]}"
    assert np.max(np.abs(wt - ref["topk_weights"]), initial=0.0) <= atol
    sid = out.sorted_token_ids[:npp].cpu().numpy()
    sw = out.sorted_weights[:npp].cpu().numpy()
    eid = out.expert_ids[: npp // B].cpu().numpy()
    assert np.array_equal(sid, ref["sorted_token_ids"])
    assert np.array_equal(eid, ref["expert_ids"])
    real = sid != T * K
    assert np.all(sw[~real] == 0.0)
    assert np.array_equal(sw[real], wt.reshape(-1)[sid[real]])
    assert out.status_word() == 0
    check_sort_invariants(ref["topk_ids"], E, B, out.sorted_token_ids.cpu().numpy(),
                          out.expert_ids.cpu().numpy(), ref["num_tokens_post_pad"])
    return out


SHAPES = [
    # E, K, B
    (896, 8, 32),     # segment kernel, 28 experts per lane
    (256, 8, 64),     # segment kernel, 8 experts per lane
    (4096, 32, 128),  # segment kernel, 128 experts per lane, K = 32
    (384, 16, 16),    # two tokens per warp once units are deep enough
    (129, 7, 1),      # E % 8 != 0: generic kernel, unaligned rows
    (64, 6, 4),       # 2 experts per lane: generic kernel
    (1, 1, 8),        # one expert
    (160, 1, 2),
]


@pytest.mark.parametrize("T", [1, 8, 17, 64, 65, 700, 5000])
@pytest.mark.parametrize("E,K,B", SHAPES)
def test_shapes(E, K, B, T):
    _check(_logits(T, E, 2.0, seed=E + T), K, 1.0, B)


@pytest.mark.parametrize("T", [1, 2, 31, 33, 152, 153, 997])
def test_ragged_token_counts_with_scale(T):
    _check(_logits(T, 896, 1.0, seed=T), 8, 2.5, 32)


@pytest.mark.parametrize("T,E", [(8192, 896), (16384, 4096)])
def test_full_size(T, E):
    _check(_logits(T, E, 1.0, seed=7), 8, 2.5, 64)


def test_poisoned_buffers_do_not_matter():
    for T in (1, 40, 3000):
        _check(_logits(T, 896, 1.0, seed=3), 8, 1.0, 32, poison=True)


@pytest.mark.parametrize("T", [1, 40, 3000])
def test_exact_ties_go_to_lower_index(T):
    # logits on a coarse grid: many exact ties at and around the K-th value
    rng = np.random.default_rng(T)
    x = np.round(rng.standard_normal((T, 896)) * 2) / 2
    _check(datagen.float32_to_bf16_bits(x.astype(np.float32)), 16, 1.0, 32)


@pytest.mark.parametrize("T", [1, 40, 3000])
def test_constant_rows(T):
    logits = np.full((T, 896), datagen.float32_to_bf16_bits(np.float32([0.5]))[0], np.uint16)
    out = _check(logits, 8, 2.0, 16)
    assert np.all(out.topk_ids.cpu().numpy() == np.arange(8))
    assert np.all(out.topk_weights.cpu().numpy() == np.float32(0.25))


@pytest.mark.parametrize("T", [1, 40, 3000])
def test_signed_zeros_tie(T):
    # rows of -0 and +0 (bf16 0x8000 / 0x0000) with a few negatives: the zeros are equal
    rng = np.random.default_rng(11)
    logits = np.where(rng.random((T, 256)) < 0.5, 0x8000, 0x0000).astype(np.uint16)
    neg = datagen.float32_to_bf16_bits(np.float32([-1.0]))[0]
    logits[:, ::5] = neg
    out = _check(logits, 8, 1.0, 8)
    ids = out.topk_ids.cpu().numpy()
    zeros = np.nonzero(np.arange(256) % 5 != 0)[0][:8]
    assert np.all(ids == zeros)


@pytest.mark.parametrize("T", [1, 40, 3000])
def test_logits_beyond_fp16_range(T):
    # unit bounds are kept in fp16: magnitudes past 65504 must still select exactly
    rng = np.random.default_rng(5)
    x = rng.standard_normal((T, 896)).astype(np.float32) * 1e5
    x[:, 3] = 3.0e38
    x[:, 500] = -3.0e38
    _check(datagen.float32_to_bf16_bits(x), 8, 1.0, 32)


@pytest.mark.parametrize("K", [2, 3, 4, 8])
def test_weights_with_near_equal_top_logits(K):
    # a handful of logits a few bf16 steps apart at the top of every row (sums of the softmax
    # terms near 2..K, weights near R / 2): the largest weight errors the arithmetic allows
    rng = np.random.default_rng(40 + K)
    T, E, R = 20000, 64, 2.5
    x = rng.standard_normal((T, E)).astype(np.float32) - 4.0
    top = rng.integers(0, E, (T, K))
    x[np.arange(T)[:, None], top] = 1.0 + rng.integers(0, 6, (T, K)) * 2.0 ** -7
    bits = datagen.float32_to_bf16_bits(x)
    out = _run(bits, K, R, 16)
    ref = oracle.route_sort_softmax(bits, K, R, 16)
    assert np.array_equal(out.topk_ids.cpu().numpy(), ref["topk_ids"])
    err = np.max(np.abs(out.topk_weights.cpu().numpy() - ref["topk_weights"]))
    print(f"softmax K={K} R={R}: largest weight difference {err:.3e} over {T} tokens")
    assert err <= WEIGHT_ATOL
