"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each oracle step is checked against an independent statement of the same fact: a library
conversion, a float64 evaluation, brute-force enumeration, an independent full sort, a
textbook argsort, a stable library sort, invariants, and hand-worked examples whose values
were computed on paper (tests/golden/).  A plausible slip in the oracle -- a dropped bias,
a wrong sign, max instead of the top-2 sum, the biased key in the weights, an unstable
placement, a wrong sentinel -- fails at least one of these.
"""
import itertools
import math

import numpy as np
import pytest
import torch

from _support import check_sort_invariants, load_golden
from moe_expert_routing_sort_gb300 import datagen

ALL_BF16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def _finite_bf16():
    f = torch.from_numpy(ALL_BF16.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    return ALL_BF16[np.isfinite(f)], f[np.isfinite(f)]


def _ulp32(x):
    x = np.abs(np.asarray(x, np.float32))
    return np.spacing(x).astype(np.float64)


# ------------------------------------------------------------------- O1: bf16 decode
def test_bf16_decode_matches_torch_all_patterns(oracle_mod):
    got = oracle_mod.bf16_to_float_array(ALL_BF16).view(np.uint32)
    ref = (torch.from_numpy(ALL_BF16.view(np.int16).copy()).view(torch.bfloat16)
           .float().numpy().view(np.uint32))
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ O2: sigmoid score
def test_sigmoid_special_values(oracle_mod):
    assert oracle_mod.sigmoid(0.0) == 0.5
    assert oracle_mod.sigmoid(-0.0) == 0.5
    assert oracle_mod.sigmoid(math.inf) == 1.0
    assert oracle_mod.sigmoid(-math.inf) == 0.0
    assert oracle_mod.sigmoid(100.0) == 1.0
    assert oracle_mod.sigmoid(-100.0) == 0.0


def test_sigmoid_vs_float64_all_finite_bf16(oracle_mod):
    _, x = _finite_bf16()
    s32 = oracle_mod.sigmoid_array(x).astype(np.float64)
    with np.errstate(over="ignore"):
        e64 = np.exp(-x.astype(np.float64))
    s64 = 1.0 / (1.0 + e64)
    # where expf(-x) overflows binary32 (x < -88.72) the formula's value is exactly 0
    overflow = e64 > np.finfo(np.float32).max
    assert np.all(s32[overflow] == 0.0)
    # elsewhere: expf (<= 1 ulp), the add and the divide (<= 0.5 ulp each) keep the result
    # within 2 ulp; below the normal range an absolute floor of a few subnormal steps
    tol = np.maximum(2.0 * _ulp32(s64), 4e-45)
    ok = ~overflow
    assert np.all(np.abs(s32[ok] - s64[ok]) <= tol[ok])


def test_sigmoid_monotone_and_symmetric(oracle_mod):
    _, x = _finite_bf16()
    order = np.argsort(x, kind="stable")
    s = oracle_mod.sigmoid_array(x[order])
    assert np.all(np.diff(s.astype(np.float64)) >= 0.0)
    xs = x[order]
    mid = np.abs(xs) < 30
    sp = oracle_mod.sigmoid_array(xs[mid]).astype(np.float64)
    sn = oracle_mod.sigmoid_array(-xs[mid]).astype(np.float64)
    assert np.all(np.abs(sp + sn - 1.0) <= 2.5e-7)


def test_sigmoid_vs_torch_float32(oracle_mod):
    _, x = _finite_bf16()
    s = oracle_mod.sigmoid_array(x).astype(np.float64)
    ref = torch.sigmoid(torch.from_numpy(x)).double().numpy()
    tol = np.maximum(3.0 * _ulp32(ref), 4e-45)
    assert np.all(np.abs(s - ref) <= tol)


# ------------------------------------------------------------------------ keys (R2)
def test_keys_add_bias_to_unbiased_score(oracle_mod):
    rng = np.random.default_rng(11)
    E = 512
    row = datagen.float32_to_bf16_bits(rng.standard_normal(E).astype(np.float32) * 2)
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    s, key = oracle_mod.scores_row(row, bias)
    x = oracle_mod.bf16_to_float_array(row).astype(np.float64)
    s64 = 1.0 / (1.0 + np.exp(-x))
    assert np.all(np.abs(s - s64) <= 2 * _ulp32(s64))
    k64 = s64 + bias.astype(np.float64)
    # the score's own error (<= 2 ulp of s) carries over; the add rounds once more
    assert np.all(np.abs(key - k64) <= 2 * _ulp32(s64) + _ulp32(k64))


# ------------------------------------------------------------- O3: group scores (R3)
@pytest.mark.parametrize("E,G", [(16, 4), (24, 8), (12, 12), (30, 5), (8, 1)])
def test_group_score_is_best_pair_sum(oracle_mod, E, G):
    rng = np.random.default_rng(E * 100 + G)
    g = E // G
    for _ in range(20):
        key = rng.uniform(0.3, 1.1, E).astype(np.float32)
        if rng.random() < 0.3:  # plant exact ties inside groups
            key[1::3] = key[0]
        gs = oracle_mod.group_scores_row(key, G)
        for j in range(G):
            grp = key[j * g:(j + 1) * g]
            if g == 1:
                ref = grp[0]
            else:
                ref = max(np.float32(grp[a]) + np.float32(grp[b])
                          for a, b in itertools.combinations(range(g), 2))
            assert gs[j] == np.float32(ref)


# ---------------------------------------------------------- O4: kept groups (R4)
def _beats(gs, a, b):
    return gs[a] > gs[b] or (gs[a] == gs[b] and a < b)


@pytest.mark.parametrize("G,Kg", [(8, 4), (8, 1), (8, 8), (6, 3), (5, 2), (1, 1)])
def test_kept_groups_by_subset_enumeration(oracle_mod, G, Kg):
    rng = np.random.default_rng(G * 10 + Kg)
    for trial in range(40):
        gs = rng.uniform(0.5, 2.2, G).astype(np.float32)
        if trial % 4 == 0:  # ties between groups
            gs[rng.integers(0, G, G // 2 + 1)] = gs[0]
        winners = [
            set(S) for S in itertools.combinations(range(G), Kg)
            if all(_beats(gs, a, b) for a in S for b in range(G) if b not in S)
        ]
        assert len(winners) == 1
        kept = oracle_mod.kept_groups_row(gs, Kg)
        assert set(np.nonzero(kept)[0]) == winners[0]


# ---------------------------------------------------------------- O5: top-k (R4, R5)
@pytest.mark.parametrize("E,G,Kg,K", [(64, 8, 4, 6), (24, 4, 2, 5), (12, 6, 3, 6),
                                      (32, 1, 1, 7), (16, 16, 5, 5)])
def test_topk_matches_independent_full_sort(oracle_mod, E, G, Kg, K):
    rng = np.random.default_rng(E + G + Kg + K)
    g = E // G
    for trial in range(30):
        key = rng.uniform(0.2, 1.1, E).astype(np.float32)
        if trial % 3 == 0:
            key[rng.integers(0, E, E // 3)] = key[1]  # exact ties
        gs = oracle_mod.group_scores_row(key, G)
        kept = oracle_mod.kept_groups_row(gs, Kg)
        ids = oracle_mod.topk_row(key, G, kept, K)
        everything = sorted(range(E), key=lambda e: (-float(key[e]), e))
        ref = [e for e in everything if kept[e // g]][:K]
        assert list(ids) == ref
        assert len(set(ids.tolist())) == K
        assert all(kept[e // g] for e in ids)


def test_topk_single_group_is_textbook_argsort(oracle_mod):
    rng = np.random.default_rng(5)
    for _ in range(20):
        E, K = 896, 16
        key = rng.uniform(0.2, 1.1, E).astype(np.float32)
        key[rng.integers(0, E, 40)] = key[3]
        kept = np.ones(1, np.int32)
        ids = oracle_mod.topk_row(key, 1, kept, K)
        ref = np.argsort(-key, kind="stable")[:K]
        assert np.array_equal(ids, ref)


# ------------------------------------------------------------------ O6: weights (R6)
def test_weights_use_unbiased_scores_and_sum_to_scale(oracle_mod):
    rng = np.random.default_rng(9)
    w_ = datagen.workload("prefill_T512_E896")
    inp = datagen.make_inputs(w_, T=64)
    ids, w = oracle_mod.route(inp.logits_bf16, inp.bias, w_.n_group, w_.topk_group, w_.topk,
                              w_.routed_scale)
    x = oracle_mod.bf16_to_float_array(inp.logits_bf16).astype(np.float64)
    s64 = 1.0 / (1.0 + np.exp(-x))
    for t in range(ids.shape[0]):
        sel = s64[t, ids[t]]
        ref = sel / sel.sum() * w_.routed_scale
        assert np.all(np.abs(w[t] - ref) <= 1e-6)
        assert abs(float(w[t].astype(np.float64).sum()) - w_.routed_scale) <= \
            w_.topk * 2 * np.spacing(np.float32(w_.routed_scale))
        assert np.all(w[t] > 0) and np.all(w[t] <= w_.routed_scale)
    del rng


# ------------------------------------------------------------- whole route step
@pytest.mark.parametrize("name", ["tiny_T4_E64", "decode_T1_E896_G8", "decode_T1_E896_G1",
                                  "prefill_T512_E896", "skewed_T8192_E896",
                                  "wide_T16384_E4096"])
def test_route_invariants_on_workloads(oracle_mod, name):
    w_ = datagen.workload(name)
    inp = datagen.make_inputs(w_, T=min(w_.T, 48))
    ids, wts = oracle_mod.route(inp.logits_bf16, inp.bias, w_.n_group, w_.topk_group,
                                w_.topk, w_.routed_scale)
    g = w_.E // w_.n_group
    for t in range(ids.shape[0]):
        s, key = oracle_mod.scores_row(inp.logits_bf16[t], inp.bias)
        gs = oracle_mod.group_scores_row(key, w_.n_group)
        kept = oracle_mod.kept_groups_row(gs, w_.topk_group)
        assert len(set(ids[t].tolist())) == w_.topk
        assert all(kept[e // g] for e in ids[t])
        assert kept.sum() == w_.topk_group
        ks = key[ids[t]]
        assert np.all(ks[:-1] >= ks[1:])
        # nothing outside the selection (inside the kept groups) beats the last slot
        cand = [e for e in range(w_.E) if kept[e // g] and e not in set(ids[t].tolist())]
        last = (float(ks[-1]), int(ids[t][-1]))
        assert all((float(key[e]), -e) < (last[0], -last[1]) for e in cand)


def test_route_golden_worked_examples(oracle_mod):
    for name, c in load_golden("route_sort_worked_examples.txt").items():
        logits = c["logits_bf16"].reshape(c["T"], c["E"])
        res = oracle_mod.route_sort(logits, c["bias"], c["n_group"], c["topk_group"],
                                    c["topk"], c["routed_scale"], c["block_m"])
        assert np.array_equal(res.topk_ids.reshape(-1), c["topk_ids"]), name
        assert np.array_equal(res.topk_weights.reshape(-1), c["topk_weights"]), name
        assert res.num_tokens_post_pad == c["num_tokens_post_pad"], name
        assert np.array_equal(res.sorted_token_ids, c["sorted_token_ids"]), name
        assert np.array_equal(res.sorted_weights, c["sorted_weights"]), name
        assert np.array_equal(res.expert_ids, c["expert_ids"]), name


# --------------------------------------------------------------- O7/O8: sort step
def test_sort_golden_worked_examples(oracle_mod):
    for name, c in load_golden("sort_worked_examples.txt").items():
        ids = c["topk_ids"].reshape(c["T"], c["topk"])
        w = c["topk_weights"].reshape(c["T"], c["topk"])
        res = oracle_mod.sort(ids, w, c["E"], c["block_m"])
        assert res.num_tokens_post_pad == c["num_tokens_post_pad"], name
        assert np.array_equal(res.sorted_token_ids, c["sorted_token_ids"]), name
        assert np.array_equal(res.sorted_weights, c["sorted_weights"]), name
        assert np.array_equal(res.expert_ids, c["expert_ids"]), name
        assert res.flags == c["flags"], name


def _stable_sort_reference(ids, w, E, B):
    """Segments from Python's stable sort of the valid routes by expert."""
    flat = ids.reshape(-1)
    N = flat.size
    valid = [r for r in range(N) if 0 <= flat[r] < E]
    order = sorted(valid, key=lambda r: flat[r])  # stable: keeps (token, slot) order
    out_ids, out_w, owners = [], [], []
    for e in range(E):
        seg = [r for r in order if flat[r] == e]
        if not seg:
            continue
        padded = seg + [N] * ((-len(seg)) % B)
        out_ids += padded
        out_w += [float(w.reshape(-1)[r]) for r in seg] + [0.0] * (len(padded) - len(seg))
        owners += [e] * (len(padded) // B)
    return (np.array(out_ids, np.int32), np.array(out_w, np.float32),
            np.array(owners, np.int32))


@pytest.mark.parametrize("dist", ["uniform", "shared", "one_expert", "every_third_dropped",
                                  "dup_in_token"])
@pytest.mark.parametrize("B", [1, 4, 16])
def test_sort_matches_stable_sort(oracle_mod, dist, B):
    rng = np.random.default_rng(hash((dist, B)) % 2**32)
    T, K, E = 37, 5, 29
    if dist == "uniform":
        ids = np.stack([rng.permutation(E)[:K] for _ in range(T)])
    elif dist == "shared":
        ids = np.stack([np.concatenate([[0], 1 + rng.permutation(E - 1)[:K - 1]])
                        for _ in range(T)])
    elif dist == "one_expert":
        ids = np.full((T, K), 7)
    elif dist == "every_third_dropped":
        ids = np.stack([rng.permutation(E)[:K] for _ in range(T)])
        ids.reshape(-1)[::3] = -1
    else:
        ids = rng.integers(0, E, (T, K))
    ids = ids.astype(np.int32)
    w = rng.uniform(0.01, 1.0, (T, K)).astype(np.float32)
    res = oracle_mod.sort(ids, w, E, B)
    ref_ids, ref_w, ref_owner = _stable_sort_reference(ids, w, E, B)
    assert np.array_equal(res.sorted_token_ids, ref_ids)
    assert np.array_equal(res.sorted_weights, ref_w)
    assert np.array_equal(res.expert_ids, ref_owner)
    check_sort_invariants(ids, E, B, res.sorted_token_ids, res.expert_ids,
                          res.num_tokens_post_pad, res.sorted_weights, w)


def test_sort_empty_and_max_padded(oracle_mod):
    ids = np.zeros((0, 4), np.int32)
    res = oracle_mod.sort(ids, np.zeros((0, 4), np.float32), 16, 8)
    assert res.num_tokens_post_pad == 0 and res.flags == 0
    # worst case: N routes over min(E, N) experts, each padded by B-1
    assert oracle_mod.max_padded(1, 896, 16, 32) == 16 + 16 * 31
    assert oracle_mod.max_padded(16384, 4096, 8, 128) == 131072 + 4096 * 127
    rng = np.random.default_rng(3)
    for _ in range(50):
        T, K, E, B = (int(rng.integers(1, 9)), int(rng.integers(1, 5)),
                      int(rng.integers(1, 40)), int(2 ** rng.integers(0, 5)))
        ids = rng.integers(0, E, (T, K)).astype(np.int32)
        res = oracle_mod.sort(ids, np.ones((T, K), np.float32), E, B)
        assert res.num_tokens_post_pad <= oracle_mod.max_padded(T, E, K, B)


# ---------------------------------------------------------- near-tie margin helper
def test_margins_detect_planted_ties(oracle_mod):
    w_ = datagen.workload("decode_T1_E896_G1")
    inp = datagen.make_inputs(w_, T=4)
    m = oracle_mod.margins(inp.logits_bf16, inp.bias, 1, 1, 16)
    assert np.all(m > 0)
    # make experts 10 and 11 tie exactly and both land in the top-16 of token 0
    logits = inp.logits_bf16.copy()
    bias = inp.bias.copy()
    logits[0, 10] = logits[0, 11] = datagen.float32_to_bf16_bits(np.float32([6.0]))[0]
    bias[10] = bias[11] = 0.0
    m2 = oracle_mod.margins(logits, bias, 1, 1, 16)
    assert m2[0] == 0.0


def test_margins_match_a_direct_computation(oracle_mod):
    # the three gaps of the margin, recomputed here in float64 from float64 keys: they agree
    # with the oracle's float32 values to float32 rounding
    rng = np.random.default_rng(31)
    T, E, G, Kg, K = 30, 48, 6, 3, 5
    logits = datagen.float32_to_bf16_bits(rng.standard_normal((T, E)).astype(np.float32))
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    m = oracle_mod.margins(logits, bias, G, Kg, K)
    x = (logits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    key = 1.0 / (1.0 + np.exp(-x)) + bias.astype(np.float64)
    g = E // G
    for t in range(T):
        kg = key[t].reshape(G, g)
        gs = np.sort(kg, axis=1)[:, -2:].sum(axis=1)
        order = np.argsort(-gs, kind="stable")
        gaps = [gs[order[Kg - 1]] - gs[order[Kg]]]
        cand = np.sort(kg[order[:Kg]].ravel())[::-1]
        gaps.append(cand[K - 1] - cand[K])
        gaps += list(cand[:K - 1] - cand[1:K])
        assert abs(m[t] - min(gaps)) < 1e-6, (t, m[t], min(gaps))


# ----------------------------------------------------- softmax variant (reading R13)
def test_softmax_topk_is_argsort_of_logits(oracle_mod):
    # selection is on the logits themselves: a textbook stable argsort of -x (ties -> lower
    # index), on coarse values so that exact ties are frequent
    rng = np.random.default_rng(5)
    T, E, K = 40, 96, 7
    x = np.round(rng.standard_normal((T, E)) * 4) / 4
    logits = datagen.float32_to_bf16_bits(x.astype(np.float32))
    ids, _ = oracle_mod.route_softmax(logits, K, 1.0)
    for t in range(T):
        want = np.argsort(-x[t], kind="stable")[:K]
        assert np.array_equal(ids[t], want)


def test_softmax_weights_are_renormalised_softmax(oracle_mod):
    rng = np.random.default_rng(6)
    T, E, K, R = 64, 200, 8, 2.5
    logits = datagen.float32_to_bf16_bits(rng.standard_normal((T, E)).astype(np.float32) * 3)
    ids, w = oracle_mod.route_softmax(logits, K, R)
    x = (logits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for t in range(T):
        p = np.exp(x[t] - x[t].max())
        p = p / p.sum()                       # softmax over all E experts
        sel = p[ids[t]]
        ref = sel / sel.sum() * R             # restricted to the top-K, renormalised
        assert np.allclose(w[t], ref, rtol=0, atol=2e-7 * R)
        assert np.all(np.diff(w[t]) <= 0)     # slots in descending order
        assert abs(w[t].astype(np.float64).sum() - R) < 1e-5


def test_softmax_two_experts_closed_form(oracle_mod):
    # K = 2: w_0 = R * sigmoid(x_0 - x_1) exactly in real arithmetic; x = [2, 0, 1, 0]
    logits = datagen.float32_to_bf16_bits(np.float32([[2.0, 0.0, 1.0, 0.0]]))
    ids, w = oracle_mod.route_softmax(logits, 2, 1.0)
    assert ids.tolist() == [[0, 2]]
    assert abs(w[0, 0] - 1 / (1 + math.exp(-1))) < 1e-7
    assert abs(w[0, 1] - 1 / (1 + math.exp(1))) < 1e-7
    # ties: [1, 3, 3, 0] -> slots 1 then 2 (lower index first), equal weights
    logits = datagen.float32_to_bf16_bits(np.float32([[1.0, 3.0, 3.0, 0.0]]))
    ids, w = oracle_mod.route_softmax(logits, 2, 4.0)
    assert ids.tolist() == [[1, 2]] and w.tolist() == [[2.0, 2.0]]


# -------------------------------------------- gate projection (reading R14)
def _bf16_rne_exact(v) -> int:
    # independent rounding of an exact rational v (a Fraction): comparison against the two
    # bracketing finite bf16 values from the full table, ties to the even pattern, +0 for 0
    # (on |v| over the non-negative patterns 0x0000..0x7f80; the sign is put back after)
    from fractions import Fraction
    v = Fraction(v)
    if v == 0:
        return 0x0000
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    bits = np.arange(0x7F81, dtype=np.uint32)
    vals = (bits << 16).view(np.float32).astype(np.float64)  # ascending, ends at +inf
    i = int(np.searchsorted(vals, float(a), side="left"))
    # float(a) may round: step to the exact bracket
    while i > 0 and Fraction(float(vals[i - 1])) >= a:
        i -= 1
    while np.isfinite(vals[i]) and Fraction(float(vals[i])) < a:
        i += 1
    if np.isfinite(vals[i]) and Fraction(float(vals[i])) == a:
        return int(bits[i]) | sign
    lo, hi = i - 1, i
    dl = a - Fraction(float(vals[lo]))
    dh = (Fraction(float(vals[hi])) - a) if np.isfinite(vals[hi]) else None
    if dh is None:
        # past the largest finite bf16: round to nearest with the infinity step 2^120
        pick = hi if dl >= Fraction(2) ** 119 else lo
    elif dl < dh:
        pick = lo
    elif dh < dl:
        pick = hi
    else:
        pick = lo if (int(bits[lo]) & 1) == 0 else hi
    return int(bits[pick]) | sign


def _bf16_value(b):
    from fractions import Fraction
    return Fraction(float((np.uint32(b) << np.uint32(16)).view(np.float32)))


def _bf16_of(x: float) -> int:
    b = int(datagen.float32_to_bf16_bits(np.float32([x]))[0])
    assert float(_bf16_value(b)) == x, x  # only exact bf16 values here
    return b


def _gate_one(oracle_mod, pairs):
    """The oracle's logit for one hidden row and one gate row given as (h, w) float pairs."""
    hb = np.array([[_bf16_of(h) for h, _ in pairs]], np.uint16)
    wb = np.array([[_bf16_of(w) for _, w in pairs]], np.uint16)
    return int(oracle_mod.gate_logits(hb, wb)[0, 0])


def test_gate_logits_round_the_exact_sum_once(oracle_mod):
    # ties: 1 + 2^-8 lies halfway between 1 (0x3f80) and 1 + 2^-7 (0x3f81): even is 0x3f80;
    # 1 + 3 * 2^-8 lies halfway between 0x3f81 and 0x3f82: even is 0x3f82
    assert _gate_one(oracle_mod, [(1.0, 1.0), (2 ** -4, 2 ** -4)]) == 0x3F80
    assert _gate_one(oracle_mod, [(1.0, 1.0), (2 ** -4, 2 ** -4), (2 ** -7, 1.0)]) == 0x3F82
    assert _gate_one(oracle_mod, [(-1.0, 1.0), (2 ** -4, -2 ** -4), (-(2 ** -7), 1.0)]) == 0xBF82
    # just above a tie rounds up, even when the excess is far below a double's precision
    assert _gate_one(oracle_mod, [(1.0, 1.0), (2 ** -4, 2 ** -4), (2 ** -60, 2 ** -60)]) == 0x3F81
    # cancellation: 2^60 + 2^-30 - 2^60 = 2^-30 exactly (a sum in double gives 0)
    assert _gate_one(oracle_mod, [(2 ** 30, 2 ** 30), (2 ** -15, 2 ** -15),
                                  (2 ** 30, -2 ** 30)]) == _bf16_of(2 ** -30)
    # exact zero is +0; the smallest subnormal survives; overflow gives infinity
    assert _gate_one(oracle_mod, [(1.0, 1.0), (1.0, -1.0)]) == 0x0000
    assert _gate_one(oracle_mod, [(2 ** -70, 2 ** -63)]) == 0x0001
    assert _gate_one(oracle_mod, [(2 ** -70, 2 ** -64)]) == 0x0000  # half the smallest: even
    assert _gate_one(oracle_mod, [(2 ** 100, 2 ** 100)]) == 0x7F80
    assert _gate_one(oracle_mod, [(-(2 ** 100), 2 ** 100)]) == 0xFF80


def test_gate_logits_equal_exact_rational_rounding(oracle_mod):
    # random rows with widely spread exponents (so sums in double would lose bits), checked
    # entry by entry against the exact rational dot product rounded once
    rng = np.random.default_rng(24)
    T, E, H = 3, 6, 64
    hx = rng.standard_normal((T, H)) * 2.0 ** rng.integers(-40, 40, (T, H))
    wx = rng.standard_normal((E, H)) * 2.0 ** rng.integers(-40, 40, (E, H))
    hb = datagen.float32_to_bf16_bits(hx.astype(np.float32))
    wb = datagen.float32_to_bf16_bits(wx.astype(np.float32))
    got = oracle_mod.gate_logits(hb, wb)
    for t in range(T):
        for e in range(E):
            exact = sum(_bf16_value(hb[t, h]) * _bf16_value(wb[e, h]) for h in range(H))
            assert got[t, e] == _bf16_rne_exact(exact), (t, e)


def test_gate_logits_exact_on_a_coarse_grid(oracle_mod):
    # hidden = i/16, w = j/64 with small integers: every partial sum is a multiple of 2^-10
    # below 2^9, so the dot products are exact in float32; torch's float32 -> bf16
    # conversion (one rounding, nearest-even) must then give the same bits
    rng = np.random.default_rng(22)
    T, E, H = 5, 48, 1024
    h = rng.integers(-16, 17, (T, H)) / 16.0
    w = rng.integers(-3, 4, (E, H)) / 64.0
    hb = datagen.float32_to_bf16_bits(h.astype(np.float32))
    wb = datagen.float32_to_bf16_bits(w.astype(np.float32))
    got = oracle_mod.gate_logits(hb, wb)
    exact = (h @ w.T).astype(np.float32)
    assert np.array_equal((h @ w.T), exact.astype(np.float64))  # representable exactly
    want = torch.from_numpy(exact).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_gate_logits_within_half_ulp_of_float64(oracle_mod):
    rng = np.random.default_rng(23)
    T, E, H = 3, 40, 777
    hb = datagen.float32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wb = datagen.float32_to_bf16_bits((rng.standard_normal((E, H)) * 0.03).astype(np.float32))
    got = oracle_mod.gate_logits(hb, wb)
    hx = (hb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    wx = (wb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = hx @ wx.T
    g = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    # the bf16 spacing at |ref| is 2^(floor(log2|ref|) - 7)
    spacing = 2.0 ** (np.floor(np.log2(np.abs(ref))) - 7)
    assert np.all(np.abs(g - ref) <= 0.5 * spacing * (1 + 1e-12))
    for t in range(T):  # and the row/column roles are not swapped
        for e in (0, 17, 39):
            exact = sum(_bf16_value(hb[t, h]) * _bf16_value(wb[e, h]) for h in range(H))
            assert got[t, e] == _bf16_rne_exact(exact)
