"""Shared test helpers: golden-file parsing, near-tie redraw callback, output invariants."""
from __future__ import annotations

import os

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# A token whose selection hinges on a key or group-score gap below this is redrawn, so that
# a one-ulp difference between two correct sigmoid evaluations cannot change the ids.
NEAR_TIE = 1e-6
# Weights agree within this absolute tolerance (IEEE expf on both sides, no fast-math).
WEIGHT_ATOL = 1e-6

_INT_KEYS = {"T", "E", "n_group", "topk_group", "topk", "block_m", "num_tokens_post_pad",
             "flags"}
_INT_ARRAYS = {"topk_ids", "sorted_token_ids", "expert_ids"}
_FLOAT_ARRAYS = {"bias", "topk_weights", "sorted_weights"}


def load_golden(fname: str) -> dict:
    """Parse ``[case]`` blocks of ``key = values`` lines; ``#`` starts a comment."""
    cases: dict = {}
    cur = None
    with open(os.path.join(GOLDEN_DIR, fname)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("[") and line.endswith("]"):
                cur = cases.setdefault(line[1:-1], {})
                continue
            key, _, val = line.partition("=")
            key = key.strip()
            toks = val.split()
            if key in _INT_KEYS:
                cur[key] = int(toks[0])
            elif key == "routed_scale":
                cur[key] = float(toks[0])
            elif key == "logits_bf16":
                cur[key] = np.array([int(t, 16) for t in toks], np.uint16)
            elif key in _INT_ARRAYS:
                cur[key] = np.array([int(t) for t in toks], np.int32)
            elif key in _FLOAT_ARRAYS:
                cur[key] = np.array([float(t) for t in toks], np.float64).astype(np.float32)
            else:
                raise ValueError(f"unknown golden key {key!r} in {fname}")
    return cases


def redraw_callback(oracle_mod, w):
    """needs_redraw(logits, bias) -> rows whose oracle selection margin is below NEAR_TIE."""

    def needs(logits, bias):
        m = oracle_mod.margins(logits, bias, w.n_group, w.topk_group, w.topk)
        return np.nonzero(m < NEAR_TIE)[0]

    return needs


def gate_redraw_callback(oracle_mod, n_group, topk_group, topk):
    """needs_redraw(hidden, w_gate, bias) -> hidden rows whose logits (from the oracle's gate
    projection) have an oracle selection margin below NEAR_TIE."""

    def needs(hidden, w_gate, bias):
        logits = oracle_mod.gate_logits(hidden, w_gate)
        m = oracle_mod.margins(logits, bias, n_group, topk_group, topk)
        return np.nonzero(m < NEAR_TIE)[0]

    return needs


def check_sort_invariants(topk_ids, E, block_m, sorted_token_ids, expert_ids, npp,
                          sorted_weights=None, topk_weights=None):
    """Properties the sort output must have for any valid input (dropped ids allowed).

    Checked: counts, padding to block_m, sentinel rows, expert ownership of every block,
    a row-slot bijection over the valid routes, and token-then-slot order in each segment.
    """
    ids = np.asarray(topk_ids).reshape(-1)
    N = ids.size
    sid = np.asarray(sorted_token_ids)[:npp]
    eid = np.asarray(expert_ids)[: npp // block_m]
    assert npp % block_m == 0
    valid = (ids >= 0) & (ids < E)
    cnt = np.bincount(ids[valid], minlength=E)
    pad = (cnt + block_m - 1) // block_m * block_m
    assert npp == int(pad.sum())
    # every block is owned by one expert, non-decreasing, covering exactly nonempty experts
    assert np.all(np.diff(eid) >= 0)
    owners, nblk = np.unique(eid, return_counts=True)
    assert np.array_equal(owners, np.nonzero(cnt)[0])
    assert np.array_equal(nblk * block_m, pad[owners])
    # row-slot bijection over valid routes; sentinel rows elsewhere
    real = sid != N
    assert np.array_equal(np.sort(sid[real]), np.nonzero(valid)[0])
    # ownership and order inside each segment
    owner_of_row = np.repeat(eid, block_m)
    assert np.all(ids[sid[real]] == owner_of_row[real])
    off = np.concatenate([[0], np.cumsum(pad)[:-1]])
    for e in owners:
        seg = sid[off[e]: off[e] + pad[e]]
        head, tail = seg[: cnt[e]], seg[cnt[e]:]
        assert np.all(head != N) and np.all(tail == N)
        assert np.all(np.diff(head) > 0), "segment not in token-then-slot order"
    if sorted_weights is not None and topk_weights is not None:
        sw = np.asarray(sorted_weights)[:npp]
        tw = np.asarray(topk_weights).reshape(-1)
        assert np.array_equal(sw[real], tw[sid[real]])
        assert np.all(sw[~real] == 0.0)


def ids_for(dist, T, K, E, rng):
    """Route ids [T, K] int32 for moe_sort tests: distinct uniform experts per token, one
    expert shared by every token, all routes to one expert, every third route dropped (-1),
    all dropped, or repeated ids inside a token."""
    if dist == "uniform":
        ids = np.stack([rng.permutation(E)[:K] for _ in range(T)])
    elif dist == "shared":
        ids = np.stack([np.concatenate([[0], 1 + rng.permutation(E - 1)[:K - 1]])
                        for _ in range(T)])
    elif dist == "one_expert":
        ids = np.full((T, K), E // 2)
    elif dist == "every_third_dropped":
        ids = np.stack([rng.permutation(E)[:K] for _ in range(T)])
        ids.reshape(-1)[::3] = -1
    elif dist == "all_dropped":
        ids = np.full((T, K), -1)
    elif dist == "dup_in_token":
        ids = rng.integers(0, E, (T, K))
    else:
        raise ValueError(dist)
    return ids.astype(np.int32)
