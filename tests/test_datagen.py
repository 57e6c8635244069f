"""The seeded input generator: determinism, bf16 rounding, skew, redraw mechanics."""
import numpy as np
import torch

from moe_expert_routing_sort_gb300 import datagen


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 3,
                        np.float32([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0, 1e-30])])
    ours = datagen.float32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_inputs_are_deterministic_and_shaped():
    for name, w in datagen.WORKLOADS.items():
        if w.T * w.E > 2_000_000:
            w = datagen.workload(name, T=64)
        a = datagen.make_inputs(w)
        b = datagen.make_inputs(w)
        assert a.logits_bf16.shape == (w.T, w.E) and a.logits_bf16.dtype == np.uint16
        assert a.bias.shape == (w.E,) and a.bias.dtype == np.float32
        assert np.array_equal(a.logits_bf16, b.logits_bf16)
        assert np.array_equal(a.bias, b.bias)
        assert np.all(np.abs(a.bias) <= w.bias_half_range)


def test_decode_variants_share_inputs():
    a = datagen.make_inputs(datagen.workload("decode_T1_E896_G8"))
    b = datagen.make_inputs(datagen.workload("decode_T1_E896_G1"))
    assert np.array_equal(a.logits_bf16, b.logits_bf16) and np.array_equal(a.bias, b.bias)


def test_skew_makes_a_few_experts_hot():
    w = datagen.workload("skewed_T8192_E896", T=2048)
    x = torch.from_numpy(datagen.make_inputs(w).logits_bf16.view(np.int16)).view(
        torch.bfloat16).float().numpy()
    col = x.mean(axis=0)
    assert col.max() > -0.1 and np.median(col) < -2.5


def test_redraw_replaces_only_named_rows():
    w = datagen.workload("prefill_T512_E896", T=16)
    base = datagen.make_inputs(w)
    calls = []

    def needs(logits, bias):
        calls.append(logits.shape[0])
        return [3, 7] if len(calls) == 1 else []

    out = datagen.make_inputs(w, needs_redraw=needs)
    assert out.redrawn_rows == 2 and calls == [16, 2]
    keep = [r for r in range(16) if r not in (3, 7)]
    assert np.array_equal(out.logits_bf16[keep], base.logits_bf16[keep])
    assert not np.array_equal(out.logits_bf16[3], base.logits_bf16[3])


def test_gate_grids_make_every_fp32_sum_exact():
    # the recipe's claim: products are multiples of 2^-10, partial sums stay below 2^9, so a
    # float32 accumulation in any order equals the exact sum (checked here in three orders,
    # including a pairwise tree, against float64, which holds these sums exactly)
    g = datagen.make_gate_inputs(3, 40, 8192, seed=9)
    h = (g.hidden_bf16.astype(np.uint32) << 16).view(np.float32)
    w = (g.w_gate_bf16.astype(np.uint32) << 16).view(np.float32)
    assert np.all(np.abs(h) <= 1) and np.all(np.abs(w) <= 3 / 64)
    assert np.all(np.mod(h * 16, 1) == 0) and np.all(np.mod(w * 64, 1) == 0)
    exact = h.astype(np.float64) @ w.astype(np.float64).T
    rng = np.random.default_rng(1)
    for t in range(3):
        for e in range(0, 40, 7):
            p = (h[t] * w[e]).astype(np.float32)
            for order in (np.arange(8192), rng.permutation(8192)):
                acc = np.float32(0)
                for v in p[order]:
                    acc = np.float32(acc + v)
                assert float(acc) == exact[t, e]
            assert float(np.sum(p, dtype=np.float32)) == exact[t, e]  # numpy's pairwise tree


def test_gate_inputs_deterministic_and_redraw():
    a = datagen.make_gate_inputs(4, 64, 256, seed=2)
    b = datagen.make_gate_inputs(4, 64, 256, seed=2)
    assert np.array_equal(a.hidden_bf16, b.hidden_bf16) and np.array_equal(a.bias, b.bias)
    calls = []

    def needs(hidden, w, bias):
        calls.append(len(hidden))
        return [1] if len(calls) == 1 else []

    c = datagen.make_gate_inputs(4, 64, 256, seed=2, needs_redraw=needs)
    assert c.redrawn_rows == 1 and calls == [4, 1]
    assert np.array_equal(c.hidden_bf16[[0, 2, 3]], a.hidden_bf16[[0, 2, 3]])
    assert not np.array_equal(c.hidden_bf16[1], a.hidden_bf16[1])
