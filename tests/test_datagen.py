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
