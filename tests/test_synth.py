"""The seeded generators: determinism, shapes and the bf16 encoding."""

import numpy as np
import torch

import synth


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 10,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0, -0.0,
                                  3.0e38, 1e-39], dtype=np.float32)])
    ours = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(synth.bf16_bits_to_f32(ours),
                                  torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_workloads_deterministic_and_shaped():
    for w in synth.ROUTER_WORKLOADS.values():
        s = w.with_tokens(64)
        a, b = synth.router_logits(s), synth.router_logits(s)
        assert a.shape == (64, w.E) and np.array_equal(a, b)
        assert a.dtype == (np.float32 if w.dtype == "fp32" else np.uint16)
        c = synth.router_logits(s, seed=1)
        assert not np.array_equal(a, c)


def test_zipf_bias_and_hot_tokens():
    w = synth.ROUTER_WORKLOADS["zipf-hot-top8-T131072-E256"].with_tokens(4000)
    z = synth.bf16_bits_to_f32(synth.router_logits(w)).astype(np.float64)
    col_mean = z.mean(axis=0)
    # the Zipf log-bias spreads the expert means over 1.5 * 1.2 * ln(256) ~ 10 nats
    assert col_mean.max() - col_mean.min() > 6.0
    s = synth.SINKHORN_WORKLOADS["taot-sinkhorn-B1024-R64"]
    m0, m1 = synth.sinkhorn_microbatch_logits(s, 0), synth.sinkhorn_microbatch_logits(s, 1)
    assert m0.shape == (4096, 384) and not np.array_equal(m0, m1)
