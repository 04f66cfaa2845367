"""The seeded generator: shapes, determinism, bf16 casts, the recipe's
structure (outlier channels, sink scaling, planted segments)."""

import numpy as np
import torch

from workloads import WORKLOADS, bf16_bits, bf16_bits_to_float32, generate, retrieval_budget


def test_bf16_cast_is_torch_rne():
    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bf16_bits(x), ref)
    np.testing.assert_array_equal(bf16_bits_to_float32(ref),
                                  torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_budgets():
    assert WORKLOADS["tiny_4k_1h"].r == 8
    assert WORKLOADS["llama3_8b_128k_b1"].n_clusters == 8192
    assert WORKLOADS["llama3_8b_128k_b1"].r == 148
    w3 = WORKLOADS["llama3_8b_128k_b16"]
    assert [retrieval_budget(w3, f) for f in (0.01, 0.02, 0.03)] == [82, 164, 246]
    w4 = WORKLOADS["llama3_8b_1m_b1"]
    assert w4.n_clusters == 65536 and w4.r == 656


def test_generator_shapes_and_determinism():
    w = WORKLOADS["llama3_8b_128k_b1"]
    a = generate(w, N=9000)
    b = generate(w, N=9000)
    assert a["K"].shape == (1, 8, 9000, 128) and a["K"].dtype == np.uint16
    assert a["q"].shape == (1, 32, 128)
    for k in ("K", "V", "q", "labels"):
        np.testing.assert_array_equal(a[k], b[k])
    K = bf16_bits_to_float32(a["K"]).astype(np.float64)
    # sinks carry 4x norm: their norms stand well above the rest
    nrm = np.linalg.norm(K[0, 0], axis=1)
    assert nrm[:4].min() > 2.0 * np.median(nrm[4:])
    # two planted segments for 9000 tokens at 8192 per segment
    assert a["labels"][0, 0, :8192].max() < 512 and a["labels"][0, 0, 8192:].min() >= 512
