"""The seeded input generator: deterministic, chunk-independent, shaped as the
workloads state, and free of the method's arithmetic."""
import numpy as np
import torch

from online_kv_cache_encode_gb300 import workloads as W


def test_chunking_is_independent_of_the_range():
    w = W.WORKLOADS["gqa32k"]
    whole = W.kv_tokens(w, 0, 0, 100, 900)
    part = W.kv_tokens(w, 0, 0, 300, 700)
    np.testing.assert_array_equal(whole[200:600], part)
    np.testing.assert_array_equal(W.kv_tokens(w, 1, 0, 5, 6), W.kv_tokens(w, 1, 0, 0, 10)[5:6])
    assert not np.array_equal(W.kv_tokens(w, 0, 0, 0, 10), W.kv_tokens(w, 1, 0, 0, 10))


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32) * 100
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(W.bf16_round(x), ref)


def test_distribution_features():
    w = W.WORKLOADS["tiny"]
    K = W.kv_tokens(w, 0, 0, 0, 1024)
    V = W.kv_tokens(w, 1, 0, 0, 1024)
    assert K.dtype == np.float32 and K.shape == (1024, 1, 128)
    big = np.abs(K[:, 0]).mean(axis=0)
    assert set(np.argsort(big)[-4:]) == {7, 33, 90, 121}
    assert np.abs(V).mean() < 1.0
    w = W.WORKLOADS["swa8x4096"]
    K0 = W.kv_tokens(w, 0, 0, 0, 512)
    K1 = W.kv_tokens(w, 0, 1, 0, 512)
    ch0 = W.outlier_channels(w, 0, 0)
    assert ch0.shape == (20, 4) and all(len(set(r)) == 4 for r in ch0)
    assert not np.array_equal(ch0, W.outlier_channels(w, 0, 1))  # per layer
    assert np.array_equal(K0, W.bf16_round(K0))
    # per-token factor shared across heads: log-ratio of a token's row norms across heads is not noisy
    assert K1.shape == (512, 20, 128)


def test_block_tables_and_lengths():
    for name, w in W.WORKLOADS.items():
        bt = W.block_table(w)
        assert bt.shape == (w.batch, w.max_blocks())
        assert len(np.unique(bt)) == bt.size and bt.min() >= 0 and bt.max() < w.num_blocks()
    w = W.WORKLOADS["qjl64"]
    assert w.batch == 64 and min(w.lens) >= 1024 and max(w.lens) <= 16384
    assert W.WORKLOADS["gqa32k"].bytes_per_token_head() == 134
    assert W.WORKLOADS["long128k3"].bytes_per_token_head() == 102
    assert W.WORKLOADS["qjl64"].bytes_per_token_head() == 88
    w = W.WORKLOADS["gqa32k"]
    s = W.slots(w, W.block_table(w), 0, 0, 40)
    assert s[17] == W.block_table(w)[0, 1] * 16 + 1
