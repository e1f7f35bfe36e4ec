"""CPU checks of the seeded input generator (shapes, determinism, page tables,
length distribution).  The generator holds no method arithmetic."""
import numpy as np

from rotated_int2_kv_kvq_gb300 import workloads as W


def test_tokens_are_regenerable_by_range():
    wl = W.WORKLOADS["qwen3_8b_32k"]
    a = W.tokens(wl, 0, 3, 0, 1000, 3000)
    b = W.tokens(wl, 0, 3, 0, 2000, 1000)
    assert np.array_equal(a[1000:2000], b)
    assert np.array_equal(W.token_at(wl, 0, 3, 0, 2500), a[1500])
    assert not np.array_equal(W.tokens(wl, 0, 4, 0, 1000, 10), a[:10])
    many = W.tokens_many(wl, 0, [3, 5], 1, [1000, 7], [10, 20])
    assert np.array_equal(many[0], W.tokens(wl, 0, 3, 1, 1000, 10))
    assert many[1].shape == (20, 8, 128)


def test_key_distribution_recipe():
    wl = W.WORKLOADS["qwen3_8b_32k"]
    k = W.bf16_bits_to_float(W.tokens(wl, 0, 0, 0, 0, 4096)).astype(np.float64)
    mu = W.key_mean(wl).astype(np.float64)
    # per-channel offsets dominate: the calibration mean tracks the data mean
    assert np.abs(k.mean(axis=0) - mu).max() < 1.0
    spread = k.std(axis=0)
    assert np.median(spread) < 1.2 and spread.max() > 5.0     # 4 heavy outlier channels per head
    v = W.bf16_bits_to_float(W.tokens(wl, 0, 0, 1, 0, 4096))
    assert abs(v.mean()) < 0.02 and abs(v.std() - 1) < 0.02


def test_page_tables_partition_the_pool():
    for name in ["tiny_1k", "qwen3_8b_32k", "ragged_64", "full_stack_36l", "long_128k"]:
        wl = W.WORKLOADS[name]
        pt, npool = W.page_table(wl)
        used = pt[pt >= 0]
        assert len(np.unique(used)) == len(used) == npool
        assert used.min() == 0 and used.max() == npool - 1
        cap = W.capacity(wl)
        for b in range(wl.batch):
            assert (pt[b] >= 0).sum() * 16 >= cap[b]


def test_ragged_lengths():
    wl = W.WORKLOADS["ragged_64"]
    L = W.seq_lens(wl)
    assert L.shape == (64,) and L.min() >= 1024 and L.max() <= 65536
    assert np.array_equal(L, W.seq_lens(wl))


def test_rotations_deterministic():
    wl = W.WORKLOADS["tiny_1k"]
    assert np.array_equal(W.rotations(wl), W.rotations(wl))
    assert not np.array_equal(W.rotations(wl, 0), W.rotations(wl, 1))


def test_effective_bits_match_the_pages_accounting():
    """INT2 with fp16 scale/zero per 128-element group is 2 + 32/128 = 2.25
    bits; keeping 64 sink and 256 recent tokens in BF16 brings a 64K context to
    the 2.32 bits the OptR page prints ("Assumptions & free parameters")."""
    assert W.effective_bits(128) == 2.25
    assert round(W.effective_bits_window(65536, 64, 256), 2) == 2.32
    assert W.effective_bits_window(320, 64, 256) == 16.0        # all of it in the window
    assert W.effective_bits_window(100, 0, 0) == 2.25
    assert abs(W.effective_bits_window(32768, 64, 256) - (32448 * 2.25 + 320 * 16) / 32768) < 1e-12
