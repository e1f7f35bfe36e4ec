"""GPU parity of the decode with a BF16 sink + recent window (kvq_decode_window)
against the float64 oracle run on the GPU's own INT2 and BF16 pool bytes.

The OptR setting keeps the first 64 (sink) and the last 256 (recent) tokens
in BF16 beside the INT2 cache ("Assumptions & free parameters" of the OptR
page).  Checked here: window sizes that are and are not multiples of the page,
contexts shorter than the window, the two degenerate windows (empty: the plain
INT2 decode; covering the context: the plain BF16 decode), a BF16 cache that
holds the window pages only, the rotated-basis output, and GQA groups.
Tolerance: 1e-3 relative L2 and 5e-3 max-abs per output vector.
"""
import numpy as np
import pytest
import torch

from kvq_testlib import (Cache, assert_close_attention, oracle_window, window_decode,
                         window_page_table, window_positions)
from rotated_int2_kv_kvq_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _caches(wl, n, num_heads=None, num_kv_heads=None, out_rotated=False, window_only=None):
    """INT2 cache with positions [0, n) of sequence 0, and a BF16 cache with
    all of them, or (window_only = (sink, recent)) with the window pages only."""
    ci = Cache(wl, num_heads=num_heads, num_kv_heads=num_kv_heads, out_rotated=out_rotated)
    Ks, Vs = ci.append_range([0], 0, n)
    Kt, Vt = Ks[0][:, :ci.Hkv].copy(), Vs[0][:, :ci.Hkv].copy()
    if window_only is None:
        cb = Cache(wl, kind="bf16", num_heads=num_heads, num_kv_heads=num_kv_heads)
        cb.append(Kt, Vt, np.zeros(n), np.arange(n))
    else:
        sink, recent = window_only
        pt, npool = window_page_table([n], ci.pt_np.shape[1], sink, recent)
        cb = Cache(wl, kind="bf16", num_heads=num_heads, num_kv_heads=num_kv_heads,
                   page_table=pt, num_pool_pages=npool)
        pos = np.array(window_positions(n, sink, recent), np.int32)
        cb.append(Kt[pos], Vt[pos], np.zeros(len(pos)), pos)
    return ci, cb


@pytest.fixture(scope="module")
def tiny():
    wl = W.WORKLOADS["tiny_1k"]
    return _caches(wl, wl.ctx)


@pytest.mark.parametrize("sink,recent", [(64, 256), (5, 37), (16, 16), (0, 256), (64, 0),
                                         (100, 3)])
@pytest.mark.parametrize("seq_len", [1, 17, 100, 320, 321, 700, 1024])
@pytest.mark.parametrize("splits", [0, 3])
def test_tiny_window(tiny, sink, recent, seq_len, splits):
    ci, cb = tiny
    q = W.queries(ci.wl, 0, seq_len + sink)
    got = window_decode(ci, cb, q, [seq_len], sink, recent, splits)
    want = oracle_window(ci, cb, q, [seq_len], [[0, h] for h in range(4)], sink, recent)
    assert_close_attention(got[0], want, f"len {seq_len} window {sink}+{recent} splits {splits}")
    assert ci.status() == 0


def test_empty_window_is_int2_decode(tiny):
    ci, cb = tiny
    q = W.queries(ci.wl, 0, 77)
    for n in (1, 500, 1024):
        got = window_decode(ci, cb, q, [n], 0, 0, 4)
        plain = ci.decode(q, [n], 4)
        assert np.abs(got - plain).max() <= 1e-5 * max(1.0, np.abs(plain).max()), n


def test_full_window_is_bf16_decode(tiny):
    ci, cb = tiny
    q = W.queries(ci.wl, 0, 78)
    for n, (sink, recent) in [(300, (64, 256)), (1024, (1024, 0)), (1024, (0, 1024)),
                              (200, (150, 60))]:
        got = window_decode(ci, cb, q, [n], sink, recent, 2)
        plain = cb.decode(q, [n], 2)
        assert np.abs(got - plain).max() <= 1e-5 * max(1.0, np.abs(plain).max()), (n, sink, recent)


def test_empty_context(tiny):
    ci, cb = tiny
    got = window_decode(ci, cb, W.queries(ci.wl), [0], 64, 256, 2)
    assert not np.any(got)
    assert ci.status() == 0


def test_window_pages_only():
    """A BF16 cache holding only the pages of window positions (other table
    entries -1) gives the same output and raises no status bit."""
    wl = W.WORKLOADS["tiny_1k"]
    sink, recent = 64, 256
    ci, cb = _caches(wl, 1000, window_only=(sink, recent))
    q = W.queries(wl, 0, 5)
    got = window_decode(ci, cb, q, [1000], sink, recent, 0)
    want = oracle_window(ci, cb, q, [1000], [[0, h] for h in range(4)], sink, recent)
    assert_close_attention(got[0], want, "window pages only")
    assert ci.status() == 0 and cb.status() == 0


def test_window_out_rotated(tiny):
    ci, cb = tiny
    wl = ci.wl
    cr, _ = _caches(wl, 700, out_rotated=True, window_only=(64, 256))
    q = W.queries(wl, 0, 6)
    rot = window_decode(cr, cb, q, [700], 64, 256, 3)[0]
    plain = window_decode(ci, cb, q, [700], 64, 256, 3)[0]
    RV = ci.R[1, 0].astype(np.float64)
    assert np.allclose(rot @ RV.T, plain, rtol=0, atol=1e-4 * np.abs(plain).max())
    want = oracle_window(cr, cb, q, [700], [[0, h] for h in range(4)], 64, 256)
    assert_close_attention(rot, want, "rotated output with window")


@pytest.mark.parametrize("G", [1, 2])
def test_window_gqa_group_sizes(G):
    wl = W.WORKLOADS["tiny_1k"]
    ci, cb = _caches(wl, 400, num_heads=G, num_kv_heads=1)
    q = W.queries(wl, 0, 12)[:, :G].copy()
    got = window_decode(ci, cb, q, [400], 64, 256, 3)
    want = oracle_window(ci, cb, q, [400], [[0, h] for h in range(G)], 64, 256)
    assert_close_attention(got[0], want, f"G={G}")


def test_ragged_batch_window():
    """64 sequences of log-uniform lengths (some shorter than the window), a
    BF16 cache of the window pages only, the automatic split choice."""
    wl = W.WORKLOADS["ragged_64"]
    sink, recent = 64, 256
    ci = Cache(wl)
    lens = W.seq_lens(wl)
    pt, npool = window_page_table(lens, ci.pt_np.shape[1], sink, recent)
    cb = Cache(wl, kind="bf16", page_table=pt, num_pool_pages=npool)
    for g0 in range(0, wl.batch, 8):
        seqs = list(range(g0, g0 + 8))
        Ks, Vs = ci.append_range(seqs, 0, [int(x) for x in lens[g0:g0 + 8]])
        for s, k, v in zip(seqs, Ks, Vs):
            pos = np.array(window_positions(lens[s], sink, recent), np.int32)
            cb.append(k[pos], v[pos], np.full(len(pos), s), pos)
    q = W.queries(wl, 0, 3)
    got = window_decode(ci, cb, q, lens, sink, recent, 0)
    rng = np.random.default_rng(31)
    bs = [int(np.argmax(lens)), int(np.argmin(lens))] + [int(b) for b in rng.integers(0, 64, 8)]
    pairs = [[b, int(rng.integers(0, 32))] for b in bs]
    want = oracle_window(ci, cb, q, lens, pairs, sink, recent)
    assert_close_attention(got[[p[0] for p in pairs], [p[1] for p in pairs]], want, "ragged")
    assert ci.status() == 0 and cb.status() == 0


def test_window_rejects_rotated_query(tiny):
    """The window's BF16 tokens need the plain query: KVQ_Q_ROTATED is refused."""
    from rotated_int2_kv_kvq_gb300 import kvq as K
    ci, cb = tiny
    cq = Cache(ci.wl, q_rotated=True)
    out = torch.empty((1, 4, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(K.kvq_workspace_bytes(cq.h, 1, 2), dtype=torch.uint8, device="cuda")
    q = torch.zeros((1, 4, 128), dtype=torch.int16, device="cuda")
    sl = torch.tensor([100], dtype=torch.int32, device="cuda")
    with pytest.raises(K.KvqError) as e:
        K.kvq_decode_window(cq.h, cq.pool, cq.npool, cb.pool, cb.npool, cb.pt, q, cq.pt, sl, 64,
                            256, out, ws, 2)
    assert e.value.code == K.KVQ_EINVAL


def _step_tokens(wl, lens, Hkv):
    Kn = np.stack([W.token_at(wl, 0, b, 0, int(L))[:Hkv] for b, L in enumerate(lens)])
    Vn = np.stack([W.token_at(wl, 0, b, 1, int(L))[:Hkv] for b, L in enumerate(lens)])
    return Kn, Vn


@pytest.mark.parametrize("sink,recent,splits,B", [(64, 256, 0, 16), (5, 37, 3, 16),
                                                   (64, 256, 0, 41)])
def test_append_decode_window_equals_separate_calls(sink, recent, splits, B):
    """kvq_append_decode_window against kvq_append + kvq_bf16_append +
    kvq_decode_window on identical caches: both pools byte for byte and the
    outputs bit for bit, over three steps with ragged lengths and a sequence
    that takes no token in one step.  B = 41: the step preparation groups
    several sequences per append CTA (the last group short), each writing its
    tokens' BF16 copies too."""
    from kvq_testlib import i32, u16
    from rotated_int2_kv_kvq_gb300 import kvq as K
    if B == 16:
        wl = W.WORKLOADS["qwen3_8b_32k"]
        kw = {}
        lens = np.concatenate([np.array([0, 1, 15, 16, 17, 300, 1000, 2047]), np.array([700] * 8)])
    else:
        wl = W.WORKLOADS["ragged_64"]
        rng = np.random.default_rng(B)
        pt = rng.permutation(B * 48).astype(np.int32).reshape(B, 48)   # 768 tokens each
        kw = dict(page_table=pt, num_pool_pages=B * 48)
        lens = rng.integers(1, 700, size=B)
        lens[:6] = [0, 1, 15, 16, 17, 300]
    pairs = []
    for _ in range(2):
        ci, cb = Cache(wl, **kw), Cache(wl, kind="bf16", **kw)
        Ks, Vs = ci.append_range(range(len(lens)), 0, [int(x) for x in lens])
        for b, L in enumerate(lens):
            if L:
                cb.append(Ks[b][:, :ci.Hkv].copy(), Vs[b][:, :ci.Hkv].copy(), np.full(L, b),
                          np.arange(L))
        pairs.append((ci, cb))
    (a, ab), (s, sb) = pairs
    assert B == len(lens)
    for step in range(3):
        Kn, Vn = _step_tokens(wl, lens, a.Hkv)
        q = W.queries(wl, 0, 60 + step)[:B].copy()
        lens_after = lens + 1
        if step == 1:
            lens_after[0] = 0              # sequence 0 takes no token this step
        out = torch.empty((B, a.H, 128), dtype=torch.float32, device="cuda")
        ws = torch.empty(K.kvq_workspace_bytes(a.h, B, splits), dtype=torch.uint8, device="cuda")
        K.kvq_append_decode_window(a.h, a.pool, a.npool, ab.pool, ab.npool, ab.pt, u16(Kn), u16(Vn),
                                   u16(q), a.pt, i32(lens_after), sink, recent, out, ws, splits)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        sel = [b for b, L in enumerate(lens_after) if L >= 1]
        pos = np.array([lens_after[b] - 1 for b in sel])
        s.append(Kn[sel], Vn[sel], np.array(sel), pos)
        sb.append(Kn[sel], Vn[sel], np.array(sel), pos)
        want = window_decode(s, sb, q, lens_after, sink, recent, splits).astype(np.float32)
        assert np.array_equal(a.pool_host(), s.pool_host()), f"INT2 pool differs at step {step}"
        assert np.array_equal(ab.pool_host(), sb.pool_host()), f"BF16 pool differs at step {step}"
        assert np.array_equal(got, want), f"output differs at step {step}"
        lens = np.maximum(lens_after, lens)
    assert a.status() == 0 and s.status() == 0 and ab.status() == 0


def test_append_decode_window_bad_bf16_page_flagged():
    """A new position whose BF16 page id is out of range: the status bit is set,
    the BF16 pool is left as it was, the INT2 copy is still stored."""
    from kvq_testlib import i32, u16
    from rotated_int2_kv_kvq_gb300 import kvq as K
    wl = W.WORKLOADS["tiny_1k"]
    ci = Cache(wl)
    pt = np.arange(64, dtype=np.int32).reshape(1, 64)
    pt[0, 10] = 9999                                  # the BF16 page of position 160
    cb = Cache(wl, kind="bf16", page_table=pt, num_pool_pages=64)
    Ks, Vs = ci.append_range([0], 0, 160)
    cb.append(Ks[0][:, :ci.Hkv].copy(), Vs[0][:, :ci.Hkv].copy(), np.zeros(160), np.arange(160))
    before_b, before_i = cb.pool_host().copy(), ci.pool_host().copy()
    Kn, Vn = _step_tokens(wl, [160], ci.Hkv)
    out = torch.empty((1, ci.H, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(K.kvq_workspace_bytes(ci.h, 1, 2), dtype=torch.uint8, device="cuda")
    K.kvq_append_decode_window(ci.h, ci.pool, ci.npool, cb.pool, cb.npool, cb.pt, u16(Kn), u16(Vn),
                               u16(W.queries(wl)), ci.pt, i32([161]), 16, 16, out, ws, 2)
    torch.cuda.synchronize()
    assert ci.status() & K.KVQ_STATUS_BAD_PAGE
    assert np.array_equal(cb.pool_host(), before_b)
    assert not np.array_equal(ci.pool_host(), before_i)
