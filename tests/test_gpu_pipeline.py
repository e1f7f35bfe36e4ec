"""GPU checks of the fused step (kvq_append_decode) and of the CUDA-graph step
over a stack of layers.

* kvq_append_decode against kvq_append followed by kvq_decode on an identical
  cache: the pools byte for byte and the outputs bit for bit (the same fp32
  operation sequences run in both), over several steps, with ragged lengths, a
  sequence without a new token, a rotated query and GQA groups;
* the graph replay of a multi-layer step against the same step run eagerly:
  outputs bit for bit at every step, pools byte for byte at the end, and one
  layer's output against the float64 oracle.
"""
import numpy as np
import pytest
import torch

from kvq_testlib import Cache, assert_close_attention, i32, u16
from rotated_int2_kv_kvq_gb300 import kvq as K
from rotated_int2_kv_kvq_gb300 import workloads as W
from rotated_int2_kv_kvq_gb300.pipeline import DecodeStepGraph, LayerCache

pytestmark = pytest.mark.gpu

D = 128


def _pair(wl, lens, **kw):
    """Two identical caches holding positions [0, lens[b]) of every sequence."""
    cs = [Cache(wl, **kw), Cache(wl, **kw)]
    for c in cs:
        c.append_range(range(len(lens)), 0, [int(x) for x in lens])
    return cs


def _new_tokens(wl, lens, Hkv, layer=0):
    Kn = np.stack([W.token_at(wl, layer, b, 0, int(L))[:Hkv] for b, L in enumerate(lens)])
    Vn = np.stack([W.token_at(wl, layer, b, 1, int(L))[:Hkv] for b, L in enumerate(lens)])
    return Kn, Vn


def _fused(c, Kn, Vn, q, lens_after, splits):
    B = c.pt_np.shape[0]
    out = torch.empty((B, c.H, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(K.kvq_workspace_bytes(c.h, B, splits), dtype=torch.uint8, device="cuda")
    K.kvq_append_decode(c.h, c.pool, c.npool, u16(Kn), u16(Vn), u16(q), c.pt, i32(lens_after), out,
                        ws, splits)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _separate(c, Kn, Vn, q, lens_after, splits):
    sel = [b for b, L in enumerate(lens_after) if L >= 1]
    c.append(Kn[sel], Vn[sel], np.array(sel), np.array([lens_after[b] - 1 for b in sel]))
    return c.decode(q, lens_after, splits).astype(np.float32)


@pytest.mark.parametrize("name,splits", [("tiny_1k", 0), ("tiny_1k", 3), ("qwen3_8b_32k", 0)])
def test_append_decode_equals_append_then_decode(name, splits):
    wl = W.WORKLOADS[name]
    if name == "tiny_1k":
        lens = np.array([500])
    else:
        lens = np.concatenate([np.array([0, 1, 15, 16, 17, 300, 1000, 2047]),
                               np.array([4000] * 8)])
    a, b = _pair(wl, lens)
    for step in range(3):
        Kn, Vn = _new_tokens(wl, lens, a.Hkv)
        q = W.queries(wl, 0, 40 + step)
        lens_after = lens + 1
        if name != "tiny_1k" and step == 1:
            lens_after[0] = 0          # sequence 0 takes no token this step
        got = _fused(a, Kn, Vn, q, lens_after, splits)
        want = _separate(b, Kn, Vn, q, lens_after, splits)
        assert np.array_equal(a.pool_host(), b.pool_host()), f"pool differs at step {step}"
        assert np.array_equal(got, want), f"output differs at step {step}"
        lens = np.maximum(lens_after, lens)
    assert a.status() == 0 and b.status() == 0


@pytest.mark.parametrize("B", [24, 25, 48, 57, 64])
def test_append_decode_large_batch(B):
    """Batches whose per-sequence preparation CTAs would exceed one wave: the
    step preparation groups 2 (B = 24, 25), 4 (B = 48) or 8 (B = 57, 64)
    sequences per append CTA (B = 25 and 57 end with a group of one); B = 25
    decodes on the plain schedule (one wave of 12 splits), the others on the
    length-balanced one; all take the KV-head combine in 256-thread CTAs.  Fused step against append + decode (pools byte for byte,
    outputs bit for bit) and against the float64 oracle, on sampled (sequence,
    head) pairs plus every head of the last sequence and of sequence 1."""
    wl = W.WORKLOADS["ragged_64"]
    pt, npool = W.page_table(wl)
    pt = pt[:B].copy()
    rng = np.random.default_rng(5 + B)
    cap = (pt >= 0).sum(axis=1) * 16 - 2          # room for the two new tokens
    lens = rng.integers(1, 2500, size=B)
    lens[:6] = [0, 1, 15, 16, 17, 2047]
    lens = np.minimum(lens, cap)
    kw = dict(page_table=pt, num_pool_pages=int(pt.max()) + 1)
    a, b = _pair(wl, lens, **kw)
    for step in range(2):
        Kn, Vn = _new_tokens(wl, lens, a.Hkv)
        q = W.queries(wl, 0, 60 + step)[:B].copy()
        lens_after = lens + 1
        if step == 1:
            lens_after[0] = 0          # sequence 0 takes no token this step
        got = _fused(a, Kn, Vn, q, lens_after, 0)
        want = _separate(b, Kn, Vn, q, lens_after, 0)
        assert np.array_equal(a.pool_host(), b.pool_host()), f"pool differs at step {step}"
        assert np.array_equal(got, want), f"output differs at step {step}"
        lens = np.maximum(lens_after, lens)
    pairs = [[int(x), int(y)] for x, y in zip(rng.integers(0, B, 12), rng.integers(0, wl.num_heads, 12))]
    pairs += [[bb, hh] for bb in (1, B - 1) for hh in range(wl.num_heads)]
    oracle_out = a.oracle_decode(a.pool_host(), q, lens_after, pairs)
    assert_close_attention(got[[p[0] for p in pairs], [p[1] for p in pairs]], oracle_out,
                           f"large batch B={B}")
    assert a.status() == 0 and b.status() == 0


def test_append_decode_rotated_query_and_gqa():
    wl = W.WORKLOADS["tiny_1k"]
    for G, q_rot in ((1, False), (2, False), (4, True)):
        a, b = _pair(wl, [200], num_heads=G, num_kv_heads=1, q_rotated=q_rot)
        Kn, Vn = _new_tokens(wl, [200], 1)
        q = W.queries(wl, 0, 50)[:, :G].copy()
        got = _fused(a, Kn, Vn, q, [201], 2)
        want = _separate(b, Kn, Vn, q, [201], 2)
        assert np.array_equal(a.pool_host(), b.pool_host()), (G, q_rot)
        assert np.array_equal(got, want), (G, q_rot)


def test_append_decode_bad_page_flagged():
    wl = W.WORKLOADS["tiny_1k"]
    pt = np.arange(64, dtype=np.int32).reshape(1, 64)
    pt[0, 10] = 9999                                  # the page of position 160
    c = Cache(wl, page_table=pt, num_pool_pages=64)
    c.append_range([0], 0, 160)
    before = c.pool_host().copy()
    Kn, Vn = _new_tokens(wl, [160], 1)
    _fused(c, Kn, Vn, W.queries(wl), [161], 2)
    assert c.status() & K.KVQ_STATUS_BAD_PAGE
    assert np.array_equal(c.pool_host(), before)      # nothing stored


def _stack(wl, layers, prefill):
    caches = []
    for l in layers:
        c = Cache(wl, layer=l)
        c.append_range(range(wl.batch), 0, prefill)
        caches.append(c)
    return caches


@pytest.mark.parametrize("fused", [True, False])
def test_graph_replay_equals_eager(fused):
    wl = W.WORKLOADS["full_stack_36l"]
    layers, prefill, steps = [0, 1, 2], 256, 4
    eager_c, graph_c = _stack(wl, layers, prefill), _stack(wl, layers, prefill)
    mk = lambda cs: DecodeStepGraph([LayerCache(c.h, c.pool, c.npool, c.pt) for c in cs],
                                    wl.batch, wl.num_heads, wl.num_kv_heads, fused=fused)
    eager, graph = mk(eager_c), mk(graph_c)
    B = wl.batch

    def inputs(step):
        pos = prefill + step
        Kn = np.stack([np.stack([W.token_at(wl, l, b, 0, pos) for b in range(B)]) for l in layers])
        Vn = np.stack([np.stack([W.token_at(wl, l, b, 1, pos) for b in range(B)]) for l in layers])
        q = np.stack([W.queries(wl, l, step) for l in layers])
        lens = np.full(B, pos + 1, np.int32)
        return dict(K_new=u16(Kn), V_new=u16(Vn), q=u16(q), seq_lens=i32(lens),
                    positions=i32(lens - 1)), q, lens

    # capture() runs step 0 eagerly before capturing; run step 0 eagerly on the
    # other stack too
    x0, _, _ = inputs(0)
    graph.load(**x0)
    graph.capture()
    eager.load(**x0)
    eager.run()
    torch.cuda.synchronize()
    assert torch.equal(graph.out, eager.out)
    for step in range(1, steps):
        x, q, lens = inputs(step)
        graph.load(**x)
        graph.replay()
        eager.load(**x)
        eager.run()
        torch.cuda.synchronize()
        assert torch.equal(graph.out, eager.out), f"step {step}"
    for a, b in zip(eager_c, graph_c):
        assert np.array_equal(a.pool_host(), b.pool_host())
        assert a.status() == 0 and b.status() == 0
    # the last step of layer 1 against the oracle
    c = graph_c[1]
    pairs = [[b, (5 * b + 3) % 32] for b in range(B)]
    want = c.oracle_decode(c.pool_host(), q[1], lens, pairs)
    got = graph.out[1].cpu().numpy().astype(np.float64)
    assert_close_attention(got[[p[0] for p in pairs], [p[1] for p in pairs]], want, "graph")


@pytest.mark.parametrize("G,B", [(1, 16), (2, 16), (2, 40)])
def test_append_decode_group_sizes(G, B):
    """The fused step with G = 1 and 2 query heads per KV head (the query CTAs
    leave the unused head columns of their fragments empty): against append +
    decode bit for bit and against the float64 oracle on every head of two
    sequences.  B = 40: groups of four sequences per append CTA."""
    wl = W.WORKLOADS["ragged_64"]
    Hkv = 8
    rng = np.random.default_rng(70 + 10 * G + B)
    pt = rng.permutation(B * 64).astype(np.int32).reshape(B, 64)     # 1024 tokens each
    kw = dict(page_table=pt, num_pool_pages=B * 64, num_heads=Hkv * G, num_kv_heads=Hkv)
    lens = rng.integers(1, 1000, size=B)
    lens[:4] = [0, 1, 16, 17]
    a, b = _pair(wl, lens, **kw)
    for step in range(2):
        Kn, Vn = _new_tokens(wl, lens, Hkv)
        q = W.queries(wl, 0, 80 + step)[:B, :Hkv * G].copy()
        lens_after = lens + 1
        got = _fused(a, Kn, Vn, q, lens_after, 0)
        want = _separate(b, Kn, Vn, q, lens_after, 0)
        assert np.array_equal(a.pool_host(), b.pool_host()), f"pool differs at step {step}"
        assert np.array_equal(got, want), f"output differs at step {step}"
        lens = lens_after
    pairs = [[bb, hh] for bb in (2, B - 1) for hh in range(Hkv * G)]
    want = a.oracle_decode(a.pool_host(), q, lens, pairs)
    assert_close_attention(got[[p[0] for p in pairs], [p[1] for p in pairs]], want,
                           f"fused step G={G} B={B}")
    assert a.status() == 0 and b.status() == 0
