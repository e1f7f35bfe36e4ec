"""GPU parity of the INT2 path through the C ABI against the CPU oracle.

* appended bytes (codes, page placement, fp16 scale/zero): bit-exact; a code
  may differ only where the oracle's pre-rounding value lies within 1 ulp of a
  rounding boundary, and such cases are counted;
* dequantisation export: bit-exact (same fp32 fmaf on both sides);
* decode attention: within 1e-3 relative L2 and 5e-3 max-abs of the float64
  oracle run on the GPU's own pool bytes.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
from kvq_testlib import (Cache, assert_boundary_count, assert_close_attention, compare_codes, i32,
                         oracle_window, u16, window_decode, window_page_table, window_positions)
from rotated_int2_kv_kvq_gb300 import kvq as K
from rotated_int2_kv_kvq_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _block_fn(wl, layer):
    @functools.lru_cache(maxsize=256)
    def blk(seq, which, b):
        return W.tokens(wl, layer, seq, which, b * 1024, 1024)

    return (lambda s, p: blk(s, 0, p // 1024)[p % 1024],
            lambda s, p: blk(s, 1, p // 1024)[p % 1024])


# ---------------------------------------------------------------------------
# tiny workload: everything checked exhaustively
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def tiny():
    wl = W.WORKLOADS["tiny_1k"]
    c = Cache(wl)
    Ks, Vs = c.append_range([0], 0, wl.ctx)
    return c, Ks[0], Vs[0]


def test_tiny_append_bitexact(tiny):
    c, Kt, Vt = tiny
    pool = c.pool_host()
    ref = np.zeros_like(pool)
    n = Kt.shape[0]
    oracle.append_int2(ref, c.npool, 1, Kt, Vt, np.zeros(n), np.arange(n), c.pt_np, c.R, c.mu,
                       c.wl.clip_k, c.wl.clip_v)
    if not np.array_equal(pool, ref):
        # only boundary cases may differ: check token by token
        Ktok, Vtok = (lambda s, p: Kt[p]), (lambda s, p: Vt[p])
        near = compare_codes(c, pool, [(0, p, 0) for p in range(n)], Ktok, Vtok)
        assert_boundary_count(near, n, "tiny")
    assert c.status() == 0


def test_tiny_dequant_bitexact(tiny):
    c, _, _ = tiny
    n = c.wl.ctx
    Ko = torch.empty((n, 1, 128), dtype=torch.float32, device="cuda")
    Vo = torch.empty_like(Ko)
    K.kvq_dequant(c.h, c.pool, c.npool, c.pt, 0, 0, n, Ko, Vo)
    Kr, Vr = oracle.dequant_int2(c.pool_host(), c.npool, 1, c.pt_np, 0, 0, n)
    assert np.array_equal(Ko.cpu().numpy(), Kr) and np.array_equal(Vo.cpu().numpy(), Vr)


@pytest.mark.parametrize("seq_len", [1, 2, 15, 16, 17, 100, 333, 1023, 1024])
@pytest.mark.parametrize("splits", [0, 1, 2, 7, 64])
def test_tiny_decode(tiny, seq_len, splits):
    c, _, _ = tiny
    q = W.queries(c.wl, 0, seq_len)
    got = c.decode(q, [seq_len], splits)
    want = c.oracle_decode(c.pool_host(), q, [seq_len], [[0, h] for h in range(4)])
    assert_close_attention(got[0], want, f"len {seq_len} splits {splits}")


def test_tiny_decode_empty_context(tiny):
    c, _, _ = tiny
    got = c.decode(W.queries(c.wl), [0], 3)
    assert not np.any(got)
    assert c.status() == 0


def test_split_count_invariance(tiny):
    c, _, _ = tiny
    q = W.queries(c.wl, 0, 5)
    outs = [c.decode(q, [1000], s) for s in (1, 2, 7, 63, 64)]
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 1e-5 * max(1.0, np.abs(outs[0]).max())


def test_out_rotated_flag(tiny):
    c, Kt, Vt = tiny
    c2 = Cache(c.wl, out_rotated=True)
    c2.append(Kt, Vt, np.zeros(Kt.shape[0]), np.arange(Kt.shape[0]))
    q = W.queries(c.wl, 0, 9)
    rot = c2.decode(q, [500], 4)[0]
    plain = c.decode(q, [500], 4)[0]
    RV = c.R[1, 0].astype(np.float64)
    assert np.allclose(rot @ RV.T, plain, rtol=0, atol=1e-4 * np.abs(plain).max())
    want = c2.oracle_decode(c2.pool_host(), q, [500], [[0, h] for h in range(4)])
    assert_close_attention(rot, want, "rotated output")


def _rotate_queries(q_bits, RK, G):
    """bf16(q R_K) per query head, the query a caller with R_K folded into its
    projection passes under KVQ_Q_ROTATED."""
    q = W.bf16_bits_to_float(q_bits).astype(np.float64)
    out = np.empty_like(q)
    for h in range(q.shape[1]):
        out[:, h] = q[:, h] @ RK[h // G].astype(np.float64)
    return W.to_bf16_bits(out.astype(np.float32))


@pytest.mark.parametrize("out_rotated", [False, True])
def test_q_rotated_flag(tiny, out_rotated):
    """KVQ_Q_ROTATED: the caller passes q R_K; decode skips the query rotation.
    Oracle: the same pool with R_K replaced by the identity for the query."""
    c, Kt, Vt = tiny
    c2 = Cache(c.wl, q_rotated=True, out_rotated=out_rotated)
    c2.append(Kt, Vt, np.zeros(Kt.shape[0]), np.arange(Kt.shape[0]))
    assert np.array_equal(c2.pool_host(), c.pool_host())    # append ignores the flags
    q = W.queries(c.wl, 0, 10)
    qr = _rotate_queries(q, c.R[0], 4)
    got = c2.decode(qr, [777], 3)
    R_id = c.R.copy()
    R_id[0] = np.eye(128, dtype=np.float32)
    want = oracle.decode_pairs("int2", c2.pool_host(), c2.npool, 4, 1, qr, c2.pt_np, [777],
                               [[0, h] for h in range(4)], R=R_id, out_rotated=out_rotated)
    assert_close_attention(got[0], want, f"q rotated, out_rotated={out_rotated}")
    # against the unfolded path: only the bf16 rounding of q R_K differs
    plain = c.decode(q, [777], 3)[0]
    if out_rotated:
        plain = plain @ c.R[1, 0].astype(np.float64)
    assert np.abs(got[0] - plain).max() <= 2e-2 * np.abs(plain).max()


@pytest.mark.parametrize("G", [1, 2])
def test_gqa_group_sizes(G):
    wl = W.WORKLOADS["tiny_1k"]
    c = Cache(wl, num_heads=G, num_kv_heads=1)
    c.append_range([0], 0, 300)
    q = W.queries(wl, 0, 11)[:, :G].copy()
    got = c.decode(q, [300], 3)
    want = c.oracle_decode(c.pool_host(), q, [300], [[0, h] for h in range(G)])
    assert_close_attention(got[0], want, f"G={G}")


@pytest.mark.parametrize("Hkv", [2, 4, 6])
@pytest.mark.parametrize("splits", [0, 3])
def test_kv_head_counts_sharing_a_cta(Hkv, splits):
    """Hkv = 2, 4, 6 (G = 4): the decode CTA serves 2, 4 or 2 KV heads, so 4, 2
    or 4 warps share each head and their partials merge through shared memory."""
    wl = W.WORKLOADS["qwen3_8b_32k"]
    B, L = 2, 3001
    pt, _ = W.page_table(wl)
    pt = pt[:B].copy()
    c = Cache(wl, page_table=pt, num_pool_pages=int(pt.max()) + 1, num_heads=4 * Hkv,
              num_kv_heads=Hkv)
    c.append_range(range(B), 0, L)
    q = W.queries(wl, 0, 40 + Hkv, batch=B)[:, :4 * Hkv].copy()
    lens = [L, L - 1000]
    got = c.decode(q, lens, splits)
    pairs = [[b, h] for b in range(B) for h in range(4 * Hkv)]
    want = c.oracle_decode(c.pool_host(), q, lens, pairs)
    assert_close_attention(got.reshape(-1, 128), want, f"Hkv={Hkv} splits={splits}")
    assert c.status() == 0


@pytest.mark.parametrize("Hkv,splits", [(8, 128), (2, 200)])
def test_balanced_schedule(Hkv, splits):
    """Several sequences whose batch x splits CTAs exceed one wave take the
    length-balanced schedule: one chunk size for the batch, chunks per
    sequence in proportion to its length, partials in per-sequence slots.
    Lengths include an empty sequence, a one-page one and page-boundary cases;
    with Hkv = 2 two KV heads share a CTA (four warps per head, merged through
    shared memory)."""
    wl = W.WORKLOADS["qwen3_8b_32k"]
    lens = [3001, 0, 17, 1200, 2999, 16, 600]
    B = len(lens)
    pt, _ = W.page_table(wl)
    pt = pt[:B].copy()
    c = Cache(wl, page_table=pt, num_pool_pages=int(pt.max()) + 1, num_heads=4 * Hkv,
              num_kv_heads=Hkv)
    c.append_range([b for b in range(B) if lens[b] > 0], 0, [L for L in lens if L > 0])
    q = W.queries(wl, 0, 70 + Hkv, batch=B)[:, :4 * Hkv].copy()
    got = c.decode(q, lens, splits)
    pairs = [[b, h] for b in range(B) for h in range(4 * Hkv)]
    want = c.oracle_decode(c.pool_host(), q, lens, pairs)
    assert np.all(got[1] == 0.0), "an empty sequence decodes to zeros"
    assert_close_attention(got.reshape(-1, 128), want, f"balanced Hkv={Hkv} splits={splits}")
    assert c.status() == 0


@pytest.mark.parametrize("Hkv", [8, 2])
def test_single_split_long_context(Hkv):
    """One split over 21,000 tokens: 1,313 pages, more than the 1,024 page ids
    a CTA stages at a time, so the second sub-chunk's ids are reloaded (with
    Hkv = 2 four warps share each head and take every fourth page)."""
    wl = W.WORKLOADS["qwen3_8b_32k"]
    L = 21000
    pt, _ = W.page_table(wl)
    pt = pt[:1].copy()
    c = Cache(wl, page_table=pt, num_pool_pages=int(pt.max()) + 1, num_heads=4 * Hkv,
              num_kv_heads=Hkv)
    for s0 in range(0, L, 7000):
        c.append_range([0], s0, 7000)
    q = W.queries(wl, 0, 50 + Hkv, batch=1)[:, :4 * Hkv].copy()
    got = c.decode(q, [L], 1)
    pairs = [[0, h] for h in range(0, 4 * Hkv, 3)]
    want = c.oracle_decode(c.pool_host(), q, [L], pairs)
    assert_close_attention(got[0, [p[1] for p in pairs]], want, f"1 split Hkv={Hkv}")
    # the automatic split count: the same tolerance against the oracle, and
    # both split counts agree far more closely than that
    auto = c.decode(q, [L], 0)
    assert_close_attention(auto[0, [p[1] for p in pairs]], want, f"auto splits Hkv={Hkv}")
    for h in range(4 * Hkv):
        d = np.linalg.norm(auto[0, h] - got[0, h]) / np.linalg.norm(got[0, h])
        assert d <= 1e-4, (h, d)
    assert c.status() == 0


def test_multi_sequence_interleaved_append():
    """Tokens of several sequences in one call, in shuffled order, including
    several tokens of one page: every byte still lands where the oracle puts it."""
    wl = W.WORKLOADS["qwen3_8b_32k"]
    B, n_per = 3, 70
    pt = np.arange(B * 5, dtype=np.int32).reshape(B, 5)[:, ::-1].copy()
    c = Cache(wl, page_table=pt, num_pool_pages=B * 5)
    seqs = np.repeat(np.arange(B), n_per).astype(np.int32)
    pos = np.tile(np.arange(n_per), B).astype(np.int32)
    perm = np.random.default_rng(0).permutation(B * n_per)
    seqs, pos = seqs[perm], pos[perm]
    Kt = np.stack([W.token_at(wl, 0, s, 0, p) for s, p in zip(seqs, pos)])
    Vt = np.stack([W.token_at(wl, 0, s, 1, p) for s, p in zip(seqs, pos)])
    c.append(Kt, Vt, seqs, pos)
    ref = np.zeros(c.npool * 8 * 1152, np.uint8)
    oracle.append_int2(ref, c.npool, 8, Kt, Vt, seqs, pos, pt, c.R, c.mu, wl.clip_k, wl.clip_v)
    pool = c.pool_host()
    if not np.array_equal(pool, ref):
        near = compare_codes(c, pool, [(s, p, kv) for s, p in zip(seqs, pos) for kv in range(8)],
                             lambda s, p: Kt[np.nonzero((seqs == s) & (pos == p))[0][0]],
                             lambda s, p: Vt[np.nonzero((seqs == s) & (pos == p))[0][0]])
        assert_boundary_count(near, len(seqs) * 8, "interleaved")
    q = W.queries(wl, 0, 1, batch=B)
    got = c.decode(q, [n_per] * B, 2)
    pairs = [[b, h] for b in range(B) for h in range(0, 32, 5)]
    want = c.oracle_decode(pool, q, [n_per] * B, pairs)
    assert_close_attention(got[[p[0] for p in pairs], [p[1] for p in pairs]], want)


# ---------------------------------------------------------------------------
# full-size workloads, sampled outputs
# ---------------------------------------------------------------------------

def _sample_tokens(rng, lens, Hkv, n):
    out = []
    for _ in range(n):
        s = int(rng.integers(0, len(lens)))
        out.append((s, int(rng.integers(0, lens[s])), int(rng.integers(0, Hkv))))
    return out


@pytest.fixture(scope="module")
def qwen32k():
    wl = W.WORKLOADS["qwen3_8b_32k"]
    c = Cache(wl)
    for g0 in range(0, wl.batch, 4):
        c.append_range(range(g0, g0 + 4), 0, wl.ctx)
    return c


def test_qwen32k_codes_sampled(qwen32k):
    c = qwen32k
    rng = np.random.default_rng(21)
    samples = _sample_tokens(rng, [c.wl.ctx] * c.wl.batch, 8, 1500)
    samples += [(0, 0, 0), (15, 32767, 7), (3, 16, 2), (9, 32752, 5)]
    Ktok, Vtok = _block_fn(c.wl, 0)
    near = compare_codes(c, c.pool_host(), samples, Ktok, Vtok)
    assert_boundary_count(near, len(samples), "qwen32k")
    assert c.status() == 0


def test_qwen32k_decode_sampled(qwen32k):
    c = qwen32k
    q = W.queries(c.wl)
    lens = [c.wl.ctx] * c.wl.batch
    got = c.decode(q, lens, 0)          # the automatic split choice, as the bench runs it
    rng = np.random.default_rng(22)
    pairs = [[int(rng.integers(0, 16)), int(rng.integers(0, 32))] for _ in range(12)]
    pairs += [[0, 0], [15, 31]]
    want = c.oracle_decode(c.pool_host(), q, lens, pairs)
    assert_close_attention(got[[p[0] for p in pairs], [p[1] for p in pairs]], want, "qwen32k")


def test_qwen32k_window_decode_sampled(qwen32k):
    """The OptR setting at full size: 64 sink + 256 recent tokens from a BF16
    cache that holds the window pages only, the rest from the INT2 cache, the
    automatic split choice."""
    c = qwen32k
    sink, recent = 64, 256
    lens = [c.wl.ctx] * c.wl.batch
    pt, npool = window_page_table(lens, c.pt_np.shape[1], sink, recent)
    cb = Cache(c.wl, kind="bf16", page_table=pt, num_pool_pages=npool)
    pos = np.array(window_positions(c.wl.ctx, sink, recent), np.int32)
    assert len(pos) == sink + recent
    for b in range(c.wl.batch):
        Kw = np.concatenate([W.tokens(c.wl, 0, b, 0, 0, sink),
                             W.tokens(c.wl, 0, b, 0, c.wl.ctx - recent, recent)])
        Vw = np.concatenate([W.tokens(c.wl, 0, b, 1, 0, sink),
                             W.tokens(c.wl, 0, b, 1, c.wl.ctx - recent, recent)])
        cb.append(Kw, Vw, np.full(len(pos), b), pos)
    q = W.queries(c.wl, 0, 2)
    got = window_decode(c, cb, q, lens, sink, recent, 0)
    rng = np.random.default_rng(25)
    pairs = [[int(rng.integers(0, 16)), int(rng.integers(0, 32))] for _ in range(8)]
    pairs += [[0, 0], [15, 31]]
    want = oracle_window(c, cb, q, lens, pairs, sink, recent)
    assert_close_attention(got[[p[0] for p in pairs], [p[1] for p in pairs]], want, "window 32k")
    assert c.status() == 0 and cb.status() == 0


@pytest.mark.parametrize("splits", [64, 128, 256])
def test_long_128k_decode(splits, long128k):
    c = long128k
    q = W.queries(c.wl, 0, splits)
    got = c.decode(q, [c.wl.ctx], splits)
    pairs = [[0, h] for h in (0, 7, 13, 22, 31)]
    want = c.oracle_decode(c.pool_host(), q, [c.wl.ctx], pairs)
    assert_close_attention(got[0, [p[1] for p in pairs]], want, f"128k splits {splits}")


@pytest.fixture(scope="module")
def long128k():
    wl = W.WORKLOADS["long_128k"]
    c = Cache(wl)
    for s0 in range(0, wl.ctx, 32768):
        c.append_range([0], s0, 32768)
    return c


def test_ragged_batch_decode():
    wl = W.WORKLOADS["ragged_64"]
    c = Cache(wl)
    lens = W.seq_lens(wl)
    for g0 in range(0, wl.batch, 8):
        c.append_range(range(g0, g0 + 8), 0, [int(x) for x in lens[g0:g0 + 8]])
    q = W.queries(wl)
    got = c.decode(q, lens, 0)
    rng = np.random.default_rng(23)
    pairs = [[int(b), int(rng.integers(0, 32))] for b in
             [int(np.argmax(lens)), int(np.argmin(lens))] + list(rng.integers(0, 64, 8))]
    want = c.oracle_decode(c.pool_host(), q, lens, pairs)
    assert_close_attention(got[[p[0] for p in pairs], [p[1] for p in pairs]], want, "ragged")
    Ktok, Vtok = _block_fn(wl, 0)
    near = compare_codes(c, c.pool_host(), _sample_tokens(rng, lens, 8, 400), Ktok, Vtok)
    assert_boundary_count(near, 400, "ragged")
    assert c.status() == 0


@pytest.mark.parametrize("layer", [0, 17, 35])
def test_full_stack_sampled_layers(layer):
    """Prefill 8192 tokens per sequence for batch 8, then 128 decode steps, each
    appending one token and decoding; outputs checked at steps 0, 63, 127."""
    wl = W.WORKLOADS["full_stack_36l"]
    c = Cache(wl, layer=layer)
    c.append_range(range(wl.batch), 0, wl.prefill)
    B = wl.batch
    Knew = W.tokens_many(wl, layer, range(B), 0, wl.prefill, wl.decode_steps)
    Vnew = W.tokens_many(wl, layer, range(B), 1, wl.prefill, wl.decode_steps)
    checked = 0
    for step in range(wl.decode_steps):
        pos = wl.prefill + step
        c.append(np.stack([Knew[b][step] for b in range(B)]), np.stack([Vnew[b][step] for b in range(B)]),
                 np.arange(B), np.full(B, pos))
        q = W.queries(wl, layer, step)
        lens = [pos + 1] * B
        got = c.decode(q, lens, 0)
        if step in (0, 63, 127):
            pairs = [[b, (7 * b + step) % 32] for b in range(B)]
            want = c.oracle_decode(c.pool_host(), q, lens, pairs)
            assert_close_attention(got[[p[0] for p in pairs], [p[1] for p in pairs]], want,
                                   f"layer {layer} step {step}")
            checked += 1
    assert checked == 3
    Ktok, Vtok = _block_fn(wl, layer)
    rng = np.random.default_rng(24 + layer)
    near = compare_codes(c, c.pool_host(), _sample_tokens(rng, [wl.prefill + 128] * B, 8, 300),
                         Ktok, Vtok)
    assert_boundary_count(near, 300, f"full stack layer {layer}")
    assert c.status() == 0


@pytest.mark.parametrize("out_rotated,G,splits", [(True, 4, 3), (False, 2, 0)])
def test_small_combine_large_batch(out_rotated, G, splits):
    """More (sequence, KV head) pairs than one wave of one-per-SM KV-head
    combine CTAs: the combine in 256-thread CTAs (four per SM, R_V^T read from
    global memory), checked on every (sequence, head) output against the
    oracle.  Odd batch, plain and rotated-basis output, G = 2 (half of each
    CTA's head warps idle), an empty sequence (output 0)."""
    wl = W.WORKLOADS["ragged_64"]
    B, Hkv = 21, 8
    pt, _ = W.page_table(wl)
    pt = pt[:B].copy()
    c = Cache(wl, out_rotated=out_rotated, page_table=pt, num_pool_pages=int(pt.max()) + 1,
              num_heads=Hkv * G, num_kv_heads=Hkv)
    rng = np.random.default_rng(40 + G)
    lens = rng.integers(1, 400, size=B)
    lens[3], lens[B - 1] = 0, 77
    lens = np.minimum(lens, (pt >= 0).sum(axis=1) * 16)
    c.append_range(range(B), 0, [int(x) for x in lens])
    q = W.queries(wl, 0, 70)[:B, :Hkv * G].copy()
    got = c.decode(q, lens, splits)
    assert c.status() == 0
    assert np.all(got[3] == 0.0)
    pairs = [[b, h] for b in range(B) if lens[b] > 0 for h in range(Hkv * G)]
    want = c.oracle_decode(c.pool_host(), q, lens, pairs)
    assert_close_attention(got[[p[0] for p in pairs], [p[1] for p in pairs]], want,
                           f"small-CTA combine, out_rotated={out_rotated}, G={G}")
