"""GPU tests of the BF16 comparison cache and of the error paths of the C ABI.

Error paths are made on the host (bad arguments) or with bad data that the
kernels check themselves (page ids outside the pool, positions beyond the page
table, seq_len beyond capacity): they must report a status bit, skip the bad
item and leave the GPU usable.  Nothing here faults or hangs the GPU.
"""
import numpy as np
import pytest
import torch

import oracle
from kvq_testlib import Cache, assert_close_attention, i32, u16
from rotated_int2_kv_kvq_gb300 import kvq as K
from rotated_int2_kv_kvq_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_bf16_append_bytes_and_decode():
    wl = W.WORKLOADS["tiny_1k"]
    c = Cache(wl, kind="bf16")
    Ks, Vs = c.append_range([0], 0, wl.ctx)
    pool = c.pool_host()
    ref = np.zeros_like(pool)
    oracle.append_bf16(ref, c.npool, 1, Ks[0], Vs[0], np.zeros(wl.ctx), np.arange(wl.ctx), c.pt_np)
    assert np.array_equal(pool, ref)
    for L, splits in [(1024, 0), (17, 1), (500, 7)]:
        q = W.queries(wl, 0, L)
        got = c.decode(q, [L], splits)
        want = c.oracle_decode(pool, q, [L], [[0, h] for h in range(4)])
        assert_close_attention(got[0], want, f"bf16 len {L}")


def test_bf16_qwen_shape():
    wl = W.WORKLOADS["qwen3_8b_32k"]
    B, L = 4, 3000
    pt, _ = W.page_table(wl)
    pt = pt[:B].copy()
    c = Cache(wl, kind="bf16", page_table=pt, num_pool_pages=int(pt.max()) + 1)
    c.append_range(range(B), 0, L)
    q = W.queries(wl, 0, 0, batch=B)
    got = c.decode(q, [L] * B, 0)
    pairs = [[b, h] for b in range(B) for h in (0, 9, 31)]
    want = c.oracle_decode(c.pool_host(), q, [L] * B, pairs)
    assert_close_attention(got[[p[0] for p in pairs], [p[1] for p in pairs]], want, "bf16 qwen")


def test_bf16_qwen_full_context():
    """The BF16 comparison kernel at the full 32K context of two sequences."""
    wl = W.WORKLOADS["qwen3_8b_32k"]
    B = 2
    pt, _ = W.page_table(wl)
    pt = pt[:B].copy()
    c = Cache(wl, kind="bf16", page_table=pt, num_pool_pages=int(pt.max()) + 1)
    for s0 in range(0, wl.ctx, 8192):
        c.append_range(range(B), s0, 8192)
    q = W.queries(wl, 0, 3, batch=B)
    lens = [wl.ctx, wl.ctx - 5]
    got = c.decode(q, lens, 0)
    pairs = [[b, h] for b in range(B) for h in (0, 13, 31)]
    want = c.oracle_decode(c.pool_host(), q, lens, pairs)
    assert_close_attention(got[[p[0] for p in pairs], [p[1] for p in pairs]], want, "bf16 32k")
    assert c.status() == 0


def test_host_argument_errors():
    wl = W.WORKLOADS["tiny_1k"]
    lay = K.make_layout(4, 1)
    bad = [K.make_layout(4, 1, head_dim=64), K.make_layout(4, 1, group=64),
           K.make_layout(4, 1, page_size=32), K.make_layout(8, 1), K.make_layout(6, 4),
           K.make_layout(4, 1, clip_k=0.0), K.make_layout(4, 1, clip_v=1.5)]
    for b in bad:
        with pytest.raises(K.KvqError) as e:
            K.kvq_create(b)
        assert e.value.code == K.KVQ_EINVAL
    h = K.kvq_create(lay)
    pt = i32(np.zeros((1, 4)))
    pool = torch.zeros(4 * 1152, dtype=torch.uint8, device="cuda")
    Kt = u16(W.tokens(wl, 0, 0, 0, 0, 3))
    # before the rotation bank is set
    with pytest.raises(K.KvqError) as e:
        K.kvq_append(h, pool, 4, Kt, Kt, i32([0, 0, 0]), i32([0, 1, 2]), pt)
    assert e.value.code == K.KVQ_ENOTREADY
    K.kvq_set_rotation(h, torch.from_numpy(W.rotations(wl)).cuda(),
                       torch.from_numpy(W.key_mean(wl)).cuda())
    out = torch.empty((1, 4, 128), dtype=torch.float32, device="cuda")
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(K.KvqError) as e:
        K.kvq_decode(h, pool, 4, u16(W.queries(wl)), pt, i32([3]), out, small, 2)
    assert e.value.code == K.KVQ_ENOSPACE
    ws = torch.empty(K.kvq_workspace_bytes(h, 1, 2), dtype=torch.uint8, device="cuda")
    with pytest.raises(K.KvqError) as e:
        K.kvq_decode(h, pool, 0, u16(W.queries(wl)), pt, i32([3]), out, ws, 2)
    assert e.value.code == K.KVQ_EINVAL
    with pytest.raises(K.KvqError) as e:
        K.kvq_decode(h, pool, 4, u16(W.queries(wl)), pt, i32([3]), out, ws, 5000)
    assert e.value.code == K.KVQ_EINVAL
    # misaligned workspace
    with pytest.raises(K.KvqError) as e:
        K.kvq_decode(h, pool, 4, u16(W.queries(wl)), pt, i32([3]), out, ws[8:], 2)
    assert e.value.code == K.KVQ_EINVAL
    assert K.kvq_get_status(h) == 0


def test_device_data_errors_are_reported_and_skipped():
    wl = W.WORKLOADS["tiny_1k"]
    pt, npool = W.page_table(wl)
    c = Cache(wl)
    n = 40
    Kt, Vt = W.tokens(wl, 0, 0, 0, 0, n), W.tokens(wl, 0, 0, 1, 0, n)
    seqs = np.zeros(n, np.int32)
    pos = np.arange(n, dtype=np.int32)
    seqs[5] = 3                 # no such sequence
    pos[6] = 64 * 16 + 2        # beyond the page table
    pos[7] = -1
    c.append(Kt, Vt, seqs, pos)
    bits = c.status()
    assert bits & K.KVQ_STATUS_BAD_SEQ and bits & K.KVQ_STATUS_BAD_POS
    assert c.status() == 0      # read clears
    # the good tokens were written exactly as the oracle writes them
    ref = np.zeros_like(c.pool_host())
    oracle.append_int2(ref, c.npool, 1, Kt, Vt, seqs, pos, c.pt_np, c.R, c.mu, wl.clip_k, wl.clip_v)
    assert np.array_equal(c.pool_host(), ref)
    # a page table entry outside the pool: append and decode skip it
    bad_pt = c.pt_np.copy()
    bad_pt[0, 1] = npool + 100
    c2 = Cache(wl, page_table=bad_pt, num_pool_pages=npool)
    c2.append(Kt[:32], Vt[:32], np.zeros(32), np.arange(32))
    assert c2.status() & K.KVQ_STATUS_BAD_PAGE
    q = W.queries(wl)
    got = c2.decode(q, [32], 2)
    assert c2.status() & K.KVQ_STATUS_BAD_PAGE
    # decode over the good page only equals decode of a 16-token context
    want = c2.oracle_decode(c2.pool_host(), q, [16], [[0, h] for h in range(4)])
    assert_close_attention(got[0], want, "bad page skipped")
    # seq_len beyond capacity: reported, treated as empty
    got = c.decode(q, [64 * 16 + 1], 2)
    assert c.status() & K.KVQ_STATUS_BAD_SEQLEN and not np.any(got)
    # the context is still usable
    got = c.decode(q, [33], 2)
    assert c.status() == 0


def test_bounded_wait_gives_up_and_leaves_the_gpu_usable():
    """A wait that nothing completes runs out after its limit, sets
    KVQ_STATUS_TIMEOUT and returns; the next decode on the same stream is
    correct and reports no error."""
    import time
    wl = W.WORKLOADS["tiny_1k"]
    c = Cache(wl)
    c.append_range([0], 0, 200)
    assert c.status() == 0
    t0 = time.perf_counter()
    K.kvq_selftest_wait_timeout(c.h, 2000)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 1.0
    assert c.status() == K.KVQ_STATUS_TIMEOUT
    assert c.status() == 0                        # reading clears the word
    q = W.queries(wl, 0, 77)
    got = c.decode(q, [200], 2)
    want = c.oracle_decode(c.pool_host(), q, [200], [[0, h] for h in range(4)])
    assert_close_attention(got[0], want, "after a timed-out wait")
    assert c.status() == 0
    with pytest.raises(K.KvqError) as e:
        K.kvq_selftest_wait_timeout(c.h, 0)
    assert e.value.code == K.KVQ_EINVAL
