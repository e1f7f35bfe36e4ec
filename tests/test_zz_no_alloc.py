"""kvq_decode_static: the decode step for callers that cannot allocate a
workspace (an attention-op signature without a workspace argument, or a
process that forbids device allocation on the decode path).  It must give the
same output as kvq_decode with a caller-allocated workspace, call after call,
while the library's fixed scratch array is reused.  This file is collected last
so that a run stopping at the first failure has run every other test first."""
import numpy as np
import pytest
import torch

from kvq_testlib import Cache, i32, u16
from rotated_int2_kv_kvq_gb300 import kvq as K
from rotated_int2_kv_kvq_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _static(c, q_np, lens, splits):
    B = c.pt_np.shape[0]
    out = torch.empty((B, c.H, 128), dtype=torch.float32, device="cuda")
    K.kvq_decode_static(c.h, c.pool, c.npool, u16(q_np), c.pt, i32(lens), out, splits)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("splits", [0, 3])
def test_static_decode_matches_workspace_decode(splits):
    wl = W.WORKLOADS["qwen3_8b_32k"]
    B, L = 4, 2000
    pt, _ = W.page_table(wl)
    pt = pt[:B].copy()
    c = Cache(wl, page_table=pt, num_pool_pages=int(pt.max()) + 1)
    c.append_range(range(B), 0, L)
    if splits == 0:
        # the automatic split count's scratch fits the fixed array, so both
        # calls run the same kernels on the same split count
        auto = K.kvq_auto_splits(c.h, B, pt.shape[1])
        assert K.kvq_workspace_bytes(c.h, B, auto) <= 16 << 20
    for call in range(2):                    # two calls in a row share the array
        q = W.queries(wl, 0, 100 + call, batch=B)
        lens = [L - 37 * call] * B
        want = c.decode(q, lens, splits)
        got = _static(c, q, lens, splits)
        for b in range(B):
            assert np.array_equal(got[b], want[b]), (call, b, np.abs(got[b] - want[b]).max())
    assert c.status() == 0


def test_static_decode_rejects_oversized_scratch():
    wl = W.WORKLOADS["tiny_1k"]
    c = Cache(wl)
    big_batch = 4000
    pt = torch.zeros((big_batch, 4), dtype=torch.int32, device="cuda")
    out = torch.empty((big_batch, 4, 128), dtype=torch.float32, device="cuda")
    q = torch.zeros((big_batch, 4, 128), dtype=torch.int16, device="cuda")
    with pytest.raises(K.KvqError) as e:
        K.kvq_decode_static(c.h, c.pool, c.npool, q, pt,
                            torch.zeros(big_batch, dtype=torch.int32, device="cuda"), out, 1024)
    assert e.value.code == K.KVQ_ENOSPACE
