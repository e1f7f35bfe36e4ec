"""Helpers shared by the GPU tests: build a cache on the device through the
C ABI from a seeded workload, read it back, and compare with the oracle."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from rotated_int2_kv_kvq_gb300 import kvq as K
from rotated_int2_kv_kvq_gb300 import workloads as W

D = 128


def u16(a: np.ndarray) -> torch.Tensor:
    """uint16 numpy -> int16 CUDA tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


class Cache:
    """One layer of one workload on the device: handle, pool, page table."""

    def __init__(self, wl: W.Workload, layer: int = 0, kind: str = "int2", out_rotated=False,
                 page_table=None, num_pool_pages=None, num_heads=None, num_kv_heads=None,
                 q_rotated=False):
        self.wl, self.layer, self.kind = wl, layer, kind
        self.H = num_heads or wl.num_heads
        self.Hkv = num_kv_heads or wl.num_kv_heads
        self.layout = K.make_layout(self.H, self.Hkv, wl.clip_k, wl.clip_v, 0.0, out_rotated,
                                    q_rotated=q_rotated)
        self.h = K.kvq_create(self.layout)
        if page_table is None:
            page_table, num_pool_pages = W.page_table(wl, layer)
        self.pt_np = np.ascontiguousarray(page_table, np.int32)
        self.npool = int(num_pool_pages)
        self.pt = i32(self.pt_np)
        rec = K.INT2_RECORD_BYTES if kind == "int2" else K.BF16_RECORD_BYTES
        self.rec = rec
        self.pool = torch.zeros(self.npool * self.Hkv * rec, dtype=torch.uint8, device="cuda")
        self.R = W.rotations(wl, layer)[:, :self.Hkv].copy()
        self.mu = W.key_mean(wl, layer)[:self.Hkv].copy()
        if kind == "int2":
            K.kvq_set_rotation(self.h, torch.from_numpy(self.R).cuda(),
                               torch.from_numpy(self.mu).cuda())

    # -- append ------------------------------------------------------------------
    def append(self, Kt: np.ndarray, Vt: np.ndarray, seq_idx, positions):
        fn = K.kvq_append if self.kind == "int2" else K.kvq_bf16_append
        fn(self.h, self.pool, self.npool, u16(Kt), u16(Vt), i32(seq_idx), i32(positions), self.pt)

    def append_range(self, seqs, start, n, layer=None):
        """Append positions [start, start+n) of each sequence in `seqs` (n may be
        per sequence).  Returns (Kt, Vt) lists of the appended host tokens."""
        layer = self.layer if layer is None else layer
        seqs = list(seqs)
        nn = n if hasattr(n, "__len__") else [n] * len(seqs)
        st = start if hasattr(start, "__len__") else [start] * len(seqs)
        Ks = W.tokens_many(self.wl, layer, seqs, 0, st, nn)
        Vs = W.tokens_many(self.wl, layer, seqs, 1, st, nn)
        for s, k, v, a, m in zip(seqs, Ks, Vs, st, nn):
            if m == 0:
                continue
            self.append(k[:, :self.Hkv].copy(), v[:, :self.Hkv].copy(), np.full(m, s, np.int32),
                        np.arange(a, a + m, dtype=np.int32))
        return Ks, Vs

    # -- decode ------------------------------------------------------------------
    def decode(self, q_np: np.ndarray, seq_lens, num_splits=0):
        B = self.pt_np.shape[0]
        out = torch.empty((B, self.H, D), dtype=torch.float32, device="cuda")
        if self.kind == "int2":
            ws = torch.empty(K.kvq_workspace_bytes(self.h, B, num_splits), dtype=torch.uint8,
                             device="cuda")
            K.kvq_decode(self.h, self.pool, self.npool, u16(q_np), self.pt, i32(seq_lens), out, ws,
                         num_splits)
        else:
            ws = torch.empty(K.kvq_bf16_workspace_bytes(self.h, B, num_splits),
                             dtype=torch.uint8, device="cuda")
            K.kvq_bf16_decode(self.h, self.pool, self.npool, u16(q_np), self.pt, i32(seq_lens),
                              out, ws, num_splits)
        torch.cuda.synchronize()
        return out.cpu().numpy().astype(np.float64)

    def pool_host(self) -> np.ndarray:
        torch.cuda.synchronize()
        return self.pool.cpu().numpy()

    def status(self) -> int:
        return K.kvq_get_status(self.h)

    def oracle_decode(self, pool_np, q_np, seq_lens, pairs):
        return oracle.decode_pairs(self.kind, pool_np, self.npool, self.H, self.Hkv, q_np,
                                   self.pt_np, seq_lens, pairs, R=self.R,
                                   out_rotated=bool(self.layout.flags & K.KVQ_OUT_ROTATED))


def rel_l2(a, b) -> float:
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    n = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (n if n > 0 else 1.0))


# Tolerances of the decode attention outputs against the float64 oracle run on
# the same dequantised cache: 1e-3 relative L2 and 5e-3 max-abs per
# (sequence, head) output vector.
REL_L2_TOL = 1e-3
MAX_ABS_TOL = 5e-3


def assert_close_attention(got, want, what=""):
    got, want = np.asarray(got), np.asarray(want)
    assert got.shape == want.shape
    for i in range(got.shape[0]):
        r = rel_l2(got[i], want[i])
        m = float(np.abs(got[i] - want[i]).max())
        assert r <= REL_L2_TOL and m <= MAX_ABS_TOL, f"{what} row {i}: rel_l2 {r:.3g} max_abs {m:.3g}"


def compare_codes(cache: Cache, pool_np: np.ndarray, samples, Ktok, Vtok):
    """Check the GPU pool's bytes for sampled (seq, pos, kv) against the oracle
    quantiser.  Ktok/Vtok: callables (seq, pos) -> bf16 [Hkv, D].  Returns the
    number of code mismatches that sit within 1 ulp of a rounding boundary
    (allowed); raises on any other difference."""
    recs = pool_np.reshape(cache.npool, cache.Hkv, K.INT2_RECORD_BYTES)
    near = 0
    for (s, p, kv) in samples:
        page = cache.pt_np[s, p // 16]
        rec = recs[page, kv]
        for which, x, R, mu, clip in [
                (0, Ktok(s, p)[kv], cache.R[0, kv], cache.mu[kv], cache.wl.clip_k),
                (1, Vtok(s, p)[kv], cache.R[1, kv], None, cache.wl.clip_v)]:
            c, s16, z16, r, t = oracle.quantize(x, R, clip, mu=mu)
            c2, s2, z2 = oracle.int2_load(rec, which, p % 16)
            assert (s16, z16) == (s2, z2), (s, p, kv, which, hex(s16), hex(s2), hex(z16), hex(z2))
            bad = np.nonzero(c != c2)[0]
            for i in bad:
                frac = abs(float(t[i]) - math.floor(float(t[i])) - 0.5)
                assert frac <= np.spacing(np.float32(t[i])), (s, p, kv, which, i, t[i], c[i], c2[i])
                near += 1
    return near


# Code disagreements allowed where the oracle's pre-rounding value lies within
# 1 ulp of a k + 1/2 boundary.  With the fixed fp32 operation order on both
# sides none are expected; a test fails if more than this fraction of the
# codes it checked sit in that band.
BOUNDARY_FRACTION = 1e-4


def assert_boundary_count(near, checked_token_heads, what=""):
    """Report the boundary-case count (pytest -rP, or -s, shows it) and bound it:
    each token-head holds 2 x 128 codes."""
    codes = 2 * 128 * checked_token_heads
    print(f"{what} boundary-case code differences: {near} of {codes} codes")
    assert near <= BOUNDARY_FRACTION * codes, (what, near, codes)


# ---- BF16 sink + recent window ---------------------------------------------------

def window_page_table(lens, max_pages, sink, recent):
    """A BF16 page table that maps only the pages holding a window position
    (p < sink or p >= len - recent) of each sequence; other entries are -1.
    Returns (table int32 [B, max_pages], num_pool_pages)."""
    pt = np.full((len(lens), max_pages), -1, np.int32)
    n = 0
    for b, L in enumerate(lens):
        for pg in range((int(L) + 15) // 16):
            first, last = 16 * pg, min(16 * pg + 16, int(L)) - 1
            if first < sink or last >= int(L) - recent:
                pt[b, pg] = n
                n += 1
    return pt, max(n, 1)


def window_positions(L, sink, recent):
    return [p for p in range(int(L)) if p < sink or p >= int(L) - recent]


def window_decode(ci: Cache, cb: Cache, q_np, seq_lens, sink, recent, num_splits=0):
    """kvq_decode_window over INT2 cache `ci` and BF16 cache `cb`."""
    B = ci.pt_np.shape[0]
    out = torch.empty((B, ci.H, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(K.kvq_workspace_bytes(ci.h, B, num_splits), dtype=torch.uint8, device="cuda")
    K.kvq_decode_window(ci.h, ci.pool, ci.npool, cb.pool, cb.npool, cb.pt, u16(q_np), ci.pt,
                        i32(seq_lens), int(sink), int(recent), out, ws, num_splits)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def oracle_window(ci: Cache, cb: Cache, q_np, seq_lens, pairs, sink, recent):
    return oracle.decode_window_pairs(
        ci.pool_host(), ci.npool, cb.pool_host(), cb.npool, cb.pt_np, ci.H, ci.Hkv, q_np,
        ci.pt_np, seq_lens, pairs, sink, recent, ci.R, ci.mu,
        out_rotated=bool(ci.layout.flags & K.KVQ_OUT_ROTATED))
