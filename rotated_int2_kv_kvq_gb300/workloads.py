"""Seeded synthetic workloads for the rotated INT2 KV-cache path.

This module only draws inputs: keys, values, queries, the calibration
stand-ins (rotation R and key mean mu), page tables and sequence lengths.  It
holds none of the method's arithmetic (no centring, rotation of data,
quantisation or attention), so the CUDA path and the CPU oracle can both take
their inputs from it.

Every array is a pure function of (workload seed, layer, sequence, block): any
token range can be regenerated on its own, so a check can look at a sample of
a workload without generating all of it.

The shapes follow the serving setting of "Output-Aware Rotation for INT2
KV-Cache Quantization" (pith.science review of arXiv 2608.02691): Qwen3-8B
(32 query heads, 8 KV heads, head_dim 128; "Core claim"), contexts up to 128K
("If this is right", second item), a paged cache ("If this is right", third
item).  The pages give no data distribution; the recipe is:

* keys: per (layer, KV head, channel) an offset ~ N(0, 4) (variance 4, std 2);
  per token noise ~ N(0, 1).  Four channels per head are outliers:
  - ``gauss_x8`` (tiny workload): the whole channel (offset + noise) times 8;
  - ``student_t`` (the others): offset + 8 * Student-t(3) noise.
* values: N(0, 1).  queries: N(0, 1).  All rounded to bf16 (nearest even).
* R: per (layer, K|V, KV head) the Q factor of a QR decomposition of a seeded
  Gaussian matrix, with the signs of diag(R_qr) folded in (Haar-distributed
  orthogonal), stored fp32.  It stands in for the calibrated rotation
  R0 exp(A - A^T) ("Core claim"), which needs model traces.
* mu: the float64 per-channel mean of a separate 4096-token calibration draw
  of keys from the same distribution, stored fp32 (the pages estimate mu from
  calibration traces: "Load-bearing premise").
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

D = 128
PAGE = 16
_BLOCK = 1024          # tokens per independently seeded block
_CALIB_TOKENS = 4096
_N_OUTLIERS = 4


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    batch: int
    num_heads: int
    num_kv_heads: int
    ctx: int                      # context per sequence (max for ragged)
    key_kind: str                 # "gauss_x8" or "student_t"
    clip_k: float
    clip_v: float
    layers: int = 1
    ragged: bool = False          # lengths log-uniform in [min_ctx, ctx]
    min_ctx: int = 0
    prefill: int = 0              # full-stack: tokens appended before decoding
    decode_steps: int = 0         # full-stack: decode steps per layer
    splits: tuple = field(default=())   # split counts the workload exercises
    description: str = ""


# The five synthetic workloads.  Clip ratios: the tiny workload states 0.95;
# the others use the pages' c_K = 0.96, c_V = 0.92 ("Assumptions & free
# parameters").
WORKLOADS = {
    "tiny_1k": Workload(
        "tiny_1k", 1001, batch=1, num_heads=4, num_kv_heads=1, ctx=1024,
        key_kind="gauss_x8", clip_k=0.95, clip_v=0.95,
        description="1 sequence, 1 KV head / 4 query heads, ctx 1024, shuffled 64-page pool"),
    "qwen3_8b_32k": Workload(
        "qwen3_8b_32k", 1002, batch=16, num_heads=32, num_kv_heads=8, ctx=32768,
        key_kind="student_t", clip_k=0.96, clip_v=0.92,
        description="Qwen3-8B-shaped layer, batch 16, ctx 32768, shuffled pool of 32768 pages"),
    "long_128k": Workload(
        "long_128k", 1003, batch=1, num_heads=32, num_kv_heads=8, ctx=131072,
        key_kind="student_t", clip_k=0.96, clip_v=0.92, splits=(64, 128, 256),
        description="batch 1, ctx 131072, split-K over 64-256 chunks"),
    "ragged_64": Workload(
        "ragged_64", 1004, batch=64, num_heads=32, num_kv_heads=8, ctx=65536,
        key_kind="student_t", clip_k=0.96, clip_v=0.92, ragged=True, min_ctx=1024,
        description="64 sequences, lengths log-uniform in [1024, 65536], shared shuffled pool"),
    "full_stack_36l": Workload(
        "full_stack_36l", 1005, batch=8, num_heads=32, num_kv_heads=8, ctx=8192 + 128,
        key_kind="student_t", clip_k=0.96, clip_v=0.92, layers=36, prefill=8192,
        decode_steps=128,
        description="36 layers, batch 8: append an 8192-token prefill, then 128 decode steps"),
}


def _rng(*key) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


def to_bf16_bits(x) -> np.ndarray:
    """float array -> bf16 bit patterns (uint16), round to nearest even (finite
    and infinite inputs; no NaNs are generated)."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32)
    u = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (u >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_float(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ---- calibration stand-ins ------------------------------------------------------

def rotations(wl: Workload, layer: int = 0) -> np.ndarray:
    """fp32 [2, Hkv, D, D]: key rotations then value rotations (row-vector
    convention, r = x R)."""
    out = np.empty((2, wl.num_kv_heads, D, D), np.float32)
    for which in range(2):
        for kv in range(wl.num_kv_heads):
            g = _rng(wl.seed, 7, layer, which, kv).standard_normal((D, D))
            q, r = np.linalg.qr(g)
            q = q * np.sign(np.diag(r))[None, :]
            out[which, kv] = q.astype(np.float32)
    return out


def _key_params(wl: Workload, layer: int):
    g = _rng(wl.seed, 3, layer)
    offsets = g.normal(0.0, 2.0, size=(wl.num_kv_heads, D))
    outliers = np.stack([g.choice(D, _N_OUTLIERS, replace=False)
                         for _ in range(wl.num_kv_heads)])
    return offsets, outliers


def _draw_keys(wl: Workload, layer: int, g: np.random.Generator, n: int) -> np.ndarray:
    """float32 [n, Hkv, D] keys (before bf16 rounding)."""
    offsets, outliers = _key_params(wl, layer)
    k = g.standard_normal((n, wl.num_kv_heads, D), dtype=np.float32)
    k += offsets.astype(np.float32)[None]
    for kv in range(wl.num_kv_heads):
        ch = outliers[kv]
        if wl.key_kind == "gauss_x8":
            k[:, kv, ch] *= np.float32(8.0)
        else:
            t = g.standard_t(3, size=(n, len(ch)))
            k[:, kv, ch] = (offsets[kv, ch][None] + 8.0 * t).astype(np.float32)
    return k


def key_mean(wl: Workload, layer: int = 0) -> np.ndarray:
    """fp32 [Hkv, D]: per-channel mean of a calibration draw of bf16 keys."""
    k = _draw_keys(wl, layer, _rng(wl.seed, 5, layer), _CALIB_TOKENS)
    kb = bf16_bits_to_float(to_bf16_bits(k)).astype(np.float64)
    return kb.mean(axis=0).astype(np.float32)


# ---- tokens ---------------------------------------------------------------------

def _block(wl: Workload, layer: int, seq: int, which: int, blk: int) -> np.ndarray:
    g = _rng(wl.seed, 11, layer, seq, which, blk)
    if which == 0:
        x = _draw_keys(wl, layer, g, _BLOCK)
    else:
        x = g.standard_normal((_BLOCK, wl.num_kv_heads, D), dtype=np.float32)
    return to_bf16_bits(x)


def tokens(wl: Workload, layer: int, seq: int, which: int, start: int, n: int) -> np.ndarray:
    """bf16 bits [n, Hkv, D] of keys (which=0) or values (which=1) of sequence
    ``seq`` at positions [start, start + n)."""
    out = np.empty((n, wl.num_kv_heads, D), np.uint16)
    pos = start
    while pos < start + n:
        blk = pos // _BLOCK
        off = pos - blk * _BLOCK
        take = min(_BLOCK - off, start + n - pos)
        out[pos - start:pos - start + take] = _block(wl, layer, seq, which, blk)[off:off + take]
        pos += take
    return out


def tokens_many(wl: Workload, layer: int, seqs, which: int, start, n, workers: int = 8):
    """[len(seqs)] arrays of tokens(), drawn in parallel threads (numpy releases
    the GIL while drawing).  start and n may be scalars or per-sequence lists."""
    from concurrent.futures import ThreadPoolExecutor

    seqs = list(seqs)
    st = start if hasattr(start, "__len__") else [start] * len(seqs)
    nn = n if hasattr(n, "__len__") else [n] * len(seqs)
    with ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(lambda i: tokens(wl, layer, seqs[i], which, int(st[i]), int(nn[i])),
                           range(len(seqs))))


def token_at(wl: Workload, layer: int, seq: int, which: int, pos: int) -> np.ndarray:
    return tokens(wl, layer, seq, which, pos, 1)[0]


def queries(wl: Workload, layer: int = 0, step: int = 0, batch: int | None = None) -> np.ndarray:
    """bf16 bits [batch, H, D], N(0, 1)."""
    b = wl.batch if batch is None else batch
    g = _rng(wl.seed, 13, layer, step)
    return to_bf16_bits(g.standard_normal((b, wl.num_heads, D), dtype=np.float32))


# ---- sequence lengths and page tables ---------------------------------------------

def seq_lens(wl: Workload) -> np.ndarray:
    """int32 [batch]: context length of each sequence (before any decode step)."""
    if not wl.ragged:
        return np.full(wl.batch, wl.prefill if wl.prefill else wl.ctx, np.int32)
    g = _rng(wl.seed, 17)
    u = g.uniform(math.log(wl.min_ctx), math.log(wl.ctx), size=wl.batch)
    return np.floor(np.exp(u)).astype(np.int32)


def capacity(wl: Workload) -> np.ndarray:
    """int32 [batch]: positions each sequence's page table must cover."""
    if wl.prefill:
        return np.full(wl.batch, wl.prefill + wl.decode_steps, np.int32)
    if wl.ragged:
        return seq_lens(wl) + 1            # one decode token per step
    return np.full(wl.batch, wl.ctx, np.int32)


def page_table(wl: Workload, layer: int = 0):
    """(page_table int32 [batch, max_pages], num_pool_pages).  Each sequence
    gets ceil(capacity / 16) pages drawn from one shuffled pool; unused table
    entries are -1."""
    cap = capacity(wl)
    pages = (cap + PAGE - 1) // PAGE
    num_pool = int(pages.sum())
    max_pages = int(pages.max())
    perm = _rng(wl.seed, 19, layer).permutation(num_pool).astype(np.int32)
    pt = np.full((wl.batch, max_pages), -1, np.int32)
    o = 0
    for b in range(wl.batch):
        pt[b, :pages[b]] = perm[o:o + pages[b]]
        o += pages[b]
    return pt, num_pool


def cache_bytes_per_token_head(kind: str = "int2") -> int:
    """Algorithmic bytes of one token of one KV head: INT2 codes of K and V
    (2 x 32 B) plus fp16 scale/zero (2 x 4 B); BF16: 2 x 256 B."""
    return 72 if kind == "int2" else 512


def effective_bits(group: int = 128) -> float:
    """Bits per cached element: 2-bit code plus two fp16 per group."""
    return 2.0 + 32.0 / group


def effective_bits_window(ctx: int, sink: int = 64, recent: int = 256, group: int = 128) -> float:
    """Bits per cached element of a context of `ctx` tokens whose first `sink`
    and last `recent` tokens stay in BF16 (16 bits) and the rest in INT2 with
    fp16 scale/zero per group (the OptR accounting, "Assumptions & free
    parameters" of the OptR page)."""
    n16 = min(ctx, sink + recent)
    return ((ctx - n16) * effective_bits(group) + n16 * 16.0) / ctx


# ---- calibration traces (rotation calibration) -----------------------------------

def calibration_traces(wl: Workload, layer: int = 0, T: int = 4096, Nq: int = 64,
                       Dm: int = 4096, heads=None, seq: int = 0):
    """Synthetic calibration chunk of one sequence for the KV heads `heads`
    (default all): keys and values at positions [0, T) (the token recipe above),
    the queries of the last Nq positions (N(0, 1), bf16) and a Gaussian stand-in
    for the KV head's slice of the output projection, N(0, 1/(H*D)).
    Returns (K bits [Hs, T, D], V bits [Hs, T, D], Q bits [Hs, Nq, G, D],
    W_O fp32 [Hs, Dm, G*D])."""
    heads = list(range(wl.num_kv_heads)) if heads is None else list(heads)
    G = wl.num_heads // wl.num_kv_heads
    Kt = tokens(wl, layer, seq, 0, 0, T)
    Vt = tokens(wl, layer, seq, 1, 0, T)
    g = _rng(wl.seed, 23, layer, seq)
    q = to_bf16_bits(g.standard_normal((Nq, wl.num_heads, D), dtype=np.float32))
    w = g.standard_normal((wl.num_kv_heads, Dm, G * D), dtype=np.float32) / np.float32(
        np.sqrt(wl.num_heads * D))
    K = np.ascontiguousarray(Kt[:, heads].transpose(1, 0, 2))
    V = np.ascontiguousarray(Vt[:, heads].transpose(1, 0, 2))
    Q = np.ascontiguousarray(np.stack([q[:, h * G:(h + 1) * G] for h in heads]))
    return K, V, Q, np.ascontiguousarray(w[heads])
