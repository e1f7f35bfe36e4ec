"""CPU oracle of the rotated INT2 KV-cache hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product (``rotated_int2_kv_kvq_gb300``) never imports it, and
the two share no code: this wrapper only marshals numpy arrays into
``kvq_oracle.c``, which restates the method from its description on
"Output-Aware Rotation for INT2 KV-Cache Quantization" (pith.science review of
arXiv 2608.02691): key centring, per-head rotation, clipping, grouping and
rounding ("What carries the argument"; clip ratios from "Assumptions & free
parameters"), dequantisation and float64 attention, inverse value rotation.

Build: ``oracle/build_oracle.py`` (called by ``__graft_entry__.build()``)
compiles ``kvq_oracle.c`` with gcc into ``oracle/libkvq_oracle.so``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq_oracle.so")

PAGE = 16
DIM = 128
INT2_RECORD_BYTES = 1152
BF16_RECORD_BYTES = 8192

_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        from . import build_oracle

        build_oracle.build()
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    i32 = ctypes.c_int
    f32 = ctypes.c_float
    f64 = ctypes.c_double
    lib.kvqo_f16_to_f32.argtypes = [ctypes.c_uint16]
    lib.kvqo_f16_to_f32.restype = f32
    lib.kvqo_f32_to_f16.argtypes = [f32]
    lib.kvqo_f32_to_f16.restype = ctypes.c_uint16
    lib.kvqo_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.kvqo_bf16_to_f32.restype = f32
    lib.kvqo_quantize.argtypes = [P, P, P, i32, f32, P, P, P, P, P]
    lib.kvqo_quantize.restype = None
    lib.kvqo_int2_locate.argtypes = [i32, i32, i32, P, P]
    lib.kvqo_int2_locate.restype = None
    lib.kvqo_int2_meta_offset.argtypes = [i32, i32]
    lib.kvqo_int2_meta_offset.restype = i32
    lib.kvqo_int2_store.argtypes = [P, i32, i32, P, ctypes.c_uint16, ctypes.c_uint16]
    lib.kvqo_int2_store.restype = None
    lib.kvqo_int2_load.argtypes = [P, i32, i32, P, P, P]
    lib.kvqo_int2_load.restype = None
    lib.kvqo_bf16_locate.argtypes = [i32, i32, i32]
    lib.kvqo_bf16_locate.restype = i32
    lib.kvqo_append_int2.argtypes = [P, i32, i32, P, P, P, P, i32, P, i32, i32, P, P, f32, f32]
    lib.kvqo_append_int2.restype = i32
    lib.kvqo_append_bf16.argtypes = [P, i32, i32, P, P, P, P, i32, P, i32, i32]
    lib.kvqo_append_bf16.restype = i32
    lib.kvqo_dequant_int2.argtypes = [P, i32, i32, P, i32, i32, i32, i32, P, P]
    lib.kvqo_dequant_int2.restype = i32
    lib.kvqo_rotate_f64.argtypes = [P, P, i32, P]
    lib.kvqo_rotate_f64.restype = None
    lib.kvqo_rotate_t_f64.argtypes = [P, P, i32, P]
    lib.kvqo_rotate_t_f64.restype = None
    lib.kvqo_attend_f64.argtypes = [P, P, P, i32, i32, f64, P]
    lib.kvqo_attend_f64.restype = None
    lib.kvqo_decode_pairs.argtypes = [i32, P, i32, i32, i32, P, P, i32, P, P, i32, P, f64, i32, P]
    lib.kvqo_decode_pairs.restype = i32
    lib.kvqo_decode_window_pairs.argtypes = [P, i32, P, i32, P, i32, i32, P, P, i32, P, P, i32,
                                             i32, i32, P, P, f64, i32, P]
    lib.kvqo_decode_window_pairs.restype = i32
    _lib = lib
    return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- number formats --------------------------------------------------------

def f32_to_f16_bits(x: float) -> int:
    """binary32 -> binary16 bit pattern, round to nearest even."""
    return int(_load().kvqo_f32_to_f16(float(np.float32(x))))


def f16_bits_to_f32(h: int) -> float:
    return float(_load().kvqo_f16_to_f32(int(h)))


def bf16_bits_to_f32(b: int) -> float:
    return float(_load().kvqo_bf16_to_f32(int(b)))


# ---- quantiser ----------------------------------------------------------------

def quantize(x_bf16, R, clip, mu=None):
    """Quantise one vector (bf16 bit patterns, uint16 [D]) with rotation R
    (fp32 [D, D], row-vector convention) and key mean mu (fp32 [D] or None for
    values).  Returns (codes uint8 [D], s16, z16, r fp32 [D], t fp32 [D])."""
    lib = _load()
    x = _c(x_bf16, np.uint16)
    D = x.shape[0]
    Rm = _c(R, np.float32)
    assert Rm.shape == (D, D)
    m = None if mu is None else _c(mu, np.float32)
    codes = np.zeros(D, np.uint8)
    s16 = np.zeros(1, np.uint16)
    z16 = np.zeros(1, np.uint16)
    r = np.zeros(D, np.float32)
    t = np.zeros(D, np.float32)
    lib.kvqo_quantize(_p(x), _p(m), _p(Rm), D, float(np.float32(clip)), _p(codes), _p(s16),
                      _p(z16), _p(r), _p(t))
    return codes, int(s16[0]), int(z16[0]), r, t


# ---- page records ---------------------------------------------------------------

def int2_locate(which: int, tau: int, d: int):
    """(byte offset, bit shift) of the code of (slot tau, element d)."""
    lib = _load()
    byte = ctypes.c_int()
    shift = ctypes.c_int()
    lib.kvqo_int2_locate(which, tau, d, ctypes.byref(byte), ctypes.byref(shift))
    return byte.value, shift.value


def int2_meta_offset(which: int, tau: int) -> int:
    return int(_load().kvqo_int2_meta_offset(which, tau))


def int2_store(rec, which, tau, codes, s16, z16):
    assert rec.dtype == np.uint8 and rec.flags.c_contiguous and rec.size == INT2_RECORD_BYTES
    c = _c(codes, np.uint8)
    _load().kvqo_int2_store(_p(rec), which, tau, _p(c), int(s16), int(z16))


def int2_load(rec, which, tau):
    rec = _c(rec, np.uint8)
    codes = np.zeros(DIM, np.uint8)
    s16 = np.zeros(1, np.uint16)
    z16 = np.zeros(1, np.uint16)
    _load().kvqo_int2_load(_p(rec), which, tau, _p(codes), _p(s16), _p(z16))
    return codes, int(s16[0]), int(z16[0])


def bf16_locate(which: int, tau: int, d: int) -> int:
    return int(_load().kvqo_bf16_locate(which, tau, d))


# ---- append / dequant / decode -------------------------------------------------

def append_int2(pool, num_pool_pages, Hkv, K, V, seq_idx, positions, page_table, R, mu,
                clip_k, clip_v):
    """Quantise tokens into ``pool`` (uint8, modified in place).
    K, V: uint16 [n, Hkv, D]; R: fp32 [2, Hkv, D, D]; mu: fp32 [Hkv, D].
    Returns the number of skipped tokens."""
    assert pool.dtype == np.uint8 and pool.flags.c_contiguous
    K = _c(K, np.uint16)
    V = _c(V, np.uint16)
    si = _c(seq_idx, np.int32)
    ps = _c(positions, np.int32)
    pt = _c(page_table, np.int32)
    Rm = _c(R, np.float32)
    m = _c(mu, np.float32)
    return int(_load().kvqo_append_int2(_p(pool), num_pool_pages, Hkv, _p(K), _p(V), _p(si),
                                        _p(ps), K.shape[0], _p(pt), pt.shape[0], pt.shape[1],
                                        _p(Rm), _p(m), float(np.float32(clip_k)),
                                        float(np.float32(clip_v))))


def append_bf16(pool, num_pool_pages, Hkv, K, V, seq_idx, positions, page_table):
    assert pool.dtype == np.uint8 and pool.flags.c_contiguous
    K = _c(K, np.uint16)
    V = _c(V, np.uint16)
    si = _c(seq_idx, np.int32)
    ps = _c(positions, np.int32)
    pt = _c(page_table, np.int32)
    return int(_load().kvqo_append_bf16(_p(pool), num_pool_pages, Hkv, _p(K), _p(V), _p(si),
                                        _p(ps), K.shape[0], _p(pt), pt.shape[0], pt.shape[1]))


def dequant_int2(pool, num_pool_pages, Hkv, page_table, b, start, length):
    """fp32 [length, Hkv, D] keys and values, rotated basis, fmaf(code, s, z)."""
    pool = _c(pool, np.uint8)
    pt = _c(page_table, np.int32)
    Ko = np.zeros((length, Hkv, DIM), np.float32)
    Vo = np.zeros((length, Hkv, DIM), np.float32)
    _load().kvqo_dequant_int2(_p(pool), num_pool_pages, Hkv, _p(pt), pt.shape[1], b, start,
                              length, _p(Ko), _p(Vo))
    return Ko, Vo


def rotate_f64(x, M):
    x = _c(x, np.float64)
    Mm = _c(M, np.float32)
    y = np.zeros_like(x)
    _load().kvqo_rotate_f64(_p(x), _p(Mm), x.shape[0], _p(y))
    return y


def rotate_t_f64(x, M):
    x = _c(x, np.float64)
    Mm = _c(M, np.float32)
    y = np.zeros_like(x)
    _load().kvqo_rotate_t_f64(_p(x), _p(Mm), x.shape[0], _p(y))
    return y


def attend_f64(q, keys, values, scale):
    q = _c(q, np.float64)
    k = _c(keys, np.float64)
    v = _c(values, np.float64)
    T, D = k.shape
    out = np.zeros(D, np.float64)
    _load().kvqo_attend_f64(_p(q), _p(k), _p(v), T, D, float(scale), _p(out))
    return out


def decode_pairs(kind, pool, num_pool_pages, H, Hkv, q, page_table, seq_lens, pairs, R=None,
                 sm_scale=None, out_rotated=False):
    """Decode the listed (b, hq) pairs in float64.  kind: 'int2' or 'bf16'.
    q: uint16 [batch, H, D]; pairs: int [npairs, 2].  Returns float64 [npairs, D]."""
    pool = _c(pool, np.uint8)
    q = _c(q, np.uint16)
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32)
    pr = _c(pairs, np.int32).reshape(-1, 2)
    Rm = None if R is None else _c(R, np.float32)
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(DIM)
    out = np.zeros((pr.shape[0], DIM), np.float64)
    _load().kvqo_decode_pairs(0 if kind == "int2" else 1, _p(pool), num_pool_pages, H, Hkv,
                              _p(q), _p(pt), pt.shape[1], _p(sl), _p(pr), pr.shape[0], _p(Rm),
                              float(sm_scale), 1 if out_rotated else 0, _p(out))
    return out


def decode_window_pairs(pool, num_pool_pages, bf16_pool, bf16_num_pool_pages, bf16_page_table, H,
                        Hkv, q, page_table, seq_lens, pairs, sink, recent, R, mu, sm_scale=None,
                        out_rotated=False):
    """Decode (b, hq) pairs with a BF16 window of `sink` first and `recent` last
    tokens over an INT2 cache; float64 [npairs, D]."""
    pool = _c(pool, np.uint8)
    bp = _c(bf16_pool, np.uint8)
    bpt = _c(bf16_page_table, np.int32)
    q = _c(q, np.uint16)
    pt = _c(page_table, np.int32)
    assert bpt.shape == pt.shape
    sl = _c(seq_lens, np.int32)
    pr = _c(pairs, np.int32).reshape(-1, 2)
    Rm = _c(R, np.float32)
    m = _c(mu, np.float32)
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(DIM)
    out = np.zeros((pr.shape[0], DIM), np.float64)
    _load().kvqo_decode_window_pairs(_p(pool), num_pool_pages, _p(bp), bf16_num_pool_pages,
                                     _p(bpt), H, Hkv, _p(q), _p(pt), pt.shape[1], _p(sl), _p(pr),
                                     pr.shape[0], int(sink), int(recent), _p(Rm), _p(m),
                                     float(sm_scale), 1 if out_rotated else 0, _p(out))
    return out
