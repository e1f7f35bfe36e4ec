"""Thin Python binding of libkvq.so (include/kvq.h).

Argument marshalling only: every function forwards to the C entry point of the
same name, passing device pointers of torch CUDA tensors and the current CUDA
stream.  Every step of the hot path runs in the library's kernels; there is no
CPU fallback.  If libkvq.so is missing the import fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

KVQ_OK, KVQ_EINVAL, KVQ_ENOSPACE, KVQ_ECUDA, KVQ_ENOTREADY = 0, 1, 2, 3, 4
KVQ_STATUS_BAD_PAGE = 1
KVQ_STATUS_BAD_POS = 2
KVQ_STATUS_BAD_SEQLEN = 4
KVQ_STATUS_BAD_SEQ = 8
KVQ_STATUS_TIMEOUT = 16
KVQ_OUT_ROTATED = 1
KVQ_Q_ROTATED = 2
INT2_RECORD_BYTES = 1152
BF16_RECORD_BYTES = 8192

# Every entry point of include/kvq.h, with its ctypes signature.
_P, _I, _SZ, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
SIGNATURES = {
    "kvq_create": ([_P, _P], _I),
    "kvq_destroy": ([_P], _I),
    "kvq_page_bytes": ([_P], _SZ),
    "kvq_bf16_page_bytes": ([_P], _SZ),
    "kvq_set_rotation": ([_P, _P, _P, _P], _I),
    "kvq_append": ([_P, _P, _I, _P, _P, _P, _P, _I, _P, _I, _I, _P], _I),
    "kvq_workspace_bytes": ([_P, _I, _I], _SZ),
    "kvq_decode": ([_P, _P, _I, _P, _P, _I, _P, _I, _P, _P, _SZ, _I, _P], _I),
    "kvq_dequant": ([_P, _P, _I, _P, _I, _I, _I, _I, _P, _P, _P], _I),
    "kvq_bf16_append": ([_P, _P, _I, _P, _P, _P, _P, _I, _P, _I, _I, _P], _I),
    "kvq_bf16_workspace_bytes": ([_P, _I, _I], _SZ),
    "kvq_bf16_decode": ([_P, _P, _I, _P, _P, _I, _P, _I, _P, _P, _SZ, _I, _P], _I),
    "kvq_decode_static": ([_P, _P, _I, _P, _P, _I, _P, _I, _P, _I, _P], _I),
    "kvq_optr_workspace_bytes": ([_I, _I, _I, _I, _I], _SZ),
    "kvq_optr_calibrate": ([_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _F, _F, _F, _F, _I, _F, _P,
                            _P, _P, _SZ, _P], _I),
    "kvq_optr_loss_grad": ([_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _F, _F, _F, _F, _P, _P, _I,
                            _P, _P, _P, _SZ, _P], _I),
    "kvq_append_decode": ([_P, _P, _I, _P, _P, _P, _P, _I, _P, _I, _P, _P, _SZ, _I, _P], _I),
    "kvq_decode_window": ([_P, _P, _I, _P, _I, _P, _P, _P, _I, _P, _I, _I, _I, _P, _P, _SZ, _I,
                           _P], _I),
    "kvq_append_decode_window": ([_P, _P, _I, _P, _I, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _P,
                                  _P, _SZ, _I, _P], _I),
    "kvq_get_status": ([_P, _P, _P], _I),
    "kvq_selftest_wait_timeout": ([_P, _I, _P], _I),
    "kvq_auto_splits": ([_P, _I, _I], _I),
    "kvq_profile_enable": ([_P, _I], _I),
    "kvq_profile_read": ([_P, _P, _P], _I),
    "kvq_strerror": ([_I], ctypes.c_char_p),
}


class KvqLayout(ctypes.Structure):
    _fields_ = [("num_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("group", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("clip_k", ctypes.c_float),
                ("clip_v", ctypes.c_float), ("sm_scale", ctypes.c_float),
                ("flags", ctypes.c_uint32)]


class KvqError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {code} ({strerror(code)})")
        self.code = code


_lib = None


def load_library():
    """Load libkvq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def strerror(code: int) -> str:
    return load_library().kvq_strerror(int(code)).decode()


def _check(fn, rc):
    if rc != KVQ_OK:
        raise KvqError(fn, rc)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t, dtypes, name):
    """Device pointer of a contiguous CUDA tensor of one of `dtypes` (None -> NULL)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


_BF16 = (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (
    torch.bfloat16, torch.int16)
_U8 = (torch.uint8,)
_I32 = (torch.int32,)
_F32 = (torch.float32,)


class Handle:
    """Owns a kvq_handle*; destroyed with the object."""

    def __init__(self, ptr: int, layout: KvqLayout):
        self.ptr = ctypes.c_void_p(ptr)
        self.layout = layout

    def __del__(self):
        if getattr(self, "ptr", None) and self.ptr.value and _lib is not None:
            _lib.kvq_destroy(self.ptr)
            self.ptr = ctypes.c_void_p(0)

    @property
    def _as_parameter_(self):
        return self.ptr


def make_layout(num_heads, num_kv_heads, clip_k=0.96, clip_v=0.92, sm_scale=0.0,
                out_rotated=False, head_dim=128, group=128, page_size=16,
                q_rotated=False) -> KvqLayout:
    flags = (KVQ_OUT_ROTATED if out_rotated else 0) | (KVQ_Q_ROTATED if q_rotated else 0)
    return KvqLayout(num_heads, num_kv_heads, head_dim, group, page_size, clip_k, clip_v,
                     sm_scale, flags)


# ---- entry points (same names as the C ABI) ------------------------------------

def kvq_create(layout: KvqLayout) -> Handle:
    out = ctypes.c_void_p()
    _check("kvq_create", load_library().kvq_create(ctypes.byref(layout), ctypes.byref(out)))
    return Handle(out.value, layout)


def kvq_destroy(h: Handle) -> None:
    _check("kvq_destroy", load_library().kvq_destroy(h.ptr))
    h.ptr = ctypes.c_void_p(0)


def kvq_page_bytes(h: Handle) -> int:
    return int(load_library().kvq_page_bytes(h.ptr))


def kvq_bf16_page_bytes(h: Handle) -> int:
    return int(load_library().kvq_bf16_page_bytes(h.ptr))


def kvq_set_rotation(h: Handle, R: torch.Tensor, mu: torch.Tensor, stream=None) -> None:
    _check("kvq_set_rotation", load_library().kvq_set_rotation(
        h.ptr, _ptr(R, _F32, "R"), _ptr(mu, _F32, "mu"), _stream(stream)))


def _append(fn, h, pool, num_pool_pages, K, V, seq_idx, positions, page_table, stream):
    n = int(K.shape[0])
    batch, max_pages = int(page_table.shape[0]), int(page_table.shape[1])
    _check(fn, getattr(load_library(), fn)(
        h.ptr, _ptr(pool, _U8, "pool"), int(num_pool_pages), _ptr(K, _BF16, "K"),
        _ptr(V, _BF16, "V"), _ptr(seq_idx, _I32, "seq_idx"), _ptr(positions, _I32, "positions"),
        n, _ptr(page_table, _I32, "page_table"), batch, max_pages, _stream(stream)))


def kvq_append(h, pool, num_pool_pages, K, V, seq_idx, positions, page_table, stream=None):
    """K, V: [n, Hkv, 128] bf16; seq_idx, positions: int32 [n]; page_table: int32 [B, P]."""
    _append("kvq_append", h, pool, num_pool_pages, K, V, seq_idx, positions, page_table, stream)


def kvq_bf16_append(h, pool, num_pool_pages, K, V, seq_idx, positions, page_table, stream=None):
    _append("kvq_bf16_append", h, pool, num_pool_pages, K, V, seq_idx, positions, page_table,
            stream)


def kvq_workspace_bytes(h: Handle, batch: int, num_splits: int = 0) -> int:
    return int(load_library().kvq_workspace_bytes(h.ptr, int(batch), int(num_splits)))


def kvq_bf16_workspace_bytes(h: Handle, batch: int, num_splits: int = 0) -> int:
    return int(load_library().kvq_bf16_workspace_bytes(h.ptr, int(batch), int(num_splits)))


def kvq_auto_splits(h: Handle, batch: int, max_pages: int) -> int:
    return int(load_library().kvq_auto_splits(h.ptr, int(batch), int(max_pages)))


def _decode(fn, h, pool, num_pool_pages, q, page_table, seq_lens, out, workspace, num_splits,
            stream):
    batch, max_pages = int(page_table.shape[0]), int(page_table.shape[1])
    _check(fn, getattr(load_library(), fn)(
        h.ptr, _ptr(pool, _U8, "pool"), int(num_pool_pages), _ptr(q, _BF16, "q"),
        _ptr(page_table, _I32, "page_table"), max_pages, _ptr(seq_lens, _I32, "seq_lens"),
        batch, _ptr(out, _F32, "out"), _ptr(workspace, _U8, "workspace"),
        int(workspace.numel()), int(num_splits), _stream(stream)))


def kvq_decode(h, pool, num_pool_pages, q, page_table, seq_lens, out, workspace, num_splits=0,
               stream=None):
    """q: [B, H, 128] bf16; out: [B, H, 128] fp32; workspace: uint8, >= kvq_workspace_bytes."""
    _decode("kvq_decode", h, pool, num_pool_pages, q, page_table, seq_lens, out, workspace,
            num_splits, stream)


def kvq_bf16_decode(h, pool, num_pool_pages, q, page_table, seq_lens, out, workspace,
                    num_splits=0, stream=None):
    _decode("kvq_bf16_decode", h, pool, num_pool_pages, q, page_table, seq_lens, out, workspace,
            num_splits, stream)


def kvq_decode_static(h, pool, num_pool_pages, q, page_table, seq_lens, out, num_splits=0,
                      stream=None):
    """kvq_decode with the library's fixed 16 MiB scratch array instead of a
    caller-supplied workspace (for callers that cannot allocate one)."""
    batch, max_pages = int(page_table.shape[0]), int(page_table.shape[1])
    _check("kvq_decode_static", load_library().kvq_decode_static(
        h.ptr, _ptr(pool, _U8, "pool"), int(num_pool_pages), _ptr(q, _BF16, "q"),
        _ptr(page_table, _I32, "page_table"), max_pages, _ptr(seq_lens, _I32, "seq_lens"),
        batch, _ptr(out, _F32, "out"), int(num_splits), _stream(stream)))


def kvq_append_decode(h, pool, num_pool_pages, K_new, V_new, q, page_table, seq_lens, out,
                      workspace, num_splits=0, stream=None):
    """One decode step: append K_new[b], V_new[b] ([B, Hkv, 128] bf16) at
    position seq_lens[b] - 1 of every sequence, then decode (as kvq_decode)."""
    batch, max_pages = int(page_table.shape[0]), int(page_table.shape[1])
    _check("kvq_append_decode", load_library().kvq_append_decode(
        h.ptr, _ptr(pool, _U8, "pool"), int(num_pool_pages), _ptr(K_new, _BF16, "K_new"),
        _ptr(V_new, _BF16, "V_new"), _ptr(q, _BF16, "q"), _ptr(page_table, _I32, "page_table"),
        max_pages, _ptr(seq_lens, _I32, "seq_lens"), batch, _ptr(out, _F32, "out"),
        _ptr(workspace, _U8, "workspace"), int(workspace.numel()), int(num_splits),
        _stream(stream)))


def kvq_decode_window(h, pool, num_pool_pages, bf16_pool, bf16_num_pool_pages, bf16_page_table,
                      q, page_table, seq_lens, sink, recent, out, workspace, num_splits=0,
                      stream=None):
    """Decode with a BF16 window: positions < sink and >= len - recent from the
    BF16 cache (bf16_page_table: int32 [B, P], same shape as page_table), the
    others from the INT2 cache, in one softmax.  Workspace as for kvq_decode."""
    batch, max_pages = int(page_table.shape[0]), int(page_table.shape[1])
    if tuple(bf16_page_table.shape) != (batch, max_pages):
        raise ValueError("bf16_page_table must have the shape of page_table")
    _check("kvq_decode_window", load_library().kvq_decode_window(
        h.ptr, _ptr(pool, _U8, "pool"), int(num_pool_pages), _ptr(bf16_pool, _U8, "bf16_pool"),
        int(bf16_num_pool_pages), _ptr(bf16_page_table, _I32, "bf16_page_table"),
        _ptr(q, _BF16, "q"), _ptr(page_table, _I32, "page_table"), max_pages,
        _ptr(seq_lens, _I32, "seq_lens"), batch, int(sink), int(recent), _ptr(out, _F32, "out"),
        _ptr(workspace, _U8, "workspace"), int(workspace.numel()), int(num_splits),
        _stream(stream)))


def kvq_append_decode_window(h, pool, num_pool_pages, bf16_pool, bf16_num_pool_pages,
                             bf16_page_table, K_new, V_new, q, page_table, seq_lens, sink, recent,
                             out, workspace, num_splits=0, stream=None):
    """One windowed decode step: append K_new[b], V_new[b] ([B, Hkv, 128] bf16) at
    position seq_lens[b] - 1 to the INT2 and the BF16 cache, then decode as
    kvq_decode_window."""
    batch, max_pages = int(page_table.shape[0]), int(page_table.shape[1])
    if tuple(bf16_page_table.shape) != (batch, max_pages):
        raise ValueError("bf16_page_table must have the shape of page_table")
    _check("kvq_append_decode_window", load_library().kvq_append_decode_window(
        h.ptr, _ptr(pool, _U8, "pool"), int(num_pool_pages), _ptr(bf16_pool, _U8, "bf16_pool"),
        int(bf16_num_pool_pages), _ptr(bf16_page_table, _I32, "bf16_page_table"),
        _ptr(K_new, _BF16, "K_new"), _ptr(V_new, _BF16, "V_new"), _ptr(q, _BF16, "q"),
        _ptr(page_table, _I32, "page_table"), max_pages, _ptr(seq_lens, _I32, "seq_lens"), batch,
        int(sink), int(recent), _ptr(out, _F32, "out"), _ptr(workspace, _U8, "workspace"),
        int(workspace.numel()), int(num_splits), _stream(stream)))


def kvq_dequant(h, pool, num_pool_pages, page_table, seq, start, length, K_out=None, V_out=None,
                stream=None):
    _check("kvq_dequant", load_library().kvq_dequant(
        h.ptr, _ptr(pool, _U8, "pool"), int(num_pool_pages), _ptr(page_table, _I32, "page_table"),
        int(page_table.shape[1]), int(seq), int(start), int(length), _ptr(K_out, _F32, "K_out"),
        _ptr(V_out, _F32, "V_out"), _stream(stream)))


def kvq_get_status(h: Handle, stream=None) -> int:
    bits = ctypes.c_uint32()
    _check("kvq_get_status", load_library().kvq_get_status(h.ptr, ctypes.byref(bits),
                                                           _stream(stream)))
    return int(bits.value)


def kvq_selftest_wait_timeout(h: Handle, limit_us: int, stream=None) -> None:
    _check("kvq_selftest_wait_timeout",
           load_library().kvq_selftest_wait_timeout(h.ptr, int(limit_us), _stream(stream)))


def kvq_profile_enable(h: Handle, enable: bool = True) -> None:
    _check("kvq_profile_enable", load_library().kvq_profile_enable(h.ptr, 1 if enable else 0))


def kvq_profile_read(h: Handle):
    """(total milliseconds of the split-K attention kernel, launches) since enable."""
    ms = ctypes.c_double()
    n = ctypes.c_int()
    _check("kvq_profile_read", load_library().kvq_profile_read(h.ptr, ctypes.byref(ms),
                                                               ctypes.byref(n)))
    return float(ms.value), int(n.value)


def kvq_optr_workspace_bytes(num_kv_heads, T, Nq, G, Dm) -> int:
    return int(load_library().kvq_optr_workspace_bytes(int(num_kv_heads), int(T), int(Nq), int(G),
                                                       int(Dm)))


def kvq_optr_calibrate(K, V, Q, W_O, R0, mu, clip_k, clip_v, lambda_k=1.0, lr=1e-3, steps=80,
                       sm_scale=0.0, workspace=None, stream=None):
    """OptR calibration of the key and value rotations of every KV head.
    K, V: bf16 [Hkv, T, 128]; Q: bf16 [Hkv, Nq, G, 128]; W_O: fp32 [Hkv, Dm, G*128];
    R0: fp32 [2, Hkv, 128, 128]; mu: fp32 [Hkv, 128].  Returns (R fp32
    [2, Hkv, 128, 128], history fp32 [2, steps + 1, Hkv]) as CUDA tensors."""
    Hkv, T = int(K.shape[0]), int(K.shape[1])
    Nq, G, Dm = int(Q.shape[1]), int(Q.shape[2]), int(W_O.shape[1])
    R = torch.empty((2, Hkv, 128, 128), dtype=torch.float32, device=K.device)
    hist = torch.empty((2, int(steps) + 1, Hkv), dtype=torch.float32, device=K.device)
    if workspace is None:
        workspace = torch.empty(kvq_optr_workspace_bytes(Hkv, T, Nq, G, Dm), dtype=torch.uint8,
                                device=K.device)
    _check("kvq_optr_calibrate", load_library().kvq_optr_calibrate(
        Hkv, T, Nq, G, Dm, _ptr(K, _BF16, "K"), _ptr(V, _BF16, "V"), _ptr(Q, _BF16, "Q"),
        _ptr(W_O, _F32, "W_O"), _ptr(R0, _F32, "R0"), _ptr(mu, _F32, "mu"), float(clip_k),
        float(clip_v), float(lambda_k), float(lr), int(steps), float(sm_scale), _ptr(R, _F32, "R"),
        _ptr(hist, _F32, "history"), _ptr(workspace, _U8, "workspace"), int(workspace.numel()),
        _stream(stream)))
    return R, hist


def kvq_optr_loss_grad(K, V, Q, W_O, R0, mu, clip_k, clip_v, A_key, A_value=None, which=0,
                       lambda_k=1.0, sm_scale=0.0, workspace=None, stream=None):
    """Loss [Hkv] and d loss / dA [Hkv, 128, 128] of the key (which = 0) or value
    (which = 1) calibration objective, as CUDA tensors."""
    Hkv, T = int(K.shape[0]), int(K.shape[1])
    Nq, G, Dm = int(Q.shape[1]), int(Q.shape[2]), int(W_O.shape[1])
    loss = torch.empty(Hkv, dtype=torch.float32, device=K.device)
    grad = torch.empty((Hkv, 128, 128), dtype=torch.float32, device=K.device)
    if workspace is None:
        workspace = torch.empty(kvq_optr_workspace_bytes(Hkv, T, Nq, G, Dm), dtype=torch.uint8,
                                device=K.device)
    _check("kvq_optr_loss_grad", load_library().kvq_optr_loss_grad(
        Hkv, T, Nq, G, Dm, _ptr(K, _BF16, "K"), _ptr(V, _BF16, "V"), _ptr(Q, _BF16, "Q"),
        _ptr(W_O, _F32, "W_O"), _ptr(R0, _F32, "R0"), _ptr(mu, _F32, "mu"), float(clip_k),
        float(clip_v), float(lambda_k), float(sm_scale), _ptr(A_key, _F32, "A_key"),
        _ptr(A_value, _F32, "A_value"), int(which), _ptr(loss, _F32, "loss"),
        _ptr(grad, _F32, "grad"), _ptr(workspace, _U8, "workspace"), int(workspace.numel()),
        _stream(stream)))
    return loss, grad


def kvq_strerror(code: int) -> str:
    return strerror(code)
