"""CPU checks of the C-ABI library: it builds, loads, exports every entry point
include/kvq.h declares, and its host-only paths behave (no GPU needed: nothing
here launches a kernel or allocates device memory)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def lib():
    from rotated_int2_kv_kvq_gb300 import build, kvq

    if not os.path.exists(kvq.LIB_PATH):
        build.build()
    return kvq.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["kvq_create", "kvq_destroy", "kvq_set_rotation", "kvq_append", "kvq_decode",
              "kvq_dequant", "kvq_workspace_bytes", "kvq_get_status", "kvq_strerror",
              "kvq_bf16_append", "kvq_bf16_decode"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from rotated_int2_kv_kvq_gb300 import kvq

    out = subprocess.run(["nm", "-D", "--defined-only", kvq.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (kvq_\w+)$", out, flags=re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    # and the binding covers exactly the declared entry points
    assert sorted(kvq.SIGNATURES) == declared_functions()


def test_layout_struct_matches_header(lib):
    from rotated_int2_kv_kvq_gb300 import kvq

    assert ctypes.sizeof(kvq.KvqLayout) == 9 * 4
    text = open(HEADER).read()
    for name, value in [("KVQ_OK", 0), ("KVQ_EINVAL", 1), ("KVQ_ENOSPACE", 2), ("KVQ_ECUDA", 3),
                        ("KVQ_ENOTREADY", 4), ("KVQ_INT2_RECORD_BYTES", 1152),
                        ("KVQ_BF16_RECORD_BYTES", 8192), ("KVQ_OUT_ROTATED", 1),
                        ("KVQ_Q_ROTATED", 2)]:
        m = re.search(r"#define\s+%s\s+(\d+)" % name, text)
        assert m and int(m.group(1)) == value


def test_host_only_paths(lib):
    from rotated_int2_kv_kvq_gb300 import kvq

    assert lib.kvq_strerror(0) == b"ok"
    for c in range(-1, 6):
        assert lib.kvq_strerror(c)
    assert lib.kvq_page_bytes(None) == 0
    assert lib.kvq_workspace_bytes(None, 4, 0) == 0
    assert lib.kvq_auto_splits(None, 4, 10) == 0
    assert lib.kvq_destroy(None) == 0
    out = ctypes.c_void_p()
    assert lib.kvq_create(None, ctypes.byref(out)) == kvq.KVQ_EINVAL
    # unsupported layouts are rejected on the host, before any CUDA call
    for bad in [kvq.make_layout(32, 8, head_dim=64), kvq.make_layout(32, 8, group=32),
                kvq.make_layout(32, 8, page_size=8), kvq.make_layout(64, 8),
                kvq.make_layout(30, 8), kvq.make_layout(32, 8, clip_k=-1.0),
                kvq.make_layout(32, 8, clip_v=0.0), kvq.make_layout(32, 0)]:
        assert lib.kvq_create(ctypes.byref(bad), ctypes.byref(out)) == kvq.KVQ_EINVAL
        assert not out.value
    assert lib.kvq_create(ctypes.byref(kvq.make_layout(32, 8)), None) == kvq.KVQ_EINVAL
    # null handles are argument errors
    assert lib.kvq_append(None, None, 0, None, None, None, None, 1, None, 1, 1, None) == 1
    assert lib.kvq_decode(None, None, 0, None, None, 0, None, 0, None, None, 0, 0, None) == 1
    assert lib.kvq_get_status(None, None, None) == 1
    assert lib.kvq_append_decode(None, None, 0, None, None, None, None, 0, None, 0, None, None, 0,
                                 0, None) == 1
    assert lib.kvq_decode_window(None, None, 0, None, 0, None, None, None, 0, None, 0, 64, 256,
                                 None, None, 0, 0, None) == 1
    assert lib.kvq_append_decode_window(None, None, 0, None, 0, None, None, None, None, None, 0,
                                        None, 0, 64, 256, None, None, 0, 0, None) == 1
    # a layout with both folding flags is valid; an unknown flag is not
    both = kvq.make_layout(32, 8, out_rotated=True, q_rotated=True)
    assert both.flags == kvq.KVQ_OUT_ROTATED | kvq.KVQ_Q_ROTATED
    bad = kvq.make_layout(32, 8)
    bad.flags = 4
    assert lib.kvq_create(ctypes.byref(bad), ctypes.byref(out)) == kvq.KVQ_EINVAL
