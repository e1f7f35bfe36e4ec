"""Rotated INT2 KV cache for GB300 (sm_103a).

- ``rotated_int2_kv_kvq_gb300.kvq``: the Python binding of libkvq.so, the C ABI
  declared in ``include/kvq.h`` (quantise-on-append, split-K INT2 decode
  attention, the BF16 comparison cache, dequantisation for tests).
- ``rotated_int2_kv_kvq_gb300.workloads``: seeded synthetic inputs.
- ``rotated_int2_kv_kvq_gb300.build``: builds libkvq.so in-tree with nvcc.
"""
