"""Compile the CPU oracle (kvq_oracle.c) into oracle/libkvq_oracle.so.

Test infrastructure: called by ``__graft_entry__.build()`` and, lazily, by the
oracle wrapper.  ``-ffp-contract=off`` keeps gcc from fusing multiply-adds that
the oracle writes as separate operations (it fuses by default on aarch64)."""
import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))


def build(verbose: bool = False) -> str:
    src = os.path.join(_HERE, "kvq_oracle.c")
    out = os.path.join(_HERE, "libkvq_oracle.so")
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", tmp, src, "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose=True))
