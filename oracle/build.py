"""Build step of the CPU oracle (test infrastructure, not product code).

Compiles ``zero_oracle.c`` and ``gen_oracle.c`` into ``oracle/_build/liboracle.so``
with gcc, ``-O2 -ffp-contract=off`` and no fast-math, so that each fp32 / fp64
operation in the oracle is one IEEE operation rounded to nearest-even and no
multiply-add is contracted (gcc on aarch64 contracts by default).
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = ("zero_oracle.c", "gen_oracle.c")
LIB = os.path.join(HERE, "_build", "liboracle.so")


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(HERE, s) for s in SOURCES] + [os.path.join(HERE, "zero_oracle.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False):
    """Compile the oracle if its library is missing or older than its sources."""
    if not force and not _stale():
        return LIB
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    tmp = LIB + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
           "-Wall", "-Wextra", "-shared", "-fPIC", "-o", tmp]
    cmd += [os.path.join(HERE, s) for s in SOURCES] + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
