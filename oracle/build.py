"""Compile the C oracle into two shared libraries (float and double builds).

Test infrastructure: the test suite, the smoke check and the benchmark's
CPU-baseline leg load these; the CUDA library never does.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gdn_ref.c")
LIBS = {"f32": os.path.join(HERE, "libgdn_ref_f32.so"),
        "f64": os.path.join(HERE, "libgdn_ref_f64.so")}
CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra"]


def _stale(lib):
    if not os.path.exists(lib):
        return True
    mt = os.path.getmtime(lib)
    return any(os.path.getmtime(os.path.join(HERE, f)) > mt for f in ("gdn_ref.c", "gdn_ref.h"))


def build(force=False):
    """Build both oracle libraries (skips ones that are up to date)."""
    cc = os.environ.get("CC", "gcc")
    for prec, lib in LIBS.items():
        if not force and not _stale(lib):
            continue
        extra = ["-DGDN_REF_DOUBLE"] if prec == "f64" else []
        tmp = lib + ".tmp"
        cmd = [cc, *CFLAGS, *extra, SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib)
    return dict(LIBS)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
