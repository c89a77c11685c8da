"""Compile the C oracle into oracle/_build/libpa_oracle.so.

TEST INFRASTRUCTURE ONLY: building the checker is not using it.  The product
library never links or loads what this produces.
"""
import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pa_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libpa_oracle.so")


def _compile(extra):
    os.makedirs(OUT_DIR, exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=OUT_DIR)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", *extra, SRC, "-o", tmp, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        os.unlink(tmp)
        return r.stderr
    os.replace(tmp, LIB)
    return None


def build(force=False):
    """Build the oracle (OpenMP when the compiler supports it); return the .so path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    err = _compile(["-fopenmp"])
    if err is not None:
        err2 = _compile([])
        if err2 is not None:
            raise RuntimeError("oracle build failed:\n" + err + "\n" + err2)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
