"""Build the fp64 CPU oracle (test infrastructure only) into oracle/_build/.

The oracle is plain C compiled with gcc; OpenMP is used when the compiler
supports it (it only spreads independent output rows over host cores).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile oracle.c into a shared library; returns its path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    cc = os.environ.get("CC", "gcc")
    base = [cc, "-O2", "-std=c11", "-fPIC", "-shared", SRC, "-o", LIB + ".tmp", "-lm"]
    for extra in (["-fopenmp"], []):
        cmd = base[:2] + extra + base[2:]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose:
            print(" ".join(cmd), r.stdout, r.stderr, file=sys.stderr)
        if r.returncode == 0:
            os.replace(LIB + ".tmp", LIB)
            return LIB
    raise RuntimeError("oracle build failed:\n" + r.stderr)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
