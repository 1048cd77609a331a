"""Builds liboracle.so (test infrastructure) with gcc: plain C99 + OpenMP,
no fast-math and no FMA contraction, so x86 and Arm give the same sums."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))


def build(verbose: bool = False) -> str:
    out = os.path.join(HERE, "liboracle.so")
    cc = os.environ.get("CC", "gcc")
    cmd = [cc, "-std=c99", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-Wall", "-Wno-unknown-pragmas", "-o", out + ".tmp",
           os.path.join(HERE, "oracle.c"), "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True, cwd=HERE)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build(verbose=True))
