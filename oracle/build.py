"""Compile the fp64 CPU oracle (moe_oracle.c) into liboracle.so with gcc.

Test infrastructure only: the oracle checks the CUDA library and is never
linked into it.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Build liboracle.so next to its source if missing or stale; return its path.

    MOE_ORACLE_LIB, when set, names another build of this source to use instead
    (the mutation tests point it at copies with a planted mistake).
    """
    override = os.environ.get("MOE_ORACLE_LIB")
    if override:
        return override
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    # -O2 without -ffast-math: no reassociation, so each sum runs in the
    # order the loops state.
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
           "-shared", "-pthread", "-o", LIB + ".tmp", SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
