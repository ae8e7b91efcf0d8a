"""Build step for the CPU oracle (test infrastructure only).

Compiles moe_oracle.cpp into oracle/libmoe_oracle.so with the host C++
compiler. Plain C++17, no architecture flags, so the same source builds on
x86_64 and aarch64 hosts.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.cpp")
LIB = os.path.join(HERE, "libmoe_oracle.so")


def build_oracle(force: bool = False) -> str:
    deps = [SRC, os.path.join(HERE, "moe_oracle.h")]
    if not force and os.path.exists(LIB) and all(
        os.path.getmtime(LIB) >= os.path.getmtime(p) for p in deps
    ):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["g++", "-std=c++17", "-O2", "-fPIC", "-shared", "-pthread",
           "-Wall", "-Wextra", "-o", tmp, SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
