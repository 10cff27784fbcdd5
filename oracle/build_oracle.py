"""Builds the C++ oracle (oracle/moe_oracle.cpp) into oracle/lib/libmoe_oracle.so
with the host compiler: plain -O2, no target-specific flags, so the same
source builds on x86-64 and on Arm.  Rebuilt when the source changes.

TEST INFRASTRUCTURE ONLY (see oracle/moe_oracle_cpp.py)."""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.cpp")
LIB = os.path.join(HERE, "lib", "libmoe_oracle.so")
STAMP = LIB + ".stamp"
FLAGS = ["-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", "-fvisibility=hidden"]


def _fingerprint() -> str:
    h = hashlib.sha256(open(SRC, "rb").read())
    h.update(" ".join(FLAGS).encode())
    return h.hexdigest()


def build(force: bool = False) -> str:
    fp = _fingerprint()
    if not force and os.path.exists(LIB) and os.path.exists(STAMP) and open(STAMP).read().strip() == fp:
        return LIB
    cxx = os.environ.get("CXX") or shutil.which("g++") or shutil.which("c++")
    if not cxx:
        raise RuntimeError("no C++ compiler found for the oracle")
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    tmp = LIB + ".tmp"
    r = subprocess.run([cxx, *FLAGS, SRC, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"oracle build failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(fp)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
