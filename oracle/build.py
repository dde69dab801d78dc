"""Build the fp64 CPU oracle (plain C) into a shared library beside it.

Test infrastructure only: the oracle is what the CUDA path is checked against.
"""
from __future__ import annotations

import os
import subprocess
from pathlib import Path

HERE = Path(__file__).resolve().parent
SOURCE = HERE / "cconv_oracle.c"
OUT_DIR = HERE / "_build"
LIB = OUT_DIR / "libcconv_oracle.so"

# -ffp-contract=off: no fused multiply-adds, so x86 and Arm hosts round identically.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(source: Path = SOURCE, out: Path = LIB, force: bool = False) -> Path:
    """Compile `source` into `out` (skipped when `out` is newer than `source`)."""
    out = Path(out)
    if not force and out.exists() and out.stat().st_mtime >= Path(source).stat().st_mtime:
        return out
    out.parent.mkdir(parents=True, exist_ok=True)
    tmp = out.with_suffix(f".{os.getpid()}.tmp")
    cmd = ["gcc", *CFLAGS, "-o", str(tmp), str(source), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True))
