"""Build the CPU oracle (test infrastructure) as a shared library with gcc.

The oracle is compiled with -ffp-contract=off so that every FP32 multiply and
add rounds on its own (GCC contracts a*b+c into an FMA by default on aarch64),
and without -ffast-math so that subnormals and IEEE division are kept.
"""
from __future__ import annotations

import os
import platform
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "nvfp4_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fvisibility=hidden", "-Wall", "-Wextra", "-Werror"]


def library_path() -> str:
    return os.path.join(OUT_DIR, f"liboracle_{platform.machine()}.so")


def build(force: bool = False) -> str:
    """Compile the oracle if the library is missing or older than its source."""
    out = library_path()
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(SRC)):
        return out
    os.makedirs(OUT_DIR, exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=OUT_DIR)
    os.close(fd)
    try:
        subprocess.run(["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, out)  # atomic: concurrent builders never see a partial file
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return out


def build_variant(source_text: str, out_path: str) -> str:
    """Compile a modified copy of the oracle source (used by the mutation tests,
    which plant a mistake and check that the pins catch it)."""
    d = os.path.dirname(out_path)
    src = os.path.join(d, "variant.c")
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", *[f for f in CFLAGS if f != "-Werror"], src, "-o", out_path, "-lm"],
                   check=True)
    return out_path


if __name__ == "__main__":
    print(build(force=True))
