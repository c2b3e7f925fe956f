"""Builds the oracle's shared library with gcc.

Test infrastructure only (see ``oracle/__init__.py``).
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pa_oracle.c")
DEFAULT_LIB = os.path.join(HERE, "liboracle.so")


def build(out_path: str = DEFAULT_LIB, mutation: int = 0, force: bool = False) -> str:
    """Compile pa_oracle.c into ``out_path`` (skipped when up to date)."""
    if (not force and mutation == 0 and os.path.exists(out_path)
            and os.path.getmtime(out_path) >= max(os.path.getmtime(SRC),
                                                  os.path.getmtime(SRC[:-2] + ".h"))):
        return out_path
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-pthread",
           f"-DORACLE_MUTATION={int(mutation)}", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


if __name__ == "__main__":
    print(build(force=True))
