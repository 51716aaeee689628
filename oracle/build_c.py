"""Compile the oracle's C part (``rowacc.c``) into ``librowacc.so``.

TEST INFRASTRUCTURE ONLY.  Plain gcc, no architecture flags, so the same
source builds on x86-64 and aarch64 hosts.
"""

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))


def build():
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        raise RuntimeError("no C compiler for the oracle")
    src = os.path.join(HERE, "rowacc.c")
    out = os.path.join(HERE, "librowacc.so")
    tmp = out + ".tmp"
    cmd = [cc, "-O2", "-fPIC", "-shared", "-fopenmp", "-o", tmp, src, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("oracle C build failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build())
