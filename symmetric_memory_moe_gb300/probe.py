"""Hardware probes behind the combine's roofline analysis, built from
``csrc/probes`` with nvcc for sm_103a and run on the current GPU.

  python -m symmetric_memory_moe_gb300.probe l2        # steady-state L2 / HBM copy bandwidth
  python -m symmetric_memory_moe_gb300.probe release   # st.release.gpu latency under load

Each prints its table to stdout.  The binaries go to ``_build/probes``.
"""
from __future__ import annotations

import os
import subprocess
import sys

from . import build as _build

PROBES = {"l2": "l2_bandwidth", "release": "release_latency"}


def binary(name: str) -> str:
    src = os.path.join(_build.CSRC, "probes", PROBES[name] + ".cu")
    out_dir = os.path.join(_build.BUILD_DIR, "probes")
    exe = os.path.join(out_dir, PROBES[name])
    if not os.path.exists(exe) or os.path.getmtime(exe) < os.path.getmtime(src):
        os.makedirs(out_dir, exist_ok=True)
        subprocess.run([_build._nvcc(), *_build.ARCH, "-O3", "-std=c++17", "-o", exe, src],
                       check=True)
    return exe


def main(argv=None) -> int:
    argv = sys.argv[1:] if argv is None else argv
    if len(argv) != 1 or argv[0] not in PROBES:
        print(__doc__)
        return 2
    return subprocess.run([binary(argv[0])]).returncode


if __name__ == "__main__":
    sys.exit(main())
