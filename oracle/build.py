"""Build the fp64 CPU oracle (test infrastructure) into ``oracle/libsporacle.so``.

Plain ``g++``; no architecture-specific flags so that the same source gives the same results
on x86_64 and aarch64 hosts. ``-ffp-contract=off`` keeps every multiply and add separately
rounded (GCC would otherwise fuse them into FMAs on aarch64).
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "sp_oracle.cpp")
LIBRARY = os.path.join(HERE, "libsporacle.so")

FLAGS = ["-std=c++17", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
         "-Wall", "-Wextra"]


def build(source: str = SOURCE, library: str = LIBRARY, extra_flags: list[str] | None = None) -> str:
    """Compile ``source`` into the shared library ``library`` if it is missing or stale."""
    if (os.path.exists(library) and os.path.getmtime(library) >= os.path.getmtime(source)
            and not extra_flags):
        return library
    tmp = library + f".tmp{os.getpid()}"
    cmd = ["g++", *FLAGS, *(extra_flags or []), source, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, library)
    return library


if __name__ == "__main__":
    print(build())
    sys.exit(0)
