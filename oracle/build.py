"""Build the CPU oracle (test infrastructure) as two shared libraries.

``python -m oracle.build`` compiles ``pa_oracle.c`` with gcc into a float build
and a double build, next to this file.  Plain C, no fast-math: the oracle keeps
IEEE semantics and the summation order written in the source.
"""
from __future__ import annotations

import os
import subprocess
import sys

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "pa_oracle.c")
LIBS = {"f32": "libpa_oracle_f32.so", "f64": "libpa_oracle_f64.so"}
_FLAGS = {"f32": ["-DORACLE_F32"], "f64": []}


def build(src: str = SRC, out_dir: str = _HERE, extra=(), verbose: bool = False,
          precisions=("f32", "f64")) -> dict:
    """Compile the builds named in ``precisions``; returns {precision: path}.
    ``extra`` adds gcc flags."""
    cc = os.environ.get("CC", "gcc")
    procs, paths = [], {}
    for prec in precisions:
        name = LIBS[prec]
        out = os.path.join(out_dir, name)
        cmd = [cc, "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", *_FLAGS[prec], *extra,
               src, "-o", out, "-lm"]
        if verbose:
            print(" ".join(cmd))
        procs.append((subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT),
                      cmd))
        paths[prec] = out
    for p, cmd in procs:
        log, _ = p.communicate()
        if p.returncode != 0:
            raise RuntimeError(f"oracle build failed: {' '.join(cmd)}\n{log.decode()}")
    return paths


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
