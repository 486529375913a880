"""Build liberi.so (the C-ABI library) for sm_103a, in-tree.

    python -m electron_repulsion_integrals_gb300.build [--force] [--jobs N]

Every ``csrc/*.cu`` and ``csrc/generated/*.cu`` is compiled to an object in
parallel with ``nvcc -gencode arch=compute_103a,code=sm_103a -O3 -lineinfo``,
then linked into ``_build/liberi.so``.  ptxas's per-kernel resource report
(registers, spill stores/loads, stack) is parsed into ``_build/ptxas.json``.
Objects are rebuilt only when their source or a shared header is newer.
"""

from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import json
import os
import re
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "liberi.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-Xptxas", "-v", "--expt-relaxed-constexpr"]


def nvcc():
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return p


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu"))) + sorted(glob.glob(os.path.join(CSRC, "generated", "*.cu")))


def _headers_mtime():
    hs = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.join(CSRC, "generated", "registry.inc")]
    return max(os.path.getmtime(h) for h in hs if os.path.exists(h))


def _compile(src, force):
    rel = os.path.relpath(src, CSRC).replace(os.sep, "_")
    obj = os.path.join(BUILD, "obj", rel + ".o")
    log = obj + ".ptxas.txt"
    if not force and os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), _headers_mtime()):
        return obj, None
    os.makedirs(os.path.dirname(obj), exist_ok=True)
    cmd = [nvcc()] + ARCH + FLAGS + ["-I", INCLUDE, "-c", src, "-o", obj + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr[-6000:]}")
    os.replace(obj + ".tmp", obj)
    with open(log, "w") as f:
        f.write(r.stderr)
    return obj, r.stderr


_FN = re.compile(r"Compiling entry function '([^']+)'")
_USE = re.compile(r"Used (\d+) registers")
_SPILL = re.compile(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads")


def parse_ptxas(text):
    out = {}
    cur = None
    for line in text.splitlines():
        m = _FN.search(line)
        if m:
            cur = m.group(1)
            out[cur] = {}
            continue
        if cur is None:
            continue
        m = _SPILL.search(line)
        if m:
            out[cur].update(stack=int(m.group(1)), spill_stores=int(m.group(2)), spill_loads=int(m.group(3)))
        m = _USE.search(line)
        if m:
            out[cur]["registers"] = int(m.group(1))
    return out


def build(force: bool = False, jobs: int | None = None, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    jobs = jobs or max(1, min(len(srcs), os.cpu_count() or 4))
    objs = []
    with cf.ThreadPoolExecutor(jobs) as ex:
        futs = {ex.submit(_compile, s, force): s for s in srcs}
        for fu in cf.as_completed(futs):
            obj, _ = fu.result()
            objs.append(obj)
            if verbose:
                print("compiled", os.path.basename(futs[fu]), flush=True)
    objs.sort()
    newest = max(os.path.getmtime(o) for o in objs)
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < newest:
        tmp = LIB + ".tmp%d" % os.getpid()
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
        os.replace(tmp, LIB)
    report = {}
    for log in glob.glob(os.path.join(BUILD, "obj", "*.ptxas.txt")):
        with open(log) as f:
            report.update(parse_ptxas(f.read()))
    with open(os.path.join(BUILD, "ptxas.json"), "w") as f:
        json.dump(report, f, indent=1, sort_keys=True)
    return LIB


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--jobs", type=int, default=None)
    a = ap.parse_args()
    print(build(a.force, a.jobs, verbose=True))


if __name__ == "__main__":
    main()
