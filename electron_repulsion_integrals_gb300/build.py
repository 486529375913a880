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


def _compile(src, force, objdir=None, extra=()):
    rel = os.path.relpath(src, CSRC).replace(os.sep, "_") if objdir is None else os.path.basename(src)
    obj = os.path.join(objdir or os.path.join(BUILD, "obj"), rel + ".o")
    log = obj + ".ptxas.txt"
    if not force and os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), _headers_mtime()):
        return obj, None
    os.makedirs(os.path.dirname(obj), exist_ok=True)
    cmd = [nvcc()] + ARCH + FLAGS + ["-I", INCLUDE, "-I", os.path.join(CSRC, "generated")] + list(extra) + \
        ["-c", src, "-o", obj + ".tmp"]
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


def build_variant(name: str, entries, force: bool = False, jobs: int | None = None) -> str:
    """Build a complete library over another set of class kernels: `entries`
    lists (class, opts) pairs, each class emitted with the generator switches
    `opts` (see gen.emit.emit_class; {"tier": "coop"} emits the cooperative
    tier).  Used to measure one design choice at a time (the ablations of
    FusionRCG section V-B, where every variant is compiled as a complete
    library).  Returns the path of _build/variants/<name>/liberi.so."""
    from .gen.emit import emit_class
    from .gen.coop import emit_coop_class
    vdir = os.path.join(BUILD, "variants", name)
    gdir = os.path.join(vdir, "generated")
    os.makedirs(gdir, exist_ok=True)
    stats = {}
    srcs = []
    classes = [tuple(c) for c, _ in entries]
    for cls, opts in entries:
        cls = tuple(cls)
        if opts.get("tier") == "coop":
            src, meta = emit_coop_class(cls)
        else:
            src, meta = emit_class(cls, **opts)
        path = os.path.join(gdir, "c{}{}{}{}.cu".format(*cls))
        if not os.path.exists(path) or open(path).read() != src:
            with open(path, "w") as f:
                f.write(src)
        srcs.append(path)
        stats["{}{}{}{}".format(*cls)] = meta
    dreg = os.path.join(gdir, "registry_deriv.inc")   # no derivative kernels in a variant
    if not os.path.exists(dreg):
        with open(dreg, "w") as f:
            f.write("")
    reg = os.path.join(gdir, "registry.inc")
    text = "".join("ERI_CLASS({}, {}, {}, {})\n".format(*c) for c in classes)
    if not os.path.exists(reg) or open(reg).read() != text:
        with open(reg, "w") as f:
            f.write(text)
    with open(os.path.join(vdir, "classes.json"), "w") as f:
        json.dump({"entries": [[list(c), o] for c, o in entries], "classes": stats}, f, indent=1, sort_keys=True,
                  default=str)
    runtime = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    objdir = os.path.join(vdir, "obj")
    extra = ["-DERI_REGISTRY_INC=\"" + reg + "\"", "-DERI_DERIV_REGISTRY_INC=\"" + dreg + "\""]
    jobs = jobs or max(1, min(len(srcs) + len(runtime), os.cpu_count() or 4))
    objs = []
    with cf.ThreadPoolExecutor(jobs) as ex:
        futs = [ex.submit(_compile, s_, force or s_ in runtime and _newer(reg, s_, objdir), objdir,
                          extra if s_ in runtime else ()) for s_ in runtime + srcs]
        for fu in futs:
            objs.append(fu.result()[0])
    lib = os.path.join(vdir, "liberi.so")
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs):
        tmp = lib + ".tmp%d" % os.getpid()
        r = subprocess.run([nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"], capture_output=True,
                           text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
        os.replace(tmp, lib)
    report = {}
    for log in glob.glob(os.path.join(objdir, "*.ptxas.txt")):
        with open(log) as f:
            report.update(parse_ptxas(f.read()))
    with open(os.path.join(vdir, "ptxas.json"), "w") as f:
        json.dump(report, f, indent=1, sort_keys=True)
    return lib


def _newer(path, src, objdir):
    """True when `path` changed after the object of `src` in `objdir` was built."""
    obj = os.path.join(objdir, os.path.basename(src) + ".o")
    return not os.path.exists(obj) or os.path.getmtime(path) > os.path.getmtime(obj)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--jobs", type=int, default=None)
    a = ap.parse_args()
    print(build(a.force, a.jobs, verbose=True))


if __name__ == "__main__":
    main()
