"""GB300 electron repulsion integrals: thin Python binding of liberi.so.

Every call below marshals arguments and forwards them to the C ABI declared in
``include/eri.h``; all integral work runs in the library's CUDA kernels.  The
binding loads ``_build/liberi.so`` and raises ``RuntimeError`` if it is missing
(build it with ``python -m electron_repulsion_integrals_gb300.build``): there is
no fallback implementation.

PyTorch serves only as the device-memory and stream provider: tensors are
passed by ``data_ptr()`` and streams by ``cuda_stream``.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import workloads  # noqa: F401  (seeded inputs; no integral arithmetic)

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "liberi.so")

ERI_OK = 0
ERI_ERR_INVALID_ARG = -1
ERI_ERR_UNSUPPORTED_L = -2
STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported angular momentum or basis", -3: "output buffer too small",
          -4: "CUDA error", -5: "out of memory", -6: "non-finite or non-positive shell data", -7: "not implemented",
          -8: "class needs more scratch than the static no-allocation array holds"}

_lib = None

# C layout of eri_shell: double center[3]; int L; int nprim; const double* exps; const double* coefs;
SHELL_DTYPE = np.dtype([("center", "<f8", (3,)), ("L", "<i4"), ("nprim", "<i4"), ("exps", "<u8"), ("coefs", "<u8")],
                       align=True)


class EriError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({code})")
        self.code = code


class _Options(ctypes.Structure):
    _fields_ = [("spherical", ctypes.c_int), ("schwarz_tau", ctypes.c_double), ("flags", ctypes.c_int)]


class ClassStats(ctypes.Structure):
    _fields_ = [("vrr_ops", ctypes.c_longlong), ("vrr_flops", ctypes.c_longlong), ("hrr_ops", ctypes.c_longlong),
                ("hrr_flops", ctypes.c_longlong), ("scratch_slots", ctypes.c_int), ("staged", ctypes.c_int)]


def lib():
    """The loaded liberi.so (raises if it has not been built).  The environment
    variable ERI_GB300_LIBRARY may name another build of the same C ABI (the
    ablation libraries of build.build_variant)."""
    global _lib
    if _lib is None:
        path = os.environ.get("ERI_GB300_LIBRARY") or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"liberi.so not found at {path}; run `python -m electron_repulsion_integrals_gb300.build` "
                               "(there is no CPU fallback)")
        L = ctypes.CDLL(path)
        vp, ip, dp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int), ctypes.c_void_p
        L.eri_plan_create.argtypes = [vp, ctypes.c_int, ctypes.POINTER(_Options), vp, ctypes.POINTER(vp)]
        L.eri_plan_create_flat.argtypes = [ctypes.c_int, vp, vp, vp, vp, vp, ctypes.POINTER(_Options), vp,
                                           ctypes.POINTER(vp)]
        L.eri_plan_destroy.argtypes = [vp]
        L.eri_plan_nbf.argtypes = [vp, ip]
        L.eri_plan_shell_info.argtypes = [vp, ctypes.c_int, ip, ip]
        L.eri_compute_class.argtypes = [vp] + [ctypes.c_int] * 4 + [vp, ctypes.c_longlong, dp, ctypes.c_longlong, vp]
        L.eri_compute_class_noalloc.argtypes = [vp] + [ctypes.c_int] * 4 + [vp, ctypes.c_longlong, dp,
                                                                             ctypes.c_longlong, vp]
        L.eri_compute_class_deriv.argtypes = [vp] + [ctypes.c_int] * 4 + [vp, ctypes.c_longlong, dp, ctypes.c_longlong,
                                                                          vp]
        L.eri_schwarz.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp, ctypes.c_longlong, dp, vp]
        L.eri_build_J.argtypes = [vp, dp, dp, vp]
        L.eri_build_JK.argtypes = [vp, dp, dp, dp, vp]
        L.eri_plan_quartet_count.argtypes = [vp] + [ctypes.c_int] * 4 + [ctypes.POINTER(ctypes.c_longlong)]
        L.eri_plan_class_work.argtypes = [vp] + [ctypes.c_int] * 4 + [ctypes.POINTER(ctypes.c_longlong),
                                                                     ctypes.POINTER(ctypes.c_double)]
        L.eri_plan_class_quartets.argtypes = [vp] + [ctypes.c_int] * 4 + [ctypes.c_longlong, ctypes.c_longlong, vp,
                                                                         vp]
        L.eri_compute_screened.argtypes = [vp] + [ctypes.c_int] * 4 + [ctypes.c_longlong, ctypes.c_longlong, dp,
                                                                      ctypes.c_longlong, vp]
        L.eri_class_info.argtypes = [ctypes.c_int] * 4 + [ctypes.POINTER(ClassStats)]
        L.eri_fp64_probe.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_longlong, dp,
                                     ctypes.POINTER(ctypes.c_longlong), vp]
        L.eri_status_string.argtypes = [ctypes.c_int]
        L.eri_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _check(fn, rc):
    if rc != ERI_OK:
        raise EriError(fn, rc)


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def shell_records(shells):
    """numpy array of eri_shell records pointing into `shells`' arrays.
    The returned tuple (records, keepalive) must outlive the call."""
    n = shells.n
    rec = np.zeros(n, dtype=SHELL_DTYPE)
    rec["center"] = shells.centers
    rec["L"] = shells.L
    rec["nprim"] = shells.nprim
    exps = np.ascontiguousarray(shells.exps, dtype=np.float64)
    coefs = np.ascontiguousarray(shells.coefs, dtype=np.float64)
    rec["exps"] = exps.ctypes.data + 8 * shells.off.astype(np.uint64)
    rec["coefs"] = coefs.ctypes.data + 8 * shells.off.astype(np.uint64)
    return rec, (exps, coefs)


def eri_plan_create(shells, spherical=True, schwarz_tau=0.0, stream=None):
    """Plan over an array of eri_shell records (one pointer pair per shell)."""
    rec, keep = shell_records(shells)
    opt = _Options(int(bool(spherical)), float(schwarz_tau), 0)
    out = ctypes.c_void_p()
    rc = lib().eri_plan_create(rec.ctypes.data_as(ctypes.c_void_p), shells.n, ctypes.byref(opt),
                               ctypes.c_void_p(_stream_handle(stream)), ctypes.byref(out))
    del keep
    _check("eri_plan_create", rc)
    return out


def eri_plan_create_flat(shells, spherical=True, schwarz_tau=0.0, stream=None):
    """Plan over flat shell arrays (centers, L, nprim, exps, coefs)."""
    c = np.ascontiguousarray(shells.centers, dtype=np.float64)
    L = np.ascontiguousarray(shells.L, dtype=np.int32)
    n = np.ascontiguousarray(shells.nprim, dtype=np.int32)
    e = np.ascontiguousarray(shells.exps, dtype=np.float64)
    f = np.ascontiguousarray(shells.coefs, dtype=np.float64)
    opt = _Options(int(bool(spherical)), float(schwarz_tau), 0)
    out = ctypes.c_void_p()
    rc = lib().eri_plan_create_flat(int(len(L)), c.ctypes.data, L.ctypes.data, n.ctypes.data, e.ctypes.data,
                                    f.ctypes.data, ctypes.byref(opt), ctypes.c_void_p(_stream_handle(stream)),
                                    ctypes.byref(out))
    _check("eri_plan_create_flat", rc)
    return out


def eri_plan_destroy(plan):
    _check("eri_plan_destroy", lib().eri_plan_destroy(plan))


def eri_plan_nbf(plan):
    n = ctypes.c_int()
    _check("eri_plan_nbf", lib().eri_plan_nbf(plan, ctypes.byref(n)))
    return n.value


def eri_plan_shell_info(plan, s):
    nf, first = ctypes.c_int(), ctypes.c_int()
    _check("eri_plan_shell_info", lib().eri_plan_shell_info(plan, int(s), ctypes.byref(nf), ctypes.byref(first)))
    return nf.value, first.value


def eri_compute_class(plan, cls, quartets, out, stream=None, n=None):
    """quartets: int32 CUDA tensor (n,4); out: float64 CUDA tensor with >= n*B elements.
    quartets None with n = the class's screened quartet count: every screened quartet."""
    if quartets is not None:
        n = quartets.shape[0]
    n = n or 0
    rc = lib().eri_compute_class(plan, *[int(x) for x in cls], _ptr(quartets), int(n), _ptr(out), int(out.numel()),
                                 ctypes.c_void_p(_stream_handle(stream)))
    _check("eri_compute_class", rc)


def eri_compute_class_noalloc(plan, cls, quartets, out, stream=None):
    """eri_compute_class without device allocation (static scratch array; see include/eri.h)."""
    n = quartets.shape[0] if quartets is not None else 0
    rc = lib().eri_compute_class_noalloc(plan, *[int(x) for x in cls], _ptr(quartets), int(n), _ptr(out),
                                         int(out.numel()), ctypes.c_void_p(_stream_handle(stream)))
    _check("eri_compute_class_noalloc", rc)


def eri_compute_class_deriv(plan, cls, quartets, out, stream=None):
    """First derivatives of the blocks of eri_compute_class: out holds, per
    quartet, 12 blocks [shell position 0..3][axis x, y, z][block]."""
    n = int(quartets.shape[0])
    rc = lib().eri_compute_class_deriv(plan, *[int(x) for x in cls], _ptr(quartets) if n else None, n,
                                       _ptr(out) if n else None, int(out.numel()),
                                       ctypes.c_void_p(_stream_handle(stream)))
    _check("eri_compute_class_deriv", rc)


def eri_schwarz(plan, la, lb, pairs, q_out, stream=None):
    rc = lib().eri_schwarz(plan, int(la), int(lb), _ptr(pairs), int(pairs.shape[0]), _ptr(q_out),
                           ctypes.c_void_p(_stream_handle(stream)))
    _check("eri_schwarz", rc)


def eri_build_J(plan, D, J, stream=None):
    _check("eri_build_J", lib().eri_build_J(plan, _ptr(D), _ptr(J), ctypes.c_void_p(_stream_handle(stream))))


def eri_build_JK(plan, D, J, K, stream=None):
    _check("eri_build_JK", lib().eri_build_JK(plan, _ptr(D), _ptr(J), _ptr(K),
                                              ctypes.c_void_p(_stream_handle(stream))))


def eri_plan_quartet_count(plan, cls):
    n = ctypes.c_longlong()
    _check("eri_plan_quartet_count", lib().eri_plan_quartet_count(plan, *[int(x) for x in cls], ctypes.byref(n)))
    return n.value


def eri_plan_class_work(plan, cls):
    """(unique quartets, primitive quartets) of a class in the screened plan."""
    n, pq = ctypes.c_longlong(), ctypes.c_double()
    _check("eri_plan_class_work", lib().eri_plan_class_work(plan, *[int(x) for x in cls], ctypes.byref(n),
                                                           ctypes.byref(pq)))
    return n.value, pq.value


def eri_plan_class_quartets(plan, cls, first, count, quartets, stream=None):
    """Write quartets [first, first + count) of a class's screened list into
    the device int32 tensor `quartets` ([count, 4])."""
    if count and (quartets.dtype.itemsize != 4 or not quartets.is_contiguous() or quartets.numel() < 4 * count):
        raise ValueError("quartets must be a contiguous int32 tensor of at least 4 x count elements")
    _check("eri_plan_class_quartets", lib().eri_plan_class_quartets(
        plan, *[int(x) for x in cls], int(first), int(count), _ptr(quartets) if count else None,
        ctypes.c_void_p(_stream_handle(stream))))


def eri_compute_screened(plan, cls, first, count, out, stream=None):
    """Blocks of quartets [first, first + count) of a class's screened list
    into the device float64 tensor `out`."""
    _check("eri_compute_screened", lib().eri_compute_screened(
        plan, *[int(x) for x in cls], int(first), int(count), _ptr(out), int(out.numel()) if out is not None else 0,
        ctypes.c_void_p(_stream_handle(stream))))


def eri_class_info(cls):
    s = ClassStats()
    _check("eri_class_info", lib().eri_class_info(*[int(x) for x in cls], ctypes.byref(s)))
    return {f: getattr(s, f) for f, _ in ClassStats._fields_}


FP64_PROBE_OPS = {"fma": 0, "mul": 1, "add": 2}


def eri_fp64_probe(op, blocks, threads, iters, sink, stream=None):
    """Launch the FP64 rate probe (see include/eri.h) for op "fma", "mul" or
    "add"; returns the number of operations launched."""
    n = ctypes.c_longlong()
    _check("eri_fp64_probe", lib().eri_fp64_probe(FP64_PROBE_OPS[op], int(blocks), int(threads), int(iters),
                                                  _ptr(sink), ctypes.byref(n), ctypes.c_void_p(_stream_handle(stream))))
    return n.value


def nfunc(l, spherical=True):
    return 2 * l + 1 if (spherical and l >= 2) else (l + 1) * (l + 2) // 2


def block_size(cls, spherical=True):
    return int(np.prod([nfunc(l, spherical) for l in cls]))


class Plan:
    """Owning wrapper around an eri_plan handle."""

    def __init__(self, shells, spherical=True, schwarz_tau=0.0, stream=None):
        self.shells = shells
        self.spherical = spherical
        self.handle = eri_plan_create_flat(shells, spherical, schwarz_tau, stream)
        self.nbf = eri_plan_nbf(self.handle)

    def compute_class(self, cls, quartets, out=None, stream=None):
        import torch
        n = quartets.shape[0]
        if out is None:
            out = torch.empty(n * block_size(cls, self.spherical), dtype=torch.float64, device=quartets.device)
        eri_compute_class(self.handle, cls, quartets, out, stream)
        return out

    def compute_class_deriv(self, cls, quartets, out=None, stream=None):
        import torch
        n = int(quartets.shape[0])
        if out is None:
            out = torch.empty(max(n, 1) * 12 * block_size(cls, self.spherical), dtype=torch.float64,
                              device=quartets.device)
        eri_compute_class_deriv(self.handle, cls, quartets, out, stream)
        return out

    def schwarz(self, la, lb, pairs, stream=None):
        import torch
        q = torch.empty(pairs.shape[0], dtype=torch.float64, device=pairs.device)
        eri_schwarz(self.handle, la, lb, pairs, q, stream)
        return q

    def build_J(self, D, J=None, stream=None):
        import torch
        if J is None:
            J = torch.empty_like(D)
        eri_build_J(self.handle, D, J, stream)
        return J

    def build_JK(self, D, J=None, K=None, stream=None):
        import torch
        J = torch.empty_like(D) if J is None else J
        K = torch.empty_like(D) if K is None else K
        eri_build_JK(self.handle, D, J, K, stream)
        return J, K

    def quartet_count(self, cls):
        return eri_plan_quartet_count(self.handle, cls)

    def class_quartets(self, cls, first=0, count=None, out=None, stream=None):
        """The screened unique quartets of canonical class `cls` (all of them,
        or [first, first + count)) as a device int32 tensor [count, 4]."""
        import torch
        if count is None:
            count = self.quartet_count(cls) - first
        if out is None:
            out = torch.empty((max(count, 1), 4), dtype=torch.int32, device=torch.device("cuda", torch.cuda.current_device()))
        eri_plan_class_quartets(self.handle, cls, first, count, out, stream)
        return out[:count]

    def compute_screened(self, cls, first=0, count=None, out=None, stream=None):
        """Blocks of the screened quartets [first, first + count) of canonical
        class `cls` (all of them by default), flat float64 on the device."""
        import torch
        if count is None:
            count = self.quartet_count(cls) - first
        if out is None:
            out = torch.empty(max(count, 1) * block_size(cls, self.spherical), dtype=torch.float64,
                              device=torch.device("cuda", torch.cuda.current_device()))
        eri_compute_screened(self.handle, cls, first, count, out, stream)
        return out

    def close(self):
        if self.handle:
            eri_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
