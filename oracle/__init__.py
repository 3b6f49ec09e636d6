"""fp64 CPU oracle for packed-tree KDA: loader and numpy-facing wrappers.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg import this package.  It shares no code with the
CUDA library (``prefix_shared_chunkwise_gb300``) and never imports it.

* ``kda_forest``: tree -> trajectories -> token-by-token recurrence, fwd + exact bwd
  (``kda_oracle.c``).
* ``plan_twin``: the minimum-call recurrence and brute force (``plan_twin.py``).
* ``chunkwise``: fp64 chunkwise form and a plan-following tree executor, used to pin
  the chunkwise reading and the replay rule on small inputs (``chunkwise.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_kda_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain C, -O2, OpenMP)."""
    src = os.path.join(_HERE, "kda_oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               src, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        d = ctypes.POINTER(ctypes.c_double)
        i32 = ctypes.POINTER(ctypes.c_int32)
        i64 = ctypes.POINTER(ctypes.c_int64)
        lib.oracle_kda_forest.restype = ctypes.c_int
        lib.oracle_kda_forest.argtypes = [
            ctypes.c_int32, i32, i64, i64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_int32, ctypes.c_double, d, d, d, d, d, d, d, d, d, d, d, d, d, d, d, d,
            ctypes.c_int32, d]
        _lib = lib
    return _lib


def _p(a, ty):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ty))


def kda_forest(parent, seg_len, seg_offset, q, k, v, g, beta, *, chunk=64, scale=1.0,
               h0=None, W=None, d_final=None, n_threads=0):
    """Run the oracle over every trajectory of the forest.

    Inputs are compact ``[C, H, d]`` arrays (``beta``: ``[C, H]``), converted to fp64;
    ``seg_offset[v]`` is the compact row of segment v's first token.  Returns a dict
    with ``o``, ``final`` (``[n_leaves, H, dk, dv]``, leaves in increasing segment id),
    ``occ_diff`` (largest disagreement between occurrences of one row) and, when ``W``
    is given, ``dq, dk, dv, dg, dbeta`` (and ``dh0`` when ``h0`` is given)."""
    lib = _load()
    parent = np.ascontiguousarray(parent, np.int32)
    seg_len = np.ascontiguousarray(seg_len, np.int64)
    seg_offset = np.ascontiguousarray(seg_offset, np.int64)
    f = lambda a: None if a is None else np.ascontiguousarray(a, np.float64)
    q, k, v, g, beta, h0, W, d_final = map(f, (q, k, v, g, beta, h0, W, d_final))
    C, H, dk = q.shape
    dv = v.shape[2]
    n_leaves = int(np.sum(np.bincount(parent[parent >= 0], minlength=len(parent)) == 0))
    n_roots = int(np.sum(parent < 0))
    o = np.zeros((C, H, dv))
    final = np.zeros((n_leaves, H, dk, dv))
    grads = None
    if W is not None:
        grads = dict(dq=np.zeros((C, H, dk)), dk=np.zeros((C, H, dk)), dv=np.zeros((C, H, dv)),
                     dg=np.zeros((C, H, dk)), dbeta=np.zeros((C, H)))
        if h0 is not None:
            grads["dh0"] = np.zeros((n_roots, H, dk, dv))
    occ = ctypes.c_double(0.0)
    D = ctypes.c_double
    gp = (lambda n: _p(grads[n], D) if grads and n in grads else None)
    rc = lib.oracle_kda_forest(
        len(parent), _p(parent, ctypes.c_int32), _p(seg_len, ctypes.c_int64),
        _p(seg_offset, ctypes.c_int64), H, dk, dv, chunk, scale,
        _p(q, D), _p(k, D), _p(v, D), _p(g, D), _p(beta, D), _p(h0, D), _p(W, D),
        _p(d_final, D), _p(o, D), _p(final, D), gp("dq"), gp("dk"), gp("dv"), gp("dg"),
        gp("dbeta"), gp("dh0"), n_threads, ctypes.byref(occ))
    if rc != 0:
        raise RuntimeError(f"oracle_kda_forest failed: {rc}")
    out = dict(o=o, final=final, occ_diff=occ.value)
    if grads:
        out.update(grads)
    return out
