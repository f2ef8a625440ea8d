"""ctypes front end of the plain C++ float64 oracle (``oracle/opd_ref.cpp``).

TEST INFRASTRUCTURE ONLY -- used by ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py``; the CUDA library and its binding never import it.

``build()`` compiles the oracle with the host C++ compiler into
``oracle/_build/liboracle_opd.so`` (float64 throughout, no fast-math, no
floating-point contraction).  The functions below marshal numpy arrays and return
the same quantities as ``oracle/opd.py``.
"""

from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "opd_ref.cpp")
LIB = os.path.join(HERE, "_build", "liboracle_opd.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the C++ oracle (skipped when the library is newer than its source)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        raise RuntimeError("no host C++ compiler: the C++ oracle cannot be built")
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = [cxx, "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", "-ffp-contract=off", "-fno-fast-math",
           SRC, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"C++ oracle build failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB)
        P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        L.oracle_row_forward.argtypes = [P, P, I, D, D, P, P]
        L.oracle_row_forward.restype = None
        L.oracle_row_grad.argtypes = [P, P, I, D, D, D, P]
        L.oracle_row_grad.restype = None
        L.oracle_verify_packed.argtypes = [P, I, I64, P, P, I, I, I, P, P, P, P]
        L.oracle_verify_packed.restype = None
        L.oracle_opd_rows.argtypes = [P, I, I64, P, I, I64, P, I, I, D, D, P, I64, P, D, I, P, P, P, P]
        L.oracle_opd_rows.restype = None
        _lib = L
    return _lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def row_forward(z, t, c, beta=1.0) -> dict:
    """The same keys as ``oracle.opd.row_forward`` for one pair of rows."""
    z, t = _f64(z), _f64(t)
    out = np.zeros(7)
    ints = np.zeros(2, dtype=np.int32)
    lib().oracle_row_forward(_ptr(z), _ptr(t), len(z), float(c), float(beta), _ptr(out), _ptr(ints))
    return dict(kl=out[0], ce=out[1], loss_row=out[2], lse_z=out[3], lse_t=out[4], S=out[5], S_l1=out[6],
                argmax=int(ints[0]), n_clipped=int(ints[1]))


def row_grad(z, t, c, beta, g=1.0) -> np.ndarray:
    z, t = _f64(z), _f64(t)
    dz = np.empty(len(z))
    lib().oracle_row_grad(_ptr(z), _ptr(t), len(z), float(c), float(beta), float(g), _ptr(dz))
    return dz


def _storage(arr, dtype):
    """A packed logit array as the oracle reads it: float32, or uint16 bfloat16 bit patterns."""
    if dtype == "bf16":
        return np.ascontiguousarray(arr, dtype=np.uint16), 1
    return np.ascontiguousarray(arr, dtype=np.float32), 0


def verify_packed(target, t_dtype, tokens, doff, vocab, threads=1):
    """Greedy verification of every request: (target_argmax [N_t], accept_len, bonus_token, accept_rate)."""
    t, tb = _storage(target, t_dtype)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    doff = np.ascontiguousarray(doff, dtype=np.int32)
    R = len(doff) - 1
    Nt = int(doff[-1]) + R
    am = np.empty(Nt, dtype=np.int32)
    L = np.empty(R, dtype=np.int32)
    bonus = np.empty(R, dtype=np.int32)
    rate = np.empty(R, dtype=np.float32)
    lib().oracle_verify_packed(_ptr(t), tb, t.shape[1], _ptr(tokens), _ptr(doff), R, int(vocab), int(threads),
                               _ptr(am), _ptr(L), _ptr(bonus), _ptr(rate))
    return am, L, bonus, rate


def opd_rows(draft, d_dtype, target, t_dtype, doff, vocab, c, beta=1.0, rows=None, grad=False, grad_row=None,
             grad_scale=1.0, threads=1):
    """Forward (and gradient) of the listed draft rows (all rows when ``rows`` is None).

    Returns (per_row, grads, loss): per_row[d] holds the keys of
    ``oracle.opd.row_forward``, grads[d] the gradient row (when ``grad``), and loss the
    mean over all draft rows (None unless every row is computed)."""
    z, zb = _storage(draft, d_dtype)
    t, tb = _storage(target, t_dtype)
    doff = np.ascontiguousarray(doff, dtype=np.int32)
    R = len(doff) - 1
    rl = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    n = int(doff[-1]) if rl is None else len(rl)
    stats = np.zeros((n, 8))
    ints = np.zeros((n, 2), dtype=np.int32)
    g = np.empty((n, int(vocab))) if grad else None
    gr = None if grad_row is None else np.ascontiguousarray(grad_row, dtype=np.float64)
    loss = np.zeros(1)
    lib().oracle_opd_rows(_ptr(z), zb, z.shape[1], _ptr(t), tb, t.shape[1], _ptr(doff), R, int(vocab), float(c),
                          float(beta), _ptr(rl), n, _ptr(gr), float(grad_scale), int(threads), _ptr(stats),
                          _ptr(ints), _ptr(g), _ptr(loss))
    ids = range(n) if rl is None else [int(x) for x in rl]
    per, grads = {}, {}
    for k, d in enumerate(ids):
        s = stats[k]
        per[d] = dict(kl=s[0], ce=s[1], loss_row=s[2], lse_z=s[3], lse_t=s[4], S=s[5], S_l1=s[6],
                      argmax=int(ints[k, 0]), n_clipped=int(ints[k, 1]))
        if grad:
            grads[d] = g[k]
    return per, grads, (float(loss[0]) if rl is None else None)
