"""CPU oracle for the tensor-parallel MLP block and the vocabulary-parallel
cross-entropy -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The library under ``vocab_ce_gb300``
never imports, links or runs it, and this package never imports the library.

The arithmetic lives in ``oracle.c`` (plain fp64 loops); this module builds it
with gcc into ``liboracle.so`` and marshals numpy arrays to it. Every input is
widened to float64 before the call, so the oracle sees the exact bf16 or fp32
values the GPU reads.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "oracle.c")
LIB_PATH = os.path.join(_HERE, "liboracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False, quiet: bool = True) -> str:
    """Compile oracle.c with gcc (OpenMP when available). Returns the .so path."""
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= os.path.getmtime(SRC):
        return LIB_PATH
    base = ["gcc", "-O3", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-shared", "-fPIC", SRC, "-o", LIB_PATH + ".tmp", "-lm"]
    last = None
    for extra in (["-fopenmp"], []):
        r = subprocess.run(base[:1] + extra + base[1:], capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(LIB_PATH + ".tmp", LIB_PATH)
            return LIB_PATH
        last = r.stderr
    raise RuntimeError("oracle build failed:\n" + (last or ""))


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(LIB_PATH)
        D = ctypes.c_double
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_gelu.restype = D
        lib.oracle_gelu.argtypes = [D]
        lib.oracle_gelu_grad.restype = D
        lib.oracle_gelu_grad.argtypes = [D]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        lib.oracle_mlp_forward.restype = None
        lib.oracle_mlp_forward.argtypes = [I64, I64, I64, P, P, P, P, P, P, P, P]
        lib.oracle_mlp_backward.restype = None
        lib.oracle_mlp_backward.argtypes = [I64, I64, I64, P, P, P, P, P, P, P, P, P, P]
        lib.oracle_mlp_backward_cols.restype = None
        lib.oracle_mlp_backward_cols.argtypes = [I64, I64, I64, P, P, P, P, P, I64, P, P, P, P]
        lib.oracle_bias_grad.restype = None
        lib.oracle_bias_grad.argtypes = [I64, I64, P, P]
        lib.oracle_mlp_sharded.restype = None
        lib.oracle_mlp_sharded.argtypes = [I64, I64, I64, ctypes.c_int, P, P, P, P, P, P, P, P, P, P]
        lib.oracle_ce.restype = None
        lib.oracle_ce.argtypes = [I64, I64, I64, I64, P, P, P, D, P, P, P, P]
        lib.oracle_ce_sharded.restype = None
        lib.oracle_ce_sharded.argtypes = [I64, I64, I64, I64, ctypes.c_int, P, P, P, P, P, P, P]
        lib.oracle_swish.restype = D
        lib.oracle_swish.argtypes = [D]
        lib.oracle_swish_grad.restype = D
        lib.oracle_swish_grad.argtypes = [D]
        lib.oracle_swiglu_forward.restype = None
        lib.oracle_swiglu_forward.argtypes = [I64, I64, I64, P, P, P, P, P, P, P, P]
        lib.oracle_swiglu_backward.restype = None
        lib.oracle_swiglu_backward.argtypes = [I64, I64, I64, P, P, P, P, P, P, P, P, P, P]
        lib.oracle_swiglu_backward_cols.restype = None
        lib.oracle_swiglu_backward_cols.argtypes = [I64, I64, I64, P, P, P, P, P, I64, P, P, P, P, P, P]
        lib.oracle_swiglu_sharded.restype = None
        lib.oracle_swiglu_sharded.argtypes = [I64, I64, I64, ctypes.c_int, P, P, P, P, P, P, P, P, P, P]
        lib.oracle_linear_forward.restype = None
        lib.oracle_linear_forward.argtypes = [I64, I64, I64, P, P, P, P]
        lib.oracle_linear_backward.restype = None
        lib.oracle_linear_backward.argtypes = [I64, I64, I64, P, P, P, P, P, P]
        lib.oracle_linear_sharded.restype = None
        lib.oracle_linear_sharded.argtypes = [I64, I64, I64, ctypes.c_int, ctypes.c_int, P, P, P, P, P, P, P]
        lib.oracle_qkv_column.restype = I64
        lib.oracle_qkv_column.argtypes = [ctypes.c_int, I64, I64, I64, I64, I64]
        lib.oracle_mlp_seq_parallel.restype = None
        lib.oracle_mlp_seq_parallel.argtypes = [I64, I64, I64, ctypes.c_int, P, P, P, P, P, P, P, P, P, P]
        _lib = lib
        return lib


def _f64(x) -> Optional[np.ndarray]:
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def gelu(x: float) -> float:
    return float(_load().oracle_gelu(float(x)))


def gelu_grad(x: float) -> float:
    return float(_load().oracle_gelu_grad(float(x)))


def mlp_forward(X, A, bA, B, bB) -> Dict[str, np.ndarray]:
    """U = X A + bA, Y = GeLU(U), Z = Y B + bB (unsharded), all float64."""
    X, A, bA, B, bB = map(_f64, (X, A, bA, B, bB))
    T, h = X.shape
    f = A.shape[1]
    U = np.empty((T, f)); Y = np.empty((T, f)); Z = np.empty((T, h))
    _load().oracle_mlp_forward(T, h, f, _ptr(X), _ptr(A), _ptr(bA), _ptr(B), _ptr(bB),
                               _ptr(U), _ptr(Y), _ptr(Z))
    return {"U": U, "Y": Y, "Z": Z}


def mlp_backward(X, A, bA, B, dZ, want: Sequence[str] = ("dX", "dA", "dbA", "dB", "dbB")) -> Dict[str, np.ndarray]:
    """Chain-rule gradients of the unsharded block for upstream gradient dZ."""
    X, A, bA, B, dZ = map(_f64, (X, A, bA, B, dZ))
    T, h = X.shape
    f = A.shape[1]
    shapes = {"dX": (T, h), "dA": (h, f), "dbA": (f,), "dB": (f, h), "dbB": (h,)}
    out = {k: np.empty(shapes[k]) for k in want}
    _load().oracle_mlp_backward(T, h, f, _ptr(X), _ptr(A), _ptr(bA), _ptr(B), _ptr(dZ),
                                _ptr(out.get("dX")), _ptr(out.get("dA")), _ptr(out.get("dbA")),
                                _ptr(out.get("dB")), _ptr(out.get("dbB")))
    return out


def mlp_backward_cols(X, A, bA, B, dZ, cols) -> Dict[str, np.ndarray]:
    """dA[:, cols], dbA[cols], dB[cols, :] of the unsharded block."""
    X, A, bA, B, dZ = map(_f64, (X, A, bA, B, dZ))
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    T, h = X.shape
    f = A.shape[1]
    n = len(cols)
    dA = np.empty((h, n)); dbA = np.empty((n,)); dB = np.empty((n, h))
    _load().oracle_mlp_backward_cols(T, h, f, _ptr(X), _ptr(A), _ptr(bA), _ptr(B), _ptr(dZ),
                                     n, _ptr(cols), _ptr(dA), _ptr(dbA), _ptr(dB))
    return {"dA": dA, "dbA": dbA, "dB": dB}


def bias_grad(dZ) -> np.ndarray:
    """dbB = sum over tokens of dZ."""
    dZ = _f64(dZ)
    T, h = dZ.shape
    out = np.empty((h,))
    _load().oracle_bias_grad(T, h, _ptr(dZ), _ptr(out))
    return out


def mlp_sharded(X, A, bA, B, bB, dZ, t: int) -> Dict[str, np.ndarray]:
    """The block computed shard by shard (column/row partition, g and f*)."""
    X, A, bA, B, bB, dZ = map(_f64, (X, A, bA, B, bB, dZ))
    T, h = X.shape
    f = A.shape[1]
    if f % t:
        raise ValueError("f must divide by t")
    Z = np.empty((T, h)); dX = np.empty((T, h)); dA = np.empty((h, f)); dB = np.empty((f, h))
    _load().oracle_mlp_sharded(T, h, f, t, _ptr(X), _ptr(A), _ptr(bA), _ptr(B), _ptr(bB), _ptr(dZ),
                               _ptr(Z), _ptr(dX), _ptr(dA), _ptr(dB))
    return {"Z": Z, "dX": dX, "dA": dA, "dB": dB}


def ce(H, E, targets, v_valid: int, grad_scale: float = 1.0, grads: bool = True,
       want_dE: bool = True) -> Dict[str, np.ndarray]:
    """Unsharded softmax cross-entropy over l = H E^T restricted to ids < v_valid."""
    H, E = _f64(H), _f64(E)
    tg = np.ascontiguousarray(np.asarray(targets, dtype=np.int32))
    T, h = H.shape
    v_pad = E.shape[0]
    loss = np.empty((T,)); lse = np.empty((T,))
    dH = np.empty((T, h)) if grads else None
    dE = np.empty((v_pad, h)) if (grads and want_dE) else None
    _load().oracle_ce(T, h, v_pad, v_valid, _ptr(H), _ptr(E), _ptr(tg), float(grad_scale),
                      _ptr(loss), _ptr(lse), _ptr(dH), _ptr(dE))
    return {"loss": loss, "lse": lse, "dH": dH, "dE": dE}


def ce_sharded(H, E, targets, v_valid: int, t: int) -> Dict[str, np.ndarray]:
    """Per-shard (max, sum-exp, target logit) and the combined loss."""
    H, E = _f64(H), _f64(E)
    tg = np.ascontiguousarray(np.asarray(targets, dtype=np.int32))
    T, h = H.shape
    v_pad = E.shape[0]
    if v_pad % t:
        raise ValueError("v_pad must divide by t")
    m = np.empty((t, T)); s = np.empty((t, T)); tau = np.empty((T,)); loss = np.empty((T,))
    _load().oracle_ce_sharded(T, h, v_pad, v_valid, t, _ptr(H), _ptr(E), _ptr(tg),
                              _ptr(m), _ptr(s), _ptr(tau), _ptr(loss))
    return {"m": m, "s": s, "tau": tau, "loss": loss}


def swish(x: float) -> float:
    return float(_load().oracle_swish(float(x)))


def swish_grad(x: float) -> float:
    return float(_load().oracle_swish_grad(float(x)))


def swiglu_forward(X, W1, b1, W2, b2) -> Dict[str, np.ndarray]:
    """GU = X W1 + b1 ([G | Up]), Y = Swish(G) * Up, Z = Y W2 + b2 (unsharded)."""
    X, W1, b1, W2, b2 = map(_f64, (X, W1, b1, W2, b2))
    T, h = X.shape
    f = W1.shape[1] // 2
    GU = np.empty((T, 2 * f)); Y = np.empty((T, f)); Z = np.empty((T, h))
    _load().oracle_swiglu_forward(T, h, f, _ptr(X), _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2),
                                  _ptr(GU), _ptr(Y), _ptr(Z))
    return {"GU": GU, "Y": Y, "Z": Z}


def swiglu_backward(X, W1, b1, W2, dZ,
                    want: Sequence[str] = ("dX", "dW1", "db1", "dW2", "db2")) -> Dict[str, np.ndarray]:
    """Chain-rule gradients of the unsharded SwiGLU block for upstream dZ."""
    X, W1, b1, W2, dZ = map(_f64, (X, W1, b1, W2, dZ))
    T, h = X.shape
    f = W1.shape[1] // 2
    shapes = {"dX": (T, h), "dW1": (h, 2 * f), "db1": (2 * f,), "dW2": (f, h), "db2": (h,)}
    out = {k: np.empty(shapes[k]) for k in want}
    _load().oracle_swiglu_backward(T, h, f, _ptr(X), _ptr(W1), _ptr(b1), _ptr(W2), _ptr(dZ),
                                   _ptr(out.get("dX")), _ptr(out.get("dW1")), _ptr(out.get("db1")),
                                   _ptr(out.get("dW2")), _ptr(out.get("db2")))
    return out


def swiglu_backward_cols(X, W1, b1, W2, dZ, cols) -> Dict[str, np.ndarray]:
    """dW1[:, cols] (gate), dW1[:, f + cols] (up), db1 at both, dW2[cols, :]."""
    X, W1, b1, W2, dZ = map(_f64, (X, W1, b1, W2, dZ))
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    T, h = X.shape
    f = W1.shape[1] // 2
    n = len(cols)
    dWg = np.empty((h, n)); dWu = np.empty((h, n)); dbg = np.empty((n,)); dbu = np.empty((n,))
    dW2 = np.empty((n, h))
    _load().oracle_swiglu_backward_cols(T, h, f, _ptr(X), _ptr(W1), _ptr(b1), _ptr(W2), _ptr(dZ),
                                        n, _ptr(cols), _ptr(dWg), _ptr(dWu), _ptr(dbg), _ptr(dbu), _ptr(dW2))
    return {"dW1_gate": dWg, "dW1_up": dWu, "db1_gate": dbg, "db1_up": dbu, "dW2": dW2}


def swiglu_sharded(X, W1, b1, W2, b2, dZ, t: int) -> Dict[str, np.ndarray]:
    """The SwiGLU block computed shard by shard (gate/up columns, W2 rows)."""
    X, W1, b1, W2, b2, dZ = map(_f64, (X, W1, b1, W2, b2, dZ))
    T, h = X.shape
    f = W1.shape[1] // 2
    if f % t:
        raise ValueError("f must divide by t")
    Z = np.empty((T, h)); dX = np.empty((T, h)); dW1 = np.empty((h, 2 * f)); dW2 = np.empty((f, h))
    _load().oracle_swiglu_sharded(T, h, f, t, _ptr(X), _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2), _ptr(dZ),
                                  _ptr(Z), _ptr(dX), _ptr(dW1), _ptr(dW2))
    return {"Z": Z, "dX": dX, "dW1": dW1, "dW2": dW2}


def linear_forward(X, W, b=None) -> np.ndarray:
    """Y = X W + b."""
    X, W, b = map(_f64, (X, W, b))
    T, n_in = X.shape
    n_out = W.shape[1]
    Y = np.empty((T, n_out))
    _load().oracle_linear_forward(T, n_in, n_out, _ptr(X), _ptr(W), _ptr(b), _ptr(Y))
    return Y


def linear_backward(X, W, dY, want: Sequence[str] = ("dX", "dW", "db")) -> Dict[str, np.ndarray]:
    """dX = dY W^T, dW = X^T dY, db = sum over tokens of dY."""
    X, W, dY = map(_f64, (X, W, dY))
    T, n_in = X.shape
    n_out = W.shape[1]
    shapes = {"dX": (T, n_in), "dW": (n_in, n_out), "db": (n_out,)}
    out = {k: np.empty(shapes[k]) for k in want}
    _load().oracle_linear_backward(T, n_in, n_out, _ptr(X), _ptr(W), _ptr(dY), _ptr(out.get("dX")),
                                   _ptr(out.get("dW")), _ptr(out.get("db")))
    return out


def linear_sharded(X, W, b, dY, t: int, mode: str) -> Dict[str, np.ndarray]:
    """The linear layer computed shard by shard; mode "column" or "row"."""
    X, W, b, dY = map(_f64, (X, W, b, dY))
    T, n_in = X.shape
    n_out = W.shape[1]
    m = {"column": 0, "row": 1}[mode]
    if (n_out if m == 0 else n_in) % t:
        raise ValueError("the split dimension must divide by t")
    Y = np.empty((T, n_out)); dX = np.empty((T, n_in)); dW = np.empty((n_in, n_out))
    _load().oracle_linear_sharded(T, n_in, n_out, t, m, _ptr(X), _ptr(W), _ptr(b), _ptr(dY),
                                  _ptr(Y), _ptr(dX), _ptr(dW))
    return {"Y": Y, "dX": dX, "dW": dW}


def qkv_column(kind: str, head: int, j: int, n_q: int, n_kv: int, d: int) -> int:
    """Column of the fused QKV projection holding element j of a query,
    key or value head (layout grouped by key/value head)."""
    k = {"q": 0, "k": 1, "v": 2}[kind]
    return int(_load().oracle_qkv_column(k, head, j, n_q, n_kv, d))


def qkv_columns(kind: str, n_q: int, n_kv: int, d: int) -> np.ndarray:
    """[heads, d] array of the columns of every head of one kind."""
    n = n_q if kind == "q" else n_kv
    return np.array([[qkv_column(kind, hh, j, n_q, n_kv, d) for j in range(d)] for hh in range(n)],
                    dtype=np.int64)


def _ptr_array(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def mlp_seq_parallel(X_chunks, A, bA, B, bB, dZ_chunks) -> Dict[str, object]:
    """The block with sequence-parallel entry (all-gather of the X chunks) and
    exit (reduce-scatter into Z chunks), and the mirrored backward."""
    Xc = [_f64(x) for x in X_chunks]
    dZc = [_f64(x) for x in dZ_chunks]
    A, bA, B, bB = map(_f64, (A, bA, B, bB))
    t = len(Xc)
    rows, h = Xc[0].shape
    f = A.shape[1]
    if any(x.shape != (rows, h) for x in Xc + dZc) or len(dZc) != t or f % t:
        raise ValueError("t chunks of equal shape and f % t == 0 required")
    Zc = [np.empty((rows, h)) for _ in range(t)]
    dXc = [np.empty((rows, h)) for _ in range(t)]
    dA = np.empty((h, f)); dB = np.empty((f, h))
    _load().oracle_mlp_seq_parallel(rows * t, h, f, t, _ptr_array(Xc), _ptr(A), _ptr(bA), _ptr(B), _ptr(bB),
                                    _ptr_array(dZc), _ptr_array(Zc), _ptr_array(dXc), _ptr(dA), _ptr(dB))
    return {"Z": Zc, "dX": dXc, "dA": dA, "dB": dB}
