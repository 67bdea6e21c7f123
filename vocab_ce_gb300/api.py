"""Python face of libtpce: the same calls as the C ABI, on torch tensors.

Only argument marshalling happens here (checking devices and dtypes,
allocating outputs and workspace with torch, passing raw pointers and the
current CUDA stream). Every arithmetic step runs in the library's kernels.
"""

from __future__ import annotations

import ctypes
from typing import Dict, Optional

import torch

from ._lib import TPCE_BF16, TPCE_COLUMN_PARALLEL, TPCE_F32, TPCE_ROW_PARALLEL, TpceError, check, lib

_DT = {torch.bfloat16: TPCE_BF16, torch.float32: TPCE_F32}


def _ptr(x: Optional[torch.Tensor]):
    return None if x is None else ctypes.c_void_p(x.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(x: torch.Tensor, name: str, dtype=None, shape=None):
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if x.device.index != torch.cuda.current_device():
        # the library launches on the current device's stream
        raise ValueError(f"{name} is on {x.device}, not on the current device cuda:{torch.cuda.current_device()}")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous (row-major)")
    if dtype is not None and x.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {x.dtype}")
    if shape is not None and tuple(x.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(x.shape)}")


def _workspace(nbytes: int, device, ws: Optional[torch.Tensor]) -> Optional[torch.Tensor]:
    if nbytes == 0:
        return ws
    if ws is not None and ws.numel() * ws.element_size() >= nbytes:
        return ws
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def tail_workspace_bytes() -> int:
    """Workspace with which the bf16 forward calls split a short last wave of tiles."""
    return int(lib().tpce_tail_workspace_bytes())


def _fwd_workspace(dt, T: int, full_bytes, dev, ws: Optional[torch.Tensor]) -> Optional[torch.Tensor]:
    """The forward's workspace: required on the fp32 path (transposed operands),
    optional on the bf16 path, where it lets short last waves of tiles split."""
    if T == 0:
        return None
    if dt == torch.float32:
        return _workspace(full_bytes(), dev, ws)
    return _workspace(tail_workspace_bytes(), dev, ws)


def pad_vocab(v: int, t: int, divisor: int = 128) -> int:
    """Smallest multiple of divisor * t that is >= v (Megatron's vocabulary padding)."""
    r = lib().tpce_pad_vocab(v, t, divisor)
    if r < 0:
        raise ValueError("pad_vocab: v >= 0, t >= 1 and divisor >= 1 required")
    return int(r)


def mlp_workspace_bytes(T: int, h: int, f: int, t: int, dtype=torch.bfloat16) -> int:
    return int(lib().tpce_mlp_workspace_bytes(T, h, f, t, _DT[dtype]))


def ce_workspace_bytes(T: int, h: int, v_pad: int, t: int, grads: bool = True, dtype=torch.bfloat16) -> int:
    return int(lib().tpce_ce_workspace_bytes(T, h, v_pad, t, _DT[dtype], 1 if grads else 0))


def tp_mlp_forward(X: torch.Tensor, A: torch.Tensor, B: torch.Tensor, t: int,
                   bA: Optional[torch.Tensor] = None, bB: Optional[torch.Tensor] = None,
                   out: Optional[Dict[str, torch.Tensor]] = None, ws: Optional[torch.Tensor] = None,
                   stream=None) -> Dict[str, torch.Tensor]:
    """Z = sum_i GeLU(X A_i + bA_i) B_i + bB over t shards; returns Z, U, Y."""
    T, h = X.shape
    f = A.shape[1]
    dt = X.dtype
    for name, x, shp in (("X", X, (T, h)), ("A", A, (h, f)), ("B", B, (f, h))):
        _need(x, name, dt, shp)
    for name, b, n in (("bA", bA, f), ("bB", bB, h)):
        if b is not None:
            _need(b, name, torch.float32, (n,))
    out = dict(out or {})
    Z = out.get("Z") if out.get("Z") is not None else torch.empty((T, h), dtype=dt, device=X.device)
    U = out.get("U") if out.get("U") is not None else torch.empty((T, f), dtype=dt, device=X.device)
    Y = out.get("Y") if out.get("Y") is not None else torch.empty((T, f), dtype=dt, device=X.device)
    w = _fwd_workspace(dt, T, lambda: mlp_workspace_bytes(T, h, f, t, dt), X.device, ws)
    st = lib().tp_mlp_forward(_ptr(X), _ptr(A), _ptr(bA), _ptr(B), _ptr(bB), T, h, f, t, _DT[dt],
                              _ptr(Z), _ptr(U), _ptr(Y), _ptr(w),
                              0 if w is None else w.numel() * w.element_size(), _stream(stream))
    check(st, "tp_mlp_forward")
    return {"Z": Z, "U": U, "Y": Y}


def tp_mlp_backward(dZ: torch.Tensor, X: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                    U: torch.Tensor, Y: torch.Tensor, t: int, bias_grads: bool = True,
                    out: Optional[Dict[str, torch.Tensor]] = None, ws: Optional[torch.Tensor] = None,
                    stream=None) -> Dict[str, torch.Tensor]:
    """dX (f* sum over shards), dA, dB and optionally dbA, dbB."""
    T, h = X.shape
    f = A.shape[1]
    dt = X.dtype
    for name, x, shp in (("dZ", dZ, (T, h)), ("X", X, (T, h)), ("A", A, (h, f)), ("B", B, (f, h)),
                         ("U", U, (T, f)), ("Y", Y, (T, f))):
        _need(x, name, dt, shp)
    out = dict(out or {})
    dev = X.device

    def get(k, shp, d):
        return out.get(k) if out.get(k) is not None else torch.empty(shp, dtype=d, device=dev)

    dX, dA, dB = get("dX", (T, h), dt), get("dA", (h, f), dt), get("dB", (f, h), dt)
    dbA = get("dbA", (f,), torch.float32) if bias_grads else None
    dbB = get("dbB", (h,), torch.float32) if bias_grads else None
    nbytes = mlp_workspace_bytes(T, h, f, t, dt) if T > 0 else 0
    w = _workspace(nbytes, dev, ws)
    st = lib().tp_mlp_backward(_ptr(dZ), _ptr(X), _ptr(A), _ptr(B), _ptr(U), _ptr(Y), T, h, f, t, _DT[dt],
                               _ptr(dX), _ptr(dA), _ptr(dbA), _ptr(dB), _ptr(dbB), _ptr(w),
                               0 if w is None else w.numel() * w.element_size(), _stream(stream))
    check(st, "tp_mlp_backward")
    res = {"dX": dX, "dA": dA, "dB": dB}
    if bias_grads:
        res.update(dbA=dbA, dbB=dbB)
    return res


def swiglu_workspace_bytes(T: int, h: int, f: int, t: int, dtype=torch.bfloat16) -> int:
    return int(lib().tpce_swiglu_workspace_bytes(T, h, f, t, _DT[dtype]))


def tp_swiglu_forward(X: torch.Tensor, W1: torch.Tensor, W2: torch.Tensor, t: int,
                      b1: Optional[torch.Tensor] = None, b2: Optional[torch.Tensor] = None,
                      out: Optional[Dict[str, torch.Tensor]] = None, ws: Optional[torch.Tensor] = None,
                      stream=None) -> Dict[str, torch.Tensor]:
    """Z = sum_i (Swish(X Wg_i + bg_i) * (X Wu_i + bu_i)) W2_i + b2 over t shards,
    W1 = [W_gate | W_up] of shape [h, 2f]; returns Z, GU = [G | Up], Y."""
    T, h = X.shape
    f = W2.shape[0]
    dt = X.dtype
    for name, x, shp in (("X", X, (T, h)), ("W1", W1, (h, 2 * f)), ("W2", W2, (f, h))):
        _need(x, name, dt, shp)
    for name, b, n in (("b1", b1, 2 * f), ("b2", b2, h)):
        if b is not None:
            _need(b, name, torch.float32, (n,))
    out = dict(out or {})
    Z = out.get("Z") if out.get("Z") is not None else torch.empty((T, h), dtype=dt, device=X.device)
    GU = out.get("GU") if out.get("GU") is not None else torch.empty((T, 2 * f), dtype=dt, device=X.device)
    Y = out.get("Y") if out.get("Y") is not None else torch.empty((T, f), dtype=dt, device=X.device)
    w = _fwd_workspace(dt, T, lambda: swiglu_workspace_bytes(T, h, f, t, dt), X.device, ws)
    st = lib().tp_swiglu_forward(_ptr(X), _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2), T, h, f, t, _DT[dt],
                                 _ptr(Z), _ptr(GU), _ptr(Y), _ptr(w),
                                 0 if w is None else w.numel() * w.element_size(), _stream(stream))
    check(st, "tp_swiglu_forward")
    return {"Z": Z, "GU": GU, "Y": Y}


def tp_swiglu_backward(dZ: torch.Tensor, X: torch.Tensor, W1: torch.Tensor, W2: torch.Tensor,
                       GU: torch.Tensor, Y: torch.Tensor, t: int, bias_grads: bool = True,
                       out: Optional[Dict[str, torch.Tensor]] = None, ws: Optional[torch.Tensor] = None,
                       stream=None) -> Dict[str, torch.Tensor]:
    """dX (f* sum over shards), dW1, dW2 and optionally db1, db2."""
    T, h = X.shape
    f = W2.shape[0]
    dt = X.dtype
    for name, x, shp in (("dZ", dZ, (T, h)), ("X", X, (T, h)), ("W1", W1, (h, 2 * f)), ("W2", W2, (f, h)),
                         ("GU", GU, (T, 2 * f)), ("Y", Y, (T, f))):
        _need(x, name, dt, shp)
    out = dict(out or {})
    dev = X.device

    def get(k, shp, d):
        return out.get(k) if out.get(k) is not None else torch.empty(shp, dtype=d, device=dev)

    dX, dW1, dW2 = get("dX", (T, h), dt), get("dW1", (h, 2 * f), dt), get("dW2", (f, h), dt)
    db1 = get("db1", (2 * f,), torch.float32) if bias_grads else None
    db2 = get("db2", (h,), torch.float32) if bias_grads else None
    nbytes = swiglu_workspace_bytes(T, h, f, t, dt) if T > 0 else 0
    w = _workspace(nbytes, dev, ws)
    st = lib().tp_swiglu_backward(_ptr(dZ), _ptr(X), _ptr(W1), _ptr(W2), _ptr(GU), _ptr(Y), T, h, f, t, _DT[dt],
                                  _ptr(dX), _ptr(dW1), _ptr(db1), _ptr(dW2), _ptr(db2), _ptr(w),
                                  0 if w is None else w.numel() * w.element_size(), _stream(stream))
    check(st, "tp_swiglu_backward")
    res = {"dX": dX, "dW1": dW1, "dW2": dW2}
    if bias_grads:
        res.update(db1=db1, db2=db2)
    return res


def _ptr_list(xs):
    return (ctypes.c_void_p * len(xs))(*[x.data_ptr() for x in xs])


def _chunks(xs, name, t, rows, h, dt, dev):
    if len(xs) != t:
        raise ValueError(f"{name}: {t} sequence chunks expected, got {len(xs)}")
    for i, x in enumerate(xs):
        _need(x, f"{name}[{i}]", dt, (rows, h))
        if x.device != dev:
            raise ValueError(f"{name}[{i}] is on {x.device}, expected {dev}")


def _mlp_sp(glu, X_chunks, W1, W2, t, b1, b2, out, ws, stream):
    rows, h = X_chunks[0].shape
    T = rows * t
    f = W2.shape[0]
    fw = 2 * f if glu else f
    dt, dev = X_chunks[0].dtype, X_chunks[0].device
    _chunks(X_chunks, "X_chunks", t, rows, h, dt, dev)
    _need(W1, "W1" if glu else "A", dt, (h, fw))
    _need(W2, "W2" if glu else "B", dt, (f, h))
    for name, b, n in (("b1", b1, fw), ("b2", b2, h)):
        if b is not None:
            _need(b, name, torch.float32, (n,))
    out = dict(out or {})
    Zc = out.get("Z")
    if Zc is None:
        Zc = [torch.empty((rows, h), dtype=dt, device=dev) for _ in range(t)]
    if isinstance(Zc, torch.Tensor):
        raise ValueError("out['Z'] must be a list of t sequence-chunk tensors")
    _chunks(Zc, "Z", t, rows, h, dt, dev)
    ukey = "GU" if glu else "U"
    U = out.get(ukey) if out.get(ukey) is not None else torch.empty((T, fw), dtype=dt, device=dev)
    Y = out.get("Y") if out.get("Y") is not None else torch.empty((T, f), dtype=dt, device=dev)
    q = swiglu_workspace_bytes if glu else mlp_workspace_bytes
    w = _fwd_workspace(dt, T, lambda: q(T, h, f, t, dt), dev, ws)
    xp, zp = _ptr_list(X_chunks), _ptr_list(Zc)
    fn = lib().tp_swiglu_forward_sp if glu else lib().tp_mlp_forward_sp
    st = fn(xp, _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2), T, h, f, t, _DT[dt], zp, _ptr(U), _ptr(Y), _ptr(w),
            0 if w is None else w.numel() * w.element_size(), _stream(stream))
    check(st, "tp_swiglu_forward_sp" if glu else "tp_mlp_forward_sp")
    return {"Z": Zc, ukey: U, "Y": Y}


def _mlp_sp_bwd(glu, dZ_chunks, X_chunks, W1, W2, U, Y, t, bias_grads, out, ws, stream):
    rows, h = X_chunks[0].shape
    T = rows * t
    f = W2.shape[0]
    fw = 2 * f if glu else f
    dt, dev = X_chunks[0].dtype, X_chunks[0].device
    _chunks(X_chunks, "X_chunks", t, rows, h, dt, dev)
    _chunks(dZ_chunks, "dZ_chunks", t, rows, h, dt, dev)
    for name, x, shp in (("W1" if glu else "A", W1, (h, fw)), ("W2" if glu else "B", W2, (f, h)),
                         ("GU" if glu else "U", U, (T, fw)), ("Y", Y, (T, f))):
        _need(x, name, dt, shp)
    out = dict(out or {})
    k1, k2, kb1, kb2 = ("dW1", "dW2", "db1", "db2") if glu else ("dA", "dB", "dbA", "dbB")
    dXc = out.get("dX")
    if dXc is None:
        dXc = [torch.empty((rows, h), dtype=dt, device=dev) for _ in range(t)]
    if isinstance(dXc, torch.Tensor):
        raise ValueError("out['dX'] must be a list of t sequence-chunk tensors")
    _chunks(dXc, "dX", t, rows, h, dt, dev)

    def get(k, shp, d):
        return out.get(k) if out.get(k) is not None else torch.empty(shp, dtype=d, device=dev)

    d1, d2 = get(k1, (h, fw), dt), get(k2, (f, h), dt)
    db1 = get(kb1, (fw,), torch.float32) if bias_grads else None
    db2 = get(kb2, (h,), torch.float32) if bias_grads else None
    q = swiglu_workspace_bytes if glu else mlp_workspace_bytes
    w = _workspace(q(T, h, f, t, dt) if T > 0 else 0, dev, ws)
    dzp, xp, dxp = _ptr_list(dZ_chunks), _ptr_list(X_chunks), _ptr_list(dXc)
    fn = lib().tp_swiglu_backward_sp if glu else lib().tp_mlp_backward_sp
    st = fn(dzp, xp, _ptr(W1), _ptr(W2), _ptr(U), _ptr(Y), T, h, f, t, _DT[dt], dxp, _ptr(d1), _ptr(db1), _ptr(d2),
            _ptr(db2), _ptr(w), 0 if w is None else w.numel() * w.element_size(), _stream(stream))
    check(st, "tp_swiglu_backward_sp" if glu else "tp_mlp_backward_sp")
    res = {"dX": dXc, k1: d1, k2: d2}
    if bias_grads:
        res.update({kb1: db1, kb2: db2})
    return res


def tp_mlp_forward_sp(X_chunks, A: torch.Tensor, B: torch.Tensor, t: int, bA: Optional[torch.Tensor] = None,
                      bB: Optional[torch.Tensor] = None, out=None, ws: Optional[torch.Tensor] = None, stream=None):
    """The GeLU block with sequence-parallel entry and exit: X and Z as t
    sequence chunks [T/t, h] (lists of tensors); returns Z (list), U, Y."""
    return _mlp_sp(False, X_chunks, A, B, t, bA, bB, out, ws, stream)


def tp_mlp_backward_sp(dZ_chunks, X_chunks, A: torch.Tensor, B: torch.Tensor, U: torch.Tensor, Y: torch.Tensor,
                       t: int, bias_grads: bool = True, out=None, ws: Optional[torch.Tensor] = None, stream=None):
    """Backward of tp_mlp_forward_sp: dX (list of chunks), dA, dB, dbA, dbB."""
    return _mlp_sp_bwd(False, dZ_chunks, X_chunks, A, B, U, Y, t, bias_grads, out, ws, stream)


def tp_swiglu_forward_sp(X_chunks, W1: torch.Tensor, W2: torch.Tensor, t: int, b1: Optional[torch.Tensor] = None,
                         b2: Optional[torch.Tensor] = None, out=None, ws: Optional[torch.Tensor] = None, stream=None):
    """The SwiGLU block with sequence-parallel entry and exit; returns Z (list), GU, Y."""
    return _mlp_sp(True, X_chunks, W1, W2, t, b1, b2, out, ws, stream)


def tp_swiglu_backward_sp(dZ_chunks, X_chunks, W1: torch.Tensor, W2: torch.Tensor, GU: torch.Tensor,
                          Y: torch.Tensor, t: int, bias_grads: bool = True, out=None,
                          ws: Optional[torch.Tensor] = None, stream=None):
    """Backward of tp_swiglu_forward_sp: dX (list of chunks), dW1, dW2, db1, db2."""
    return _mlp_sp_bwd(True, dZ_chunks, X_chunks, W1, W2, GU, Y, t, bias_grads, out, ws, stream)


_PAR = {"column": TPCE_COLUMN_PARALLEL, "row": TPCE_ROW_PARALLEL}


def _wsize(w: Optional[torch.Tensor]) -> int:
    return 0 if w is None else w.numel() * w.element_size()


def linear_workspace_bytes(T: int, n_in: int, n_out: int, t: int, parallel: str = "column",
                           dtype=torch.bfloat16) -> int:
    return int(lib().tpce_linear_workspace_bytes(T, n_in, n_out, t, _PAR[parallel], _DT[dtype]))


def tp_linear_forward(X: torch.Tensor, W: torch.Tensor, t: int, parallel: str = "column",
                      b: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                      ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Y = X W + b over t shards of W's columns ("column") or rows ("row")."""
    T, n_in = X.shape
    n_out = W.shape[1]
    dt = X.dtype
    _need(X, "X", dt, (T, n_in))
    _need(W, "W", dt, (n_in, n_out))
    if b is not None:
        _need(b, "b", torch.float32, (n_out,))
    Y = out if out is not None else torch.empty((T, n_out), dtype=dt, device=X.device)
    w = _fwd_workspace(dt, T, lambda: linear_workspace_bytes(T, n_in, n_out, t, parallel, dt), X.device, ws)
    st = lib().tp_linear_forward(_ptr(X), _ptr(W), _ptr(b), T, n_in, n_out, t, _PAR[parallel], _DT[dt], _ptr(Y),
                                 _ptr(w), _wsize(w), _stream(stream))
    check(st, "tp_linear_forward")
    return Y


def tp_linear_backward(dY: torch.Tensor, X: torch.Tensor, W: torch.Tensor, t: int, parallel: str = "column",
                       bias_grad: bool = True, out: Optional[Dict[str, torch.Tensor]] = None,
                       ws: Optional[torch.Tensor] = None, stream=None) -> Dict[str, torch.Tensor]:
    """dX = dY W^T, dW = X^T dY and optionally db = sum over tokens of dY."""
    T, n_in = X.shape
    n_out = W.shape[1]
    dt = X.dtype
    for name, x, shp in (("dY", dY, (T, n_out)), ("X", X, (T, n_in)), ("W", W, (n_in, n_out))):
        _need(x, name, dt, shp)
    out = dict(out or {})
    dev = X.device
    dX = out.get("dX") if out.get("dX") is not None else torch.empty((T, n_in), dtype=dt, device=dev)
    dW = out.get("dW") if out.get("dW") is not None else torch.empty((n_in, n_out), dtype=dt, device=dev)
    db = None
    if bias_grad:
        db = out.get("db") if out.get("db") is not None else torch.empty(n_out, dtype=torch.float32, device=dev)
    w = _workspace(linear_workspace_bytes(T, n_in, n_out, t, parallel, dt) if T > 0 else 0, dev, ws)
    st = lib().tp_linear_backward(_ptr(dY), _ptr(X), _ptr(W), T, n_in, n_out, t, _PAR[parallel], _DT[dt],
                                  _ptr(dX), _ptr(dW), _ptr(db), _ptr(w), _wsize(w), _stream(stream))
    check(st, "tp_linear_backward")
    res = {"dX": dX, "dW": dW}
    if bias_grad:
        res["db"] = db
    return res


def attn_workspace_bytes(T: int, h: int, n_heads: int, n_kv_heads: int, head_dim: int, t: int,
                         dtype=torch.bfloat16) -> int:
    return int(lib().tpce_attn_workspace_bytes(T, h, n_heads, n_kv_heads, head_dim, t, _DT[dtype]))


def tp_attn_qkv_forward(X: torch.Tensor, Wqkv: torch.Tensor, n_heads: int, n_kv_heads: int, head_dim: int, t: int,
                        bqkv: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                        ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """QKV = X Wqkv + bqkv, column-parallel by (grouped-query) heads."""
    T, h = X.shape
    n = (n_heads + 2 * n_kv_heads) * head_dim
    dt = X.dtype
    _need(X, "X", dt, (T, h))
    _need(Wqkv, "Wqkv", dt, (h, n))
    if bqkv is not None:
        _need(bqkv, "bqkv", torch.float32, (n,))
    QKV = out if out is not None else torch.empty((T, n), dtype=dt, device=X.device)
    w = _fwd_workspace(dt, T, lambda: attn_workspace_bytes(T, h, n_heads, n_kv_heads, head_dim, t, dt), X.device, ws)
    st = lib().tp_attn_qkv_forward(_ptr(X), _ptr(Wqkv), _ptr(bqkv), T, h, n_heads, n_kv_heads, head_dim, t, _DT[dt],
                                   _ptr(QKV), _ptr(w), _wsize(w), _stream(stream))
    check(st, "tp_attn_qkv_forward")
    return QKV


def tp_attn_qkv_backward(dQKV: torch.Tensor, X: torch.Tensor, Wqkv: torch.Tensor, n_heads: int, n_kv_heads: int,
                         head_dim: int, t: int, bias_grad: bool = True, out: Optional[Dict[str, torch.Tensor]] = None,
                         ws: Optional[torch.Tensor] = None, stream=None) -> Dict[str, torch.Tensor]:
    """dX (f* sum over shards), dWqkv and optionally dbqkv."""
    T, h = X.shape
    n = (n_heads + 2 * n_kv_heads) * head_dim
    dt = X.dtype
    for name, x, shp in (("dQKV", dQKV, (T, n)), ("X", X, (T, h)), ("Wqkv", Wqkv, (h, n))):
        _need(x, name, dt, shp)
    out = dict(out or {})
    dev = X.device
    dX = out.get("dX") if out.get("dX") is not None else torch.empty((T, h), dtype=dt, device=dev)
    dW = out.get("dWqkv") if out.get("dWqkv") is not None else torch.empty((h, n), dtype=dt, device=dev)
    db = None
    if bias_grad:
        db = out.get("dbqkv") if out.get("dbqkv") is not None else torch.empty(n, dtype=torch.float32, device=dev)
    w = _workspace(attn_workspace_bytes(T, h, n_heads, n_kv_heads, head_dim, t, dt) if T > 0 else 0, dev, ws)
    st = lib().tp_attn_qkv_backward(_ptr(dQKV), _ptr(X), _ptr(Wqkv), T, h, n_heads, n_kv_heads, head_dim, t,
                                    _DT[dt], _ptr(dX), _ptr(dW), _ptr(db), _ptr(w), _wsize(w), _stream(stream))
    check(st, "tp_attn_qkv_backward")
    res = {"dX": dX, "dWqkv": dW}
    if bias_grad:
        res["dbqkv"] = db
    return res


def tp_attn_out_forward(O: torch.Tensor, Wo: torch.Tensor, n_heads: int, head_dim: int, t: int,
                        bo: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                        ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Z = sum_i O_i Wo_i + bo: the row-parallel output projection."""
    T, hq = O.shape
    h = Wo.shape[1]
    dt = O.dtype
    _need(O, "O", dt, (T, n_heads * head_dim))
    _need(Wo, "Wo", dt, (n_heads * head_dim, h))
    if bo is not None:
        _need(bo, "bo", torch.float32, (h,))
    Z = out if out is not None else torch.empty((T, h), dtype=dt, device=O.device)
    w = _fwd_workspace(dt, T, lambda: linear_workspace_bytes(T, hq, h, t, "row", dt), O.device, ws)
    st = lib().tp_attn_out_forward(_ptr(O), _ptr(Wo), _ptr(bo), T, h, n_heads, head_dim, t, _DT[dt], _ptr(Z),
                                   _ptr(w), _wsize(w), _stream(stream))
    check(st, "tp_attn_out_forward")
    return Z


def tp_attn_out_backward(dZ: torch.Tensor, O: torch.Tensor, Wo: torch.Tensor, n_heads: int, head_dim: int, t: int,
                         bias_grad: bool = True, out: Optional[Dict[str, torch.Tensor]] = None,
                         ws: Optional[torch.Tensor] = None, stream=None) -> Dict[str, torch.Tensor]:
    """dO (each shard's own head columns), dWo and optionally dbo."""
    T, hq = O.shape
    h = Wo.shape[1]
    dt = O.dtype
    for name, x, shp in (("dZ", dZ, (T, h)), ("O", O, (T, n_heads * head_dim)), ("Wo", Wo, (n_heads * head_dim, h))):
        _need(x, name, dt, shp)
    out = dict(out or {})
    dev = O.device
    dO = out.get("dO") if out.get("dO") is not None else torch.empty((T, hq), dtype=dt, device=dev)
    dW = out.get("dWo") if out.get("dWo") is not None else torch.empty((hq, h), dtype=dt, device=dev)
    db = None
    if bias_grad:
        db = out.get("dbo") if out.get("dbo") is not None else torch.empty(h, dtype=torch.float32, device=dev)
    w = _workspace(linear_workspace_bytes(T, hq, h, t, "row", dt) if T > 0 else 0, dev, ws)
    st = lib().tp_attn_out_backward(_ptr(dZ), _ptr(O), _ptr(Wo), T, h, n_heads, head_dim, t, _DT[dt], _ptr(dO),
                                    _ptr(dW), _ptr(db), _ptr(w), _wsize(w), _stream(stream))
    check(st, "tp_attn_out_backward")
    res = {"dO": dO, "dWo": dW}
    if bias_grad:
        res["dbo"] = db
    return res


def _chunk_list(out, key, t, rows, cols, dt, dev):
    xs = out.get(key) if out else None
    if xs is None:
        xs = [torch.empty((rows, cols), dtype=dt, device=dev) for _ in range(t)]
    if isinstance(xs, torch.Tensor):
        raise ValueError(f"out['{key}'] must be a list of t sequence-chunk tensors")
    _chunks(xs, key, t, rows, cols, dt, dev)
    return xs


def _wsz(T, n_in, n_out, t, parallel, dt, dev, ws, need):
    w = _workspace(linear_workspace_bytes(T, n_in, n_out, t, parallel, dt) if need else 0, dev, ws)
    return w, (0 if w is None else w.numel() * w.element_size())


def _wsz_fwd(T, n_in, n_out, t, parallel, dt, dev, ws):
    w = _fwd_workspace(dt, T, lambda: linear_workspace_bytes(T, n_in, n_out, t, parallel, dt), dev, ws)
    return w, (0 if w is None else w.numel() * w.element_size())


def tp_column_linear_forward_sp(X_chunks, W: torch.Tensor, t: int, b: Optional[torch.Tensor] = None,
                                out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                                stream=None) -> torch.Tensor:
    """Y = X W + b, column-parallel, X given as t sequence chunks (the all-gather entry)."""
    rows, n_in = X_chunks[0].shape
    T, n_out = rows * t, W.shape[1]
    dt, dev = X_chunks[0].dtype, X_chunks[0].device
    _chunks(X_chunks, "X_chunks", t, rows, n_in, dt, dev)
    _need(W, "W", dt, (n_in, n_out))
    if b is not None:
        _need(b, "b", torch.float32, (n_out,))
    Y = out if out is not None else torch.empty((T, n_out), dtype=dt, device=dev)
    w, wb = _wsz_fwd(T, n_in, n_out, t, "column", dt, dev, ws)
    xp = _ptr_list(X_chunks)
    check(lib().tp_column_linear_forward_sp(xp, _ptr(W), _ptr(b), T, n_in, n_out, t, _DT[dt], _ptr(Y), _ptr(w), wb,
                                            _stream(stream)), "tp_column_linear_forward_sp")
    return Y


def tp_column_linear_backward_sp(dY: torch.Tensor, X_chunks, W: torch.Tensor, t: int, bias_grad: bool = True,
                                 out=None, ws: Optional[torch.Tensor] = None, stream=None) -> Dict[str, object]:
    """dX as t sequence chunks (the f* sum reduce-scattered), dW, db."""
    rows, n_in = X_chunks[0].shape
    T, n_out = rows * t, W.shape[1]
    dt, dev = X_chunks[0].dtype, X_chunks[0].device
    _chunks(X_chunks, "X_chunks", t, rows, n_in, dt, dev)
    _need(dY, "dY", dt, (T, n_out))
    _need(W, "W", dt, (n_in, n_out))
    out = dict(out or {})
    dXc = _chunk_list(out, "dX", t, rows, n_in, dt, dev)
    dW = out.get("dW") if out.get("dW") is not None else torch.empty((n_in, n_out), dtype=dt, device=dev)
    db = (out.get("db") if out.get("db") is not None else torch.empty(n_out, dtype=torch.float32, device=dev)) \
        if bias_grad else None
    w, wb = _wsz(T, n_in, n_out, t, "column", dt, dev, ws, T > 0)
    xp, dxp = _ptr_list(X_chunks), _ptr_list(dXc)
    check(lib().tp_column_linear_backward_sp(_ptr(dY), xp, _ptr(W), T, n_in, n_out, t, _DT[dt], dxp, _ptr(dW),
                                             _ptr(db), _ptr(w), wb, _stream(stream)), "tp_column_linear_backward_sp")
    res = {"dX": dXc, "dW": dW}
    if bias_grad:
        res["db"] = db
    return res


def tp_row_linear_forward_sp(X: torch.Tensor, W: torch.Tensor, t: int, b: Optional[torch.Tensor] = None,
                             out=None, ws: Optional[torch.Tensor] = None, stream=None):
    """Y = sum_i X_i W_i + b, row-parallel, Y returned as t sequence chunks (the reduce-scatter exit)."""
    T, n_in = X.shape
    n_out = W.shape[1]
    dt, dev = X.dtype, X.device
    _need(X, "X", dt, (T, n_in))
    _need(W, "W", dt, (n_in, n_out))
    if b is not None:
        _need(b, "b", torch.float32, (n_out,))
    if T % t:
        raise ValueError("T must divide by t")
    Yc = _chunk_list({"Y": out} if out is not None else None, "Y", t, T // t, n_out, dt, dev)
    w, wb = _wsz_fwd(T, n_in, n_out, t, "row", dt, dev, ws)
    yp = _ptr_list(Yc)
    check(lib().tp_row_linear_forward_sp(_ptr(X), _ptr(W), _ptr(b), T, n_in, n_out, t, _DT[dt], yp, _ptr(w), wb,
                                         _stream(stream)), "tp_row_linear_forward_sp")
    return Yc


def tp_row_linear_backward_sp(dY_chunks, X: torch.Tensor, W: torch.Tensor, t: int, bias_grad: bool = True, out=None,
                              ws: Optional[torch.Tensor] = None, stream=None) -> Dict[str, torch.Tensor]:
    """dX (each shard's columns), dW, db from the gathered dY chunks."""
    T, n_in = X.shape
    n_out = W.shape[1]
    dt, dev = X.dtype, X.device
    _need(X, "X", dt, (T, n_in))
    _need(W, "W", dt, (n_in, n_out))
    _chunks(dY_chunks, "dY_chunks", t, T // t, n_out, dt, dev)
    out = dict(out or {})
    dX = out.get("dX") if out.get("dX") is not None else torch.empty((T, n_in), dtype=dt, device=dev)
    dW = out.get("dW") if out.get("dW") is not None else torch.empty((n_in, n_out), dtype=dt, device=dev)
    db = (out.get("db") if out.get("db") is not None else torch.empty(n_out, dtype=torch.float32, device=dev)) \
        if bias_grad else None
    w, wb = _wsz(T, n_in, n_out, t, "row", dt, dev, ws, T > 0)
    dyp = _ptr_list(dY_chunks)
    check(lib().tp_row_linear_backward_sp(dyp, _ptr(X), _ptr(W), T, n_in, n_out, t, _DT[dt], _ptr(dX), _ptr(dW),
                                          _ptr(db), _ptr(w), wb, _stream(stream)), "tp_row_linear_backward_sp")
    res = {"dX": dX, "dW": dW}
    if bias_grad:
        res["db"] = db
    return res


def tp_attn_qkv_forward_sp(X_chunks, Wqkv: torch.Tensor, n_heads: int, n_kv_heads: int, head_dim: int, t: int,
                           bqkv: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                           ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """QKV projection with the sequence-parallel entry: X as t sequence chunks."""
    rows, h = X_chunks[0].shape
    T, n = rows * t, (n_heads + 2 * n_kv_heads) * head_dim
    dt, dev = X_chunks[0].dtype, X_chunks[0].device
    _chunks(X_chunks, "X_chunks", t, rows, h, dt, dev)
    _need(Wqkv, "Wqkv", dt, (h, n))
    if bqkv is not None:
        _need(bqkv, "bqkv", torch.float32, (n,))
    QKV = out if out is not None else torch.empty((T, n), dtype=dt, device=dev)
    w, wb = _wsz_fwd(T, h, n, t, "column", dt, dev, ws)
    xp = _ptr_list(X_chunks)
    check(lib().tp_attn_qkv_forward_sp(xp, _ptr(Wqkv), _ptr(bqkv), T, h, n_heads, n_kv_heads, head_dim, t, _DT[dt],
                                       _ptr(QKV), _ptr(w), wb, _stream(stream)), "tp_attn_qkv_forward_sp")
    return QKV


def tp_attn_qkv_backward_sp(dQKV: torch.Tensor, X_chunks, Wqkv: torch.Tensor, n_heads: int, n_kv_heads: int,
                            head_dim: int, t: int, bias_grad: bool = True, out=None,
                            ws: Optional[torch.Tensor] = None, stream=None) -> Dict[str, object]:
    """dX as t sequence chunks, dWqkv, dbqkv."""
    rows, h = X_chunks[0].shape
    T, n = rows * t, (n_heads + 2 * n_kv_heads) * head_dim
    dt, dev = X_chunks[0].dtype, X_chunks[0].device
    _chunks(X_chunks, "X_chunks", t, rows, h, dt, dev)
    _need(dQKV, "dQKV", dt, (T, n))
    _need(Wqkv, "Wqkv", dt, (h, n))
    out = dict(out or {})
    dXc = _chunk_list(out, "dX", t, rows, h, dt, dev)
    dW = out.get("dWqkv") if out.get("dWqkv") is not None else torch.empty((h, n), dtype=dt, device=dev)
    db = (out.get("dbqkv") if out.get("dbqkv") is not None else torch.empty(n, dtype=torch.float32, device=dev)) \
        if bias_grad else None
    w, wb = _wsz(T, h, n, t, "column", dt, dev, ws, T > 0)
    xp, dxp = _ptr_list(X_chunks), _ptr_list(dXc)
    check(lib().tp_attn_qkv_backward_sp(_ptr(dQKV), xp, _ptr(Wqkv), T, h, n_heads, n_kv_heads, head_dim, t, _DT[dt],
                                        dxp, _ptr(dW), _ptr(db), _ptr(w), wb, _stream(stream)),
          "tp_attn_qkv_backward_sp")
    res = {"dX": dXc, "dWqkv": dW}
    if bias_grad:
        res["dbqkv"] = db
    return res


def tp_attn_out_forward_sp(O: torch.Tensor, Wo: torch.Tensor, n_heads: int, head_dim: int, t: int,
                           bo: Optional[torch.Tensor] = None, out=None, ws: Optional[torch.Tensor] = None,
                           stream=None):
    """Output projection with the sequence-parallel exit: Z as t sequence chunks."""
    T, hq = O.shape
    h = Wo.shape[1]
    dt, dev = O.dtype, O.device
    _need(O, "O", dt, (T, n_heads * head_dim))
    _need(Wo, "Wo", dt, (hq, h))
    if bo is not None:
        _need(bo, "bo", torch.float32, (h,))
    if T % t:
        raise ValueError("T must divide by t")
    Zc = _chunk_list({"Z": out} if out is not None else None, "Z", t, T // t, h, dt, dev)
    w, wb = _wsz_fwd(T, hq, h, t, "row", dt, dev, ws)
    zp = _ptr_list(Zc)
    check(lib().tp_attn_out_forward_sp(_ptr(O), _ptr(Wo), _ptr(bo), T, h, n_heads, head_dim, t, _DT[dt], zp, _ptr(w),
                                       wb, _stream(stream)), "tp_attn_out_forward_sp")
    return Zc


def tp_attn_out_backward_sp(dZ_chunks, O: torch.Tensor, Wo: torch.Tensor, n_heads: int, head_dim: int, t: int,
                            bias_grad: bool = True, out=None, ws: Optional[torch.Tensor] = None,
                            stream=None) -> Dict[str, torch.Tensor]:
    """dO, dWo, dbo from the gathered dZ chunks."""
    T, hq = O.shape
    h = Wo.shape[1]
    dt, dev = O.dtype, O.device
    _need(O, "O", dt, (T, n_heads * head_dim))
    _need(Wo, "Wo", dt, (hq, h))
    _chunks(dZ_chunks, "dZ_chunks", t, T // t, h, dt, dev)
    out = dict(out or {})
    dO = out.get("dO") if out.get("dO") is not None else torch.empty((T, hq), dtype=dt, device=dev)
    dW = out.get("dWo") if out.get("dWo") is not None else torch.empty((hq, h), dtype=dt, device=dev)
    db = (out.get("dbo") if out.get("dbo") is not None else torch.empty(h, dtype=torch.float32, device=dev)) \
        if bias_grad else None
    w, wb = _wsz(T, hq, h, t, "row", dt, dev, ws, T > 0)
    dzp = _ptr_list(dZ_chunks)
    check(lib().tp_attn_out_backward_sp(dzp, _ptr(O), _ptr(Wo), T, h, n_heads, head_dim, t, _DT[dt], _ptr(dO),
                                        _ptr(dW), _ptr(db), _ptr(w), wb, _stream(stream)), "tp_attn_out_backward_sp")
    res = {"dO": dO, "dWo": dW}
    if bias_grad:
        res["dbo"] = db
    return res


def vocab_parallel_ce(H: torch.Tensor, E: torch.Tensor, targets: torch.Tensor, v_valid: int, t: int,
                      grad_scale: float = 1.0, grads: bool = True, want_dH: bool = True, want_dE: bool = True,
                      out: Optional[Dict[str, torch.Tensor]] = None, ws: Optional[torch.Tensor] = None,
                      stream=None) -> Dict[str, torch.Tensor]:
    """Per-token loss and lse; with grads, dH and dE of grad_scale * sum(loss)."""
    T, h = H.shape
    v_pad = E.shape[0]
    dt = H.dtype
    _need(H, "H", dt, (T, h))
    _need(E, "E", dt, (v_pad, h))
    _need(targets, "targets", torch.int32, (T,))
    out = dict(out or {})
    dev = H.device
    loss = out.get("loss") if out.get("loss") is not None else torch.empty(T, dtype=torch.float32, device=dev)
    lse = out.get("lse") if out.get("lse") is not None else torch.empty(T, dtype=torch.float32, device=dev)
    dH = dE = None
    if grads and want_dH:
        dH = out.get("dH") if out.get("dH") is not None else torch.empty((T, h), dtype=dt, device=dev)
    if grads and want_dE:
        dE = out.get("dE") if out.get("dE") is not None else torch.empty((v_pad, h), dtype=dt, device=dev)
    with_g = dH is not None or dE is not None
    nbytes = ce_workspace_bytes(T, h, v_pad, t, with_g, dt) if T > 0 else 0
    w = _workspace(nbytes, dev, ws)
    st = lib().vocab_parallel_ce(_ptr(H), _ptr(E), _ptr(targets), T, h, v_pad, v_valid, t, float(grad_scale),
                                 _DT[dt], _ptr(loss), _ptr(lse), _ptr(dH), _ptr(dE), _ptr(w),
                                 0 if w is None else w.numel() * w.element_size(), _stream(stream))
    check(st, "vocab_parallel_ce")
    res = {"loss": loss, "lse": lse}
    if dH is not None:
        res["dH"] = dH
    if dE is not None:
        res["dE"] = dE
    return res


CE_STATIC_SCRATCH_BYTES = 16 << 20  # TPCE_CE_STATIC_SCRATCH_BYTES in include/tpce.h


def vocab_parallel_ce_loss_static(H: torch.Tensor, E: torch.Tensor, targets: torch.Tensor, v_valid: int, t: int,
                                  loss: torch.Tensor, lse: Optional[torch.Tensor] = None,
                                  stream=None) -> Dict[str, torch.Tensor]:
    """Forward-only fused CE into caller-provided loss (and lse) buffers, with
    the library's static device scratch instead of a workspace: for callers
    that cannot allocate device memory. Nothing is allocated here either."""
    T, h = H.shape
    v_pad = E.shape[0]
    dt = H.dtype
    _need(H, "H", dt, (T, h))
    _need(E, "E", dt, (v_pad, h))
    _need(targets, "targets", torch.int32, (T,))
    _need(loss, "loss", torch.float32, (T,))
    if lse is not None:
        _need(lse, "lse", torch.float32, (T,))
    st = lib().vocab_parallel_ce_loss_static(_ptr(H), _ptr(E), _ptr(targets), T, h, v_pad, v_valid, t, _DT[dt],
                                             _ptr(loss), _ptr(lse), _stream(stream))
    check(st, "vocab_parallel_ce_loss_static")
    res = {"loss": loss}
    if lse is not None:
        res["lse"] = lse
    return res


def device_status(clear: bool = True, stream=None) -> int:
    """Synchronise and return the device status word's code (0 = OK)."""
    detail = ctypes.c_uint32(0)
    return int(lib().tpce_device_status(_stream(stream), 1 if clear else 0, ctypes.byref(detail)))


def device_status_detail(clear: bool = True, stream=None):
    detail = ctypes.c_uint32(0)
    code = int(lib().tpce_device_status(_stream(stream), 1 if clear else 0, ctypes.byref(detail)))
    return code, int(detail.value)


def profile_enable(on: bool = True) -> None:
    check(lib().tpce_profile_enable(1 if on else 0), "tpce_profile_enable")


def profile_read() -> Dict[str, Dict[str, float]]:
    """Per-kernel launches and total ms recorded since profile_enable(True)."""
    L = lib()
    n = L.tpce_profile_count()
    if n < 0:
        raise TpceError(5, "tpce_profile_count")
    res = {}
    for i in range(n):
        name = ctypes.c_char_p()
        launches = ctypes.c_int64()
        ms = ctypes.c_double()
        check(L.tpce_profile_get(i, ctypes.byref(name), ctypes.byref(launches), ctypes.byref(ms)),
              "tpce_profile_get")
        res[name.value.decode()] = {"launches": int(launches.value), "ms": float(ms.value)}
    return res


__all__ = ["TpceError", "pad_vocab", "mlp_workspace_bytes", "ce_workspace_bytes", "tp_mlp_forward",
           "tp_mlp_backward", "vocab_parallel_ce", "vocab_parallel_ce_loss_static", "device_status", "device_status_detail",
           "profile_enable", "profile_read"]
