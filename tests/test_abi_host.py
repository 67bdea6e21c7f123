"""Host-side tests of the C ABI that need no GPU: the library loads, exports
every symbol include/tpce.h declares, and its host logic (padding rule,
workspace sizes, argument validation) behaves as documented. No call here
reaches a kernel: every compute entry point is called only with arguments the
host checks reject before any CUDA call."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from vocab_ce_gb300 import build
    build.build()
    from vocab_ce_gb300._lib import lib
    return lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "tpce.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", src)) - {"if", "sizeof"})


def test_library_exports_every_declared_symbol(L):
    names = header_functions()
    assert "tp_mlp_forward" in names and "vocab_parallel_ce" in names
    for n in names:
        assert hasattr(L, n), f"missing export {n}"


def test_binding_declares_every_symbol():
    from vocab_ce_gb300._lib import SIGNATURES
    assert set(header_functions()) == set(SIGNATURES)


def test_status_strings(L):
    for code, name in enumerate(["TPCE_OK", "TPCE_ERR_INVALID", "TPCE_ERR_SHAPE", "TPCE_ERR_ALIGN",
                                 "TPCE_ERR_WORKSPACE", "TPCE_ERR_CUDA", "TPCE_ERR_TIMEOUT",
                                 "TPCE_ERR_UNSUPPORTED"]):
        assert L.tpce_status_string(code).decode() == name
    assert L.tpce_version() >= 100


def test_vocab_padding_golden(L):
    rows = [l.split() for l in open(os.path.join(ROOT, "tests", "golden", "vocab_padding.txt"))
            if l.strip() and not l.startswith("#")]
    assert rows
    for v, t, d, vp in rows:
        assert L.tpce_pad_vocab(int(v), int(t), int(d)) == int(vp)


def test_vocab_padding_rule(L):
    import vocab_ce_gb300 as tp
    for v in (1, 127, 128, 129, 50257, 128256):
        for t in (1, 2, 4, 8, 16):
            p = tp.pad_vocab(v, t)
            assert p >= v and p % (128 * t) == 0 and p - v < 128 * t
    assert tp.pad_vocab(128256, 8) == 129024 == 8 * 126 * 128
    assert L.tpce_pad_vocab(-1, 8, 128) == -1 and L.tpce_pad_vocab(10, 0, 128) == -1


def test_workspace_sizes(L):
    import vocab_ce_gb300 as tp
    # every workspace starts with the GEMMs' split-tail scratch: at most 64
    # K parts of one CTA pair's 256 x 256 fp32 tile, plus their tickets
    tail = tp.tail_workspace_bytes()
    assert tail == 64 * 2 * 128 * 256 * 4 + 4096
    # MLP backward holds dU [T, f] in bf16 plus a small column-sum buffer; from
    # widths of 6144 on, the weight gradients read K-major copies: X^T [h, T]
    # (for dA, when f >= 6144) and Y^T [f, T] (for dB, when h >= 6144), rows
    # padded to 8 tokens
    def copies(T, h, fw, f):
        Tp = (T + 7) // 8 * 8
        return (h * Tp * 2 if fw >= 6144 else 0) + (f * Tp * 2 if h >= 6144 else 0)
    for T, h, f in ((32, 64, 256), (4096, 8192, 32768), (8192, 3072, 12288), (300, 6144, 6144)):
        b = tp.mlp_workspace_bytes(T, h, f, 8 if f % 512 == 0 else 2) - tail
        base = T * f * 2 + copies(T, h, f, f)
        assert b >= base and b < base + 64 * max(f, h) * 4 + 4096, (T, h, f)
    # CE: the forward keeps statistics only; the backward scratch stays far
    # below the T x v_pad logits (the logits are never materialised)
    T, h, vp, t = 16384, 8192, 129024, 8
    fwd = tp.ce_workspace_bytes(T, h, vp, t, grads=False) - tail
    bwd = tp.ce_workspace_bytes(T, h, vp, t, grads=True) - tail
    assert fwd < 0.02 * T * vp * 2
    # the dl scratch holds at most half the vocabulary and at most 1 GiB
    assert bwd <= 2 ** 30 + T * h * 4 + fwd + 4096
    assert bwd < 0.5 * T * vp * 2
    # pass 1 hands the combine one (max, sumexp) pair per shard and token; a
    # shard cut into several runs ("parts") also needs the parts' pairs and a
    # ticket per 32-token slab and shard for the fold. At the 129K config
    # each shard's 63 tiles are cut into 9 runs of 7 (4608 work units keep the
    # 76 CTA pairs 99.4% busy), at the 8.3B config 25 tiles into 5 runs of 5,
    # and one run per shard wherever the units fit in one wave; the one-CTA
    # kernel (fp32) makes one part per 128-id tile
    def rup(x):
        return (x + 255) // 256 * 256

    def fwd_ws(T, h, vp, t, dt=None):
        kw = {} if dt is None else {"dtype": dt}
        return tp.ce_workspace_bytes(T, h, vp, t, grads=False, **kw) - tail

    def expect(T, t, parts):
        fold = rup(parts * T * 8) + rup((T + 31) // 32 * t * 4) if parts > t else 0
        return rup(t * T * 8) + fold + 2 * rup(T * 4)
    for (Tq, hq, vq, tq, parts) in ((16384, 8192, 129024, 8, 72), (8192, 3072, 51200, 8, 40),
                                    (1000, 256, 4096, 8, 8), (6400, 64, 6144, 4, 12)):
        assert fwd_ws(Tq, hq, vq, tq) == expect(Tq, tq, parts), (Tq, vq, tq)
    assert fwd_ws(100, 64, 512, 2, dt=__import__("torch").float32) == expect(100, 2, 4)
    # the 8.3B block: 4 of 8 shards per chunk
    T2, h2, vp2 = 8192, 3072, 51200
    b2 = tp.ce_workspace_bytes(T2, h2, vp2, 8, grads=True) - tp.ce_workspace_bytes(T2, h2, vp2, 8, grads=False)
    assert b2 <= T2 * (vp2 // 2) * 2 + T2 * h2 * 4 + 1024
    # 66,000 tokens: one 8,192-id shard (1.08 GB of dl) exceeds the 1 GiB bound,
    # so each shard is cut into two 4,096-id chunks
    T3, h3, vp3 = 66000, 16, 16384
    b3 = tp.ce_workspace_bytes(T3, h3, vp3, 2, grads=True) - tp.ce_workspace_bytes(T3, h3, vp3, 2, grads=False)
    assert T3 * 4096 * 2 <= b3 <= T3 * 4096 * 2 + T3 * h3 * 4 + 4096
    # fp32 adds transposed operand copies: A^T, B^T, Y^T, dZ^T, X^T, dU^T
    T, h, f = 32, 64, 256
    assert tp.mlp_workspace_bytes(T, h, f, 2, dtype=__import__("torch").float32) >= 4 * (T * f + 2 * f * h + 2 * f * T + 2 * h * T)
    # invalid shapes give 0
    assert L.tpce_mlp_workspace_bytes(10, 64, 100, 3, 0) == 0
    assert L.tpce_ce_workspace_bytes(10, 64, 1000, 8, 0, 1) == 0


P = ctypes.c_void_p
FAKE = P(1 << 20)      # an aligned address that is never dereferenced
MISALIGNED = P((1 << 20) + 8)


def mlp_fwd(L, T=64, h=64, f=256, t=2, dtype=0, X=FAKE):
    return L.tp_mlp_forward(X, FAKE, None, FAKE, None, T, h, f, t, dtype, FAKE, FAKE, FAKE, None, 0, None)


def test_mlp_validation(L):
    assert mlp_fwd(L, f=256, t=3) == 2                 # f % t
    assert mlp_fwd(L, f=256, t=8) == 2                 # f / t = 32 is not whole 64-wide blocks
    assert mlp_fwd(L, h=60) == 2                       # 16-byte row pitch
    assert mlp_fwd(L, T=-1) == 2
    assert mlp_fwd(L, X=MISALIGNED) == 3
    assert mlp_fwd(L, X=None) == 1
    assert mlp_fwd(L, dtype=1) == 4                    # the fp32 (tf32) forward needs its workspace
    assert mlp_fwd(L, dtype=5) == 1
    assert mlp_fwd(L, T=0) == 0                        # empty batch: nothing to do
    # backward with T > 0 and no workspace
    st = L.tp_mlp_backward(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 64, 256, 2, 0,
                           FAKE, FAKE, None, FAKE, None, None, 0, None)
    assert st == 4


def test_swiglu_validation_and_workspace(L):
    import vocab_ce_gb300 as tp
    import torch

    def fwd(T=64, h=64, f=256, t=2, dtype=0, X=FAKE):
        return L.tp_swiglu_forward(X, FAKE, None, FAKE, None, T, h, f, t, dtype, FAKE, FAKE, FAKE, None, 0, None)
    assert fwd(f=256, t=3) == 2                        # f % t
    assert fwd(f=256, t=8) == 2                        # f / t = 32 is not whole 64-wide blocks
    assert fwd(h=60) == 2
    assert fwd(X=MISALIGNED) == 3
    assert fwd(X=None) == 1
    assert fwd(dtype=1) == 4                           # the fp32 forward needs its workspace
    assert fwd(T=0) == 0
    st = L.tp_swiglu_backward(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 64, 256, 2, 0,
                              FAKE, FAKE, None, FAKE, None, None, 0, None)
    assert st == 4
    # the backward holds [dG | dUp] [T, 2f] in bf16 plus a small column-sum buffer
    T, h, f = 4096, 8192, 28672
    b = tp.swiglu_workspace_bytes(T, h, f, 8) - tp.tail_workspace_bytes()
    Tp = (T + 7) // 8 * 8
    cp = (h * Tp * 2 if 2 * f >= 6144 else 0) + (f * Tp * 2 if h >= 6144 else 0)  # X^T, Y^T
    assert T * 2 * f * 2 + cp <= b < T * 2 * f * 2 + cp + 64 * 2 * f * 4 + 4096
    # fp32: transposed W1 [2f, h], W2, Y, dZ, X and [dG | dUp]
    T, h, f = 32, 64, 256
    b32 = tp.swiglu_workspace_bytes(T, h, f, 2, dtype=torch.float32)
    assert b32 >= 4 * (T * 2 * f + 2 * f * h + f * h + f * T + 2 * h * T + 2 * f * T)
    assert L.tpce_swiglu_workspace_bytes(10, 64, 100, 3, 0) == 0


def test_linear_and_attention_validation(L):
    def lin(T=64, n_in=128, n_out=256, t=2, par=0, dtype=0, X=FAKE):
        return L.tp_linear_forward(X, FAKE, None, T, n_in, n_out, t, par, dtype, FAKE, None, 0, None)
    # only invalid requests are tried: each is rejected before any launch
    assert lin(n_out=256, t=3) == 2        # column: n_out % t
    assert lin(n_out=256, t=8) == 2        # column: a shard of 32 columns is not whole 64-wide blocks
    assert lin(n_in=128, t=4, par=1) == 2  # row: a shard of 32 rows
    assert lin(n_in=60) == 2
    assert lin(par=2) == 1
    assert lin(X=MISALIGNED) == 3
    assert lin(X=None) == 1
    assert lin(dtype=1) == 4               # the fp32 forward needs its workspace
    assert lin(T=0) == 0
    st = L.tp_linear_backward(FAKE, FAKE, FAKE, 64, 128, 256, 2, 0, 0, FAKE, FAKE, None, None, 0, None)
    assert st == 4                         # the backward needs the bias-gradient workspace

    def qkv(nq=8, nkv=2, d=64, t=2):
        return L.tp_attn_qkv_forward(None, FAKE, None, 64, 256, nq, nkv, d, t, 0, FAKE, None, 0, None)
    assert qkv(nkv=2, t=4) == 2            # key/value heads must split evenly over the shards
    assert qkv(nq=8, nkv=3, t=1) == 2      # query heads share key/value heads evenly
    assert qkv(d=60) == 2
    assert L.tp_attn_out_forward(FAKE, FAKE, None, 64, 256, 6, 64, 4, 0, FAKE, None, 0, None) == 2
    assert L.tpce_attn_workspace_bytes(64, 256, 8, 2, 64, 4, 0) == 0
    assert L.tpce_attn_workspace_bytes(64, 256, 8, 2, 64, 2, 0) > 0
    assert L.tpce_linear_workspace_bytes(64, 128, 256, 3, 0, 0) == 0


def test_seq_parallel_validation(L):
    import ctypes as C

    def arr(ptrs):
        return (C.c_void_p * len(ptrs))(*ptrs)
    good = [1 << 20] * 4

    def fwd(T=512, h=64, f=256, t=4, X=None, Z=None):
        X = arr(good[:t] if X is None else X)
        Z = arr(good[:t] if Z is None else Z)
        return L.tp_mlp_forward_sp(X, FAKE, None, FAKE, None, T, h, f, t, 0, Z, FAKE, FAKE, None, 0, None)
    assert fwd(T=500) == 2                                  # T % t
    assert fwd(T=256) == 2                                  # chunks of 64 rows: not whole 128-row blocks
    assert fwd(X=[1 << 20, 0, 1 << 20, 1 << 20]) == 1       # a null chunk
    assert fwd(Z=[1 << 20, (1 << 20) + 8, 1 << 20, 1 << 20]) == 3   # a misaligned chunk
    assert L.tp_mlp_forward_sp(None, FAKE, None, FAKE, None, 512, 64, 256, 4, 0, arr(good), FAKE, FAKE, None, 0,
                               None) == 1
    assert fwd(T=0) == 0
    # more chunks than the library maps
    big = arr([1 << 20] * 32)
    assert L.tp_mlp_forward_sp(big, FAKE, None, FAKE, None, 32 * 128, 64, 32 * 64, 32, 0, big, FAKE, FAKE, None, 0,
                               None) == 2
    # backward: the workspace check comes after the chunk checks
    st = L.tp_mlp_backward_sp(arr(good), arr(good), FAKE, FAKE, FAKE, FAKE, 512, 64, 256, 4, 0, arr(good), FAKE,
                              None, FAKE, None, None, 0, None)
    assert st == 4
    st = L.tp_swiglu_backward_sp(arr(good), arr(good[:3] + [0]), FAKE, FAKE, FAKE, FAKE, 512, 64, 256, 4, 0,
                                 arr(good), FAKE, None, FAKE, None, None, 0, None)
    assert st == 1


def test_linear_seq_parallel_validation(L):
    import ctypes as C

    def arr(ptrs):
        return (C.c_void_p * len(ptrs))(*ptrs)
    good = [1 << 20] * 4
    # column entry: X chunks of 64 rows are not whole 128-row blocks
    assert L.tp_column_linear_forward_sp(arr(good), FAKE, None, 256, 128, 256, 4, 0, FAKE, None, 0, None) == 2
    assert L.tp_column_linear_forward_sp(arr(good[:3] + [0]), FAKE, None, 512, 128, 256, 4, 0, FAKE, None, 0,
                                         None) == 1
    assert L.tp_column_linear_forward_sp(arr(good), FAKE, None, 0, 128, 256, 4, 0, FAKE, None, 0, None) == 0
    # row exit: a misaligned Y chunk
    assert L.tp_row_linear_forward_sp(FAKE, FAKE, None, 512, 256, 128, 4, 0, arr(good[:3] + [(1 << 20) + 4]), None,
                                      0, None) == 3
    # backward without its workspace, after the chunk checks pass
    assert L.tp_row_linear_backward_sp(arr(good), FAKE, FAKE, 512, 256, 128, 4, 0, FAKE, FAKE, None, None, 0,
                                       None) == 4
    assert L.tp_column_linear_backward_sp(FAKE, arr(good), FAKE, 512, 128, 256, 4, 0, arr(good), FAKE, None, None,
                                          0, None) == 4
    # attention: the head rules still apply
    assert L.tp_attn_qkv_forward_sp(arr(good), FAKE, None, 512, 256, 8, 2, 64, 4, 0, FAKE, None, 0, None) == 2
    assert L.tp_attn_out_forward_sp(FAKE, FAKE, None, 512, 256, 6, 64, 4, 0, arr(good), None, 0, None) == 2


def test_ce_validation(L):
    def ce(T=64, h=64, vp=512, vv=500, t=2, ws=None, wsb=0, H=FAKE, tg=FAKE):
        return L.vocab_parallel_ce(H, FAKE, tg, T, h, vp, vv, t, 1.0, 0, FAKE, None, FAKE, FAKE, ws, wsb, None)
    assert ce(vp=512, t=3) == 2          # v_pad % t
    assert ce(vp=384, t=2) == 2          # shard of 192 ids is not a multiple of 128
    assert ce(vv=513) == 2               # v_valid > v_pad
    assert ce(vv=0) == 2
    assert ce(H=MISALIGNED) == 3
    assert ce(tg=P((1 << 20) + 2)) == 3
    assert ce(tg=None) == 1
    assert ce() == 4                     # no workspace


def test_profile_api_without_launches(L):
    assert L.tpce_profile_enable(1) == 0
    assert L.tpce_profile_count() == 0
    assert L.tpce_profile_enable(0) == 0


def test_missing_library_fails_loudly(tmp_path):
    # a process whose library build is missing gets an error at its first call,
    # never a result from some other implementation
    import subprocess
    import sys
    code = ("import vocab_ce_gb300 as tp\n"
            "try:\n"
            "    tp.pad_vocab(50257, 8)\n"
            "except Exception as e:\n"
            "    print('raised', type(e).__name__)\n"
            "else:\n"
            "    print('no error')\n")
    env = dict(__import__("os").environ, TPCE_LIBRARY=str(tmp_path / "libtpce.so"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=300,
                       cwd=__import__("os").path.dirname(__import__("os").path.dirname(__file__)))
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.startswith("raised"), r.stdout


def test_python_binding_rejects_bad_tensors_before_the_library():
    # host tensors, wrong dtypes and non-contiguous views are refused in Python,
    # before any pointer reaches the library (no GPU needed)
    import torch
    import vocab_ce_gb300 as tp
    X = torch.zeros(32, 64, dtype=torch.bfloat16)
    A = torch.zeros(64, 256, dtype=torch.bfloat16)
    B = torch.zeros(256, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        tp.tp_mlp_forward(X, A, B, 2)
    H = torch.zeros(32, 64, dtype=torch.bfloat16)
    E = torch.zeros(512, 64, dtype=torch.bfloat16)
    y = torch.zeros(32, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        tp.vocab_parallel_ce(H, E, y, 512, 2)


def test_dimensions_beyond_32_bit_coordinates_are_rejected(L):
    # kernel coordinates are 32-bit: a dimension at or above 2^31 is a shape
    # error, reported by the size queries before any call could be made
    big = 1 << 31
    assert L.tpce_mlp_workspace_bytes(big, 64, 256, 2, 0) == 0
    assert L.tpce_mlp_workspace_bytes(64, big, 256, 2, 0) == 0
    assert L.tpce_ce_workspace_bytes(big, 64, 512, 2, 0, 1) == 0
    assert L.tpce_ce_workspace_bytes(64, 64, big, 2, 0, 1) == 0
