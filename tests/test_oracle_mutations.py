"""Planted mistakes: each is a plausible slip written into a scratch copy of
the oracle (oracle/oracle.c), and each must make one of the oracle's pin
files fail -- the pins check the oracle against what the pages and the
mathematics fix, so a pin that let a slip through would prove nothing. The
unchanged copy must pass the same files. CPU only: the copies are built with
gcc and run in subprocesses, several at a time; nothing here touches the
CUDA library."""

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = ("test_oracle_pins.py", "test_oracle_pins_swiglu.py", "test_oracle_pins_linear.py")

# (name, pin file, text in oracle.c, the slip put in its place)
MUTATIONS = [
    # the row-parallel bias bB left out of Z
    ('drop_bB', 'test_oracle_pins.py',
     'Z[t * h + n] = bB ? bB[n] : 0.0;',
     'Z[t * h + n] = 0.0;'),
    # GeLU' = Phi - x phi instead of Phi + x phi
    ('gelu_grad_sign', 'test_oracle_pins.py',
     'return Phi + x * phi;',
     'return Phi - x * phi;'),
    # dA built from the wrong (transposed) index pair
    ('transpose_dA', 'test_oracle_pins.py',
     'dA[k * f + jj] += x * dU[tt * f + jj];',
     'dA[k * f + jj] += X[tt * h + (jj % h)] * dU[tt * f + k % f];'),
    # log-sum-exp without the max subtraction
    ('no_max_sub', 'test_oracle_pins.py',
     'S += exp(l[j] - m);\n        double L = m + log(S);',
     'S += exp(l[j]);\n        double L = log(S);'),
    # padded vocabulary rows of dE not zero
    ('pad_leak', 'test_oracle_pins.py',
     'for (j = 0; j < v_pad; j++) {\n            for (int64_t k = 0; k < h; k++)\n                dE[j * h + k] = 0.0;\n            if (j >= v_valid) continue;',
     'for (j = 0; j < v_pad; j++) {\n            for (int64_t k = 0; k < h; k++)\n                dE[j * h + k] = 0.0;\n            if (j >= v_valid) { for (int64_t k = 0; k < h; k++) dE[j*h+k] = 1e-3; continue; }'),
    # bB added once per shard instead of once
    ('bias_per_shard', 'test_oracle_pins.py',
     'Z[tt * h + n] += bB ? bB[n] : 0.0;',
     'Z[tt * h + n] += bB ? t * bB[n] : 0.0;'),
    # shard sums combined without exp(m_i - m)
    ('combine_no_rescale', 'test_oracle_pins.py',
     'S += si * exp(m_shard[(int64_t)i * T + tok] - M);',
     'S += si;'),
    # dX from a shifted, scaled A
    ('dX_wrong_operand', 'test_oracle_pins.py',
     'acc += dU[t * f + jj] * A[kk * f + jj];',
     'acc += dU[t * f + jj] * A[(kk * f + jj) % (h*f)] * 1.0001;'),
    # bA left out of U
    ('U_no_bias', 'test_oracle_pins.py',
     'u[j] = bA ? bA[j] : 0.0;',
     'u[j] = 0.0;'),
    # Swish applied to the up half instead of the gate
    ('swap_gate_up', 'test_oracle_pins_swiglu.py',
     'y[j] = oracle_swish(gu[j]) * gu[f + j];',
     'y[j] = oracle_swish(gu[f + j]) * gu[j];'),
    # Swish(x) = sigmoid(x) instead of x sigmoid(x)
    ('swish_is_sigmoid', 'test_oracle_pins_swiglu.py',
     'return x / (1.0 + exp(-x));',
     'return 1.0 / (1.0 + exp(-x));'),
    # Swish with exp(x) instead of exp(-x)
    ('swish_neg', 'test_oracle_pins_swiglu.py',
     'return x / (1.0 + exp(-x));',
     'return x / (1.0 + exp(x));'),
    # a term of Swish' dropped
    ('swish_grad_drop', 'test_oracle_pins_swiglu.py',
     'return s + x * s * (1.0 - s);',
     'return s + x * s;'),
    # dG without the factor Up
    ('dG_no_u', 'test_oracle_pins_swiglu.py',
     'dGU[t * f2 + jj] = dy * u * oracle_swish_grad(g);',
     'dGU[t * f2 + jj] = dy * oracle_swish_grad(g);'),
    # a shard gathering the wrong up columns of W1
    ('shard_up_cols', 'test_oracle_pins_swiglu.py',
     'W1i[k * fs2 + fs + j] = W1[k * f2 + u0 + j];',
     'W1i[k * fs2 + fs + j] = W1[k * f2 + g0 + fs + j];'),
    # dX summed over the gate half of W1 only
    ('dX_only_gate', 'test_oracle_pins_swiglu.py',
     'for (int64_t jj = 0; jj < f2; jj++)\n                    acc += dGU[t * f2 + jj] * W1[kk * f2 + jj];',
     'for (int64_t jj = 0; jj < f; jj++)\n                    acc += dGU[t * f2 + jj] * W1[kk * f2 + jj];'),
    # the up bias taken from the gate biases
    ('cols_up_bias', 'test_oracle_pins_swiglu.py',
     'double g = b1 ? b1[j] : 0.0, u = b1 ? b1[f + j] : 0.0;',
     'double g = b1 ? b1[j] : 0.0, u = b1 ? b1[j] : 0.0;'),
    # the row-parallel bias added by every shard
    ('row_bias_per_shard', 'test_oracle_pins_linear.py',
     'bi[j] = (mode == 0 && b) ? b[c0 + j] : 0.0;',
     'bi[j] = b ? b[c0 + j] : 0.0;'),
    # K heads read one head-block off
    ('qkv_k_offset', 'test_oracle_pins_linear.py',
     'return head * gw + (qpg + kind - 1) * d + j;',
     'return head * gw + (qpg + kind) * d + j;'),
    # query heads not grouped with their KV head
    ('qkv_q_group', 'test_oracle_pins_linear.py',
     'return (head / qpg) * gw + (head % qpg) * d + j;',
     'return head * d + j;'),
    # dX with W indexed transposed
    ('dX_transposed', 'test_oracle_pins_linear.py',
     'acc += dY[t * n_out + jj] * W[kk * n_out + jj];',
     'acc += dY[t * n_out + jj] * W[(jj * n_in + kk) % (n_in * n_out)];'),
    # the bias gradient left at zero
    ('db_missing', 'test_oracle_pins_linear.py',
     'acc += dY[t * n_out + j];',
     'acc += 0.0;'),
    # every column-parallel shard reading column block 0
    ('shard_col_offset', 'test_oracle_pins_linear.py',
     'int64_t c0 = mode == 0 ? (int64_t)i * out_s : 0;',
     'int64_t c0 = 0;'),
    # the reduce-scatter writing rank r's rows from rank r + 1
    ('rs_wrong_rank', 'test_oracle_pins.py',
     'Z_chunks[r][e] += Zi[(int64_t)r * rows * h + e];',
     'Z_chunks[r][e] += Zi[(int64_t)((r + 1) % t) * rows * h + e];'),
    # the sequence-parallel dX partials overwritten, not summed
    ('dx_not_summed', 'test_oracle_pins.py',
     'dX_chunks[r][e] += dXi[(int64_t)r * rows * h + e];',
     'dX_chunks[r][e] = dXi[(int64_t)r * rows * h + e];'),
    # the all-gather repeating chunk 0
    ('gather_one_chunk', 'test_oracle_pins.py',
     'memcpy(X + (int64_t)r * rows * h, X_chunks[r], sizeof(double) * (size_t)(rows * h));',
     'memcpy(X + (int64_t)r * rows * h, X_chunks[0], sizeof(double) * (size_t)(rows * h));'),
    # the exit bias added twice
    ('bias_per_rank_twice', 'test_oracle_pins.py',
     'Z_chunks[r][rr * h + n] += bB ? bB[n] : 0.0;',
     'Z_chunks[r][rr * h + n] += bB ? 2 * bB[n] : 0.0;'),
]


def _scratch_copy(dst):
    ignore = shutil.ignore_patterns("*.so", "*.so.tmp", "__pycache__", "abi_c")
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(dst, "oracle"), ignore=ignore)
    shutil.copytree(os.path.join(ROOT, "tests"), os.path.join(dst, "tests"), ignore=ignore)
    shutil.copy(os.path.join(ROOT, "pytest.ini"), dst)


def _run_pins(dst, pins):
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider"] +
                       [os.path.join("tests", p) for p in pins], cwd=dst, env=env, capture_output=True, text=True,
                       timeout=600)
    tail = r.stdout.strip().splitlines()[-1] if r.stdout.strip() else r.stderr[-300:]
    return r.returncode, tail


def _mutant(case, root):
    name, pins, old, new = case
    dst = os.path.join(root, name)
    _scratch_copy(dst)
    path = os.path.join(dst, "oracle", "oracle.c")
    src = open(path).read()
    assert old in src, f"{name}: the text to change is no longer in oracle.c"
    open(path, "w").write(src.replace(old, new, 1))
    return _run_pins(dst, (pins,))


def test_unchanged_copy_passes_the_pins(tmp_path):
    _scratch_copy(str(tmp_path / "clean"))
    rc, tail = _run_pins(str(tmp_path / "clean"), PINS)
    assert rc == 0, tail


def test_every_planted_mistake_fails_a_pin(tmp_path):
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(lambda c: _mutant(c, str(tmp_path)), MUTATIONS))
    survivors, broken = [], []
    for (name, *_), (rc, tail) in zip(MUTATIONS, results):
        if rc == 0:
            survivors.append(name)
        elif "failed" not in tail:  # a copy that did not build or collect proves nothing
            broken.append(f"{name}: {tail}")
    assert not broken, broken
    assert not survivors, f"slips no pin caught: {survivors}"
