"""Plants one plausible mistake at a time in a scratch copy of the oracle and
checks that the pin suite (test_oracle_pins.py, test_oracle_hybrid_pins.py,
test_oracle_covariance_pins.py, test_oracle_second_order_pins.py,
test_oracle_reorder_pins.py, test_golden.py) rejects every mutant. The mistakes are planted on the CPU only, in a temporary directory."""

import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "H transposed": ("H[j] = kc.T @ v[r]", "H[j] = (kc.T @ v[r]).T"),
    "H not centred": ("kc = k[r] - kbar[j]", "kc = k[r]"),
    "key centroid as a sum": ("kbar[j] = k[r].mean(axis=0)", "kbar[j] = k[r].sum(axis=0)"),
    "value sum as a mean": ("vsum[j] = v[r].sum(axis=0)", "vsum[j] = v[r].mean(axis=0)"),
    "block mass B for a partial block": ("alpha @ nj[U].astype(np.float64)",
                                         "alpha @ np.full(len(U), 64.0)"),
    "first-order sign": ("num = num + w @ H[U].reshape(-1, d)", "num = num - w @ H[U].reshape(-1, d)"),
    "first-order term without the scale": ("w = (alpha[:, :, None] * qp[:, None, :])",
                                           "w = (alpha[:, :, None] * q[rows][:, None, :])"),
    "ties to the higher index": ("order = np.lexsort((cand, -r[a, cand]))",
                                 "order = np.lexsort((-cand, -r[a, cand]))"),
    "band off by one": ("forced = (np.abs(idx - i) <= band) | (idx < n_sink)",
                        "forced = (np.abs(idx - i) < band) | (idx < n_sink)"),
    "shift ignores centroid logits": ("            m = np.maximum(m, a.max(axis=1))", "            pass"),
    "global H as a sum": ("return np.asarray(H, dtype=np.float64).mean(axis=0)",
                          "return np.asarray(H, dtype=np.float64).sum(axis=0)"),
    "hybrid first order weighted by every block": (
        "alpha.sum(axis=1)[:, None] * (qp @ Hbar)",
        "(alpha.sum(axis=1) + pe.sum(axis=1))[:, None] * (qp @ Hbar)"),
    "hybrid first order without the scale": ("alpha.sum(axis=1)[:, None] * (qp @ Hbar)",
                                              "alpha.sum(axis=1)[:, None] * (q[rows] @ Hbar)"),
    "spectral norm as the Frobenius norm": ("np.linalg.svd(a, compute_uv=False)[0] for a in A",
                                            "np.sqrt((a * a).sum()) for a in A"),
    "heterogeneity not centred on Hbar": ("A = np.asarray(H, np.float64) - np.asarray(Hbar, np.float64)[None]",
                                          "A = np.asarray(H, np.float64)"),
    "covariance bias ignored": ("r = r + np.asarray(bias, np.float64)[None, :]", "r = r"),
    "covariance bias subtracted": ("r = r + np.asarray(bias, np.float64)[None, :]",
                                   "r = r - np.asarray(bias, np.float64)[None, :]"),
    "second order without the squared scale": ("return 0.5 * scale * scale * (q2 @ var.T)",
                                               "return 0.5 * scale * (q2 @ var.T)"),
    "second order with the sample variance": ("k[block_rows(j, n, B)].var(axis=0)",
                                              "k[block_rows(j, n, B)].var(axis=0, ddof=1)"),
    "second order pools the squared mean": ("(q[block_rows(i, n, B)] ** 2).mean(axis=0)",
                                            "q[block_rows(i, n, B)].mean(axis=0) ** 2"),
    "second-order gate at ln 64 for every block": (
        "lim = np.log(np.asarray(nj, dtype=np.float64))[None, :]",
        "lim = np.full((1, len(nj)), np.log(64.0))"),
    "second-order gate clamps": ("return np.where(w > lim, 0.0, w)", "return np.minimum(w, lim)"),
    "Morton with t and y bits swapped": ("c |= ((t >> b) & 1) << (3 * b + 2)",
                                        "c |= ((t >> b) & 1) << (3 * b + 1)"),
    "sink blocks off by one": ("forced = (np.abs(idx - i) <= band) | (idx < n_sink)",
                               "forced = (np.abs(idx - i) <= band) | (idx <= n_sink)"),
    "restore ignores the permutation": ("y[np.asarray(perm)] = np.transpose(o, (1, 0, 2))",
                                        "y[:] = np.transpose(o, (1, 0, 2))"),
    "rank bonus gated instead of clamped": (
        "return np.minimum(w, np.log(np.asarray(nj, dtype=np.float64))[None, :])",
        "return gate_second_order(w, nj)"),
    "pair bonus ignored": ("        r = r + np.asarray(bonus, np.float64)", "        r = r"),
    "margin one rank too high": ("gaps[a] = s[topk - 1] - s[topk]", "gaps[a] = s[topk - 2] - s[topk - 1]"),
    "margin one rank too low": ("gaps[a] = s[topk - 1] - s[topk]", "gaps[a] = s[topk] - s[min(topk + 1, len(s) - 1)]"),
    "margin counts band blocks as candidates": (
        "cand = r[a, (np.abs(idx - i) > band) & (idx >= n_sink)]", "cand = r[a, idx >= n_sink]"),
    "margin counts sink blocks as candidates": (
        "cand = r[a, (np.abs(idx - i) > band) & (idx >= n_sink)]", "cand = r[a, np.abs(idx - i) > band]"),
    "margin infinite one candidate early": ("if 0 < topk < len(cand):", "if 0 < topk < len(cand) - 1:"),
    "margin ignores the bias": (
        "r = route_scores(np.asarray(qbar, np.float64)[want], kbar, scale, bias, bon)",
        "r = route_scores(np.asarray(qbar, np.float64)[want], kbar, scale, None, bon)"),
    "second-order spread subtracted": ("a = a + np.asarray(spread, dtype=np.float64)[i, U][None, :]",
                                       "a = a - np.asarray(spread, dtype=np.float64)[i, U][None, :]"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    dst = tmp_path / "repo"
    os.makedirs(dst)
    shutil.copytree(os.path.join(ROOT, "oracle"), dst / "oracle")
    shutil.copytree(os.path.join(ROOT, "tests"), dst / "tests",
                    ignore=shutil.ignore_patterns("__pycache__", "test_oracle_mutations.py"))
    pkg = dst / "piecewise_sparse_attention_gb300"
    os.makedirs(pkg)
    for f in ("__init__.py", "workloads.py"):
        src = os.path.join(ROOT, "piecewise_sparse_attention_gb300", f)
        if os.path.exists(src):
            shutil.copy(src, pkg / f)
    shutil.copy(os.path.join(ROOT, "pytest.ini"), dst / "pytest.ini")
    path = dst / "oracle" / "pisa_oracle.py"
    src = path.read_text()
    assert src.count(old) >= 1, name
    path.write_text(src.replace(old, new))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py", "tests/test_oracle_hybrid_pins.py",
                        "tests/test_oracle_covariance_pins.py",
                        "tests/test_oracle_second_order_pins.py",
                        "tests/test_oracle_reorder_pins.py", "tests/test_golden.py"],
                       cwd=dst, capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"mutant '{name}' survived:\n{r.stdout[-2000:]}"
