"""The oracle's CPU pins fail on plausible mistakes planted in a copy of the oracle.

Each case copies oracle/, synth/, the pin tests with their golden fixtures and the
test configuration into a temporary tree, replaces one line of the copied oracle
with a mistake, and runs the pin tests there: every planted mistake must make them
fail.  The mistakes exist only in those copies, on the CPU.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle", "moe_oracle.py")

# (what the mistake is, the oracle's line, the line with the mistake)
MUTATIONS = [
    ("top-k ties to the higher index", 'order = np.argsort(-sel, axis=1, kind="stable")',
     'order = sel.shape[1] - 1 - np.argsort(-sel[:, ::-1], axis=1, kind="stable")'),
    ("slot order reversed", "return order[:, :k].astype(np.int32)", "return order[:, :k][:, ::-1].astype(np.int32)"),
    ("softmax gate normalised over all experts",
     "            zs = z[t, idx[t]].astype(np.float64)\n            e = np.exp(zs - zs.max())\n            w[t] = e / e.sum()",
     "            zs = z[t, idx[t]].astype(np.float64)\n            e = np.exp(zs - zs.max())\n"
     "            w[t] = e / np.exp(z[t].astype(np.float64) - zs.max()).sum()"),
    ("selection bias leaks into the sigmoid gate", "    return sel, s\n", "    return sel, sel\n"),
    ("logit bias dropped", "z = z + logit_bias.astype(np.float64)[None, :]", "z = z"),
    ("SiLU sign", "return a / (1.0 + np.exp(-a))", "return a / (1.0 + np.exp(a))"),
    ("W1 in place of W3", "h = silu(a) * (xr @ W3.T)", "h = silu(a) * (xr @ W1.T)"),
    ("ReLU left out", "    else:\n        h = np.maximum(a, 0.0)\n    return h @ W2.T", "    else:\n        h = a\n    return h @ W2.T"),
    ("capacity off by one", "return int(-((-Fraction(alpha) * T * k) // N))",
     "return int(-((-Fraction(alpha) * T * k) // N)) + 1"),
    ("capacity rounded down", "return int(-((-Fraction(alpha) * T * k) // N))",
     "return int((Fraction(alpha) * T * k) // N)"),
    ("capacity never applied", "limit = cap if cap > 0 else T * k", "limit = T * k"),
    ("every slot weighted by slot 0's gate", "out[t] += w[t, j] * y_rows[r]", "out[t] += w[t, 0] * y_rows[r]"),
    ("N missing from the balance loss", "aux = N * float(np.sum(f * P))", "aux = float(np.sum(f * P))"),
    ("P averaged over the wrong axis", "P = router_probabilities(z, gate).mean(axis=0)",
     "P = router_probabilities(z, gate).mean(axis=1)"),
    ("z-loss without the square", "return float(np.mean(lse ** 2))", "return float(np.mean(np.abs(lse)))"),
    ("bias update with the wrong sign", "out[i] += gamma", "out[i] -= gamma"),
    ("sequence loss on the batch's P", "P = p[s0:s1].mean(axis=0)", "P = p.mean(axis=0)"),
    ("E4M3 ties rounded up", "r = np.minimum(np.rint(a / quantum) * quantum, 448.0)",
     "r = np.minimum(np.floor(a / quantum + 0.5) * quantum, 448.0)"),
    ("FP8 scale from the wrong maximum", "(amax / np.float32(E4M3_MAX))", "(amax / np.float32(240.0))"),
    # the backward pass (pinned by central differences)
    ("SiLU derivative without a (1 - sig)", "da = dh * u * (sig * (1.0 + a * (1.0 - sig)))   # d SiLU(a) / da",
     "da = dh * u * sig   # d SiLU(a) / da"),
    ("up-projection gradient without a", "du = dh * a * sig\n        dW2 = dy.T @ h",
     "du = dh * sig\n        dW2 = dy.T @ h"),
    ("dW1 from the up-projection gradient", "dW1 = da.T @ xr", "dW1 = du.T @ xr"),
    ("ReLU backward passes negatives", "    da = dh * (a > 0)\n    return da @ W1, da.T @ xr, None, dy.T @ h",
     "    da = dh\n    return da @ W1, da.T @ xr, None, dy.T @ h"),
    ("softmax gate Jacobian uncentred", "dz[idx_t] = w_t * (g - np.sum(w_t * g))", "dz[idx_t] = w_t * g"),
    ("sigmoid derivative without (1 - s)", "dz[idx_t] = ds * s * (1.0 - s)", "dz[idx_t] = ds * s"),
]


def _run_mutant(case):
    name, old, new = case
    with tempfile.TemporaryDirectory() as tmp:
        for d in ("oracle", "synth"):
            shutil.copytree(os.path.join(ROOT, d), os.path.join(tmp, d),
                            ignore=shutil.ignore_patterns("__pycache__"))
        os.makedirs(os.path.join(tmp, "tests"))
        for f in ("conftest.py", "test_oracle_pins.py"):
            shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(tmp, "tests", f))
        shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(tmp, "tests", "golden"))
        path = os.path.join(tmp, "oracle", "moe_oracle.py")
        with open(path) as fh:
            src = fh.read()
        with open(path, "w") as fh:
            fh.write(src.replace(old, new, 1))
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                            os.path.join("tests", "test_oracle_pins.py")],
                           cwd=tmp, capture_output=True, text=True, timeout=600)
        return name, r.returncode, r.stdout[-400:]


def test_each_mutation_targets_exactly_one_line():
    with open(ORACLE) as fh:
        src = fh.read()
    for name, old, _ in MUTATIONS:
        assert src.count(old) == 1, name


def test_pins_catch_every_planted_mistake():
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(_run_mutant, MUTATIONS))
    survivors = [(name, out) for name, rc, out in results if rc == 0]
    assert not survivors, f"pins passed with a planted mistake: {[s[0] for s in survivors]}"


def test_unmutated_copy_passes():
    """The copied tree itself is sound: with no mistake planted the pins pass there."""
    name, rc, out = _run_mutant(("none", "", ""))
    assert rc == 0, out
