"""Mutation check of the oracle's pins, planted on the CPU: each mutant is
the oracle's source with one plausible mistake (a sign, a wrong count, a
wrong mean, a clipped weight, a missing term, ...), loaded as a module of its
own and put in place of `oracle` while the fixed pins of test_oracle.py run
(sampler mutants: in place of the sampler oracle, against its own pins).
Every mutant must fail at least one pin; the unmutated source must fail
none (so the harness itself is sound).  The oracle package is never
modified."""

import inspect
import types

import numpy as np
import pytest

import oracle
import oracle.rz_oracle
import oracle.rz_sampler
import test_oracle as pins
import test_oracle_sampler as sampler_pins

SRC = open(oracle.rz_oracle.__file__).read()
SAMPLER_SRC = open(oracle.rz_sampler.__file__).read()

# name -> [(fragment of the oracle's source, replacement)]; every fragment
# must occur in the source (all occurrences are replaced).
MUTANTS = {
    "one-hot sign in dz": [("p[np.arange(e - s), tokens[s:e]] -= 1.0",
                            "p[np.arange(e - s), tokens[s:e]] += 1.0")],
    "dW sign": [("dW += dz.T @ Hd[s:e]", "dW -= dz.T @ Hd[s:e]")],
    "T in place of T_i": [("total += A[i] * w[s:e][v].sum() / Ti",
                           "total += A[i] * w[s:e][v].sum() / T"),
                          ("np.where(v, A[i] * w[s:e] / (B * Ti), 0.0)",
                           "np.where(v, A[i] * w[s:e] / (B * T), 0.0)")],
    "1/T in place of 1/B in the loss": [("loss = -total / B if B > 0 else 0.0",
                                         "loss = -total / T if T > 0 else 0.0")],
    "weight dropped from c (plain REINFORCE)": [("np.where(v, A[i] * w[s:e] / (B * Ti), 0.0)",
                                                 "np.where(v, A[i] / (B * Ti), 0.0)")],
    "weight clipped at 2": [("    w = np.exp(lp - lm)\n    c = np.zeros",
                             "    w = np.minimum(np.exp(lp - lm), 2.0)\n    c = np.zeros")],
    "global instead of group mean": [("(g - g.mean(axis=1, keepdims=True))", "(g - g.mean())")],
    "advantage divided by the group std": [
        ("(g - g.mean(axis=1, keepdims=True))",
         "((g - g.mean(axis=1, keepdims=True)) / (g.std(axis=1, keepdims=True) + 1e-6))")],
    "D3 with + log w": [("np.mean(w - 1.0 - np.log(w))", "np.mean(w - 1.0 + np.log(w))")],
    "mask ignored in T_i": [("        Ti = int(v.sum())\n", "        Ti = e - s\n")],
    "log-sum-exp without the max": [("return m[:, 0] + np.log(np.exp(z - m).sum(axis=1))",
                                     "return np.log(np.exp(z).sum(axis=1))")],
    "gather off by one": [("lp[s:s + _ROW_BLOCK] = z[np.arange(r.shape[0]), tokens[r]] - l",
                           "lp[s:s + _ROW_BLOCK] = z[np.arange(r.shape[0]), "
                           "(tokens[r] + 1) % z.shape[1]] - l")],
    "SC mean over all responses": [("abar = A[nonempty].mean() if nonempty.any() else 0.0",
                                    "abar = A.mean() if B > 0 else 0.0")],
    "SC without centring": [("abar = A[nonempty].mean() if nonempty.any() else 0.0",
                             "abar = 0.0")],
    "one-hot sign in the given-logits dz": [("p[np.arange(rr.shape[0]), tokens[rr]] -= 1.0",
                                             "p[np.arange(rr.shape[0]), tokens[rr]] += 1.0")],
    "dH sign": [("dH[s:e] = dz @ Wd", "dH[s:e] = -(dz @ Wd)")],
    "k1 sign": [('"k1": float(np.mean(-d))', '"k1": float(np.mean(d))')],
    "k2 without the 1/2": [("np.mean(d * d / 2.0)", "np.mean(d * d)")],
    "mean in place of median": [("np.max(x) / np.median(x)", "np.max(x) / np.mean(x)")],
    "SC counts ignore the mask": [("counts = np.array([int(valid[cu[i]:cu[i + 1]].sum())",
                                   "counts = np.array([int(cu[i + 1] - cu[i])")],
    "strided instead of contiguous groups": [("g = r.reshape(B // G, G)",
                                              "g = r.reshape(G, B // G).T")],
    "w without the exponential": [("    w = np.exp(lp - lm)\n    c = np.zeros",
                                   "    w = 1.0 + (lp - lm)\n    c = np.zeros")],
}


# mistakes in the sampler oracle, against the sampler's pins
SAMPLER_MUTANTS = {
    "U on the closed interval": [("+ 0.5) * 2.0 ** -23", "+ 0.0) * 2.0 ** -23")],
    "Philox with 7 rounds": [("    for _ in range(10):", "    for _ in range(7):")],
    "recorded log mu of the wrong token": [("logmu = z[rows, final] - lse",
                                            "logmu = z[rows, (final + 1) % V] - lse")],
    "chunk kept against the sum before it": [("rep = u1 * R < Wc", "rep = u1 * (R - Wc) < Wc")],
    "segment kept against the sum before it": [("rep = (u3 * Rp < Qg) & (cand >= 0)",
                                                "rep = (u3 * (Rp - Qg) < Qg) & (cand >= 0)")],
    "draw by column instead of by class": [
        ("return np.array([j for k in range(4) for j in range(k, n, 4)], dtype=np.int64)",
         "return np.arange(n, dtype=np.int64)")],
    "one tile per segment": [("    tps = (nt + n - 1) // n\n", "    tps = 1\n")],
    "both draws from word 0": [("u1, u2 = uniform_of(x[:, 0]), uniform_of(x[:, 1])",
                                "u1, u2 = uniform_of(x[:, 0]), uniform_of(x[:, 0])")],
}


def _module(pairs):
    src = SRC
    for old, new in pairs:
        assert old in src, "mutation target not in the oracle source: %r" % old
        src = src.replace(old, new)
    mod = types.ModuleType("oracle_mutant")
    mod.__dict__["__file__"] = oracle.rz_oracle.__file__
    exec(compile(src, "<oracle mutant>", "exec"), mod.__dict__)
    names = [n for n in dir(oracle) if not n.startswith("_") and callable(getattr(oracle, n))]
    return types.SimpleNamespace(**{n: getattr(mod, n) for n in names})


def _pins():
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if name.startswith("test_") and not inspect.signature(fn).parameters:
            out.append((name, fn))
    return out


def _failing_pins(ns, monkeypatch):
    monkeypatch.setattr(pins, "oracle", ns)
    failed = []
    with np.errstate(all="ignore"):
        for name, fn in _pins():
            try:
                fn()
            except Exception:  # an assertion, or a crash on a broken shape
                failed.append(name)
    monkeypatch.undo()
    return failed


def test_unmutated_source_passes_every_pin(monkeypatch):
    assert len(_pins()) >= 25
    assert _failing_pins(_module([]), monkeypatch) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_every_mutant_fails_a_pin(name, monkeypatch):
    failed = _failing_pins(_module(MUTANTS[name]), monkeypatch)
    assert failed, "no pin catches the mutant %r" % name


def _sampler_module(pairs):
    src = SAMPLER_SRC
    for old, new in pairs:
        assert old in src, "mutation target not in the sampler source: %r" % old
        src = src.replace(old, new)
    mod = types.ModuleType("sampler_mutant")
    exec(compile(src, "<sampler mutant>", "exec"), mod.__dict__)
    return mod


def _failing_sampler_pins(mod, monkeypatch, first_only=False):
    """Sampler pins that fail with `mod` in place of the sampler oracle; the
    cheap ones (known answers, the U grid) run before the sampling ones, and
    first_only stops at the first failure."""
    monkeypatch.setattr(sampler_pins, "rz_sampler", mod)
    fns = [(n, f) for n, f in inspect.getmembers(sampler_pins, inspect.isfunction)
           if n.startswith("test_") and not inspect.signature(f).parameters]
    fns.sort(key=lambda nf: ("sampling" in nf[0], nf[0]))
    failed = []
    with np.errstate(all="ignore"):
        for name, fn in fns:
            try:
                fn()
            except Exception:
                failed.append(name)
                if first_only:
                    break
    monkeypatch.undo()
    return failed


def test_unmutated_sampler_passes_every_pin(monkeypatch):
    assert _failing_sampler_pins(_sampler_module([]), monkeypatch) == []


@pytest.mark.parametrize("name", sorted(SAMPLER_MUTANTS))
def test_every_sampler_mutant_fails_a_pin(name, monkeypatch):
    failed = _failing_sampler_pins(_sampler_module(SAMPLER_MUTANTS[name]), monkeypatch,
                                   first_only=True)
    assert failed, "no sampler pin catches the mutant %r" % name
