"""The product path has no fallback: without librz.so every entry point
raises, no module of the package touches the CPU oracle, and the library
itself refuses (rather than computes) when there is no sm_103 device."""

import ast
import os

import pytest
import torch

import invariant_logprobs_gb300 as rz

PKG = os.path.dirname(os.path.abspath(rz.__file__))


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(rz, "_lib", None)
    monkeypatch.setattr(rz, "LIB_PATH", str(tmp_path / "librz.so"))
    with pytest.raises(RuntimeError, match="not built"):
        rz.load()
    # every wrapper goes through load() before touching its arguments
    for name in ("rz_token_logprob", "rz_loss_fwd_bwd", "rz_sc_loss_fwd_bwd",
                 "rz_logits_loss_fwd_bwd", "rz_group_advantage", "rz_is_loss", "rz_d3",
                 "rz_is_stats", "rz_lmhead_logits", "rz_sample_logprob",
                 "rz_token_logprob_noalloc", "rz_loss_fwd_bwd_shard", "rz_sum_partials",
                 "rz_loss_fwd_bwd_ref"):
        fn = getattr(rz, name)
        n_required = fn.__code__.co_argcount - len(fn.__defaults__ or ())
        with pytest.raises(RuntimeError, match="not built"):
            fn(*([None] * n_required))


def test_package_never_imports_the_oracle():
    for root, _, files in os.walk(PKG):
        for f in files:
            if not f.endswith(".py"):
                continue
            tree = ast.parse(open(os.path.join(root, f)).read())
            for node in ast.walk(tree):
                if isinstance(node, ast.Import):
                    names = [a.name for a in node.names]
                elif isinstance(node, ast.ImportFrom):
                    names = [node.module or ""]
                else:
                    continue
                assert not any(n == "oracle" or n.startswith("oracle.") for n in names), (f, names)


def test_library_refuses_without_a_gpu():
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import ctypes
    from invariant_logprobs_gb300 import build
    lib = rz.load(build.build())
    # a well-formed group-advantage call: no sm_103 device, so nothing runs
    fake = ctypes.c_void_p(1 << 20)
    assert lib.rz_group_advantage(fake, 8, 4, fake, None) == rz.RZ_ERR_UNSUPPORTED
