"""CPU checks of the C ABI boundary: the library builds and loads without a
GPU, exports every function include/rz.h declares, and its host-side
argument checks return the documented status codes before touching CUDA."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rz.h")


@pytest.fixture(scope="module")
def lib():
    from invariant_logprobs_gb300 import build
    import invariant_logprobs_gb300 as rz
    path = build.build()
    return rz.load(path)


def _declared():
    src = open(HEADER).read()
    return re.findall(r"^RZ_API\s+[\w\s\*]+?\b(rz_\w+)\s*\(", src, flags=re.M)


def test_header_declares_the_boundary():
    names = set(_declared())
    for n in ["rz_token_logprob", "rz_loss_fwd_bwd", "rz_group_advantage", "rz_d3",
              "rz_is_loss", "rz_logits_loss_fwd_bwd", "rz_workspace_size", "rz_status_string",
              "rz_lmhead_logits"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    import invariant_logprobs_gb300 as rz
    assert rz.status_string(0) == "ok"
    for s in range(1, 5):
        assert rz.status_string(s) and rz.status_string(s) != "unknown status"
    assert rz.status_string(99) == "unknown status"


def test_workspace_sizes(lib):
    import invariant_logprobs_gb300 as rz
    V = 151936
    # logprob pass: per row S=60 (max, sum) pairs + one gathered logit
    # (594 vocab tiles in groups of 10)
    s = rz.workspace_size(rz.RZ_OP_TOKEN_LOGPROB, 1000, 2560, V, 0)
    assert s >= 1000 * (60 * 8 + 4)
    # independent of d, monotone in T
    assert s == rz.workspace_size(rz.RZ_OP_TOKEN_LOGPROB, 1000, 64, V, 0)
    assert rz.workspace_size(rz.RZ_OP_TOKEN_LOGPROB, 2000, 64, V, 0) > s
    # learner: one chunk of at most 38912 rows x V kept fp16 terms (dz in
    # place) plus a running max per 32 columns (2.125 bytes per logit), split
    # states of one chunk, log pi
    big = rz.workspace_size(rz.RZ_OP_LOSS_FWD_BWD, 1_114_112, 2560, V, 128)
    per_row = V * 2 + (V + 31) // 32 * 4
    assert 38912 * per_row <= big < 38912 * per_row + 38912 * (64 * 8 + 16) + 1_114_112 * 4 + 10**6
    # a short batch only needs its own rows (rounded up to 128)
    small = rz.workspace_size(rz.RZ_OP_LOSS_FWD_BWD, 300, 256, 1024, 8)
    assert 384 * (1024 * 2 + 32 * 4) < small < 384 * (1024 * 2 + 32 * 4) + (1 << 20)
    assert rz.workspace_size(rz.RZ_OP_IS_LOSS, 10, 0, 0, 256) >= 256 * 24
    assert rz.workspace_size(99, 10, 10, 10, 10) == 0
    # a vocabulary so large that 38,912 rows of kept terms would pass 40 GiB:
    # the chunk shrinks to the largest multiple of 128 rows that fits
    V = 1 << 20
    per_row = V * 2 + (V // 128) * 4 * 4
    rows = (40 << 30) // per_row // 128 * 128
    assert rows == 19200
    huge = rz.workspace_size(rz.RZ_OP_LOSS_FWD_BWD, 10**6, 64, V, 8)
    assert rows * per_row <= huge < rows * per_row + rows * (64 * 8 + 16) + 10**6 * 4 + 10**6
    assert huge <= (40 << 30) + (64 << 20)


def _no_gpu():
    """Calls with fake pointers run only where no GPU is visible: there the
    library cannot launch anything even if a check were missed."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("fake-pointer calls are kept off machines with a GPU")


def test_host_side_argument_checks(lib):
    _no_gpu()
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: every call below fails validation first
    null = None
    # B % G != 0
    assert lib.rz_group_advantage(fake, 10, 4, fake, null) == 1
    assert lib.rz_group_advantage(fake, 8, 0, fake, null) == 1
    # Checks that answer 2 (alignment, d % 8) come before the workspace
    # check, so these calls pass no workspace: a missing check would answer 3
    # here instead of 2 (without a GPU, a call that passes every check
    # also answers 2).
    # d not a multiple of 8
    assert lib.rz_token_logprob(fake, fake, fake, 5, 12, 100, fake, null, null, 0,
                                null, null) == 2
    # missing pointers
    assert lib.rz_token_logprob(null, fake, fake, 5, 16, 100, fake, null, fake, 1 << 20,
                                null, null) == 1
    # V out of range
    assert lib.rz_token_logprob(fake, fake, fake, 5, 16, 0, fake, null, fake, 1 << 20,
                                null, null) == 1
    # misaligned H
    assert lib.rz_token_logprob(P((1 << 20) + 2), fake, fake, 5, 16, 100, fake, null, null,
                                0, null, null) == 2
    # workspace too small / missing
    assert lib.rz_token_logprob(fake, fake, fake, 5, 16, 100, fake, null, fake, 8,
                                null, null) == 3
    assert lib.rz_token_logprob(fake, fake, fake, 5, 16, 100, fake, null, null, 1 << 30,
                                null, null) == 3
    # B = 0 with tokens
    assert lib.rz_loss_fwd_bwd(fake, fake, fake, fake, fake, fake, null, 0, 5, 16, 100, fake,
                               fake, null, fake, fake, fake, 1 << 30, null, null) == 1
    # logits variant needs V % 8 == 0
    assert lib.rz_logits_loss_fwd_bwd(fake, fake, fake, fake, fake, null, 2, 10, 100, fake, fake,
                                      fake, null, 0, null, null) == 2
    # is_loss: missing outputs
    assert lib.rz_is_loss(fake, fake, fake, fake, null, 2, 10, null, fake, null, fake, 1 << 20,
                          null, null) == 1
    assert lib.rz_d3(fake, fake, -1, fake, null) == 1
    # shard of a data-parallel step: the batch cannot hold fewer responses
    # than the shard, nor none when the shard has some
    assert lib.rz_loss_fwd_bwd_shard(fake, fake, fake, fake, null, fake, fake, null, 4, 3, 5, 16,
                                     100, fake, fake, null, fake, fake, fake, 1 << 30, null,
                                     null) == 1
    assert lib.rz_loss_fwd_bwd_shard(fake, fake, fake, fake, null, fake, fake, null, 4, 0, 5, 16,
                                     100, fake, fake, null, fake, fake, fake, 1 << 30, null,
                                     null) == 1
    # ... and is otherwise checked as rz_loss_fwd_bwd (d % 8 answers 2)
    assert lib.rz_loss_fwd_bwd_shard(fake, fake, fake, fake, null, fake, fake, null, 4, 8, 5, 12,
                                     100, fake, fake, null, fake, fake, null, 0, null, null) == 2
    # the reference variant needs its reference rows
    assert lib.rz_loss_fwd_bwd_ref(fake, fake, fake, fake, null, fake, fake, null, 2, 5, 16, 100,
                                   fake, fake, null, fake, fake, fake, 1 << 30, null, null) == 1
    assert lib.rz_loss_fwd_bwd_ref(fake, fake, fake, fake, fake, fake, fake, null, 2, 5, 12, 100,
                                   fake, fake, null, fake, fake, null, 0, null, null) == 2
    # its workspace has no running maxima but the chunk's rows of H scaled
    T, d, V, B = 5000, 512, 151936, 8
    plain = lib.rz_workspace_size(1, T, d, V, B)
    ref = lib.rz_workspace_size(6, T, d, V, B)
    rows = 5120  # the chunk of 5,000 rows, rounded to whole 128-row blocks
    assert ref - plain == rows * d * 2 - rows * ((V + 127) // 128 * 4) * 4
    # the exchange sum: at least one part, non-negative count, pointers
    assert lib.rz_sum_partials(fake, 0, 10, fake, null) == 1
    assert lib.rz_sum_partials(fake, 2, -1, fake, null) == 1
    assert lib.rz_sum_partials(null, 2, 10, fake, null) == 1
    assert lib.rz_sum_partials(null, 2, 0, null, null) == 0  # nothing to add


def test_valid_call_without_gpu_reports_unsupported(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    fake = ctypes.c_void_p(1 << 20)
    # valid arguments, but no sm_103 device: refused, nothing launched
    assert lib.rz_d3(fake, fake, 10, fake, None) == 2


def test_peak_to_median_host_function(lib):
    import numpy as np
    import invariant_logprobs_gb300 as rz
    import oracle
    rng = np.random.default_rng(4)
    for n in (1, 2, 7, 100):
        x = (rng.random(n) + 0.1).astype(np.float32)
        assert rz.rz_peak_to_median(list(x)) == pytest.approx(oracle.peak_to_median(x), rel=1e-12)
    out = ctypes.c_double(0)
    assert lib.rz_peak_to_median(None, 3, ctypes.byref(out)) == 1


def _declared_arity():
    """name -> number of parameters, parsed from the prototypes in rz.h."""
    src = open(HEADER).read()
    out = {}
    for m in re.finditer(r"^RZ_API\s+[\w\s\*]+?\b(rz_\w+)\s*\(([^)]*)\)\s*;", src, flags=re.M):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_the_header(lib):
    import invariant_logprobs_gb300 as rz
    arity = _declared_arity()
    assert set(arity) == set(_declared())
    for name, n in arity.items():
        assert name in rz._SIGNATURES, name
        assert len(rz._SIGNATURES[name][1]) == n, name


def test_more_host_side_argument_checks(lib):
    _no_gpu()
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: every call below fails validation first
    odd = P((1 << 20) + 8)  # 8-byte but not 16-byte aligned
    null = None
    big = 1 << 40
    # Score Centering learner: B = 0 with tokens, missing dW, d % 8, misaligned
    # dW, workspace too small
    sc = lib.rz_sc_loss_fwd_bwd
    assert sc(fake, fake, fake, fake, fake, null, 0, 5, 16, 100, fake, null, fake, fake,
              fake, big, null, null) == 1
    assert sc(fake, fake, fake, fake, fake, null, 2, 5, 16, 100, fake, null, fake, null,
              fake, big, null, null) == 1
    # (the 2-answers pass no workspace, as above)
    assert sc(fake, fake, fake, fake, fake, null, 2, 5, 12, 100, fake, null, fake, fake,
              null, 0, null, null) == 2
    assert sc(fake, fake, fake, fake, fake, null, 2, 5, 16, 100, fake, null, fake, odd,
              null, 0, null, null) == 2
    assert sc(fake, fake, fake, fake, fake, null, 2, 5, 16, 100, fake, null, fake, fake,
              fake, 64, null, null) == 3
    # IS learner: D3 output and log mu are required
    isl = lib.rz_loss_fwd_bwd
    assert isl(fake, fake, fake, fake, fake, fake, null, 2, 5, 16, 100, fake, null, null,
               fake, fake, fake, big, null, null) == 1
    assert isl(fake, fake, fake, null, fake, fake, null, 2, 5, 16, 100, fake, fake, null,
               fake, fake, fake, big, null, null) == 1
    # fused sampler: missing tokens_out, d % 8, missing workspace; T = 0 is a no-op
    smp = lib.rz_sample_logprob
    assert smp(fake, fake, null, 5, 16, 100, 1, null, fake, null, fake, big, null, null) == 1
    assert smp(fake, fake, null, 5, 20, 100, 1, fake, fake, null, null, 0, null, null) == 2
    assert smp(fake, fake, null, 5, 16, 100, 1, fake, fake, null, null, big, null, null) == 3
    assert smp(null, null, null, 0, 16, 100, 1, null, null, null, null, 0, null, null) == 0
    # logits: missing output, misaligned W
    assert lib.rz_lmhead_logits(fake, fake, 5, 16, 100, null, null, null) == 1
    assert lib.rz_lmhead_logits(fake, odd, 5, 16, 100, fake, null, null) == 2
    # no-alloc entry point: past its built-in scratch, bad d
    assert lib.rz_token_logprob_noalloc(fake, fake, fake, 10_000_000, 16, 151936, fake, null,
                                        null, null) == 5
    assert lib.rz_token_logprob_noalloc(fake, fake, fake, 5, 7, 100, fake, null, null,
                                        null) == 1
    # self-test: the wait limit must be 1 us .. 2 s and the flag present
    assert lib.rz_selftest_wait_timeout(fake, null, 0, null) == 1
    assert lib.rz_selftest_wait_timeout(fake, null, 2_000_001, null) == 1
    assert lib.rz_selftest_wait_timeout(null, null, 1000, null) == 1
    # diagnostics: negative T
    assert lib.rz_is_stats(fake, fake, -1, fake, null) == 1
    assert lib.rz_d3(null, null, 5, fake, null) == 1


def test_vocab_splits_depend_on_v_only(lib):
    """The logprob pass keeps T x S split states (8 bytes each) plus one
    gathered logit per row; S groups consecutive 256-column vocab tiles,
    at most 64 groups, and is a function of V alone (never of T), which is
    what fixes each row's reduction order whatever batch it is in."""
    import invariant_logprobs_gb300 as rz

    def splits(V, T=512):
        # past the decode-sized batches (at most 64 rows), which also hold
        # their logits
        ws = rz.workspace_size(rz.RZ_OP_TOKEN_LOGPROB, T, 64, V, 0)
        return (ws - 2048) // (T * 8)  # T * 4 bytes of gathered logits -> 2048 bytes at T = 512

    def rule(V):
        tiles = -(-V // 256)
        per = -(-tiles // min(tiles, 64))
        return -(-tiles // per)

    for V, want in [(1, 1), (256, 1), (257, 2), (16384, 64), (16385, 33), (151936, 60),
                    (1 << 24, 64)]:
        assert splits(V) == want == rule(V), V
    for T in (512, 1024, 4096):
        assert splits(151936, T) == 60
    # a decode-sized batch's workspace adds its logits, [T, V rounded up to 64] fp32
    for T in (1, 7, 64):
        extra = rz.workspace_size(rz.RZ_OP_TOKEN_LOGPROB, T, 64, 151936, 0) - \
            (-(-T * 60 * 8 // 256) * 256 + -(-T * 4 // 256) * 256)
        assert extra == -(-T * 151936 * 4 // 256) * 256, T


def test_profile_classes_and_host_side_behaviour(lib):
    """The timing hook's class ids match the binding's names; without a
    recorded call it returns zeros; a short output array is refused."""
    import invariant_logprobs_gb300 as rz
    src = open(HEADER).read()
    ids = {m.group(1): int(m.group(2))
           for m in re.finditer(r"#define RZ_PROF_(\w+)\s+(\d+)", src)}
    assert ids.pop("CLASSES") == len(rz.RZ_PROF_NAMES)
    assert sorted(ids.values()) == list(range(len(rz.RZ_PROF_NAMES)))
    assert [n.lower() for n, _ in sorted(ids.items(), key=lambda kv: kv[1])] == \
        [n.lower() for n in rz.RZ_PROF_NAMES]
    rz.rz_profile_begin()
    got = rz.rz_profile_end()
    assert got == {n: (0.0, 0) for n in rz.RZ_PROF_NAMES}
    ms = (ctypes.c_float * 3)()
    assert lib.rz_profile_end(ms, None, 3) == rz.RZ_ERR_INVALID_ARG
    assert lib.rz_profile_end(None, None, len(rz.RZ_PROF_NAMES)) == rz.RZ_ERR_INVALID_ARG
