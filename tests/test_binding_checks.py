"""CPU checks of the Python binding's argument marshalling.

Tensors here are host tensors of a subclass that reports itself as a CUDA
tensor on a chosen device; nothing is ever dereferenced as a device pointer.
A valid call must pass every binding check and reach the library, whose
only answer without an sm_103 device is RZ_ERR_UNSUPPORTED (its own
argument checks run first, so a wrongly marshalled call can come back as 1
or 3 instead).  Bad buffers (wrong dtype, too small, another device, a
non-byte workspace) must be refused in Python before the library is called.
"""


import pytest
import torch

import invariant_logprobs_gb300 as rz


def _fake_cls(index):
    class FakeCuda(torch.Tensor):
        @property
        def is_cuda(self):
            return True

        @property
        def device(self):
            return torch.device("cuda", index)

    return FakeCuda


CUDA0 = _fake_cls(0)
CUDA1 = _fake_cls(1)


class _Stream:
    def __init__(self, index=0):
        self.device = torch.device("cuda", index)
        self.cuda_stream = 0


def dev(t, cls=CUDA0):
    return t.as_subclass(cls)


def zeros(*shape, dtype=torch.float32, cls=CUDA0):
    return dev(torch.zeros(*shape, dtype=dtype), cls)


def workspace(nbytes, cls=CUDA0):
    """A uint8 buffer whose start is 256-byte aligned, as the library asks."""
    buf = torch.zeros(nbytes + 512, dtype=torch.uint8)
    off = (-buf.data_ptr()) % 256
    return dev(buf[off:off + max(nbytes, 256)], cls)


# Host tensors posing as device tensors must never reach a real GPU: with
# one present the library would launch on them.
pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="fake device tensors are kept off machines with a GPU")


@pytest.fixture(scope="module")
def lib():
    from invariant_logprobs_gb300 import build
    return rz.load(build.build())


@pytest.fixture(autouse=True)
def current_device_0(monkeypatch):
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)


T, d, V, B = 6, 16, 104, 2
S = _Stream()


def _problem():
    H = zeros(T, d, dtype=torch.bfloat16)
    W = zeros(V, d, dtype=torch.bfloat16)
    tok = zeros(T, dtype=torch.int32)
    logmu = zeros(T)
    cu = dev(torch.tensor([0, 2, T], dtype=torch.int64))
    adv = zeros(B)
    return H, W, tok, logmu, cu, adv


def _unsupported(fn, *a, **k):
    with pytest.raises(rz.RzError) as e:
        fn(*a, **k)
    assert e.value.status == rz.RZ_ERR_UNSUPPORTED, e.value


def test_valid_calls_reach_the_library(lib):
    H, W, tok, logmu, cu, adv = _problem()
    err = zeros(1, dtype=torch.int32)
    lp, lse = zeros(T), zeros(T)
    _unsupported(rz.rz_token_logprob, H, W, tok, logprob_out=lp, lse_out=lse,
                 ws=workspace(rz.workspace_size(rz.RZ_OP_TOKEN_LOGPROB, T, d, V, 0)),
                 err_flag=err, stream=S)
    _unsupported(rz.rz_token_logprob_noalloc, H, W, tok, lp, lse_out=lse, err_flag=err, stream=S)
    _unsupported(rz.rz_sample_logprob, H, W, 5, row_ids=zeros(T, dtype=torch.int64),
                 tokens_out=zeros(T, dtype=torch.int32), logprob_out=lp, lse_out=lse,
                 ws=workspace(rz.workspace_size(rz.RZ_OP_SAMPLE, T, d, V, 0)), err_flag=err,
                 stream=S)
    _unsupported(rz.rz_lmhead_logits, H, W, logits_out=zeros(T, V), err_flag=err, stream=S)
    learn_ws = workspace(rz.workspace_size(rz.RZ_OP_LOSS_FWD_BWD, T, d, V, B))
    outs = dict(logprob_out=lp, dH=zeros(T, d, dtype=torch.bfloat16), dW=zeros(V, d),
                loss_out=zeros(1), ws=learn_ws, err_flag=err, stream=S,
                action_mask=zeros(T, dtype=torch.uint8))
    _unsupported(rz.rz_loss_fwd_bwd, H, W, tok, logmu, cu, adv, d3_out=zeros(1), **outs)
    ref_outs = dict(outs, ws=workspace(rz.workspace_size(rz.RZ_OP_LOSS_FWD_BWD_REF, T, d, V, B)))
    _unsupported(rz.rz_loss_fwd_bwd_ref, H, W, tok, logmu, zeros(T), cu, adv, d3_out=zeros(1),
                 **ref_outs)
    _unsupported(rz.rz_loss_fwd_bwd_shard, H, W, tok, logmu, cu, adv, 2 * B, d3_out=zeros(1),
                 ref_lse=zeros(T), **ref_outs)
    _unsupported(rz.rz_sc_loss_fwd_bwd, H, W, tok, cu, adv, **outs)
    _unsupported(rz.rz_logits_loss_fwd_bwd, zeros(T, V, dtype=torch.bfloat16), tok, logmu, cu,
                 adv, logprob_out=lp, loss_out=zeros(1), d3_out=zeros(1),
                 ws=workspace(rz.workspace_size(rz.RZ_OP_LOGITS_LOSS, T, 0, V, B)),
                 err_flag=err, stream=S)
    _unsupported(rz.rz_is_loss, lp, logmu, cu, adv, loss_out=zeros(1), d3_out=zeros(1),
                 coef_out=zeros(T), ws=workspace(rz.workspace_size(rz.RZ_OP_IS_LOSS, T, 0, 0, B)),
                 err_flag=err, stream=S)
    _unsupported(rz.rz_d3, lp, logmu, d3_out=zeros(1), stream=S)
    _unsupported(rz.rz_is_stats, lp, logmu, stats_out=zeros(7), stream=S)
    _unsupported(rz.rz_group_advantage, zeros(4), 2, adv_out=zeros(4), stream=S)
    _unsupported(rz.rz_selftest_wait_timeout, err, zeros(1, dtype=torch.int32), stream=S)


def test_output_buffers_are_checked_before_the_call(lib):
    H, W, tok, logmu, cu, adv = _problem()
    lws = workspace(rz.workspace_size(rz.RZ_OP_LOGITS_LOSS, T, 0, V, B))
    logits = zeros(T, V, dtype=torch.bfloat16)
    # a bf16 logprob buffer would take 4 bytes per row into 2
    with pytest.raises(TypeError):
        rz.rz_logits_loss_fwd_bwd(logits, tok, logmu, cu, adv, ws=lws, stream=S,
                                  logprob_out=zeros(T, dtype=torch.bfloat16),
                                  loss_out=zeros(1), d3_out=zeros(1))
    # empty scalar outputs
    with pytest.raises(ValueError):
        rz.rz_logits_loss_fwd_bwd(logits, tok, logmu, cu, adv, ws=lws, stream=S,
                                  logprob_out=zeros(T), loss_out=zeros(0), d3_out=zeros(1))
    with pytest.raises(ValueError):
        rz.rz_d3(zeros(T), logmu, d3_out=zeros(0), stream=S)
    with pytest.raises(ValueError):
        rz.rz_is_stats(zeros(T), logmu, stats_out=zeros(6), stream=S)
    # the error flag is one int32
    with pytest.raises(TypeError):
        rz.rz_token_logprob(H, W, tok, logprob_out=zeros(T), err_flag=zeros(1, dtype=torch.int64),
                            ws=workspace(4096), stream=S)
    # the workspace is counted in bytes: only uint8 is accepted
    with pytest.raises(TypeError):
        rz.rz_token_logprob(H, W, tok, logprob_out=zeros(T), ws=zeros(4096), stream=S)
    # sampler outputs
    with pytest.raises(TypeError):
        rz.rz_sample_logprob(H, W, 1, tokens_out=zeros(T), logprob_out=zeros(T),
                             ws=workspace(1 << 16), stream=S)
    with pytest.raises(ValueError):
        rz.rz_sample_logprob(H, W, 1, tokens_out=zeros(T - 1, dtype=torch.int32),
                             logprob_out=zeros(T), ws=workspace(1 << 16), stream=S)
    with pytest.raises(TypeError):
        rz.rz_selftest_wait_timeout(zeros(1, dtype=torch.int32), done_out=zeros(1), stream=S)


def test_device_mismatches_are_refused(lib):
    H, W, tok, logmu, cu, adv = _problem()
    # one tensor on another device
    with pytest.raises(ValueError):
        rz.rz_token_logprob(H, W, tok, logprob_out=zeros(T, cls=CUDA1), ws=workspace(4096),
                            stream=S)
    # everything on cuda:1 while the current device is cuda:0
    H1, W1, t1 = dev(torch.zeros(T, d, dtype=torch.bfloat16), CUDA1), \
        dev(torch.zeros(V, d, dtype=torch.bfloat16), CUDA1), \
        dev(torch.zeros(T, dtype=torch.int32), CUDA1)
    with pytest.raises(ValueError, match="current device"):
        rz.rz_token_logprob(H1, W1, t1, logprob_out=zeros(T, cls=CUDA1),
                            ws=workspace(4096, CUDA1), stream=_Stream(1))
    # a stream of another device
    with pytest.raises(ValueError, match="stream"):
        rz.rz_token_logprob(H, W, tok, logprob_out=zeros(T), ws=workspace(4096),
                            stream=_Stream(1))
