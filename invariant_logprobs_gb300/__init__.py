"""Python binding of the rz C ABI (include/rz.h).

Argument marshalling only: each function below checks dtypes/devices,
allocates outputs and scratch with torch when the caller did not pass them,
and calls the C entry point of the same name on the current CUDA stream.
Every step of the computation runs in librz.so's CUDA kernels; there is no
Python, torch or CPU implementation behind these names.  If the library is
missing, load() raises -- it never falls back.

Build the library with ``python -m invariant_logprobs_gb300.build`` (or
``__graft_entry__.build()``).
"""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librz.so")
# the debug build with device bounds checks (build.build(checks=True)); used
# instead of librz.so when the environment sets RZ_LIB_VARIANT=checks
LIB_PATH_CHECKS = os.path.join(_HERE, "librz_checks.so")

RZ_OK = 0
RZ_ERR_INVALID_ARG = 1
RZ_ERR_UNSUPPORTED = 2
RZ_ERR_WORKSPACE = 3
RZ_ERR_CUDA = 4
RZ_ERR_TOO_LARGE = 5

RZ_DEVERR_TOKEN_RANGE = 1
RZ_DEVERR_CU_SEQLENS = 2
RZ_DEVERR_TIMEOUT = 4
RZ_DEVERR_RANGE = 8

RZ_PROF_NAMES = ("logprob_gemm", "keep_gemm", "merge", "dz", "dH_gemm", "dW_gemm",
                 "logits_rows", "small")  # index = RZ_PROF_* class

RZ_OP_TOKEN_LOGPROB = 0
RZ_OP_LOSS_FWD_BWD = 1
RZ_OP_LOGITS_LOSS = 2
RZ_OP_IS_LOSS = 3
RZ_OP_SAMPLE = 4
RZ_OP_SC_LOSS_FWD_BWD = 5
RZ_OP_LOSS_FWD_BWD_REF = 6

_lib = None

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "rz_workspace_size": (_SZ, [ctypes.c_int, _I64, _I32, _I32, _I32]),
    "rz_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "rz_token_logprob": (ctypes.c_int, [_P, _P, _P, _I64, _I32, _I32, _P, _P, _P, _SZ, _P, _P]),
    "rz_group_advantage": (ctypes.c_int, [_P, _I32, _I32, _P, _P]),
    "rz_is_loss": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _I64, _P, _P, _P, _P, _SZ, _P, _P]),
    "rz_d3": (ctypes.c_int, [_P, _P, _I64, _P, _P]),
    "rz_loss_fwd_bwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I32, _I64, _I32, _I32,
                                       _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "rz_loss_fwd_bwd_shard": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I64,
                                             _I32, _I32, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "rz_loss_fwd_bwd_ref": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I32, _I64, _I32,
                                           _I32, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "rz_sum_partials": (ctypes.c_int, [_P, _I32, _I64, _P, _P]),
    "rz_sc_loss_fwd_bwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I32, _I64, _I32, _I32,
                                          _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "rz_logits_loss_fwd_bwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I32, _I64, _I32,
                                              _P, _P, _P, _P, _SZ, _P, _P]),
    "rz_lmhead_logits": (ctypes.c_int, [_P, _P, _I64, _I32, _I32, _P, _P, _P]),
    "rz_token_logprob_noalloc": (ctypes.c_int, [_P, _P, _P, _I64, _I32, _I32, _P, _P, _P, _P]),
    "rz_noalloc_scratch_bytes": (_SZ, []),
    "rz_is_stats": (ctypes.c_int, [_P, _P, _I64, _P, _P]),
    "rz_selftest_wait_timeout": (ctypes.c_int, [_P, _P, ctypes.c_uint32, _P]),
    "rz_sample_logprob": (ctypes.c_int, [_P, _P, _P, _I64, _I32, _I32, ctypes.c_uint64,
                                         _P, _P, _P, _P, _SZ, _P, _P]),
    "rz_peak_to_median": (ctypes.c_int, [_P, _I64, _P]),
    "rz_profile_begin": (ctypes.c_int, []),
    "rz_debug_check_failures": (ctypes.c_int, [_P, _P]),
    "rz_profile_end": (ctypes.c_int, [_P, _P, _I32]),
}


class RzError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__("%s failed: %s (status %d)" % (fn, status_string(status), status))
        self.status = status


def load(path=None):
    """Load librz.so (raises OSError/RuntimeError if it is missing)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or (LIB_PATH_CHECKS if os.environ.get("RZ_LIB_VARIANT") == "checks" else LIB_PATH)
    if not os.path.exists(p):
        raise RuntimeError("librz.so not built at %s: run invariant_logprobs_gb300.build" % p)
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def status_string(status):
    return load().rz_status_string(int(status)).decode()


def workspace_size(op, T, d, V, B):
    return int(load().rz_workspace_size(int(op), int(T), int(d), int(V), int(B)))


# ----------------------------------------------------------------- helpers
def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    """The stream handle to launch on: the given torch stream, which must
    belong to the current device (the library launches there), else the
    current device's current stream."""
    torch = _torch()
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dev = getattr(stream, "device", None)
    if dev is not None and dev.index is not None and dev.index != torch.cuda.current_device():
        raise ValueError("stream is on %s but the current device is cuda:%d"
                         % (dev, torch.cuda.current_device()))
    return ctypes.c_void_p(stream.cuda_stream)


def _check(name, status):
    if status != RZ_OK:
        raise RzError(name, status)


def _need(t, dtype, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise TypeError("%s must be a contiguous CUDA tensor of %s" % (name, dtype))


def _out(t, dtype, name, shape=None, min_numel=1):
    """Check a caller-supplied output buffer (None is allowed: the wrapper
    allocates it): dtype, contiguity and device as _need, then the exact
    shape or at least min_numel elements, so that the library never writes
    past its end."""
    if t is None:
        return
    _need(t, dtype, name)
    if shape is not None:
        _shape(t, shape, name)
    elif t.numel() < min_numel:
        raise ValueError("%s needs at least %d elements, got %d" % (name, min_numel, t.numel()))


def _ws_bytes(ws):
    """Size in bytes of a caller workspace (a contiguous CUDA uint8 tensor)."""
    _need(ws, _torch().uint8, "ws")
    return ws.numel()


def _shape(t, shape, name):
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def _same_device(*ts):
    """All tensors on one CUDA device, and that the current device: the
    library launches on the current device's context."""
    devs = {t.device for t in ts if t is not None}
    if len(devs) > 1:
        raise ValueError("all tensors must be on one CUDA device, got %s" % sorted(map(str, devs)))
    if devs:
        dev = next(iter(devs))
        cur = _torch().cuda.current_device()
        if dev.type == "cuda" and dev.index is not None and dev.index != cur:
            raise ValueError("tensors are on %s but the current device is cuda:%d; call under "
                             "torch.cuda.device(%s)" % (dev, cur, dev))


def alloc_workspace(op, T, d, V, B, device):
    torch = _torch()
    n = workspace_size(op, T, d, V, B)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def new_err_flag(device):
    torch = _torch()
    return torch.zeros(1, dtype=torch.int32, device=device)


# ----------------------------------------------------------------- entry points
def rz_token_logprob(H, W, tokens, logprob_out=None, lse_out=None, ws=None, err_flag=None,
                     stream=None):
    """Rollout-side per-token logprob (see include/rz.h).  Returns
    (logprob [T] fp32, lse [T] fp32): lse is each row's log-sum-exp, the
    reference rz_loss_fwd_bwd_ref takes (allocated here unless given)."""
    torch = _torch()
    lib = load()
    _need(H, torch.bfloat16, "H")
    _need(W, torch.bfloat16, "W")
    _need(tokens, torch.int32, "tokens")
    T, d = H.shape
    V = W.shape[0]
    _shape(W, (V, d), "W")
    _shape(tokens, (T,), "tokens")
    if logprob_out is None:
        logprob_out = torch.empty(T, dtype=torch.float32, device=H.device)
    _need(logprob_out, torch.float32, "logprob_out")
    _shape(logprob_out, (T,), "logprob_out")
    _out(lse_out, torch.float32, "lse_out", (T,))
    _out(err_flag, torch.int32, "err_flag")
    _same_device(H, W, tokens, logprob_out, lse_out, ws, err_flag)
    if ws is None:
        ws = alloc_workspace(RZ_OP_TOKEN_LOGPROB, T, d, V, 0, H.device)
    ws_bytes, strm = _ws_bytes(ws), _stream(stream)  # checked before allocating lse
    if lse_out is None:
        lse_out = torch.empty(T, dtype=torch.float32, device=H.device)
    st = lib.rz_token_logprob(_ptr(H), _ptr(W), _ptr(tokens), T, d, V, _ptr(logprob_out),
                              _ptr(lse_out), _ptr(ws), ws_bytes, _ptr(err_flag), strm)
    _check("rz_token_logprob", st)
    return logprob_out, lse_out


def rz_group_advantage(rewards, G, adv_out=None, stream=None):
    torch = _torch()
    lib = load()
    _need(rewards, torch.float32, "rewards")
    B = rewards.shape[0]
    if adv_out is None:
        adv_out = torch.empty_like(rewards)
    _need(adv_out, torch.float32, "adv_out")
    _shape(adv_out, (B,), "adv_out")
    _same_device(rewards, adv_out)
    _check("rz_group_advantage",
           lib.rz_group_advantage(_ptr(rewards), B, int(G), _ptr(adv_out), _stream(stream)))
    return adv_out


def rz_is_loss(logpi, logmu, cu_seqlens, adv, loss_out=None, d3_out=None, coef_out=None,
               ws=None, err_flag=None, stream=None, action_mask=None):
    torch = _torch()
    lib = load()
    _need(cu_seqlens, torch.int64, "cu_seqlens")
    _need(logpi, torch.float32, "logpi")
    _need(logmu, torch.float32, "logmu")
    _need(adv, torch.float32, "adv")
    B = cu_seqlens.shape[0] - 1
    T = logpi.shape[0]
    _shape(logmu, (T,), "logmu")
    _shape(adv, (B,), "adv")
    _out(coef_out, torch.float32, "coef_out", (T,))
    _out(loss_out, torch.float32, "loss_out")
    _out(d3_out, torch.float32, "d3_out")
    _out(err_flag, torch.int32, "err_flag")
    _shape(action_mask, (T,), "action_mask")
    _same_device(logpi, logmu, cu_seqlens, adv, coef_out, loss_out, d3_out, action_mask, ws,
                 err_flag)
    dev = cu_seqlens.device
    if loss_out is None:
        loss_out = torch.empty(1, dtype=torch.float32, device=dev)
    if d3_out is None:
        d3_out = torch.empty(1, dtype=torch.float32, device=dev)
    if ws is None:
        ws = alloc_workspace(RZ_OP_IS_LOSS, T, 0, 0, B, dev)
    if action_mask is not None:
        _need(action_mask, torch.uint8, "action_mask")
    st = lib.rz_is_loss(_ptr(logpi), _ptr(logmu), _ptr(cu_seqlens), _ptr(adv),
                        _ptr(action_mask), B, T,
                        _ptr(loss_out), _ptr(d3_out), _ptr(coef_out), _ptr(ws), _ws_bytes(ws),
                        _ptr(err_flag), _stream(stream))
    _check("rz_is_loss", st)
    return loss_out, d3_out, coef_out


def rz_d3(logpi, logmu, d3_out=None, stream=None):
    torch = _torch()
    lib = load()
    _need(logpi, torch.float32, "logpi")
    _need(logmu, torch.float32, "logmu")
    _shape(logmu, tuple(logpi.shape), "logmu")
    _out(d3_out, torch.float32, "d3_out")
    _same_device(logpi, logmu, d3_out)
    if d3_out is None:
        d3_out = torch.empty(1, dtype=torch.float32, device=logpi.device)
    _check("rz_d3", lib.rz_d3(_ptr(logpi), _ptr(logmu), logpi.shape[0], _ptr(d3_out),
                              _stream(stream)))
    return d3_out


def rz_loss_fwd_bwd(H, W, tokens, logmu, cu_seqlens, adv, logprob_out=None, dH=None, dW=None,
                    loss_out=None, d3_out=None, ws=None, err_flag=None, stream=None,
                    want_logprob=True, action_mask=None):
    """Learner-side fused logprob + loss forward/backward (see include/rz.h).
    Returns dict(loss, d3, logprob, dH, dW) of device tensors."""
    return _learner(None, None, H, W, tokens, logmu, cu_seqlens, adv, logprob_out, dH, dW,
                    loss_out, d3_out, ws, err_flag, stream, want_logprob, action_mask)


def rz_loss_fwd_bwd_ref(H, W, tokens, logmu, ref_lse, cu_seqlens, adv, logprob_out=None,
                        dH=None, dW=None, loss_out=None, d3_out=None, ws=None, err_flag=None,
                        stream=None, want_logprob=True, action_mask=None):
    """rz_loss_fwd_bwd with the rollout's log-sum-exp of every row (ref_lse
    [T] fp32, e.g. the lse rz_token_logprob returned with logmu) as the
    reference of the kept softmax terms; no dz pass (see include/rz.h)."""
    load()
    if ref_lse is None:
        raise TypeError("rz_loss_fwd_bwd_ref needs ref_lse (use rz_loss_fwd_bwd without one)")
    return _learner(None, ref_lse, H, W, tokens, logmu, cu_seqlens, adv, logprob_out, dH, dW,
                    loss_out, d3_out, ws, err_flag, stream, want_logprob, action_mask)


def rz_loss_fwd_bwd_shard(H, W, tokens, logmu, cu_seqlens, adv, B_total, logprob_out=None,
                          dH=None, dW=None, loss_out=None, d3_out=None, ws=None, err_flag=None,
                          stream=None, want_logprob=True, action_mask=None, ref_lse=None):
    """One shard (contiguous whole responses) of a data-parallel learner step,
    normalised by the batch's B_total responses (see include/rz.h); ref_lse
    as in rz_loss_fwd_bwd_ref.  Returns dict(loss, d3, logprob, dH, dW): the
    shard's loss share, its D3, its dH rows and its dW partial."""
    load()
    return _learner(int(B_total), ref_lse, H, W, tokens, logmu, cu_seqlens, adv, logprob_out,
                    dH, dW, loss_out, d3_out, ws, err_flag, stream, want_logprob, action_mask)


def rz_sum_partials(parts, out=None, stream=None):
    """out[i] = parts[0][i] + parts[1][i] + ... in row order (fp32): the
    fixed-order sum of the data-parallel exchange.  parts: [n, ...] fp32."""
    torch = _torch()
    lib = load()
    _need(parts, torch.float32, "parts")
    if parts.dim() < 1 or parts.shape[0] < 1:
        raise ValueError("parts must have a leading rank dimension of at least 1")
    shape = tuple(parts.shape[1:])
    count = 1
    for x in shape:
        count *= int(x)
    _out(out, torch.float32, "out", shape)
    _same_device(parts, out)
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=parts.device)
    st = lib.rz_sum_partials(_ptr(parts), int(parts.shape[0]), count, _ptr(out), _stream(stream))
    _check("rz_sum_partials", st)
    return out


def _learner(B_total, ref_lse, H, W, tokens, logmu, cu_seqlens, adv, logprob_out, dH, dW,
             loss_out, d3_out, ws, err_flag, stream, want_logprob, action_mask):
    torch = _torch()
    lib = load()
    _need(H, torch.bfloat16, "H")
    _need(W, torch.bfloat16, "W")
    _need(tokens, torch.int32, "tokens")
    _need(logmu, torch.float32, "logmu")
    _need(cu_seqlens, torch.int64, "cu_seqlens")
    _need(adv, torch.float32, "adv")
    T, d = H.shape
    V = W.shape[0]
    B = cu_seqlens.shape[0] - 1
    _shape(W, (V, d), "W")
    _shape(tokens, (T,), "tokens")
    _shape(logmu, (T,), "logmu")
    _shape(adv, (B,), "adv")
    _shape(action_mask, (T,), "action_mask")
    if ref_lse is not None:
        _need(ref_lse, torch.float32, "ref_lse")
        _shape(ref_lse, (T,), "ref_lse")
    _out(logprob_out, torch.float32, "logprob_out", (T,))
    _out(dH, torch.bfloat16, "dH", (T, d))
    _out(dW, torch.float32, "dW", (V, d))
    _out(loss_out, torch.float32, "loss_out")
    _out(d3_out, torch.float32, "d3_out")
    _out(err_flag, torch.int32, "err_flag")
    _same_device(H, W, tokens, logmu, ref_lse, cu_seqlens, adv, action_mask, logprob_out, dH,
                 dW, loss_out, d3_out, ws, err_flag)
    dev = H.device
    if want_logprob and logprob_out is None:
        logprob_out = torch.empty(T, dtype=torch.float32, device=dev)
    if dH is None:
        dH = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    if dW is None:
        dW = torch.empty((V, d), dtype=torch.float32, device=dev)
    if loss_out is None:
        loss_out = torch.empty(1, dtype=torch.float32, device=dev)
    if d3_out is None:
        d3_out = torch.empty(1, dtype=torch.float32, device=dev)
    if ws is None:
        ws = alloc_workspace(RZ_OP_LOSS_FWD_BWD if ref_lse is None else RZ_OP_LOSS_FWD_BWD_REF,
                             T, d, V, B, dev)
    if action_mask is not None:
        _need(action_mask, torch.uint8, "action_mask")
    if B_total is None and ref_lse is None:
        name = "rz_loss_fwd_bwd"
        st = lib.rz_loss_fwd_bwd(_ptr(H), _ptr(W), _ptr(tokens), _ptr(logmu), _ptr(cu_seqlens),
                                 _ptr(adv), _ptr(action_mask), B, T, d, V, _ptr(loss_out),
                                 _ptr(d3_out), _ptr(logprob_out), _ptr(dH), _ptr(dW), _ptr(ws),
                                 _ws_bytes(ws), _ptr(err_flag), _stream(stream))
    elif B_total is None:
        name = "rz_loss_fwd_bwd_ref"
        st = lib.rz_loss_fwd_bwd_ref(_ptr(H), _ptr(W), _ptr(tokens), _ptr(logmu), _ptr(ref_lse),
                                     _ptr(cu_seqlens), _ptr(adv), _ptr(action_mask), B, T, d, V,
                                     _ptr(loss_out), _ptr(d3_out), _ptr(logprob_out), _ptr(dH),
                                     _ptr(dW), _ptr(ws), _ws_bytes(ws), _ptr(err_flag),
                                     _stream(stream))
    else:
        name = "rz_loss_fwd_bwd_shard"
        st = lib.rz_loss_fwd_bwd_shard(_ptr(H), _ptr(W), _ptr(tokens), _ptr(logmu),
                                       _ptr(ref_lse), _ptr(cu_seqlens), _ptr(adv),
                                       _ptr(action_mask), B,
                                       B_total, T, d, V, _ptr(loss_out), _ptr(d3_out),
                                       _ptr(logprob_out), _ptr(dH), _ptr(dW), _ptr(ws),
                                       _ws_bytes(ws), _ptr(err_flag), _stream(stream))
    _check(name, st)
    return {"loss": loss_out, "d3": d3_out, "logprob": logprob_out, "dH": dH, "dW": dW}


def rz_sc_loss_fwd_bwd(H, W, tokens, cu_seqlens, adv, logprob_out=None, dH=None, dW=None,
                       loss_out=None, ws=None, err_flag=None, stream=None, want_logprob=True,
                       action_mask=None):
    """Score Centering comparison estimator: the learner step without
    importance weights, advantages centred over the batch (see include/rz.h).
    Returns dict(loss, logprob, dH, dW) of device tensors."""
    torch = _torch()
    lib = load()
    _need(H, torch.bfloat16, "H")
    _need(W, torch.bfloat16, "W")
    _need(tokens, torch.int32, "tokens")
    _need(cu_seqlens, torch.int64, "cu_seqlens")
    _need(adv, torch.float32, "adv")
    T, d = H.shape
    V = W.shape[0]
    B = cu_seqlens.shape[0] - 1
    _shape(W, (V, d), "W")
    _shape(tokens, (T,), "tokens")
    _shape(adv, (B,), "adv")
    _shape(action_mask, (T,), "action_mask")
    _out(logprob_out, torch.float32, "logprob_out", (T,))
    _out(dH, torch.bfloat16, "dH", (T, d))
    _out(dW, torch.float32, "dW", (V, d))
    _out(loss_out, torch.float32, "loss_out")
    _out(err_flag, torch.int32, "err_flag")
    _same_device(H, W, tokens, cu_seqlens, adv, action_mask, logprob_out, dH, dW, loss_out, ws,
                 err_flag)
    dev = H.device
    if want_logprob and logprob_out is None:
        logprob_out = torch.empty(T, dtype=torch.float32, device=dev)
    if dH is None:
        dH = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    if dW is None:
        dW = torch.empty((V, d), dtype=torch.float32, device=dev)
    if loss_out is None:
        loss_out = torch.empty(1, dtype=torch.float32, device=dev)
    if ws is None:
        ws = alloc_workspace(RZ_OP_SC_LOSS_FWD_BWD, T, d, V, B, dev)
    if action_mask is not None:
        _need(action_mask, torch.uint8, "action_mask")
    st = lib.rz_sc_loss_fwd_bwd(_ptr(H), _ptr(W), _ptr(tokens), _ptr(cu_seqlens), _ptr(adv),
                                _ptr(action_mask), B, T, d, V, _ptr(loss_out),
                                _ptr(logprob_out), _ptr(dH), _ptr(dW), _ptr(ws), _ws_bytes(ws),
                                _ptr(err_flag), _stream(stream))
    _check("rz_sc_loss_fwd_bwd", st)
    return {"loss": loss_out, "logprob": logprob_out, "dH": dH, "dW": dW}


def rz_logits_loss_fwd_bwd(logits_inout, tokens, logmu, cu_seqlens, adv, logprob_out=None,
                           loss_out=None, d3_out=None, ws=None, err_flag=None, stream=None,
                           action_mask=None):
    """Given-logits variant; overwrites logits_inout with dz (see include/rz.h)."""
    torch = _torch()
    lib = load()
    _need(logits_inout, torch.bfloat16, "logits_inout")
    _need(tokens, torch.int32, "tokens")
    _need(logmu, torch.float32, "logmu")
    _need(cu_seqlens, torch.int64, "cu_seqlens")
    _need(adv, torch.float32, "adv")
    T, V = logits_inout.shape
    B = cu_seqlens.shape[0] - 1
    _shape(tokens, (T,), "tokens")
    _shape(logmu, (T,), "logmu")
    _shape(adv, (B,), "adv")
    _shape(action_mask, (T,), "action_mask")
    _out(logprob_out, torch.float32, "logprob_out", (T,))
    _out(loss_out, torch.float32, "loss_out")
    _out(d3_out, torch.float32, "d3_out")
    _out(err_flag, torch.int32, "err_flag")
    _same_device(logits_inout, tokens, logmu, cu_seqlens, adv, action_mask, logprob_out,
                 loss_out, d3_out, ws, err_flag)
    dev = logits_inout.device
    if logprob_out is None:
        logprob_out = torch.empty(T, dtype=torch.float32, device=dev)
    if loss_out is None:
        loss_out = torch.empty(1, dtype=torch.float32, device=dev)
    if d3_out is None:
        d3_out = torch.empty(1, dtype=torch.float32, device=dev)
    if ws is None:
        ws = alloc_workspace(RZ_OP_LOGITS_LOSS, T, 0, V, B, dev)
    if action_mask is not None:
        _need(action_mask, torch.uint8, "action_mask")
    st = lib.rz_logits_loss_fwd_bwd(_ptr(logits_inout), _ptr(tokens), _ptr(logmu),
                                    _ptr(cu_seqlens), _ptr(adv), _ptr(action_mask), B, T, V,
                                    _ptr(loss_out),
                                    _ptr(d3_out), _ptr(logprob_out), _ptr(ws), _ws_bytes(ws),
                                    _ptr(err_flag), _stream(stream))
    _check("rz_logits_loss_fwd_bwd", st)
    return {"loss": loss_out, "d3": d3_out, "logprob": logprob_out}


def rz_lmhead_logits(H, W, logits_out=None, err_flag=None, stream=None):
    torch = _torch()
    lib = load()
    _need(H, torch.bfloat16, "H")
    _need(W, torch.bfloat16, "W")
    T, d = H.shape
    V = W.shape[0]
    _shape(W, (V, d), "W")
    if logits_out is None:
        logits_out = torch.empty((T, V), dtype=torch.float32, device=H.device)
    _need(logits_out, torch.float32, "logits_out")
    _shape(logits_out, (T, V), "logits_out")
    _out(err_flag, torch.int32, "err_flag")
    _same_device(H, W, logits_out, err_flag)
    st = lib.rz_lmhead_logits(_ptr(H), _ptr(W), T, d, V, _ptr(logits_out), _ptr(err_flag),
                              _stream(stream))
    _check("rz_lmhead_logits", st)
    return logits_out


def rz_token_logprob_noalloc(H, W, tokens, logprob_out, lse_out=None, err_flag=None,
                             stream=None):
    """rz_token_logprob for callers that cannot allocate device memory: the
    library's built-in scratch replaces the workspace, and nothing is
    allocated here either -- the caller passes the output buffers.  See
    include/rz.h for the size limit, first-call set-up and the rule that
    overlapping calls race."""
    torch = _torch()
    lib = load()
    _need(H, torch.bfloat16, "H")
    _need(W, torch.bfloat16, "W")
    _need(tokens, torch.int32, "tokens")
    _need(logprob_out, torch.float32, "logprob_out")
    T, d = H.shape
    V = W.shape[0]
    _shape(W, (V, d), "W")
    _shape(tokens, (T,), "tokens")
    _shape(logprob_out, (T,), "logprob_out")
    _out(lse_out, torch.float32, "lse_out", (T,))
    _out(err_flag, torch.int32, "err_flag")
    _same_device(H, W, tokens, logprob_out, lse_out, err_flag)
    st = lib.rz_token_logprob_noalloc(_ptr(H), _ptr(W), _ptr(tokens), T, d, V,
                                      _ptr(logprob_out), _ptr(lse_out), _ptr(err_flag),
                                      _stream(stream))
    _check("rz_token_logprob_noalloc", st)
    return logprob_out, lse_out


def noalloc_scratch_bytes():
    return int(load().rz_noalloc_scratch_bytes())


IS_STATS_FIELDS = ("d3", "k1", "k2", "w_mean", "w_max", "w_min", "absd_max")


def rz_is_stats(logpi, logmu, stats_out=None, stream=None):
    """Per-update IS diagnostics (see include/rz.h): a [7] fp32 device tensor
    in the order of IS_STATS_FIELDS."""
    torch = _torch()
    lib = load()
    _need(logpi, torch.float32, "logpi")
    _need(logmu, torch.float32, "logmu")
    _shape(logmu, tuple(logpi.shape), "logmu")
    _out(stats_out, torch.float32, "stats_out", min_numel=len(IS_STATS_FIELDS))
    _same_device(logpi, logmu, stats_out)
    if stats_out is None:
        stats_out = torch.empty(7, dtype=torch.float32, device=logpi.device)
    _check("rz_is_stats", lib.rz_is_stats(_ptr(logpi), _ptr(logmu), logpi.shape[0],
                                          _ptr(stats_out), _stream(stream)))
    return stats_out


def rz_peak_to_median(series):
    """max/median of a host sequence of per-update values (host function)."""
    buf = (ctypes.c_float * len(series))(*[float(x) for x in series])
    out = ctypes.c_double(0.0)
    _check("rz_peak_to_median", load().rz_peak_to_median(
        ctypes.cast(buf, ctypes.c_void_p), len(series), ctypes.byref(out)))
    return out.value


def rz_sample_logprob(H, W, seed, row_ids=None, tokens_out=None, logprob_out=None,
                      lse_out=None, ws=None, err_flag=None, stream=None):
    """Rollout with fused sampling (see include/rz.h): returns (tokens [T]
    int32, log mu [T] fp32)."""
    torch = _torch()
    lib = load()
    _need(H, torch.bfloat16, "H")
    _need(W, torch.bfloat16, "W")
    if row_ids is not None:
        _need(row_ids, torch.int64, "row_ids")
    T, d = H.shape
    V = W.shape[0]
    _shape(W, (V, d), "W")
    _shape(row_ids, (T,), "row_ids")
    _out(tokens_out, torch.int32, "tokens_out", (T,))
    _out(logprob_out, torch.float32, "logprob_out", (T,))
    _out(lse_out, torch.float32, "lse_out", (T,))
    _out(err_flag, torch.int32, "err_flag")
    _same_device(H, W, row_ids, tokens_out, logprob_out, lse_out, ws, err_flag)
    if tokens_out is None:
        tokens_out = torch.empty(T, dtype=torch.int32, device=H.device)
    if logprob_out is None:
        logprob_out = torch.empty(T, dtype=torch.float32, device=H.device)
    if ws is None:
        ws = alloc_workspace(RZ_OP_SAMPLE, T, d, V, 0, H.device)
    st = lib.rz_sample_logprob(_ptr(H), _ptr(W), _ptr(row_ids), T, d, V,
                               ctypes.c_uint64(int(seed) & 0xFFFFFFFFFFFFFFFF),
                               _ptr(tokens_out), _ptr(logprob_out), _ptr(lse_out), _ptr(ws),
                               _ws_bytes(ws), _ptr(err_flag), _stream(stream))
    _check("rz_sample_logprob", st)
    return tokens_out, logprob_out


def rz_selftest_wait_timeout(err_flag, done_out=None, limit_us=50000, stream=None):
    """Run the bounded-wait self-test (see include/rz.h)."""
    torch = _torch()
    _need(err_flag, torch.int32, "err_flag")
    _out(done_out, torch.int32, "done_out")
    _same_device(err_flag, done_out)
    _check("rz_selftest_wait_timeout", load().rz_selftest_wait_timeout(
        _ptr(err_flag), _ptr(done_out), int(limit_us), _stream(stream)))


def rz_profile_begin():
    """Start launch-class timing (see rz_profile_begin in include/rz.h)."""
    _check("rz_profile_begin", load().rz_profile_begin())


def rz_profile_end():
    """Stop launch-class timing; blocks until the recorded events complete.
    Returns {class name: (milliseconds, kernel launches)} for every class."""
    n = len(RZ_PROF_NAMES)
    ms = (ctypes.c_float * n)()
    launches = (ctypes.c_int32 * n)()
    _check("rz_profile_end", load().rz_profile_end(ms, launches, n))
    return {name: (float(ms[i]), int(launches[i])) for i, name in enumerate(RZ_PROF_NAMES)}


def rz_debug_check_failures():
    """(failed device bounds checks since the last read, site of the first)
    from the debug build, cleared on read; None with the normal build, which
    has no checks."""
    n = ctypes.c_uint32(0)
    site = ctypes.c_int32(0)
    st = load().rz_debug_check_failures(ctypes.byref(n), ctypes.byref(site))
    if st == RZ_ERR_UNSUPPORTED:
        return None
    _check("rz_debug_check_failures", st)
    return int(n.value), int(site.value)
