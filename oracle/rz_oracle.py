"""Plain float64 definitions of what the REINFORCE Zero hot path computes.

TEST INFRASTRUCTURE ONLY (see the package docstring): the CUDA library never
imports this module and this module never imports the CUDA library.

Sources (web pages on REINFORCE Zero; cited by title and section):

* [RZ-page]  "REINFORCE Zero -- Kernel Alignment Unlocks Stable Asynchronous
  RL with Importance Sampling", project page (hujian.website):
  - section 02 "The mechanism", block "A minimal REINFORCE objective": the
    loss  L = -(1/B) sum_i (1/T_i) sum_t A_i * pi(a_it|h_it) / mu_i(a_it|h_it),
    T_i = valid action tokens of response i, mu the recorded behaviour
    probability, gradient through the numerator pi only;
  - section "The full IS correction", items 01-04: w = p/q, E_q[w s] = 0,
    g_IS = E_q[w A s] = Cov_p(A, s); item 03 "Score centering":
    g_SC = Cov_q(A, s) (the comparison estimator without IS).
* [vLLM-zh]  "Zero Mismatch, Simple Async RL: REINFORCE Zero, DeepSeek-V4.1
  and Kimi K3.1" (Chinese rendering, todayforai.com):
  - section 3: the D3 diagnostic, the per-update mean over all tokens of
    w - 1 - log w; the log-gap decomposition;
  - section 4 "方案" items 1-3: logprob of the sampled token; unclipped
    token-level ratio pi/mu from the recorded logprob; advantage = reward
    minus the mean reward of its group; tokens averaged within a response;
    and the loss equation.
  - section 5: "diff 0" = bitwise-equal logprob for every sampled token.

Readings where the pages are silent (each is also listed in the design
notes): temperature 1 and no logit processing; groups are contiguous blocks
of G responses; advantage = r - group mean (no std division); B counts every
response of the call; a response with T_i = 0 adds 0 to the loss; D3 is the
flat mean over the T tokens of the call; mu enters only through the given
log mu array (never differentiated).

Rows are processed in blocks only to bound memory; each row's arithmetic is
the per-row definition, unchanged by the blocking.
"""

import numpy as np

_ROW_BLOCK = 256


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def lmhead_logits(H, W):
    """z_tv = sum_k H_tk W_vk (LM-head projection; the pages' pi(a|h) is the
    softmax of these logits) [vLLM-zh s.4 item 1].  Library matmul, fp64."""
    return _f64(H) @ _f64(W).T


def logsumexp_rows(z):
    """LSE_t = m_t + log sum_v exp(z_tv - m_t), m_t = max_v z_tv (the
    normaliser of the softmax policy)."""
    z = _f64(z)
    m = z.max(axis=1, keepdims=True)
    return m[:, 0] + np.log(np.exp(z - m).sum(axis=1))


def token_logprob_rows(H, W, tokens, rows):
    """log pi for a subset of rows (used to check full-size runs row by row).

    Returns (logpi[rows], lse[rows]) in fp64.  log pi(a_t|h_t) = z_{t,a_t} -
    LSE_t [vLLM-zh s.4 item 1; RZ-page s.02 objective numerator].
    """
    rows = np.asarray(rows, dtype=np.int64)
    tokens = np.asarray(tokens, dtype=np.int64)
    Wd = _f64(W)
    lp = np.empty(rows.shape[0], dtype=np.float64)
    lse = np.empty(rows.shape[0], dtype=np.float64)
    for s in range(0, rows.shape[0], _ROW_BLOCK):
        r = rows[s:s + _ROW_BLOCK]
        z = _f64(H[r]) @ Wd.T
        l = logsumexp_rows(z)
        lse[s:s + _ROW_BLOCK] = l
        lp[s:s + _ROW_BLOCK] = z[np.arange(r.shape[0]), tokens[r]] - l
    return lp, lse


def token_logprob(H, W, tokens):
    """Per-token logprob of the sampled token for every row.

    This is what the rollout records as log mu (with the rollout's weights)
    and what the learner recomputes as log pi [vLLM-zh s.4 items 1-2].
    Returns (logpi [T], lse [T]) in fp64.
    """
    T = np.asarray(tokens).shape[0]
    return token_logprob_rows(H, W, tokens, np.arange(T))


def group_advantage(rewards, G):
    """A_i = r_i - (1/G) sum_{j in group(i)} r_j, groups = contiguous blocks
    of G responses [vLLM-zh s.4 item 3: reward minus the group's mean reward;
    no value model]."""
    r = _f64(rewards)
    B = r.shape[0]
    if G <= 0 or B % G != 0:
        raise ValueError("B must be a multiple of G")
    g = r.reshape(B // G, G)
    return (g - g.mean(axis=1, keepdims=True)).reshape(B)


def d3(logpi, logmu):
    """D3 = mean over all tokens of (w - 1 - log w), w = pi/mu
    [vLLM-zh s.3, Figure 1 caption text].  Empty input gives 0."""
    lp = _f64(logpi)
    if lp.shape[0] == 0:
        return 0.0
    w = np.exp(lp - _f64(logmu))
    return float(np.mean(w - 1.0 - np.log(w)))


def is_loss(logpi, logmu, cu_seqlens, adv, mask=None):
    """The REINFORCE Zero loss and its per-token gradient coefficient.

    w_t = pi/mu = exp(log pi_t - log mu_t), never clipped [vLLM-zh s.4 item 2].
    L = -(1/B) sum_i (1/T_i) sum_{t in i} A_i w_t     [RZ-page s.02 objective]
    D3 = mean_t (w_t - 1 - log w_t)                      [vLLM-zh s.3]
    c_t = A_i w_t / (B T_i) = -dL/dlog pi_t  (the derivative of w through the
    numerator only: dw/dlog pi = w)                      [RZ-page s.02]

    mask (optional, [T], nonzero = valid action token): "T_i counts valid
    action tokens" [RZ-page s.02]; a masked-out token (e.g. a tool output
    inside an agentic response) is in no sum: T_i counts the valid tokens of
    response i, D3 averages over all valid tokens, and c_t = 0.

    Returns dict(loss, d3, w [T], c [T]) in fp64.
    """
    lp = _f64(logpi)
    lm = _f64(logmu)
    A = _f64(adv)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    B = A.shape[0]
    T = lp.shape[0]
    valid = np.ones(T, dtype=bool) if mask is None else (np.asarray(mask) != 0)
    w = np.exp(lp - lm)
    c = np.zeros(T, dtype=np.float64)
    total = 0.0
    for i in range(B):
        s, e = int(cu[i]), int(cu[i + 1])
        v = valid[s:e]
        Ti = int(v.sum())
        if Ti == 0:
            continue
        total += A[i] * w[s:e][v].sum() / Ti
        c[s:e] = np.where(v, A[i] * w[s:e] / (B * Ti), 0.0)
    loss = -total / B if B > 0 else 0.0
    return {"loss": loss, "d3": d3(lp[valid], lm[valid]), "w": w, "c": c}


def loss_fwd_bwd(H, W, tokens, logmu, cu_seqlens, adv, mask=None):
    """Learner step: log pi, loss, D3 and the gradients dH, dW.

    dL/dz_tv = c_t (softmax_v(z_t) - [v = a_t]) because
    dL/dlog pi_t = -c_t and dlog pi_t/dz_tv = [v = a_t] - p_tv; mu and A are
    constants [RZ-page s.02: differentiate through the numerator].
    z = H W^T gives dH = dz W and dW = dz^T H.  `mask` as in is_loss.
    Returns dict(loss, d3, logpi, lse, c, dH, dW) in fp64.
    """
    Hd = _f64(H)
    Wd = _f64(W)
    tokens = np.asarray(tokens, dtype=np.int64)
    T = tokens.shape[0]
    logpi, lse = token_logprob(Hd, Wd, tokens)
    r = is_loss(logpi, logmu, cu_seqlens, adv, mask)
    c = r["c"]
    dH = np.zeros_like(Hd)
    dW = np.zeros_like(Wd)
    for s in range(0, T, _ROW_BLOCK):
        e = min(T, s + _ROW_BLOCK)
        z = Hd[s:e] @ Wd.T
        p = np.exp(z - lse[s:e, None])
        p[np.arange(e - s), tokens[s:e]] -= 1.0
        dz = c[s:e, None] * p
        dH[s:e] = dz @ Wd
        dW += dz.T @ Hd[s:e]
    return {"loss": r["loss"], "d3": r["d3"], "logpi": logpi, "lse": lse,
            "c": c, "dH": dH, "dW": dW}


def sc_loss(logpi, cu_seqlens, adv, mask=None):
    """Score Centering (SC), the comparison estimator without importance
    weights [RZ-page "The full IS correction", items 02-03]: the update
    E_q[A s] taken on the sampler's tokens carries the drift E_q[A] E_q[s];
    SC centres the sampler score and keeps g_SC = Cov_q(A, s).

    Per-token form (a reading: the pages give only the expectation): each
    sampled token's score s_t = grad log pi_t is centred by the batch
    estimate of its mean, with the token weights of the IS loss,
        g_SC = (1/B) sum_i (A_i/T_i) sum_t (s_t - sbar),
        sbar = (1/B+) sum_{j: T_j > 0} (1/T_j) sum_t s_t,
    B+ = number of responses with T_j > 0.  This equals
    (1/B) sum_i ((A_i - Abar)/T_i) sum_t s_t with Abar the mean of A_i over
    those B+ responses, so adding a constant to every advantage changes
    nothing (the centred scores sum to zero).  Its surrogate loss
    (gradient -g_SC) is
        L_SC = -(1/B) sum_i ((A_i - Abar)/T_i) sum_{t in i} log pi_t,
    c_t = -dL_SC/dlog pi_t = (A_i - Abar)/(B T_i).  T_i, B and the mask as in
    is_loss; a response with T_i = 0 adds nothing.

    Returns dict(loss, abar, c [T]) in fp64.
    """
    lp = _f64(logpi)
    A = _f64(adv)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    B = A.shape[0]
    T = lp.shape[0]
    valid = np.ones(T, dtype=bool) if mask is None else (np.asarray(mask) != 0)
    counts = np.array([int(valid[cu[i]:cu[i + 1]].sum()) for i in range(B)], dtype=np.int64)
    nonempty = counts > 0
    abar = A[nonempty].mean() if nonempty.any() else 0.0
    c = np.zeros(T, dtype=np.float64)
    total = 0.0
    for i in range(B):
        if counts[i] == 0:
            continue
        s, e = int(cu[i]), int(cu[i + 1])
        v = valid[s:e]
        total += (A[i] - abar) * lp[s:e][v].sum() / counts[i]
        c[s:e] = np.where(v, (A[i] - abar) / (B * counts[i]), 0.0)
    loss = -total / B if B > 0 else 0.0
    return {"loss": loss, "abar": abar, "c": c}


def sc_loss_fwd_bwd(H, W, tokens, cu_seqlens, adv, mask=None):
    """Learner step of the Score Centering estimator (sc_loss): log pi, L_SC
    and dH, dW with dz_tv = c_t (softmax_v(z_t) - [v = a_t]), as in
    loss_fwd_bwd but with c_t from sc_loss (no log mu, no weight).
    Returns dict(loss, abar, logpi, lse, c, dH, dW) in fp64.
    """
    Hd = _f64(H)
    Wd = _f64(W)
    tokens = np.asarray(tokens, dtype=np.int64)
    T = tokens.shape[0]
    logpi, lse = token_logprob(Hd, Wd, tokens)
    r = sc_loss(logpi, cu_seqlens, adv, mask)
    c = r["c"]
    dH = np.zeros_like(Hd)
    dW = np.zeros_like(Wd)
    for s in range(0, T, _ROW_BLOCK):
        e = min(T, s + _ROW_BLOCK)
        z = Hd[s:e] @ Wd.T
        p = np.exp(z - lse[s:e, None])
        p[np.arange(e - s), tokens[s:e]] -= 1.0
        dz = c[s:e, None] * p
        dH[s:e] = dz @ Wd
        dW += dz.T @ Hd[s:e]
    return {"loss": r["loss"], "abar": r["abar"], "logpi": logpi, "lse": lse, "c": c,
            "dH": dH, "dW": dW}


def logits_loss_fwd_bwd(logits, tokens, logmu, cu_seqlens, adv, rows=None, mask=None):
    """The same loss and dlogits, starting from given logits z [T, V].

    Returns dict(loss, d3, logpi, lse, c) and, for the requested rows (all
    when rows is None), dz [len(rows), V] = c_t (softmax(z_t) - onehot(a_t)).
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    T = tokens.shape[0]
    logpi = np.empty(T, dtype=np.float64)
    lse = np.empty(T, dtype=np.float64)
    for s in range(0, T, _ROW_BLOCK):
        e = min(T, s + _ROW_BLOCK)
        z = _f64(logits[s:e])
        l = logsumexp_rows(z)
        lse[s:e] = l
        logpi[s:e] = z[np.arange(e - s), tokens[s:e]] - l
    r = is_loss(logpi, logmu, cu_seqlens, adv, mask)
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    dz = np.empty((rows.shape[0], np.asarray(logits[:1]).shape[1]), np.float64)
    for s in range(0, rows.shape[0], _ROW_BLOCK):
        rr = rows[s:s + _ROW_BLOCK]
        z = _f64(logits[rr])
        p = np.exp(z - lse[rr, None])
        p[np.arange(rr.shape[0]), tokens[rr]] -= 1.0
        dz[s:s + _ROW_BLOCK] = r["c"][rr, None] * p
    return {"loss": r["loss"], "d3": r["d3"], "logpi": logpi, "lse": lse,
            "c": r["c"], "dz": dz, "rows": rows}


def is_stats(logpi, logmu):
    """Per-update importance-sampling diagnostics over the T sampled tokens.

    d_t = log pi_t - log mu_t, w_t = exp(d_t).  Returned in fp64:
      d3   mean(w - 1 - log w): the D3 diagnostic [vLLM-zh s.3]; for tokens
           drawn from mu it is also the "k3" estimator of KL(mu || pi);
      k1   mean(-d) = mean(log mu - log pi): the plain estimator of KL(mu||pi);
      k2   mean(d^2 / 2);
      w_mean, w_max, w_min, absd_max.
    The pages plot a "sampled rollout-to-learner KL" without defining it
    ([RZ-page] Figure 1, [vLLM-zh] s.4 Figure 3); k1 and k3 are the two
    readings offered.  Empty input gives zeros.
    """
    lp = _f64(logpi)
    lm = _f64(logmu)
    if lp.shape[0] == 0:
        return {"d3": 0.0, "k1": 0.0, "k2": 0.0, "w_mean": 0.0, "w_max": 0.0,
                "w_min": 0.0, "absd_max": 0.0}
    d = lp - lm
    w = np.exp(d)
    return {"d3": float(np.mean(w - 1.0 - np.log(w))), "k1": float(np.mean(-d)),
            "k2": float(np.mean(d * d / 2.0)), "w_mean": float(np.mean(w)),
            "w_max": float(np.max(w)), "w_min": float(np.min(w)),
            "absd_max": float(np.max(np.abs(d)))}


def peak_to_median(series):
    """max(series) / median(series) of a per-update diagnostic series (the
    statistic the pages report for D3 across updates: 1.50x aligned vs
    442.54x standard kernels [vLLM-zh s.3, Figure 1]).  The median of an even
    count is the mean of the two middle values."""
    x = _f64(series)
    return float(np.max(x) / np.median(x))
