"""Oracle of the fused rollout sampler: Gumbel-max sampling of a_t from
softmax(z_t) with counter-based noise, and the recorded log mu(a_t).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages say the rollout records the logprob of every token it samples
([vLLM-zh] s.4 item 2) but not how it samples; the reading taken here is
exact sampling at temperature 1 by the Gumbel-max rule
    a_t = argmax_v ( z_tv + G_tv ),   G = -log(-log U),
whose argmax is distributed as softmax(z_t).  U comes from the counter-based
generator Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random
Numbers: As Easy as 1, 2, 3", SC 2011), written here from that definition:
    key (k0, k1) = seed (low, high 32 bits)
    counter (c0, c1, c2, c3) = (v // 4, row_id low, row_id high, 0)
    U_tv = ((x >> 9) + 1/2) * 2^-23,  x = output word (v mod 4).
Ties of the key go to the smallest vocabulary index.
"""

import numpy as np

_M0 = 0xD2511F53
_M1 = 0xCD9E8D57
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
_MASK = 0xFFFFFFFF


def philox4x32_10(ctr, key):
    """Philox4x32 with 10 rounds, vectorised over leading axes.

    ctr: uint array [..., 4]; key: uint array [..., 2] (broadcastable).
    Each round: (hi0, lo0) = M0 * c0, (hi1, lo1) = M1 * c2 (64-bit products),
    c <- (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0); then the key is bumped by
    (W0, W1).  Returns uint64 array [..., 4] holding 32-bit values.
    """
    c = np.array(ctr, dtype=np.uint64) & _MASK
    k = np.array(key, dtype=np.uint64) & _MASK
    c0, c1, c2, c3 = c[..., 0], c[..., 1], c[..., 2], c[..., 3]
    k0, k1 = k[..., 0] + 0 * c0, k[..., 1] + 0 * c0
    for _ in range(10):
        p0 = c0 * np.uint64(_M0)
        p1 = c2 * np.uint64(_M1)
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(_MASK)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(_MASK)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        k0 = (k0 + np.uint64(_W0)) & np.uint64(_MASK)
        k1 = (k1 + np.uint64(_W1)) & np.uint64(_MASK)
    return np.stack([c0, c1, c2, c3], axis=-1)


def uniforms(row_id, V, seed):
    """U_tv for one row, v = 0..V-1, as float64 (exactly the 23-bit values)."""
    ngroups = (V + 3) // 4
    g = np.arange(ngroups, dtype=np.uint64)
    rid = np.uint64(int(row_id) & 0xFFFFFFFFFFFFFFFF)
    ctr = np.stack([g, np.full_like(g, rid & np.uint64(_MASK)),
                    np.full_like(g, rid >> np.uint64(32)), np.zeros_like(g)], axis=-1)
    key = np.array([seed & _MASK, (seed >> 32) & _MASK], dtype=np.uint64)
    x = philox4x32_10(ctr, key).reshape(-1)[:V]
    return ((x >> np.uint64(9)).astype(np.float64) + 0.5) * 2.0 ** -23


def gumbel_keys(z_row, row_id, seed):
    """z_v + G_v for one row (fp64)."""
    u = uniforms(row_id, z_row.shape[0], seed)
    return np.asarray(z_row, np.float64) - np.log(-np.log(u))


def sample_rows(H, W, row_ids, seed):
    """Sampled token and its recorded log mu for every row of H (fp64 logits
    from the exact bf16 values).  Returns (tokens [T] int64, logmu [T],
    keys_margin [T]) where keys_margin is the gap between the best and the
    second-best key (small margins mark rows whose argmax a different
    rounding could flip)."""
    H = np.asarray(H, np.float64)
    W = np.asarray(W, np.float64)
    T = H.shape[0]
    tok = np.empty(T, dtype=np.int64)
    lmu = np.empty(T, dtype=np.float64)
    margin = np.empty(T, dtype=np.float64)
    for t in range(T):
        z = H[t] @ W.T
        k = gumbel_keys(z, row_ids[t], seed)
        a = int(np.argmax(k))
        top2 = np.partition(k, -2)[-2:] if k.shape[0] > 1 else np.array([-np.inf, k[0]])
        margin[t] = top2[1] - top2[0]
        m = z.max()
        lse = m + np.log(np.exp(z - m).sum())
        tok[t] = a
        lmu[t] = z[a] - lse
    return tok, lmu, margin


def key_of(H_row, W, row_id, seed):
    """Every token's Gumbel key z_v + G_v for one row (fp64) and the row's
    logits z, for checking that a token drawn elsewhere holds the best key
    (or one within a near-tie of it)."""
    z = np.asarray(W, np.float64) @ np.asarray(H_row, np.float64)
    return gumbel_keys(z, row_id, seed), z
