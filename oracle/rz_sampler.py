"""Oracle of the fused rollout sampler: exact sampling of a_t from
softmax(z_t), streamed over the vocabulary with counter-based uniforms, and
the recorded log mu(a_t).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages say the rollout records the logprob of every token it samples
([vLLM-zh] s.4 item 2) but not how it samples.  The reading taken here is
exact sampling at temperature 1 by a two-level weighted reservoir, which
draws a token with probability exactly its softmax weight q_v / sum q,
q_v = exp(z_v - max z):

* chunks c = 0, 1, ... are the columns [32c, 32c + 32) of the row;
* segments g = 0 .. S-1 group whole 256-column tiles: with n_t = ceil(V/256)
  tiles, n = min(n_t, 64), tps = ceil(n_t / n) tiles per segment and
  S = ceil(n_t / tps) segments, segment g holds columns
  [256 tps g, 256 tps (g + 1)) (clipped at V);
* inside a segment the chunks are taken in order; with R the sum of q over
  the segment's chunks so far (this one included) and W the chunk's sum,
  the segment's candidate becomes a draw from this chunk when U1 R < W;
  the draw visits the chunk's columns by class (column mod 4 = 0, 1, 2, 3)
  and, inside a class, by column, and takes the first at which the running
  sum of q passes U2 W;
* the segments are taken in order the same way: with R' the sum of the
  segments' totals so far, the sample becomes segment g's candidate when
  U3 R' < its total.

For a stream of blocks with weights W_1 .. W_n, keeping block k with
probability W_k / R_k and no later one gives W_k / R_n, so every token is
drawn with probability q_v / sum q, in both levels.

U1, U2 are words 0 and 1 of Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3", SC 2011; written here from
that definition) at counter (c, row id low 32 bits, row id high 32 bits, 0)
under key (seed low, seed high); U3 is word 0 at counter (g, row id low,
row id high, 1).  A word x maps to U = ((x >> 9) + 1/2) 2^-23 in (0, 1).
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


def uniform_of(x):
    """((x >> 9) + 1/2) 2^-23 for 32-bit words x (exact in float64)."""
    return ((np.asarray(x, np.uint64) >> np.uint64(9)).astype(np.float64) + 0.5) * 2.0 ** -23


def row_words(counter0, row_ids, counter3, seed):
    """Philox words at counter (counter0, row id lo, row id hi, counter3) for
    every row id; returns uint64 [T, 4]."""
    rid = np.asarray(row_ids).astype(np.int64).astype(np.uint64)
    ctr = np.stack([np.full_like(rid, np.uint64(counter0)), rid & np.uint64(_MASK),
                    rid >> np.uint64(32), np.full_like(rid, np.uint64(counter3))], axis=-1)
    key = np.array([seed & _MASK, (seed >> 32) & _MASK], dtype=np.uint64)
    return philox4x32_10(ctr, key)


def segments(V):
    """Column ranges [a, b) of the segments (groups of 256-column tiles)."""
    nt = (V + 255) // 256
    n = min(nt, 64)
    tps = (nt + n - 1) // n
    S = (nt + tps - 1) // tps
    return [(256 * tps * g, min(256 * tps * (g + 1), V)) for g in range(S)]


def draw_order(n):
    """Positions 0 .. n-1 of a chunk in draw order: by class j mod 4, then j."""
    return np.array([j for k in range(4) for j in range(k, n, 4)], dtype=np.int64)


def sample_rows(H, W, row_ids, seed):
    """Sampled token and its recorded log mu for every row of H (fp64 logits
    from the exact bf16 values).  Returns (tokens [T] int64, logmu [T],
    margin [T]): margin is the smallest relative distance, over every
    decision the row's sample depends on, between the uniform's threshold
    and the value it is compared with (tiny margins mark rows whose sample a
    different rounding could change)."""
    H = np.asarray(H, np.float64)
    W = np.asarray(W, np.float64)
    z = H @ W.T
    T, V = z.shape
    M = z.max(axis=1, keepdims=True)
    q = np.exp(z - M)
    rows = np.arange(T)
    margin = np.full(T, np.inf)
    final = np.full(T, -1, dtype=np.int64)
    Rp = np.zeros(T)
    for g, (a, b) in enumerate(segments(V)):
        R = np.zeros(T)
        cand = np.full(T, -1, dtype=np.int64)
        for c0 in range(a, b, 32):
            c1 = min(c0 + 32, b)
            qc = q[:, c0:c1]
            Wc = qc.sum(axis=1)
            R = R + Wc
            x = row_words(c0 // 32, row_ids, 0, seed)
            u1, u2 = uniform_of(x[:, 0]), uniform_of(x[:, 1])
            rep = u1 * R < Wc
            with np.errstate(divide="ignore", invalid="ignore"):
                margin = np.minimum(margin, np.where(Wc > 0, np.abs(u1 * R - Wc) / Wc, np.inf))
            order = draw_order(c1 - c0)
            cs = np.cumsum(qc[:, order], axis=1)
            tgt = u2 * Wc
            past = cs > tgt[:, None]
            pos = np.where(past.any(axis=1), past.argmax(axis=1),
                           (qc[:, order] > 0).shape[1] - 1 -
                           np.argmax((qc[:, order] > 0)[:, ::-1], axis=1))
            # boundaries next to the drawn position, relative to W
            hi = np.abs(cs[rows, pos] - tgt)
            lo = np.where(pos > 0, np.abs(cs[rows, np.maximum(pos - 1, 0)] - tgt), np.inf)
            with np.errstate(divide="ignore", invalid="ignore"):
                dm = np.where(rep & (Wc > 0), np.minimum(hi, lo) / Wc, np.inf)
            margin = np.minimum(margin, dm)
            cand = np.where(rep, c0 + order[pos], cand)
        Qg = q[:, a:b].sum(axis=1)
        Rp = Rp + Qg
        u3 = uniform_of(row_words(g, row_ids, 1, seed)[:, 0])
        rep = (u3 * Rp < Qg) & (cand >= 0)
        with np.errstate(divide="ignore", invalid="ignore"):
            margin = np.minimum(margin, np.where(Qg > 0, np.abs(u3 * Rp - Qg) / Qg, np.inf))
        final = np.where(rep, cand, final)
    lse = M[:, 0] + np.log(q.sum(axis=1))
    logmu = z[rows, final] - lse
    return final, logmu, margin
