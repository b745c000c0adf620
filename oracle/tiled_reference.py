"""Tiled online-softmax attention in numpy float64 -- test infrastructure only.

Restates the forward algorithm of "FlashAttention V2 in depth" (section 6.1,
full forward algorithm) in its own order: an outer loop over query tiles of
B_r rows, an inner loop over key/value tiles of B_c rows, running row maximum
m (starting at -inf), running row sum l (starting at 0) and an unnormalised
accumulator O~ (starting at 0), each rescaled by exp(m_old - m_new) when a tile
raises the maximum (section 3.2, deferred rescaling), one division by l after
the inner loop, and L = m + log l.  With ``local_max=True`` it follows the
two-factor update of the Flash Attention 2 page (inner-loop steps 2-5: tile
max m_ij, P~ = exp(S - m_ij), l_ij, then both old and new terms rescaled to
m_new), which is algebraically the same.

``fa1_update=True`` instead keeps O normalised after every tile with the
FlashAttention V1 update of section 3.2 (multiply the old O by
l_old*exp(m_old - m_new)/l_new, add exp(S - m_new)V_j/l_new), which is also
exact.

The flags ``rescale_output``, ``m_init`` and ``normalize_in_loop`` exist only so
tests can plant, one at a time, the three slips that Lesson 6.6 ("Worked
example, step by step") names, and check that each one breaks exactness:
``normalize_in_loop`` divides the running output by l after every tile and
then keeps adding unnormalised terms to it.

``trace`` (optional list) receives, after every inner step, a dict with the
tile's S, the running m, l and O~, so the per-step values printed in the
pages' worked examples can be compared.
"""
from __future__ import annotations

import math

import numpy as np


def tiled_attention(Q, K, V, B_r: int, B_c: int, scale: float = 1.0, causal: bool = False,
                    local_max: bool = False, fa1_update: bool = False, rescale_output: bool = True,
                    m_init: float = -math.inf, normalize_in_loop: bool = False, trace=None):
    """O [N, d_v] and L [N] for one head; Q [N, d], K [N_k, d], V [N_k, d_v] float arrays."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    N, d = Q.shape
    N_k = K.shape[0]                                 # keys (equal to N whenever causal)
    O = np.zeros((N, V.shape[1]))
    L = np.zeros(N)
    for i in range(0, N, B_r):                       # outer loop over query tiles
        Qi = Q[i:i + B_r]
        rows = Qi.shape[0]
        m = np.full(rows, m_init)
        l = np.zeros(rows)
        Ot = np.zeros((rows, V.shape[1]))
        kv_end = min(N_k, i + B_r) if causal else N_k  # causal: stop at the diagonal
        for j in range(0, kv_end, B_c):              # inner loop over key/value tiles
            Kj = K[j:j + B_c]
            Vj = V[j:j + B_c]
            S = scale * (Qi @ Kj.T)
            if causal and i < j + Kj.shape[0] - 1:   # tile crosses the diagonal
                qpos = np.arange(i, i + rows)[:, None]
                kpos = np.arange(j, j + Kj.shape[0])[None, :]
                S = np.where(kpos <= qpos, S, -np.inf)
            with np.errstate(invalid="ignore", over="ignore"):
                if local_max:
                    m_ij = S.max(axis=1)
                    Pt = np.exp(S - np.where(np.isfinite(m_ij), m_ij, 0.0)[:, None])
                    l_ij = Pt.sum(axis=1)
                    m_new = np.maximum(m, m_ij)
                    safe = np.where(np.isfinite(m_new), m_new, 0.0)
                    a_old = np.exp(m - safe)
                    a_new = np.exp(np.where(np.isfinite(m_ij), m_ij, -np.inf) - safe)
                    l = a_old * l + a_new * l_ij
                    Ot = (a_old[:, None] if rescale_output else 1.0) * Ot + a_new[:, None] * (Pt @ Vj)
                else:
                    m_new = np.maximum(m, S.max(axis=1))
                    safe = np.where(np.isfinite(m_new), m_new, 0.0)
                    alpha = np.exp(m - safe)
                    P = np.exp(S - safe[:, None])
                    l_prev = l
                    l = alpha * l + P.sum(axis=1)
                    if fa1_update:
                        Ot = ((l_prev * alpha) / l)[:, None] * Ot + (P / l[:, None]) @ Vj
                    else:
                        Ot = (alpha[:, None] if rescale_output else 1.0) * Ot + P @ Vj
                if normalize_in_loop:
                    Ot = Ot / l[:, None]
            m = m_new
            if trace is not None:
                trace.append({"i": i, "j": j, "S": S.copy(), "m": m.copy(), "l": l.copy(), "O_tilde": Ot.copy()})
        if normalize_in_loop or fa1_update:
            O[i:i + B_r] = Ot
        else:
            O[i:i + B_r] = Ot / l[:, None]
        L[i:i + B_r] = m + np.log(l)
    return O, L


def split_keys_attention(Q, K, V, scale: float, chunk: int, visible=None, merge_rescale: bool = True):
    """Split-over-keys attention (the decoding regime) in numpy float64 -- test infrastructure only.

    The keys are cut into chunks of ``chunk`` rows; for every query row each
    chunk yields the online-softmax state of its visible keys on its own --
    local maximum m_c (-inf when the chunk shows the row nothing), l_c =
    sum exp(s - m_c) and O~_c = sum exp(s - m_c) v -- and the states are then
    merged with the same rescaling step the tiled loop applies between key
    tiles (Lesson 6.6, "Online softmax"; FlashAttention V2 in depth, section
    3.2): M = max_c m_c, l = sum_c exp(m_c - M) l_c, O = sum_c exp(m_c - M)
    O~_c / l, L = M + log l.  A row that sees no key gets O = 0, L = -inf.
    ``visible`` is a boolean [N_q, N_k] mask (None: every key visible).
    ``merge_rescale=False`` plants the slip of merging without the factors
    exp(m_c - M), so tests can check that it breaks exactness.

    Q [N_q, d], K [N_k, d], V [N_k, d_v]; returns O [N_q, d_v], L [N_q].
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    n_q, n_k = Q.shape[0], K.shape[0]
    if visible is None:
        visible = np.ones((n_q, n_k), dtype=bool)
    states = []
    for c0 in range(0, n_k, chunk):
        S = scale * (Q @ K[c0:c0 + chunk].T)
        S = np.where(visible[:, c0:c0 + chunk], S, -np.inf)
        m = S.max(axis=1)
        shift = np.where(np.isneginf(m), 0.0, m)
        P = np.exp(S - shift[:, None])                 # exp(-inf) = 0 for hidden keys
        states.append((m, P.sum(axis=1), P @ V[c0:c0 + chunk]))
    M = np.max([s[0] for s in states], axis=0)
    l = np.zeros(n_q)
    Ot = np.zeros((n_q, V.shape[1]))
    for m, lc, Oc in states:
        if merge_rescale:
            f = np.where(np.isneginf(m), 0.0, np.exp(m - np.where(np.isneginf(M), 0.0, M)))
        else:
            f = np.ones(n_q)
        l += f * lc
        Ot += f[:, None] * Oc
    empty = ~(l > 0)
    O = np.where(empty[:, None], 0.0, Ot / np.where(empty, 1.0, l)[:, None])
    L = np.where(empty, -np.inf, M + np.log(np.where(empty, 1.0, l)))
    return O, L
