"""Single-query attention over a cache, in float64 (oracle; test infrastructure only).

Three independent statements of the same result:

* ``cached_attention``: form A. The new key/value are appended to the
  history, scores are the scaled dot products of the single query with every
  row, a softmax with the maximum subtracted turns them into weights, and the
  output is the weighted sum of the value rows. This is knowledge point 2 of
  "KV缓存原理与显存估算" (LLM Systems Wiki): z_i = q.k_i / sqrt(d),
  a_i = exp(z_i - z_max) / sum_j exp(z_j - z_max), o = sum_i a_i v_i, with the
  append performed before the attention. The scale is an argument here; the
  page's default 1/sqrt(d) is used when it is omitted.
* ``causal_attention_full`` / ``decode_by_recompute``: form B. No cache: all
  t tokens' K/V are kept, the full t x t (or seq_len x total_len) score matrix
  is built, the causal mask of "单请求 KV Cache" (change 3: row i may see
  columns 0..past_len+i) sets the rest to -inf, and the last row is taken, as
  the no-cache generator of "KV-Cache——为什么AI回复越来越快" section 05 does
  with its last-token query.
* ``attention_loops``: form C, plain Python loops over scalars with
  ``math.exp``; used on tiny inputs to pin the NumPy forms.
"""

from __future__ import annotations

import math

import numpy as np


def _as_f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def stable_softmax(z: np.ndarray, axis: int = -1) -> np.ndarray:
    """softmax(z) computed as exp(z - max z) / sum exp(z - max z).

    Subtracting the row maximum leaves the softmax unchanged and keeps every
    exponent <= 0 ("KV-Cache——为什么AI回复越来越快" section 05, the stable
    softmax of the single-head attention class; LLM Systems Wiki knowledge
    point 2). Masked entries are -inf and receive weight exactly 0.
    """
    z = _as_f64(z)
    m = np.max(z, axis=axis, keepdims=True)
    e = np.exp(z - m)
    return e / np.sum(e, axis=axis, keepdims=True)


def cached_attention(query, past_keys, past_values, new_key, new_value, scale=None):
    """Form A: append (new_key, new_value) to the history, then attend.

    query: [d]; past_keys: [T, d]; past_values: [T, dv]; new_key: [d];
    new_value: [dv]. Returns (output [dv], weights [T+1], keys [T+1, d],
    values [T+1, dv]). Input checks follow the page: non-empty dimensions,
    K/V rows paired, all values finite.
    """
    q = _as_f64(query).reshape(-1)
    pk = _as_f64(past_keys).reshape(-1, q.shape[0]) if np.size(past_keys) else np.zeros((0, q.shape[0]))
    nv = _as_f64(new_value).reshape(-1)
    pv = _as_f64(past_values).reshape(-1, nv.shape[0]) if np.size(past_values) else np.zeros((0, nv.shape[0]))
    nk = _as_f64(new_key).reshape(-1)
    if q.shape[0] == 0 or nv.shape[0] == 0:
        raise ValueError("query and value rows must be non-empty")
    if nk.shape[0] != q.shape[0]:
        raise ValueError("key width must equal query width")
    if pk.shape[0] != pv.shape[0]:
        raise ValueError("history keys and values must pair up")
    keys = np.concatenate([pk, nk[None, :]], axis=0)
    values = np.concatenate([pv, nv[None, :]], axis=0)
    for arr in (q, keys, values):
        if not np.all(np.isfinite(arr)):
            raise ValueError("inputs must be finite")
    s = (1.0 / math.sqrt(q.shape[0])) if scale is None else float(scale)
    z = (keys @ q) * s
    a = stable_softmax(z)
    out = a @ values
    return out, a, keys, values


def attend_rows(q, K, V, scale):
    """Output of one query over the rows of K/V (form A without the append).

    q: [d]; K: [n, d]; V: [n, dv]; n >= 1. Returns (out [dv], lse) where lse
    is the natural log of sum_i exp(z_i), z_i = scale * q.k_i.
    """
    q = _as_f64(q)
    K = _as_f64(K)
    V = _as_f64(V)
    if K.shape[0] == 0:
        raise ValueError("attention needs at least one cached row")
    z = (K @ q) * float(scale)
    m = np.max(z)
    e = np.exp(z - m)
    tot = np.sum(e)
    return (e / tot) @ V, float(m + math.log(tot))


def causal_attention_full(Q, K, V, scale, past_len: int = 0):
    """Form B: full attention of seq_len queries over total_len keys with the causal mask.

    Q: [seq_len, d]; K: [total_len, d]; V: [total_len, dv];
    total_len = past_len + seq_len. Row i may see columns 0..past_len+i
    ("单请求 KV Cache", change 3); every other score is -inf. Returns
    [seq_len, dv].
    """
    Q = _as_f64(Q)
    K = _as_f64(K)
    V = _as_f64(V)
    seq_len, total_len = Q.shape[0], K.shape[0]
    if total_len != past_len + seq_len:
        raise ValueError("total_len must equal past_len + seq_len")
    scores = (Q @ K.T) * float(scale)
    cols = np.arange(total_len)[None, :]
    rows = np.arange(seq_len)[:, None]
    masked = cols > (past_len + rows)
    scores = np.where(masked, -np.inf, scores)
    return stable_softmax(scores, axis=-1) @ V


def decode_by_recompute(Q_all, K_all, V_all, scale):
    """Decode output for the last of t tokens by recomputing everything.

    Q_all, K_all: [t, d]; V_all: [t, dv]. Builds the full t x t causal
    attention (past_len = 0) and returns its last row, as the no-cache
    generator does with its last-token query.
    """
    return causal_attention_full(Q_all, K_all, V_all, scale, past_len=0)[-1]


def attention_loops(q, K, V, scale):
    """Form C: the same result with scalar Python loops (tiny inputs only)."""
    q = [float(x) for x in q]
    K = [[float(x) for x in row] for row in K]
    V = [[float(x) for x in row] for row in V]
    n = len(K)
    z = []
    for i in range(n):
        acc = 0.0
        for j in range(len(q)):
            acc += q[j] * K[i][j]
        z.append(acc * scale)
    peak = max(z)
    w = [math.exp(zi - peak) for zi in z]
    tot = sum(w)
    w = [wi / tot for wi in w]
    dv = len(V[0])
    out = []
    for c in range(dv):
        acc = 0.0
        for i in range(n):
            acc += w[i] * V[i][c]
        out.append(acc)
    return out
