"""The dense mask-matrix formulation, fp64 numpy, for tiny inputs.

TEST INFRASTRUCTURE (see the package docstring). This follows the structure of
kopitiam-runtime 0.2.4 src/attention.rs step by step, in numpy:

* ``repeat_kv_heads`` -- each KV head's data repeated ``group_size`` times
  contiguously (a broadcast over a new axis after the head axis, then a reshape),
  so query head g lines up with KV head g // group_size; identity for group 1.
* ``causal_mask``     -- additive bias [1, seq_q, seq_kv]: 0 where key j is visible
  to row i (j <= position_offset + i), -inf elsewhere.
* ``attention``       -- per head: scores = q k^T * scale, + mask, softmax over the
  key axis, probs @ v, heads back to [seq, H, dv].

It is a second, independent route to the same numbers as the C loops in
``gqa_oracle.c``; the tests require the two to agree to 1e-12.
"""
import numpy as np


def repeat_kv_heads(x: np.ndarray, group_size: int) -> np.ndarray:
    """x [n_kv, seq, d] -> [n_kv * group_size, seq, d]."""
    if group_size == 1:
        return x
    n_kv, seq, d = x.shape
    return np.broadcast_to(x.reshape(n_kv, 1, seq, d), (n_kv, group_size, seq, d)).reshape(
        n_kv * group_size, seq, d)


def causal_mask(seq_q: int, seq_kv: int, position_offset: int) -> np.ndarray:
    """[1, seq_q, seq_kv] additive bias, 0 = visible, -inf = masked."""
    mask = np.zeros((1, seq_q, seq_kv), np.float64)
    for i in range(seq_q):
        last_visible = position_offset + i
        mask[0, i, last_visible + 1:] = -np.inf
    return mask


def softmax_last(x: np.ndarray) -> np.ndarray:
    m = np.max(x, axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attention(q: np.ndarray, k_full: np.ndarray, v_full: np.ndarray, position_offset: int,
              scale: float) -> np.ndarray:
    """One sequence. q [seq_q, H, dk]; k_full [Hkv, seq_kv, dk]; v_full [Hkv, seq_kv, dv]
    (the cache after this pass's rows were appended). Returns [seq_q, H, dv]."""
    seq_q, H, _ = q.shape
    Hkv, seq_kv, _ = k_full.shape
    group = H // Hkv
    qh = np.transpose(q, (1, 0, 2))                        # [H, seq_q, dk]
    k_rep = repeat_kv_heads(k_full, group)                 # [H, seq_kv, dk]
    v_rep = repeat_kv_heads(v_full, group)                 # [H, seq_kv, dv]
    scores = np.matmul(qh, np.transpose(k_rep, (0, 2, 1))) * scale
    scores = scores + causal_mask(seq_q, seq_kv, position_offset)
    probs = softmax_last(scores)
    return np.transpose(np.matmul(probs, v_rep), (1, 0, 2))


def probabilities(q: np.ndarray, k_full: np.ndarray, position_offset: int, scale: float) -> np.ndarray:
    """The softmax weights [H, seq_q, seq_kv] of :func:`attention`."""
    seq_q, H, _ = q.shape
    Hkv = k_full.shape[0]
    k_rep = repeat_kv_heads(k_full, H // Hkv)
    scores = np.matmul(np.transpose(q, (1, 0, 2)), np.transpose(k_rep, (0, 2, 1))) * scale
    return softmax_last(scores + causal_mask(seq_q, k_full.shape[1], position_offset))


def attention_arms(q: np.ndarray, k_full: np.ndarray, v_full: np.ndarray, position_offset: int, scale: float,
                   window: int = 0, softcap: float = 0.0, sinks=None, slopes=None) -> np.ndarray:
    """`attention` with the arms of the attention row, as one additive bias matrix
    and one extra key: per head, scores = q k^T * scale; softcap c > 0 maps them
    to c * tanh(scores / c); ALiBi adds slope_h * (j - p); the mask takes keys
    past the row's position and, with a window W > 0, keys at or before p - W;
    a sink z_h is one more key column with logit z_h and a zero value vector.
    Shapes as in `attention`."""
    seq_q, H, _ = q.shape
    Hkv, seq_kv, dv = v_full.shape
    group = H // Hkv
    qh = np.transpose(q, (1, 0, 2))
    k_rep = repeat_kv_heads(k_full, group)
    v_rep = repeat_kv_heads(v_full, group)
    scores = np.matmul(qh, np.transpose(k_rep, (0, 2, 1))) * scale          # [H, seq_q, seq_kv]
    if softcap > 0:
        scores = softcap * np.tanh(scores / softcap)
    pos = position_offset + np.arange(seq_q)[:, None]                          # [seq_q, 1]
    keys = np.arange(seq_kv)[None, :]                                          # [1, seq_kv]
    if slopes is not None:
        scores = scores + np.asarray(slopes, np.float64)[:, None, None] * (keys - pos)[None]
    visible = keys <= pos
    if window > 0:
        visible = visible & (keys > pos - window)
    scores = np.where(visible[None], scores, -np.inf)
    if sinks is not None:  # the extra key: logit z_h for every row, value 0
        z = np.broadcast_to(np.asarray(sinks, np.float64)[:, None, None], (H, seq_q, 1))
        scores = np.concatenate([scores, z], axis=2)
        v_rep = np.concatenate([v_rep, np.zeros((H, 1, dv))], axis=1)
    probs = softmax_last(scores)
    return np.transpose(np.matmul(probs, v_rep), (1, 0, 2))
