"""Textbook attention on contiguous tensors, used to pin the oracle.

The paged cache is first gathered into a contiguous [n, Hk, D] array with
numpy fancy indexing (logical token t -> block_table[t // S], offset t % S,
the paging rule of the tutorial page "LLM 推理服务引擎深度拆解", section 2.2),
then softmax(scale * q K^T) V is evaluated with numpy matrix products per
head.  Float conversion goes through torch/numpy (library routines), not the
oracle's own bit decoding.
"""
import numpy as np
import torch


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).numpy()


def gather(cache64: np.ndarray, bt_row, n: int) -> np.ndarray:
    S = cache64.shape[2]
    t = np.arange(n)
    bt_row = np.asarray(bt_row)
    return cache64[bt_row[t // S], :, t % S, :]          # [n, Hk, D]


def softmax_attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """q [D], K/V [n, D] -> [D]."""
    if K.shape[0] == 0:
        return np.zeros(q.shape[0])
    s = scale * (K @ q)
    w = np.exp(s - s.max())
    return (w / w.sum()) @ V


def decode(q, key_cache, value_cache, block_tables, context_lens, scale):
    q64, k64, v64 = to_f64(q), to_f64(key_cache), to_f64(value_cache)
    B, H, D = q64.shape
    Hk = k64.shape[1]
    G = H // Hk
    out = np.zeros((B, H, D))
    bt = block_tables.numpy()
    for i in range(B):
        n = int(context_lens[i])
        K, V = gather(k64, bt[i], n), gather(v64, bt[i], n)
        for h in range(H):
            out[i, h] = softmax_attend(q64[i, h], K[:, h // G], V[:, h // G], scale)
    return out


def prefill(q, cu_q_lens, key_cache, value_cache, block_tables, context_lens, scale):
    q64, k64, v64 = to_f64(q), to_f64(key_cache), to_f64(value_cache)
    NT, H, D = q64.shape
    Hk = k64.shape[1]
    G = H // Hk
    out = np.zeros((NT, H, D))
    bt = block_tables.numpy()
    cu = cu_q_lens.numpy()
    for i in range(cu.shape[0] - 1):
        C = int(cu[i + 1] - cu[i])
        P = int(context_lens[i]) - C
        K, V = gather(k64, bt[i], P + C), gather(v64, bt[i], P + C)
        for j in range(C):
            n = P + j + 1
            for h in range(H):
                out[cu[i] + j, h] = softmax_attend(q64[cu[i] + j, h], K[:n, h // G],
                                                   V[:n, h // G], scale)
    return out
