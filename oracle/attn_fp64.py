"""fp64 CPU oracle of the tensor-parallel self-attention block.

TEST INFRASTRUCTURE ONLY — used by ``tests/``, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py``; never by the product path.

What the block computes ("tensor-parallel-megatron" reading, attention section;
"Tensor Parallelism（TP）与 Sequence Parallelism（SP）", §2 "attention 的道理是一样的"):

    QKV = X·Wqkvᵀ              fused Q, K, V projection, [3h, h] weight, split by
                               columns so that each tensor shard owns whole heads
    O_j = softmax(Q_j·K_jᵀ/√d)·V_j   per head j, on the shard that owns it
    Z   = O·Woᵀ                output projection [h, h], split by rows; the shards'
                               partial sums are added (g: all-reduce, or the
                               reduce-scatter under sequence parallelism)

with h = a·d (a heads of width d; "Tensor Parallelism（TP）与 Sequence
Parallelism（SP）", §0 notation).  Activations ``[s, b, h]`` are flattened to
``[M, h]`` with row ``m = t·b + bi`` (token t of sequence bi).

Readings taken where the pages are silent (each listed in the design notes):

A1. Row layout of Wqkv.  The pages give the fused weight's interleaving per
    query group, [q₁ q₂ k₁ v₁ | q₃ q₄ k₂ v₂ | …] for grouped-query attention; with
    one query head per group (multi-head attention, as the pages' parameter count
    3h² + h² assumes) that is, per head j, rows [3dj, 3dj+d) = Wq_j,
    [3dj+d, 3dj+2d) = Wk_j, [3dj+2d, 3dj+3d) = Wv_j.  Tensor shard i owns heads
    [i·a/tp, (i+1)·a/tp), i.e. the contiguous rows [i·3h/tp, (i+1)·3h/tp).
A2. O's column layout: head j occupies columns [jd, (j+1)d) (heads concatenated),
    so shard i's slice of O is columns [i·h/tp, (i+1)·h/tp) — exactly the rows of
    Wo's input dimension it owns.
A3. Mask.  The printed formula softmax(QKᵀ/√d)V has no mask; ``causal=True``
    adds the decoder mask (key u visible to query t iff u ≤ t) of the GPT-style
    models the pages measure.  Both are provided; the unmasked form is the
    definition.
A4. No bias, no dropout on the probabilities, no softmax scaling other than
    1/√d (dropout here is the caller's, as in the MLP block).
A5. ``lse2`` is the base-2 log-sum-exp of the scaled scores of each query row,
    log2 Σ_u 2^(x_tu) with x = (q·k/√d)·log2(e): the statistic a streaming
    softmax keeps for its backward pass.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "LOG2E",
    "qkv_head_rows",
    "split_qkv",
    "merge_qkv",
    "attention_core_forward",
    "attention_core_backward",
    "attn_forward",
    "attn_backward",
    "attn_forward_sharded",
    "attn_backward_sharded",
]

LOG2E = 1.4426950408889634


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def qkv_head_rows(heads, d, j):
    """Rows of Wqkv (or columns of QKV) holding head j's q, k and v (reading A1)."""
    base = 3 * d * j
    return (range(base, base + d), range(base + d, base + 2 * d), range(base + 2 * d, base + 3 * d))


def split_qkv(QKV, heads):
    """[M, 3h] head-interleaved → Q, K, V, each [M, h] with head j in columns [jd, (j+1)d)."""
    QKV = _f64(QKV)
    M, three_h = QKV.shape
    h = three_h // 3
    d = h // heads
    r = QKV.reshape(M, heads, 3, d)
    return (r[:, :, 0, :].reshape(M, h), r[:, :, 1, :].reshape(M, h), r[:, :, 2, :].reshape(M, h))


def merge_qkv(Q, K, V, heads):
    """Inverse of split_qkv."""
    M, h = Q.shape
    d = h // heads
    out = np.empty((M, heads, 3, d))
    out[:, :, 0, :] = _f64(Q).reshape(M, heads, d)
    out[:, :, 1, :] = _f64(K).reshape(M, heads, d)
    out[:, :, 2, :] = _f64(V).reshape(M, heads, d)
    return out.reshape(M, 3 * h)


def _per_sequence(T, s, b, heads):
    """[M, h] with m = t·b + bi → [b, heads, s, d]."""
    M, h = T.shape
    d = h // heads
    return _f64(T).reshape(s, b, heads, d).transpose(1, 2, 0, 3)


def _from_per_sequence(T):
    """[b, heads, s, d] → [M, h]."""
    b, heads, s, d = T.shape
    return T.transpose(2, 0, 1, 3).reshape(s * b, heads * d)


def _scores(q, k, causal):
    """Scaled scores x = (q·kᵀ/√d)·log2(e) with masked entries at −inf.  q, k: [..., s, d]."""
    d = q.shape[-1]
    x = np.einsum("...td,...ud->...tu", q, k) * (LOG2E / math.sqrt(d))
    if causal:
        s = q.shape[-2]
        x = np.where(np.triu(np.ones((s, s), dtype=bool), k=1), -np.inf, x)
    return x


def attention_core_forward(Q, K, V, s, b, heads, causal=False):
    """O = softmax(QKᵀ/√d)V per sequence and head.  Q, K, V: [M, h].

    Returns {"O": [M, h], "lse2": [b, heads, s], "P": [b, heads, s, s]}."""
    q, k, v = (_per_sequence(T, s, b, heads) for T in (Q, K, V))
    x = _scores(q, k, causal)
    mx = x.max(axis=-1, keepdims=True)
    e = np.exp2(x - mx)
    den = e.sum(axis=-1, keepdims=True)
    P = e / den
    o = np.einsum("...tu,...ud->...td", P, v)
    lse2 = (mx + np.log2(den))[..., 0]
    return {"O": _from_per_sequence(o), "lse2": lse2, "P": P}


def attention_core_backward(Q, K, V, dO, s, b, heads, causal=False):
    """Gradients of the attention core given dO = ∂L/∂O: dQ, dK, dV, each [M, h].

    dV = Pᵀ·dO, dP = dO·Vᵀ, dS = P ⊙ (dP − rowsum(dP ⊙ P)) (softmax Jacobian),
    dQ = dS·K/√d, dK = dSᵀ·Q/√d."""
    q, k, v, do = (_per_sequence(T, s, b, heads) for T in (Q, K, V, dO))
    d = q.shape[-1]
    P = attention_core_forward(Q, K, V, s, b, heads, causal)["P"]
    dv = np.einsum("...tu,...td->...ud", P, do)
    dP = np.einsum("...td,...ud->...tu", do, v)
    dS = P * (dP - (dP * P).sum(axis=-1, keepdims=True))
    dq = np.einsum("...tu,...ud->...td", dS, k) / math.sqrt(d)
    dk = np.einsum("...tu,...td->...ud", dS, q) / math.sqrt(d)
    return {"dQ": _from_per_sequence(dq), "dK": _from_per_sequence(dk), "dV": _from_per_sequence(dv)}


def attn_forward(X, Wqkv, Wo, s, b, heads, causal=False):
    """The unsharded block.  X: [M, h] (or [s, b, h]); Wqkv: [3h, h]; Wo: [h, h]."""
    X = _f64(X).reshape(s * b, -1)
    QKV = X @ _f64(Wqkv).T
    Q, K, V = split_qkv(QKV, heads)
    core = attention_core_forward(Q, K, V, s, b, heads, causal)
    Z = core["O"] @ _f64(Wo).T
    return {"QKV": QKV, "O": core["O"], "lse2": core["lse2"], "Z": Z}


def attn_backward(X, Wqkv, Wo, dZ, s, b, heads, causal=False):
    """Gradients of the unsharded block given dZ: dX, dWqkv, dWo (and dO, dQKV)."""
    X = _f64(X).reshape(s * b, -1)
    dZ = _f64(dZ).reshape(s * b, -1)
    fw = attn_forward(X, Wqkv, Wo, s, b, heads, causal)
    dWo = dZ.T @ fw["O"]
    dO = dZ @ _f64(Wo)
    Q, K, V = split_qkv(fw["QKV"], heads)
    g = attention_core_backward(Q, K, V, dO, s, b, heads, causal)
    dQKV = merge_qkv(g["dQ"], g["dK"], g["dV"], heads)
    dWqkv = dQKV.T @ X
    dX = dQKV @ _f64(Wqkv)
    return {"dX": dX, "dWqkv": dWqkv, "dWo": dWo, "dO": dO, "dQKV": dQKV}


def attn_forward_sharded(X, Wqkv, Wo, s, b, heads, tp, causal=False):
    """The tensor-parallel form: shard i takes Wqkv rows [i·3h/tp, (i+1)·3h/tp)
    (its heads) and Wo columns [i·h/tp, (i+1)·h/tp); Z is the sum of the shards'
    partial outputs (g)."""
    X = _f64(X).reshape(s * b, -1)
    h = X.shape[1]
    hs, a_s = h // tp, heads // tp
    Z = np.zeros((s * b, h))
    for i in range(tp):
        QKV_i = X @ _f64(Wqkv)[3 * hs * i: 3 * hs * (i + 1)].T
        Q, K, V = split_qkv(QKV_i, a_s)
        O_i = attention_core_forward(Q, K, V, s, b, a_s, causal)["O"]
        Z += O_i @ _f64(Wo)[:, hs * i: hs * (i + 1)].T
    return Z


def attn_backward_sharded(X, Wqkv, Wo, dZ, s, b, heads, tp, causal=False):
    """Shard-local gradients: dWqkv and dWo are concatenations of the shards'
    blocks; dX is the sum of the shards' partial input gradients (f backward)."""
    X = _f64(X).reshape(s * b, -1)
    dZ = _f64(dZ).reshape(s * b, -1)
    h = X.shape[1]
    hs, a_s = h // tp, heads // tp
    dX = np.zeros_like(X)
    dWqkv = np.zeros((3 * h, h))
    dWo = np.zeros((h, h))
    for i in range(tp):
        rq = slice(3 * hs * i, 3 * hs * (i + 1))
        ro = slice(hs * i, hs * (i + 1))
        Wqkv_i = _f64(Wqkv)[rq]
        Wo_i = _f64(Wo)[:, ro]
        QKV_i = X @ Wqkv_i.T
        Q, K, V = split_qkv(QKV_i, a_s)
        O_i = attention_core_forward(Q, K, V, s, b, a_s, causal)["O"]
        dWo[:, ro] = dZ.T @ O_i
        dO_i = dZ @ Wo_i
        g = attention_core_backward(Q, K, V, dO_i, s, b, a_s, causal)
        dQKV_i = merge_qkv(g["dQ"], g["dK"], g["dV"], a_s)
        dWqkv[rq] = dQKV_i.T @ X
        dX += dQKV_i @ Wqkv_i
    return {"dX": dX, "dWqkv": dWqkv, "dWo": dWo}
