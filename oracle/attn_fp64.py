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

A1. Row layout of Wqkv.  The pages give the fused weight as [h + 2·h_kv, h] and
    its interleaving per query group, [q₁ q₂ k₁ v₁ | q₃ q₄ k₂ v₂ | …] for
    grouped-query attention: with G key/value heads (groups) and r = a/G query
    heads per group, group g holds rows [g·(r+2)·d, (g+1)·(r+2)·d): its r query
    heads' q rows in head order, then its k rows, then its v rows.  Query head j
    belongs to group j // r.  With one query head per group (multi-head
    attention, G = a, as the pages' parameter count 3h² + h² assumes) that is,
    per head j, rows [3dj, 3dj+d) = Wq_j, [3dj+d, 3dj+2d) = Wk_j,
    [3dj+2d, 3dj+3d) = Wv_j.  Tensor shard i owns groups [i·G/tp, (i+1)·G/tp),
    i.e. the contiguous rows [i·(h+2h_kv)/tp, (i+1)·(h+2h_kv)/tp); G must be a
    multiple of tp (the pages' fallback when it is not, an all-gather of QKV
    before slicing, is not taken).
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
A6. Grouped-query attention: query head j attends with its group's key and
    value head g(j) = j // r, O_j = softmax(Q_j·K_gᵀ/√d)·V_g; a key/value head
    shared by r query heads receives the sum of their gradients.  The head
    width d = h/a is free (the pages use 128 and 96).

``kv_heads`` (G) defaults to ``heads`` (multi-head attention) everywhere.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "LOG2E",
    "qkv_width",
    "qkv_head_rows",
    "qkv_row_labels",
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


def qkv_width(heads, d, kv_heads=None):
    """Rows of the fused Wqkv: h + 2·h_kv = (a + 2G)·d."""
    G = heads if kv_heads is None else kv_heads
    return (heads + 2 * G) * d


def qkv_head_rows(heads, d, j, kv_heads=None):
    """Rows of Wqkv (or columns of QKV) holding query head j's q, and its
    group's k and v (reading A1)."""
    G = heads if kv_heads is None else kv_heads
    r = heads // G
    g = j // r
    base = g * (r + 2) * d
    q0 = base + (j - g * r) * d
    k0 = base + r * d
    return (range(q0, q0 + d), range(k0, k0 + d), range(k0 + d, k0 + 2 * d))


def qkv_row_labels(heads, kv_heads):
    """The fused weight's head blocks in row order, as the pages print them:
    'q1', 'q2', 'k1', 'v1', 'q3', … (query heads numbered 1…a, groups 1…G)."""
    r = heads // kv_heads
    out = []
    for g in range(kv_heads):
        out += [f"q{g * r + i + 1}" for i in range(r)] + [f"k{g + 1}", f"v{g + 1}"]
    return out


def split_qkv(QKV, heads, kv_heads=None):
    """[M, h + 2h_kv] group-interleaved → Q [M, h] (query head j in columns
    [jd, (j+1)d)), K and V [M, h_kv] (group g in columns [gd, (g+1)d))."""
    G = heads if kv_heads is None else kv_heads
    QKV = _f64(QKV)
    M, width = QKV.shape
    d = width // (heads + 2 * G)
    r = heads // G
    t = QKV.reshape(M, G, r + 2, d)
    return (t[:, :, :r, :].reshape(M, heads * d), t[:, :, r, :].reshape(M, G * d), t[:, :, r + 1, :].reshape(M, G * d))


def merge_qkv(Q, K, V, heads, kv_heads=None):
    """Inverse of split_qkv."""
    G = heads if kv_heads is None else kv_heads
    M, h = Q.shape
    d = h // heads
    r = heads // G
    out = np.empty((M, G, r + 2, d))
    out[:, :, :r, :] = _f64(Q).reshape(M, G, r, d)
    out[:, :, r, :] = _f64(K).reshape(M, G, d)
    out[:, :, r + 1, :] = _f64(V).reshape(M, G, d)
    return out.reshape(M, (heads + 2 * G) * d)


def _group_of(heads, kv_heads):
    """g(j) for every query head j (reading A6)."""
    return np.arange(heads) // (heads // kv_heads)


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


def attention_core_forward(Q, K, V, s, b, heads, causal=False, kv_heads=None):
    """O_j = softmax(Q_j·K_gᵀ/√d)·V_g per sequence and query head j, g = g(j).
    Q: [M, h]; K, V: [M, h_kv].

    Returns {"O": [M, h], "lse2": [b, heads, s], "P": [b, heads, s, s]}."""
    G = heads if kv_heads is None else kv_heads
    q = _per_sequence(Q, s, b, heads)
    grp = _group_of(heads, G)
    k = _per_sequence(K, s, b, G)[:, grp]  # query head j sees its group's keys and values
    v = _per_sequence(V, s, b, G)[:, grp]
    x = _scores(q, k, causal)
    mx = x.max(axis=-1, keepdims=True)
    e = np.exp2(x - mx)
    den = e.sum(axis=-1, keepdims=True)
    P = e / den
    o = np.einsum("...tu,...ud->...td", P, v)
    lse2 = (mx + np.log2(den))[..., 0]
    return {"O": _from_per_sequence(o), "lse2": lse2, "P": P}


def attention_core_backward(Q, K, V, dO, s, b, heads, causal=False, kv_heads=None):
    """Gradients of the attention core given dO = ∂L/∂O: dQ [M, h], dK, dV [M, h_kv].

    Per query head j (group g): dV_j = P_jᵀ·dO_j, dP_j = dO_j·V_gᵀ,
    dS_j = P_j ⊙ (dP_j − rowsum(dP_j ⊙ P_j)) (softmax Jacobian),
    dQ_j = dS_j·K_g/√d, dK_j = dS_jᵀ·Q_j/√d; a group's dK and dV are the sums
    over its query heads (reading A6)."""
    G = heads if kv_heads is None else kv_heads
    q, do = (_per_sequence(T, s, b, heads) for T in (Q, dO))
    grp = _group_of(heads, G)
    k = _per_sequence(K, s, b, G)[:, grp]
    v = _per_sequence(V, s, b, G)[:, grp]
    d = q.shape[-1]
    P = attention_core_forward(Q, K, V, s, b, heads, causal, G)["P"]
    dv = np.einsum("...tu,...td->...ud", P, do)
    dP = np.einsum("...td,...ud->...tu", do, v)
    dS = P * (dP - (dP * P).sum(axis=-1, keepdims=True))
    dq = np.einsum("...tu,...ud->...td", dS, k) / math.sqrt(d)
    dk = np.einsum("...tu,...td->...ud", dS, q) / math.sqrt(d)
    dk_g = np.zeros((dk.shape[0], G) + dk.shape[2:])
    dv_g = np.zeros_like(dk_g)
    for j in range(heads):  # a shared key/value head collects its query heads' gradients
        dk_g[:, grp[j]] += dk[:, j]
        dv_g[:, grp[j]] += dv[:, j]
    return {"dQ": _from_per_sequence(dq), "dK": _from_per_sequence(dk_g), "dV": _from_per_sequence(dv_g)}


def attn_forward(X, Wqkv, Wo, s, b, heads, causal=False, kv_heads=None):
    """The unsharded block.  X: [M, h] (or [s, b, h]); Wqkv: [h + 2h_kv, h]; Wo: [h, h]."""
    X = _f64(X).reshape(s * b, -1)
    QKV = X @ _f64(Wqkv).T
    Q, K, V = split_qkv(QKV, heads, kv_heads)
    core = attention_core_forward(Q, K, V, s, b, heads, causal, kv_heads)
    Z = core["O"] @ _f64(Wo).T
    return {"QKV": QKV, "O": core["O"], "lse2": core["lse2"], "Z": Z}


def attn_backward(X, Wqkv, Wo, dZ, s, b, heads, causal=False, kv_heads=None):
    """Gradients of the unsharded block given dZ: dX, dWqkv, dWo (and dO, dQKV)."""
    X = _f64(X).reshape(s * b, -1)
    dZ = _f64(dZ).reshape(s * b, -1)
    fw = attn_forward(X, Wqkv, Wo, s, b, heads, causal, kv_heads)
    dWo = dZ.T @ fw["O"]
    dO = dZ @ _f64(Wo)
    Q, K, V = split_qkv(fw["QKV"], heads, kv_heads)
    g = attention_core_backward(Q, K, V, dO, s, b, heads, causal, kv_heads)
    dQKV = merge_qkv(g["dQ"], g["dK"], g["dV"], heads, kv_heads)
    dWqkv = dQKV.T @ X
    dX = dQKV @ _f64(Wqkv)
    return {"dX": dX, "dWqkv": dWqkv, "dWo": dWo, "dO": dO, "dQKV": dQKV}


def attn_forward_sharded(X, Wqkv, Wo, s, b, heads, tp, causal=False, kv_heads=None):
    """The tensor-parallel form: shard i takes Wqkv rows
    [i·(h+2h_kv)/tp, (i+1)·(h+2h_kv)/tp) (its groups, with their query heads)
    and Wo columns [i·h/tp, (i+1)·h/tp); Z is the sum of the shards' partial
    outputs (g)."""
    G = heads if kv_heads is None else kv_heads
    X = _f64(X).reshape(s * b, -1)
    h = X.shape[1]
    hs, a_s, g_s = h // tp, heads // tp, G // tp
    ws = (Wqkv.shape[0]) // tp
    Z = np.zeros((s * b, h))
    for i in range(tp):
        QKV_i = X @ _f64(Wqkv)[ws * i: ws * (i + 1)].T
        Q, K, V = split_qkv(QKV_i, a_s, g_s)
        O_i = attention_core_forward(Q, K, V, s, b, a_s, causal, g_s)["O"]
        Z += O_i @ _f64(Wo)[:, hs * i: hs * (i + 1)].T
    return Z


def attn_backward_sharded(X, Wqkv, Wo, dZ, s, b, heads, tp, causal=False, kv_heads=None):
    """Shard-local gradients: dWqkv and dWo are concatenations of the shards'
    blocks; dX is the sum of the shards' partial input gradients (f backward)."""
    G = heads if kv_heads is None else kv_heads
    X = _f64(X).reshape(s * b, -1)
    dZ = _f64(dZ).reshape(s * b, -1)
    h = X.shape[1]
    hs, a_s, g_s = h // tp, heads // tp, G // tp
    ws = (Wqkv.shape[0]) // tp
    dX = np.zeros_like(X)
    dWqkv = np.zeros((Wqkv.shape[0], h))
    dWo = np.zeros((h, h))
    for i in range(tp):
        rq = slice(ws * i, ws * (i + 1))
        ro = slice(hs * i, hs * (i + 1))
        Wqkv_i = _f64(Wqkv)[rq]
        Wo_i = _f64(Wo)[:, ro]
        QKV_i = X @ Wqkv_i.T
        Q, K, V = split_qkv(QKV_i, a_s, g_s)
        O_i = attention_core_forward(Q, K, V, s, b, a_s, causal, g_s)["O"]
        dWo[:, ro] = dZ.T @ O_i
        dO_i = dZ @ Wo_i
        g = attention_core_backward(Q, K, V, dO_i, s, b, a_s, causal, g_s)
        dQKV_i = merge_qkv(g["dQ"], g["dK"], g["dV"], a_s, g_s)
        dWqkv[rq] = dQKV_i.T @ X
        dX += dQKV_i @ Wqkv_i
    return {"dX": dX, "dWqkv": dWqkv, "dWo": dWo}
