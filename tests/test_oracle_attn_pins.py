"""Pins of the attention-block oracle (oracle/attn_fp64.py) against things other
than itself: explicit loops, closed forms, an independent library routine,
finite differences, invariances the definition implies, and the pages' sizes."""
import math

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle as O


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _case(s, b, heads, d, seed=0, wscale=0.3):
    h = heads * d
    X = _rand((s * b, h), seed)
    Wqkv = _rand((3 * h, h), seed + 1, wscale)
    Wo = _rand((h, h), seed + 2, wscale)
    dZ = _rand((s * b, h), seed + 3)
    return X, Wqkv, Wo, dZ


def _loops_forward(X, Wqkv, Wo, s, b, heads, causal):
    """Scalar loops, written from the formula without NumPy vector algebra."""
    M, h = X.shape
    d = h // heads
    QKV = [[sum(X[m][c] * Wqkv[r][c] for c in range(h)) for r in range(3 * h)] for m in range(M)]
    Ocat = [[0.0] * h for _ in range(M)]
    for bi in range(b):
        for j in range(heads):
            qr, kr, vr = (list(r) for r in O.qkv_head_rows(heads, d, j))
            for t in range(s):
                mt = t * b + bi
                scores = []
                for u in range(s):
                    if causal and u > t:
                        continue
                    mu = u * b + bi
                    dot = sum(QKV[mt][qr[e]] * QKV[mu][kr[e]] for e in range(d))
                    scores.append((u, dot / math.sqrt(d)))
                top = max(v for _, v in scores)
                w = [(u, math.exp(v - top)) for u, v in scores]
                tot = sum(x for _, x in w)
                for e in range(d):
                    Ocat[mt][j * d + e] = sum(x / tot * QKV[u * b + bi][vr[e]] for u, x in w)
    Z = [[sum(Ocat[m][c] * Wo[n][c] for c in range(h)) for n in range(h)] for m in range(M)]
    return np.array(Ocat), np.array(Z)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_matches_scalar_loops(causal):
    s, b, heads, d = 3, 2, 2, 2
    X, Wqkv, Wo, _ = _case(s, b, heads, d, seed=5)
    fw = O.attn_forward(X, Wqkv, Wo, s, b, heads, causal)
    Ol, Zl = _loops_forward(X, Wqkv, Wo, s, b, heads, causal)
    assert np.allclose(fw["O"], Ol, rtol=1e-12, atol=1e-12)
    assert np.allclose(fw["Z"], Zl, rtol=1e-12, atol=1e-12)


def test_zero_queries_give_the_mean_of_the_values():
    """Wq = 0: every score is 0, the weights are uniform over the visible keys, so
    O_t is the mean of V over all keys (unmasked) or over keys ≤ t (causal)."""
    s, b, heads, d = 5, 2, 2, 3
    X, Wqkv, Wo, _ = _case(s, b, heads, d, seed=7)
    for j in range(heads):
        Wqkv[list(O.qkv_head_rows(heads, d, j)[0])] = 0.0
    Q, K, V = O.split_qkv(X @ Wqkv.T, heads)
    Vs = V.reshape(s, b, heads * d)
    full = O.attn_forward(X, Wqkv, Wo, s, b, heads, False)["O"].reshape(s, b, -1)
    caus = O.attn_forward(X, Wqkv, Wo, s, b, heads, True)["O"].reshape(s, b, -1)
    assert np.allclose(full, np.broadcast_to(Vs.mean(axis=0), full.shape), atol=1e-12)
    prefix = np.cumsum(Vs, axis=0) / np.arange(1, s + 1)[:, None, None]
    assert np.allclose(caus, prefix, atol=1e-12)


def test_single_token_and_first_causal_row_return_v():
    X, Wqkv, Wo, _ = _case(1, 3, 2, 4, seed=9)
    fw = O.attn_forward(X, Wqkv, Wo, 1, 3, 2, False)
    assert np.allclose(fw["O"], O.split_qkv(fw["QKV"], 2)[2], atol=1e-13)
    s, b = 6, 2
    X, Wqkv, Wo, _ = _case(s, b, 2, 4, seed=10)
    fw = O.attn_forward(X, Wqkv, Wo, s, b, 2, True)
    V = O.split_qkv(fw["QKV"], 2)[2]
    assert np.allclose(fw["O"][:b], V[:b], atol=1e-13)  # token 0 of every sequence


def test_lse2_against_scipy_logsumexp():
    s, b, heads, d = 7, 2, 3, 4
    X, Wqkv, Wo, _ = _case(s, b, heads, d, seed=11)
    for causal in (False, True):
        fw = O.attn_forward(X, Wqkv, Wo, s, b, heads, causal)
        Q, K, V = O.split_qkv(fw["QKV"], heads)
        for bi in range(b):
            for j in range(heads):
                q = Q.reshape(s, b, heads, d)[:, bi, j]
                k = K.reshape(s, b, heads, d)[:, bi, j]
                nat = q @ k.T / math.sqrt(d)
                if causal:
                    nat = np.where(np.triu(np.ones((s, s), bool), 1), -np.inf, nat)
                ref = logsumexp(nat, axis=1) / math.log(2.0)
                assert np.allclose(fw["lse2"][bi, j], ref, atol=1e-12)


def test_permutation_equivariance_without_mask():
    s, b, heads, d = 6, 1, 2, 3
    X, Wqkv, Wo, _ = _case(s, b, heads, d, seed=12)
    perm = np.random.default_rng(3).permutation(s)
    a = O.attn_forward(X, Wqkv, Wo, s, b, heads, False)["Z"]
    p = O.attn_forward(X[perm], Wqkv, Wo, s, b, heads, False)["Z"]
    assert np.allclose(p, a[perm], atol=1e-12)
    # the causal form is not equivariant (a planted swap of the mask would pass otherwise)
    c = O.attn_forward(X, Wqkv, Wo, s, b, heads, True)["Z"]
    cp = O.attn_forward(X[perm], Wqkv, Wo, s, b, heads, True)["Z"]
    assert not np.allclose(cp, c[perm], atol=1e-6)


def test_output_is_linear_in_values():
    """Scaling Wv by c scales O and Z by c (the weights do not depend on V)."""
    s, b, heads, d = 4, 2, 2, 3
    X, Wqkv, Wo, _ = _case(s, b, heads, d, seed=13)
    W2 = Wqkv.copy()
    for j in range(heads):
        W2[list(O.qkv_head_rows(heads, d, j)[2])] *= 2.5
    a = O.attn_forward(X, Wqkv, Wo, s, b, heads, True)
    c = O.attn_forward(X, W2, Wo, s, b, heads, True)
    assert np.allclose(c["O"], 2.5 * a["O"], atol=1e-12)
    assert np.allclose(c["Z"], 2.5 * a["Z"], atol=1e-12)


def _loss(X, Wqkv, Wo, dZ, s, b, heads, causal):
    return float((O.attn_forward(X, Wqkv, Wo, s, b, heads, causal)["Z"] * dZ).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_by_central_differences(causal):
    s, b, heads, d = 4, 2, 2, 2
    X, Wqkv, Wo, dZ = _case(s, b, heads, d, seed=21, wscale=0.5)
    g = O.attn_backward(X, Wqkv, Wo, dZ, s, b, heads, causal)
    eps = 1e-6
    rng = np.random.default_rng(4)
    for name, T in (("dX", X), ("dWqkv", Wqkv), ("dWo", Wo)):
        for _ in range(12):
            idx = tuple(int(rng.integers(0, n)) for n in T.shape)
            old = T[idx]
            T[idx] = old + eps
            lp = _loss(X, Wqkv, Wo, dZ, s, b, heads, causal)
            T[idx] = old - eps
            lm = _loss(X, Wqkv, Wo, dZ, s, b, heads, causal)
            T[idx] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(g[name][idx] - fd) <= 1e-6 * max(1.0, abs(fd)), (name, idx, g[name][idx], fd)


@pytest.mark.parametrize("causal", [False, True])
def test_core_gradients_by_central_differences(causal):
    """dQ, dK, dV of the core alone (the softmax Jacobian and the 1/√d factors)."""
    s, b, heads, d = 5, 1, 2, 3
    rng = np.random.default_rng(8)
    Q, K, V, dO = (rng.standard_normal((s * b, heads * d)) for _ in range(4))
    g = O.attention_core_backward(Q, K, V, dO, s, b, heads, causal)

    def loss():
        return float((O.attention_core_forward(Q, K, V, s, b, heads, causal)["O"] * dO).sum())

    eps = 1e-6
    for name, T in (("dQ", Q), ("dK", K), ("dV", V)):
        for idx in [(0, 0), (2, 3), (s * b - 1, heads * d - 1), (3, 1)]:
            old = T[idx]
            T[idx] = old + eps
            lp = loss()
            T[idx] = old - eps
            lm = loss()
            T[idx] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(g[name][idx] - fd) <= 1e-6 * max(1.0, abs(fd)), (name, idx)


@pytest.mark.parametrize("causal", [False, True])
def test_sharded_by_heads_equals_unsharded(causal):
    s, b, heads, d, tp = 5, 2, 4, 3, 2
    X, Wqkv, Wo, dZ = _case(s, b, heads, d, seed=31)
    full = O.attn_forward(X, Wqkv, Wo, s, b, heads, causal)
    assert np.allclose(O.attn_forward_sharded(X, Wqkv, Wo, s, b, heads, tp, causal), full["Z"], atol=1e-12)
    gb = O.attn_backward(X, Wqkv, Wo, dZ, s, b, heads, causal)
    gs = O.attn_backward_sharded(X, Wqkv, Wo, dZ, s, b, heads, tp, causal)
    for k in ("dX", "dWqkv", "dWo"):
        assert np.allclose(gs[k], gb[k], atol=1e-11), k


def test_splitting_qkv_by_whole_blocks_instead_of_heads_is_wrong():
    """Reading A1 matters: taking Q, K, V as the three contiguous [h] blocks of
    QKV (instead of per-head interleaving) changes the result."""
    s, b, heads, d = 4, 1, 2, 3
    X, Wqkv, Wo, _ = _case(s, b, heads, d, seed=41)
    QKV = X @ Wqkv.T
    h = heads * d
    Qb, Kb, Vb = QKV[:, :h], QKV[:, h:2 * h], QKV[:, 2 * h:]
    wrong = O.attention_core_forward(Qb, Kb, Vb, s, b, heads)["O"]
    right = O.attn_forward(X, Wqkv, Wo, s, b, heads)["O"]
    assert not np.allclose(wrong, right, atol=1e-3)
    Q, K, V = O.split_qkv(QKV, heads)
    assert np.array_equal(O.merge_qkv(Q, K, V, heads), QKV)


def test_attention_parameter_count_per_shard():
    """Attention weights per layer and shard: (3h² + h²)/tp ("Tensor Parallelism（TP）与
    Sequence Parallelism（SP）" calculator, MHA: QKV 3h² + output h²); with the MLP's
    2hf/tp the page's default case (h=4096, f=16384, TP=8) gives 25,165,824."""
    h, f, tp = 4096, 16384, 8
    heads = 32
    d = h // heads
    shard_qkv_rows = len(range(0, 3 * h // tp))
    assert shard_qkv_rows * h + h * (h // tp) == 4 * h * h // tp
    assert (2 * h * f + 4 * h * h) // tp == 25_165_824
    # each shard's heads are whole: its Wqkv rows hold q, k, v of heads [i·a/tp, (i+1)·a/tp)
    i = 3
    rows = set(range(3 * h // tp * i, 3 * h // tp * (i + 1)))
    for j in range(heads // tp * i, heads // tp * (i + 1)):
        for r in O.qkv_head_rows(heads, d, j):
            assert set(r) <= rows


# ---------------------------------------------------------------- grouped-query attention (reading A6)


def _gqa_case(s, b, heads, kv, d, seed=0, wscale=0.3):
    h = heads * d
    X = _rand((s * b, h), seed)
    Wqkv = _rand((O.qkv_width(heads, d, kv), h), seed + 1, wscale)
    Wo = _rand((h, h), seed + 2, wscale)
    dZ = _rand((s * b, h), seed + 3)
    return X, Wqkv, Wo, dZ


def test_fused_weight_rows_follow_the_printed_interleave():
    """The "tensor-parallel-megatron" reading (attention section) prints the GQA
    fused weight as [q₁ q₂ k₁ v₁ | q₃ q₄ k₂ v₂ | …] and its shape as
    [h + 2·h_kv, h]: four query heads in two groups, block by block."""
    assert O.qkv_row_labels(4, 2) == ["q1", "q2", "k1", "v1", "q3", "q4", "k2", "v2"]
    assert O.qkv_row_labels(2, 2) == ["q1", "k1", "v1", "q2", "k2", "v2"]  # MHA
    d = 3
    assert O.qkv_width(4, d, 2) == 4 * d + 2 * 2 * d
    labels = O.qkv_row_labels(4, 2)
    for j in range(4):
        q, k, v = O.qkv_head_rows(4, d, j, 2)
        assert labels[q.start // d] == f"q{j + 1}"
        assert labels[k.start // d] == f"k{j // 2 + 1}" and labels[v.start // d] == f"v{j // 2 + 1}"
        assert len(q) == len(k) == len(v) == d


def _loops_forward_gqa(X, Wqkv, Wo, s, b, heads, kv, causal):
    """Scalar loops from reading A6: query head j uses the k and v rows of its
    group j // (heads/kv), located by the printed labels."""
    M, h = X.shape
    d = h // heads
    labels = O.qkv_row_labels(heads, kv)
    row0 = {lab: i * d for i, lab in enumerate(labels)}
    QKV = [[sum(X[m][c] * Wqkv[r][c] for c in range(h)) for r in range(len(labels) * d)] for m in range(M)]
    Ocat = [[0.0] * h for _ in range(M)]
    r = heads // kv
    for bi in range(b):
        for j in range(heads):
            qb, kb, vb = row0[f"q{j + 1}"], row0[f"k{j // r + 1}"], row0[f"v{j // r + 1}"]
            for t in range(s):
                mt = t * b + bi
                sc = []
                for u in range(s):
                    if causal and u > t:
                        continue
                    dot = sum(QKV[mt][qb + e] * QKV[u * b + bi][kb + e] for e in range(d))
                    sc.append((u, dot / math.sqrt(d)))
                top = max(v for _, v in sc)
                w = [(u, math.exp(v - top)) for u, v in sc]
                tot = sum(x for _, x in w)
                for e in range(d):
                    Ocat[mt][j * d + e] = sum(x / tot * QKV[u * b + bi][vb + e] for u, x in w)
    Z = [[sum(Ocat[m][c] * Wo[n][c] for c in range(h)) for n in range(h)] for m in range(M)]
    return np.array(Ocat), np.array(Z)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_forward_matches_scalar_loops(causal):
    s, b, heads, kv, d = 3, 2, 4, 2, 2
    X, Wqkv, Wo, _ = _gqa_case(s, b, heads, kv, d, seed=51)
    fw = O.attn_forward(X, Wqkv, Wo, s, b, heads, causal, kv)
    Ol, Zl = _loops_forward_gqa(X, Wqkv, Wo, s, b, heads, kv, causal)
    assert np.allclose(fw["O"], Ol, rtol=1e-12, atol=1e-12)
    assert np.allclose(fw["Z"], Zl, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_gradients_by_central_differences(causal):
    """A key/value head shared by several query heads: its weights' gradient is
    the sum over the heads that read it, which finite differences see directly."""
    s, b, heads, kv, d = 4, 2, 4, 2, 2
    X, Wqkv, Wo, dZ = _gqa_case(s, b, heads, kv, d, seed=61, wscale=0.5)
    g = O.attn_backward(X, Wqkv, Wo, dZ, s, b, heads, causal, kv)

    def loss():
        return float((O.attn_forward(X, Wqkv, Wo, s, b, heads, causal, kv)["Z"] * dZ).sum())

    eps = 1e-6
    rng = np.random.default_rng(6)
    k_rows = [r for j in range(heads) for r in O.qkv_head_rows(heads, d, j, kv)[1]]
    for name, T, picks in (("dX", X, None), ("dWqkv", Wqkv, k_rows), ("dWqkv", Wqkv, None), ("dWo", Wo, None)):
        for _ in range(10):
            idx = tuple(int(rng.integers(0, n)) for n in T.shape)
            if picks is not None:  # a row of a shared key head
                idx = (int(picks[rng.integers(0, len(picks))]), idx[1])
            old = T[idx]
            T[idx] = old + eps
            lp = loss()
            T[idx] = old - eps
            lm = loss()
            T[idx] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(g[name][idx] - fd) <= 1e-6 * max(1.0, abs(fd)), (name, idx, g[name][idx], fd)


def test_gqa_with_one_group_per_head_is_multi_head_attention():
    """kv_heads = heads is the MHA layout (reading A1): both calls agree bit for bit."""
    s, b, heads, d = 4, 2, 2, 3
    X, Wqkv, Wo, dZ = _case(s, b, heads, d, seed=71)
    a = O.attn_backward(X, Wqkv, Wo, dZ, s, b, heads, True)
    g = O.attn_backward(X, Wqkv, Wo, dZ, s, b, heads, True, heads)
    for k in ("dX", "dWqkv", "dWo"):
        assert np.array_equal(a[k], g[k]), k


def test_gqa_is_not_attention_with_separate_key_heads():
    """Sharing matters: giving every query head its own copy of the key/value
    weights and then perturbing one copy changes only that head's output, while
    perturbing a shared group's weights changes every head of the group."""
    s, b, heads, kv, d = 4, 1, 4, 2, 2
    X, Wqkv, Wo, _ = _gqa_case(s, b, heads, kv, d, seed=81)
    base = O.attn_forward(X, Wqkv, Wo, s, b, heads, False, kv)["O"]
    W2 = Wqkv.copy()
    W2[list(O.qkv_head_rows(heads, d, 0, kv)[1])] += 0.5  # group 0's k rows (heads 0 and 1)
    o2 = O.attn_forward(X, W2, Wo, s, b, heads, False, kv)["O"]
    changed = [not np.allclose(o2[:, j * d:(j + 1) * d], base[:, j * d:(j + 1) * d]) for j in range(heads)]
    assert changed == [True, True, False, False]


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_sharded_by_groups_equals_unsharded(causal):
    s, b, heads, kv, d, tp = 4, 2, 8, 4, 2, 2
    X, Wqkv, Wo, dZ = _gqa_case(s, b, heads, kv, d, seed=91)
    full = O.attn_forward(X, Wqkv, Wo, s, b, heads, causal, kv)
    assert np.allclose(O.attn_forward_sharded(X, Wqkv, Wo, s, b, heads, tp, causal, kv), full["Z"], atol=1e-12)
    gb = O.attn_backward(X, Wqkv, Wo, dZ, s, b, heads, causal, kv)
    gs = O.attn_backward_sharded(X, Wqkv, Wo, dZ, s, b, heads, tp, causal, kv)
    for k in ("dX", "dWqkv", "dWo"):
        assert np.allclose(gs[k], gb[k], atol=1e-11), k
    # shard i's Wqkv rows are exactly its groups' blocks, query heads included
    ws = O.qkv_width(heads, d, kv) // tp
    for i in range(tp):
        rows = set(range(ws * i, ws * (i + 1)))
        for j in range(heads // tp * i, heads // tp * (i + 1)):
            for r in O.qkv_head_rows(heads, d, j, kv):
                assert set(r) <= rows


def test_gqa_workload_sizes():
    """The pages' GQA numbers: 8 KV heads × 128 = h_kv 1024 against MHA's 8192 at
    64 heads × 128 (an 8× smaller KV); the fused weight of the Llama-70B-like width
    is [8192 + 2·1024, 8192]."""
    assert 8 * 128 == 1024 and 64 * 128 == 8192 and 8192 // 1024 == 8
    assert O.qkv_width(64, 128, 8) == 8192 + 2 * 1024
    assert O.qkv_width(64, 128) == 3 * 8192
