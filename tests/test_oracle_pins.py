"""Pins of the fp64 CPU oracle against things other than itself (CPU only).

Each test ties one oracle function to a value the pages print, a closed form, a
finite difference, a brute-force loop or an independent library routine, chosen
so that a plausible slip (a dropped term, a wrong sign or index, a transposed
operand, a wrong shard order) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import erf, expit

import oracle as O
from synthetic import integer_block_inputs

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_values.json")))
ACTS = ["gelu", "swiglu", "identity", "relu"]


# ---------------------------------------------------------------- activations


def test_gelu_closed_forms():
    assert O.gelu_tanh(0.0) == 0.0
    assert O.gelu_tanh_grad(0.0) == 0.5
    x = np.linspace(-7, 7, 2001)
    # tanh is odd, so gelu(x) - gelu(-x) = x exactly (up to rounding).
    np.testing.assert_allclose(O.gelu_tanh(x) - O.gelu_tanh(-x), x, atol=1e-12)
    # asymptotes: gelu(x) -> x for x -> +inf, -> 0 for x -> -inf
    assert abs(O.gelu_tanh(12.0) - 12.0) < 1e-12 and abs(O.gelu_tanh(-12.0)) < 1e-12


def test_gelu_tanh_is_within_its_bound_of_the_erf_definition():
    """The tanh form approximates x·Φ(x) (Hendrycks & Gimpel); |diff| < 4.8e-4 on R."""
    x = np.linspace(-8, 8, 40001)
    exact = 0.5 * x * (1.0 + erf(x / math.sqrt(2.0)))
    assert np.abs(O.gelu_tanh(x) - exact).max() < 4.8e-4


@pytest.mark.parametrize("fn,grad", [(O.gelu_tanh, O.gelu_tanh_grad), (O.silu, O.silu_grad)])
def test_activation_grad_finite_difference(fn, grad):
    x = np.linspace(-6, 6, 1201)
    eps = 1e-6
    fd = (fn(x + eps) - fn(x - eps)) / (2 * eps)
    np.testing.assert_allclose(grad(x), fd, rtol=1e-7, atol=1e-8)


def test_silu_against_library_sigmoid():
    x = np.linspace(-30, 30, 3001)
    np.testing.assert_allclose(O.silu(x), x * expit(x), rtol=1e-14, atol=1e-300)
    assert O.silu(0.0) == 0.0 and O.silu_grad(0.0) == 0.5
    np.testing.assert_allclose(O.silu(x) - O.silu(-x), x, atol=1e-12)


def test_relu_counterexample_from_the_page():
    g = GOLDEN["relu_counterexample"]
    z0, z1 = g["Z0"], g["Z1"]
    assert O.act_forward(np.array([z0]), "relu")[0] + O.act_forward(np.array([z1]), "relu")[0] == g["sum_of_relu"]
    assert O.act_forward(np.array([z0 + z1]), "relu")[0] == g["relu_of_sum"]
    assert O.relu_grad(np.array([-1.0, 0.5]))[1] == 1.0 and O.relu_grad(np.array([-1.0]))[0] == 0.0


def test_row_first_partition_is_not_the_block():
    """GeLU(X1A1 + X2A2) != GeLU(X1A1) + GeLU(X2A2): the rejected row-first split is far
    from the block on random data, well beyond the 2e-2 tolerance used for parity."""
    rng = np.random.default_rng(0)
    X = rng.standard_normal((32, 64))
    W1 = rng.standard_normal((128, 64)) * 0.2
    W2 = rng.standard_normal((64, 128)) * 0.2
    right = O.mlp_forward(X, W1, W2, "gelu")["Z"]
    wrong = O.mlp_forward_row_first_wrong(X, W1, W2, "gelu", 2)
    assert np.abs(wrong - right).max() / np.abs(right).max() > 0.2
    # For the identity activation the row-first split IS exact (linearity).
    np.testing.assert_allclose(O.mlp_forward_row_first_wrong(X, W1, W2, "identity", 2),
                               O.mlp_forward(X, W1, W2, "identity")["Z"], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- brute force


def _brute_forward(X, W1, W2, act):
    """Pure-Python loops in the pages' math layout: A[k][j] = W1[j][k], B[j][i] = W2[i][j]."""
    M, h = X.shape
    n1 = W1.shape[0]
    U = [[sum(X[m][k] * W1[j][k] for k in range(h)) for j in range(n1)] for m in range(M)]
    Y = O.act_forward(np.array(U), act).tolist()
    f = len(Y[0])
    Z = [[sum(Y[m][j] * W2[i][j] for j in range(f)) for i in range(W2.shape[0])] for m in range(M)]
    return np.array(U), np.array(Y), np.array(Z)


@pytest.mark.parametrize("act", ACTS)
def test_forward_matches_brute_force_loops(act):
    rng = np.random.default_rng(1)
    M, h, f = 5, 7, 6
    n1 = 2 * f if act == "swiglu" else f
    X = rng.standard_normal((M, h))
    W1 = rng.standard_normal((n1, h))
    W2 = rng.standard_normal((h, f))
    U, Y, Z = _brute_forward(X, W1, W2, act)
    out = O.mlp_forward(X, W1, W2, act)
    np.testing.assert_allclose(out["U"], U, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(out["Y"], Y, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(out["Z"], Z, rtol=1e-12, atol=1e-12)


def test_tiny_config_matmuls_match_brute_force():
    """The tiny TP config ([16,2,64], f=256) checked entry by entry with loops on a slice."""
    from synthetic import CONFIGS, block_inputs

    cfg = CONFIGS["tiny_tp2_f32"]
    t = block_inputs(cfg)
    X = O.flatten_sbh(t["X"].double().numpy())
    W1 = t["W1"].double().numpy()
    W2 = t["W2"].double().numpy()
    out = O.mlp_forward(X, W1, W2, "gelu")
    for m in (0, 17, 31):
        for j in (0, 100, 255):
            u = sum(X[m, k] * W1[j, k] for k in range(cfg.h))
            assert abs(out["U"][m, j] - u) < 1e-12
        for i in (0, 33, 63):
            z = sum(out["Y"][m, j] * W2[i, j] for j in range(cfg.f))
            assert abs(out["Z"][m, i] - z) < 1e-12


# ---------------------------------------------------------------- gradients


@pytest.mark.parametrize("act", ACTS)
def test_backward_matches_central_finite_differences(act):
    """L = Σ Z ⊙ dZ, so ∂L/∂Z = dZ; every entry of X, W1, W2 perturbed in fp64."""
    rng = np.random.default_rng(2)
    M, h, f = 4, 5, 6
    n1 = 2 * f if act == "swiglu" else f
    X = rng.standard_normal((M, h))
    W1 = rng.standard_normal((n1, h)) * 0.7
    W2 = rng.standard_normal((h, f)) * 0.7
    dZ = rng.standard_normal((M, h))
    g = O.mlp_backward(X, W1, W2, dZ, act)

    def loss(X_, W1_, W2_):
        return float(np.sum(O.mlp_forward(X_, W1_, W2_, act)["Z"] * dZ))

    eps = 1e-6
    for name, T, grad in (("X", X, g["dX"]), ("W1", W1, g["dW1"]), ("W2", W2, g["dW2"])):
        fd = np.zeros_like(T)
        for idx in np.ndindex(*T.shape):
            Tp, Tm = T.copy(), T.copy()
            Tp[idx] += eps
            Tm[idx] -= eps
            args_p = {"X": X, "W1": W1, "W2": W2}
            args_m = dict(args_p)
            args_p[name], args_m[name] = Tp, Tm
            fd[idx] = (loss(args_p["X"], args_p["W1"], args_p["W2"])
                       - loss(args_m["X"], args_m["W1"], args_m["W2"])) / (2 * eps)
        np.testing.assert_allclose(grad, fd, rtol=2e-6, atol=2e-7, err_msg=f"{act}: d{name}")


def test_scalar_chain_rule_example():
    """L = y1·y2 with y1 = x·w1, y2 = x·w2: the column-parallel input gradient sums the
    two paths and equals the page's closed form 2·x·w1·w2."""
    for c in GOLDEN["scalar_chain_rule"]["cases"]:
        x, w1, w2 = c["x"], c["w1"], c["w2"]
        X = np.array([[x]])
        W_sh = [np.array([[w1]]), np.array([[w2]])]
        y1, y2 = (O.column_parallel_linear(X, W_sh)[i][0, 0] for i in range(2))
        dY_sh = [np.array([[y2]]), np.array([[y1]])]  # ∂L/∂y1 = y2, ∂L/∂y2 = y1
        out = O.column_parallel_linear_backward(X, W_sh, dY_sh)
        assert out["dX"][0, 0] == c["dL_dx"]


# ---------------------------------------------------------------- the pages' worked examples


def test_worked_example_column_and_row_split():
    """Y = XW, X ∈ R^{B×4}, W ∈ R^{4×8}, 2 GPUs, integer data so fp64 is exact."""
    g = GOLDEN["worked_example_shapes"]
    rng = np.random.default_rng(3)
    B = 3
    X = rng.integers(-4, 5, (B, g["in_features"])).astype(np.float64)
    W = rng.integers(-4, 5, (g["in_features"], g["out_features"])).astype(np.float64)
    full = np.array([[sum(X[m, k] * W[k, j] for k in range(4)) for j in range(8)] for m in range(B)])
    col = O.column_parallel_linear(X, [W[:, :4], W[:, 4:]])
    assert [c.shape for c in col] == [(B, 4), (B, 4)]
    assert list(W[:, :4].shape) == g["column_shard"]
    assert np.array_equal(np.concatenate(col, axis=1), full)  # concatenation, not a sum
    row = O.row_parallel_linear([X[:, :2], X[:, 2:]], [W[:2], W[2:]])
    assert list(W[:2].shape) == g["row_shard"]
    assert [r.shape for r in row] == [(B, 8), (B, 8)]  # each partial is full-size
    assert np.array_equal(row[0] + row[1], full)  # partial sums add up
    assert not np.array_equal(row[0], full)


def test_worked_two_layer_mlp_relu_sharded_equals_unsharded():
    """W1 ∈ R^{4×8} column-split, ReLU local, W2 ∈ R^{8×4} row-split; integer data."""
    t = integer_block_inputs(3, 1, 4, 8, "relu", seed=11)
    X = O.flatten_sbh(t["X"].double().numpy())
    W1 = t["W1"].double().numpy()  # storage [8, 4] = (math W1 ∈ R^{4×8})ᵀ
    W2 = t["W2"].double().numpy()  # storage [4, 8] = (math W2 ∈ R^{8×4})ᵀ
    dZ = O.flatten_sbh(t["dZ"].double().numpy())
    _, _, Zb = _brute_forward(X, W1, W2, "relu")
    sh = O.mlp_forward_sharded(X, W1, W2, "relu", 2)
    assert np.array_equal(sh["Z"], Zb)
    assert np.array_equal(sh["partials"][0] + sh["partials"][1], Zb)
    bs = O.mlp_backward_sharded(X, W1, W2, dZ, "relu", 2)
    bu = O.mlp_backward(X, W1, W2, dZ, "relu")
    for k in ("dX", "dW1", "dW2"):
        assert np.array_equal(bs[k], bu[k]), k


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("tp", [1, 2, 4])
def test_sharded_block_equals_unsharded(act, tp):
    """Z = Σ_i Y_i·B_i and dX = Σ_i dU_i·A_iᵀ equal the single-device block; weight
    gradients concatenate."""
    rng = np.random.default_rng(4)
    M, h, f = 6, 8, 8
    n1 = 2 * f if act == "swiglu" else f
    X = rng.standard_normal((M, h))
    W1 = rng.standard_normal((n1, h)) * 0.5
    W2 = rng.standard_normal((h, f)) * 0.5
    dZ = rng.standard_normal((M, h))
    fu = O.mlp_forward(X, W1, W2, act)
    fs = O.mlp_forward_sharded(X, W1, W2, act, tp)
    np.testing.assert_allclose(fs["Z"], fu["Z"], rtol=1e-12, atol=1e-12)
    bu = O.mlp_backward(X, W1, W2, dZ, act)
    bs = O.mlp_backward_sharded(X, W1, W2, dZ, act, tp)
    for k in ("dX", "dW1", "dW2"):
        np.testing.assert_allclose(bs[k], bu[k], rtol=1e-12, atol=1e-12, err_msg=k)


def test_tp1_reduces_to_two_plain_gemms():
    """tp = 1, identity activation: Z = X·W1ᵀ·W2ᵀ = X·(W2·W1)ᵀ, evaluated with einsum."""
    rng = np.random.default_rng(5)
    X = rng.standard_normal((9, 8))
    W1 = rng.standard_normal((16, 8))
    W2 = rng.standard_normal((8, 16))
    Z = O.mlp_forward_sharded(X, W1, W2, "identity", 1)["Z"]
    np.testing.assert_allclose(Z, np.einsum("mk,ik->mi", X, np.einsum("ij,jk->ik", W2, W1)),
                               rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- sequence parallelism


def test_split_gather_roundtrip_and_divisibility():
    T = np.arange(8 * 3 * 2).reshape(8, 3, 2)
    ch = O.split_dim0(T, 4)
    assert [c.shape for c in ch] == [(2, 3, 2)] * 4
    assert np.array_equal(ch[1], T[2:4])  # chunk i = rows [i·s/tp, (i+1)·s/tp)
    assert np.array_equal(O.gather_dim0(ch), T)
    with pytest.raises(ValueError, match=GOLDEN["sp_divisibility_message"]["message"]):
        O.split_dim0(T, 3)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_sp_invariant(act):
    """AG → TP block → RS equals TP block → all-reduce → split (bit-identical: the same
    sharded arithmetic), and equals the unsharded block up to fp64 rounding."""
    rng = np.random.default_rng(6)
    tp, s, b, h, f = 4, 8, 2, 8, 8
    n1 = 2 * f if act == "swiglu" else f
    X3 = rng.standard_normal((s, b, h))
    dZ3 = rng.standard_normal((s, b, h))
    W1 = rng.standard_normal((n1, h)) * 0.5
    W2 = rng.standard_normal((h, f)) * 0.5
    X, dZ = X3.reshape(s * b, h), dZ3.reshape(s * b, h)
    Xc = [c.reshape(-1, h) for c in O.split_dim0(X3, tp)]
    dZc = [c.reshape(-1, h) for c in O.split_dim0(dZ3, tp)]
    sp = O.mlp_forward_sp(Xc, W1, W2, act, tp)
    ar = O.split_dim0(O.mlp_forward_sharded(X, W1, W2, act, tp)["Z"], tp)
    for a, c in zip(sp["Z_chunks"], ar):
        assert np.array_equal(a, c)
    for a, c in zip(sp["Z_chunks"], O.split_dim0(O.mlp_forward(X, W1, W2, act)["Z"], tp)):
        np.testing.assert_allclose(a, c, rtol=1e-12, atol=1e-12)
    bsp = O.mlp_backward_sp(Xc, W1, W2, dZc, act, tp)
    bu = O.mlp_backward(X, W1, W2, dZ, act)
    for a, c in zip(bsp["dX_chunks"], O.split_dim0(bu["dX"], tp)):
        np.testing.assert_allclose(a, c, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(bsp["dW1"], bu["dW1"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(bsp["dW2"], bu["dW2"], rtol=1e-12, atol=1e-12)


def test_sizes_printed_on_the_pages():
    """Byte and parameter counts of the pages' examples, from the oracle's shard shapes."""
    for key in ("allreduce_payload_8p3b", "allreduce_payload_default"):
        g = GOLDEN[key]
        M, h, f, tp = g["b"] * g["s"], g["h"], g["f"], g["tp"]
        # the g output is one [s, b, h] tensor
        assert M * h * g["elem_bytes"] / 2**20 == g["allreduce_MiB"]
        # MLP part of the per-GPU parameters: W1 shard rows × h + W2 shard columns × h = 2hf/tp
        w1_rows = O.fc1_shard_rows(f, tp, "gelu")[0].size
        w2_cols = O.shard_ranges(f, tp)[0][1] - O.shard_ranges(f, tp)[0][0]
        mlp = w1_rows * h + h * w2_cols
        attn = 4 * h * h // tp  # QKV 3h² + output h², also split by TP
        assert mlp + attn == g["params_per_gpu_per_layer"]
    g = GOLDEN["llama70b_activation"]
    full = np.zeros((g["s"], g["b"], 1), dtype=np.int8)  # shape carrier; bytes scaled by h·e
    per_row = g["h"] * g["elem_bytes"]
    assert full.shape[0] * g["b"] * per_row / 2**20 == g["full_MiB"]
    assert O.split_dim0(full, g["tp"])[0].shape[0] * g["b"] * per_row / 2**20 == g["per_rank_MiB"]


# ---------------------------------------------------------------- fp32 shard sum, rounding


def test_shard_sum_fp32_is_fixed_order():
    big = np.float32(2**24)
    P = np.array([[big], [1.0], [-big]], dtype=np.float32)
    # ((2^24 + 1) → 2^24 by nearest-even) − 2^24 = 0 in shard order 0, 1, 2 …
    assert O.shard_sum_fp32(P)[0] == 0.0
    # … whereas a different order keeps the 1.
    assert O.shard_sum_fp32(P[[0, 2, 1]])[0] == 1.0
    # integer partials: exact, equals the fp64 sum
    rng = np.random.default_rng(7)
    Q = rng.integers(-1000, 1000, (8, 64)).astype(np.float32)
    assert np.array_equal(O.shard_sum_fp32(Q), Q.astype(np.float64).sum(0).astype(np.float32))
    # random partials: same as torch's float32 additions in the same order
    R = rng.standard_normal((8, 4096)).astype(np.float32)
    acc = torch.from_numpy(R[0]).clone()
    for i in range(1, 8):
        acc = acc + torch.from_numpy(R[i])
    assert np.array_equal(O.shard_sum_fp32(R), acc.numpy())


def test_bf16_rounding_against_torch_and_known_bits():
    vals = np.array([1.0, 1 + 2**-8, 1 + 3 * 2**-8, -2.5, 3.0e38, 1e-40, 0.0, -0.0, np.inf],
                    dtype=np.float32)
    bits = O.round_f32_to_bf16_bits(vals)
    assert bits[0] == 0x3F80 and bits[1] == 0x3F80 and bits[2] == 0x3F82
    rng = np.random.default_rng(8)
    r = np.concatenate([vals, (rng.standard_normal(100000) * 10.0 ** rng.integers(-30, 30, 100000)).astype(np.float32)])
    ref = torch.from_numpy(r).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.round_f32_to_bf16_bits(r), ref)
    assert np.array_equal(O.round_to_storage(r, "f16"), r.astype(np.float16).astype(np.float32))


# ---------------------------------------------------------------- sampled reference


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_sampled_reference_matches_full_oracle(act):
    rng = np.random.default_rng(9)
    M, h, f = 40, 24, 32
    n1 = 2 * f if act == "swiglu" else f
    X = rng.standard_normal((M, h))
    W1 = rng.standard_normal((n1, h)) * 0.3
    W2 = rng.standard_normal((h, f)) * 0.3
    dZ = rng.standard_normal((M, h))
    rows, feats = np.array([0, 7, 39]), np.array([1, 17, 31])
    s = O.sampled_reference(X, W1, W2, dZ, act, rows, feats, chunk=10)
    full = O.mlp_backward(X, W1, W2, dZ, act)
    np.testing.assert_allclose(s["Z_rows"], full["Z"][rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["dX_rows"], full["dX"][rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["dW1_rows"], full["dW1"][s["dW1_row_index"]], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["dW2_cols"], full["dW2"][:, feats], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_weight_gradients_accumulate_over_micro_batches(act):
    """Gradient accumulation (main_grad): the loss of two micro-batches is the sum of
    their losses, so dW of the concatenated batch equals the sum of the two dW."""
    rng = np.random.default_rng(12)
    h, f = 8, 12
    n1 = 2 * f if act == "swiglu" else f
    W1 = rng.standard_normal((n1, h)) * 0.5
    W2 = rng.standard_normal((h, f)) * 0.5
    X1, X2 = rng.standard_normal((5, h)), rng.standard_normal((7, h))
    dZ1, dZ2 = rng.standard_normal((5, h)), rng.standard_normal((7, h))
    g1 = O.mlp_backward(X1, W1, W2, dZ1, act)
    g2 = O.mlp_backward(X2, W1, W2, dZ2, act)
    g = O.mlp_backward(np.vstack([X1, X2]), W1, W2, np.vstack([dZ1, dZ2]), act)
    np.testing.assert_allclose(g1["dW1"] + g2["dW1"], g["dW1"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g1["dW2"] + g2["dW2"], g["dW2"], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- SP region: LayerNorm, dropout + residual


def test_layernorm_forward_closed_forms():
    rng = np.random.default_rng(13)
    X = rng.standard_normal((6, 16)) * 3 + 1.5
    out = O.layernorm_forward(X, np.ones(16), np.zeros(16), 0.0)
    # normalised rows have mean 0 and (population) variance 1
    np.testing.assert_allclose(out["Y"].mean(-1), 0, atol=1e-12)
    np.testing.assert_allclose((out["Y"] ** 2).mean(-1), 1, atol=1e-12)
    # affine part and statistics against numpy's own routines
    g, b = rng.standard_normal(16), rng.standard_normal(16)
    o2 = O.layernorm_forward(X, g, b, 1e-5)
    np.testing.assert_allclose(o2["mean"], np.mean(X, -1), rtol=1e-14)
    np.testing.assert_allclose(o2["rstd"], 1 / np.sqrt(np.var(X, -1) + 1e-5), rtol=1e-14)
    # a constant row maps to beta (x − μ = 0)
    c = O.layernorm_forward(np.full((1, 16), 7.0), g, b, 1e-5)
    np.testing.assert_allclose(c["Y"][0], b, atol=1e-12)
    # shift invariance
    np.testing.assert_allclose(O.layernorm_forward(X + 10.0, g, b, 1e-5)["Y"], o2["Y"], atol=1e-9)


def test_layernorm_backward_finite_differences():
    rng = np.random.default_rng(14)
    X = rng.standard_normal((3, 8))
    g, b = rng.standard_normal(8), rng.standard_normal(8)
    dY = rng.standard_normal((3, 8))
    eps = 1e-3
    gr = O.layernorm_backward(X, g, dY, eps)

    def loss(X_, g_, b_):
        return float(np.sum(O.layernorm_forward(X_, g_, b_, eps)["Y"] * dY))

    h = 1e-6
    for name, T, grad in (("X", X, gr["dX"]), ("g", g, gr["dgamma"]), ("b", b, gr["dbeta"])):
        fd = np.zeros_like(T)
        for idx in np.ndindex(*T.shape):
            Tp, Tm = T.copy(), T.copy()
            Tp[idx] += h
            Tm[idx] -= h
            args_p = {"X": X, "g": g, "b": b}
            args_m = dict(args_p)
            args_p[name], args_m[name] = Tp, Tm
            fd[idx] = (loss(args_p["X"], args_p["g"], args_p["b"]) - loss(args_m["X"], args_m["g"], args_m["b"])) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-7, err_msg=name)


def test_residual_dropout_closed_forms():
    R = np.array([[1.0, 2.0, 3.0, 4.0]])
    Z = np.array([[10.0, 20.0, 30.0, 40.0]])
    keep = np.array([[1, 0, 1, 0]])
    out = O.residual_dropout_forward(R, Z, keep, 0.5)
    assert np.array_equal(out, np.array([[21.0, 2.0, 63.0, 4.0]]))
    assert np.array_equal(O.residual_dropout_forward(R, Z, np.ones_like(keep), 0.0), R + Z)
    bw = O.residual_dropout_backward(np.ones((1, 4)), keep, 0.5)
    assert np.array_equal(bw["dZ"], np.array([[2.0, 0.0, 2.0, 0.0]])) and np.array_equal(bw["dR"], np.ones((1, 4)))
