"""fp64 CPU oracle of the Megatron tensor-parallel MLP block, with sequence parallelism.

TEST INFRASTRUCTURE ONLY — used by ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py``; never by the product path.

What the block computes (math convention of the pages, A ∈ R^{h×f}, B ∈ R^{f×h}):

    Z = act(X·A)·B                      ("Tensor Parallelism（TP）与 Sequence
                                         Parallelism（SP）", §2 column-parallel 与
                                         row-parallel 的配合)

Storage follows torch's ``[out, in]`` weight convention ("tensor-parallelism-
matrix-split", §一个 Linear，两种拆法, note on nn.Linear; "tensor-parallel-megatron"
reading, MLP section: column shard [4h/TP, h], row shard [h, 4h/TP]):
``W1 = Aᵀ`` is ``[f, h]`` and ``W2 = Bᵀ`` is ``[h, f]``.  Activations ``[s, b, h]``
are flattened to ``[M, h]`` with row ``m = s_idx * b + b_idx`` (sequence-first
layout, "Tensor Parallelism（TP）与 Sequence Parallelism（SP）", §1); the block is
token-wise, so the flattening does not change any value.

Readings taken where the pages are silent (each listed in the design notes):

1. GeLU is the tanh form 0.5·x·(1 + tanh(√(2/π)(x + 0.044715x³))) (Hendrycks &
   Gimpel 2016); its derivative is taken analytically.  The pages name GeLU but
   print no formula.
2. SwiGLU: fc1 has 2F outputs, rows [0, F) are the gate and rows [F, 2F) the up
   projection; Y = silu(G) ⊙ Up with silu(x) = x·σ(x).  Tensor shard i owns gate
   rows [i·F/tp, (i+1)·F/tp) and the matching up rows, so the product stays local.
3. No bias, no dropout, no LayerNorm inside the block.
4. The shard sums of g (forward all-reduce / reduce-scatter) and of f's backward
   run in fixed shard order i = 0 … tp−1 in float32, then round to the storage
   type (round-to-nearest-even).  ``shard_sum_fp32`` is that definition.
5. Chunk i of a sequence-parallel split is rows [i·s/tp, (i+1)·s/tp) of dim 0.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "GELU_C",
    "GELU_K",
    "gelu_tanh",
    "gelu_tanh_grad",
    "silu",
    "silu_grad",
    "relu",
    "relu_grad",
    "act_forward",
    "act_backward",
    "flatten_sbh",
    "mlp_forward",
    "mlp_backward",
    "shard_ranges",
    "fc1_shard_rows",
    "column_parallel_linear",
    "row_parallel_linear",
    "column_parallel_linear_backward",
    "row_parallel_linear_backward",
    "mlp_forward_sharded",
    "mlp_backward_sharded",
    "mlp_forward_row_first_wrong",
    "split_dim0",
    "gather_dim0",
    "all_reduce",
    "reduce_scatter_dim0",
    "mlp_forward_sp",
    "mlp_backward_sp",
    "shard_sum_fp32",
    "round_f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "round_to_storage",
    "sampled_reference",
    "layernorm_forward",
    "layernorm_backward",
    "residual_dropout_forward",
    "residual_dropout_backward",
]

# --------------------------------------------------------------------------
# Activations (element-wise, hence local per tensor shard: "Tensor Parallelism
# （TP）与 Sequence Parallelism（SP）", §2; "tensor-parallelism-matrix-split",
# §Forward：Column + Row — ReLU is element-wise so each GPU applies it locally).
# --------------------------------------------------------------------------

GELU_C = math.sqrt(2.0 / math.pi)
GELU_K = 0.044715


def gelu_tanh(x):
    """tanh-form GeLU (reading 1)."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(GELU_C * (x + GELU_K * x**3)))


def gelu_tanh_grad(x):
    """d/dx of ``gelu_tanh``: 0.5(1+t) + 0.5·x·(1−t²)·c·(1 + 3k·x²), t = tanh(c(x + k·x³))."""
    x = np.asarray(x, dtype=np.float64)
    t = np.tanh(GELU_C * (x + GELU_K * x**3))
    return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * GELU_C * (1.0 + 3.0 * GELU_K * x * x)


def _sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    pos = x >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-x[pos]))
    ex = np.exp(x[~pos])
    out[~pos] = ex / (1.0 + ex)
    return out


def silu(x):
    """silu(x) = x·σ(x) (reading 2)."""
    x = np.asarray(x, dtype=np.float64)
    return x * _sigmoid(x)


def silu_grad(x):
    """d/dx silu = σ(x)·(1 + x·(1 − σ(x)))."""
    x = np.asarray(x, dtype=np.float64)
    s = _sigmoid(x)
    return s * (1.0 + x * (1.0 - s))


def relu(x):
    """ReLU of the pages' two-layer example ("tensor-parallelism-matrix-split", §两层之间的通信能不能省掉)."""
    x = np.asarray(x, dtype=np.float64)
    return np.where(x > 0, x, 0.0)


def relu_grad(x):
    """ReLU backward is the element-wise mask x > 0 (same page, §Backward 的通信)."""
    x = np.asarray(x, dtype=np.float64)
    return (x > 0).astype(np.float64)


def act_forward(U, act):
    """Y = act(U).  For SwiGLU, U = [G | Up] along the last axis (reading 2)."""
    U = np.asarray(U, dtype=np.float64)
    if act == "gelu":
        return gelu_tanh(U)
    if act == "relu":
        return relu(U)
    if act == "identity":
        return U.copy()
    if act == "swiglu":
        F = U.shape[-1] // 2
        G, Up = U[..., :F], U[..., F:]
        return silu(G) * Up
    raise ValueError(f"unknown activation {act!r}")


def act_backward(U, dY, act):
    """dU from dY through the activation, element-wise (local per shard)."""
    U = np.asarray(U, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    if act == "gelu":
        return dY * gelu_tanh_grad(U)
    if act == "relu":
        return dY * relu_grad(U)
    if act == "identity":
        return dY.copy()
    if act == "swiglu":
        F = U.shape[-1] // 2
        G, Up = U[..., :F], U[..., F:]
        dG = dY * Up * silu_grad(G)
        dUp = dY * silu(G)
        return np.concatenate([dG, dUp], axis=-1)
    raise ValueError(f"unknown activation {act!r}")


# --------------------------------------------------------------------------
# The unpartitioned block: the plain definition the partitioned method reaches
# exactly ("tensor-parallelism-matrix-split", §Column Parallel / §Row Parallel:
# concatenation and partial sums restore the single-device product).
# --------------------------------------------------------------------------


def flatten_sbh(T):
    """[s, b, h] → [s·b, h], row m = s_idx·b + b_idx (a view for contiguous input)."""
    T = np.asarray(T, dtype=np.float64)
    return T.reshape(-1, T.shape[-1])


def mlp_forward(X, W1, W2, act="gelu"):
    """U = X·A = X·W1ᵀ, Y = act(U), Z = Y·B = Y·W2ᵀ.  X is [M, h]."""
    X = np.asarray(X, dtype=np.float64)
    W1 = np.asarray(W1, dtype=np.float64)
    W2 = np.asarray(W2, dtype=np.float64)
    U = X @ W1.T
    Y = act_forward(U, act)
    Z = Y @ W2.T
    return {"U": U, "Y": Y, "Z": Z}


def mlp_backward(X, W1, W2, dZ, act="gelu"):
    """Gradients of the block given dZ = ∂L/∂Z.

    With Y = XW: dW = Xᵀ·dY and dX = dY·Wᵀ ("tensor-parallelism-matrix-split",
    §Backward：为什么有些梯度需要求和 / 两种梯度), applied to both layers:
        dB = Yᵀ·dZ  (stored dW2 = dBᵀ = dZᵀ·Y,  [h, f])
        dY = dZ·Bᵀ = dZ·W2
        dU = act'(U) ⊙ dY
        dA = Xᵀ·dU  (stored dW1 = dAᵀ = dUᵀ·X,  [f, h])
        dX = dU·Aᵀ = dU·W1
    """
    X = np.asarray(X, dtype=np.float64)
    W1 = np.asarray(W1, dtype=np.float64)
    W2 = np.asarray(W2, dtype=np.float64)
    dZ = np.asarray(dZ, dtype=np.float64)
    fw = mlp_forward(X, W1, W2, act)
    U, Y = fw["U"], fw["Y"]
    dW2 = dZ.T @ Y
    dY = dZ @ W2
    dU = act_backward(U, dY, act)
    dW1 = dU.T @ X
    dX = dU @ W1
    return {"U": U, "Y": Y, "Z": fw["Z"], "dY": dY, "dU": dU, "dW1": dW1, "dW2": dW2, "dX": dX}


# --------------------------------------------------------------------------
# Tensor-parallel (sharded) formulation, used for the invariants only.
# --------------------------------------------------------------------------


def shard_ranges(n, tp):
    """tp equal contiguous ranges of [0, n); n must be divisible by tp
    ("tensor-parallel-megatron" reading, constraints: divide()/ensure_divisibility)."""
    if tp <= 0 or n % tp != 0:
        raise ValueError(f"{n} is not divisible by tp={tp}")
    w = n // tp
    return [(i * w, (i + 1) * w) for i in range(tp)]


def fc1_shard_rows(f, tp, act):
    """Row indices of W1 owned by shard i: a column block of A (reading 2 for SwiGLU)."""
    out = []
    for lo, hi in shard_ranges(f, tp):
        if act == "swiglu":
            out.append(np.concatenate([np.arange(lo, hi), f + np.arange(lo, hi)]))
        else:
            out.append(np.arange(lo, hi))
    return out


def column_parallel_linear(X, W_col_shards):
    """Y = X·[W_0 | W_1 | …] = [X·W_0 | X·W_1 | …] (math layout W ∈ R^{in×out};
    "tensor-parallelism-matrix-split", §Column Parallel).  Returns the shard outputs."""
    X = np.asarray(X, dtype=np.float64)
    return [X @ np.asarray(W, dtype=np.float64) for W in W_col_shards]


def row_parallel_linear(X_col_shards, W_row_shards):
    """Y = Σ_i X_i·W_i for W = [W_0; W_1; …], X = [X_0 | X_1 | …]
    (same page, §Row Parallel).  Returns the per-shard partial sums."""
    return [np.asarray(Xi, dtype=np.float64) @ np.asarray(Wi, dtype=np.float64)
            for Xi, Wi in zip(X_col_shards, W_row_shards)]


def column_parallel_linear_backward(X, W_col_shards, dY_shards):
    """Column-parallel backward: dW_i = Xᵀ·dY_i (local) and dX = Σ_i dY_i·W_iᵀ — the
    sum over shards comes from the multivariable chain rule, because X feeds every
    shard ("tensor-parallelism-matrix-split", §从多变量链式法则看为什么要求和)."""
    X = np.asarray(X, dtype=np.float64)
    dW = [X.T @ np.asarray(dYi, dtype=np.float64) for dYi in dY_shards]
    contribs = [np.asarray(dYi, dtype=np.float64) @ np.asarray(Wi, dtype=np.float64).T
                for dYi, Wi in zip(dY_shards, W_col_shards)]
    dX = contribs[0].copy()
    for c in contribs[1:]:
        dX = dX + c
    return {"dX": dX, "dX_contribs": contribs, "dW": dW}


def row_parallel_linear_backward(X_col_shards, W_row_shards, dY):
    """Row-parallel backward: dX_i = dY·W_iᵀ and dW_i = X_iᵀ·dY, both local — no sum
    (same page, §Row Parallel 的 backward)."""
    dY = np.asarray(dY, dtype=np.float64)
    dX = [dY @ np.asarray(Wi, dtype=np.float64).T for Wi in W_row_shards]
    dW = [np.asarray(Xi, dtype=np.float64).T @ dY for Xi in X_col_shards]
    return {"dX": dX, "dW": dW}


def mlp_forward_sharded(X, W1, W2, act, tp):
    """Column → act → row with tp shards: Y_i = act(X·A_i) locally, then g sums the
    partials Z = Σ_i Y_i·B_i ("Tensor Parallelism（TP）与 Sequence Parallelism（SP）",
    §2 and its f/g table; "tensor-parallelism-matrix-split", §Forward：Column + Row)."""
    X = np.asarray(X, dtype=np.float64)
    W1 = np.asarray(W1, dtype=np.float64)
    W2 = np.asarray(W2, dtype=np.float64)
    f = W2.shape[1]
    rows = fc1_shard_rows(f, tp, act)
    U_sh, Y_sh, P_sh = [], [], []
    for i, (lo, hi) in enumerate(shard_ranges(f, tp)):
        Ui = X @ W1[rows[i]].T
        Yi = act_forward(Ui, act)
        Pi = Yi @ W2[:, lo:hi].T
        U_sh.append(Ui)
        Y_sh.append(Yi)
        P_sh.append(Pi)
    return {"U": U_sh, "Y": Y_sh, "partials": P_sh, "Z": all_reduce(P_sh)}


def mlp_backward_sharded(X, W1, W2, dZ, act, tp):
    """Backward of the sharded block.  g's backward is identity (every shard sees the
    full dZ); f's backward sums the input-gradient contributions of the shards:
    dX = Σ_i dU_i·A_iᵀ; weight gradients stay local and concatenate
    ("Tensor Parallelism（TP）与 Sequence Parallelism（SP）", §5 table;
    "tensor-parallelism-matrix-split", §Backward 的通信)."""
    X = np.asarray(X, dtype=np.float64)
    W1 = np.asarray(W1, dtype=np.float64)
    W2 = np.asarray(W2, dtype=np.float64)
    dZ = np.asarray(dZ, dtype=np.float64)
    f = W2.shape[1]
    rows = fc1_shard_rows(f, tp, act)
    G_sh, dW1_sh, dW2_sh = [], [], []
    for i, (lo, hi) in enumerate(shard_ranges(f, tp)):
        Ui = X @ W1[rows[i]].T
        Yi = act_forward(Ui, act)
        dW2_sh.append(dZ.T @ Yi)
        dYi = dZ @ W2[:, lo:hi]
        dUi = act_backward(Ui, dYi, act)
        dW1_sh.append(dUi.T @ X)
        G_sh.append(dUi @ W1[rows[i]])
    dW1 = np.zeros_like(W1)
    for i in range(tp):
        dW1[rows[i]] = dW1_sh[i]
    return {"dX_partials": G_sh, "dX": all_reduce(G_sh), "dW1": dW1,
            "dW2": np.concatenate(dW2_sh, axis=1)}


def mlp_forward_row_first_wrong(X, W1, W2, act, tp):
    """The partition the pages reject: split A by rows (X by columns), apply the
    activation to each partial sum, then sum — act(X₁A₁ + X₂A₂) ≠ Σ act(XᵢAᵢ)
    ("tensor-parallelism-matrix-split", §为什么不反过来 Row + Column; "tensor-parallel-
    megatron" reading, GeLU non-additivity).  Used only to show it differs."""
    X = np.asarray(X, dtype=np.float64)
    W1 = np.asarray(W1, dtype=np.float64)
    W2 = np.asarray(W2, dtype=np.float64)
    h = X.shape[1]
    Y = 0.0
    for lo, hi in shard_ranges(h, tp):
        Y = Y + act_forward(X[:, lo:hi] @ W1[:, lo:hi].T, act)
    return Y @ W2.T


# --------------------------------------------------------------------------
# Sequence parallelism: split / gather / reduce-scatter along dim 0
# ("Tensor Parallelism（TP）与 Sequence Parallelism（SP）", §1 `s` 在前的设计 and
# `s` 需被 TP 整除; "Sequence Parallel 与 Context Parallel", §SP：all-gather 进、
# reduce-scatter 出).
# --------------------------------------------------------------------------


def split_dim0(T, tp):
    """Chunk i = rows [i·n/tp, (i+1)·n/tp) of dim 0 (reading 5); n % tp != 0 is an error."""
    T = np.asarray(T)
    n = T.shape[0]
    if tp <= 0 or n % tp != 0:
        raise ValueError("First dimension of the tensor should be divisible by tensor parallel size")
    w = n // tp
    return [T[i * w:(i + 1) * w].copy() for i in range(tp)]


def gather_dim0(chunks):
    """All-gather along dim 0 = concatenation of the chunks in rank order."""
    return np.concatenate([np.asarray(c) for c in chunks], axis=0)


def all_reduce(partials):
    """Sum of the tp partials, in shard order 0 … tp−1 (fp64 here)."""
    out = np.array(partials[0], dtype=np.float64, copy=True)
    for p in partials[1:]:
        out = out + np.asarray(p, dtype=np.float64)
    return out


def reduce_scatter_dim0(partials, tp):
    """Reduce-scatter along dim 0: sum the partials, then rank i keeps chunk i."""
    return split_dim0(all_reduce(partials), tp)


def mlp_forward_sp(X_chunks, W1, W2, act, tp):
    """SP forward: AG(dim 0) → sharded block → RS(dim 0) ("Sequence Parallel 与 Context
    Parallel", §SP：all-gather 进、reduce-scatter 出).  X_chunks are [s/tp·b, h]."""
    X = gather_dim0(X_chunks)
    sh = mlp_forward_sharded(X, W1, W2, act, tp)
    return {"U": sh["U"], "Y": sh["Y"], "Z_chunks": reduce_scatter_dim0(sh["partials"], tp)}


def mlp_backward_sp(X_chunks, W1, W2, dZ_chunks, act, tp):
    """SP backward: the RS's backward all-gathers dZ, the input is re-gathered for the
    weight gradients (forward kept only local chunks), and the AG's backward
    reduce-scatters the input-gradient partials (same page and section)."""
    X = gather_dim0(X_chunks)
    dZ = gather_dim0(dZ_chunks)
    sh = mlp_backward_sharded(X, W1, W2, dZ, act, tp)
    return {"dX_chunks": reduce_scatter_dim0(sh["dX_partials"], tp),
            "dW1": sh["dW1"], "dW2": sh["dW2"]}


# --------------------------------------------------------------------------
# float32 fixed-order shard sum and rounding to the storage type (reading 4).
# --------------------------------------------------------------------------


def shard_sum_fp32(partials):
    """acc = P_0; acc = fl32(acc + P_i) for i = 1 … tp−1 (IEEE float32, nearest-even)."""
    P = np.asarray(partials, dtype=np.float32)
    acc = P[0].copy()
    for i in range(1, P.shape[0]):
        acc = np.add(acc, P[i], dtype=np.float32)
    return acc


def round_f32_to_bf16_bits(x):
    """IEEE round-to-nearest-even of float32 to bfloat16 (the top 16 bits), as uint16.

    bfloat16 keeps the sign, the 8 exponent bits and the top 7 fraction bits of a
    float32.  Rounding adds half an ulp minus one (0x7FFF) plus the lowest kept bit
    (ties go to even) and truncates; a carry into the exponent is the correct
    round-up.  NaN maps to the canonical quiet NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) & np.uint64(0xFFFF)
    r = r.astype(np.uint16)
    r[np.isnan(x)] = np.uint16(0x7FC0)
    return r


def bf16_bits_to_f32(bits):
    """Exact widening of bfloat16 bit patterns to float32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def round_to_storage(x_f32, dtype):
    """float32 → storage dtype with round-to-nearest-even, returned widened to float32."""
    x = np.asarray(x_f32, dtype=np.float32)
    if dtype == "f32":
        return x.copy()
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float32)
    if dtype == "bf16":
        return bf16_bits_to_f32(round_f32_to_bf16_bits(x))
    raise ValueError(dtype)


# --------------------------------------------------------------------------
# Sampled reference at full size: the same plain definition restricted to a few
# token rows (Z, dX) and a few ffn features (dW1 rows, dW2 columns).
# --------------------------------------------------------------------------


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def sampled_reference(X, W1, W2, dZ, act, rows, feats, chunk=4096):
    """Z[rows], dX[rows], U[rows], Y[rows], dU[rows], dW1[feature rows] and
    dW2[:, feats] of ``mlp_backward``.

    X, dZ: [M, h]; W1: [fc1_rows, h]; W2: [h, f]; any float dtype (converted to
    fp64 slice by slice).  ``feats`` index the ffn width f (F for SwiGLU; the
    returned dW1 rows are then the gate rows feats and the up rows F + feats).
    """
    rows = np.asarray(rows, dtype=np.int64)
    feats = np.asarray(feats, dtype=np.int64)
    f = W2.shape[1]
    Xr = _f64(X[rows])
    dZr = _f64(dZ[rows])
    nrow = W1.shape[0]
    # U[rows] = X[rows]·W1ᵀ, chunked over W1's rows to bound the fp64 working set.
    Ur = np.empty((rows.size, nrow))
    for lo in range(0, nrow, chunk):
        Ur[:, lo:lo + chunk] = Xr @ _f64(W1[lo:lo + chunk]).T
    Yr = act_forward(Ur, act)
    Zr = np.zeros((rows.size, W2.shape[0]))
    dYr = np.empty((rows.size, f))
    for lo in range(0, f, chunk):
        W2c = _f64(W2[:, lo:lo + chunk])
        Zr += Yr[:, lo:lo + chunk] @ W2c.T
        dYr[:, lo:lo + chunk] = dZr @ W2c
    dUr = act_backward(Ur, dYr, act)
    dXr = np.zeros((rows.size, X.shape[1]))
    for lo in range(0, nrow, chunk):
        dXr += dUr[:, lo:lo + chunk] @ _f64(W1[lo:lo + chunk])
    # Feature columns need every token: U[:, j] = X·W1[j], dY[:, j] = dZ·W2[:, j].
    Xf = _f64(X)
    dZf = _f64(dZ)
    if act == "swiglu":
        w1_rows = np.concatenate([feats, f + feats])
    else:
        w1_rows = feats
    Uc = Xf @ _f64(W1[w1_rows]).T
    Yc = act_forward(Uc, act)
    dYc = dZf @ _f64(W2[:, feats])
    dUc = act_backward(Uc, dYc, act)
    dW1_rows = dUc.T @ Xf
    dW2_cols = dZf.T @ Yc
    return {"Z_rows": Zr, "dX_rows": dXr, "U_rows": Ur, "Y_rows": Yr, "dU_rows": dUr,
            "dW1_rows": dW1_rows, "dW1_row_index": w1_rows, "dW2_cols": dW2_cols}


# --------------------------------------------------------------------------
# Sequence-parallel region around the block ("Sequence Parallel 与 Context
# Parallel", §SP：all-gather 进、reduce-scatter 出: LayerNorm and dropout run on the
# sequence chunks [s/tp, b, h]; "tensor-parallel-megatron" reading, SP section:
# LayerNorm, dropout and the residual are split along the sequence).  All of it
# is token-wise, so the oracle works on full [M, h] tensors; chunking does not
# change a value.  Reading: the LayerNorm is the standard one over h with affine
# gamma, beta and variance without Bessel's correction; dropout scales kept
# values by 1/(1-p) ("inverted" dropout) and its keep-mask is an input.
# --------------------------------------------------------------------------


def layernorm_forward(X, gamma, beta, eps):
    """y = (x − μ)/√(σ² + eps)·γ + β per row, μ and σ² over the last axis."""
    X = np.asarray(X, dtype=np.float64)
    mu = X.mean(axis=-1, keepdims=True)
    var = ((X - mu) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (X - mu) * rstd
    return {"Y": xhat * np.asarray(gamma, dtype=np.float64) + np.asarray(beta, dtype=np.float64),
            "mean": mu[..., 0], "rstd": rstd[..., 0]}


def layernorm_backward(X, gamma, dY, eps):
    """Gradients of layernorm_forward: dX, dγ = Σ_rows dY·x̂, dβ = Σ_rows dY.

    dX = rstd·(g − mean(g) − x̂·mean(g·x̂)) with g = dY·γ (the gradient through the
    mean and the variance written out)."""
    X = np.asarray(X, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    gamma = np.asarray(gamma, dtype=np.float64)
    fw = layernorm_forward(X, gamma, np.zeros_like(gamma), eps)
    rstd = fw["rstd"][..., None]
    xhat = (X - fw["mean"][..., None]) * rstd
    g = dY * gamma
    dX = rstd * (g - g.mean(axis=-1, keepdims=True) - xhat * (g * xhat).mean(axis=-1, keepdims=True))
    rows = dY.reshape(-1, dY.shape[-1])
    return {"dX": dX, "dgamma": (rows * xhat.reshape(rows.shape)).sum(axis=0), "dbeta": rows.sum(axis=0)}


def residual_dropout_forward(R, Z, keep, p):
    """out = R + keep·Z/(1 − p); keep ∈ {0, 1} is drawn by the caller."""
    return np.asarray(R, dtype=np.float64) + np.asarray(keep, dtype=np.float64) * np.asarray(Z, dtype=np.float64) / (1.0 - p)


def residual_dropout_backward(dOut, keep, p):
    """dR = dOut (identity branch), dZ = keep·dOut/(1 − p)."""
    dOut = np.asarray(dOut, dtype=np.float64)
    return {"dR": dOut.copy(), "dZ": np.asarray(keep, dtype=np.float64) * dOut / (1.0 - p)}
