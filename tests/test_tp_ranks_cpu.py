"""The tensor-parallel MLP block partitioned across ranks, on the CPU (gloo).

One process per tensor shard, as the pages place them on GPUs ("Tensor
Parallelism（TP）与 Sequence Parallelism（SP）", §5 forward/backward communication
table; §4 on keeping the TP group inside one NVLink domain).  Rank i holds

* W1 rows [i·f/tp, (i+1)·f/tp) — for SwiGLU the gate rows and the matching up
  rows (the column split of A),
* W2 columns [i·f/tp, (i+1)·f/tp) (the row split of B),
* under SP, the dim-0 chunk i of X and of dZ (rows [i·s/tp, (i+1)·s/tp)).

The ranks exchange only at the f/g points:

* SP on: all-gather X on dim 0 before fc1; reduce-scatter the fc2 partials on
  dim 0 after it; in backward all-gather dZ, re-gather X for the weight
  gradient, and reduce-scatter the fc1 input-gradient partials.
* SP off: all-reduce the fc2 partials (g forward) and the fc1 input-gradient
  partials (f backward); X and dZ are replicated.

The reduce-scatter sends chunk j of every rank's partial to rank j
(all_to_all) and rank j adds them in rank order 0…tp−1: the same fixed-order
float32 sum the one-GPU library computes over its logical shards, so it can be
compared with the oracle's shard sum bit for bit.  The per-rank arithmetic is
the oracle's own (fp64), so the test pins the partitioning and the exchanges —
chunk ownership, shard ranges, the dual collectives of backward — against the
unpartitioned block, with no GPU involved.
"""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


# ---------------------------------------------------------------- collectives on dim 0


def all_gather_dim0(dist, local):
    """Concatenation of every rank's chunk along dim 0, in rank order."""
    import torch

    parts = [torch.empty_like(local) for _ in range(dist.get_world_size())]
    dist.all_gather(parts, local)
    return torch.cat(parts, 0)


def reduce_scatter_dim0_fixed_order(dist, partial):
    """Rank j receives chunk j of every rank's partial and adds them in rank
    order 0…tp−1 (float32 partials give a float32 fixed-order sum)."""
    import torch

    world = dist.get_world_size()
    rows = partial.shape[0] // world
    recv = torch.empty_like(partial)
    dist.all_to_all_single(recv, partial.contiguous())  # recv[i·rows:(i+1)·rows] = rank i's chunk j
    acc = recv[:rows].clone()
    for i in range(1, world):
        acc += recv[i * rows:(i + 1) * rows]
    return acc


def all_reduce_fixed_order(dist, partial):
    """Every rank gets the rank-ordered sum of all partials."""
    import torch

    parts = [torch.empty_like(partial) for _ in range(dist.get_world_size())]
    dist.all_gather(parts, partial.contiguous())
    acc = parts[0].clone()
    for p in parts[1:]:
        acc += p
    return acc


# ---------------------------------------------------------------- one rank's block


def _rank_block(rank, world, port, s, b, h, f, act, sp, q):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch
    import torch.distributed as dist

    import oracle as O
    from synthetic import BlockConfig, block_inputs

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = BlockConfig("ranks", s, b, h, f, world, sp, "f32", act)
        inp = block_inputs(cfg)
        X = inp["X"].double().reshape(s * b, h)
        dZ = inp["dZ"].double().reshape(s * b, h)
        W1 = inp["W1"].double()
        W2 = inp["W2"].double()
        M, ft = s * b, f // world
        rpc = M // world  # rows of one SP chunk ([s/tp, b, h] flattened)
        cols = slice(rank * ft, (rank + 1) * ft)
        # this rank's weights: the column shard of A (gate and up rows for SwiGLU), the row shard of B
        w1_rows = (torch.cat([W1[cols], W1[f + rank * ft:f + (rank + 1) * ft]]) if act == "swiglu" else W1[cols])
        w2_cols = W2[:, cols]
        x_local = X[rank * rpc:(rank + 1) * rpc] if sp else X
        dz_local = dZ[rank * rpc:(rank + 1) * rpc] if sp else dZ

        # forward: f = all-gather (SP) / identity; local fc1 + act + fc2; g = RS (SP) / AR
        Xf = all_gather_dim0(dist, x_local) if sp else x_local
        U = (Xf @ w1_rows.T).numpy()
        Y = torch.from_numpy(O.act_forward(U, act))
        P = Y @ w2_cols.T
        Z = reduce_scatter_dim0_fixed_order(dist, P) if sp else all_reduce_fixed_order(dist, P)

        # backward: g's dual = all-gather dZ (SP) / identity; f's dual = RS (SP) / AR
        dZf = all_gather_dim0(dist, dz_local) if sp else dz_local
        dY = (dZf @ w2_cols).numpy()
        dU = torch.from_numpy(O.act_backward(U, dY, act))
        dW2 = dZf.T @ Y                              # [h, f/tp]: no exchange
        Xg = all_gather_dim0(dist, x_local) if sp else x_local  # the re-gather of X for the weight gradient
        dW1 = dU.T @ Xg                              # [f/tp (2f/tp), h]: no exchange
        G = dU @ w1_rows
        dX = reduce_scatter_dim0_fixed_order(dist, G) if sp else all_reduce_fixed_order(dist, G)

        # the cross-rank float32 reduce-scatter against the oracle's fixed-order shard sum
        P32 = P.float()
        rs32 = reduce_scatter_dim0_fixed_order(dist, P32) if sp else all_reduce_fixed_order(dist, P32)
        all_p = [torch.empty_like(P32) for _ in range(world)]
        dist.all_gather(all_p, P32)
        ref32 = O.shard_sum_fp32(np.stack([p.numpy() for p in all_p]))
        ref32 = ref32[rank * rpc:(rank + 1) * rpc] if sp else ref32
        rs_bits_equal = bool(np.array_equal(rs32.numpy().view(np.uint32), ref32.astype(np.float32).view(np.uint32)))

        q.put((rank, {"Z": Z.numpy(), "dX": dX.numpy(), "dW1": dW1.numpy(), "dW2": dW2.numpy(),
                      "rs_bits_equal": rs_bits_equal, "x_rows": x_local.shape[0]}))
    finally:
        dist.destroy_process_group()


def _run(world, s, b, h, f, act, sp):
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_block, args=(r, world, port, s, b, h, f, act, sp, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    try:
        for _ in range(world):
            r, d = q.get(timeout=180)
            out[r] = d
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    return [out[r] for r in range(world)]


@pytest.mark.parametrize("world,sp,act", [(2, True, "gelu"), (2, False, "gelu"), (4, True, "swiglu"),
                                          (4, False, "gelu")])
def test_partitioned_block_across_ranks_equals_the_unpartitioned_block(world, sp, act):
    sys.path.insert(0, ROOT)
    import oracle as O
    from synthetic import BlockConfig, block_inputs

    s, b, h, f = 16, 2, 64, 128
    res = _run(world, s, b, h, f, act, sp)
    inp = block_inputs(BlockConfig("ranks", s, b, h, f, world, sp, "f32", act))
    X = inp["X"].double().numpy().reshape(s * b, h)
    dZ = inp["dZ"].double().numpy().reshape(s * b, h)
    ref = O.mlp_backward(X, inp["W1"].double().numpy(), inp["W2"].double().numpy(), dZ, act)
    M, ft = s * b, f // world
    if sp:
        # rank i owns dim-0 chunk i of Z and dX, and only that chunk of the input
        assert all(r["x_rows"] == M // world for r in res)
        Z = np.concatenate([r["Z"] for r in res])
        dX = np.concatenate([r["dX"] for r in res])
    else:
        # all-reduce: every rank holds the whole (replicated) Z and dX, bit for bit the same
        for r in res[1:]:
            assert np.array_equal(r["Z"], res[0]["Z"]) and np.array_equal(r["dX"], res[0]["dX"])
        Z, dX = res[0]["Z"], res[0]["dX"]
    # weight gradients stay sharded: W1's rows and W2's columns, no exchange
    if act == "swiglu":
        dW1 = np.concatenate([r["dW1"][:ft] for r in res] + [r["dW1"][ft:] for r in res])
    else:
        dW1 = np.concatenate([r["dW1"] for r in res])
    dW2 = np.concatenate([r["dW2"] for r in res], axis=1)
    for k, v in {"Z": Z, "dX": dX, "dW1": dW1, "dW2": dW2}.items():
        np.testing.assert_allclose(v, ref[k], rtol=1e-10, atol=1e-10, err_msg=k)
    # the cross-rank fp32 reduce-scatter / all-reduce is the oracle's fixed-order shard sum, bit for bit
    assert all(r["rs_bits_equal"] for r in res)


def test_fixed_order_sum_is_what_makes_ranks_agree_bit_for_bit():
    """Why the exchange adds in rank order: float32 addition does not associate,
    so another order of the same partials gives other bits ([2²⁴, 1, −2²⁴] sums
    to 0 in order 0, 1, 2 and to 1 in order 0, 2, 1)."""
    sys.path.insert(0, ROOT)
    import oracle as O

    p = np.array([[2.0 ** 24], [1.0], [-(2.0 ** 24)]], dtype=np.float32)
    assert O.shard_sum_fp32(p)[0] == 0.0
    assert O.shard_sum_fp32(p[[0, 2, 1]])[0] == 1.0
