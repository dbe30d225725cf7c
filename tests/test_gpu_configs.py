"""Parity at the five workload configurations, in the launch configuration the
benchmark times.  The tiny and TP+SP configurations are compared element by
element against the full fp64 oracle.  At the 8.3B, 22B and Llama-70B widths the
oracle computes sampled token rows (whole rows of Z, dX, U, Y and dU) and
sampled ffn features (rows of dW1, columns of dW2) one by one.  The samples take
at least one token in every 256-row block and one feature in every 256-column
block, so every 256×256 output tile of all six GEMMs holds elements compared with
the oracle; the fused/partials cross-check then covers every element."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_common import TOL, assert_block_close, oracle_block, rel_err, run_block
from synthetic import CONFIGS, block_inputs

pytestmark = pytest.mark.gpu


def _dt(cfg):
    return cfg.torch_dtype


@pytest.mark.parametrize("mode", ["fused", "partials"])
@pytest.mark.parametrize("name", ["tiny_tp2_f32", "tpsp4_bf16"])
def test_small_configs_full_parity(cuda_lib, name, mode):
    cfg = CONFIGS[name]
    inp = block_inputs(cfg)
    out = run_block(cuda_lib, inp, cfg.s, cfg.b, cfg.h, cfg.f, cfg.tp, cfg.sp, cfg.act, mode, _dt(cfg))
    errs = assert_block_close(out, oracle_block(inp, cfg.act), _dt(cfg))
    print(name, mode, errs)


TILE = 256  # the pair GEMM's output tile is 256 × 256


def _sample_indices(n, seed, chunk=None, tile=TILE):
    """One random index inside every `tile`-wide block of [0, n), the first and
    last index, and both sides of every `chunk` boundary (SP chunks, TP shards)."""
    rng = np.random.default_rng(seed)
    idx = {int(lo + rng.integers(0, min(tile, n - lo))) for lo in range(0, n, tile)}
    idx |= {0, n - 1}
    if chunk:
        for j in range(1, n // chunk):
            idx |= {j * chunk - 1, j * chunk}
    return np.array(sorted(idx))


def test_samples_hit_every_tile():
    rows = _sample_indices(8192, 1, chunk=1024)
    assert len({r // TILE for r in rows}) == 8192 // TILE
    feats = _sample_indices(28672, 2, chunk=3584)
    assert len({f // TILE for f in feats}) == 28672 // TILE
    assert {3583, 3584, 0, 28671} <= set(feats.tolist())
    ragged = _sample_indices(300, 3)
    assert len({r // TILE for r in ragged}) == 2 and 299 in ragged


@pytest.mark.parametrize("name", ["w8p3b_tp8_f16", "w22b_tpsp8_bf16", "llama70b_swiglu_tpsp8_bf16"])
def test_large_configs_sampled_parity(cuda_lib, name):
    cfg = CONFIGS[name]
    inp = block_inputs(cfg)
    dt = _dt(cfg)
    M = cfg.M
    fused = run_block(cuda_lib, inp, cfg.s, cfg.b, cfg.h, cfg.f, cfg.tp, cfg.sp, cfg.act, "fused", dt)
    rows = _sample_indices(M, 1, chunk=M // cfg.tp)  # every 256-row block, the SP chunk boundaries
    feats = _sample_indices(cfg.f, 2, chunk=cfg.f // cfg.tp)  # every 256-column block, the TP shard boundaries
    X = inp["X"].float().numpy().reshape(M, cfg.h)
    dZ = inp["dZ"].float().numpy().reshape(M, cfg.h)
    ref = O.sampled_reference(X, inp["W1"].float().numpy(), inp["W2"].float().numpy(), dZ, cfg.act, rows, feats)
    errs = {
        "Z": rel_err(fused["Z"][rows], ref["Z_rows"]),
        "dX": rel_err(fused["dX"][rows], ref["dX_rows"]),
        "dW1": rel_err(fused["dW1"][ref["dW1_row_index"]], ref["dW1_rows"]),
        "dW2": rel_err(fused["dW2"][:, feats], ref["dW2_cols"]),
        "U": rel_err(fused["U"][rows], ref["U_rows"]),
        "Y": rel_err(fused["Y"][rows], ref["Y_rows"]),
        "dU": rel_err(fused["dU"][rows], ref["dU_rows"]),
    }
    print(name, "fused sampled", len(rows), "rows", len(feats), "features", errs)
    assert all(e <= TOL[dt] for e in errs.values()), errs
    for k in ("Z", "dX", "dW1", "dW2", "U", "Y", "dU"):
        assert np.isfinite(fused[k]).all(), k
    # PARTIALS mode on the same inputs: a different summation order of the same
    # sums, so both agree to the storage precision on every element.
    del fused["_raw"]
    torch.cuda.empty_cache()
    part = run_block(cuda_lib, inp, cfg.s, cfg.b, cfg.h, cfg.f, cfg.tp, cfg.sp, cfg.act, "partials", dt)
    for k in ("Z", "dX", "dW1", "dW2"):
        assert rel_err(part[k], fused[k]) <= TOL[dt], k
    errs_p = {
        "Z": rel_err(part["Z"][rows], ref["Z_rows"]),
        "dX": rel_err(part["dX"][rows], ref["dX_rows"]),
    }
    print(name, "partials sampled", errs_p)
    assert all(e <= TOL[dt] for e in errs_p.values()), errs_p
    # forward-only tensors and the weight gradients do not depend on the mode
    for k in ("U", "Y", "dU", "dW1", "dW2"):
        assert np.array_equal(part[k], fused[k]), k
