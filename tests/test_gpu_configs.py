"""Parity at the five workload configurations, in the launch configuration the
benchmark times.  The tiny and TP+SP configurations are compared element by
element against the full fp64 oracle; at the 8.3B, 22B and Llama-70B widths the
oracle computes sampled token rows (Z, dX) and sampled ffn features (rows of
dW1, columns of dW2) one by one, plus the fused/partials cross-check on every
element."""
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


def _sample_indices(n, k, seed, chunk=None):
    rng = np.random.default_rng(seed)
    idx = set(rng.choice(n, size=min(k, n), replace=False).tolist())
    idx |= {0, n - 1}
    if chunk:
        for j in range(1, n // chunk):
            idx |= {j * chunk - 1, j * chunk}
    return np.array(sorted(idx))


@pytest.mark.parametrize("name", ["w8p3b_tp8_f16", "w22b_tpsp8_bf16", "llama70b_swiglu_tpsp8_bf16"])
def test_large_configs_sampled_parity(cuda_lib, name):
    cfg = CONFIGS[name]
    inp = block_inputs(cfg)
    dt = _dt(cfg)
    M = cfg.M
    fused = run_block(cuda_lib, inp, cfg.s, cfg.b, cfg.h, cfg.f, cfg.tp, cfg.sp, cfg.act, "fused", dt)
    rows = _sample_indices(M, 12, 1, chunk=M // cfg.tp)  # includes the SP chunk boundaries
    feats = _sample_indices(cfg.f, 12, 2, chunk=cfg.f // cfg.tp)  # includes the TP shard boundaries
    X = inp["X"].float().numpy().reshape(M, cfg.h)
    dZ = inp["dZ"].float().numpy().reshape(M, cfg.h)
    ref = O.sampled_reference(X, inp["W1"].float().numpy(), inp["W2"].float().numpy(), dZ, cfg.act, rows, feats)
    errs = {
        "Z": rel_err(fused["Z"][rows], ref["Z_rows"]),
        "dX": rel_err(fused["dX"][rows], ref["dX_rows"]),
        "dW1": rel_err(fused["dW1"][ref["dW1_row_index"]], ref["dW1_rows"]),
        "dW2": rel_err(fused["dW2"][:, feats], ref["dW2_cols"]),
    }
    print(name, "fused sampled", errs)
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
