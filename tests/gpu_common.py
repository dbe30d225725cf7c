"""Helpers shared by the GPU parity tests: run the block through the C ABI and
compare with the fp64 oracle on the same dtype-rounded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O

TOL = {torch.float32: 1e-5, torch.float16: 2e-2, torch.bfloat16: 2e-2}


def rel_err(a, ref) -> float:
    """‖a − ref‖∞ / ‖ref‖∞ (per tensor)."""
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    if den == 0:
        return float(np.abs(a).max())
    return float(np.abs(a - ref).max() / den)


def to_np(t) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def chunks(t, tp):
    return [c.contiguous() for c in t.chunk(tp, 0)]


def run_block(tpmlp, inp, s, b, h, f, tp, sp, act, mode, dtype, check_status=True):
    """Forward + backward on cuda:0 through the C ABI; returns float64 arrays."""
    dev = "cuda"
    blk = tpmlp.MLPBlock(s, b, h, f, tp, sp, dtype, act, mode)
    X = inp["X"].to(dev)
    dZ = inp["dZ"].to(dev)
    W1 = inp["W1"].to(dev)
    W2 = inp["W2"].to(dev)
    x = chunks(X, tp) if sp else X
    dz = chunks(dZ, tp) if sp else dZ
    fw = blk.forward(x, W1, W2)
    ws_after_fwd = blk.workspace.clone() if mode == "partials" else None
    bw = blk.backward(x, W1, W2, fw, dz)
    torch.cuda.synchronize()
    if check_status:
        assert tpmlp.device_status() == 0, tpmlp.last_error()
    Z = torch.cat(fw["z"], 0) if sp else fw["z"]
    dX = torch.cat(bw["dx"], 0) if sp else bw["dx"]
    M = s * b
    return {
        "Z": to_np(Z).reshape(M, h),
        "dX": to_np(dX).reshape(M, h),
        "U": to_np(fw["u"]),
        "Y": to_np(fw["y"]),
        "dU": to_np(bw["du"]),
        "dW1": to_np(bw["dw1"]),
        "dW2": to_np(bw["dw2"]),
        "_raw": {"Z": Z, "dX": dX, "fw": fw, "bw": bw, "ws_after_fwd": ws_after_fwd, "blk": blk},
    }


def oracle_block(inp, act):
    X = O.flatten_sbh(to_np(inp["X"]))
    dZ = O.flatten_sbh(to_np(inp["dZ"]))
    return O.mlp_backward(X, to_np(inp["W1"]), to_np(inp["W2"]), dZ, act)


def assert_block_close(out, ref, dtype, keys=("Z", "dX", "dW1", "dW2", "U", "Y", "dU"), tol=None):
    tol = TOL[dtype] if tol is None else tol
    errs = {k: rel_err(out[k], ref[k]) for k in keys}
    bad = {k: e for k, e in errs.items() if not e <= tol}
    assert not bad, f"relative error above {tol}: {bad} (all: {errs})"
    return errs
