"""tpmlp_forward_noalloc: the forward for callers that cannot hand the library a
device workspace (their device memory belongs to a memory manager that does not
let them allocate where they call the block, or their loop cannot afford
cudaMalloc's implicit synchronisation).  It runs on the library's built-in 64 MiB
scratch array and must give the same results as tpmlp_forward with a caller
workspace — checked here through the C ABI on two calls in a row with different
inputs, so that stale scratch contents from the first call cannot hide an error
in the second.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_common import TOL, rel_err, to_np
from synthetic import CONFIGS, BlockConfig, block_inputs

pytestmark = pytest.mark.gpu

CASES = [
    # TP+SP config, PARTIALS mode: tp fp32 partials (≈34 MB of scratch)
    (CONFIGS["tpsp4_bf16"], "partials"),
    (CONFIGS["tpsp4_bf16"], "fused"),
    # SwiGLU with SP, ragged shapes, fp16
    (BlockConfig("nz", 96, 2, 136, 288, 4, True, "f16", "swiglu"), "partials"),
    # 765-token SP chunks (not whole 128-row blocks): the forward gathers X into
    # ≈47.8 MiB of scratch, which fits, while forward and backward together
    # (X and dZ gathered) would need ≈95.6 MiB, which does not
    (BlockConfig("between", 6120, 1, 4096, 2048, 8, True, "bf16", "gelu"), "fused"),
]


def _run_reference_forward(tpmlp, cfg, mode, t):
    blk = tpmlp.MLPBlock(cfg.s, cfg.b, cfg.h, cfg.f, cfg.tp, cfg.sp, cfg.torch_dtype, cfg.act, mode)
    x = [c.contiguous() for c in t["X"].cuda().chunk(cfg.tp)] if cfg.sp else t["X"].cuda()
    W1, W2 = t["W1"].cuda(), t["W2"].cuda()
    out = blk.forward(x, W1, W2)
    return blk, x, W1, W2, out


def _cat(z, sp):
    return torch.cat(z) if sp else z


@pytest.mark.parametrize("cfg,mode", CASES, ids=[f"{c.name}-{m}" for c, m in CASES])
def test_noalloc_forward_matches_workspace_forward_twice(cuda_lib, cfg, mode):
    tpmlp = cuda_lib
    need = tpmlp.forward_workspace_size(cfg.s, cfg.b, cfg.h, cfg.f, cfg.tp, cfg.sp, cfg.torch_dtype, cfg.act, mode)
    assert need <= tpmlp.NOALLOC_SCRATCH_BYTES
    if cfg.name == "between":
        assert tpmlp.workspace_size(cfg.s, cfg.b, cfg.h, cfg.f, cfg.tp, cfg.sp, cfg.torch_dtype, cfg.act,
                                    mode) > tpmlp.NOALLOC_SCRATCH_BYTES
    for call, seed in enumerate((101, 202)):
        t = block_inputs(cfg, seed=seed)
        blk, x, W1, W2, ref = _run_reference_forward(tpmlp, cfg, mode, t)
        got = blk.alloc_forward()
        for k in ("u", "y"):
            got[k].fill_(float("nan"))
        for zz in (got["z"] if cfg.sp else [got["z"]]):
            zz.fill_(float("nan"))
        tpmlp.forward_noalloc(x, W1, W2, got["u"], got["y"], got["z"], s=cfg.s, b=cfg.b, h=cfg.h, f=cfg.f,
                              tp=cfg.tp, sp=cfg.sp, act=cfg.act, mode=mode)
        torch.cuda.synchronize()
        assert tpmlp.device_status() == 0, tpmlp.last_error()
        tol = TOL[cfg.torch_dtype]
        for k in ("u", "y"):
            e = rel_err(to_np(got[k]), to_np(ref[k]))
            assert e <= tol, (call, k, e)
        a, r = to_np(_cat(got["z"], cfg.sp)), to_np(_cat(ref["z"], cfg.sp))
        assert np.isfinite(a).all(), call
        assert rel_err(a, r) <= tol, (call, "z", rel_err(a, r))


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_lib):
    """The 22B-width TP+SP config in PARTIALS mode needs 8·4096·6144·4 bytes
    (≈0.8 GB) of scratch for its float32 partials; its SP chunks are read in
    place, so no gathered X adds to that."""
    tpmlp = cuda_lib
    cfg = CONFIGS["w22b_tpsp8_bf16"]
    need = tpmlp.forward_workspace_size(cfg.s, cfg.b, cfg.h, cfg.f, cfg.tp, cfg.sp, cfg.torch_dtype, cfg.act,
                                        "partials")
    assert need == 8 * 4096 * 6144 * 4
    assert need > tpmlp.NOALLOC_SCRATCH_BYTES
    lib = tpmlp.load()
    fake = 1 << 20  # never dereferenced: the size check fails first
    arr = (ctypes.c_void_p * cfg.tp)(*([fake] * cfg.tp))
    rc = lib.tpmlp_forward_noalloc(cfg.s, cfg.b, cfg.h, cfg.f, cfg.tp, 1, 2, 0, 0, arr, fake, fake, fake, fake, arr,
                                   None)
    assert rc == -4  # TPMLP_ERR_WORKSPACE
    msg = tpmlp.last_error()
    assert str(need) in msg and str(tpmlp.NOALLOC_SCRATCH_BYTES) in msg
