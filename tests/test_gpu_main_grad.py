"""Gradient-accumulation fusion: tpmlp_backward_main_grad adds each weight-gradient
GEMM's float32 accumulator into float32 main_grad buffers.

Checks: (1) on a zeroed main_grad, one call leaves exactly the accumulator, so
rounding it to the storage type reproduces tpmlp_backward's dW bit for bit, and
dX, dU are unchanged; (2) two micro-batches accumulate to the oracle's gradient
of the concatenated batch; (3) s = 0 leaves main_grad untouched."""
import pytest
import torch

from gpu_common import TOL, chunks, oracle_block, rel_err, to_np
from synthetic import CONFIGS, BlockConfig, block_inputs

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def _setup(tpmlp, cfg, mode, t):
    blk = tpmlp.MLPBlock(cfg.s, cfg.b, cfg.h, cfg.f, cfg.tp, cfg.sp, cfg.torch_dtype, cfg.act, mode)
    X, dZ, W1, W2 = (t[k].cuda() for k in ("X", "dZ", "W1", "W2"))
    x = chunks(X, cfg.tp) if cfg.sp else X
    dz = chunks(dZ, cfg.tp) if cfg.sp else dZ
    return blk, x, dz, W1, W2


CASES = [(BlockConfig("mg", 128, 2, 256, 512, 4, True, dt, act, seed=3), mode)
         for dt in ("bf16", "f16", "f32") for act in ("gelu", "swiglu") for mode in ("fused", "partials")]
CASES.append((BlockConfig("mg-fused-ag", 256, 2, 256, 512, 4, True, "bf16", "gelu", seed=4), "fused"))


@pytest.mark.parametrize("cfg,mode", CASES, ids=[f"{c.name}-{c.dtype}-{c.act}-{m}" for c, m in CASES])
def test_main_grad_first_call_equals_the_accumulator(cuda_lib, cfg, mode):
    tpmlp = cuda_lib
    t = block_inputs(cfg)
    blk, x, dz, W1, W2 = _setup(tpmlp, cfg, mode, t)
    fw = blk.forward(x, W1, W2)
    ref = blk.backward(x, W1, W2, fw, dz)
    mg1 = torch.zeros(blk.n1, cfg.h, dtype=torch.float32, device="cuda")
    mg2 = torch.zeros(cfg.h, cfg.f, dtype=torch.float32, device="cuda")
    got = blk.backward_main_grad(x, W1, W2, fw, dz, mg1, mg2)
    torch.cuda.synchronize()
    assert tpmlp.device_status() == 0, tpmlp.last_error()
    assert torch.equal(mg1.to(cfg.torch_dtype), ref["dw1"])
    assert torch.equal(mg2.to(cfg.torch_dtype), ref["dw2"])
    assert torch.equal(got["du"], ref["du"])
    gx = torch.cat(got["dx"]) if cfg.sp else got["dx"]
    rx = torch.cat(ref["dx"]) if cfg.sp else ref["dx"]
    assert torch.equal(gx, rx)


@pytest.mark.parametrize("name", ["tpsp4_bf16", "tiny_tp2_f32"])
def test_main_grad_accumulates_micro_batches(cuda_lib, name):
    tpmlp = cuda_lib
    cfg = CONFIGS[name]
    mode = "fused"
    t1 = block_inputs(cfg, seed=21)
    t2 = block_inputs(cfg, seed=22)
    t2["W1"], t2["W2"] = t1["W1"], t1["W2"]  # same layer, two micro-batches
    n1 = cfg.fc1_rows
    mg1 = torch.zeros(n1, cfg.h, dtype=torch.float32, device="cuda")
    mg2 = torch.zeros(cfg.h, cfg.f, dtype=torch.float32, device="cuda")
    for t in (t1, t2):
        blk, x, dz, W1, W2 = _setup(tpmlp, cfg, mode, t)
        fw = blk.forward(x, W1, W2)
        blk.backward_main_grad(x, W1, W2, fw, dz, mg1, mg2)
    torch.cuda.synchronize()
    assert tpmlp.device_status() == 0, tpmlp.last_error()
    r1, r2 = oracle_block(t1, cfg.act), oracle_block(t2, cfg.act)
    tol = TOL[cfg.torch_dtype]
    assert rel_err(to_np(mg1), r1["dW1"] + r2["dW1"]) <= tol
    assert rel_err(to_np(mg2), r1["dW2"] + r2["dW2"]) <= tol


def test_main_grad_untouched_for_an_empty_sequence(cuda_lib):
    tpmlp = cuda_lib
    h, f, tp = 64, 128, 2
    d = torch.bfloat16
    dummy = torch.zeros(64, dtype=d, device="cuda")
    W1 = torch.randn(f, h, device="cuda").to(d)
    W2 = torch.randn(h, f, device="cuda").to(d)
    mg1 = torch.randn(f, h, device="cuda")
    mg2 = torch.randn(h, f, device="cuda")
    keep1, keep2 = mg1.clone(), mg2.clone()
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    tpmlp.backward_main_grad([dummy, dummy], W1, W2, dummy, dummy, [dummy, dummy], [dummy, dummy], mg1, mg2, dummy,
                             s=0, b=1, h=h, f=f, tp=tp, sp=True, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(mg1, keep1) and torch.equal(mg2, keep2)
