"""The sequence-parallel region around the block on the GPU, against the fp64
oracle: LayerNorm forward/backward on the [s/tp, b, h] chunks, dropout +
residual, and the whole MLP sublayer R → LayerNorm → block → dropout + residual
(forward and backward) with the LayerNorm's output chunks fed to the block as
its SP input chunks (fc1 reads them in place)."""
import pytest
import torch

import oracle as O
from gpu_common import TOL, chunks, rel_err, to_np
from synthetic import BlockConfig, block_inputs, sp_region_inputs

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
EPS = 1e-5


def _flat(t):
    return to_np(t).reshape(-1, t.shape[-1])


# Shapes: warp-per-row kernels (h < 1024, or rows not a whole number of
# 8-element vectors) and the streamed kernels (h >= 1024) with 1..4 vectors per
# thread, a ragged last vector column (h = 2056: 257 vectors), fewer rows than
# CTAs, and the widest ring (h = 8192); the 16-bit forward's two-warps-per-row
# kernel with 8, 10 (predicated), 12 and 16 vectors a lane (h = 4096, 5120,
# 6144, 8192).
LN_SHAPES = [(64, 2, 136, 2), (9, 1, 5, 3), (512, 4, 1024, 4), (16, 2, 64, 1), (24, 1, 64, 2),
             (40, 2, 2056, 4), (48, 1, 6144, 2), (9, 1, 1032, 3), (24, 1, 8192, 3), (6, 1, 1030, 3),
             (32, 2, 4096, 2), (24, 1, 5120, 4)]


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("s,b,h,tp", LN_SHAPES)
def test_layernorm_forward_and_backward(cuda_lib, dt, s, b, h, tp):
    tpmlp = cuda_lib
    inp = sp_region_inputs(s, b, h, 0.1, seed=s + h, dtype=dt)
    R = inp["R"].cuda()
    gamma, beta = inp["gamma"].cuda(), inp["beta"].cuda()
    dY = inp["dOut"].cuda()
    x = chunks(R, tp)
    y = [torch.full_like(c, float("nan")) for c in x]
    mean = torch.empty(s * b, device="cuda")
    rstd = torch.empty(s * b, device="cuda")
    tpmlp.sp_layernorm_forward(x, gamma, beta, EPS, y, mean, rstd, s=s, b=b, h=h, tp=tp)
    ref = O.layernorm_forward(_flat(inp["R"]), to_np(inp["gamma"]), to_np(inp["beta"]), EPS)
    tol = TOL[DT[dt]]
    assert rel_err(_flat(torch.cat(y)), ref["Y"]) <= tol
    assert rel_err(to_np(mean), ref["mean"]) <= 1e-5
    assert rel_err(to_np(rstd), ref["rstd"]) <= 1e-5
    # backward, written and accumulated
    dy = chunks(dY, tp)
    dx = [torch.full_like(c, float("nan")) for c in x]
    dg = torch.empty(h, device="cuda")
    db = torch.empty(h, device="cuda")
    tpmlp.sp_layernorm_backward(x, gamma, mean, rstd, dy, dx, dg, db, s=s, b=b, h=h, tp=tp)
    rb = O.layernorm_backward(_flat(inp["R"]), to_np(inp["gamma"]), _flat(inp["dOut"]), EPS)
    assert rel_err(_flat(torch.cat(dx)), rb["dX"]) <= tol
    assert rel_err(to_np(dg), rb["dgamma"]) <= tol
    assert rel_err(to_np(db), rb["dbeta"]) <= tol
    base = [torch.ones_like(c) for c in x]
    tpmlp.sp_layernorm_backward(x, gamma, mean, rstd, dy, base, dg, db, s=s, b=b, h=h, tp=tp, accumulate=True)
    assert rel_err(_flat(torch.cat(base)), rb["dX"] + 1.0) <= tol
    # deterministic parameter gradients
    dg2 = torch.empty(h, device="cuda")
    db2 = torch.empty(h, device="cuda")
    tpmlp.sp_layernorm_backward(x, gamma, mean, rstd, dy, dx, dg2, db2, s=s, b=b, h=h, tp=tp)
    torch.cuda.synchronize()
    assert torch.equal(dg, dg2) and torch.equal(db, db2)
    assert tpmlp.device_status() == 0


@pytest.mark.parametrize("s,b,h,tp", [(16, 2, 136, 2), (40, 2, 2056, 4), (48, 1, 6144, 2)])
def test_layernorm_statistics_with_a_large_mean(cuda_lib, s, b, h, tp):
    """Rows at 1000 + 0.5·N(0, 1) in float32: the variance is 4·10⁻⁶ of the mean
    square, so E[x²] − E[x]² in float32 would cancel it away; mean and rstd must
    still match the fp64 oracle to 1e-5 (warp-per-row and streamed kernels)."""
    tpmlp = cuda_lib
    inp = sp_region_inputs(s, b, h, 0.1, seed=7 + h, dtype="f32")
    R = (inp["R"] * 0.5 + 1000.0).cuda()
    gamma, beta = inp["gamma"].cuda(), inp["beta"].cuda()
    x = chunks(R, tp)
    y = [torch.full_like(c, float("nan")) for c in x]
    mean = torch.empty(s * b, device="cuda")
    rstd = torch.empty(s * b, device="cuda")
    tpmlp.sp_layernorm_forward(x, gamma, beta, EPS, y, mean, rstd, s=s, b=b, h=h, tp=tp)
    torch.cuda.synchronize()
    ref = O.layernorm_forward(_flat(R.cpu()), to_np(inp["gamma"]), to_np(inp["beta"]), EPS)
    assert rel_err(to_np(mean), ref["mean"]) <= 1e-5
    assert rel_err(to_np(rstd), ref["rstd"]) <= 1e-5
    # Y carries the float32 rounding of a mean near 1000 (half an ulp, 3·10⁻⁵)
    # in every x − mean, about 10⁻⁴ of the normalised values
    assert rel_err(_flat(torch.cat(y)), ref["Y"]) <= 1e-4
    assert tpmlp.device_status() == 0


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("p", [0.0, 0.1])
@pytest.mark.parametrize("s,b,h,tp", [(64, 2, 136, 2), (9, 1, 5, 3)])
def test_residual_dropout(cuda_lib, dt, p, s, b, h, tp):
    tpmlp = cuda_lib
    inp = sp_region_inputs(s, b, h, p, seed=7 + s, dtype=dt)
    Z = block_inputs(BlockConfig("z", s, b, h, 8 * tp, tp, True, dt, "gelu", seed=3))["X"]
    r, z = chunks(inp["R"].cuda(), tp), chunks(Z.cuda(), tp)
    keep = chunks(inp["keep"].cuda(), tp)
    out = [torch.empty_like(c) for c in r]
    tpmlp.sp_residual_dropout_forward(r, z, keep, p, out, s=s, b=b, h=h, tp=tp)
    ref = O.residual_dropout_forward(_flat(inp["R"]), _flat(Z), _flat(inp["keep"]), p)
    tol = TOL[DT[dt]]
    assert rel_err(_flat(torch.cat(out)), ref) <= tol
    dout = chunks(inp["dOut"].cuda(), tp)
    dz = [torch.empty_like(c) for c in r]
    tpmlp.sp_residual_dropout_backward(dout, keep, p, dz, s=s, b=b, h=h, tp=tp)
    rb = O.residual_dropout_backward(_flat(inp["dOut"]), _flat(inp["keep"]), p)
    assert rel_err(_flat(torch.cat(dz)), rb["dZ"]) <= tol
    torch.cuda.synchronize()
    assert tpmlp.device_status() == 0


@pytest.mark.parametrize("act,mode", [("gelu", "fused"), ("swiglu", "partials")])
def test_sp_mlp_sublayer_end_to_end(cuda_lib, act, mode):
    """out = R + dropout(MLP(LN(R))) and its gradients, all on SP chunks (128-row
    chunks, so fc1 reads the LayerNorm output in place)."""
    tpmlp = cuda_lib
    s, b, h, f, tp, p = 256, 2, 256, 512, 4, 0.1
    reg = sp_region_inputs(s, b, h, p, seed=31)
    w = block_inputs(BlockConfig("w", s, b, h, f, tp, True, "bf16", act, seed=32))
    dev = "cuda"
    R = chunks(reg["R"].to(dev), tp)
    gamma, beta = reg["gamma"].to(dev), reg["beta"].to(dev)
    keep = chunks(reg["keep"].to(dev), tp)
    W1, W2 = w["W1"].to(dev), w["W2"].to(dev)
    M = s * b
    mean, rstd = torch.empty(M, device=dev), torch.empty(M, device=dev)
    Xn = [torch.empty_like(c) for c in R]
    tpmlp.sp_layernorm_forward(R, gamma, beta, EPS, Xn, mean, rstd, s=s, b=b, h=h, tp=tp)
    blk = tpmlp.MLPBlock(s, b, h, f, tp, True, torch.bfloat16, act, mode)
    fw = blk.forward(Xn, W1, W2)
    out = [torch.empty_like(c) for c in R]
    tpmlp.sp_residual_dropout_forward(R, fw["z"], keep, p, out, s=s, b=b, h=h, tp=tp)
    # backward
    dOut = chunks(reg["dOut"].to(dev), tp)
    dZ = [torch.empty_like(c) for c in R]
    tpmlp.sp_residual_dropout_backward(dOut, keep, p, dZ, s=s, b=b, h=h, tp=tp)
    bw = blk.backward(Xn, W1, W2, fw, dZ)
    dR = [c.clone() for c in dOut]  # residual branch
    dg, db = torch.empty(h, device=dev), torch.empty(h, device=dev)
    tpmlp.sp_layernorm_backward(R, gamma, mean, rstd, bw["dx"], dR, dg, db, s=s, b=b, h=h, tp=tp, accumulate=True)
    torch.cuda.synchronize()
    assert tpmlp.device_status() == 0
    # oracle composition in fp64
    R64 = _flat(reg["R"])
    ln = O.layernorm_forward(R64, to_np(reg["gamma"]), to_np(reg["beta"]), EPS)
    W1n, W2n = to_np(w["W1"]), to_np(w["W2"])
    mf = O.mlp_forward(ln["Y"], W1n, W2n, act)
    keep64 = _flat(reg["keep"])
    out_ref = O.residual_dropout_forward(R64, mf["Z"], keep64, p)
    rd = O.residual_dropout_backward(_flat(reg["dOut"]), keep64, p)
    mb = O.mlp_backward(ln["Y"], W1n, W2n, rd["dZ"], act)
    lb = O.layernorm_backward(R64, to_np(reg["gamma"]), mb["dX"], EPS)
    tol = 2e-2
    assert rel_err(_flat(torch.cat(out)), out_ref) <= tol
    assert rel_err(_flat(torch.cat(dR)), rd["dR"] + lb["dX"]) <= tol
    assert rel_err(to_np(dg), lb["dgamma"]) <= tol
    assert rel_err(to_np(db), lb["dbeta"]) <= tol
    assert rel_err(to_np(bw["dw1"]), mb["dW1"]) <= tol
    assert rel_err(to_np(bw["dw2"]), mb["dW2"]) <= tol
    assert M == len(mean)


def test_sp_region_at_the_22b_width(cuda_lib):
    """LayerNorm forward/backward (accumulating into the residual gradient) and
    dropout + residual on the [4096, 1, 6144] bf16 residual stream in 8 sequence
    chunks — the shapes the benchmark's SP-region step runs — against the oracle,
    every element."""
    tpmlp = cuda_lib
    s, b, h, tp, p = 4096, 1, 6144, 8, 0.1
    inp = sp_region_inputs(s, b, h, p, seed=61)
    Z = block_inputs(BlockConfig("z", s, b, h, 8 * tp, tp, True, "bf16", "gelu", seed=62))["X"]
    dev = "cuda"
    R = chunks(inp["R"].to(dev), tp)
    gamma, beta = inp["gamma"].to(dev), inp["beta"].to(dev)
    M = s * b
    mean, rstd = torch.empty(M, device=dev), torch.empty(M, device=dev)
    Y = [torch.empty_like(c) for c in R]
    tpmlp.sp_layernorm_forward(R, gamma, beta, EPS, Y, mean, rstd, s=s, b=b, h=h, tp=tp)
    dY = chunks(inp["dOut"].to(dev), tp)
    dR = [torch.ones_like(c) for c in R]
    dg, db = torch.empty(h, device=dev), torch.empty(h, device=dev)
    tpmlp.sp_layernorm_backward(R, gamma, mean, rstd, dY, dR, dg, db, s=s, b=b, h=h, tp=tp, accumulate=True)
    keep = chunks(inp["keep"].to(dev), tp)
    out = [torch.empty_like(c) for c in R]
    tpmlp.sp_residual_dropout_forward(R, chunks(Z.to(dev), tp), keep, p, out, s=s, b=b, h=h, tp=tp)
    dz = [torch.empty_like(c) for c in R]
    tpmlp.sp_residual_dropout_backward(dY, keep, p, dz, s=s, b=b, h=h, tp=tp)
    torch.cuda.synchronize()
    assert tpmlp.device_status() == 0
    R64, g64 = _flat(inp["R"]), to_np(inp["gamma"])
    ref = O.layernorm_forward(R64, g64, to_np(inp["beta"]), EPS)
    assert rel_err(_flat(torch.cat(Y)), ref["Y"]) <= 2e-2
    assert rel_err(to_np(mean), ref["mean"]) <= 1e-5
    assert rel_err(to_np(rstd), ref["rstd"]) <= 1e-5
    rb = O.layernorm_backward(R64, g64, _flat(inp["dOut"]), EPS)
    assert rel_err(_flat(torch.cat(dR)), rb["dX"] + 1.0) <= 2e-2
    assert rel_err(to_np(dg), rb["dgamma"]) <= 2e-2
    assert rel_err(to_np(db), rb["dbeta"]) <= 2e-2
    keep64 = _flat(inp["keep"])
    assert rel_err(_flat(torch.cat(out)), O.residual_dropout_forward(R64, _flat(Z), keep64, p)) <= 2e-2
    assert rel_err(_flat(torch.cat(dz)), O.residual_dropout_backward(_flat(inp["dOut"]), keep64, p)["dZ"]) <= 2e-2
