"""Block-level parity of the CUDA path (through the C ABI) against the fp64 oracle
on shapes that span several tiles and ragged tails, plus the invariants the
method fixes: exact results on integer data, SP on/off identity, independence of
the fused result from tp, the shard sum of the partials, determinism, and the
degenerate and error cases."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_common import TOL, assert_block_close, oracle_block, rel_err, run_block, to_np
from synthetic import BlockConfig, block_inputs, integer_block_inputs

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def _cfg(s, b, h, f, tp, sp, dt, act):
    return BlockConfig("t", s, b, h, f, tp, sp, dt, act, seed=s * 31 + h + f + tp)


# Ragged on purpose: M = 192 (1.5 M-tiles), h = 136 (ragged N and K tiles),
# f/tp = 136 (a shard's K range ends inside a 64-wide K block).
@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("act", ["gelu", "swiglu", "relu", "identity"])
@pytest.mark.parametrize("mode", ["fused", "partials"])
@pytest.mark.parametrize("sp", [False, True])
def test_block_parity_ragged(cuda_lib, dt, act, mode, sp):
    cfg = _cfg(64, 3, 136, 272, 2, sp, dt, act)
    inp = block_inputs(cfg)
    out = run_block(cuda_lib, inp, cfg.s, cfg.b, cfg.h, cfg.f, cfg.tp, sp, act, mode, DT[dt])
    assert_block_close(out, oracle_block(inp, act), DT[dt])


@pytest.mark.parametrize("act", ["gelu", "swiglu", "relu"])
@pytest.mark.parametrize("mode", ["fused", "partials"])
@pytest.mark.parametrize("shape", [(16, 2, 64, 256, 2, False), (12, 1, 5, 6, 2, True), (33, 3, 70, 96, 4, False),
                                   (64, 2, 100, 120, 8, True)])
def test_block_parity_float32(cuda_lib, act, mode, shape):
    s, b, h, f, tp, sp = shape
    cfg = _cfg(s, b, h, f, tp, sp, "f32", act)
    inp = block_inputs(cfg)
    out = run_block(cuda_lib, inp, s, b, h, f, tp, sp, act, mode, torch.float32)
    assert_block_close(out, oracle_block(inp, act), torch.float32)


@pytest.mark.parametrize("mode", ["fused", "partials"])
def test_worked_two_layer_relu_example_exact(cuda_lib, mode):
    """W1 ∈ R^{4×8} column-split over 2 shards, ReLU local, W2 ∈ R^{8×4} row-split,
    B = 3 tokens, integer data: every float32 operation is exact."""
    inp = integer_block_inputs(3, 1, 4, 8, "relu", seed=11)
    out = run_block(cuda_lib, inp, 3, 1, 4, 8, 2, False, "relu", mode, torch.float32)
    ref = oracle_block(inp, "relu")
    for k in ("Z", "dX", "dW1", "dW2", "U", "Y", "dU"):
        assert np.array_equal(out[k], ref[k]), k


@pytest.mark.parametrize("dt,s,b,h,f", [("f16", 32, 2, 16, 32), ("bf16", 8, 2, 8, 16), ("f16", 32, 2, 16, 64)])
@pytest.mark.parametrize("act", ["identity", "relu"])
@pytest.mark.parametrize("mode", ["fused", "partials"])
@pytest.mark.parametrize("sp", [False, True])
def test_tensor_core_path_exact_on_integer_data(cuda_lib, dt, s, b, h, f, act, mode, sp):
    """Entries in {-1, 0, 1}: products and sums are small integers, exact in the
    float32 accumulator and in the 16-bit storage, so the GPU equals the oracle."""
    inp = integer_block_inputs(s, b, h, f, act, seed=5, dtype=dt, lo=-1, hi=1)
    out = run_block(cuda_lib, inp, s, b, h, f, 2, sp, act, mode, DT[dt])
    ref = oracle_block(inp, act)
    for k in ("Z", "dX", "dW1", "dW2", "U", "Y", "dU"):
        assert np.array_equal(out[k], ref[k]), k


# (s, b, h, f, tp): 64-row chunks -> the SP chunks are gathered by the copy kernel;
# 128-row chunks -> the all-gather is fused into the GEMMs' loads; 3 chunks of 128
# rows -> M = 384, so the last 256-row tile's second half starts past M.
SP_SHAPES = [(128, 2, 256, 512, 4), (256, 2, 256, 512, 4), (192, 2, 256, 288, 3)]


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("mode", ["fused", "partials"])
@pytest.mark.parametrize("shape", SP_SHAPES, ids=["gathered", "fused-gather", "fused-gather-3chunks"])
def test_sp_on_and_off_are_bit_identical(cuda_lib, dt, act, mode, shape):
    """AG → block → RS equals block → all-reduce → split, bit for bit, whether the
    all-gather is a separate copy or fused into the GEMM loads."""
    s, b, h, f, tp = shape
    cfg = _cfg(s, b, h, f, tp, False, dt, act)
    inp = block_inputs(cfg)
    a = run_block(cuda_lib, inp, s, b, h, f, tp, False, act, mode, DT[dt])
    c = run_block(cuda_lib, inp, s, b, h, f, tp, True, act, mode, DT[dt])
    for k in ("Z", "dX", "dW1", "dW2", "U", "Y", "dU"):
        assert np.array_equal(a[k], c[k]), k
    assert_block_close(c, oracle_block(inp, act), DT[dt])


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_fused_result_is_independent_of_tp(cuda_lib, act):
    """The fused shard sum accumulates the K ranges of shards 0..tp-1 in order —
    the same order for every tp — so the result does not depend on tp."""
    cfg = _cfg(96, 2, 128, 512, 1, False, "bf16", act)
    inp = block_inputs(cfg)
    base = run_block(cuda_lib, inp, 96, 2, 128, 512, 1, False, act, "fused", torch.bfloat16)
    for tp in (2, 4, 8):
        o = run_block(cuda_lib, inp, 96, 2, 128, 512, tp, True, act, "fused", torch.bfloat16)
        for k in ("Z", "dX", "dW1", "dW2"):
            assert np.array_equal(base[k], o[k]), (tp, k)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("tp", [1, 2, 8])
def test_partials_mode_output_is_the_fixed_order_shard_sum(cuda_lib, dt, tp):
    """After the forward in PARTIALS mode the workspace holds fc2's tp float32
    partials; Z must be their fixed-order float32 sum, rounded once."""
    s, b, h, f = 64, 2, 128, 512
    cfg = _cfg(s, b, h, f, tp, False, dt, "gelu")
    inp = block_inputs(cfg)
    out = run_block(cuda_lib, inp, s, b, h, f, tp, False, "gelu", "partials", DT[dt])
    M = s * b
    ws = out["_raw"]["ws_after_fwd"]
    P = ws[: tp * M * h * 4].view(torch.float32).reshape(tp, M, h).cpu().numpy()
    ref = O.round_to_storage(O.shard_sum_fp32(P), dt)
    assert np.array_equal(out["Z"].astype(np.float32), ref)
    # and each partial is shard i's own contribution Y_i·B_i (oracle, fp64)
    sh = O.mlp_forward_sharded(O.flatten_sbh(to_np(inp["X"])), to_np(inp["W1"]), to_np(inp["W2"]), "gelu", tp)
    for i in range(tp):
        assert rel_err(P[i], sh["partials"][i]) < TOL[DT[dt]]


def test_results_are_deterministic(cuda_lib):
    cfg = _cfg(256, 2, 512, 1024, 4, True, "bf16", "gelu")
    inp = block_inputs(cfg)
    a = run_block(cuda_lib, inp, 256, 2, 512, 1024, 4, True, "gelu", "partials", torch.bfloat16)
    c = run_block(cuda_lib, inp, 256, 2, 512, 1024, 4, True, "gelu", "partials", torch.bfloat16)
    for k in ("Z", "dX", "dW1", "dW2", "dU"):
        assert np.array_equal(a[k], c[k]), k


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_empty_sequence(cuda_lib, dt):
    """s = 0: nothing to compute forward; the weight gradients are empty sums (zero)."""
    tpmlp = cuda_lib
    d = DT[dt]
    h, f, tp = 64, 128, 2
    dummy = torch.zeros(64, dtype=d, device="cuda")
    W1 = torch.randn(f, h, device="cuda").to(d)
    W2 = torch.randn(h, f, device="cuda").to(d)
    dW1 = torch.full((f, h), float("nan"), dtype=d, device="cuda")
    dW2 = torch.full((h, f), float("nan"), dtype=d, device="cuda")
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    tpmlp.forward([dummy, dummy], W1, W2, dummy, dummy, [dummy, dummy], s=0, b=1, h=h, f=f, tp=tp, sp=True,
                  workspace=ws)
    tpmlp.backward([dummy, dummy], W1, W2, dummy, dummy, [dummy, dummy], [dummy, dummy], dW1, dW2, dummy, s=0,
                   b=1, h=h, f=f, tp=tp, sp=True, workspace=ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dW1).item() == 0 and torch.count_nonzero(dW2).item() == 0
    assert tpmlp.device_status() == 0


def test_misaligned_pointer_is_rejected(cuda_lib):
    tpmlp = cuda_lib
    blk = tpmlp.MLPBlock(16, 2, 64, 256, 2, False, torch.bfloat16)
    base = torch.zeros(16 * 2 * 64 + 1, dtype=torch.bfloat16, device="cuda")
    x = base[1:].view(16, 2, 64)  # 2-byte offset
    W1 = torch.zeros(256, 64, dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros(64, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tpmlp.TpmlpError) as e:
        blk.forward(x, W1, W2)
    assert e.value.status == "TPMLP_ERR_UNSUPPORTED"


def test_multi_tile_persistent_schedule(cuda_lib):
    """Many more tiles than SMs (several tiles per CTA, both accumulator buffers
    and several phases of the stage ring), ragged in every dimension."""
    s, b, h, f, tp = 1000, 2, 1048, 4160, 4
    cfg = _cfg(s, b, h, f, tp, True, "bf16", "gelu")
    inp = block_inputs(cfg)
    out = run_block(cuda_lib, inp, s, b, h, f, tp, True, "gelu", "fused", torch.bfloat16)
    assert_block_close(out, oracle_block(inp, "gelu"), torch.bfloat16)
