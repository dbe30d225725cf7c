"""Dim-0 movement and the shard sum on the GPU, bit-exact against NumPy slicing
and the oracle's float32 fixed-order sum + nearest-even rounding."""
import numpy as np
import pytest
import torch

import oracle as O
from synthetic import fp32_partials

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def _bits(t):
    t = t.contiguous().cpu()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy()
    return t.view(torch.int16).numpy()


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("s,b,h,tp", [(16, 2, 64, 2), (24, 3, 40, 8), (6, 1, 3, 3), (512, 4, 1024, 4), (8, 1, 8, 1),
                                      (4096, 1, 6144, 8)])
def test_split_gather_bit_exact(cuda_lib, dt, s, b, h, tp):
    tpmlp = cuda_lib
    g = torch.Generator().manual_seed(s * 7 + h)
    full = torch.randn(s, b, h, generator=g).to(DT[dt]).cuda()
    shards = [torch.full((s // tp, b, h), float("nan"), dtype=DT[dt], device="cuda") for _ in range(tp)]
    tpmlp.split_dim0(full, shards, s=s, b=b, h=h, tp=tp)
    ref = O.split_dim0(_bits(full), tp)
    for j in range(tp):
        assert np.array_equal(_bits(shards[j]), ref[j])
    back = torch.full_like(full, float("nan"))
    tpmlp.gather_dim0(shards, back, s=s, b=b, h=h, tp=tp)
    assert np.array_equal(_bits(back), O.gather_dim0(ref))
    assert tpmlp.device_status() == 0


def test_split_rejects_indivisible_sequence(cuda_lib):
    tpmlp = cuda_lib
    full = torch.zeros(10, 1, 8, device="cuda")
    with pytest.raises(tpmlp.TpmlpError) as e:
        tpmlp.split_dim0(full, [torch.zeros(3, 1, 8, device="cuda")] * 3, s=10, b=1, h=8, tp=3)
    assert e.value.status == "TPMLP_ERR_NOT_DIVISIBLE"


def test_empty_sequence_is_a_no_op(cuda_lib):
    tpmlp = cuda_lib
    full = torch.zeros(0, 2, 8, device="cuda", dtype=torch.bfloat16)
    shards = [torch.zeros(0, 2, 8, device="cuda", dtype=torch.bfloat16) for _ in range(2)]
    # zero-size tensors may have a NULL data pointer; use a real allocation
    dummy = torch.zeros(16, device="cuda", dtype=torch.bfloat16)
    tpmlp.split_dim0(dummy, [dummy, dummy], s=0, b=2, h=8, tp=2, dtype=torch.bfloat16)
    tpmlp.gather_dim0([dummy, dummy], dummy, s=0, b=2, h=8, tp=2, dtype=torch.bfloat16)
    assert tpmlp.device_status() == 0
    del full, shards


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("scatter", [0, 1])
@pytest.mark.parametrize("s,b,h,tp", [(16, 2, 64, 2), (12, 1, 20, 4), (9, 1, 5, 3), (512, 4, 1024, 4), (64, 1, 8, 8),
                                      (4096, 1, 6144, 8)])
def test_reduce_scatter_bit_exact(cuda_lib, dt, scatter, s, b, h, tp):
    tpmlp = cuda_lib
    P = fp32_partials(tp, s * b, h, seed=s + h + tp)
    Pd = P.cuda()
    if scatter:
        out = [torch.full((s // tp, b, h), float("nan"), dtype=DT[dt], device="cuda") for _ in range(tp)]
    else:
        out = [torch.full((s, b, h), float("nan"), dtype=DT[dt], device="cuda")]
    tpmlp.reduce_scatter_dim0(Pd, out, s=s, b=b, h=h, tp=tp, scatter=scatter)
    ref32 = O.shard_sum_fp32(P.numpy())
    ref = O.round_to_storage(ref32, dt).reshape(s, b, h)
    got = torch.cat(out, 0).float().cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    if scatter:
        for j, c in enumerate(O.split_dim0(ref, tp)):
            assert np.array_equal(out[j].float().cpu().numpy(), c)
    assert tpmlp.device_status() == 0
