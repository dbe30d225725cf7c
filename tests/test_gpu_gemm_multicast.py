"""The GEMM gives bit-identical results with and without operand multicast.

TPMLP_GEMM_MULTICAST=0 runs the 2-SM GEMM as plain CTA pairs; by default (1)
the launch asks for clusters of 4 where the GPCs have room, and the two pairs
of such a cluster, on neighbouring N tiles, share their A rows by TMA
multicast, while the remaining pairs run alone.  The switch changes which SM
loads which operand rows, never the order of the K accumulation, so every
output of the block is bit-identical with and without it; the multicast run is
also compared with the fp64 oracle.  The switch is read once per process, so
each setting runs in a child process.  The shapes cover the fused SP gather
with multicast, a ragged last M tile, SwiGLU (whose fused gate/up GEMM keeps
plain pairs) and an odd number of N tiles (plain pairs)."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from gpu_common import assert_block_close, oracle_block
from synthetic import BlockConfig, block_inputs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")
KEYS = ("Z", "dX", "dW1", "dW2", "U", "Y", "dU")
DT = {"f16": torch.float16, "bf16": torch.bfloat16}

CHILD = r"""
import sys
import numpy as np
import torch
sys.path[:0] = [{root!r}, {tests!r}]
import sp_partitioned_transformer_gb300 as tpmlp
from gpu_common import run_block
from synthetic import BlockConfig, block_inputs
tpmlp.load()
s, b, h, f, tp, sp, dt, act = {shape!r}
cfg = BlockConfig("mc", s, b, h, f, tp, sp, dt, act, seed=7)
out = run_block(tpmlp, block_inputs(cfg), s, b, h, f, tp, sp, act, "fused",
                {{"f16": torch.float16, "bf16": torch.bfloat16}}[dt])
np.savez({path!r}, **{{k: out[k] for k in {keys!r}}})
"""

SHAPES = {
    # M = 1024, f/tp = 1024, h = 1024, SP chunks of 256 rows: every GEMM multicasts
    "even": (1024, 1, 1024, 4096, 4, True, "bf16", "gelu"),
    # M = 900: the last pair tile is ragged; SwiGLU's fc1 keeps plain pairs
    "ragged_swiglu": (450, 2, 1024, 3072, 2, False, "f16", "swiglu"),
    # h = 640: three N tiles in fc2 and fc1's input gradient (plain pairs there)
    "odd_n_tiles": (320, 2, 640, 2048, 2, True, "bf16", "relu"),
}


def _run_child(shape, level, path):
    code = CHILD.format(root=ROOT, tests=TESTS, shape=shape, path=path, keys=KEYS)
    env = dict(os.environ, TPMLP_GEMM_MULTICAST=level)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, f"multicast level {level}: exit {r.returncode}\n{r.stdout[-2000:]}\n{r.stderr[-4000:]}"
    with np.load(path) as z:
        return {k: z[k] for k in KEYS}


@pytest.mark.parametrize("name", list(SHAPES))
def test_multicast_is_bit_identical(cuda_lib, tmp_path, name):
    shape = SHAPES[name]
    outs = {lv: _run_child(shape, lv, str(tmp_path / f"out_{lv}.npz")) for lv in ("0", "1")}
    for k in KEYS:
        assert np.array_equal(outs["1"][k], outs["0"][k]), (name, k)
    s, b, h, f, tp, sp, dt, act = shape
    inp = block_inputs(BlockConfig("mc", s, b, h, f, tp, sp, dt, act, seed=7))
    errs = assert_block_close(outs["1"], oracle_block(inp, act), DT[dt])
    print(name, errs)
