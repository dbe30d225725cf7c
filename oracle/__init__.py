"""CPU oracle of the tensor/sequence-parallel MLP and attention blocks (TEST INFRASTRUCTURE ONLY).

Plain NumPy float64 (plus a few float32 helpers where the method fixes float32
arithmetic: the fixed-order shard sum and the final rounding).  Nothing here is
imported by the product package; only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may use it.

Pages followed (cited by title and section):

* "Tensor Parallelism（TP）与 Sequence Parallelism（SP）" (llm-infra-atlas)
* "tensor-parallelism-matrix-split" (111qqz.com)
* "tensor-parallel-megatron" visual reading (blog.vllbc.top)
* "Sequence Parallel 与 Context Parallel" (blog.vllbc.top)

Every function is pinned by a ``-m "not gpu"`` test (``tests/test_oracle_pins.py``,
``tests/test_oracle_attn_pins.py``)
against something other than itself: values the pages print, closed forms,
finite differences, brute-force loops or an independent library routine.
"""
from .mlp_fp64 import *  # noqa: F401,F403
from .attn_fp64 import *  # noqa: F401,F403
