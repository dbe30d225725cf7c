"""The tensor-parallel attention block on the GPU, through the C ABI, against the
fp64 oracle (oracle/attn_fp64.py): Z, dX, dWqkv, dWo and the saved
intermediates (QKV, O, lse2, dO, dQKV), both masks, both 16-bit storage types,
SP chunks read in place (whole 128-row chunks) or gathered (ragged chunks),
ragged sequence lengths, several sequences per batch, and bit-identical
repeats; grouped-query attention (several query heads per key/value head, and
one key/value head for all) and the head width 96 as well as 128.  Tolerance
‖GPU − oracle‖∞ / ‖oracle‖∞ ≤ 2e-2 per tensor."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_common import chunks, rel_err, to_np
from synthetic import ATTN_CONFIGS, AttnConfig, attn_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-2


def _run(tpmlp, cfg, t=None):
    t = t or attn_inputs(cfg)
    dev = "cuda"
    X, Wqkv, Wo, dZ = (t[k].to(dev) for k in ("X", "Wqkv", "Wo", "dZ"))
    x = chunks(X, cfg.tp) if cfg.sp else X
    dz = chunks(dZ, cfg.tp) if cfg.sp else dZ
    blk = tpmlp.AttnBlock(cfg.s, cfg.b, cfg.h, cfg.heads, cfg.tp, cfg.sp, cfg.torch_dtype, cfg.causal,
                          kv_heads=cfg.groups)
    fw = blk.forward(x, Wqkv, Wo)
    bw = blk.backward(x, Wqkv, Wo, fw, dz)
    torch.cuda.synchronize()
    assert tpmlp.device_status() == 0, tpmlp.last_error()
    cat = (lambda v: torch.cat(v)) if cfg.sp else (lambda v: v)
    return t, blk, fw, bw, cat


def _flat(a, M):
    return np.asarray(a).reshape(M, -1)


CASES = [
    # name, s, b, h, heads, tp, sp, dtype, causal
    AttnConfig("ag-gathered", 192, 2, 512, 4, 2, True, "bf16", False),
    AttnConfig("ag-in-place-causal", 256, 1, 256, 2, 2, True, "bf16", True),
    AttnConfig("no-sp-f16", 128, 1, 256, 2, 1, False, "f16", False),
    AttnConfig("no-sp-f16-causal", 128, 2, 256, 2, 1, False, "f16", True),
    AttnConfig("short-ragged", 100, 3, 256, 2, 1, False, "bf16", True),
    AttnConfig("ragged-tiles", 320, 1, 512, 4, 4, True, "bf16", True),
    AttnConfig("multi-tile-in-place", 1024, 1, 512, 4, 2, True, "bf16", False),
    # grouped-query attention: 2 query heads per group, one group per shard, in place, causal
    AttnConfig("gqa-2-per-group", 256, 1, 512, 4, 2, True, "bf16", True, kv_heads=2),
    # 4 query heads per group, gathered SP chunks (96 tokens × 2 sequences), unmasked
    AttnConfig("gqa-4-per-group-gathered", 192, 2, 1024, 8, 2, True, "bf16", False, kv_heads=2),
    # one key/value head for all query heads, ragged sequence, fp16
    AttnConfig("mqa-ragged-f16", 320, 1, 512, 4, 1, False, "f16", True, kv_heads=1),
    # head width 96 (the 22B and 8.3B models' heads)
    AttnConfig("d96-in-place-causal", 256, 1, 384, 4, 2, True, "bf16", True),
    AttnConfig("d96-ragged-f16", 100, 3, 192, 2, 1, False, "f16", False),
    AttnConfig("d96-gqa-multi-tile", 640, 1, 768, 8, 2, True, "bf16", True, kv_heads=2),
]


@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_attention_block_matches_the_oracle(cuda_lib, cfg):
    tpmlp = cuda_lib
    t, blk, fw, bw, cat = _run(tpmlp, cfg)
    M, s, b, heads = cfg.M, cfg.s, cfg.b, cfg.heads
    X, Wqkv, Wo, dZ = (to_np(t[k]).reshape(-1, t[k].shape[-1]) for k in ("X", "Wqkv", "Wo", "dZ"))
    ref = O.attn_forward(X, Wqkv, Wo, s, b, heads, cfg.causal, cfg.groups)
    g = O.attn_backward(X, Wqkv, Wo, dZ, s, b, heads, cfg.causal, cfg.groups)
    lse = to_np(fw["lse"])[:, :, :s]
    errs = {
        "QKV": rel_err(to_np(fw["qkv"]), ref["QKV"]),
        "O": rel_err(to_np(fw["o"]), ref["O"]),
        "Z": rel_err(_flat(to_np(cat(fw["z"])), M), ref["Z"]),
        "dO": rel_err(to_np(bw["dout"]), g["dO"]),
        "dQKV": rel_err(to_np(bw["dqkv"]), g["dQKV"]),
        "dX": rel_err(_flat(to_np(cat(bw["dx"])), M), g["dX"]),
        "dWqkv": rel_err(to_np(bw["dwqkv"]), g["dWqkv"]),
        "dWo": rel_err(to_np(bw["dwo"]), g["dWo"]),
    }
    print(cfg.name, errs)
    bad = {k: e for k, e in errs.items() if not e <= TOL}
    assert not bad, bad
    assert np.abs(lse - ref["lse2"]).max() <= 2e-2 * max(1.0, np.abs(ref["lse2"]).max())


SPLIT_CASES = [c for c in CASES if c.name in ("gqa-4-per-group-gathered", "d96-gqa-multi-tile")]


@pytest.mark.parametrize("split", ["1", "2"])
@pytest.mark.parametrize("cfg", SPLIT_CASES, ids=[c.name for c in SPLIT_CASES])
def test_grouped_query_split_of_the_key_value_gradients(cuda_lib, cfg, split, monkeypatch):
    """The dK/dV kernel with a group's 4 query heads split over 1 or 2 CTAs per
    key tile (each CTA running its heads one after the other; with 2, float32
    partials added by the reduce kernel) instead of one head per CTA: the
    backward against the oracle (the large-shape split is chosen by the CTA
    count, so small shapes take one head per CTA unless told otherwise)."""
    tpmlp = cuda_lib
    monkeypatch.setenv("TPMLP_ATTN_KV_SPLIT", split)
    t, blk, fw, bw, cat = _run(tpmlp, cfg)
    M, s, b, heads = cfg.M, cfg.s, cfg.b, cfg.heads
    X, Wqkv, Wo, dZ = (to_np(t[k]).reshape(-1, t[k].shape[-1]) for k in ("X", "Wqkv", "Wo", "dZ"))
    g = O.attn_backward(X, Wqkv, Wo, dZ, s, b, heads, cfg.causal, cfg.groups)
    errs = {
        "dQKV": rel_err(to_np(bw["dqkv"]), g["dQKV"]),
        "dX": rel_err(_flat(to_np(cat(bw["dx"])), M), g["dX"]),
        "dWqkv": rel_err(to_np(bw["dwqkv"]), g["dWqkv"]),
    }
    bad = {k: e for k, e in errs.items() if not e <= TOL}
    assert not bad, bad


CORE_CASES = [
    AttnConfig("core", 384, 2, 512, 4, 2, True, "bf16", True),
    AttnConfig("core-gqa", 384, 2, 1024, 8, 2, True, "bf16", True, kv_heads=2),
    AttnConfig("core-d96-gqa", 384, 1, 768, 8, 2, True, "bf16", False, kv_heads=4),
]


@pytest.mark.parametrize("cfg", CORE_CASES, ids=[c.name for c in CORE_CASES])
def test_attention_core_alone_on_the_gpu_s_own_qkv(cuda_lib, cfg):
    """The core's O, lse2 and dQ/dK/dV against the oracle's core evaluated on the
    GPU's own (rounded) QKV and dO: isolates the flash kernels from the
    projections (with grouped-query attention, dK and dV sum over the query
    heads of a group)."""
    tpmlp = cuda_lib
    t, blk, fw, bw, cat = _run(tpmlp, cfg)
    Q, K, V = O.split_qkv(to_np(fw["qkv"]), cfg.heads, cfg.groups)
    core = O.attention_core_forward(Q, K, V, cfg.s, cfg.b, cfg.heads, cfg.causal, cfg.groups)
    assert rel_err(to_np(fw["o"]), core["O"]) <= 1e-2
    assert np.abs(to_np(fw["lse"])[:, :, :cfg.s] - core["lse2"]).max() <= 1e-3 * np.abs(core["lse2"]).max()
    gc = O.attention_core_backward(Q, K, V, to_np(bw["dout"]), cfg.s, cfg.b, cfg.heads, cfg.causal, cfg.groups)
    dq, dk, dv = O.split_qkv(to_np(bw["dqkv"]), cfg.heads, cfg.groups)
    assert rel_err(dq, gc["dQ"]) <= TOL
    assert rel_err(dk, gc["dK"]) <= TOL
    assert rel_err(dv, gc["dV"]) <= TOL


@pytest.mark.parametrize("kv", [4, 2], ids=["mha", "gqa"])
def test_attention_is_deterministic(cuda_lib, kv):
    tpmlp = cuda_lib
    cfg = AttnConfig("det", 256, 1, 512, 4, 2, True, "bf16", True, kv_heads=kv)
    t = attn_inputs(cfg)
    _, _, fw1, bw1, cat = _run(tpmlp, cfg, t)
    _, _, fw2, bw2, _ = _run(tpmlp, cfg, t)
    assert torch.equal(cat(fw1["z"]), cat(fw2["z"]))
    for k in ("dwqkv", "dwo", "dqkv"):
        assert torch.equal(bw1[k], bw2[k]), k
    assert torch.equal(cat(bw1["dx"]), cat(bw2["dx"]))


def test_sp_on_equals_sp_off(cuda_lib):
    """Reading the SP chunks in place (all-gather fused into the GEMM loads) and the
    reduce-scatter fused into the epilogue give the SP-off block's bits."""
    tpmlp = cuda_lib
    on = AttnConfig("sp", 256, 2, 256, 2, 2, True, "bf16", False)
    t = attn_inputs(on)
    _, _, fa, ba, cat = _run(tpmlp, on, t)
    _, _, fb, bb, _ = _run(tpmlp, on.with_(sp=False), t)
    assert torch.equal(cat(fa["z"]), fb["z"])
    assert torch.equal(cat(ba["dx"]), bb["dx"])
    assert torch.equal(ba["dwqkv"], bb["dwqkv"]) and torch.equal(ba["dwo"], bb["dwo"])


def test_llama70b_width_attention_sampled(cuda_lib):
    """The benchmark's workload ([4096, 1, 8192], 64 heads of 128, tp 8, SP, causal,
    bf16) at full size: the core of two heads (one in the first shard, one in the
    last) against the oracle's core on the GPU's own QKV and dO, and the
    projections on sampled rows."""
    tpmlp = cuda_lib
    cfg = ATTN_CONFIGS["llama70b_attn_tpsp8_bf16"]
    t, blk, fw, bw, cat = _run(tpmlp, cfg)
    s, b, d = cfg.s, cfg.b, cfg.d
    qkv = to_np(fw["qkv"])
    o = to_np(fw["o"])
    do = to_np(bw["dout"])
    dqkv = to_np(bw["dqkv"])
    for j in (3, 60):
        cols = slice(3 * d * j, 3 * d * (j + 1))
        Q, K, V = O.split_qkv(qkv[:, cols], 1)
        core = O.attention_core_forward(Q, K, V, s, b, 1, True)
        assert rel_err(o[:, d * j:d * (j + 1)], core["O"]) <= 1e-2
        gc = O.attention_core_backward(Q, K, V, do[:, d * j:d * (j + 1)], s, b, 1, True)
        dq, dk, dv = O.split_qkv(dqkv[:, cols], 1)
        assert rel_err(dq, gc["dQ"]) <= TOL
        assert rel_err(dk, gc["dK"]) <= TOL
        assert rel_err(dv, gc["dV"]) <= TOL
    # projections on sampled rows, with the oracle's fp64 products of the GPU's inputs
    rows = np.array([0, 1, 511, 512, 2047, 4095])
    X = to_np(t["X"]).reshape(-1, cfg.h)
    Wqkv, Wo = to_np(t["Wqkv"]), to_np(t["Wo"])
    assert rel_err(qkv[rows], X[rows] @ Wqkv.T) <= TOL
    z = to_np(cat(fw["z"])).reshape(-1, cfg.h)
    assert rel_err(z[rows], o[rows] @ Wo.T) <= TOL
    dZ = to_np(t["dZ"]).reshape(-1, cfg.h)
    assert rel_err(do[rows], dZ[rows] @ Wo) <= TOL
    dx = to_np(cat(bw["dx"])).reshape(-1, cfg.h)
    assert rel_err(dx[rows], dqkv[rows] @ Wqkv) <= TOL
    feats = np.array([0, 127, 4096, 8191])
    dwo = to_np(bw["dwo"])
    assert rel_err(dwo[feats], dZ[:, feats].T @ o) <= TOL
    dwqkv = to_np(bw["dwqkv"])
    qrows = np.array([0, 383, 12288, 24575])
    assert rel_err(dwqkv[qrows], dqkv[:, qrows].T @ X) <= TOL


def _sampled_projections(cfg, t, fw, bw, cat, rows, feats, qrows):
    """QKV, Z, dO, dX on sampled token rows and dWo, dWqkv on sampled features,
    against the oracle's fp64 products of the GPU's own inputs."""
    X = to_np(t["X"]).reshape(-1, cfg.h)
    Wqkv, Wo = to_np(t["Wqkv"]), to_np(t["Wo"])
    qkv, o, do, dqkv = to_np(fw["qkv"]), to_np(fw["o"]), to_np(bw["dout"]), to_np(bw["dqkv"])
    assert rel_err(qkv[rows], X[rows] @ Wqkv.T) <= TOL
    z = to_np(cat(fw["z"])).reshape(-1, cfg.h)
    assert rel_err(z[rows], o[rows] @ Wo.T) <= TOL
    dZ = to_np(t["dZ"]).reshape(-1, cfg.h)
    assert rel_err(do[rows], dZ[rows] @ Wo) <= TOL
    dx = to_np(cat(bw["dx"])).reshape(-1, cfg.h)
    assert rel_err(dx[rows], dqkv[rows] @ Wqkv) <= TOL
    dwo = to_np(bw["dwo"])
    assert rel_err(dwo[feats], dZ[:, feats].T @ o) <= TOL
    dwqkv = to_np(bw["dwqkv"])
    assert rel_err(dwqkv[qrows], dqkv[:, qrows].T @ X) <= TOL


@pytest.mark.parametrize("name,heads_checked", [("llama70b_gqa_attn_tpsp8_bf16", (3, 60)),
                                                 ("w22b_attn_tpsp8_bf16", (5, 62))])
def test_gqa_and_d96_widths_sampled(cuda_lib, name, heads_checked):
    """The Llama-70B-like grouped-query workload ([4096, 1, 8192], 64 query heads
    and 8 key/value heads of 128, tp 8, SP, causal) and the 22B model's
    attention ([4096, 1, 6144], 64 heads of 96) at full size: the core of two
    query heads (first and last shard) against the oracle's core on the GPU's own
    QKV and dO — for GQA with the whole group, whose dK/dV sum over its eight
    query heads — and the projections on sampled rows and features."""
    tpmlp = cuda_lib
    cfg = ATTN_CONFIGS[name]
    t, blk, fw, bw, cat = _run(tpmlp, cfg)
    s, b, d, heads, G = cfg.s, cfg.b, cfg.d, cfg.heads, cfg.groups
    r = heads // G
    qkv, o, do, dqkv = to_np(fw["qkv"]), to_np(fw["o"]), to_np(bw["dout"]), to_np(bw["dqkv"])
    for j in heads_checked:
        g = j // r
        cols = slice(g * (r + 2) * d, (g + 1) * (r + 2) * d)  # the whole group: its r query heads, k, v
        hcols = slice(g * r * d, (g + 1) * r * d)
        Q, K, V = O.split_qkv(qkv[:, cols], r, 1)
        core = O.attention_core_forward(Q, K, V, s, b, r, True, 1)
        assert rel_err(o[:, hcols], core["O"]) <= 1e-2
        gc = O.attention_core_backward(Q, K, V, do[:, hcols], s, b, r, True, 1)
        dq, dk, dv = O.split_qkv(dqkv[:, cols], r, 1)
        for nm, got, want in (("dQ", dq, gc["dQ"]), ("dK", dk, gc["dK"]), ("dV", dv, gc["dV"])):
            assert rel_err(got, want) <= TOL, (j, nm)
    rows = np.array([0, 1, 511, 512, 2047, 4095])
    feats = np.array([0, 127, cfg.h // 2, cfg.h - 1])
    qrows = np.array([0, d - 1, cfg.qkv_rows // 2, cfg.qkv_rows - 1])
    _sampled_projections(cfg, t, fw, bw, cat, rows, feats, qrows)


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "unmasked"])
def test_growing_scores_raise_the_softmax_reference(cuda_lib, causal):
    """Token rows of X scaled up linearly along the sequence (×1 … ×10) make the
    scores grow along the keys, so a row's maximum rises by far more than 2^15
    between key tiles many times over: the forward's exponentials must raise
    their reference maximum mid-sequence and rescale O and the row sum (the
    path that plain N(0, 1) inputs only take on each row's first tile).  Scores
    this sharp make the block output sensitive to the rounding of QKV itself, so
    the core is checked against the oracle's core on the GPU's own QKV and dO."""
    tpmlp = cuda_lib
    cfg = AttnConfig("growing", 512, 1, 256, 2, 1, False, "bf16", causal)
    t = attn_inputs(cfg)
    ramp = torch.linspace(1.0, 10.0, cfg.s).view(cfg.s, 1, 1)
    t["X"] = (t["X"].float() * ramp).to(cfg.torch_dtype)
    _, blk, fw, bw, cat = _run(tpmlp, cfg, t)
    s, d = cfg.s, cfg.d
    Q, K, V = O.split_qkv(to_np(fw["qkv"]), cfg.heads)
    # the workload does exercise the path: per row, key tiles whose maximum
    # exceeds everything before it by more than 15 (log2 units)
    x = np.einsum("thd,uhd->htu", Q.reshape(s, cfg.heads, d), K.reshape(s, cfg.heads, d)) * (O.LOG2E / np.sqrt(d))
    if causal:
        x = np.where(np.triu(np.ones((s, s), dtype=bool), k=1), -np.inf, x)
    tile_max = x.reshape(cfg.heads, s, s // 128, 128).max(axis=-1)
    running = np.maximum.accumulate(tile_max, axis=-1)
    jumps = int((tile_max[..., 1:] > running[..., :-1] + 15).sum())
    assert jumps > 20, jumps  # 27 causal, 51 unmasked
    core = O.attention_core_forward(Q, K, V, s, cfg.b, cfg.heads, causal)
    assert rel_err(to_np(fw["o"]), core["O"]) <= 1e-2
    lse = to_np(fw["lse"])[:, :, :s]
    assert np.abs(lse - core["lse2"]).max() <= 1e-3 * np.abs(core["lse2"]).max()
    gc = O.attention_core_backward(Q, K, V, to_np(bw["dout"]), s, cfg.b, cfg.heads, causal)
    dq, dk, dv = O.split_qkv(to_np(bw["dqkv"]), cfg.heads)
    for name, got, want in (("dQ", dq, gc["dQ"]), ("dK", dk, gc["dK"]), ("dV", dv, gc["dV"])):
        assert rel_err(got, want) <= TOL, name


def test_empty_sequence(cuda_lib):
    """s = 0: nothing to compute; the weight gradients are empty sums (zero).
    (Buffers are non-empty dummies: the ABI rejects NULL pointers.)"""
    tpmlp = cuda_lib
    d = torch.bfloat16
    h, heads, tp = 256, 2, 2
    dummy = torch.zeros(4096, dtype=d, device="cuda")
    lse = torch.zeros(1024, device="cuda")
    Wqkv = torch.randn(3 * h, h, device="cuda").to(d)
    Wo = torch.randn(h, h, device="cuda").to(d)
    dwqkv = torch.full((3 * h, h), 7.0, dtype=d, device="cuda")
    dwo = torch.full((h, h), 7.0, dtype=d, device="cuda")
    ws = torch.empty(max(256, tpmlp.attn_workspace_size(0, 1, h, heads, tp, True, d, True)), dtype=torch.uint8,
                     device="cuda")
    kw = dict(s=0, b=1, h=h, heads=heads, tp=tp, sp=True, causal=True, workspace=ws)
    chunks2 = [dummy, dummy]
    tpmlp.attn_forward(chunks2, Wqkv, Wo, dummy, dummy, lse, chunks2, **kw)
    tpmlp.attn_backward(chunks2, Wqkv, Wo, dummy, dummy, lse, chunks2, chunks2, dwqkv, dwo, dummy, dummy, **kw)
    torch.cuda.synchronize()
    assert tpmlp.device_status() == 0
    assert not dwqkv.any() and not dwo.any()


PAIR_CASES = [
    # s = 1024 is two 512-row pair blocks; 320 leaves the last block mostly past s
    AttnConfig("pair-causal-gqa", 1024, 1, 1024, 8, 2, True, "bf16", True, kv_heads=2),
    AttnConfig("pair-unmasked-ragged-f16", 320, 2, 512, 4, 1, False, "f16", False),
]


@pytest.mark.parametrize("cfg", PAIR_CASES, ids=[c.name for c in PAIR_CASES])
def test_two_sm_forward_matches_the_one_cta_forward_and_the_oracle(cuda_lib, cfg, monkeypatch):
    """The 2-SM (CTA pair) forward, selected with TPMLP_ATTN_FWD_PAIR=1: O and
    lse2 against the oracle's core on the GPU's own QKV, O close to the one-CTA
    forward's, and the backward run on the pair forward's O and lse2 against
    the oracle's core gradients."""
    tpmlp = cuda_lib
    t = attn_inputs(cfg)
    monkeypatch.setenv("TPMLP_ATTN_FWD_PAIR", "1")
    _, _, fp, bp, cat = _run(tpmlp, cfg, t)
    monkeypatch.setenv("TPMLP_ATTN_FWD_PAIR", "0")
    _, _, f1, b1, _ = _run(tpmlp, cfg, t)
    assert torch.equal(fp["qkv"], f1["qkv"])
    Q, K, V = O.split_qkv(to_np(fp["qkv"]), cfg.heads, cfg.groups)
    core = O.attention_core_forward(Q, K, V, cfg.s, cfg.b, cfg.heads, cfg.causal, cfg.groups)
    assert rel_err(to_np(fp["o"]), core["O"]) <= 1e-2
    assert np.abs(to_np(fp["lse"])[:, :, :cfg.s] - core["lse2"]).max() <= 1e-3 * np.abs(core["lse2"]).max()
    assert rel_err(to_np(fp["o"]), to_np(f1["o"])) <= 1e-2
    g = O.attention_core_backward(Q, K, V, to_np(bp["dout"]), cfg.s, cfg.b, cfg.heads, cfg.causal, cfg.groups)
    dq, dk, dv = O.split_qkv(to_np(bp["dqkv"]), cfg.heads, cfg.groups)
    for name, got, want in (("dQ", dq, g["dQ"]), ("dK", dk, g["dK"]), ("dV", dv, g["dV"])):
        assert rel_err(got, want) <= TOL, name
