"""Python binding of ``libtpmlp.so`` — the GB300 tensor/sequence-parallel MLP block.

Argument marshalling only: every step of the block runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current CUDA stream.  If the
library has not been built, ``load()`` raises; there is no fallback path.

Entry points mirror the C ABI in ``include/tpmlp.h``:

* ``workspace_size``, ``forward_workspace_size``, ``forward``, ``backward``
* ``split_dim0``, ``gather_dim0``, ``reduce_scatter_dim0``
* ``last_error``, ``device_status``, ``set_wait_timeout_ns``, ``wait_timeout_selftest``

``MLPBlock`` is a convenience holder that allocates outputs and the workspace
with ``torch.empty`` for one configuration and calls the entry points.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

__all__ = [
    "TpmlpError",
    "load",
    "lib_path",
    "STATUS",
    "DTYPE",
    "ACT",
    "MODE",
    "workspace_size",
    "forward_workspace_size",
    "forward",
    "forward_noalloc",
    "NOALLOC_SCRATCH_BYTES",
    "backward",
    "backward_main_grad",
    "split_dim0",
    "gather_dim0",
    "reduce_scatter_dim0",
    "last_error",
    "device_status",
    "set_wait_timeout_ns",
    "wait_timeout_selftest",
    "abi_version",
    "sp_layernorm_forward",
    "sp_layernorm_backward",
    "sp_layernorm_backward_workspace",
    "sp_residual_dropout_forward",
    "sp_residual_dropout_backward",
    "profile_start",
    "profile_stop",
    "PROFILE_KINDS",
    "MLPBlock",
    "attn_workspace_size",
    "attn_forward",
    "attn_backward",
    "AttnBlock",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_lib", "libtpmlp.so")

STATUS = {
    0: "TPMLP_OK",
    -1: "TPMLP_ERR_INVALID_ARG",
    -2: "TPMLP_ERR_NOT_DIVISIBLE",
    -3: "TPMLP_ERR_UNSUPPORTED",
    -4: "TPMLP_ERR_WORKSPACE",
    -5: "TPMLP_ERR_CUDA",
    -6: "TPMLP_ERR_TIMEOUT",
}
DTYPE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
DTYPE_NAMES = {"f32": 0, "f16": 1, "bf16": 2}
ACT = {"gelu": 0, "swiglu": 1, "identity": 2, "relu": 3}
MODE = {"partials": 0, "fused": 1}

PROFILE_KINDS = ("gemm_tc", "gemm_f32", "copy_dim0", "shard_sum", "sp_region", "attn_core")

_lib = None


class _Profile(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int * 6), ("ms", ctypes.c_double * 6), ("work", ctypes.c_double * 6)]


class TpmlpError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code
        self.status = STATUS.get(code, str(code))


def lib_path() -> str:
    return _LIB_PATH


def load(path: str | None = None):
    """Load libtpmlp.so (raises ImportError if it is missing — no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise ImportError(
            f"{p} is not built; run `python -m sp_partitioned_transformer_gb300.build` "
            "(nvcc, sm_103a) first"
        )
    lib = ctypes.CDLL(p)
    i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    vpp = ctypes.POINTER(ctypes.c_void_p)
    lib.tpmlp_abi_version.restype = i32
    lib.tpmlp_abi_version.argtypes = []
    lib.tpmlp_last_error.restype = ctypes.c_char_p
    lib.tpmlp_last_error.argtypes = []
    lib.tpmlp_workspace_size.restype = sz
    lib.tpmlp_workspace_size.argtypes = [i64, i64, i64, i64, i32, i32, i32, i32, i32]
    lib.tpmlp_forward_workspace_size.restype = sz
    lib.tpmlp_forward_workspace_size.argtypes = [i64, i64, i64, i64, i32, i32, i32, i32, i32]
    lib.tpmlp_forward.restype = i32
    lib.tpmlp_forward.argtypes = [i64, i64, i64, i64, i32, i32, i32, i32, i32,
                                  vpp, vp, vp, vp, vp, vpp, vp, sz, vp]
    lib.tpmlp_backward.restype = i32
    lib.tpmlp_backward.argtypes = [i64, i64, i64, i64, i32, i32, i32, i32, i32,
                                   vpp, vp, vp, vp, vp, vpp, vpp, vp, vp, vp, vp, sz, vp]
    lib.tpmlp_backward_main_grad.restype = i32
    lib.tpmlp_backward_main_grad.argtypes = [i64, i64, i64, i64, i32, i32, i32, i32, i32,
                                             vpp, vp, vp, vp, vp, vpp, vpp, vp, vp, vp, vp, sz, vp]
    lib.tpmlp_split_dim0.restype = i32
    lib.tpmlp_split_dim0.argtypes = [vp, vpp, i64, i64, i64, i32, i32, vp]
    lib.tpmlp_gather_dim0.restype = i32
    lib.tpmlp_gather_dim0.argtypes = [vpp, vp, i64, i64, i64, i32, i32, vp]
    lib.tpmlp_reduce_scatter_dim0.restype = i32
    lib.tpmlp_reduce_scatter_dim0.argtypes = [vp, vpp, i64, i64, i64, i32, i32, i32, vp]
    lib.tpmlp_device_status.restype = i32
    lib.tpmlp_device_status.argtypes = [vp, i32]
    lib.tpmlp_set_wait_timeout_ns.restype = None
    lib.tpmlp_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.tpmlp_wait_timeout_selftest.restype = i32
    lib.tpmlp_wait_timeout_selftest.argtypes = [ctypes.c_uint64, vp]
    lib.tpmlp_forward_noalloc.restype = i32
    lib.tpmlp_forward_noalloc.argtypes = [i64, i64, i64, i64, i32, i32, i32, i32, i32,
                                          vpp, vp, vp, vp, vp, vpp, vp]
    f32 = ctypes.c_float
    lib.tpmlp_sp_layernorm_forward.restype = i32
    lib.tpmlp_sp_layernorm_forward.argtypes = [vpp, vp, vp, f32, vpp, vp, vp, i64, i64, i64, i32, i32, vp]
    lib.tpmlp_sp_layernorm_backward_workspace.restype = sz
    lib.tpmlp_sp_layernorm_backward_workspace.argtypes = [i64, i64, i64]
    lib.tpmlp_sp_layernorm_backward.restype = i32
    lib.tpmlp_sp_layernorm_backward.argtypes = [vpp, vp, vp, vp, vpp, vpp, i32, vp, vp, vp, sz, i64, i64, i64, i32,
                                                i32, vp]
    lib.tpmlp_sp_residual_dropout_forward.restype = i32
    lib.tpmlp_sp_residual_dropout_forward.argtypes = [vpp, vpp, vpp, f32, vpp, i64, i64, i64, i32, i32, vp]
    lib.tpmlp_sp_residual_dropout_backward.restype = i32
    lib.tpmlp_sp_residual_dropout_backward.argtypes = [vpp, vpp, f32, vpp, i64, i64, i64, i32, i32, vp]
    lib.tpmlp_attn_workspace_size.restype = sz
    lib.tpmlp_attn_workspace_size.argtypes = [i64, i64, i64, i32, i32, i32, i32, i32, i32]
    lib.tpmlp_attn_forward.restype = i32
    lib.tpmlp_attn_forward.argtypes = [i64, i64, i64, i32, i32, i32, i32, i32, i32,
                                       vpp, vp, vp, vp, vp, vp, vpp, vp, sz, vp]
    lib.tpmlp_attn_backward.restype = i32
    lib.tpmlp_attn_backward.argtypes = [i64, i64, i64, i32, i32, i32, i32, i32, i32,
                                        vpp, vp, vp, vp, vp, vp, vpp, vpp, vp, vp, vp, vp, vp, sz, vp]
    lib.tpmlp_profile_start.restype = i32
    lib.tpmlp_profile_start.argtypes = []
    lib.tpmlp_profile_stop.restype = i32
    lib.tpmlp_profile_stop.argtypes = [ctypes.POINTER(_Profile)]
    _lib = lib
    return lib


# ---------------------------------------------------------------- marshalling


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _ptrs(ts):
    """Host array of device pointers (a list/tuple of tensors, or one tensor)."""
    if ts is None:
        return None
    if isinstance(ts, (list, tuple)):
        vals = [_ptr(t) for t in ts]
    else:
        vals = [_ptr(ts)]
    return (ctypes.c_void_p * len(vals))(*vals)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(dtype) -> int:
    if isinstance(dtype, str):
        return DTYPE_NAMES[dtype]
    if isinstance(dtype, int):
        return dtype
    return DTYPE[dtype]


def _check(rc: int) -> None:
    if rc != 0:
        raise TpmlpError(rc, last_error())


def abi_version() -> int:
    return load().tpmlp_abi_version()


def last_error() -> str:
    return load().tpmlp_last_error().decode(errors="replace")


def workspace_size(s, b, h, f, tp, sp, dtype, act="gelu", mode="fused") -> int:
    return int(load().tpmlp_workspace_size(s, b, h, f, tp, int(sp), _dtype_code(dtype), ACT[act], MODE[mode]))


def forward_workspace_size(s, b, h, f, tp, sp, dtype, act="gelu", mode="fused") -> int:
    return int(load().tpmlp_forward_workspace_size(s, b, h, f, tp, int(sp), _dtype_code(dtype), ACT[act],
                                                   MODE[mode]))


def forward(x, w1, w2, u, y, z, *, s, b, h, f, tp, sp, act="gelu", mode="fused", workspace=None,
            workspace_bytes=None, dtype=None, stream=None) -> None:
    """Enqueue the block's forward.  x, z: a tensor, or a list of tp SP chunks."""
    dt = _dtype_code(dtype if dtype is not None else w1.dtype)
    ws_bytes = workspace_bytes if workspace_bytes is not None else (
        0 if workspace is None or isinstance(workspace, int) else workspace.numel() * workspace.element_size())
    rc = load().tpmlp_forward(s, b, h, f, tp, int(sp), dt, ACT[act], MODE[mode], _ptrs(x), _ptr(w1), _ptr(w2),
                              _ptr(u), _ptr(y), _ptrs(z), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc)


NOALLOC_SCRATCH_BYTES = 64 << 20


def forward_noalloc(x, w1, w2, u, y, z, *, s, b, h, f, tp, sp, act="gelu", mode="fused", dtype=None,
                    stream=None) -> None:
    """The forward without a caller workspace: the library's built-in 64 MiB
    scratch is used instead (for callers that cannot allocate device memory where
    they call the block).  Calls share that scratch: do not overlap them on the GPU."""
    dt = _dtype_code(dtype if dtype is not None else w1.dtype)
    rc = load().tpmlp_forward_noalloc(s, b, h, f, tp, int(sp), dt, ACT[act], MODE[mode], _ptrs(x), _ptr(w1),
                                      _ptr(w2), _ptr(u), _ptr(y), _ptrs(z), _stream(stream))
    _check(rc)


def backward(x, w1, w2, u, y, dz, dx, dw1, dw2, du, *, s, b, h, f, tp, sp, act="gelu", mode="fused",
             workspace=None, workspace_bytes=None, dtype=None, stream=None) -> None:
    """Enqueue the block's backward.  x, dz, dx: a tensor, or a list of tp SP chunks."""
    dt = _dtype_code(dtype if dtype is not None else w1.dtype)
    ws_bytes = workspace_bytes if workspace_bytes is not None else (
        0 if workspace is None or isinstance(workspace, int) else workspace.numel() * workspace.element_size())
    rc = load().tpmlp_backward(s, b, h, f, tp, int(sp), dt, ACT[act], MODE[mode], _ptrs(x), _ptr(w1), _ptr(w2),
                               _ptr(u), _ptr(y), _ptrs(dz), _ptrs(dx), _ptr(dw1), _ptr(dw2), _ptr(du),
                               _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc)


def backward_main_grad(x, w1, w2, u, y, dz, dx, main_grad_w1, main_grad_w2, du, *, s, b, h, f, tp, sp,
                       act="gelu", mode="fused", workspace=None, workspace_bytes=None, dtype=None,
                       stream=None) -> None:
    """tpmlp_backward with the weight gradients added into float32 main_grad buffers."""
    dt = _dtype_code(dtype if dtype is not None else w1.dtype)
    ws_bytes = workspace_bytes if workspace_bytes is not None else (
        0 if workspace is None or isinstance(workspace, int) else workspace.numel() * workspace.element_size())
    rc = load().tpmlp_backward_main_grad(s, b, h, f, tp, int(sp), dt, ACT[act], MODE[mode], _ptrs(x), _ptr(w1),
                                         _ptr(w2), _ptr(u), _ptr(y), _ptrs(dz), _ptrs(dx), _ptr(main_grad_w1),
                                         _ptr(main_grad_w2), _ptr(du), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc)


def split_dim0(full, shards, *, s, b, h, tp, dtype=None, stream=None) -> None:
    dt = _dtype_code(dtype if dtype is not None else full.dtype)
    _check(load().tpmlp_split_dim0(_ptr(full), _ptrs(shards), s, b, h, tp, dt, _stream(stream)))


def gather_dim0(shards, full, *, s, b, h, tp, dtype=None, stream=None) -> None:
    dt = _dtype_code(dtype if dtype is not None else full.dtype)
    _check(load().tpmlp_gather_dim0(_ptrs(shards), _ptr(full), s, b, h, tp, dt, _stream(stream)))


def reduce_scatter_dim0(partials, out, *, s, b, h, tp, scatter, dtype=None, stream=None) -> None:
    outs = out if isinstance(out, (list, tuple)) else [out]
    dt = _dtype_code(dtype if dtype is not None else outs[0].dtype)
    _check(load().tpmlp_reduce_scatter_dim0(_ptr(partials), _ptrs(outs), s, b, h, tp, int(scatter), dt,
                                            _stream(stream)))


def device_status(reset: bool = False, stream=None) -> int:
    """Synchronise the stream and return the device status (0 = OK, -6 = a wait timed out)."""
    return int(load().tpmlp_device_status(_stream(stream), int(reset)))


def set_wait_timeout_ns(ns: int) -> None:
    load().tpmlp_set_wait_timeout_ns(int(ns))


def wait_timeout_selftest(timeout_ns: int, stream=None) -> None:
    _check(load().tpmlp_wait_timeout_selftest(int(timeout_ns), _stream(stream)))


def _as_list(t):
    return list(t) if isinstance(t, (list, tuple)) else [t]


def sp_layernorm_forward(x, gamma, beta, eps, y, mean, rstd, *, s, b, h, tp, dtype=None, stream=None) -> None:
    """LayerNorm over h on the SP chunks (lists of tp [s/tp,b,h] tensors, or one tensor with tp=1)."""
    xs, ys = _as_list(x), _as_list(y)
    dt = _dtype_code(dtype if dtype is not None else xs[0].dtype)
    _check(load().tpmlp_sp_layernorm_forward(_ptrs(xs), _ptr(gamma), _ptr(beta), float(eps), _ptrs(ys), _ptr(mean),
                                             _ptr(rstd), s, b, h, tp, dt, _stream(stream)))


def sp_layernorm_backward_workspace(s, b, h) -> int:
    return int(load().tpmlp_sp_layernorm_backward_workspace(s, b, h))


def sp_layernorm_backward(x, gamma, mean, rstd, dy, dx, dgamma, dbeta, *, s, b, h, tp, accumulate=False,
                          workspace=None, dtype=None, stream=None) -> None:
    xs, dys, dxs = _as_list(x), _as_list(dy), _as_list(dx)
    dt = _dtype_code(dtype if dtype is not None else xs[0].dtype)
    need = sp_layernorm_backward_workspace(s, b, h)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=xs[0].device)
    _check(load().tpmlp_sp_layernorm_backward(_ptrs(xs), _ptr(gamma), _ptr(mean), _ptr(rstd), _ptrs(dys),
                                              _ptrs(dxs), int(accumulate), _ptr(dgamma), _ptr(dbeta),
                                              _ptr(workspace), workspace.numel() * workspace.element_size(), s, b, h,
                                              tp, dt, _stream(stream)))


def sp_residual_dropout_forward(r, z, keep, p, out, *, s, b, h, tp, dtype=None, stream=None) -> None:
    rs = _as_list(r)
    dt = _dtype_code(dtype if dtype is not None else rs[0].dtype)
    _check(load().tpmlp_sp_residual_dropout_forward(_ptrs(rs), _ptrs(_as_list(z)), _ptrs(_as_list(keep)), float(p),
                                                    _ptrs(_as_list(out)), s, b, h, tp, dt, _stream(stream)))


def sp_residual_dropout_backward(dout, keep, p, dz, *, s, b, h, tp, dtype=None, stream=None) -> None:
    ds = _as_list(dout)
    dt = _dtype_code(dtype if dtype is not None else ds[0].dtype)
    _check(load().tpmlp_sp_residual_dropout_backward(_ptrs(ds), _ptrs(_as_list(keep)), float(p), _ptrs(_as_list(dz)),
                                                     s, b, h, tp, dt, _stream(stream)))


def profile_start() -> None:
    """Start launch accounting on this thread (CUDA events around every launch)."""
    _check(load().tpmlp_profile_start())


def profile_stop() -> dict:
    """Stop accounting; per kernel kind: launches, summed ms, algorithmic work
    (FLOPs for the GEMMs, bytes for the copy and shard-sum kernels)."""
    pr = _Profile()
    _check(load().tpmlp_profile_stop(ctypes.byref(pr)))
    return {k: {"launches": pr.launches[i], "ms": pr.ms[i], "work": pr.work[i]} for i, k in enumerate(PROFILE_KINDS)}


# ---------------------------------------------------------------- convenience


@dataclass
class MLPBlock:
    """One block configuration; allocates outputs and workspace with torch.empty.

    f is the ffn width (F for SwiGLU).  With sp, activations are lists of tp
    chunks [s/tp, b, h]; otherwise single [s, b, h] tensors.
    """

    s: int
    b: int
    h: int
    f: int
    tp: int
    sp: bool
    dtype: torch.dtype
    act: str = "gelu"
    mode: str = "fused"
    device: str = "cuda"

    def __post_init__(self):
        self.M = self.s * self.b
        self.n1 = 2 * self.f if self.act == "swiglu" else self.f
        self.ws_bytes = workspace_size(self.s, self.b, self.h, self.f, self.tp, self.sp, self.dtype, self.act,
                                       self.mode)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=self.device)

    def act_tensor(self):
        if self.sp:
            return [torch.empty(self.s // self.tp, self.b, self.h, dtype=self.dtype, device=self.device)
                    for _ in range(self.tp)]
        return torch.empty(self.s, self.b, self.h, dtype=self.dtype, device=self.device)

    def alloc_forward(self):
        return {
            "u": torch.empty(self.M, self.n1, dtype=self.dtype, device=self.device),
            "y": torch.empty(self.M, self.f, dtype=self.dtype, device=self.device),
            "z": self.act_tensor(),
        }

    def alloc_backward(self):
        return {
            "dx": self.act_tensor(),
            "dw1": torch.empty(self.n1, self.h, dtype=self.dtype, device=self.device),
            "dw2": torch.empty(self.h, self.f, dtype=self.dtype, device=self.device),
            "du": torch.empty(self.M, self.n1, dtype=self.dtype, device=self.device),
        }

    def _kw(self):
        return dict(s=self.s, b=self.b, h=self.h, f=self.f, tp=self.tp, sp=self.sp, act=self.act, mode=self.mode,
                    workspace=self.workspace, workspace_bytes=self.workspace.numel(), dtype=self.dtype)

    def forward(self, x, w1, w2, out=None, stream=None):
        out = out or self.alloc_forward()
        forward(x, w1, w2, out["u"], out["y"], out["z"], stream=stream, **self._kw())
        return out

    def backward_main_grad(self, x, w1, w2, fwd, dz, main_grad_w1, main_grad_w2, out=None, stream=None):
        """Backward whose weight gradients are added into float32 main_grad buffers."""
        out = out or self.alloc_backward()
        backward_main_grad(x, w1, w2, fwd["u"], fwd["y"], dz, out["dx"], main_grad_w1, main_grad_w2, out["du"],
                           stream=stream, **self._kw())
        return out

    def backward(self, x, w1, w2, fwd, dz, out=None, stream=None):
        out = out or self.alloc_backward()
        backward(x, w1, w2, fwd["u"], fwd["y"], dz, out["dx"], out["dw1"], out["dw2"], out["du"], stream=stream,
                 **self._kw())
        return out


# ---------------------------------------------------------------- attention block


def attn_workspace_size(s, b, h, heads, tp, sp, dtype, causal, kv_heads=None) -> int:
    kv = heads if kv_heads is None else kv_heads
    return int(load().tpmlp_attn_workspace_size(s, b, h, heads, kv, tp, int(bool(sp)), _dtype_code(dtype),
                                                 int(bool(causal))))


def attn_forward(x, wqkv, wo, qkv, o, lse, z, *, s, b, h, heads, tp, sp, causal, kv_heads=None, workspace=None,
                 dtype=None, stream=None) -> None:
    """tpmlp_attn_forward.  x, z: lists of tp chunks under sp, else single tensors;
    kv_heads None = one key/value head per query head."""
    dt = _dtype_code(dtype if dtype is not None else wqkv.dtype)
    kv = heads if kv_heads is None else kv_heads
    _check(load().tpmlp_attn_forward(s, b, h, heads, kv, tp, int(bool(sp)), dt, int(bool(causal)), _ptrs(x),
                                     _ptr(wqkv), _ptr(wo), _ptr(qkv), _ptr(o), _ptr(lse), _ptrs(z), _ptr(workspace),
                                     0 if workspace is None else workspace.numel() * workspace.element_size(),
                                     _stream(stream)))


def attn_backward(x, wqkv, wo, qkv, o, lse, dz, dx, dwqkv, dwo, dqkv, dout, *, s, b, h, heads, tp, sp, causal,
                  workspace, kv_heads=None, dtype=None, stream=None) -> None:
    """tpmlp_attn_backward.  x, dz, dx: lists of tp chunks under sp, else single tensors."""
    dt = _dtype_code(dtype if dtype is not None else wqkv.dtype)
    kv = heads if kv_heads is None else kv_heads
    _check(load().tpmlp_attn_backward(s, b, h, heads, kv, tp, int(bool(sp)), dt, int(bool(causal)), _ptrs(x),
                                      _ptr(wqkv), _ptr(wo), _ptr(qkv), _ptr(o), _ptr(lse), _ptrs(dz), _ptrs(dx),
                                      _ptr(dwqkv), _ptr(dwo), _ptr(dqkv), _ptr(dout), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream)))


class AttnBlock:
    """One attention-block configuration; allocates outputs, saved activations and
    workspace with torch.empty (the library itself allocates nothing)."""

    def __init__(self, s, b, h, heads, tp, sp, dtype, causal, device="cuda", kv_heads=None):
        self.s, self.b, self.h, self.heads, self.tp, self.sp = s, b, h, heads, tp, bool(sp)
        self.kv_heads = heads if kv_heads is None else kv_heads
        self.dtype, self.causal, self.device = dtype, bool(causal), device
        self.M = s * b
        self.s_pad = (s + 127) // 128 * 128
        self.qkv_w = h + 2 * self.kv_heads * (h // heads)  # fused projection width h + 2·h_kv
        n = attn_workspace_size(s, b, h, heads, tp, sp, dtype, causal, self.kv_heads)
        self.ws = torch.empty(max(n, 256), dtype=torch.uint8, device=device)

    def _act(self):
        if self.sp:
            return [torch.empty(self.s // self.tp, self.b, self.h, dtype=self.dtype, device=self.device)
                    for _ in range(self.tp)]
        return torch.empty(self.s, self.b, self.h, dtype=self.dtype, device=self.device)

    def _kw(self):
        return dict(s=self.s, b=self.b, h=self.h, heads=self.heads, tp=self.tp, sp=self.sp, causal=self.causal,
                    kv_heads=self.kv_heads)

    def forward(self, x, wqkv, wo, stream=None):
        qkv = torch.empty(self.M, self.qkv_w, dtype=self.dtype, device=self.device)
        o = torch.empty(self.M, self.h, dtype=self.dtype, device=self.device)
        lse = torch.empty(self.b, self.heads, self.s_pad, dtype=torch.float32, device=self.device)
        z = self._act()
        attn_forward(x, wqkv, wo, qkv, o, lse, z, workspace=self.ws, stream=stream, **self._kw())
        return {"qkv": qkv, "o": o, "lse": lse, "z": z}

    def backward(self, x, wqkv, wo, fw, dz, stream=None):
        dx = self._act()
        dwqkv = torch.empty(self.qkv_w, self.h, dtype=self.dtype, device=self.device)
        dwo = torch.empty(self.h, self.h, dtype=self.dtype, device=self.device)
        dqkv = torch.empty(self.M, self.qkv_w, dtype=self.dtype, device=self.device)
        dout = torch.empty(self.M, self.h, dtype=self.dtype, device=self.device)
        attn_backward(x, wqkv, wo, fw["qkv"], fw["o"], fw["lse"], dz, dx, dwqkv, dwo, dqkv, dout,
                      workspace=self.ws, stream=stream, **self._kw())
        return {"dx": dx, "dwqkv": dwqkv, "dwo": dwo, "dqkv": dqkv, "dout": dout}
