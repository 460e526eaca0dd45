"""Thin ctypes binding of libqmoe.so (argument marshalling only).

Every step of the layer runs in the library's CUDA kernels; PyTorch supplies
device memory and the current stream. There is no fallback: if the library is
missing or the device is not a GB300, the calls raise.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqmoe.so")

Q4K, Q5K, Q6K, MXFP4 = 0, 1, 2, 3
QTYPE = {"q4k": Q4K, "q5k": Q5K, "q6k": Q6K, "mxfp4": MXFP4}
PATH_NAMES = {0: "none", 1: "gemv", 2: "gemm_tc", 3: "decode"}

_c_int, _c_size, _vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p


class MoeDesc(ctypes.Structure):
    _fields_ = [("H", _c_int), ("E", _c_int), ("k", _c_int), ("F", _c_int),
                ("gate_type", _c_int), ("down_type", _c_int),
                ("Wr", _vp), ("Wg", _vp), ("Wu", _vp), ("Wd", _vp),
                ("Sg", _vp), ("Su", _vp), ("Sd", _vp)]


class MoeWsLayout(ctypes.Structure):
    _fields_ = [("ids", _c_size), ("w", _c_size), ("offsets", _c_size), ("perm", _c_size),
                ("y", _c_size)]


class QmoeError(RuntimeError):
    pass


_lib = None


def lib() -> ctypes.CDLL:
    """Loads libqmoe.so (built in-tree by ``quantized_moe_transformer_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise QmoeError(f"{LIB_PATH} is not built; run quantized_moe_transformer_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER
        L.qmoe_status_str.restype = ctypes.c_char_p
        L.qmoe_status_str.argtypes = [_c_int]
        L.qmoe_query_status.argtypes = [_vp]
        L.qmoe_get_gemm_threshold.argtypes = []
        L.qmoe_set_gemm_threshold.argtypes = [_c_int]
        L.qmoe_set_gemm_threshold.restype = None
        L.qmoe_last_path.argtypes = []
        L.qmoe_moe_route_workspace_bytes.restype = _c_size
        L.qmoe_moe_route_workspace_bytes.argtypes = [_c_int] * 4
        L.qmoe_moe_route.argtypes = [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp,
                                     _c_size, _vp]
        L.qmoe_moe_workspace_bytes.restype = _c_size
        L.qmoe_moe_workspace_bytes.argtypes = [P(MoeDesc), _c_int]
        L.qmoe_moe_workspace_layout.argtypes = [P(MoeDesc), _c_int, P(MoeWsLayout)]
        L.qmoe_moe_forward.argtypes = [P(MoeDesc), _vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_size,
                                       _vp]
        L.qmoe_moe_forward_host_workspace_bytes.restype = _c_size
        L.qmoe_moe_forward_host_workspace_bytes.argtypes = [P(MoeDesc), _c_int]
        L.qmoe_moe_forward_host.argtypes = [P(MoeDesc), _vp, _vp, _vp, _c_int, _vp, _c_size, _vp]
        L.qmoe_launch_count.restype = ctypes.c_longlong
        L.qmoe_launch_count.argtypes = []
        L.qmoe_profile_start.argtypes = [_c_int]
        L.qmoe_profile_stop.argtypes = [P(ctypes.c_double), P(_c_int)]
        L.qmoe_profile_read.argtypes = [P(ctypes.c_double), P(_c_int)]
        L.qmoe_moe_forward_noalloc.argtypes = [P(MoeDesc), _vp, _vp, _vp, _c_int, _vp]
        L.qmoe_last_cuda_error.argtypes = []
        L.qmoe_get_decode_max_rows.argtypes = []
        L.qmoe_set_decode_max_rows.argtypes = [_c_int]
        L.qmoe_set_decode_max_rows.restype = None
        L.qmoe_test_inject.argtypes = [_c_int, _c_int]
        _lib = L
    return _lib


def exported_symbols() -> list[str]:
    """Names of the entry points include/qmoe.h declares."""
    return ["qmoe_status_str", "qmoe_query_status", "qmoe_get_gemm_threshold",
            "qmoe_set_gemm_threshold", "qmoe_last_path", "qmoe_moe_route_workspace_bytes",
            "qmoe_moe_route", "qmoe_moe_workspace_bytes", "qmoe_moe_workspace_layout",
            "qmoe_moe_forward", "qmoe_moe_forward_host_workspace_bytes", "qmoe_moe_forward_host",
            "qmoe_launch_count", "qmoe_profile_start", "qmoe_profile_stop", "qmoe_profile_read",
            "qmoe_moe_forward_noalloc", "qmoe_get_decode_max_rows", "qmoe_set_decode_max_rows",
            "qmoe_last_cuda_error", "qmoe_rmsnorm", "qmoe_attn_workspace_bytes", "qmoe_attn_forward", "qmoe_block_workspace_bytes",
            "qmoe_block_forward", "qmoe_test_inject"]


def _check(status: int):
    if status != 0:
        msg = f"qmoe status {status}: {lib().qmoe_status_str(status).decode()}"
        if status == -6:
            msg += f" (cudaError {int(lib().qmoe_last_cuda_error())})"
        raise QmoeError(msg)


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise QmoeError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise QmoeError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class MoeLayer:
    """Device-resident weights of one routed-MoE layer plus its descriptor."""

    def __init__(self, H, E, k, F, Wr, Wg, Wu, Wd, Sg=None, Su=None, Sd=None,
                 gate_type="q4k", down_type="q5k"):
        self.H, self.E, self.k, self.F = H, E, k, F
        self.gate_type, self.down_type = gate_type, down_type
        self.Wr, self.Wg, self.Wu, self.Wd = Wr, Wg, Wu, Wd
        self.Sg, self.Su, self.Sd = Sg, Su, Sd
        self._desc = MoeDesc(H, E, k, F, QTYPE[gate_type], QTYPE[down_type],
                             _ptr(Wr), _ptr(Wg), _ptr(Wu), _ptr(Wd),
                             _ptr(Sg), _ptr(Su), _ptr(Sd))
        self._desc_ref = ctypes.byref(self._desc)

    @classmethod
    def from_arrays(cls, layer: dict, k: int, device="cuda"):
        """From the numpy dict of ``inputs.moe_layer``."""
        dev = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device)
        return cls(layer["H"], layer["E"], k, layer["F"], dev(layer["Wr"]), dev(layer["Wg"]),
                   dev(layer["Wu"]), dev(layer["Wd"]), dev(layer.get("Sg")), dev(layer.get("Su")),
                   dev(layer.get("Sd")), layer["gate_type"], layer["down_type"])

    @property
    def desc(self) -> MoeDesc:
        return self._desc

    def workspace_bytes(self, T: int) -> int:
        return int(lib().qmoe_moe_workspace_bytes(ctypes.byref(self._desc), T))

    def workspace_layout(self, T: int) -> MoeWsLayout:
        out = MoeWsLayout()
        _check(lib().qmoe_moe_workspace_layout(ctypes.byref(self._desc), T, ctypes.byref(out)))
        return out

    def workspace(self, T: int) -> torch.Tensor:
        return torch.empty(max(self.workspace_bytes(T), 256), dtype=torch.uint8,
                           device=self.Wr.device)


def moe_route(X: torch.Tensor, Wr: torch.Tensor, k: int, ws: torch.Tensor | None = None,
              stream=None):
    """ids [T,k] int32 and w [T,k] fp32 of rows X [T,H] under router Wr [H,E]."""
    T, H = X.shape
    E = Wr.shape[1]
    ids = torch.empty((T, k), dtype=torch.int32, device=X.device)
    w = torch.empty((T, k), dtype=torch.float32, device=X.device)
    need = int(lib().qmoe_moe_route_workspace_bytes(T, H, E, k))
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=X.device)
    _check(lib().qmoe_moe_route(_ptr(X), _ptr(Wr), T, H, E, k, _ptr(ids), _ptr(w), _ptr(ws),
                                ws.numel(), _stream(stream)))
    return ids, w


def moe_forward(layer: MoeLayer, X: torch.Tensor, R: torch.Tensor | None = None,
                ids: torch.Tensor | None = None, w: torch.Tensor | None = None,
                out: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """out = R + shared(X) + sum_s w_s expert_{ids_s}(X), enqueued on ``stream``."""
    T = X.shape[0]
    if out is None:
        out = torch.empty_like(X)
    if ws is None:
        ws = layer.workspace(T)
    _check(lib().qmoe_moe_forward(ctypes.byref(layer.desc), _ptr(X), _ptr(R), _ptr(ids), _ptr(w),
                                  _ptr(out), T, _ptr(ws), ws.numel(), _stream(stream)))
    return out


FAULT_SITES = {"none": 0, "decode_copy": 1, "tc_arrive": 2, "attn_final": 3}


def test_inject(site: str, wait_us: int = 0):
    """Test-only: make the next calls withhold one copy, arrival or signal at
    ``site`` so that one bounded device wait runs out after ``wait_us``."""
    _check(lib().qmoe_test_inject(FAULT_SITES[site], int(wait_us)))


def query_status(stream=None) -> int:
    return int(lib().qmoe_query_status(_stream(stream)))


def last_path() -> str:
    return PATH_NAMES[int(lib().qmoe_last_path())]


def set_gemm_threshold(rows: int):
    lib().qmoe_set_gemm_threshold(int(rows))


def get_gemm_threshold() -> int:
    return int(lib().qmoe_get_gemm_threshold())


def set_decode_max_rows(rows: int):
    lib().qmoe_set_decode_max_rows(int(rows))


def get_decode_max_rows() -> int:
    return int(lib().qmoe_get_decode_max_rows())


STAGES = {"router": 1, "route": 2, "gateup": 3, "down": 4, "combine": 5, "decode": 6}


def moe_forward_host(layer: MoeLayer, X: torch.Tensor, R: torch.Tensor | None = None,
                     out: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """The layer on HOST tensors (pinned for asynchronous copies): the library
    copies X (and R) in, runs the layer and copies the result back, then waits."""
    T = X.shape[0]
    if out is None:
        out = torch.empty_like(X)
    if ws is None:
        n = int(lib().qmoe_moe_forward_host_workspace_bytes(ctypes.byref(layer.desc), T))
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device=layer.Wr.device)
    for t in (X, R, out):
        if t is not None and (t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous()):
            raise QmoeError("moe_forward_host takes contiguous fp32 host tensors")
    if not ws.is_cuda:
        raise QmoeError("the workspace must be on a CUDA device")
    # (a per-call path: integer addresses and the layer's cached descriptor
    # reference, converted by the argument types declared in lib())
    s = stream if stream is not None else torch.cuda.current_stream()
    _check(lib().qmoe_moe_forward_host(layer._desc_ref, X.data_ptr(), None if R is None else R.data_ptr(),
                                       out.data_ptr(), T, ws.data_ptr(), ws.numel(), s.cuda_stream))
    return out


def host_workspace_bytes(layer: MoeLayer, T: int) -> int:
    return int(lib().qmoe_moe_forward_host_workspace_bytes(ctypes.byref(layer.desc), T))


def launch_count() -> int:
    return int(lib().qmoe_launch_count())


def profile_start(stage: str):
    _check(lib().qmoe_profile_start(STAGES[stage]))


def profile_read():
    """(summed kernel milliseconds, launches) of the profiled launches as the
    last replay of a graph captured with profiling on left them."""
    ms = ctypes.c_double()
    n = _c_int()
    _check(lib().qmoe_profile_read(ctypes.byref(ms), ctypes.byref(n)))
    return ms.value, n.value


def profile_stop():
    """(summed kernel milliseconds, launches) of the profiled stage."""
    ms = ctypes.c_double()
    n = _c_int()
    _check(lib().qmoe_profile_stop(ctypes.byref(ms), ctypes.byref(n)))
    return ms.value, n.value


def moe_forward_noalloc(layer: MoeLayer, X: torch.Tensor, R: torch.Tensor | None = None,
                        out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The layer with the library's fixed device scratch instead of a caller
    workspace (for callers that cannot allocate); raises for T beyond it."""
    T = X.shape[0]
    if out is None:
        out = torch.empty_like(X)
    _check(lib().qmoe_moe_forward_noalloc(ctypes.byref(layer.desc), _ptr(X), _ptr(R), _ptr(out), T,
                                          _stream(stream)))
    return out


# ---------------------------------------------------------------- block

class BlockDesc(ctypes.Structure):
    _fields_ = [("H", _c_int), ("n_heads", _c_int), ("n_kv", _c_int), ("head_dim", _c_int),
                ("rope_theta", ctypes.c_float), ("eps", ctypes.c_float),
                ("g1", _vp), ("g2", _vp), ("Wq", _vp), ("Wk", _vp), ("Wv", _vp), ("Wo", _vp),
                ("moe", MoeDesc)]


def _block_lib():
    L = lib()
    if not getattr(L, "_block_declared", False):
        P = ctypes.POINTER
        L.qmoe_rmsnorm.argtypes = [_vp, _vp, ctypes.c_float, _vp, _c_int, _c_int, _vp]
        L.qmoe_attn_workspace_bytes.restype = _c_size
        L.qmoe_attn_workspace_bytes.argtypes = [P(BlockDesc), _c_int, _c_int]
        L.qmoe_attn_forward.argtypes = [P(BlockDesc), _vp, _vp, _vp, _c_int, _vp, _vp, _c_int, _c_int, _vp,
                                        _c_size, _vp]
        L.qmoe_block_workspace_bytes.restype = _c_size
        L.qmoe_block_workspace_bytes.argtypes = [P(BlockDesc), _c_int, _c_int]
        L.qmoe_block_forward.argtypes = [P(BlockDesc), _vp, _vp, _c_int, _vp, _vp, _c_int, _c_int, _vp,
                                         _c_size, _vp]
        L._block_declared = True
    return L


class Block:
    """Device-resident weights of one attention + MoE block and its descriptor."""

    def __init__(self, H, n_heads, n_kv, head_dim, g1, g2, Wq, Wk, Wv, Wo, moe: MoeLayer,
                 rope_theta=1e7, eps=1e-6):
        self.H, self.n_heads, self.n_kv, self.head_dim = H, n_heads, n_kv, head_dim
        self.g1, self.g2, self.Wq, self.Wk, self.Wv, self.Wo = g1, g2, Wq, Wk, Wv, Wo
        self.moe = moe
        self._desc = BlockDesc(H, n_heads, n_kv, head_dim, rope_theta, eps, _ptr(g1), _ptr(g2), _ptr(Wq),
                               _ptr(Wk), _ptr(Wv), _ptr(Wo), moe.desc)

    @classmethod
    def from_arrays(cls, blk: dict, k: int, device="cuda"):
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
        moe = MoeLayer.from_arrays(blk["moe"], k, device)
        return cls(blk["H"], blk["n_heads"], blk["n_kv"], blk["head_dim"], dev(blk["g1"]), dev(blk["g2"]),
                   dev(blk["Wq"]), dev(blk["Wk"]), dev(blk["Wv"]), dev(blk["Wo"]), moe)

    @property
    def desc(self) -> BlockDesc:
        return self._desc

    def attn_workspace(self, T, pos0):
        n = int(_block_lib().qmoe_attn_workspace_bytes(ctypes.byref(self._desc), T, pos0))
        return torch.empty(max(n, 256), dtype=torch.uint8, device=self.Wq.device)

    def workspace(self, T, pos0):
        n = int(_block_lib().qmoe_block_workspace_bytes(ctypes.byref(self._desc), T, pos0))
        return torch.empty(max(n, 256), dtype=torch.uint8, device=self.Wq.device)


def cache_from_bits(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """bf16 cache tensor from uint16 bit patterns (same bytes)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def rmsnorm(X: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6, out=None, stream=None):
    T, H = X.shape
    if out is None:
        out = torch.empty_like(X)
    _check(_block_lib().qmoe_rmsnorm(_ptr(X), _ptr(gamma), eps, _ptr(out), T, H, _stream(stream)))
    return out


def attn_forward(block: Block, X: torch.Tensor, R: torch.Tensor | None, k_cache: torch.Tensor,
                 v_cache: torch.Tensor, pos0: int, out=None, ws=None, stream=None):
    """out = R + O(attention(...)) for rows at positions pos0..pos0+T-1 (R may be None)."""
    T = X.shape[0]
    if out is None:
        out = torch.empty_like(X)
    if ws is None:
        ws = block.attn_workspace(T, pos0)
    _check(_block_lib().qmoe_attn_forward(ctypes.byref(block.desc), _ptr(X), _ptr(R), _ptr(out), T,
                                          _ptr(k_cache), _ptr(v_cache), pos0, k_cache.shape[0], _ptr(ws),
                                          ws.numel(), _stream(stream)))
    return out


def block_forward(block: Block, X: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, pos0: int,
                  out=None, ws=None, stream=None):
    T = X.shape[0]
    if out is None:
        out = torch.empty_like(X)
    if ws is None:
        ws = block.workspace(T, pos0)
    _check(_block_lib().qmoe_block_forward(ctypes.byref(block.desc), _ptr(X), _ptr(out), T, _ptr(k_cache),
                                           _ptr(v_cache), pos0, k_cache.shape[0], _ptr(ws), ws.numel(),
                                           _stream(stream)))
    return out
