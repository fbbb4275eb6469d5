"""ctypes binding over the C ABI in include/flash_lora_attn.h.

Argument marshalling only: every tensor must already live on the current
CUDA device; the functions pass data pointers, strides and the current torch
stream to the library, which enqueues its own kernels.  There is no CPU or
PyTorch fallback: if libflashlora.so is missing or a call fails, an
exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libflashlora.so")

FLA_OK = 0
FLA_F32, FLA_BF16 = 0, 1
KERNELS = {"auto": 0, "simt": 1, "tensor": 2, "mma": 3, "tcgen05": 4}
STATUS = {0: "FLA_OK", 1: "FLA_ERR_INVALID_ARG", 2: "FLA_ERR_UNSUPPORTED", 3: "FLA_ERR_WORKSPACE",
          4: "FLA_ERR_CUDA", 5: "FLA_ERR_DEVICE_TIMEOUT"}

# Every symbol the header declares (tests check that the library exports them).
EXPORTED = ("lr_cache_build", "flash_lora_attn_decode_workspace_size", "flash_lora_attn_decode",
            "flash_lora_attn_prefill_workspace_size", "flash_lora_attn_prefill", "fla_status_string",
            "fla_last_error", "fla_device_error", "fla_version", "flash_lora_attn_decode_noalloc",
            "lora_value_expand", "flash_lora_attn_decode_host_io", "rebase_kv_lr_build",
            "fla_selftest_bounded_wait")


class FlaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class AttnDims(ctypes.Structure):
    _fields_ = [("n_agents", ctypes.c_int32), ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("rank", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("l_row_stride", ctypes.c_int64), ("l_agent_stride", ctypes.c_int64),
                ("softmax_scale", ctypes.c_float), ("kernel", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libflashlora.so (built by build_lib.py); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it with "
                              "`python -m attention_flash_lora_attn_b300.build_lib`")
        lib = ctypes.CDLL(path)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        dims_p = ctypes.POINTER(AttnDims)
        lib.lr_cache_build.argtypes = [vp, i64, vp, vp, i64, i64, i32, i32, i32, i32, i32, vp]
        lib.lr_cache_build.restype = ctypes.c_int
        lib.rebase_kv_lr_build.argtypes = [vp, i64, vp, vp, vp, vp, i64, i64, i32, i32, i32, i32, i32, i32, i32, vp]
        lib.rebase_kv_lr_build.restype = ctypes.c_int
        lib.flash_lora_attn_decode_workspace_size.argtypes = [dims_p, i32, i64]
        lib.flash_lora_attn_decode_workspace_size.restype = sz
        lib.flash_lora_attn_decode.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, i32, i64, vp, vp, sz, vp]
        lib.flash_lora_attn_decode.restype = ctypes.c_int
        lib.flash_lora_attn_prefill_workspace_size.argtypes = [dims_p, i32, i64]
        lib.flash_lora_attn_prefill_workspace_size.restype = sz
        lib.flash_lora_attn_prefill.argtypes = [dims_p, vp, vp, vp, vp, vp, i64, i32, vp, vp, sz, vp]
        lib.flash_lora_attn_prefill.restype = ctypes.c_int
        lib.fla_status_string.argtypes = [ctypes.c_int]
        lib.fla_status_string.restype = ctypes.c_char_p
        lib.fla_last_error.argtypes = []
        lib.fla_last_error.restype = ctypes.c_char_p
        lib.fla_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
        lib.fla_device_error.restype = ctypes.c_int
        lib.fla_version.argtypes = []
        lib.fla_version.restype = ctypes.c_char_p
        lib.flash_lora_attn_decode_noalloc.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, i32, i64, vp, vp]
        lib.flash_lora_attn_decode_noalloc.restype = ctypes.c_int
        lib.lora_value_expand.argtypes = [dims_p, vp, vp, vp, i64, vp, vp]
        lib.lora_value_expand.restype = ctypes.c_int
        lib.flash_lora_attn_decode_host_io.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, vp, i32, i64, vp, vp, vp,
                                                       sz, vp]
        lib.flash_lora_attn_decode_host_io.restype = ctypes.c_int
        lib.fla_selftest_bounded_wait.argtypes = [ctypes.c_uint64, vp, vp]
        lib.fla_selftest_bounded_wait.restype = ctypes.c_int
        _lib = lib
        return lib


def _check(status: int):
    if status != FLA_OK:
        msg = load_library().fla_last_error().decode(errors="replace")
        raise FlaError(status, msg)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return FLA_F32
    if t.dtype == torch.bfloat16:
        return FLA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: use torch.bfloat16 or torch.float32")


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors on the current device")


def _dense(t: torch.Tensor, name: str):
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# Workspaces cached per (device, stream): calls on one stream are ordered, so
# they can share one.
_workspaces = {}


def _workspace(nbytes: int, device: torch.device, stream_ptr: int) -> torch.Tensor:
    key = (device.index, stream_ptr)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def make_dims(n_agents, hq, hkv, head_dim, rank, dtype_code, l_row_stride, l_agent_stride,
              scale=None, kernel="auto") -> AttnDims:
    return AttnDims(n_agents, hq, hkv, head_dim, rank, dtype_code, l_row_stride, l_agent_stride,
                    0.0 if scale is None else float(scale), KERNELS[kernel])


def lr_cache_build(X: torch.Tensor, A_cat: torch.Tensor, L: Optional[torch.Tensor] = None, *,
                   n_agents: int = 1, kernel: str = "auto", stream=None) -> torch.Tensor:
    """L = X . A_cat for every agent at once (A_cat = [A_1 | ... | A_A], [D, A*r]).

    X [n, D] (rows may be strided), A_cat [D, A*r] contiguous, L [n, A*r]
    (rows may be strided; a column slice of a wider tensor is allowed).
    `n_agents` splits the A*r columns into agents' blocks of rank A*r/n_agents
    (the product is the same; it only names the blocks at the C ABI).
    """
    lib = load_library()
    _need_cuda(X, A_cat, L)
    n, D = X.shape
    D2, N = A_cat.shape
    if D2 != D:
        raise ValueError("A_cat must be [d_model, n_agents * rank]")
    if n_agents < 1 or N % n_agents != 0:
        raise ValueError("the A_cat columns must split evenly into n_agents blocks")
    if L is None:
        L = torch.empty((n, N), dtype=X.dtype, device=X.device)
    if X.stride(1) != 1 or L.stride(1) != 1:
        raise ValueError("X and L must have unit column stride")
    if tuple(L.shape) != (n, N):
        raise ValueError("L must be [n_tokens, n_agents * rank]")
    _dense(A_cat, "A_cat")
    if not (X.dtype == A_cat.dtype == L.dtype):
        raise TypeError("X, A_cat and L must share one dtype")
    _check(lib.lr_cache_build(X.data_ptr(), X.stride(0), A_cat.data_ptr(), L.data_ptr(), L.stride(0), n, D,
                              n_agents, N // n_agents, _dtype_code(X), KERNELS[kernel], _stream_ptr(stream)))
    return L


def rebase_kv_lr_build(X: torch.Tensor, W_cat: torch.Tensor, *, hkv: int, head_dim: int, n_agents: int,
                       rank: int, K_base: Optional[torch.Tensor] = None, V_base: Optional[torch.Tensor] = None,
                       L: Optional[torch.Tensor] = None, kernel: str = "auto", stream=None):
    """[K_base | V_base | L] = X . [W_k | W_v | A_cat] in one pass over X.

    X [n, D] (rows may be strided); W_cat [D, 2*hkv*head_dim + n_agents*rank]
    contiguous; K_base, V_base [n, hkv, head_dim] contiguous; L [n, A*r] with
    unit column stride.  Returns (K_base, V_base, L).
    """
    lib = load_library()
    _need_cuda(X, W_cat, K_base, V_base, L)
    n, D = X.shape
    kv, lr = hkv * head_dim, n_agents * rank
    if tuple(W_cat.shape) != (D, 2 * kv + lr):
        raise ValueError("W_cat must be [d_model, 2*hkv*head_dim + n_agents*rank]")
    _dense(W_cat, "W_cat")
    if K_base is None:
        K_base = torch.empty((n, hkv, head_dim), dtype=X.dtype, device=X.device)
    if V_base is None:
        V_base = torch.empty((n, hkv, head_dim), dtype=X.dtype, device=X.device)
    if L is None:
        L = torch.empty((n, lr), dtype=X.dtype, device=X.device)
    for t, nm in ((K_base, "K_base"), (V_base, "V_base")):
        _dense(t, nm)
        if tuple(t.shape) != (n, hkv, head_dim):
            raise ValueError(f"{nm} must be [n_tokens, hkv, head_dim]")
    if X.stride(1) != 1 or L.stride(1) != 1 or tuple(L.shape) != (n, lr):
        raise ValueError("X and L need unit column stride; L must be [n_tokens, n_agents*rank]")
    if not (X.dtype == W_cat.dtype == K_base.dtype == V_base.dtype == L.dtype):
        raise TypeError("X, W_cat and the outputs must share one dtype")
    _check(lib.rebase_kv_lr_build(X.data_ptr(), X.stride(0), W_cat.data_ptr(), K_base.data_ptr(), V_base.data_ptr(),
                                  L.data_ptr(), L.stride(0), n, D, hkv, head_dim, n_agents, rank, _dtype_code(X),
                                  KERNELS[kernel], _stream_ptr(stream)))
    return K_base, V_base, L


def flash_lora_attn_decode(Q, K_base, V_base, L, B, offsets, *, rank: int,
                           l_agent_stride: Optional[int] = None, scale: Optional[float] = None,
                           O: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                           kernel: str = "auto", stream=None) -> torch.Tensor:
    """Decode attention over a packed ragged base cache (see the header for layouts).

    Q [R, A, Hq, d]; K_base, V_base [N, Hkv, d]; L [N, ldL] (unit column
    stride); B [A, r, Hkv*d]; offsets int32 [R+1] on the device.  Returns O
    fp32 [R, A, Hq, d].
    """
    lib = load_library()
    _need_cuda(Q, K_base, V_base, L, B, offsets, O, workspace)
    for t, nm in ((Q, "Q"), (K_base, "K_base"), (V_base, "V_base"), (B, "B")):
        _dense(t, nm)
    if L.stride(1) != 1:
        raise ValueError("L must have unit column stride")
    if offsets.dtype != torch.int32 or not offsets.is_contiguous():
        raise TypeError("offsets must be a contiguous int32 tensor")
    R, A, hq, d = Q.shape
    N, hkv, d2 = K_base.shape
    if d2 != d or V_base.shape != K_base.shape:
        raise ValueError("K_base/V_base must be [N, Hkv, d] matching Q")
    if l_agent_stride is None:
        l_agent_stride = rank
    dims = make_dims(A, hq, hkv, d, rank, _dtype_code(Q), L.stride(0), l_agent_stride, scale, kernel)
    if O is None:
        O = torch.empty((R, A, hq, d), dtype=torch.float32, device=Q.device)
    sp = _stream_ptr(stream)
    need = lib.flash_lora_attn_decode_workspace_size(ctypes.byref(dims), R, N)
    if workspace is None and need > 0:
        workspace = _workspace(need, Q.device, sp)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.flash_lora_attn_decode(ctypes.byref(dims), Q.data_ptr(), K_base.data_ptr(), V_base.data_ptr(),
                                      L.data_ptr(), B.data_ptr(), offsets.data_ptr(), R, N, O.data_ptr(),
                                      ws_ptr, ws_bytes, sp))
    return O


class PreparedDecode:
    """A decode call marshalled once: calling it enqueues the kernels with one C call.

    For serving loops that decode many times over the same buffers (the
    queries are refreshed in place, e.g. by a host->device copy into Q):
    validation, the dims struct, the workspace and the stream are fixed at
    construction, so each call costs one ctypes call.  Arguments as for
    flash_lora_attn_decode.
    """

    def __init__(self, Q, K_base, V_base, L, B, offsets, *, rank: int, l_agent_stride: Optional[int] = None,
                 scale: Optional[float] = None, O: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None, kernel: str = "auto", stream=None):
        lib = load_library()
        _need_cuda(Q, K_base, V_base, L, B, offsets, O, workspace)
        for t, nm in ((Q, "Q"), (K_base, "K_base"), (V_base, "V_base"), (B, "B")):
            _dense(t, nm)
        if L.stride(1) != 1:
            raise ValueError("L must have unit column stride")
        if offsets.dtype != torch.int32 or not offsets.is_contiguous():
            raise TypeError("offsets must be a contiguous int32 tensor")
        R, A, hq, d = Q.shape
        N, hkv, d2 = K_base.shape
        if d2 != d or V_base.shape != K_base.shape:
            raise ValueError("K_base/V_base must be [N, Hkv, d] matching Q")
        if l_agent_stride is None:
            l_agent_stride = rank
        self.dims = make_dims(A, hq, hkv, d, rank, _dtype_code(Q), L.stride(0), l_agent_stride, scale, kernel)
        self.O = O if O is not None else torch.empty((R, A, hq, d), dtype=torch.float32, device=Q.device)
        sp = _stream_ptr(stream)
        need = lib.flash_lora_attn_decode_workspace_size(ctypes.byref(self.dims), R, N)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=Q.device)
        self._keep = (Q, K_base, V_base, L, B, offsets, workspace)  # keep the buffers alive
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        self._fn = lib.flash_lora_attn_decode
        self._args = (ctypes.byref(self.dims), Q.data_ptr(), K_base.data_ptr(), V_base.data_ptr(), L.data_ptr(),
                      B.data_ptr(), offsets.data_ptr(), R, N, self.O.data_ptr(), ws_ptr, ws_bytes, sp)

    def __call__(self) -> torch.Tensor:
        st = self._fn(*self._args)
        if st != FLA_OK:
            _check(st)
        return self.O


class PreparedDecodeHostIO:
    """A host-buffer decode marshalled once (flash_lora_attn_decode_host_io).

    Each call enqueues the copy Q_host -> Q_dev, the decode into O_dev and the
    copy O_dev -> O_host with one C call.  Q_host and O_host are CPU tensors
    (pin them for asynchronous copies); O_host is valid once the stream has
    passed the call.  Other arguments as for flash_lora_attn_decode.
    """

    def __init__(self, Q_host, Q_dev, K_base, V_base, L, B, offsets, *, rank: int, O_dev, O_host,
                 l_agent_stride: Optional[int] = None, scale: Optional[float] = None,
                 workspace: Optional[torch.Tensor] = None, kernel: str = "auto", stream=None):
        lib = load_library()
        _need_cuda(Q_dev, K_base, V_base, L, B, offsets, O_dev, workspace)
        if Q_host.is_cuda or O_host.is_cuda:
            raise ValueError("Q_host and O_host must be host (CPU) tensors")
        for t, nm in ((Q_host, "Q_host"), (Q_dev, "Q_dev"), (K_base, "K_base"), (V_base, "V_base"), (B, "B"),
                      (O_dev, "O_dev"), (O_host, "O_host")):
            _dense(t, nm)
        if Q_host.shape != Q_dev.shape or Q_host.dtype != Q_dev.dtype:
            raise ValueError("Q_host and Q_dev must have the same shape and dtype")
        R, A, hq, d = Q_dev.shape
        if tuple(O_dev.shape) != (R, A, hq, d) or O_dev.dtype != torch.float32 or O_host.shape != O_dev.shape \
                or O_host.dtype != torch.float32:
            raise ValueError("O_dev and O_host must be fp32 [R, A, Hq, d]")
        if L.stride(1) != 1:
            raise ValueError("L must have unit column stride")
        N, hkv, _ = K_base.shape
        if l_agent_stride is None:
            l_agent_stride = rank
        self.dims = make_dims(A, hq, hkv, d, rank, _dtype_code(Q_dev), L.stride(0), l_agent_stride, scale, kernel)
        sp = _stream_ptr(stream)
        need = lib.flash_lora_attn_decode_workspace_size(ctypes.byref(self.dims), R, N)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=Q_dev.device)
        self.O_host = O_host
        self._keep = (Q_host, Q_dev, K_base, V_base, L, B, offsets, O_dev, O_host, workspace)
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        self._fn = lib.flash_lora_attn_decode_host_io
        self._args = (ctypes.byref(self.dims), Q_host.data_ptr(), Q_dev.data_ptr(), K_base.data_ptr(),
                      V_base.data_ptr(), L.data_ptr(), B.data_ptr(), offsets.data_ptr(), R, N, O_dev.data_ptr(),
                      O_host.data_ptr(), ws_ptr, ws_bytes, sp)

    def __call__(self) -> torch.Tensor:
        st = self._fn(*self._args)
        if st != FLA_OK:
            _check(st)
        return self.O_host


def flash_lora_attn_prefill(Q, K_base, V_base, L, B, n0: int, *, rank: int,
                            l_agent_stride: Optional[int] = None, scale: Optional[float] = None,
                            O: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                            kernel: str = "auto", stream=None) -> torch.Tensor:
    """Causal chunked prefill: Q [A, c, Hq, d]; K_base, V_base [n0+c, Hkv, d]; L [n0+c, ldL]."""
    lib = load_library()
    _need_cuda(Q, K_base, V_base, L, B, O, workspace)
    for t, nm in ((Q, "Q"), (K_base, "K_base"), (V_base, "V_base"), (B, "B")):
        _dense(t, nm)
    if L.stride(1) != 1:
        raise ValueError("L must have unit column stride")
    A, c, hq, d = Q.shape
    N, hkv, _ = K_base.shape
    if N < n0 + c:
        raise ValueError("K_base must hold n0 + chunk tokens")
    if l_agent_stride is None:
        l_agent_stride = rank
    dims = make_dims(A, hq, hkv, d, rank, _dtype_code(Q), L.stride(0), l_agent_stride, scale, kernel)
    if O is None:
        O = torch.empty((A, c, hq, d), dtype=torch.float32, device=Q.device)
    sp = _stream_ptr(stream)
    need = lib.flash_lora_attn_prefill_workspace_size(ctypes.byref(dims), c, n0)
    if workspace is None and need > 0:
        workspace = _workspace(need, Q.device, sp)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.flash_lora_attn_prefill(ctypes.byref(dims), Q.data_ptr(), K_base.data_ptr(), V_base.data_ptr(),
                                       L.data_ptr(), B.data_ptr(), n0, c, O.data_ptr(), ws_ptr, ws_bytes, sp))
    return O


def lora_value_expand(V_base, L, B, *, rank: int, l_agent_stride: Optional[int] = None,
                      V_out: Optional[torch.Tensor] = None, kernel: str = "auto", stream=None) -> torch.Tensor:
    """Every agent's materialised value cache V_i = V_base + L_i . B_i (the form
    the reordered attention avoids; used by the naive-materialisation baseline).

    V_base [N, Hkv, d]; L [N, ldL] (unit column stride); B [A, r, Hkv*d].
    Returns V_out [A, N, Hkv, d] in V_base's dtype.
    """
    lib = load_library()
    _need_cuda(V_base, L, B, V_out)
    _dense(V_base, "V_base")
    _dense(B, "B")
    if L.stride(1) != 1:
        raise ValueError("L must have unit column stride")
    N, hkv, d = V_base.shape
    A = B.shape[0]
    if tuple(B.shape) != (A, rank, hkv * d):
        raise ValueError("B must be [A, r, Hkv*d]")
    if not (V_base.dtype == L.dtype == B.dtype):
        raise TypeError("V_base, L and B must share one dtype")
    if l_agent_stride is None:
        l_agent_stride = rank
    if V_out is None:
        V_out = torch.empty((A, N, hkv, d), dtype=V_base.dtype, device=V_base.device)
    elif tuple(V_out.shape) != (A, N, hkv, d) or V_out.dtype != V_base.dtype or not V_out.is_contiguous():
        raise ValueError("V_out must be a contiguous [A, N, Hkv, d] tensor of V_base's dtype")
    dims = make_dims(A, hkv, hkv, d, rank, _dtype_code(V_base), L.stride(0), l_agent_stride, kernel=kernel)
    _check(lib.lora_value_expand(ctypes.byref(dims), V_base.data_ptr(), L.data_ptr(), B.data_ptr(), N,
                                 V_out.data_ptr(), _stream_ptr(stream)))
    return V_out


def device_error() -> int:
    """Synchronise, then read and clear the library's device error word (0 = none)."""
    lib = load_library()
    code = ctypes.c_uint32(0)
    _check(lib.fla_device_error(ctypes.byref(code)))
    return code.value


def selftest_bounded_wait(limit_ns: int, stream=None) -> dict:
    """Runs the bounded-wait self-test (a wait that nothing completes, limited to
    limit_ns) and returns what the kernel observed plus the device error code it
    left (read and cleared)."""
    lib = load_library()
    out = torch.zeros(3, dtype=torch.int64, device="cuda")
    _check(lib.fla_selftest_bounded_wait(int(limit_ns), out.data_ptr(), _stream_ptr(stream)))
    code = device_error()  # synchronises
    o = out.cpu().tolist()
    return {"timed_out": bool(o[0]), "peer_left_on_abort": bool(o[1]), "wait_ns": int(o[2]), "device_error": code}


def version() -> str:
    return load_library().fla_version().decode()
