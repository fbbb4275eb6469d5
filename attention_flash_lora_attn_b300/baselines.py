"""Baselines the reordered decode is measured against (not part of the hot path).

* Naive materialisation (LRAgent technical summary, Metodologia section 3,
  Problema bullet): every agent's value cache V_i = V_base + L_i . B_i is
  expanded to full width (`lora_value_expand`), then each agent runs plain
  attention over its own V_i.
* Non-shared caches (LRAgent summary, section 2, the setting the shared base
  cache improves on): every agent keeps a full K / V cache of the context and
  runs plain attention over it.

Plain attention here is the library's decode call for one agent with a zero
LoRA term (B = 0 over a zero LR cache of rank 16, which the tensor-core
decode accepts): O = softmax(q . K^T * scale) . V.  That zero LR cache adds
32 bytes per token to the 2 * Hkv * d * 2 bytes of K and V it reads.
Every step runs in the library's kernels; these functions only marshal
arguments (and, for several requests, slice Q and O per agent with torch).
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from .binding import (
    PreparedDecode,
    _check,
    _dtype_code,
    _stream_ptr,
    flash_lora_attn_decode,
    load_library,
    lora_value_expand,
    make_dims,
)

ZERO_RANK = 16
_zeros = {}


def _zero_lora(n_tokens: int, hkv: int, d: int, dtype, device):
    """Zero LR cache [N, 16] and zero B [1, 16, Hkv*d] (cached per shape)."""
    key = (device.index, dtype, n_tokens, hkv * d)
    z = _zeros.get(key)
    if z is None:
        z = (torch.zeros((max(n_tokens, 1), ZERO_RANK), dtype=dtype, device=device),
             torch.zeros((1, ZERO_RANK, hkv * d), dtype=dtype, device=device))
        _zeros[key] = z
    return z


def per_agent_decode(Q, K: Sequence[torch.Tensor], V: Sequence[torch.Tensor], offsets, *,
                     scale: Optional[float] = None, O: Optional[torch.Tensor] = None,
                     kernel: str = "auto", stream=None) -> torch.Tensor:
    """Plain attention for each agent a over its own cache K[a], V[a] ([N, Hkv, d] each).

    Q [R, A, Hq, d]; offsets int32 [R+1] on the device.  Returns O fp32
    [R, A, Hq, d] with O[q, a] = softmax(Q[q, a] . K[a]^T * scale) . V[a].
    """
    R, A, hq, d = Q.shape
    if len(K) != A or len(V) != A:
        raise ValueError("K and V must hold one cache per agent")
    N, hkv, _ = K[0].shape
    L0, B0 = _zero_lora(N, hkv, d, Q.dtype, Q.device)
    if O is None:
        O = torch.empty((R, A, hq, d), dtype=torch.float32, device=Q.device)
    for a in range(A):
        qa = Q[:, a:a + 1]
        oa = O[:, a:a + 1]
        direct = qa.is_contiguous() and oa.is_contiguous()
        if not direct:
            qa = qa.contiguous()
            oa = torch.empty((R, 1, hq, d), dtype=torch.float32, device=Q.device)
        flash_lora_attn_decode(qa, K[a], V[a], L0[:max(N, 1)], B0, offsets, rank=ZERO_RANK, l_agent_stride=0,
                               scale=scale, O=oa, kernel=kernel, stream=stream)
        if not direct:
            O[:, a:a + 1].copy_(oa)
    return O


def naive_materialised_decode(Q, K_base, V_base, L, B, offsets, *, rank: int,
                              l_agent_stride: Optional[int] = None, scale: Optional[float] = None,
                              O: Optional[torch.Tensor] = None, V_i: Optional[torch.Tensor] = None,
                              kernel: str = "auto", stream=None) -> torch.Tensor:
    """Decode without the reordering: expand every V_i, then plain attention per agent.

    Same arguments and result as `flash_lora_attn_decode`.  V_i, if given, is
    the [A, N, Hkv, d] buffer the expansion writes.
    """
    V_i = lora_value_expand(V_base, L, B, rank=rank, l_agent_stride=l_agent_stride, V_out=V_i, stream=stream)
    A = Q.shape[1]
    return per_agent_decode(Q, [K_base] * A, [V_i[a] for a in range(A)], offsets, scale=scale, O=O,
                            kernel=kernel, stream=stream)


class PreparedBaselineDecode:
    """Either baseline marshalled once for a single request (R = 1): one C call
    for the expansion and one per agent, for timing loops.

    mode "naive": expand V_i from (V_base, L, B), then plain attention per
    agent over (K_base, V_i).  mode "non_shared": plain attention per agent
    over that agent's own (K[a], V[a]); L and B are not used.
    """

    def __init__(self, mode: str, Q, offsets, *, K_base=None, V_base=None, L=None, B=None, rank: int = 0,
                 l_agent_stride: Optional[int] = None, K: Optional[Sequence[torch.Tensor]] = None,
                 V: Optional[Sequence[torch.Tensor]] = None, O: Optional[torch.Tensor] = None,
                 kernel: str = "auto", stream=None):
        R, A, hq, d = Q.shape
        if R != 1:
            raise ValueError("PreparedBaselineDecode serves one request (R = 1)")
        if O is None:
            O = torch.empty((R, A, hq, d), dtype=torch.float32, device=Q.device)
        self.O = O
        self.V_i = None
        self.expand = None
        if mode == "naive":
            N, hkv, _ = K_base.shape
            if l_agent_stride is None:
                l_agent_stride = rank
            self.V_i = torch.empty((A, N, hkv, d), dtype=V_base.dtype, device=V_base.device)
            self._dims = make_dims(A, hkv, hkv, d, rank, _dtype_code(V_base), L.stride(0), l_agent_stride)
            fn = load_library().lora_value_expand
            args = (ctypes.byref(self._dims), V_base.data_ptr(), L.data_ptr(), B.data_ptr(), N,
                    self.V_i.data_ptr(), _stream_ptr(stream))

            def expand():
                st = fn(*args)
                if st != 0:
                    _check(st)
            self.expand = expand
            K = [K_base] * A
            V = [self.V_i[a] for a in range(A)]
        elif mode != "non_shared":
            raise ValueError("mode must be 'naive' or 'non_shared'")
        N, hkv, _ = K[0].shape
        L0, B0 = _zero_lora(N, hkv, d, Q.dtype, Q.device)
        self._calls = [PreparedDecode(Q[:, a:a + 1], K[a], V[a], L0[:max(N, 1)], B0, offsets, rank=ZERO_RANK,
                                      l_agent_stride=0, O=O[:, a:a + 1], kernel=kernel, stream=stream)
                       for a in range(A)]
        self._keep = (Q, offsets, K_base, V_base, L, B, K, V)

    def __call__(self) -> torch.Tensor:
        if self.expand is not None:
            self.expand()
        for c in self._calls:
            c()
        return self.O
