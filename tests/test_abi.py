"""The C-ABI library: exports, header agreement and host-side validation (no GPU needed)."""
import ctypes
import os
import re

import pytest
import torch

import attention_flash_lora_attn_b300 as fla
from attention_flash_lora_attn_b300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from attention_flash_lora_attn_b300 import build_lib
    build_lib.build()
    return fla.load_library()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"FLA_API\s+[\w\s\*]+?\b(\w+)\s*\(", txt))
    return names


def test_header_and_binding_agree():
    assert _declared() == set(binding.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert lib.fla_status_string(0) == b"FLA_OK"
    assert lib.fla_status_string(3) == b"FLA_ERR_WORKSPACE"
    assert re.match(rb"\d+\.\d+\.\d+", lib.fla_version())


def _dims(**kw):
    base = dict(n_agents=3, hq=32, hkv=8, head_dim=128, rank=16, dtype_code=1, l_row_stride=48,
                l_agent_stride=16)
    base.update(kw)
    return binding.make_dims(base["n_agents"], base["hq"], base["hkv"], base["head_dim"], base["rank"],
                             base["dtype_code"], base["l_row_stride"], base["l_agent_stride"])


def _decode(lib, dims, n_req=1, total=16, ptr=16, ws=None, ws_bytes=0):
    p = ctypes.c_void_p(ptr)
    return lib.flash_lora_attn_decode(ctypes.byref(dims), p, p, p, p, p, p, n_req, total, p, ws, ws_bytes, None)


def test_decode_rejects_bad_shapes_without_launching(lib):
    assert _decode(lib, _dims(hq=30)) == 1            # hq % hkv
    assert "multiple of hkv" in lib.fla_last_error().decode()
    assert _decode(lib, _dims(n_agents=0)) == 1
    assert _decode(lib, _dims(head_dim=130)) == 2     # not a multiple of 4
    assert _decode(lib, _dims(rank=0)) == 2
    assert _decode(lib, _dims(l_row_stride=40)) == 1  # narrower than A*r
    assert _decode(lib, _dims(l_agent_stride=8)) == 1  # between 0 and r
    assert _decode(lib, _dims(dtype_code=7)) == 1
    assert _decode(lib, _dims(), n_req=-1) == 1
    assert _decode(lib, _dims(), ptr=0) == 1          # NULL pointers


def test_decode_workspace_checks(lib):
    d = _dims()
    need = lib.flash_lora_attn_decode_workspace_size(ctypes.byref(d), 1, 16384)
    assert need > 0
    # tensor path with a missing workspace is refused before any launch
    assert _decode(lib, d, total=16384, ws=None, ws_bytes=0) == 3
    # SIMT kernels need none
    s = _dims()
    s.kernel = 1
    assert lib.flash_lora_attn_decode_workspace_size(ctypes.byref(s), 1, 16384) == 0


def test_tensor_kernel_refuses_unsupported_shapes(lib):
    d = _dims(rank=12, l_row_stride=36, l_agent_stride=12)  # rank % 8 != 0
    d.kernel = 2
    assert _decode(lib, d) == 2
    f = _dims(dtype_code=0)
    f.kernel = 2
    assert _decode(lib, f) == 2


def test_kernel_generation_selection_is_validated(lib):
    p = ctypes.c_void_p(16)
    d = _dims()
    d.kernel = 5                                       # not a fla_kernel
    assert _decode(lib, d) == 1
    h = _dims(head_dim=64)
    h.kernel = 4                                       # the tcgen05 decode kernel needs head_dim 128
    assert _decode(lib, h) == 2
    assert "tcgen05" in lib.fla_last_error().decode()
    assert lib.lr_cache_build(p, 64, p, p, 16, 8, 64, 1, 16, 1, 3, None) == 2   # build has no mma.sync kernel
    assert lib.lr_cache_build(p, 64, p, p, 16, 8, 64, 1, 16, 0, 4, None) == 2   # fp32: outside tcgen05
    # prefill: L width A*r = 96 > 64 is outside the tcgen05 kernel; refused before any launch
    w = _dims(n_agents=3, rank=32, l_row_stride=96, l_agent_stride=32)
    w.kernel = 4
    assert lib.flash_lora_attn_prefill(ctypes.byref(w), p, p, p, p, p, 1, 20, p, None, 0, None) == 2
    assert "tcgen05" in lib.fla_last_error().decode()
    f = _dims(dtype_code=0)
    f.kernel = 3
    assert lib.flash_lora_attn_prefill(ctypes.byref(f), p, p, p, p, p, 1, 20, p, None, 0, None) == 2


def test_empty_calls_are_noops(lib):
    assert _decode(lib, _dims(), n_req=0) == 0
    d = _dims()
    p = ctypes.c_void_p(16)
    assert lib.flash_lora_attn_prefill(ctypes.byref(d), p, p, p, p, p, 0, 0, p, None, 0, None) == 0
    assert lib.lr_cache_build(p, 64, p, p, 16, 0, 64, 1, 16, 1, 0, None) == 0


def test_build_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(16)
    assert lib.lr_cache_build(p, 32, p, p, 16, 8, 64, 1, 16, 1, 0, None) == 1   # ldx < d_model
    assert lib.lr_cache_build(p, 64, p, p, 8, 8, 64, 1, 16, 1, 0, None) == 1    # ldl < n_cols
    assert lib.lr_cache_build(None, 64, p, p, 16, 8, 64, 1, 16, 1, 0, None) == 1
    assert lib.lr_cache_build(p, 64, p, p, 16, 8, 64, 1, 16, 5, 0, None) == 1   # dtype
    assert lib.lr_cache_build(p, 64, p, p, 16, 8, 64, 0, 16, 1, 0, None) == 1   # n_agents < 1
    assert lib.lr_cache_build(p, 64, p, p, 16, 8, 64, 1, 0, 1, 0, None) == 1    # rank < 1
    assert lib.lr_cache_build(p, 64, p, p, 32, 8, 64, 4, 16, 1, 0, None) == 1   # ldl < n_agents * rank


def test_rebase_projection_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(16)
    ok = (p, 64, p, p, p, p, 16, 8, 64, 1, 64, 1, 16, 1, 0, None)

    def call(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return lib.rebase_kv_lr_build(*a)
    assert call(a7=0) == 0                      # n_tokens == 0: no-op
    assert call(a1=32) == 1                     # ldx < d_model
    assert call(a6=8) == 1                      # ldl < n_agents * rank
    assert call(a0=None) == 1                   # NULL X
    assert call(a4=None) == 1                   # NULL V_base
    assert call(a9=0) == 1                      # hkv < 1
    assert call(a12=0) == 1                     # rank < 1
    assert call(a13=5) == 1                     # dtype
    assert call(a14=3) == 2                     # no mma.sync kernel
    assert call(a13=0, a14=4) == 2              # fp32 is outside the tcgen05 kernel


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_valid_call_without_gpu_reports_cuda_error(lib):
    p = ctypes.c_void_p(16)
    st = lib.lr_cache_build(p, 64, p, p, 16, 8, 64, 1, 16, 1, 1, None)
    assert st == 4


def test_value_expand_validates_on_the_host(lib):
    p, odd = ctypes.c_void_p(16), ctypes.c_void_p(8)
    d = _dims()
    assert lib.lora_value_expand(ctypes.byref(d), p, p, p, 0, p, None) == 0       # empty: no-op
    assert lib.lora_value_expand(ctypes.byref(d), p, p, p, -1, p, None) == 1      # n_tokens < 0
    assert lib.lora_value_expand(ctypes.byref(d), None, p, p, 8, p, None) == 1    # V_base NULL
    assert lib.lora_value_expand(ctypes.byref(d), p, p, p, 8, odd, None) == 1     # V_out misaligned
    assert lib.lora_value_expand(ctypes.byref(_dims(hq=30)), p, p, p, 8, p, None) == 1
    d12 = _dims(hq=8, hkv=8, head_dim=12)
    assert lib.lora_value_expand(ctypes.byref(d12), p, p, p, 8, p, None) == 2     # head_dim % 8
    big = _dims(head_dim=256, rank=256, l_row_stride=768, l_agent_stride=256)
    big.dtype = 0                                                                  # fp32: the CUDA-core kernel
    assert lib.lora_value_expand(ctypes.byref(big), p, p, p, 8, p, None) == 2     # shared memory
    d5 = _dims()
    d5.kernel = 4
    assert lib.lora_value_expand(ctypes.byref(d5), p, p, p, 8, p, None) == 2      # no tcgen05 kernel


def test_decode_host_io_validates_on_the_host(lib):
    p = ctypes.c_void_p(16)
    d = _dims()

    def call(qh=p, qd=p, od=p, oh=p, n_req=1, dims=d):
        return lib.flash_lora_attn_decode_host_io(ctypes.byref(dims), qh, qd, p, p, p, p, p, n_req, 16, od, oh,
                                                  None, 0, None)
    assert call(qh=None) == 1
    assert call(oh=None) == 1
    assert call(qd=None) == 1
    assert call(n_req=-1) == 1
    assert call(dims=_dims(hq=30)) == 1     # a decode shape check, before anything is enqueued
    assert call(n_req=0) == 0               # no queries: no-op
