"""flash_lora_attn_decode_noalloc: decode for callers that cannot allocate.

Some callers cannot allocate device memory when they call the library (a
serving loop whose memory budget is fixed at start-up, a plugin whose host
framework owns every allocation).  This entry point takes no workspace; the
split-context partials live in a fixed 16 MiB array inside the library.  The
test calls it through the C ABI twice in a row and compares each result with
the regular entry point's (which gets a caller-provided workspace), within
the tolerance the parity tests use.  It must pass alone in a fresh process
and after the other tests, so it builds and loads the library itself.
"""
import ctypes

import numpy as np
import pytest
import torch

from workloads import WORKLOADS, make_decode_inputs

pytestmark = pytest.mark.gpu

ATOL, RTOL_L2 = 1e-2, 5e-3


@pytest.fixture(scope="module")
def fla():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from attention_flash_lora_attn_b300 import build_lib
    build_lib.build()
    import attention_flash_lora_attn_b300 as m
    m.load_library()
    return m


def _close(a, b):
    a, b = a.double().cpu().numpy(), b.double().cpu().numpy()
    assert np.isfinite(a).all()
    max_abs = float(np.abs(a - b).max())
    rel = float(np.linalg.norm(a - b) / np.linalg.norm(b))
    assert max_abs <= ATOL and rel <= RTOL_L2, (max_abs, rel)


def _noalloc(fla, x, rank, O):
    from attention_flash_lora_attn_b300 import binding
    lib = fla.load_library()
    R, A, hq, d = x["Q"].shape
    N, hkv, _ = x["K_base"].shape
    dims = binding.make_dims(A, hq, hkv, d, rank, binding.FLA_BF16, x["L"].stride(0), rank, None, "auto")
    st = lib.flash_lora_attn_decode_noalloc(
        ctypes.byref(dims), x["Q"].data_ptr(), x["K_base"].data_ptr(), x["V_base"].data_ptr(), x["L"].data_ptr(),
        x["B"].data_ptr(), x["offsets"].data_ptr(), R, N, O.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.fla_last_error_message()
    return O


@pytest.mark.parametrize("name,lengths", [("llama8b_decode", None), ("llama8b_decode", [3000, 17, 1, 9000])],
                         ids=["single-request", "ragged"])
def test_noalloc_matches_workspace_decode_twice(fla, name, lengths):
    w = WORKLOADS[name]
    x = {k: v.cuda() for k, v in make_decode_inputs(w, seed=21, lengths=lengths).items()}
    ws = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    ref = fla.flash_lora_attn_decode(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], x["offsets"], rank=w.rank,
                                     workspace=ws)
    for _ in range(2):  # two calls in a row share the fixed scratch array
        O = torch.full_like(ref, float("nan"))
        _noalloc(fla, x, w.rank, O)
        torch.cuda.synchronize()
        _close(O, ref)
    assert fla.device_error() == 0


def test_noalloc_rejects_calls_needing_more_scratch(fla):
    from attention_flash_lora_attn_b300 import binding
    lib = fla.load_library()
    dims = binding.make_dims(3, 32, 8, 128, 16, binding.FLA_BF16, 48, 16, None, "auto")
    p = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    st = lib.flash_lora_attn_decode_noalloc(ctypes.byref(dims), p, p, p, p, p, p, 4096, 1 << 30, p, None)
    assert st == 3  # FLA_ERR_WORKSPACE
    assert b"16777216" in lib.fla_last_error_message()
