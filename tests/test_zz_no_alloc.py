"""flash_lora_attn_decode_noalloc: decode for callers that cannot allocate.

Some callers cannot allocate device memory when they call the library (a
serving loop whose memory budget is fixed at start-up, a plugin whose host
framework owns every allocation).  This entry point takes no workspace; the
split-context partials live in a fixed 16 MiB array inside the library.  The
test calls it through the C ABI twice in a row and compares each result with
the regular entry point's (which gets a caller-provided workspace) and with
the fp64 oracle, within the tolerance the parity tests use, on both decode
kernels (12 query rows per kv head: mma.sync; 40: tcgen05, whose partial
records are laid out differently).  It must pass alone in a fresh process and
after the other tests, so it builds and loads the library itself.
"""
import ctypes

import numpy as np
import pytest
import torch

import dataclasses

import oracle
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
    assert st == 0, lib.fla_last_error()
    return O


CASES = {
    "mma-single-request": (WORKLOADS["llama8b_decode"], None),
    "mma-ragged": (WORKLOADS["llama8b_decode"], [3000, 17, 1, 9000]),
    "tcgen05-70b-group": (dataclasses.replace(WORKLOADS["llama70b_decode"], lengths=(6000,)), None),
    "tcgen05-ragged": (dataclasses.replace(WORKLOADS["llama70b_decode"], lengths=(1000, 0, 200)), None),
}


@pytest.mark.parametrize("case", list(CASES))
def test_noalloc_matches_workspace_decode_and_oracle_twice(fla, case):
    w, lengths = CASES[case]
    xh = make_decode_inputs(w, seed=21, lengths=lengths)
    x = {k: v.cuda() for k, v in xh.items()}
    ws = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    ref = fla.flash_lora_attn_decode(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], x["offsets"], rank=w.rank,
                                     workspace=ws)
    want = oracle.decode(xh["Q"], xh["K_base"], xh["V_base"], xh["L"], xh["B"], xh["offsets"].numpy(),
                         rank=w.rank)
    for _ in range(2):  # two calls in a row share the fixed scratch array
        O = torch.full_like(ref, float("nan"))
        _noalloc(fla, x, w.rank, O)
        torch.cuda.synchronize()
        _close(O, ref)
        _close(O, torch.from_numpy(want))
    assert fla.device_error() == 0


def test_noalloc_rejects_calls_needing_more_scratch(fla):
    from attention_flash_lora_attn_b300 import binding
    lib = fla.load_library()
    dims = binding.make_dims(3, 32, 8, 128, 16, binding.FLA_BF16, 48, 16, None, "auto")
    p = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    st = lib.flash_lora_attn_decode_noalloc(ctypes.byref(dims), p, p, p, p, p, p, 4096, 1 << 30, p, None)
    assert st == 3  # FLA_ERR_WORKSPACE
    assert b"16777216" in lib.fla_last_error()
