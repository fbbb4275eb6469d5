"""Failure detection without a GPU fault: the bounded waits.

Every pipeline kernel waits on mbarriers through one bounded helper; when a
wait runs out it records a code in the device error word, raises its CTA's
abort flag (so the CTA's other roles stop waiting) and returns.  The self-test
entry point runs that helper on a barrier nothing completes, with a short
limit, and a second waiter with the kernels' own limit that must leave through
the abort flag.  Afterwards the context must still be usable: a decode runs and
matches the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import WORKLOADS, make_decode_inputs

pytestmark = pytest.mark.gpu

SELFTEST_CODE = 0x401


@pytest.fixture(scope="module")
def fla():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from attention_flash_lora_attn_b300 import build_lib
    build_lib.build()
    import attention_flash_lora_attn_b300 as m
    m.load_library()
    assert m.device_error() == 0
    yield m
    assert m.device_error() == 0


@pytest.mark.parametrize("limit_ms", [1, 20])
def test_a_wait_nothing_completes_times_out_and_reports(fla, limit_ms):
    r = fla.selftest_bounded_wait(limit_ms * 1_000_000)
    assert r["timed_out"], r
    assert r["peer_left_on_abort"], r
    assert r["device_error"] == SELFTEST_CODE, r
    # the wait lasted its limit, not the kernels' 2 s
    assert limit_ms * 1e6 <= r["wait_ns"] < limit_ms * 1e6 + 50e6, r
    assert fla.device_error() == 0  # read-and-clear left it clean


def test_the_context_is_usable_after_a_timeout(fla):
    r = fla.selftest_bounded_wait(2_000_000)
    assert r["timed_out"] and r["device_error"] == SELFTEST_CODE, r
    w = WORKLOADS["tiny_decode"]
    x = make_decode_inputs(w, seed=3)
    d = {k: v.cuda() for k, v in x.items()}
    O = fla.flash_lora_attn_decode(d["Q"], d["K_base"], d["V_base"], d["L"], d["B"], d["offsets"], rank=w.rank)
    torch.cuda.synchronize()
    ref = oracle.decode(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], x["offsets"].numpy(), rank=w.rank)
    got = O.double().cpu().numpy()
    assert np.abs(got - ref).max() <= 1e-2
    assert fla.device_error() == 0


def test_limit_is_validated(fla):
    with pytest.raises(fla.FlaError) as ei:
        fla.selftest_bounded_wait(0)
    assert ei.value.status == 1
    with pytest.raises(fla.FlaError):
        fla.selftest_bounded_wait(3_000_000_000)
