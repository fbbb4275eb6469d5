"""GPU parity of the baselines the reordered decode is compared with, against
the fp64 oracle: the materialised value cache (lora_value_expand, both
kernels) and plain per-agent attention over materialised or non-shared
caches.

Same bar as the attention kernels: max-abs 1e-2 and relative L2 5e-3 on O.
The bf16 expansion is held to the rounding of the fp64 result to bf16.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from workloads import WORKLOADS, make_decode_inputs

pytestmark = pytest.mark.gpu

ATOL, RTOL_L2 = 1e-2, 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from attention_flash_lora_attn_b300 import build_lib
    build_lib.build()
    import attention_flash_lora_attn_b300 as fla
    fla.load_library()
    yield
    assert fla.device_error() == 0


def _fla():
    import attention_flash_lora_attn_b300 as fla
    return fla


def _base():
    from attention_flash_lora_attn_b300 import baselines
    return baselines


def check_attn(O_gpu, O_ref, atol=ATOL, rtol_l2=RTOL_L2, what=""):
    O_gpu = O_gpu.detach().double().cpu().numpy()
    assert np.isfinite(O_gpu).all(), f"{what}: non-finite output"
    diff = O_gpu - O_ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    nrm = float(np.linalg.norm(O_ref))
    rel = float(np.linalg.norm(diff)) / nrm if nrm > 0 else float(np.linalg.norm(diff))
    assert max_abs <= atol and rel <= rtol_l2, f"{what}: max_abs={max_abs:.3e} rel_l2={rel:.3e}"


def workload(A, hq, hkv, d, r, dtype="bf16"):
    return dataclasses.replace(WORKLOADS["llama8b_decode"], n_agents=A, hq=hq, hkv=hkv, head_dim=d,
                               rank=r, dtype=dtype, lengths=(1,))


def to_dev(x):
    return {k: v.cuda() for k, v in x.items()}


# (n_tokens, A, hkv, d, r, shared L, dtype): ragged row tails, every supported
# d / r class, fp32 and bf16; bf16 with r % 16 == 0 and d 64 / 128 takes the
# mma.sync kernel under "auto"
EXPAND = [
    (200, 2, 2, 64, 8, False, "f32"),
    (300, 3, 8, 128, 16, False, "bf16"),
    (65, 5, 8, 128, 64, False, "bf16"),
    (130, 4, 2, 64, 32, True, "bf16"),
    (1, 1, 1, 8, 1, False, "f32"),
    (129, 2, 3, 24, 5, False, "f32"),
    (100, 3, 4, 128, 8, False, "bf16"),
    (4099, 3, 8, 128, 16, False, "bf16"),
]


@pytest.mark.parametrize("kernel", ["auto", "simt"])
@pytest.mark.parametrize("case", EXPAND, ids=[f"e{i}" for i in range(len(EXPAND))])
def test_lora_value_expand_matches_the_materialised_oracle(case, kernel):
    n, A, hkv, d, r, shared, dt = case
    x = make_decode_inputs(workload(A, hkv, hkv, d, r, dt), seed=3, shared_L=shared, lengths=[n])
    x["B"].mul_(25.0)  # adapter term of the order of V_base, so a wrong product shows
    dv = to_dev(x)
    Vi = _fla().lora_value_expand(dv["V_base"], dv["L"], dv["B"], rank=r, l_agent_stride=0 if shared else r,
                                  kernel=kernel)
    got = Vi.double().cpu().numpy()
    for a in range(A):
        cols = slice(0, r) if shared else slice(a * r, (a + 1) * r)
        ref = oracle.agent_value_cache(x["V_base"], x["L"][:, cols], x["B"][a], hkv, d)
        if dt == "f32":
            np.testing.assert_allclose(got[a], ref, rtol=1e-5, atol=1e-5)
        else:
            # one rounding of the fp32-accumulated value: within half a bf16 ulp
            # of the exact value plus the accumulation error, and equal to the
            # rounded exact value nearly everywhere
            assert np.all(np.abs(got[a] - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6), f"agent {a}"
            mismatch = np.mean(got[a] != oracle.round_to_bf16(ref))
            assert mismatch < 1e-3, f"agent {a}: {mismatch:.2e} of values off the rounded exact value"


def test_lora_value_expand_kernel_selection():
    x = to_dev(make_decode_inputs(workload(2, 4, 4, 128, 8), seed=1, lengths=[64]))
    fla = _fla()
    with pytest.raises(fla.FlaError) as e:  # rank 8: outside the mma.sync kernel
        fla.lora_value_expand(x["V_base"], x["L"], x["B"], rank=8, kernel="mma")
    assert e.value.status == 2
    with pytest.raises(fla.FlaError) as e:  # no tcgen05 kernel for the expansion
        fla.lora_value_expand(x["V_base"], x["L"], x["B"], rank=8, kernel="tcgen05")
    assert e.value.status == 2


# (lengths, A, hq, hkv, d, r, shared L)
NAIVE = [
    ((300,), 2, 8, 2, 128, 16, False),
    ((0, 5, 700), 3, 32, 8, 128, 16, False),
    ((513,), 5, 64, 8, 128, 64, False),
    ((129, 64), 4, 32, 8, 128, 32, True),
    ((77,), 2, 4, 4, 64, 8, False),
]


@pytest.mark.parametrize("case", NAIVE, ids=[f"n{i}" for i in range(len(NAIVE))])
def test_naive_materialised_decode_matches_oracle(case):
    lengths, A, hq, hkv, d, r, shared = case
    x = make_decode_inputs(workload(A, hq, hkv, d, r), seed=13, shared_L=shared, lengths=list(lengths))
    dv = to_dev(x)
    O = _base().naive_materialised_decode(dv["Q"], dv["K_base"], dv["V_base"], dv["L"], dv["B"], dv["offsets"],
                                          rank=r, l_agent_stride=0 if shared else r)
    ref = oracle.decode(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], x["offsets"].numpy(), rank=r,
                        agent_stride=0 if shared else r)
    check_attn(O, ref, what=f"naive {case}")


def test_naive_materialised_decode_f32_tiny_workload():
    w = WORKLOADS["tiny_decode"]
    x = make_decode_inputs(w, seed=0)
    dv = to_dev(x)
    O = _base().naive_materialised_decode(dv["Q"], dv["K_base"], dv["V_base"], dv["L"], dv["B"], dv["offsets"],
                                          rank=w.rank)
    ref = oracle.decode(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], x["offsets"].numpy(), rank=w.rank)
    check_attn(O, ref, atol=1e-4, rtol_l2=1e-5, what="naive tiny fp32")


def _per_agent_caches(A, N, hkv, d, seed):
    gen = torch.Generator("cpu").manual_seed(seed)
    K = [torch.randn((N, hkv, d), generator=gen).to(torch.bfloat16) for _ in range(A)]
    V = [torch.randn((N, hkv, d), generator=gen).to(torch.bfloat16) for _ in range(A)]
    return K, V


@pytest.mark.parametrize("lengths", [(1000,), (3, 0, 450)])
def test_non_shared_decode_matches_oracle(lengths):
    A, hq, hkv, d = 3, 32, 8, 128
    x = make_decode_inputs(workload(A, hq, hkv, d, 16), seed=17, lengths=list(lengths))
    N = int(sum(lengths))
    K, V = _per_agent_caches(A, N, hkv, d, seed=19)
    O = _base().per_agent_decode(x["Q"].cuda(), [k.cuda() for k in K], [v.cuda() for v in V],
                                 x["offsets"].cuda())
    offs = x["offsets"].numpy()
    zL, zB = np.zeros((N, 1)), np.zeros((1, 1, hkv * d))
    for a in range(A):
        ref = oracle.decode(x["Q"][:, a:a + 1], K[a], V[a], zL, zB, offs, rank=1)
        check_attn(O[:, a:a + 1], ref, what=f"non-shared agent {a}")


def test_prepared_baselines_match_the_functions():
    A, hq, hkv, d, r = 3, 32, 8, 128, 16
    x = to_dev(make_decode_inputs(workload(A, hq, hkv, d, r), seed=23, lengths=[2500]))
    base = _base()
    naive = base.PreparedBaselineDecode("naive", x["Q"], x["offsets"], K_base=x["K_base"], V_base=x["V_base"],
                                        L=x["L"], B=x["B"], rank=r)
    got = naive().clone()
    want = base.naive_materialised_decode(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], x["offsets"], rank=r)
    assert torch.equal(got, want)
    K, V = _per_agent_caches(A, 2500, hkv, d, seed=29)
    K, V = [k.cuda() for k in K], [v.cuda() for v in V]
    ns = base.PreparedBaselineDecode("non_shared", x["Q"], x["offsets"], K=K, V=V)
    assert torch.equal(ns().clone(), base.per_agent_decode(x["Q"], K, V, x["offsets"]))
