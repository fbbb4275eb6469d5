"""GPU parity: the CUDA kernels (through the C ABI) against the fp64 oracle.

Acceptance bar: attention outputs within max-abs 1e-2 and relative L2 5e-3
of the oracle; the LR cache within relative L2 2e-3 of the fp64 product.
Every input comes from the seeded generators in `workloads`.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from workloads import WORKLOADS, make_build_inputs, make_decode_inputs, make_prefill_inputs, make_rebase_inputs

pytestmark = pytest.mark.gpu

ATOL, RTOL_L2, BUILD_RTOL_L2 = 1e-2, 5e-3, 2e-3


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


def check_attn(O_gpu, O_ref, atol=ATOL, rtol_l2=RTOL_L2, what=""):
    O_gpu = O_gpu.detach().double().cpu().numpy() if isinstance(O_gpu, torch.Tensor) else O_gpu
    assert np.isfinite(O_gpu).all(), f"{what}: non-finite output"
    diff = O_gpu - O_ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    nrm = float(np.linalg.norm(O_ref))
    rel = float(np.linalg.norm(diff)) / nrm if nrm > 0 else float(np.linalg.norm(diff))
    assert max_abs <= atol and rel <= rtol_l2, f"{what}: max_abs={max_abs:.3e} rel_l2={rel:.3e}"
    return max_abs, rel


def to_dev(x):
    return {k: v.cuda() for k, v in x.items()}


def run_decode(x, rank, kernel, shared=False, **kw):
    d = to_dev(x)
    return _fla().flash_lora_attn_decode(d["Q"], d["K_base"], d["V_base"], d["L"], d["B"], d["offsets"],
                                         rank=rank, l_agent_stride=0 if shared else rank, kernel=kernel, **kw)


def small_workload(A, hq, hkv, d, r, dtype="bf16"):
    return dataclasses.replace(WORKLOADS["llama8b_decode"], n_agents=A, hq=hq, hkv=hkv, head_dim=d,
                               rank=r, dtype=dtype, lengths=(1,))


# (lengths, A, hq, hkv, d, r, shared)
SMALL = [
    ((1,), 1, 4, 4, 64, 8, False),
    ((37,), 2, 8, 2, 128, 16, False),
    ((0, 5, 300), 3, 32, 8, 128, 16, False),
    ((129, 1, 64, 1000), 4, 32, 8, 128, 32, False),
    ((513,), 5, 64, 8, 128, 64, False),
    ((2049, 17), 3, 32, 8, 128, 16, True),
    ((700,), 2, 16, 2, 64, 32, False),
    ((96, 31), 1, 8, 8, 128, 8, False),
    ((4000,), 4, 16, 1, 128, 16, False),
]


@pytest.mark.parametrize("kernel", ["tensor", "mma", "tcgen05", "simt"])
@pytest.mark.parametrize("case", SMALL, ids=[f"s{i}" for i in range(len(SMALL))])
def test_decode_small(case, kernel):
    lengths, A, hq, hkv, d, r, shared = case
    w = small_workload(A, hq, hkv, d, r)
    x = make_decode_inputs(w, seed=11, shared_L=shared, lengths=list(lengths))
    try:
        O = run_decode(x, r, kernel, shared)
    except _fla().FlaError as e:
        if kernel in ("tensor", "mma", "tcgen05") and e.status == 2:
            pytest.skip("shape outside this tensor-core decode kernel")
        raise
    ref = oracle.decode(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], x["offsets"].numpy(), rank=r,
                        agent_stride=0 if shared else r)
    check_attn(O, ref, what=f"decode {case} {kernel}")


@pytest.mark.parametrize("kernel", ["mma", "tcgen05", "simt"])
def test_decode_lora_term_alone(kernel):
    """V_base = 0 isolates (P.L_a).B_a, so the LoRA path is checked at full weight."""
    w = small_workload(3, 32, 8, 128, 16)
    x = make_decode_inputs(w, seed=5, lengths=[1500, 77])
    x["V_base"].zero_()
    x["B"].mul_(50.0)  # LoRA term of order 1
    O = run_decode(x, 16, kernel)
    ref = oracle.decode(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], x["offsets"].numpy(), rank=16)
    assert np.abs(ref).max() > 0.5
    check_attn(O, ref, what="lora-only")


def test_decode_f32_tiny_workload():
    w = WORKLOADS["tiny_decode"]
    x = make_decode_inputs(w, seed=0)
    O = run_decode(x, w.rank, "auto")
    ref = oracle.decode(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], x["offsets"].numpy(), rank=w.rank)
    check_attn(O, ref, atol=1e-4, rtol_l2=1e-5, what="tiny fp32")


@pytest.mark.parametrize("kernel", ["mma", "tcgen05"])
def test_decode_llama8b_full(kernel):
    w = WORKLOADS["llama8b_decode"]
    x = make_decode_inputs(w, seed=0)
    O = run_decode(x, w.rank, kernel)
    ref = oracle.decode(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], x["offsets"].numpy(), rank=w.rank)
    check_attn(O, ref, what="llama8b_decode")


@pytest.mark.parametrize("kernel", ["mma", "tcgen05"])
def test_decode_ragged_sampled_requests(kernel):
    """Full 32-request ragged batch on the GPU; 6 requests re-computed by the oracle."""
    w = WORKLOADS["llama8b_ragged"]
    x = make_decode_inputs(w, seed=0)
    O = run_decode(x, w.rank, kernel).cpu()
    offs = x["offsets"].numpy()
    for q in [0, 5, 14, 23, 27, 31]:  # includes the longest (14) and shortest (23) requests
        t0, t1 = int(offs[q]), int(offs[q + 1])
        ref = oracle.decode(x["Q"][q:q + 1], x["K_base"][t0:t1], x["V_base"][t0:t1], x["L"][t0:t1], x["B"],
                            np.array([0, t1 - t0]), rank=w.rank)
        check_attn(O[q:q + 1], ref, what=f"ragged request {q}")


@pytest.mark.parametrize("kernel", ["mma", "tcgen05"])
def test_decode_llama70b_sampled_agents(kernel):
    w = WORKLOADS["llama70b_decode"]
    x = make_decode_inputs(w, seed=0)
    O = run_decode(x, w.rank, kernel).cpu()
    r = w.rank
    for a in [0, 4]:
        ref = oracle.decode(x["Q"][:, a:a + 1], x["K_base"], x["V_base"], x["L"][:, a * r:(a + 1) * r],
                            x["B"][a:a + 1], x["offsets"].numpy(), rank=r)
        check_attn(O[:, a:a + 1], ref, what=f"70b agent {a}")


@pytest.mark.parametrize("kernel", ["mma", "tcgen05"])
def test_decode_tensor_and_simt_agree_and_are_deterministic(kernel):
    w = WORKLOADS["llama8b_decode"]
    x = make_decode_inputs(w, seed=3)
    O1 = run_decode(x, w.rank, kernel)
    O2 = run_decode(x, w.rank, kernel)
    assert torch.equal(O1, O2), f"{kernel} decode is not deterministic run to run"
    O3 = run_decode(x, w.rank, "simt")
    check_attn(O1, O3.double().cpu().numpy(), what=f"{kernel} vs simt")


def test_decode_many_waves_two_ctas_per_sm():
    """40 requests: the grid spans several waves, so the mma.sync decode runs two CTAs per SM (one
    warp group each); the 8B shapes with a 48-column L window."""
    w = small_workload(3, 32, 8, 128, 16)
    lengths = [int(v) for v in np.random.default_rng(7).integers(1, 4000, size=40)]
    x = make_decode_inputs(w, seed=17, lengths=lengths)
    O = run_decode(x, 16, "mma")
    ref = oracle.decode(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], x["offsets"].numpy(), rank=16)
    check_attn(O, ref, what="many waves")


def test_decode_tcgen05_rescales_when_scores_jump():
    """Q scaled so the running max moves by far more than 2^8 between tiles: exercises the rescale
    of O, OL and l in TMEM; one request shorter than a tile and one empty request ride along."""
    w = small_workload(5, 40, 8, 128, 16)
    x = make_decode_inputs(w, seed=21, lengths=[3000, 100, 0, 1300])
    x["Q"] = (x["Q"].float() * 8.0).to(x["Q"].dtype)
    O = run_decode(x, 16, "tcgen05")
    ref = oracle.decode(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], x["offsets"].numpy(), rank=16)
    check_attn(O, ref, what="tcgen05 rescale")


def test_prepared_decode_matches_the_function():
    w = small_workload(3, 32, 8, 128, 16)
    x = to_dev(make_decode_inputs(w, seed=13, lengths=[5000, 70, 1]))
    fla = _fla()
    O1 = fla.flash_lora_attn_decode(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], x["offsets"], rank=16)
    call = fla.PreparedDecode(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], x["offsets"], rank=16)
    for _ in range(2):
        O2 = call()
        torch.cuda.synchronize()
        assert torch.equal(O1, O2)


def test_decode_host_io_matches_the_device_decode():
    """One host-buffer call (copy in, decode, copy out) gives the device decode's output, twice in a row."""
    fla = _fla()
    w = small_workload(3, 32, 8, 128, 16)
    x = make_decode_inputs(w, seed=31, lengths=[1500, 7])
    d = to_dev(x)
    Qh = x["Q"].clone().pin_memory()
    Qd = torch.empty_like(d["Q"])
    Od = torch.empty(d["Q"].shape, dtype=torch.float32, device="cuda")
    Oh = torch.empty(d["Q"].shape, dtype=torch.float32).pin_memory()
    call = fla.PreparedDecodeHostIO(Qh, Qd, d["K_base"], d["V_base"], d["L"], d["B"], d["offsets"], rank=16,
                                    O_dev=Od, O_host=Oh)
    for step in range(2):
        if step:
            Qh.copy_(make_decode_inputs(w, seed=37, lengths=[1500, 7])["Q"])
        call()
        torch.cuda.synchronize()
        want = fla.flash_lora_attn_decode(Qh.cuda(), d["K_base"], d["V_base"], d["L"], d["B"], d["offsets"], rank=16)
        assert torch.equal(Oh, want.cpu()), f"step {step}"
    ref = oracle.decode(Qh, x["K_base"], x["V_base"], x["L"], x["B"], x["offsets"].numpy(), rank=16)
    check_attn(Oh, ref, what="host io")


def test_decode_output_guard_bands():
    """Writes stay inside O: canaries around the output are untouched."""
    w = small_workload(3, 32, 8, 128, 16)
    x = to_dev(make_decode_inputs(w, seed=9, lengths=[3000, 5]))
    R, A, hq, d = x["Q"].shape
    n = R * A * hq * d
    buf = torch.full((n + 2048,), 12345.0, device="cuda")
    O = buf[1024:1024 + n].view(R, A, hq, d)
    for kernel in ("mma", "tcgen05"):
        _fla().flash_lora_attn_decode(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], x["offsets"], rank=16,
                                      O=O, kernel=kernel)
        torch.cuda.synchronize()
        assert torch.all(buf[:1024] == 12345.0) and torch.all(buf[1024 + n:] == 12345.0)


# ----------------------------------------------------------------------------- prefill

def small_prefill(A, hq, hkv, d, r, n0, c):
    return dataclasses.replace(WORKLOADS["llama8b_prefill"], n_agents=A, hq=hq, hkv=hkv, head_dim=d,
                               rank=r, n0=n0, chunk=c, d_model=64)


PREFILL_SMALL = [(1, 4, 4, 64, 8, 0, 5), (2, 8, 2, 128, 16, 37, 70), (4, 32, 8, 128, 16, 300, 129),
                 (3, 16, 4, 128, 32, 1, 200), (1, 8, 8, 64, 16, 64, 1), (5, 64, 8, 128, 64, 130, 33),
                 (2, 4, 2, 128, 16, 0, 300)]


@pytest.mark.parametrize("kernel", ["tensor", "mma", "simt"])
@pytest.mark.parametrize("case", PREFILL_SMALL, ids=[f"p{i}" for i in range(len(PREFILL_SMALL))])
def test_prefill_small(case, kernel):
    A, hq, hkv, d, r, n0, c = case
    w = small_prefill(A, hq, hkv, d, r, n0, c)
    x = make_prefill_inputs(w, seed=2, with_X=False)
    dx = to_dev(x)
    try:
        O = _fla().flash_lora_attn_prefill(dx["Q"], dx["K_base"], dx["V_base"], dx["L"], dx["B"], n0, rank=r,
                                           kernel=kernel)
    except _fla().FlaError as e:
        if kernel in ("tensor", "mma") and e.status == 2:
            pytest.skip("shape outside the tensor-core prefill kernels")
        raise
    ref = oracle.prefill(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], n0=n0, rank=r)
    check_attn(O, ref, what=f"prefill {case}")


# (A, hq, hkv, d, r, n0, chunk, shared L, Q scale): shapes inside the tcgen05 kernel.  Ragged key
# tails, partial 128-row blocks (A*G*QB < 128), L narrower than its 64-column box (shared L, small
# A*r), head_dim 64, one key in total, and Q scaled up so the running max moves often (rescales).
PREFILL_TC5 = [(4, 32, 8, 128, 16, 300, 129, False, 1.0), (4, 32, 8, 128, 16, 1000, 64, True, 1.0),
               (3, 24, 8, 128, 16, 777, 50, False, 1.0), (2, 8, 8, 64, 32, 2000, 100, False, 4.0),
               (1, 32, 8, 128, 64, 513, 300, False, 1.0), (8, 16, 8, 128, 8, 129, 17, False, 1.0),
               (2, 2, 2, 128, 16, 0, 1, False, 1.0), (2, 16, 8, 128, 16, 3000, 40, False, 8.0)]


@pytest.mark.parametrize("kernel", ["tcgen05", "mma"])
@pytest.mark.parametrize("case", PREFILL_TC5, ids=[f"t{i}" for i in range(len(PREFILL_TC5))])
def test_prefill_tcgen05_shapes(case, kernel):
    A, hq, hkv, d, r, n0, c, shared, qs = case
    if kernel == "mma" and r % 16:
        pytest.skip("the mma.sync prefill kernel needs rank % 16 == 0")
    w = small_prefill(A, hq, hkv, d, r, n0, c)
    x = make_prefill_inputs(w, seed=5, with_X=False)
    x["Q"] = (x["Q"].float() * qs).to(x["Q"].dtype)  # power-of-two scale: exact in bf16
    dx = to_dev(x)
    L = dx["L"][:, :r] if shared else dx["L"]
    O = _fla().flash_lora_attn_prefill(dx["Q"], dx["K_base"], dx["V_base"], L, dx["B"], n0, rank=r,
                                       l_agent_stride=0 if shared else r, kernel=kernel)
    ref = oracle.prefill(x["Q"], x["K_base"], x["V_base"], x["L"][:, :r] if shared else x["L"], x["B"],
                         n0=n0, rank=r, agent_stride=0 if shared else r)
    check_attn(O, ref, what=f"prefill {kernel} {case}")


@pytest.mark.parametrize("case", [(4, 32, 8, 128, 16, 1000, 200), (2, 8, 8, 64, 32, 700, 90)], ids=["d128", "d64"])
def test_prefill_tcgen05_split_tail_and_whole_range_both_match(case):
    """With its workspace the tcgen05 prefill runs pairs as two half-range items merged afterwards (every
    pair here: few pairs); with no workspace every pair runs its whole key range.  Both against the oracle."""
    A, hq, hkv, d, r, n0, c = case
    w = small_prefill(A, hq, hkv, d, r, n0, c)
    x = make_prefill_inputs(w, seed=7, with_X=False)
    dx = to_dev(x)
    ref = oracle.prefill(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], n0=n0, rank=r)
    fla = _fla()
    need = fla.load_library().flash_lora_attn_prefill_workspace_size(
        __import__("ctypes").byref(fla.binding.make_dims(A, hq, hkv, d, r, 1, A * r, r, None, "tcgen05")), c, n0)
    assert need > 0  # this shape splits
    O_split = fla.flash_lora_attn_prefill(dx["Q"], dx["K_base"], dx["V_base"], dx["L"], dx["B"], n0, rank=r,
                                          kernel="tcgen05")
    O_whole = fla.flash_lora_attn_prefill(dx["Q"], dx["K_base"], dx["V_base"], dx["L"], dx["B"], n0, rank=r,
                                          kernel="tcgen05", workspace=torch.empty(0, dtype=torch.uint8, device="cuda"))
    check_attn(O_split, ref, what=f"prefill split {case}")
    check_attn(O_whole, ref, what=f"prefill whole {case}")


def test_prefill_tcgen05_rejects_shapes_outside_it():
    w = small_prefill(3, 16, 4, 128, 32, 1, 20)  # L width A*r = 96 > 64
    dx = to_dev(make_prefill_inputs(w, seed=1, with_X=False))
    with pytest.raises(_fla().FlaError) as ei:
        _fla().flash_lora_attn_prefill(dx["Q"], dx["K_base"], dx["V_base"], dx["L"], dx["B"], 1, rank=32,
                                       kernel="tcgen05")
    assert ei.value.status == 2


@pytest.mark.parametrize("kernel", ["tcgen05", "mma"])
def test_prefill_llama8b_chunk_with_lr_build_sampled_rows(kernel):
    """Build the chunk's LR rows on the GPU, then prefill; oracle on sampled positions."""
    w = WORKLOADS["llama8b_prefill"]
    x = make_prefill_inputs(w, seed=0)
    dx = to_dev(x)
    fla = _fla()
    fla.lr_cache_build(dx["X"], dx["A_cat"], dx["L"][w.n0:], n_agents=w.n_agents)
    O = fla.flash_lora_attn_prefill(dx["Q"], dx["K_base"], dx["V_base"], dx["L"], dx["B"], w.n0,
                                    rank=w.rank, kernel=kernel).cpu()
    # oracle: its own LR rows for the chunk (fp64 product rounded to the bf16 storage type)
    L_ref = oracle.to_f64(x["L"]).copy()
    L_ref[w.n0:] = oracle.round_to_bf16(oracle.lr_cache_build(x["X"], x["A_cat"]))
    pos = [0, 1, 7, 8, 255, 256, 510, 511]
    ref = oracle.prefill(x["Q"], x["K_base"], x["V_base"], L_ref, x["B"], n0=w.n0, rank=w.rank, positions=pos)
    check_attn(O[:, pos], ref[:, pos], what="llama8b prefill")


# ----------------------------------------------------------------------------- LR-cache build

BUILD_SMALL = [(1, 64, 16, "bf16"), (100, 256, 48, "bf16"), (300, 4096, 64, "bf16"), (257, 512, 320, "bf16"),
               (130, 192, 24, "bf16"), (77, 256, 16, "f32")]


def _rel_l2(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("kernel", ["auto", "simt"])
@pytest.mark.parametrize("case", BUILD_SMALL, ids=[f"b{i}" for i in range(len(BUILD_SMALL))])
def test_lr_build_small(case, kernel):
    n, D, N, dt = case
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32
    x = make_build_inputs(n, D, 1, N, dtype, seed=4)
    dX, dA = x["X"].cuda(), x["A_cat"].cuda()
    L = _fla().lr_cache_build(dX, dA, kernel=kernel).double().cpu().numpy()
    ref = oracle.lr_cache_build(x["X"], x["A_cat"])
    assert _rel_l2(L, ref) <= (BUILD_RTOL_L2 if dt == "bf16" else 1e-6)


@pytest.mark.parametrize("case", [(128, 64, 32), (300, 4096, 64), (257, 512, 320), (1000, 1024, 512), (77, 128, 96)],
                         ids=["one-tile", "llama8b-cols", "ragged-320", "n512", "n96"])
def test_lr_build_tensor_kernel(case):
    """The tcgen05 GEMM itself (kernel="tensor" refuses to fall back)."""
    n, D, N = case
    x = make_build_inputs(n, D, 1, N, torch.bfloat16, seed=8)
    L = _fla().lr_cache_build(x["X"].cuda(), x["A_cat"].cuda(), kernel="tensor")
    ref = oracle.lr_cache_build(x["X"], x["A_cat"])
    assert _rel_l2(L.double().cpu().numpy(), ref) <= BUILD_RTOL_L2


# Enough rows that the tile count exceeds half the SMs: the plan takes the
# CTA-pair kernel (256 rows per pair, each CTA copying half of the W boxes).
# Ragged row tails (the odd CTA of the last pair past the end), odd box counts
# (a zero-filled box completes the pair), partial boxes and several column tiles.
PAIR_BUILD = [(10000, 256, 320), (9700, 128, 96), (2000, 512, 2368), (19200, 192, 64), (12345, 64, 512)]


@pytest.mark.parametrize("case", PAIR_BUILD, ids=["n320-odd-boxes", "n96-partial", "n2368-5-tiles", "n64", "n512"])
def test_lr_build_cta_pairs(case):
    n, D, N = case
    x = make_build_inputs(n, D, 1, N, torch.bfloat16, seed=9)
    L = _fla().lr_cache_build(x["X"].cuda(), x["A_cat"].cuda(), kernel="tcgen05")
    ref = oracle.lr_cache_build(x["X"], x["A_cat"])
    got = L.double().cpu().numpy()
    assert np.isfinite(got).all()
    assert _rel_l2(got, ref) <= BUILD_RTOL_L2
    # every row, the last ones included, on its own
    per_row = np.linalg.norm(got - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    assert per_row.max() <= 4 * BUILD_RTOL_L2


def test_lr_build_strided_output_leaves_other_columns():
    x = make_build_inputs(200, 512, 2, 32, torch.bfloat16, seed=6)
    L = torch.full((200, 100), 7.0, dtype=torch.bfloat16, device="cuda")
    _fla().lr_cache_build(x["X"].cuda(), x["A_cat"].cuda(), L[:, 8:72])
    Lc = L.double().cpu().numpy()
    assert (Lc[:, :8] == 7).all() and (Lc[:, 72:] == 7).all()
    assert _rel_l2(Lc[:, 8:72], oracle.lr_cache_build(x["X"], x["A_cat"])) <= BUILD_RTOL_L2


def test_lr_build_llama8b_chunk_full():
    x = make_build_inputs(512, 4096, 4, 16, torch.bfloat16, seed=0)
    L = _fla().lr_cache_build(x["X"].cuda(), x["A_cat"].cuda(), kernel="tensor")
    assert _rel_l2(L.double().cpu().numpy(), oracle.lr_cache_build(x["X"], x["A_cat"])) <= BUILD_RTOL_L2


def test_lr_build_llama70b_full_size_sampled_rows():
    """131072 x 8192 . 8192 x 320 on the GPU; 4096 sampled rows against the oracle."""
    x = make_build_inputs(131072, 8192, 5, 64, torch.bfloat16, seed=0)
    dX = x["X"].cuda()
    L = _fla().lr_cache_build(dX, x["A_cat"].cuda(), kernel="tensor")
    rows = np.sort(np.random.default_rng(0).choice(131072, 4096, replace=False))
    rows = np.concatenate([[0, 1], rows, [131070, 131071]])
    Ls = L[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    ref = oracle.lr_cache_build(x["X"][torch.from_numpy(rows)], x["A_cat"])
    assert _rel_l2(Ls, ref) <= BUILD_RTOL_L2


# ----------------------------------------------------------------------------- ReBaseShared base projection

# (n, d_model, hkv, head_dim, n_agents, rank, dtype)
REBASE = [(1, 64, 1, 64, 2, 16, "bf16"), (77, 256, 2, 64, 3, 32, "bf16"), (300, 512, 8, 128, 4, 16, "bf16"),
          (1000, 1024, 4, 128, 5, 64, "bf16"), (130, 192, 1, 48, 2, 8, "bf16"), (60, 128, 2, 16, 1, 8, "f32")]


def _rebase_check(x, K, V, L, hkv, d):
    Kr, Vr, Lr = oracle.rebase_kv_lr_build(x["X"], x["W_k"], x["W_v"], x["A_cat"], hkv=hkv, d=d)
    for got, ref, nm in ((K, Kr, "K_base"), (V, Vr, "V_base"), (L, Lr, "L")):
        g = got.double().cpu().numpy().reshape(ref.shape)
        tol = BUILD_RTOL_L2 if got.dtype == torch.bfloat16 else 1e-6
        assert _rel_l2(g, ref) <= tol, nm


@pytest.mark.parametrize("kernel", ["auto", "simt"])
@pytest.mark.parametrize("case", REBASE, ids=[f"rb{i}" for i in range(len(REBASE))])
def test_rebase_projection_small(case, kernel):
    n, D, hkv, d, A, r, dt = case
    x = make_rebase_inputs(n, D, hkv, d, A, r, torch.bfloat16 if dt == "bf16" else torch.float32, seed=12)
    W = torch.cat([x["W_k"], x["W_v"], x["A_cat"]], dim=1).cuda()
    K, V, L = _fla().rebase_kv_lr_build(x["X"].cuda(), W, hkv=hkv, head_dim=d, n_agents=A, rank=r, kernel=kernel)
    _rebase_check(x, K, V, L, hkv, d)


def test_rebase_projection_tensor_kernel_refuses_odd_widths():
    x = make_rebase_inputs(64, 128, 1, 48, 2, 8, torch.bfloat16, seed=1)
    W = torch.cat([x["W_k"], x["W_v"], x["A_cat"]], dim=1).cuda()
    with pytest.raises(_fla().FlaError) as ei:
        _fla().rebase_kv_lr_build(x["X"].cuda(), W, hkv=1, head_dim=48, n_agents=2, rank=8, kernel="tensor")
    assert ei.value.status == 2


def test_rebase_projection_llama8b_chunk_full():
    """The 512-token chunk of the 8B workload: X 512x4096 . [W_k | W_v | A_cat] (4096 x 2112), all outputs."""
    w = WORKLOADS["llama8b_prefill"]
    x = make_rebase_inputs(w.chunk, w.d_model, w.hkv, w.head_dim, w.n_agents, w.rank, torch.bfloat16, seed=0)
    W = torch.cat([x["W_k"], x["W_v"], x["A_cat"]], dim=1).cuda()
    L = torch.full((w.chunk, 104), 7.0, dtype=torch.bfloat16, device="cuda")  # L as a column slice of a wider tensor
    K, V, Ls = _fla().rebase_kv_lr_build(x["X"].cuda(), W, hkv=w.hkv, head_dim=w.head_dim, n_agents=w.n_agents,
                                         rank=w.rank, L=L[:, 8:8 + w.n_agents * w.rank], kernel="tensor")
    _rebase_check(x, K, V, Ls, w.hkv, w.head_dim)
    Lc = L.double().cpu().numpy()
    assert (Lc[:, :8] == 7).all() and (Lc[:, 8 + w.n_agents * w.rank:] == 7).all()


def test_rebase_projection_cta_pairs():
    """Three output segments through the CTA-pair kernel: 4000 rows, 512 + 512 + 96 columns in three tiles."""
    n, D, hkv, d, A, r = 4000, 256, 4, 128, 6, 16
    x = make_rebase_inputs(n, D, hkv, d, A, r, torch.bfloat16, seed=13)
    W = torch.cat([x["W_k"], x["W_v"], x["A_cat"]], dim=1).cuda()
    K, V, L = _fla().rebase_kv_lr_build(x["X"].cuda(), W, hkv=hkv, head_dim=d, n_agents=A, rank=r, kernel="tcgen05")
    _rebase_check(x, K, V, L, hkv, d)


def test_rebase_projection_llama70b_shape_sampled_rows():
    """70B shapes (8192 -> 2*1024 + 320 columns) on 16384 rows, 600 sampled rows against the oracle."""
    w = WORKLOADS["llama70b_decode"]
    n = 16384
    x = make_rebase_inputs(n, w.d_model, w.hkv, w.head_dim, w.n_agents, w.rank, torch.bfloat16, seed=3)
    W = torch.cat([x["W_k"], x["W_v"], x["A_cat"]], dim=1).cuda()
    K, V, L = _fla().rebase_kv_lr_build(x["X"].cuda(), W, hkv=w.hkv, head_dim=w.head_dim, n_agents=w.n_agents,
                                        rank=w.rank, kernel="tensor")
    rows = np.concatenate([[0, 1, 127, 128], np.sort(np.random.default_rng(1).choice(n, 592, replace=False)),
                           [n - 2, n - 1]])
    ri = torch.from_numpy(rows)
    xs = dict(x, X=x["X"][ri])
    _rebase_check(xs, K[ri.cuda()], V[ri.cuda()], L[ri.cuda()], w.hkv, w.head_dim)
