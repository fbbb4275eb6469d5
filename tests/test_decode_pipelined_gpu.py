"""Back-to-back decode calls, as a serving loop (and the benchmark) issues them.

Decode calls are launched with programmatic dependent launch: a call's decode
kernel starts its token loop while the previous call's kernels drain, and it
waits on the previous grid only before its first global write.  These tests
enqueue many calls with no synchronisation in between, all sharing one
workspace and rotating over several input sets, on a stream and captured in a
CUDA graph, and check every call's output bit for bit against the same call
made alone (itself checked against the fp64 oracle).  One case puts a PyTorch
kernel that writes Q immediately before every decode, the producer the
header's ordering rule describes.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from workloads import WORKLOADS, make_decode_inputs

pytestmark = pytest.mark.gpu

ATOL, RTOL_L2 = 1e-2, 5e-3
N_SETS, N_CALLS = 3, 12


@pytest.fixture(scope="module")
def fla():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from attention_flash_lora_attn_b300 import build_lib
    build_lib.build()
    import attention_flash_lora_attn_b300 as m
    m.load_library()
    yield m
    assert m.device_error() == 0


def _check_oracle(O, x, rank):
    ref = oracle.decode(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"], x["offsets"].numpy(), rank=rank)
    got = O.double().cpu().numpy()
    assert np.isfinite(got).all()
    max_abs = float(np.abs(got - ref).max())
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert max_abs <= ATOL and rel <= RTOL_L2, (max_abs, rel)


# the headline 8B decode (mma.sync kernel, 12 query rows per kv head) and a
# 70B-shaped group of 40 rows per kv head (tcgen05 kernel) on a shorter context
SHAPES = {
    "mma-8b": (dataclasses.replace(WORKLOADS["llama8b_decode"]), "mma"),
    "tcgen05-70b": (dataclasses.replace(WORKLOADS["llama70b_decode"], lengths=(8192,)), "tcgen05"),
    "mma-ragged": (dataclasses.replace(WORKLOADS["llama8b_ragged"], lengths=(3000, 17, 0, 9000, 640)), "mma"),
}


def _sets(w, n):
    host = [make_decode_inputs(w, seed=100 + i) for i in range(n)]
    dev = [{k: v.cuda() for k, v in x.items()} for x in host]
    return host, dev


def _isolated(fla, d, w, kernel, ws):
    O = fla.flash_lora_attn_decode(d["Q"], d["K_base"], d["V_base"], d["L"], d["B"], d["offsets"], rank=w.rank,
                                   workspace=ws, kernel=kernel)
    torch.cuda.synchronize()
    return O.clone()


@pytest.mark.parametrize("shape", list(SHAPES))
def test_back_to_back_calls_on_a_stream_and_in_a_graph(fla, shape):
    w, kernel = SHAPES[shape]
    host, dev = _sets(w, N_SETS)
    ws = torch.empty(fla.load_library().flash_lora_attn_decode_workspace_size(
        __import__("ctypes").byref(fla.binding.make_dims(w.n_agents, w.hq, w.hkv, w.head_dim, w.rank, 1,
                                                         w.n_agents * w.rank, w.rank, None, kernel)),
        w.n_req, w.total_tokens) + 256, dtype=torch.uint8, device="cuda")
    want = [_isolated(fla, d, w, kernel, ws) for d in dev]
    for i in range(N_SETS):
        _check_oracle(want[i], host[i], w.rank)

    outs = [torch.full_like(want[0], float("nan")) for _ in range(N_CALLS)]
    stream = torch.cuda.Stream()

    def enqueue():
        for i in range(N_CALLS):
            d = dev[i % N_SETS]
            fla.flash_lora_attn_decode(d["Q"], d["K_base"], d["V_base"], d["L"], d["B"], d["offsets"],
                                       rank=w.rank, O=outs[i], workspace=ws, kernel=kernel, stream=stream)

    # on a stream, nothing synchronised between the calls
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        enqueue()
    stream.synchronize()
    for i in range(N_CALLS):
        assert torch.equal(outs[i], want[i % N_SETS]), f"stream call {i}"

    # the same calls captured in one CUDA graph, replayed twice
    for o in outs:
        o.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        enqueue()
    for rep in range(2):
        for o in outs:
            o.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        for i in range(N_CALLS):
            assert torch.equal(outs[i], want[i % N_SETS]), f"graph replay {rep} call {i}"


@pytest.mark.parametrize("shape", ["mma-8b", "tcgen05-70b"])
def test_a_torch_kernel_writing_q_right_before_each_decode(fla, shape):
    """Every decode reads a Q buffer that a PyTorch copy kernel filled just before it on the same stream."""
    w, kernel = SHAPES[shape]
    host, dev = _sets(w, N_SETS)
    d0 = dev[0]
    ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    # one K/V/L/B cache, three query sets
    want = []
    for i in range(N_SETS):
        want.append(_isolated(fla, dict(d0, Q=dev[i]["Q"]), w, kernel, ws))
    x = dict(host[0], Q=host[1]["Q"])
    _check_oracle(want[1], x, w.rank)
    Qbuf = torch.empty_like(d0["Q"])
    outs = [torch.full_like(want[0], float("nan")) for _ in range(N_CALLS)]
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(N_CALLS):
            Qbuf.copy_(dev[i % N_SETS]["Q"])
            fla.flash_lora_attn_decode(Qbuf, d0["K_base"], d0["V_base"], d0["L"], d0["B"], d0["offsets"],
                                       rank=w.rank, O=outs[i], workspace=ws, kernel=kernel, stream=stream)
    stream.synchronize()
    for i in range(N_CALLS):
        assert torch.equal(outs[i], want[i % N_SETS]), f"call {i}"
