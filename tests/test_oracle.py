"""Pins for the CPU oracle: it is checked against things other than itself.

* hand-derived tiny cases (tests/golden, exact fractions by construction);
* B = 0 reduces to plain softmax attention: torch's scaled_dot_product_attention
  in fp64 (a library routine);
* Q = 0 gives the mean of V_i over the visible tokens (closed form);
* the reordered form P.V_base + (P.L_i).B_i equals the materialised one
  (LRAgent summary, Metodologia section 3, associativity);
* causal visibility: prefill row p equals decode over the first n0+p+1 tokens;
* GQA equals MHA with duplicated kv heads; ragged equals separate requests;
  token permutation invariance; n = 1 returns V_i[0]; O is affine in B;
  each agent's output depends only on its own L_i, B_i;
* lr_cache_build against hand-derived values and per-agent block structure;
* rebase_kv_lr_build against a hand-derived case, brute-force sums on integer
  inputs, one-hot hidden states (each output row is a weight row) and the
  head layout of K_base / V_base.
"""
import dataclasses
import glob
import json
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import WORKLOADS, make_build_inputs, make_decode_inputs, make_prefill_inputs


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _arr(x):
    return np.asarray(x, dtype=np.float64)


GOLDEN = sorted(os.path.basename(p) for p in
                glob.glob(os.path.join(os.path.dirname(__file__), "golden", "*.json")))


@pytest.mark.parametrize("name", GOLDEN)
def test_golden_fixture(golden_dir, name):
    c = _load(golden_dir, name)
    if c["kind"] == "decode":
        O = oracle.decode(_arr(c["Q"]), _arr(c["K_base"]), _arr(c["V_base"]), _arr(c["L"]),
                          _arr(c["B"]), c["offsets"], rank=c["rank"],
                          agent_stride=c.get("agent_stride"))
        np.testing.assert_allclose(O, _arr(c["O"]), rtol=0, atol=1e-12)
    elif c["kind"] == "prefill":
        O = oracle.prefill(_arr(c["Q"]), _arr(c["K_base"]), _arr(c["V_base"]), _arr(c["L"]),
                           _arr(c["B"]), n0=c["n0"], rank=c["rank"])
        np.testing.assert_allclose(O, _arr(c["O"]), rtol=0, atol=1e-12)
    elif c["kind"] == "rebase":
        K, V, L = oracle.rebase_kv_lr_build(_arr(c["X"]), _arr(c["W_k"]), _arr(c["W_v"]), _arr(c["A_cat"]),
                                            hkv=c["hkv"], d=c["d"])
        np.testing.assert_array_equal(K, _arr(c["K_base"]))
        np.testing.assert_array_equal(V, _arr(c["V_base"]))
        np.testing.assert_array_equal(L, _arr(c["L"]))
    else:
        L = oracle.lr_cache_build(_arr(c["X"]), _arr(c["A_cat"]))
        np.testing.assert_array_equal(L, _arr(c["L"]))


# ----------------------------------------------------------------------------
# small random cases (several agents, GQA, ragged), fp64
# ----------------------------------------------------------------------------

def _small_decode(seed=1, lengths=(7, 1, 12), A=3, hq=4, hkv=2, d=8, r=3, shared=False):
    g = np.random.default_rng(seed)
    N = int(sum(lengths))
    return dict(
        Q=g.standard_normal((len(lengths), A, hq, d)),
        K_base=g.standard_normal((N, hkv, d)),
        V_base=g.standard_normal((N, hkv, d)),
        L=g.standard_normal((N, r if shared else A * r)),
        B=g.standard_normal((A, r, hkv * d)),
        offsets=np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64),
        rank=r,
    )


def _sdpa(q, K, V, scale, mask=None):
    """torch SDPA in fp64 on CPU for one head: q [m, d], K/V [n, d]."""
    out = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, None], torch.from_numpy(K)[None, None],
        torch.from_numpy(V)[None, None],
        attn_mask=None if mask is None else torch.from_numpy(mask)[None, None], scale=scale)
    return out[0, 0].numpy()


def test_b_zero_is_plain_attention_decode():
    x = _small_decode()
    x["B"] = np.zeros_like(x["B"])
    O = oracle.decode(**x)
    R, A, hq, d = x["Q"].shape
    G = hq // x["K_base"].shape[1]
    offs = x["offsets"]
    for q in range(R):
        t0, t1 = offs[q], offs[q + 1]
        for a in range(A):
            for j in range(hq):
                ref = _sdpa(x["Q"][q, a, j][None], x["K_base"][t0:t1, j // G],
                            x["V_base"][t0:t1, j // G], 1 / np.sqrt(d))[0]
                np.testing.assert_allclose(O[q, a, j], ref, rtol=1e-12, atol=1e-12)


def test_b_zero_is_plain_attention_prefill():
    g = np.random.default_rng(2)
    A, c, hq, hkv, d, r, n0 = 2, 5, 4, 2, 8, 2, 6
    Q = g.standard_normal((A, c, hq, d))
    K = g.standard_normal((n0 + c, hkv, d))
    V = g.standard_normal((n0 + c, hkv, d))
    L = g.standard_normal((n0 + c, A * r))
    B = np.zeros((A, r, hkv * d))
    O = oracle.prefill(Q, K, V, L, B, n0=n0, rank=r)
    # boolean mask: True = attend; row p sees keys [0, n0+p]
    mask = np.arange(n0 + c)[None, :] <= (n0 + np.arange(c))[:, None]
    for a in range(A):
        for j in range(hq):
            ref = _sdpa(Q[a, :, j], K[:, j // 2], V[:, j // 2], 1 / np.sqrt(d), mask)
            np.testing.assert_allclose(O[a, :, j], ref, rtol=1e-12, atol=1e-12)


def test_q_zero_gives_mean_of_agent_values():
    x = _small_decode(seed=3)
    x["Q"] = np.zeros_like(x["Q"])
    O = oracle.decode(**x)
    r, d = x["rank"], x["Q"].shape[-1]
    hkv = x["K_base"].shape[1]
    G = x["Q"].shape[2] // hkv
    offs = x["offsets"]
    for q in range(len(offs) - 1):
        t0, t1 = offs[q], offs[q + 1]
        for a in range(x["Q"].shape[1]):
            # mean(V_base + L_a B_a) = mean(V_base) + mean(L_a) B_a
            Lm = x["L"][t0:t1, a * r:(a + 1) * r].mean(axis=0)
            for j in range(x["Q"].shape[2]):
                h = j // G
                want = x["V_base"][t0:t1, h].mean(axis=0) + Lm @ x["B"][a][:, h * d:(h + 1) * d]
                np.testing.assert_allclose(O[q, a, j], want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("shared", [False, True])
def test_reordered_equals_materialised(shared):
    x = _small_decode(seed=4, shared=shared)
    stride = 0 if shared else None
    O1 = oracle.decode(**x, agent_stride=stride)
    O2 = oracle.decode_reordered(**x, agent_stride=stride)
    np.testing.assert_allclose(O1, O2, rtol=1e-12, atol=1e-12)


def test_causal_row_equals_truncated_decode():
    g = np.random.default_rng(5)
    A, c, hq, hkv, d, r, n0 = 2, 6, 4, 2, 8, 3, 4
    Q = g.standard_normal((A, c, hq, d))
    K = g.standard_normal((n0 + c, hkv, d))
    V = g.standard_normal((n0 + c, hkv, d))
    L = g.standard_normal((n0 + c, A * r))
    B = g.standard_normal((A, r, hkv * d))
    O = oracle.prefill(Q, K, V, L, B, n0=n0, rank=r)
    for p in range(c):
        n = n0 + p + 1  # row p sees exactly n0+p+1 keys
        Od = oracle.decode(Q[None, :, p], K[:n], V[:n], L[:n], B, [0, n], rank=r)
        np.testing.assert_allclose(O[:, p], Od[0], rtol=1e-12, atol=1e-12)
        # and seeing one more key would change it
        if p + 1 < c:
            Od2 = oracle.decode(Q[None, :, p], K[:n + 1], V[:n + 1], L[:n + 1], B, [0, n + 1], rank=r)
            assert np.abs(Od2[0] - O[:, p]).max() > 1e-6


def test_gqa_equals_mha_with_duplicated_heads():
    x = _small_decode(seed=6, hq=6, hkv=2)
    O = oracle.decode(**x)
    G, d = 3, x["Q"].shape[-1]
    K2 = np.repeat(x["K_base"], G, axis=1)
    V2 = np.repeat(x["V_base"], G, axis=1)
    A, r = x["B"].shape[0], x["rank"]
    B2 = np.concatenate([np.concatenate([x["B"][:, :, h * d:(h + 1) * d]] * G, axis=2)
                         for h in range(2)], axis=2)
    assert B2.shape == (A, r, 6 * d)
    O2 = oracle.decode(x["Q"], K2, V2, x["L"], B2, x["offsets"], rank=r)
    np.testing.assert_allclose(O, O2, rtol=1e-12, atol=1e-12)


def test_ragged_equals_separate_requests():
    x = _small_decode(seed=7, lengths=(5, 9, 2))
    O = oracle.decode(**x)
    offs = x["offsets"]
    for q in range(3):
        t0, t1 = offs[q], offs[q + 1]
        Oq = oracle.decode(x["Q"][q:q + 1], x["K_base"][t0:t1], x["V_base"][t0:t1],
                           x["L"][t0:t1], x["B"], [0, t1 - t0], rank=x["rank"])
        np.testing.assert_allclose(O[q], Oq[0], rtol=1e-13, atol=1e-13)


def test_token_permutation_invariance():
    x = _small_decode(seed=8, lengths=(11,))
    O = oracle.decode(**x)
    perm = np.random.default_rng(0).permutation(11)
    y = dict(x, K_base=x["K_base"][perm], V_base=x["V_base"][perm], L=x["L"][perm])
    np.testing.assert_allclose(oracle.decode(**y), O, rtol=1e-12, atol=1e-12)


def test_single_token_returns_agent_value():
    x = _small_decode(seed=9, lengths=(1,))
    O = oracle.decode(**x)
    d, r = x["Q"].shape[-1], x["rank"]
    for a in range(x["Q"].shape[1]):
        Va = x["V_base"][0] + (x["L"][0, a * r:(a + 1) * r] @ x["B"][a]).reshape(-1, d)
        for j in range(x["Q"].shape[2]):
            np.testing.assert_allclose(O[0, a, j], Va[j // 2], rtol=1e-13, atol=1e-13)


def test_affine_in_b_and_agent_independence():
    x = _small_decode(seed=10)
    g = np.random.default_rng(11)
    B1, B2 = x["B"], g.standard_normal(x["B"].shape)
    O1 = oracle.decode(**x)
    O2 = oracle.decode(**dict(x, B=B2))
    O12 = oracle.decode(**dict(x, B=B1 + B2))
    O0 = oracle.decode(**dict(x, B=np.zeros_like(B1)))
    np.testing.assert_allclose(O12, O1 + O2 - O0, rtol=1e-11, atol=1e-11)
    # perturb agent 1's L block and B only: agents 0 and 2 are unchanged
    r = x["rank"]
    L = x["L"].copy()
    L[:, r:2 * r] += 5.0
    B = x["B"].copy()
    B[1] *= -3
    O3 = oracle.decode(**dict(x, L=L, B=B))
    np.testing.assert_array_equal(O3[:, [0, 2]], O1[:, [0, 2]])
    assert np.abs(O3[:, 1] - O1[:, 1]).max() > 1e-3


def test_lr_build_blocks_are_per_agent_products():
    g = np.random.default_rng(12)
    X = g.integers(-3, 4, size=(9, 5)).astype(np.float64)
    A = g.integers(-2, 3, size=(5, 3 * 2)).astype(np.float64)
    L = oracle.lr_cache_build(X, A)
    assert L.shape == (9, 6)
    for a in range(3):
        for t in range(9):
            for k in range(2):
                want = sum(X[t, i] * A[i, a * 2 + k] for i in range(5))
                assert L[t, a * 2 + k] == want


def test_oracle_accepts_bf16_workload_inputs_exactly():
    w = WORKLOADS["tiny_decode"]
    x = make_decode_inputs(w, seed=0)
    assert x["Q"].dtype == torch.float32
    Q64 = oracle.to_f64(x["Q"])
    assert np.array_equal(Q64, x["Q"].double().numpy())
    xb = make_build_inputs(4, 16, 2, 8, torch.bfloat16, seed=0)
    assert np.array_equal(oracle.to_f64(xb["X"]), xb["X"].float().double().numpy())


def test_round_to_bf16_ties_to_even():
    # 1 + 2^-8 is exactly halfway between bf16 neighbours 1 and 1 + 2^-7: even is 1
    v = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5])
    np.testing.assert_array_equal(oracle.round_to_bf16(v), [1.0, 1.0 + 2.0 ** -6, -2.5])


def test_workload_generators_are_deterministic():
    w = WORKLOADS["tiny_decode"]
    a = make_decode_inputs(w, seed=0)
    b = make_decode_inputs(w, seed=0)
    for k in a:
        assert torch.equal(a[k], b[k])
    p = make_prefill_inputs(dataclasses.replace(WORKLOADS["llama8b_prefill"], n0=8, chunk=4), seed=0)
    assert p["L"].shape == (12, 4 * 16) and p["X"].shape == (4, 4096)


def test_ragged_lengths_recipe():
    w = WORKLOADS["llama8b_ragged"]
    assert w.n_req == 32 and w.total_tokens == 614602
    assert min(w.lengths) == 4174 and max(w.lengths) == 31930


def test_agent_value_cache_by_brute_force():
    """V_i[t, h, j] = V_base[t, h, j] + sum_k L_i[t, k] B_i[k, h*d + j], element by element
    (LRAgent summary, Metodologia section 1).  Integer inputs make every product exact,
    so a transposed head slice or a dropped term shows as a mismatch."""
    rng = np.random.default_rng(5)
    n, hkv, d, r = 3, 2, 4, 3
    V = rng.integers(-3, 4, size=(n, hkv, d)).astype(np.float64)
    L = rng.integers(-2, 3, size=(n, r)).astype(np.float64)
    B = rng.integers(-2, 3, size=(r, hkv * d)).astype(np.float64)
    got = oracle.agent_value_cache(V, L, B, hkv, d)
    assert got.shape == (n, hkv, d)
    for t in range(n):
        for h in range(hkv):
            for j in range(d):
                want = V[t, h, j] + sum(L[t, k] * B[k, h * d + j] for k in range(r))
                assert got[t, h, j] == want
    # B = 0 leaves the base cache; a one-hot L row picks one row of B, split by head
    assert np.array_equal(oracle.agent_value_cache(V, L, np.zeros_like(B), hkv, d), V)
    one_hot = np.zeros((n, r))
    one_hot[:, 1] = 1.0
    picked = oracle.agent_value_cache(np.zeros_like(V), one_hot, B, hkv, d)
    assert np.array_equal(picked[0], B[1].reshape(hkv, d))


# ----------------------------------------------------------------------------
# ReBaseShared base projection fused with the LR build
# ----------------------------------------------------------------------------

def _int_rebase_inputs(n, D, hkv, d, A, r, seed):
    rng = np.random.default_rng(seed)
    return (rng.integers(-3, 4, (n, D)).astype(np.float64), rng.integers(-3, 4, (D, hkv * d)).astype(np.float64),
            rng.integers(-3, 4, (D, hkv * d)).astype(np.float64), rng.integers(-3, 4, (D, A * r)).astype(np.float64))


def test_rebase_projection_by_brute_force():
    """Every output element is the plain sum over d_model (integer inputs: exact)."""
    n, D, hkv, d, A, r = 5, 7, 2, 3, 3, 2
    X, Wk, Wv, Ac = _int_rebase_inputs(n, D, hkv, d, A, r, seed=3)
    K, V, L = oracle.rebase_kv_lr_build(X, Wk, Wv, Ac, hkv=hkv, d=d)
    for t in range(n):
        for h in range(hkv):
            for j in range(d):
                c = h * d + j
                assert K[t, h, j] == sum(X[t, k] * Wk[k, c] for k in range(D))
                assert V[t, h, j] == sum(X[t, k] * Wv[k, c] for k in range(D))
        for c in range(A * r):
            assert L[t, c] == sum(X[t, k] * Ac[k, c] for k in range(D))


def test_rebase_projection_one_hot_rows_select_weight_rows():
    """X = identity: token t's K/V/L rows are row t of W_k, W_v, A_cat (head h = columns [h*d, (h+1)*d))."""
    D, hkv, d, A, r = 6, 3, 2, 2, 3
    _, Wk, Wv, Ac = _int_rebase_inputs(1, D, hkv, d, A, r, seed=5)
    K, V, L = oracle.rebase_kv_lr_build(np.eye(D), Wk, Wv, Ac, hkv=hkv, d=d)
    for t in range(D):
        for h in range(hkv):
            np.testing.assert_array_equal(K[t, h], Wk[t, h * d:(h + 1) * d])
            np.testing.assert_array_equal(V[t, h], Wv[t, h * d:(h + 1) * d])
        np.testing.assert_array_equal(L[t], Ac[t])


def test_rebase_lr_block_matches_the_lr_build():
    x = make_build_inputs(9, 64, 2, 8, torch.bfloat16, seed=2)
    rng = np.random.default_rng(1)
    Wk, Wv = rng.standard_normal((64, 32)), rng.standard_normal((64, 32))
    _, _, L = oracle.rebase_kv_lr_build(x["X"], Wk, Wv, x["A_cat"], hkv=2, d=16)
    np.testing.assert_array_equal(L, oracle.lr_cache_build(x["X"], x["A_cat"]))
