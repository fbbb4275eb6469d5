"""Plain fp64 definitions of the LR-cache build and LoRA attention.

TEST INFRASTRUCTURE ONLY (see the package docstring): never called by the
CUDA library or its Python binding.

Sources are cited by page and section:
  [LRAgent-1]  LRAgent technical summary (gist.science), Metodologia,
               section 1 "Descomposicion de la Cache".
  [LRAgent-2]  same page, section 2 "Esquemas de Intercambio"
               (BaseShared and BaseLRShared bullets).
  [LRAgent-3]  same page, section 3 "Flash-LoRA-Attention".
  [PReCache]   PReCache abstract (arxivdaily), PreLRShared paragraph.
  [ReBase]     same abstract, ReBaseShared paragraph (the shared base cache
               rebuilt from adapter-free hidden states with the pretrained
               weights).

Readings taken where the pages are silent:
  * softmax scale is 1/sqrt(d) unless the caller passes another value;
  * the adapter acts on values only; keys are base-only;
  * LoRA's alpha/r factor is folded into B (no extra scale);
  * B_i has shape [r, Hkv*d]; kv head h uses columns [h*d, (h+1)*d), and the
    width-r LR cache of an agent is shared by all its heads;
  * q head j reads kv head floor(j / (Hq/Hkv));
  * a decode query sees every cached token of its request; a prefill query
    at chunk position p sees keys [0, n0 + p] (inclusive causal bound);
  * an empty context gives an all-zero output row.
"""
from __future__ import annotations

import numpy as np


def to_f64(x) -> np.ndarray:
    """Exact fp64 copy of a torch tensor (any float dtype) or numpy array."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even), as fp64.

    Used where the method stores a result in bf16 (the LR cache is kept in
    the same storage type as the rest of the KV cache).
    """
    import torch

    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).to(torch.float64).numpy()


def lr_cache_build(X, A_cat) -> np.ndarray:
    """LR cache L = X . [A_1 | ... | A_A] in fp64  ([LRAgent-2] BaseShared; [PReCache]).

    X is [n, D] (one hidden-state row per token), A_cat is [D, A*r] with agent
    i's down-projection A_i in columns [i*r, (i+1)*r).  Column block i of the
    result is agent i's LR cache L_i = X . A_i.  Building every agent's block
    in one product is PreLRShared's "precompute each agent's LR cache when the
    context is first processed".
    """
    return to_f64(X) @ to_f64(A_cat)


def rebase_kv_lr_build(X, W_k, W_v, A_cat, hkv: int, d: int):
    """Base K/V caches and every agent's LR cache from one set of hidden states, fp64.

    [ReBase]: the shared base cache is computed from adapter-free hidden
    states X with the pretrained projections, K_base = X . W_k and
    V_base = X . W_v ([LRAgent-1]: the base part of the value cache comes from
    the frozen pretrained weights; keys carry no adapter term).  [PReCache]:
    each agent's LR cache L_i = X . A_i is computed in the same pass over X.
    No rotary embedding or other position encoding is applied here.

    X [n, D]; W_k, W_v [D, Hkv*d]; A_cat [D, A*r].  Returns
    (K_base [n, Hkv, d], V_base [n, Hkv, d], L [n, A*r]).
    """
    X = to_f64(X)
    n = X.shape[0]
    K_base = (X @ to_f64(W_k)).reshape(n, hkv, d)
    V_base = (X @ to_f64(W_v)).reshape(n, hkv, d)
    L = X @ to_f64(A_cat)
    return K_base, V_base, L


def agent_value_cache(V_base, L_i, B_i, hkv: int, d: int) -> np.ndarray:
    """Materialised value cache of one agent, V_i = V_base + L_i . B_i  ([LRAgent-1]).

    V_base [n, Hkv, d]; L_i [n, r]; B_i [r, Hkv*d].  Returns [n, Hkv, d].
    This is the full-width expansion (cost n*r*d_out) that [LRAgent-3] calls
    the naive reconstruction.
    """
    V_base = to_f64(V_base)
    delta = to_f64(L_i) @ to_f64(B_i)  # [n, Hkv*d]
    return V_base + delta.reshape(V_base.shape[0], hkv, d)


def _softmax_attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """softmax(q . K^T * scale) . V for one query row; zero row if K is empty."""
    if K.shape[0] == 0:
        return np.zeros(V.shape[1])
    s = (K @ q) * scale
    w = np.exp(s - s.max())
    w /= w.sum()
    return w @ V


def _agent_cols(a: int, rank: int, agent_stride: int) -> slice:
    start = a * agent_stride
    return slice(start, start + rank)


def decode(Q, K_base, V_base, L, B, offsets, rank: int, scale: float = None,
           agent_stride: int = None) -> np.ndarray:
    """One decode token per agent per request, over a packed ragged context.

    Q [R, A, Hq, d]; K_base, V_base [N, Hkv, d]; L [N, ldL]; B [A, r, Hkv*d];
    offsets [R+1] (request q owns tokens offsets[q] .. offsets[q+1]-1).
    Agent a's LR cache is L[:, a*agent_stride : a*agent_stride + r];
    agent_stride defaults to r (one block per agent, BaseShared) and 0 means
    all agents read the same block (BaseLRShared, [LRAgent-2]).
    Returns O [R, A, Hq, d] in fp64.
    """
    Q, K, V, L, B = (to_f64(t) for t in (Q, K_base, V_base, L, B))
    offs = [int(o) for o in np.asarray(offsets).reshape(-1)]
    R, A, hq, d = Q.shape
    hkv = K.shape[1]
    G = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if agent_stride is None:
        agent_stride = rank
    O = np.zeros((R, A, hq, d))
    for q_req in range(R):
        t0, t1 = offs[q_req], offs[q_req + 1]
        Kq = K[t0:t1]
        for a in range(A):
            Va = agent_value_cache(V[t0:t1], L[t0:t1, _agent_cols(a, rank, agent_stride)],
                                   B[a], hkv, d)
            for j in range(hq):
                h = j // G
                O[q_req, a, j] = _softmax_attend(Q[q_req, a, j], Kq[:, h], Va[:, h], scale)
    return O


def decode_reordered(Q, K_base, V_base, L, B, offsets, rank: int, scale: float = None,
                     agent_stride: int = None) -> np.ndarray:
    """Same result as `decode`, evaluated as P.V_base + (P.L_i).B_i  ([LRAgent-3]).

    Used by the tests only, to check the associativity identity in fp64.
    """
    Q, K, V, L, B = (to_f64(t) for t in (Q, K_base, V_base, L, B))
    offs = [int(o) for o in np.asarray(offsets).reshape(-1)]
    R, A, hq, d = Q.shape
    hkv = K.shape[1]
    G = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if agent_stride is None:
        agent_stride = rank
    O = np.zeros((R, A, hq, d))
    for q_req in range(R):
        t0, t1 = offs[q_req], offs[q_req + 1]
        if t1 == t0:
            continue
        for a in range(A):
            La = L[t0:t1, _agent_cols(a, rank, agent_stride)]
            for j in range(hq):
                h = j // G
                s = (K[t0:t1, h] @ Q[q_req, a, j]) * scale
                p = np.exp(s - s.max())
                p /= p.sum()
                O[q_req, a, j] = p @ V[t0:t1, h] + (p @ La) @ B[a][:, h * d:(h + 1) * d]
    return O


def prefill(Q, K_base, V_base, L, B, n0: int, rank: int, scale: float = None,
            agent_stride: int = None, positions=None) -> np.ndarray:
    """Causal chunked prefill of c new tokens for every agent.

    Q [A, c, Hq, d]; K_base, V_base [n0+c, Hkv, d]; L [n0+c, ldL];
    B [A, r, Hkv*d].  The query at chunk position p (absolute position n0+p)
    sees keys 0 .. n0+p inclusive.  Returns O [A, c, Hq, d] in fp64.
    `positions` restricts the work to those chunk positions (the other rows
    of O stay zero); it selects rows, it does not change their arithmetic.
    """
    Q, K, V, L, B = (to_f64(t) for t in (Q, K_base, V_base, L, B))
    A, c, hq, d = Q.shape
    hkv = K.shape[1]
    G = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if agent_stride is None:
        agent_stride = rank
    O = np.zeros((A, c, hq, d))
    for a in range(A):
        Va = agent_value_cache(V, L[:, _agent_cols(a, rank, agent_stride)], B[a], hkv, d)
        for j in range(hq):
            h = j // G
            for p in (range(c) if positions is None else positions):
                vis = n0 + p + 1
                O[a, p, j] = _softmax_attend(Q[a, p, j], K[:vis, h], Va[:vis, h], scale)
    return O
