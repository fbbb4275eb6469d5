"""CPU oracle for Flash-LoRA-Attention over a decomposed KV cache (fp64).

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline / reference arm may import this package.  The CUDA
library never calls it and shares no code with it.

What it computes follows the plain definition on the pages, not the
kernel's reordering:

* LR cache (LRAgent summary, "Metodologia" section 2, BaseShared bullet;
  PReCache abstract, PreLRShared): agent i stores L_i = X . A_i, the LoRA
  down-projection of the context hidden states, at width r.
* Value decomposition (LRAgent summary, section 1, "Descomposicion de la
  Cache"): the agent's value cache is the shared base part plus the adapter
  output, V_i = V_base + L_i . B_i.  The oracle materialises V_i at full
  width, exactly the "naive reconstruction" that section 3
  ("Flash-LoRA-Attention", Problema bullet) describes.
* Base-cache rebuild (PReCache abstract, ReBaseShared): K_base = X . W_k and
  V_base = X . W_v from adapter-free hidden states with the pretrained
  weights, computed together with every agent's L_i = X . A_i.
* Attention: O = softmax(q . K_base^T / sqrt(d)) . V_i, softmax taken with
  the maximum subtracted, all in fp64.  Keys carry no adapter term.

`decode_reordered` evaluates the reordered form P.V_base + (P.L_i).B_i of
section 3 (Solucion bullet).  It exists only so the tests can check the
identity the kernel relies on; the attention functions never use it.

Inputs may be torch tensors or numpy arrays of any float dtype; they are
converted to fp64 exactly (bf16 and fp32 values are representable in fp64).

Pins (tests/test_oracle.py): hand-derived tiny cases in tests/golden/,
B = 0 against torch's scaled_dot_product_attention in fp64, Q = 0 against
the mean of V_i, reordered vs materialised, causal visibility, GQA against
duplicated-head MHA, ragged against separate requests, token permutation,
n = 1, lr_cache_build against brute-force sums on integer inputs, and
rebase_kv_lr_build against a hand-derived case, brute force and closed forms.
"""
from .reference import (  # noqa: F401
    lr_cache_build,
    rebase_kv_lr_build,
    agent_value_cache,
    decode,
    decode_reordered,
    prefill,
    to_f64,
    round_to_bf16,
)
