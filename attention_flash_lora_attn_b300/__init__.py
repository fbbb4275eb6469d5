"""Flash-LoRA-Attention for B300 (sm_103a).

Public API (thin wrappers over the C ABI in include/flash_lora_attn.h):
  lr_cache_build(X, A_cat, L=None)          L = X . A_cat for every agent at once
  rebase_kv_lr_build(X, W_cat, ...)         [K_base | V_base | L] = X . [W_k | W_v | A_cat] in one pass
  flash_lora_attn_decode(Q, K_base, V_base, L, B, offsets, rank=...)
  flash_lora_attn_prefill(Q, K_base, V_base, L, B, n0, rank=...)
  PreparedDecode(...)                       a decode call marshalled once, one C call per step
  PreparedDecodeHostIO(...)                 the same with host Q in / host O out in that one call
  lora_value_expand(V_base, L, B, rank=...) every agent's V_i = V_base + L_i.B_i (baseline only)
  device_error()                            read and clear the device error word

All compute runs in the library's CUDA kernels; the library must have been
built (`python -m attention_flash_lora_attn_b300.build_lib`).

`baselines` holds the naive-materialisation and non-shared-cache decodes the
reordered decode is compared with; they are not part of the hot path.
"""
from .binding import (  # noqa: F401
    EXPORTED,
    LIB_PATH,
    FlaError,
    PreparedDecode,
    PreparedDecodeHostIO,
    device_error,
    flash_lora_attn_decode,
    flash_lora_attn_prefill,
    load_library,
    lora_value_expand,
    lr_cache_build,
    rebase_kv_lr_build,
    selftest_bounded_wait,
    version,
)

__version__ = "0.1.0"
