"""KDA (Kimi Delta Attention) for NVIDIA GB300: a C-ABI CUDA library for
sm_103a (include/kda.h) with a thin Python binding.

    from linear_attention_03_gb300 import kda
    out, final_state = kda.kda_prefill(q, k, v, g, beta, init_state, cu_seqlens)
    out = kda.kda_decode_step(q, k, v, g, beta, state)
    q, k, v, g, beta = kda.kda_prologue(q_raw, k_raw, v_raw, conv_w, z_g, z_beta)

Build the library first: ``python -m linear_attention_03_gb300.build``.
Importing ``linear_attention_03_gb300.kda`` raises if it is missing.
"""
