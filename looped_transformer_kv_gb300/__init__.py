"""ResidualQuant decode attention for GB300: librq (C ABI, CUDA sm_103a) + a thin
PyTorch binding.  See include/rq.h for the boundary."""

from .rq import (  # noqa: F401
    PackedCache,
    bf16_decode_attention,
    cache_bytes,
    decode_attention,
    decode_workspace_bytes,
    encode_append,
    make_shape,
    res_bits_of,
    synth_params,
    synth_queries,
    synth_states,
)
