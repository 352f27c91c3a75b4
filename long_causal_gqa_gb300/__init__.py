"""GB300-native (sm_103a) causal grouped-query attention prefill.

The compute runs in the CUDA library libh3gqa.so (C ABI in include/h3gqa.h);
`binding` marshals arguments to it and `inputs` draws seeded synthetic inputs.
"""
from .binding import (H3GQAError, attention_fwd, causal_gqa_fwd, h3gqa_attention_fwd,  # noqa: F401
                      h3gqa_attention_plan, h3gqa_causal_fwd, h3gqa_make_plan,
                      h3gqa_status_string, h3gqa_sync_and_check, h3gqa_version)
