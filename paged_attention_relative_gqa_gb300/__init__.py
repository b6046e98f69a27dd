"""GB300 (sm_103a) paged prefill/decode attention with a per-token relative-position bias.

The compute lives in ``libinkling_attn.so`` (hand-written CUDA behind a C ABI,
declared in ``include/inkling_attn.h``).  ``binding`` marshals torch tensors into that
ABI; ``workloads`` makes seeded synthetic inputs.  Importing this package does not load
the CUDA library; the first call through ``binding`` does, and fails loudly if it is
missing.
"""

__all__ = ["binding", "workloads"]
