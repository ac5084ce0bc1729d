"""Column-sparse (Mx1-slice) attention for video diffusion transformers on GB300.

The compute path is the C-ABI library ``libsparse_attn.so`` (hand-written
sm_103a kernels); :mod:`video_dit_sparse_gb300.binding` marshals torch
tensors into it.  :mod:`video_dit_sparse_gb300.inputs` draws seeded
synthetic workloads.
"""
