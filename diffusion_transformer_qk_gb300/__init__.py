"""GB300 (sm_103a) kernels for diffusion-transformer attention prologues.

- ``qknr``: ctypes binding of ``libqknr.so`` — fused per-head QK-RMSNorm +
  RoPE (``qk_norm_rope_packed``, ``qk_norm_rope_tensor``,
  ``qk_norm_rope_separate``, ``HostPipeline``), AdaLN scale/shift
  (``adaln_modulate``) and group norm + SiLU (``group_norm_silu``).
- ``build``: compiles ``libqknr.so`` in-tree with nvcc.
- ``inputs``: seeded synthetic workloads (Wan, FLUX.2 and VAE shapes).

Importing the package loads nothing; ``qknr.load()`` (called by every
entry point) loads the library and raises if it is not built.
"""
