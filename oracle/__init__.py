"""fp64 CPU oracle for the fused DiT QK-RMSNorm + RoPE step.

Test infrastructure only: the tests, the smoke check and the benchmark's
CPU-baseline leg use it; the CUDA library and its binding never do.
"""
