"""fp64 CPU oracle for causal GQA attention forward/backward.

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline leg may import this package.  The CUDA library never uses it.
"""
