"""CPU oracle for the HiSA sparse-attention step (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may use it.
"""
