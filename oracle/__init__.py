"""Test infrastructure: the CPU oracle (plain C via ctypes).  Only tests/, the smoke
check and the benchmark's CPU-baseline leg may import this package."""
