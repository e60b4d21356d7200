"""CPU oracle for the affine-packed dequantise-into-matmul path.

Test infrastructure only: the tests, the smoke check and the benchmark's
CPU-baseline leg may import it; the library and its binding never do.
"""
