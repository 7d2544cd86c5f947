"""Plain CPU oracle for the batch-invariant router and projection GEMM.

Test infrastructure only: the library's product path never imports it."""
