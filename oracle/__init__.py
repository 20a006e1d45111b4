"""Oracle package: CPU definitions the GPU path is checked against (TEST INFRASTRUCTURE).

Only tests/, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg may import
anything here.  Nothing in the product package imports this package, and this package
imports nothing from the product package.

  gemm_ref    fp64 GEMM reference (C, OpenMP) + acceptance bound
  layout_ref  definitional shape:stride layout semantics in plain Python
"""
