"""GB300-native tiled GEMM D = alpha*A*B + beta*C with shape:stride layout addressing.

  gemm      the sm_103a GEMM through its C ABI (include/gb300_gemm.h)
  layout    the host layout library through its C ABI (include/layout_algebra.h)
  workloads seeded synthetic operands
The native library loads on first use and every entry point raises if it is missing.
"""
from .binding import GemmError, gemm, last_device_status, plan, status_string  # noqa: F401
from . import layout  # noqa: F401
