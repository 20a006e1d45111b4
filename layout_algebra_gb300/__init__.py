"""GB300-native tiled GEMM D = alpha*A*B + beta*C with layout-algebra addressing."""
