"""ctypes loader for libgb300gemm.so (argument types only; no computation here).

The library is built in-tree by ``layout_algebra_gb300.build.build()``.  Nothing in this
package falls back to another implementation: if the library is missing, every call
raises.
"""
import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgb300gemm.so")

GEMM_SYMBOLS = [
    "gb_gemm_f16", "gb_gemm_bf16", "gb_last_device_status", "gb_status_string",
    "gb_gemm_make_plan", "gb_set_wait_timeout_ns", "gb_debug_skip_k_block",
    "gb_debug_epilogue_map", "gb_debug_stage_bytes", "gb_set_kernel_variant",
    "gb_gemm_f16_ws", "gb_gemm_bf16_ws", "gb_gemm_workspace_bytes", "gb_set_schedule",
    "gb_gemm_noalloc", "gb_gemm_ex", "gb_gemm_fp8", "gb_gemm_mxfp8", "gb_mx_scales_bytes",
    "gb_mx_pack_scales", "gb_gemm_f16_host", "gb_gemm_bf16_host", "gb_gemm_fp8_host",
    "gb_gemm_host_row_blocks", "gb_host_staging_free",
]
LAYOUT_SYMBOLS = [
    "la_error_string", "la_size", "la_cosize", "la_eval", "la_eval_coord", "la_coalesce",
    "la_composition", "la_complement", "la_logical_divide", "la_zipped_divide",
    "la_local_tile", "la_local_partition", "la_print_layout", "la_logical_product",
    "la_swizzle", "la_local_tile_proj",
]


class NativeLibraryMissing(RuntimeError):
    pass


class Epilogue(ctypes.Structure):
    _fields_ = [("bias", ctypes.c_void_p), ("activation", ctypes.c_int),
                ("amax", ctypes.c_void_p), ("out_format", ctypes.c_int),
                ("out_scale", ctypes.c_float)]


class GemmPlan(ctypes.Structure):
    _fields_ = [
        ("m_tiles", ctypes.c_int64), ("n_tiles", ctypes.c_int64), ("k_blocks", ctypes.c_int64),
        ("tile_m", ctypes.c_int64), ("tile_n", ctypes.c_int64), ("tile_k", ctypes.c_int64),
        ("a_dim", ctypes.c_int64 * 2), ("a_row_bytes", ctypes.c_int64),
        ("a_box", ctypes.c_int64 * 2), ("a_boxes", ctypes.c_int64),
        ("b_dim", ctypes.c_int64 * 2), ("b_row_bytes", ctypes.c_int64),
        ("b_box", ctypes.c_int64 * 2), ("b_boxes", ctypes.c_int64),
        ("d_grid_stride", ctypes.c_int64 * 2), ("d_elem_stride", ctypes.c_int64 * 2),
        ("instr_desc", ctypes.c_uint32), ("vector_epilogue", ctypes.c_int32),
        ("variant", ctypes.c_int32),
    ]


_lib = None


def lib():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise NativeLibraryMissing(
            "libgb300gemm.so is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    i64, f32, vp, ci = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int
    cp, sz = ctypes.c_char_p, ctypes.c_size_t
    for name in ("gb_gemm_f16", "gb_gemm_bf16", "gb_gemm_f16_host", "gb_gemm_bf16_host"):
        fn = getattr(L, name)
        fn.restype = ci
        fn.argtypes = [i64, i64, i64, f32, vp, i64, ci, vp, i64, ci, f32, vp, vp, vp]
    for name in ("gb_gemm_f16_ws", "gb_gemm_bf16_ws"):
        fn = getattr(L, name)
        fn.restype = ci
        fn.argtypes = [i64, i64, i64, f32, vp, i64, ci, vp, i64, ci, f32, vp, vp, vp, sz, vp]
    L.gb_gemm_ex.restype = ci
    L.gb_gemm_ex.argtypes = [ci, i64, i64, i64, f32, vp, i64, ci, vp, i64, ci, f32, vp, vp,
                             ctypes.POINTER(Epilogue), vp, sz, vp]
    L.gb_gemm_fp8.restype = ci
    L.gb_gemm_fp8.argtypes = [ci, ci, ci, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, vp,
                              ctypes.POINTER(Epilogue), vp, sz, vp]
    L.gb_gemm_mxfp8.restype = ci
    L.gb_gemm_mxfp8.argtypes = [ci, ci, ci, i64, i64, i64, f32, vp, i64, vp, vp, i64, vp, f32, vp, vp,
                                ctypes.POINTER(Epilogue), vp, sz, vp]
    L.gb_gemm_fp8_host.restype = ci
    L.gb_gemm_fp8_host.argtypes = [ci, ci, ci, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, vp,
                                   ctypes.POINTER(Epilogue), vp]
    L.gb_gemm_host_row_blocks.restype = ci
    L.gb_gemm_host_row_blocks.argtypes = [i64, ctypes.POINTER(i64), ctypes.POINTER(ci)]
    L.gb_host_staging_free.restype = ci
    L.gb_host_staging_free.argtypes = []
    L.gb_mx_scales_bytes.restype = ci
    L.gb_mx_scales_bytes.argtypes = [ci, i64, i64, ctypes.POINTER(sz)]
    L.gb_mx_pack_scales.restype = ci
    L.gb_mx_pack_scales.argtypes = [ci, i64, i64, vp, i64, vp, vp]
    L.gb_gemm_noalloc.restype = ci
    L.gb_gemm_noalloc.argtypes = [ci, i64, i64, i64, f32, vp, i64, ci, vp, i64, ci, f32, vp, vp, vp]
    L.gb_gemm_workspace_bytes.restype = ci
    L.gb_gemm_workspace_bytes.argtypes = [ctypes.POINTER(sz)]
    L.gb_set_schedule.restype = ci
    L.gb_set_schedule.argtypes = [ci]
    L.gb_last_device_status.restype = ci
    L.gb_last_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    L.gb_status_string.restype = cp
    L.gb_status_string.argtypes = [ci]
    L.gb_gemm_make_plan.restype = ci
    L.gb_gemm_make_plan.argtypes = [ci, i64, i64, i64, i64, ci, i64, ci, ctypes.POINTER(GemmPlan)]
    L.gb_set_wait_timeout_ns.restype = ci
    L.gb_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    L.gb_debug_skip_k_block.restype = ci
    L.gb_debug_skip_k_block.argtypes = [i64]
    L.gb_debug_epilogue_map.restype = ci
    L.gb_debug_epilogue_map.argtypes = [ci, i64, i64, i64, i64, vp, vp]
    L.gb_set_kernel_variant.restype = ci
    L.gb_set_kernel_variant.argtypes = [ci]
    L.gb_debug_stage_bytes.restype = ci
    L.gb_debug_stage_bytes.argtypes = [ci, ci, i64, i64, i64, vp, i64, ci, vp, i64, ci, i64,
                                       i64, vp, vp]
    L.la_error_string.restype = cp
    L.la_error_string.argtypes = [ci]
    L.la_size.restype = ci
    L.la_size.argtypes = [cp, ctypes.POINTER(i64)]
    L.la_cosize.restype = ci
    L.la_cosize.argtypes = [cp, ctypes.POINTER(i64)]
    L.la_eval.restype = ci
    L.la_eval.argtypes = [cp, vp, i64, vp]
    L.la_eval_coord.restype = ci
    L.la_eval_coord.argtypes = [cp, vp, ci, ctypes.POINTER(i64)]
    for name in ("la_coalesce",):
        getattr(L, name).restype = ci
        getattr(L, name).argtypes = [cp, cp, sz]
    for name in ("la_composition", "la_logical_divide", "la_zipped_divide"):
        getattr(L, name).restype = ci
        getattr(L, name).argtypes = [cp, cp, cp, sz]
    L.la_complement.restype = ci
    L.la_complement.argtypes = [cp, i64, cp, sz]
    L.la_local_tile.restype = ci
    L.la_local_tile.argtypes = [cp, cp, vp, ci, ctypes.POINTER(i64), cp, sz]
    L.la_local_tile_proj.restype = ci
    L.la_local_tile_proj.argtypes = [cp, cp, vp, vp, ci, ctypes.POINTER(i64), cp, sz]
    L.la_local_partition.restype = ci
    L.la_local_partition.argtypes = [cp, cp, i64, ctypes.POINTER(i64), cp, sz]
    L.la_logical_product.restype = ci
    L.la_logical_product.argtypes = [cp, cp, cp, sz]
    L.la_swizzle.restype = ci
    L.la_swizzle.argtypes = [ci, ci, ci, vp, i64, vp]
    L.la_print_layout.restype = ci
    L.la_print_layout.argtypes = [cp, cp, sz]
    _lib = L
    return L
