"""Python face of the GEMM C ABI (include/gb300_gemm.h): argument marshalling only.

``gemm`` takes torch tensors holding the STORED operands (see include/gb300_gemm.h for
the K-major / MN-major conventions) and calls gb_gemm_f16 / gb_gemm_bf16 on the current
CUDA stream.  When the operands are host tensors it calls gb_gemm_f16_host /
gb_gemm_bf16_host, which stage them to the device, run the GEMM and copy D back into a
host tensor (the row blocks and the copy/compute overlap live in the library): that is the
end-to-end path a caller holding host buffers uses.
"""
import ctypes

import torch

from ._native import Epilogue, GemmPlan, lib

K_MAJOR, MN_MAJOR = 0, 1
F16, BF16 = 0, 1


class GemmError(RuntimeError):
    def __init__(self, status, what="gemm"):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (what, status_string(status), status))


def status_string(status):
    return lib().gb_status_string(int(status)).decode()


def major_code(m):
    if m in (K_MAJOR, "K", "k"):
        return K_MAJOR
    if m in (MN_MAJOR, "MN", "mn", "M", "N"):
        return MN_MAJOR
    raise ValueError("major must be 'K' or 'MN'")


def dtype_code(dt):
    if dt in (torch.float16, "f16", "fp16"):
        return F16
    if dt in (torch.bfloat16, "bf16"):
        return BF16
    raise TypeError("operands must be float16 or bfloat16")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


# ----------------------------------------------------------------------------- host operands


def row_blocks(M):
    """Row blocks [m0, m1) in which a host-operand call stages A, C and D (gb_gemm_host_row_blocks)."""
    bounds = (ctypes.c_int64 * 9)()
    n = ctypes.c_int()
    st = lib().gb_gemm_host_row_blocks(M, bounds, ctypes.byref(n))
    if st != 0:
        raise GemmError(st, "row_blocks")
    return [(bounds[i], bounds[i + 1]) for i in range(n.value)]


def host_staging_free():
    """Free this device's staging buffer of the host-operand calls."""
    st = lib().gb_host_staging_free()
    if st != 0:
        raise GemmError(st, "host_staging_free")


def _host_out(D, numel, dtype):
    """The host tensor that receives D: the caller's, or a new pinned one."""
    if D is None:
        return torch.empty(numel, dtype=dtype, pin_memory=True)
    if D.is_cuda:
        raise TypeError("with host operands, D must be a host tensor")
    return D


def gemm(A, B, M, N, K, *, lda, ldb, majorA="K", majorB="K", alpha=1.0, beta=0.0, C=None,
         D=None, stream=None, workspace=None):
    """D = alpha * A @ B + beta * C.  Returns D (M*N elements, row-major).

    A, B, C are flat (or any contiguous) tensors of one dtype.  Device tensors: D is
    written in place (allocated if None).  Host tensors: gb_gemm_*_host stages them to the
    device in row blocks overlapped with the GEMM, and D (a host tensor, pinned if
    allocated here) receives the result once the stream reaches the end of the call.
    """
    dt = dtype_code(A.dtype)
    if B.dtype != A.dtype or (C is not None and C.dtype != A.dtype):
        raise TypeError("A, B and C must share one dtype")

    def call(A_ptr, B_ptr, C_ptr, D_ptr, rows, s):
        if workspace is None:
            fn = lib().gb_gemm_bf16 if dt == BF16 else lib().gb_gemm_f16
            st = fn(rows, N, K, float(alpha), A_ptr, lda, major_code(majorA), B_ptr, ldb,
                    major_code(majorB), float(beta), C_ptr, D_ptr, _stream_handle(s))
        else:
            fn = lib().gb_gemm_bf16_ws if dt == BF16 else lib().gb_gemm_f16_ws
            st = fn(rows, N, K, float(alpha), A_ptr, lda, major_code(majorA), B_ptr, ldb,
                    major_code(majorB), float(beta), C_ptr, D_ptr, workspace.data_ptr(),
                    workspace.numel() * workspace.element_size(), _stream_handle(s))
        if st != 0:
            raise GemmError(st)

    if not A.is_cuda:
        if workspace is not None:
            raise ValueError("host operands take no workspace")
        D_h = _host_out(D, M * N, A.dtype)
        fn = lib().gb_gemm_bf16_host if dt == BF16 else lib().gb_gemm_f16_host
        st = fn(M, N, K, float(alpha), _ptr(A), lda, major_code(majorA), _ptr(B), ldb,
                major_code(majorB), float(beta), _ptr(C), _ptr(D_h), _stream_handle(stream))
        if st != 0:
            raise GemmError(st, "gemm (host operands)")
        return D_h
    D_d = D if D is not None else torch.empty(M * N, dtype=A.dtype, device=A.device)
    call(_ptr(A), _ptr(B), _ptr(C), _ptr(D_d), M, stream)
    return D_d


ACTIVATIONS = {"none": 0, "relu": 1, "gelu": 2}
OUT_FORMATS = {"input": 0, "e4m3": 1, "e5m2": 2}


def gemm_fused(A, B, M, N, K, *, lda, ldb, majorA="K", majorB="K", alpha=1.0, beta=0.0, C=None,
               bias=None, activation="none", amax=None, out_format="input", out_scale=1.0,
               D=None, workspace=None, stream=None):
    """D = epilogue(alpha*A@B + beta*C) through gb_gemm_ex (device tensors only).

    bias: N values of the input dtype; amax: a 1-element float32 device tensor (combined by
    max with its contents); out_format "e4m3"/"e5m2" returns float8 tensors of M*N elements.
    """
    dt = dtype_code(A.dtype)
    fmt = OUT_FORMATS[out_format]
    if D is None:
        out_dtype = {0: A.dtype, 1: torch.float8_e4m3fn, 2: torch.float8_e5m2}[fmt]
        D = torch.empty(M * N, dtype=out_dtype, device=A.device)
    epi = Epilogue(_ptr(bias), ACTIVATIONS[activation], _ptr(amax), fmt, float(out_scale))
    st = lib().gb_gemm_ex(dt, M, N, K, float(alpha), _ptr(A), lda, major_code(majorA), _ptr(B),
                          ldb, major_code(majorB), float(beta), _ptr(C), _ptr(D),
                          ctypes.byref(epi), _ptr(workspace),
                          0 if workspace is None else workspace.numel() * workspace.element_size(),
                          _stream_handle(stream))
    if st != 0:
        raise GemmError(st, "gemm_fused")
    return D


FP8_FORMATS = {"e4m3": 0, "e5m2": 1}


def fp8_format(x):
    if x in FP8_FORMATS:
        return FP8_FORMATS[x]
    if x == torch.float8_e4m3fn:
        return 0
    if x == torch.float8_e5m2:
        return 1
    raise TypeError("FP8 operands must be e4m3 (float8_e4m3fn) or e5m2 (float8_e5m2)")


def gemm_fp8(A, B, M, N, K, *, lda, ldb, a_format=None, b_format=None, out_dtype=torch.bfloat16,
             alpha=1.0, beta=0.0, C=None, bias=None, activation="none", amax=None,
             out_format="input", out_scale=1.0, D=None, workspace=None, stream=None):
    """D = epilogue(alpha*A@B + beta*C) with FP8 inputs through gb_gemm_fp8.

    A (M x K, leading dimension lda) and B (stored as N rows of K, leading dimension ldb) are
    K-major byte tensors: float8_e4m3fn / float8_e5m2, or uint8 codes with a_format /
    b_format naming the format.  C, D and bias are of out_dtype; per-tensor scales belong in
    alpha.  out_format "e4m3"/"e5m2" gives a float8 D.  Host operands (with a host bias and
    a host amax) go through gb_gemm_fp8_host, as for ``gemm``.
    """
    fa = fp8_format(a_format if a_format is not None else A.dtype)
    fb = fp8_format(b_format if b_format is not None else B.dtype)
    od = dtype_code(out_dtype)
    fmt = OUT_FORMATS[out_format]
    dd = {0: out_dtype, 1: torch.float8_e4m3fn, 2: torch.float8_e5m2}[fmt]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()

    def call(A_ptr, B_ptr, C_ptr, bias_ptr, D_ptr, rows, s):
        epi = Epilogue(bias_ptr, ACTIVATIONS[activation], _ptr(amax), fmt, float(out_scale))
        st = lib().gb_gemm_fp8(fa, fb, od, rows, N, K, float(alpha), A_ptr, lda, B_ptr, ldb,
                               float(beta), C_ptr, D_ptr, ctypes.byref(epi), _ptr(workspace),
                               ws_bytes, _stream_handle(s))
        if st != 0:
            raise GemmError(st, "gemm_fp8")

    if not A.is_cuda:
        if workspace is not None:
            raise ValueError("host operands take no workspace")
        D_h = _host_out(D, M * N, dd)
        epi = Epilogue(_ptr(bias), ACTIVATIONS[activation], _ptr(amax), fmt, float(out_scale))
        st = lib().gb_gemm_fp8_host(fa, fb, od, M, N, K, float(alpha), _ptr(A), lda, _ptr(B), ldb,
                                    float(beta), _ptr(C), _ptr(D_h), ctypes.byref(epi),
                                    _stream_handle(stream))
        if st != 0:
            raise GemmError(st, "gemm_fp8 (host operands)")
        return D_h
    if D is None:
        D = torch.empty(M * N, dtype=dd, device=A.device)
    call(_ptr(A), _ptr(B), _ptr(C), _ptr(bias), _ptr(D), M, stream)
    return D


def mx_scales_bytes(operand, rows, K):
    """Bytes of the packed scale buffer of operand 0 (A, rows = M) or 1 (B, rows = N)."""
    n = ctypes.c_size_t()
    st = lib().gb_mx_scales_bytes(int(operand), rows, K, ctypes.byref(n))
    if st != 0:
        raise GemmError(st, "mx_scales_bytes")
    return n.value


def mx_pack_scales(operand, rows, K, scales, ld=None, stream=None):
    """Pack rows x ceil(K/32) E8M0 scales (a uint8 device tensor, row pitch ld) for
    gemm_mxfp8; returns the packed uint8 device tensor."""
    ld = -(-K // 32) if ld is None else ld
    out = torch.empty(mx_scales_bytes(operand, rows, K), dtype=torch.uint8, device=scales.device)
    st = lib().gb_mx_pack_scales(int(operand), rows, K, _ptr(scales), ld, _ptr(out),
                                 _stream_handle(stream))
    if st != 0:
        raise GemmError(st, "mx_pack_scales")
    return out


def gemm_mxfp8(A, B, M, N, K, *, lda, ldb, sfa, sfb, a_format=None, b_format=None,
               out_dtype=torch.bfloat16, alpha=1.0, beta=0.0, C=None, bias=None, activation="none",
               amax=None, out_format="input", out_scale=1.0, D=None, workspace=None, stream=None):
    """Block-scaled FP8 GEMM through gb_gemm_mxfp8 (device tensors).  A, B as for gemm_fp8;
    sfa / sfb are packed scales from mx_pack_scales (operand 0 with M rows, 1 with N rows)."""
    fa = fp8_format(a_format if a_format is not None else A.dtype)
    fb = fp8_format(b_format if b_format is not None else B.dtype)
    od = dtype_code(out_dtype)
    fmt = OUT_FORMATS[out_format]
    if D is None:
        dd = {0: out_dtype, 1: torch.float8_e4m3fn, 2: torch.float8_e5m2}[fmt]
        D = torch.empty(M * N, dtype=dd, device=A.device)
    epi = Epilogue(_ptr(bias), ACTIVATIONS[activation], _ptr(amax), fmt, float(out_scale))
    st = lib().gb_gemm_mxfp8(fa, fb, od, M, N, K, float(alpha), _ptr(A), lda, _ptr(sfa), _ptr(B), ldb,
                             _ptr(sfb), float(beta), _ptr(C), _ptr(D), ctypes.byref(epi),
                             _ptr(workspace),
                             0 if workspace is None else workspace.numel() * workspace.element_size(),
                             _stream_handle(stream))
    if st != 0:
        raise GemmError(st, "gemm_mxfp8")
    return D


def raw_call(dtype, M, N, K, alpha, A_ptr, lda, majorA, B_ptr, ldb, majorB, beta, C_ptr, D_ptr,
             stream_handle):
    """Direct C-ABI call with integer pointers; returns the status code."""
    fn = lib().gb_gemm_bf16 if dtype_code(dtype) == BF16 else lib().gb_gemm_f16
    return fn(M, N, K, float(alpha), A_ptr, lda, major_code(majorA), B_ptr, ldb,
              major_code(majorB), float(beta), C_ptr, D_ptr, stream_handle)


def raw_call_ws(dtype, M, N, K, alpha, A_ptr, lda, majorA, B_ptr, ldb, majorB, beta, C_ptr,
                D_ptr, ws_ptr, ws_bytes, stream_handle):
    """Direct C-ABI call of the workspace (stream-K) entry point; returns the status."""
    fn = lib().gb_gemm_bf16_ws if dtype_code(dtype) == BF16 else lib().gb_gemm_f16_ws
    return fn(M, N, K, float(alpha), A_ptr, lda, major_code(majorA), B_ptr, ldb,
              major_code(majorB), float(beta), C_ptr, D_ptr, ws_ptr, ws_bytes, stream_handle)


def plan(dtype, M, N, K, lda, majorA, ldb, majorB):
    """Host-side plan (tile grid, copy geometry, instruction descriptor) as a dict."""
    p = GemmPlan()
    st = lib().gb_gemm_make_plan(dtype_code(dtype), M, N, K, lda, major_code(majorA), ldb,
                                 major_code(majorB), ctypes.byref(p))
    if st != 0:
        raise GemmError(st, "plan")
    out = {}
    for name, _ in GemmPlan._fields_:
        v = getattr(p, name)
        out[name] = list(v) if hasattr(v, "__len__") else v
    return out


def last_device_status(stream=None):
    """(status, detail) of the device status word; synchronises the stream."""
    detail = ctypes.c_uint32()
    st = lib().gb_last_device_status(_stream_handle(stream), ctypes.byref(detail))
    return st, detail.value


def set_wait_timeout_ns(ns):
    lib().gb_set_wait_timeout_ns(int(ns))


def debug_skip_k_block(kb):
    lib().gb_debug_skip_k_block(int(kb))


def workspace_bytes():
    """Bytes of scratch the *_ws calls need on the current device."""
    n = ctypes.c_size_t()
    st = lib().gb_gemm_workspace_bytes(ctypes.byref(n))
    if st != 0:
        raise GemmError(st, "workspace_bytes")
    return n.value


def make_workspace(device=None):
    """A zero-filled workspace for the *_ws calls (allocated once by the caller)."""
    return torch.zeros(workspace_bytes(), dtype=torch.uint8,
                       device=device if device is not None else torch.device("cuda"))


def set_schedule(schedule):
    """0 (default): stream-K, given a workspace, when the tiles are fewer than the CTAs and each
    CTA gets two stage-blocks; 1: whole tiles only; 2: stream-K whenever a workspace is given."""
    st = lib().gb_set_schedule(int(schedule))
    if st != 0:
        raise GemmError(st, "set_schedule")


def set_kernel_variant(variant):
    """0: choose by shape; 1: single-CTA 128x256 kernel; 2: CTA-pair 256x256 kernel."""
    st = lib().gb_set_kernel_variant(int(variant))
    if st != 0:
        raise GemmError(st, "set_kernel_variant")
