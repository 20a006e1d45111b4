"""Python face of the GEMM C ABI (include/gb300_gemm.h): argument marshalling only.

``gemm`` takes torch tensors holding the STORED operands (see include/gb300_gemm.h for
the K-major / MN-major conventions) and calls gb_gemm_f16 / gb_gemm_bf16 on the current
CUDA stream.  When the operands are host tensors the call stages them to the device with
torch copies, runs the same C-ABI call, and copies D back into a host tensor: that is the
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
#
# A call with host (pinned) operands stages them to the device and reads D back.  With
# K-major A and enough rows, the problem is cut into row blocks of A, C and D (multiples
# of 256 rows, so every block starts 16-byte aligned): B goes up first, then block i's A
# and C rows go up on one copy stream while block i-1 is multiplied on the caller's stream
# and block i-2's D rows come down on another, so the two copy directions and the GEMM
# overlap.  Each block is one C-ABI call on the sub-matrices (M' rows, pointers offset by
# the block's first row); a block's outputs are the same as in one call over all rows.

_copy_streams = {}


def _copy_pair(dev):
    s = _copy_streams.get(dev.index)
    if s is None:
        s = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))
        _copy_streams[dev.index] = s
    return s


def row_blocks(M, chunkable):
    """Row blocks [m0, m1) of a host-operand call: up to 8 blocks of >= 1024 rows, each a
    multiple of 256 rows except the last."""
    if not chunkable or M < 2048:
        return [(0, M)]
    n = min(8, M // 1024)
    rows = -(-M // n)
    rows = -(-rows // 256) * 256
    return [(m0, min(M, m0 + rows)) for m0 in range(0, M, rows)]


def _staged(M, N, A, a_row_elems, B, C, extras, D_host, out_dtype, launch, stream):
    """Run launch(A_d, B_d, C_d, D_d, extras_d, m0, m1, s) over row blocks with host operands
    staged to the device.  a_row_elems: elements of A per row (lda) when A's rows are
    contiguous (K-major), else None (A goes up whole before the first block)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    main = stream if stream is not None else torch.cuda.current_stream(dev)
    up, down = _copy_pair(dev)
    with torch.cuda.stream(main):
        A_d = torch.empty(A.numel(), dtype=A.dtype, device=dev)
        B_d = torch.empty(B.numel(), dtype=B.dtype, device=dev)
        C_d = torch.empty(C.numel(), dtype=C.dtype, device=dev) if C is not None else None
        D_d = torch.empty(M * N, dtype=out_dtype, device=dev)
        ex_d = [torch.empty(t.numel(), dtype=t.dtype, device=dev) if t is not None else None
                for t in extras]
    if D_host is None:
        D_host = torch.empty(M * N, dtype=out_dtype, pin_memory=True)
    up.wait_stream(main)
    down.wait_stream(main)
    blocks = row_blocks(M, a_row_elems is not None)
    with torch.cuda.stream(up):
        B_d.copy_(B, non_blocking=True)
        for t, t_d in zip(extras, ex_d):
            if t is not None:
                t_d.copy_(t, non_blocking=True)
        if a_row_elems is None:
            A_d.copy_(A, non_blocking=True)
    for m0, m1 in blocks:
        with torch.cuda.stream(up):
            if a_row_elems is not None:
                a0, a1 = m0 * a_row_elems, min(m1 * a_row_elems, A.numel())
                A_d[a0:a1].copy_(A[a0:a1], non_blocking=True)
            if C is not None:
                C_d[m0 * N:m1 * N].copy_(C[m0 * N:m1 * N], non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(up)
        main.wait_event(ready)
        launch(A_d, B_d, C_d, D_d, ex_d, m0, m1, main)
        done = torch.cuda.Event()
        done.record(main)
        down.wait_event(done)
        with torch.cuda.stream(down):
            D_host[m0 * N:m1 * N].copy_(D_d[m0 * N:m1 * N], non_blocking=True)
    # the caller's stream sees D on the host; the staging buffers (allocated on it) are
    # released only after every copy that touches them
    main.wait_stream(down)
    main.wait_stream(up)
    return D_host


def gemm(A, B, M, N, K, *, lda, ldb, majorA="K", majorB="K", alpha=1.0, beta=0.0, C=None,
         D=None, stream=None, workspace=None):
    """D = alpha * A @ B + beta * C.  Returns D (M*N elements, row-major).

    A, B, C are flat (or any contiguous) tensors of one dtype.  Device tensors: D is
    written in place (allocated if None).  Host tensors: operands are staged to the device
    in row blocks overlapped with the GEMM, and D (a host tensor, pinned if given so)
    receives the result.
    """
    dt = dtype_code(A.dtype)
    if B.dtype != A.dtype or (C is not None and C.dtype != A.dtype):
        raise TypeError("A, B and C must share one dtype")
    esz = A.element_size()

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
        k_major_a = major_code(majorA) == K_MAJOR

        def launch(A_s, B_s, C_s, D_s, _ex, m0, m1, s):
            # block rows m0..m1: A K-major starts m0 rows of lda in (M-major A is never cut)
            call(A_s.data_ptr() + m0 * lda * esz, B_s.data_ptr(),
                 None if C_s is None else C_s.data_ptr() + m0 * N * esz,
                 D_s.data_ptr() + m0 * N * esz, m1 - m0, s)

        return _staged(M, N, A, lda if k_major_a else None, B, C, [], D, A.dtype, launch, stream)
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
    alpha.  out_format "e4m3"/"e5m2" gives a float8 D.  Host operands are staged to the
    device and D (a host tensor, pinned if given so) receives the result, as for ``gemm``.
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
        csz = torch.empty(0, dtype=out_dtype).element_size()
        dsz = torch.empty(0, dtype=dd).element_size()

        def launch(A_s, B_s, C_s, D_s, ex, m0, m1, s):
            call(A_s.data_ptr() + m0 * lda, B_s.data_ptr(),
                 None if C_s is None else C_s.data_ptr() + m0 * N * csz,
                 None if ex[0] is None else ex[0].data_ptr(),
                 D_s.data_ptr() + m0 * N * dsz, m1 - m0, s)

        return _staged(M, N, A, lda, B, C, [bias], D, dd, launch, stream)
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
