"""C ABI: every declared symbol is exported, and the host-side planning and validation
(no GPU needed) behave as include/gb300_gemm.h states."""
import os
import re

import pytest

from layout_algebra_gb300 import _native, binding as G

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b((?:gb|la)_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_library_loads_and_exports_every_declared_symbol():
    lib = _native.lib()
    decl = declared_functions()
    assert len(decl) >= 20
    missing = [n for n in decl if not hasattr(lib, n)]
    assert not missing
    assert set(decl) >= set(_native.GEMM_SYMBOLS) | set(_native.LAYOUT_SYMBOLS)


def test_status_strings():
    assert G.status_string(0) == "ok"
    assert "misaligned" in G.status_string(2)
    assert "10.3" in G.status_string(3)


@pytest.fixture(params=[1, 2, 5, 6, 7], ids=["single", "pair", "pair224", "pair512", "pair448"])
def variant(request):
    G.set_kernel_variant(request.param)
    yield request.param
    G.set_kernel_variant(0)


@pytest.mark.parametrize("name,M,N,K,majors,grid1,grid2", [
    ("gemm256_int_f16", 256, 256, 256, ("K", "K"), (2, 1, 4), (1, 1, 4)),
    ("gemm4096_f16", 4096, 4096, 4096, ("K", "K"), (32, 16, 64), (16, 16, 64)),
    ("gemm8192_bf16_c", 8192, 8192, 8192, ("K", "K"), (64, 32, 128), (32, 32, 128)),
    ("gemm16384x1024x4096_mnmajor_f16", 16384, 1024, 4096, ("MN", "MN"), (128, 4, 64), (64, 4, 64)),
    ("gemm5000x3000x4104_ragged_f16", 5000, 3000, 4104, ("K", "K"), (40, 12, 65), (20, 12, 65)),
])
def test_plans_of_the_workloads(variant, name, M, N, K, majors, grid1, grid2):
    lda = K if majors[0] == "K" else M
    ldb = K if majors[1] == "K" else N
    p = G.plan("f16", M, N, K, lda, majors[0], ldb, majors[1])
    # 224-column tiles need K-major B: a forced 224 (448) variant with MN-major B runs as the
    # pair (the 512-column pair)
    want = {5: 2, 7: 6}.get(variant, variant) if majors[1] == "MN" else variant
    grid = grid1 if want == 1 else grid2
    tile_m = 128 if want == 1 else 256
    tile_n = {5: 224, 6: 512, 7: 448}.get(want, 256)
    if want in (5, 6, 7):
        grid = (grid[0], -(-N // tile_n), grid[2])
    rows_b = {1: 256, 2: 128, 5: 112, 6: 128, 7: 112}[want]    # B rows one copy box stages per CTA
    mma_n = {6: 256, 7: 224}.get(want, tile_n)                 # the wide tiles take two MMAs
    assert p["variant"] == want and p["tile_m"] == tile_m and p["tile_n"] == tile_n
    assert (p["m_tiles"], p["n_tiles"], p["k_blocks"]) == grid
    # a grid mode of extent 1 is only ever indexed at 0: its stride is immaterial
    for i, (ext, want) in enumerate(zip(grid[:2], [tile_m * N, tile_n])):
        if ext > 1:
            assert p["d_grid_stride"][i] == want
    assert p["d_elem_stride"] == [N, 1]
    if majors[0] == "K":
        assert p["a_dim"] == [K, M] and p["a_box"] == [64, 128] and p["a_boxes"] == 1
        assert p["a_row_bytes"] == 2 * lda
    else:
        assert p["a_dim"] == [M, K] and p["a_box"] == [64, 64] and p["a_boxes"] == 2
    if majors[1] == "K":
        assert p["b_dim"] == [K, N] and p["b_box"] == [64, rows_b] and p["b_boxes"] == 1
    else:
        assert p["b_dim"] == [N, K] and p["b_box"] == [64, 64] and p["b_boxes"] == rows_b // 64
    # instruction descriptor: fp32 accumulate, fp16 inputs, majors, N/8, M/16
    d = p["instr_desc"]
    assert (d >> 4) & 3 == 1 and (d >> 7) & 7 == 0 and (d >> 10) & 7 == 0
    assert (d >> 15) & 1 == (majors[0] == "MN") and (d >> 16) & 1 == (majors[1] == "MN")
    assert (d >> 17) & 63 == mma_n >> 3 and (d >> 24) & 31 == tile_m >> 4
    assert p["vector_epilogue"] == 1


def test_variant_choice_by_shape():
    """Default choice (a plan made without a GPU assumes 152 SMs, 76 CTA pairs)."""
    G.set_kernel_variant(0)
    # small outputs: narrow 128 x 64 tiles while they fit in one wave (one per SM)
    assert G.plan("f16", 128, 512, 64, 64, "K", 64, "K")["variant"] == 4      # 8 tiles
    assert G.plan("f16", 256, 256, 256, 256, "K", 256, "K")["variant"] == 4   # 8 tiles
    assert G.plan("f16", 1024, 1216, 64, 64, "K", 64, "K")["variant"] == 4    # 8 x 19 = 152 tiles
    # then the single CTA while its 128 x 256 tiles fit in one wave
    assert G.plan("f16", 1024, 1280, 64, 64, "K", 64, "K")["variant"] == 1    # 160 narrow, 40 single
    assert G.plan("f16", 2048, 2048, 512, 512, "K", 512, "K")["variant"] == 1  # 128 single tiles
    assert G.plan("f16", 19456, 256, 64, 64, "K", 64, "K")["variant"] == 1    # 152 single tiles
    # CTA pairs: the width whose waves of tiles cost least (per-k-block times 0.324 / 0.339 /
    # 0.645 us for 224 / 256 / 512 columns, plus 1 us of exposed epilogue per 512-column tile)
    assert G.plan("f16", 19584, 256, 64, 64, "K", 64, "K")["variant"] == 2    # 3 waves of 224 vs 2 of 256
    p = G.plan("f16", 4096, 4096, 4096, 4096, "K", 4096, "K")                 # 4 x 224: 83 us, 2 x 512: 85
    assert p["variant"] == 5 and (p["m_tiles"], p["n_tiles"], p["tile_n"]) == (16, 19, 224)
    assert p["b_box"] == [64, 112] and (p["instr_desc"] >> 17) & 63 == 224 >> 3
    p = G.plan("bf16", 8192, 8192, 8192, 8192, "K", 8192, "K")                # 7 x 512: 585 us, 14 x 256: 608
    assert p["variant"] == 6 and (p["m_tiles"], p["n_tiles"], p["tile_n"]) == (32, 16, 512)
    assert p["b_box"] == [64, 128] and (p["instr_desc"] >> 17) & 63 == 256 >> 3
    # rows of 4104 halves (8208 bytes) are not 128-byte aligned: a wide tile copies fewer bytes per
    # flop, and 7 columns of 448 fill their 2 waves better than 6 of 512
    assert G.plan("f16", 5000, 3000, 4104, 4104, "K", 4104, "K")["variant"] == 7
    assert G.plan("f16", 16384, 1024, 4096, 16384, "MN", 1024, "MN")["variant"] == 6   # 2 x 512 vs 4 x 256
    assert G.plan("f16", 4096, 4096, 4096, 4096, "K", 4096, "MN")["variant"] == 6   # MN-major B: no 224
    # at most 64 output columns: narrow 128 x 64 tiles
    p = G.plan("f16", 4096, 16, 4096, 4096, "K", 4096, "K")
    assert p["variant"] == 4 and (p["tile_m"], p["tile_n"]) == (128, 64)
    assert (p["m_tiles"], p["n_tiles"], p["k_blocks"]) == (32, 1, 64)
    assert p["b_box"] == [64, 64] and (p["instr_desc"] >> 17) & 63 == 64 >> 3
    with pytest.raises(G.GemmError):
        G.set_kernel_variant(8)
    # 3 was a form whose B tiles were copied into two CTA pairs at once (copy multicast); it
    # is gone, and asking for it is an argument error
    assert G.lib().gb_set_kernel_variant(3) == 1
    assert G.lib().gb_set_kernel_variant(0) == 0


def test_plan_bf16_descriptor_and_scalar_epilogue(variant):
    p = G.plan("bf16", 129, 77, 40, 40, "K", 40, "K")
    assert (p["instr_desc"] >> 7) & 7 == 1 and (p["instr_desc"] >> 10) & 7 == 1
    assert p["vector_epilogue"] == 0          # rows of 77 elements are not 16-byte aligned
    assert (p["m_tiles"], p["n_tiles"], p["k_blocks"]) == ((2, 1, 1) if variant == 1 else (1, 1, 1))


@pytest.mark.parametrize("args,status", [
    ((-1, 8, 8, 8, "K", 8, "K"), 1),
    ((8, 8, 8, 4, "K", 8, "K"), 1),           # lda < K
    ((8, 8, 8, 8, "MN", 8, "K"), 0),
    ((8, 8, 12, 12, "K", 16, "K"), 2),        # lda*2 = 24 bytes: not a multiple of 16
    ((8, 8, 8, 8, "K", 20, "K"), 2),
    ((8, 8, 8, 8, "K", 8, 7), 1),             # bad major
    ((1 << 31, 8, 8, 1 << 31, "MN", 8, "K"), 1),
])
def test_plan_validation(args, status):
    M, N, K, lda, ma, ldb, mb = args
    if isinstance(mb, int) and mb not in (0, 1):
        rc = _native.lib().gb_gemm_make_plan(0, M, N, K, lda, 0, ldb, mb,
                                             __import__("ctypes").byref(_native.GemmPlan()))
        assert rc == status
        return
    if status == 0:
        G.plan("f16", M, N, K, lda, ma, ldb, mb)
    else:
        with pytest.raises(G.GemmError) as e:
            G.plan("f16", M, N, K, lda, ma, ldb, mb)
        assert e.value.status == status


def test_gemm_call_validation_without_gpu():
    """Argument errors come back before any device is touched."""
    lib = _native.lib()
    # negative size
    assert lib.gb_gemm_f16(-1, 8, 8, 1.0, 16, 8, 0, 16, 8, 0, 0.0, None, 16, None) == 1
    # empty problem: nothing to do
    assert lib.gb_gemm_f16(0, 8, 8, 1.0, None, 8, 0, None, 8, 0, 0.0, None, None, None) == 0
    # beta != 0 needs C
    assert lib.gb_gemm_f16(8, 8, 8, 1.0, 16, 8, 0, 16, 8, 0, 1.0, None, 16, None) == 1
    # D missing
    assert lib.gb_gemm_f16(8, 8, 8, 1.0, 16, 8, 0, 16, 8, 0, 0.0, None, None, None) == 1
    # misaligned pointers
    assert lib.gb_gemm_bf16(8, 8, 8, 1.0, 18, 8, 0, 16, 8, 0, 0.0, None, 16, None) == 2
    assert lib.gb_gemm_bf16(8, 8, 8, 1.0, 16, 8, 0, 16, 8, 0, 0.0, None, 24, None) == 2


def test_host_row_blocks():
    """Row blocks of a host-operand call (gb_gemm_host_row_blocks): up to 8 blocks of >= 1024
    rows, multiples of 256 rows (every block's first row keeps 16-byte alignment), covering
    [0, M) exactly."""
    from layout_algebra_gb300 import binding as G
    assert G.row_blocks(1000) == [(0, 1000)]
    assert G.row_blocks(2047) == [(0, 2047)]
    assert G.row_blocks(8192) == [(i * 1024, (i + 1) * 1024) for i in range(8)]
    assert G.row_blocks(5000) == [(0, 1280), (1280, 2560), (2560, 3840), (3840, 5000)]
    for M in (2048, 2049, 3000, 4097, 16384, 100000):
        b = G.row_blocks(M)
        assert b[0][0] == 0 and b[-1][1] == M and len(b) <= 8
        assert all(m1 == n0 for (_, m1), (n0, _) in zip(b, b[1:]))
        assert all(m0 % 256 == 0 and m1 - m0 >= 1 for m0, m1 in b)
