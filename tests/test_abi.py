"""The C-ABI library on a CPU-only machine: it builds for sm_103a, loads,
exports every function include/gemm_gb300.h declares, and rejects bad
arguments before any device work.  No compute call is made here."""
import ctypes
import os
import re

import pytest

import dense_gemm_blackwell_tcgen05_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm_gb300.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(gemm_\w+)\s*\(", text, re.M)))


def test_header_declares_expected():
    assert declared_functions() == sorted(g.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol():
    L = g.load()
    for name in declared_functions():
        assert hasattr(L, name), name


def test_library_is_sm103a_only_and_needs_no_driver_at_load():
    path = g.library_path()
    assert os.path.exists(path)
    # statically linked runtime: loading works here without libcuda
    ctypes.CDLL(path)


def test_status_strings():
    for code in range(-6, 1):
        s = g.gemm_status_string(code)
        assert s and s != "unknown status"
    assert g.gemm_status_string(7) == "unknown status"


NULL = 0
FAKE = 0x7F0000000000   # never dereferenced: every case below fails validation first


@pytest.mark.parametrize("args, want", [
    (dict(M=-1, N=4, K=4, lda=8, ldb=8, ldd=4), g.GEMM_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=-4, lda=8, ldb=8, ldd=4), g.GEMM_ERR_INVALID_ARG),
    (dict(M=1 << 31, N=4, K=4, lda=8, ldb=8, ldd=4), g.GEMM_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=16, lda=8, ldb=16, ldd=4), g.GEMM_ERR_INVALID_ARG),    # lda < K
    (dict(M=4, N=4, K=16, lda=16, ldb=8, ldd=4), g.GEMM_ERR_INVALID_ARG),    # ldb < K
    (dict(M=4, N=8, K=16, lda=16, ldb=16, ldd=4), g.GEMM_ERR_INVALID_ARG),   # ldd < N
    (dict(M=4, N=4, K=12, lda=12, ldb=16, ldd=4), g.GEMM_ERR_ALIGNMENT),     # 24-byte pitch
    (dict(M=4, N=4, K=16, lda=16, ldb=20, ldd=4), g.GEMM_ERR_ALIGNMENT),
    (dict(M=0, N=4, K=16, lda=16, ldb=16, ldd=4), g.GEMM_OK),               # empty: no-op
    (dict(M=4, N=0, K=16, lda=16, ldb=16, ldd=4), g.GEMM_OK),
])
def test_bf16_validation(args, want):
    rc = g.gemm_bf16(FAKE, FAKE, FAKE, args["M"], args["N"], args["K"], args["lda"], args["ldb"],
                     args["ldd"], 0)
    assert rc == want


def test_bf16_null_and_misaligned_pointers():
    assert g.gemm_bf16(NULL, FAKE, FAKE, 4, 4, 16, 16, 16, 4, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_bf16(FAKE, FAKE, NULL, 4, 4, 16, 16, 16, 4, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_bf16(FAKE + 8, FAKE, FAKE, 4, 4, 16, 16, 16, 4, 0) == g.GEMM_ERR_ALIGNMENT
    # D's elements must sit at their own alignment (2 bytes for bf16)
    assert g.gemm_bf16(FAKE, FAKE, FAKE + 1, 4, 4, 16, 16, 16, 4, 0) == g.GEMM_ERR_ALIGNMENT
    e = g.GemmEpilogue()
    e.alpha, e.out_dtype = 1.0, g.DTYPE_F32
    assert g.gemm_bf16_fused(0, FAKE, FAKE, FAKE + 2, 4, 4, 16, 16, 16, 4, e, 0) == g.GEMM_ERR_ALIGNMENT
    e.out_dtype, e.bias, e.bias_dtype = g.DTYPE_BF16, FAKE + 1, g.DTYPE_BF16
    assert g.gemm_bf16_fused(0, FAKE, FAKE, FAKE, 4, 4, 16, 16, 16, 4, e, 0) == g.GEMM_ERR_ALIGNMENT


def test_variant_validation():
    assert g.gemm_bf16_variant(9, FAKE, FAKE, FAKE, 4, 4, 16, 16, 16, 4, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_bf16_variant(0x200, FAKE, FAKE, FAKE, 4, 4, 16, 16, 16, 4, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_mxfp8_variant(g.VARIANT_SYNC, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 4, 32, 32, 32, 16,
                                16, 4, 0) == g.GEMM_ERR_INVALID_ARG


def test_mxfp8_validation():
    f = lambda **k: g.gemm_mxfp8(k.get("A", FAKE), FAKE, k.get("SFA", FAKE), FAKE, FAKE, 4, 4,
                                 k.get("K", 64), k.get("lda", 64), 64, k.get("ldsfa", 16), 16, 4, 0)
    assert f(lda=40, K=40) == g.GEMM_ERR_ALIGNMENT          # E4M3 pitch must be 16-byte multiple
    assert f(K=1024, lda=1024, ldsfa=16) == g.GEMM_ERR_INVALID_ARG   # ldsfa < ceil(K/32)
    assert f(SFA=NULL) == g.GEMM_ERR_INVALID_ARG
    # scale matrices take any pitch >= ceil(K/32) and any alignment (plain-load
    # gather where TMA cannot read them): past validation, these reach the
    # device checks (no device here; the fake pointers on a GPU machine)
    past = (g.GEMM_ERR_UNSUPPORTED_DEVICE, g.GEMM_ERR_INVALID_ARG)
    assert f(ldsfa=2) in past
    assert f(ldsfa=8) in past
    assert f(SFA=FAKE + 4) in past
    assert f(SFA=FAKE + 1, ldsfa=3) in past


def test_no_device_is_reported_not_crashed():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # valid-looking arguments reach the device check, which fails cleanly
    assert g.gemm_bf16(FAKE, FAKE, FAKE, 4, 4, 16, 16, 16, 4, 0) == g.GEMM_ERR_UNSUPPORTED_DEVICE


def test_smallk_plan_and_validation():
    p = g.gemm_kernel_plan(False, g.VARIANT_SMALLK)
    assert p["tmem_cols"] == 0 and p["threads"] == 256 and p["tile_n"] == 256
    # K beyond the small-K limit, a workspace or an epilogue: refused before device work
    assert g.gemm_bf16_variant(4, FAKE, FAKE, FAKE, 4, 4, 17, 24, 24, 4, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_bf16_streamk(4, FAKE, FAKE, FAKE, 4, 4, 8, 8, 8, 4, FAKE, 1 << 20, 0) == \
        g.GEMM_ERR_INVALID_ARG
    assert g.gemm_bf16_fused(4, FAKE, FAKE, FAKE, 4, 4, 8, 8, 8, 4, g.GemmEpilogue(), 0) == \
        g.GEMM_ERR_INVALID_ARG
    assert g.gemm_bf16_variant(6, FAKE, FAKE, FAKE, 4, 4, 8, 8, 8, 4, 0) == g.GEMM_ERR_INVALID_ARG
    # the tensor-core small-K kernel takes the same limits
    assert g.gemm_bf16_variant(g.VARIANT_SMALLK_TC, FAKE, FAKE, FAKE, 4, 4, 17, 24, 24, 4, 0) == \
        g.GEMM_ERR_INVALID_ARG
    assert g.gemm_bf16_fused(g.VARIANT_SMALLK_TC, FAKE, FAKE, FAKE, 4, 4, 8, 8, 8, 4,
                             g.GemmEpilogue(), 0) == g.GEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("mx, variant", [(0, 1), (0, 2), (0, 3), (0, 0x101), (0, 0x102), (1, 1), (1, 0x101),
                                        (1, 2)])
def test_kernel_plans_fit_the_sm(mx, variant):
    p = g.gemm_kernel_plan(bool(mx), variant)
    assert 0 <= p["smem_bytes"] <= 232448
    assert p["tmem_cols"] in (128, 256, 512)
    assert p["stages"] >= 1
    if (variant & 0xFF) == 2:
        assert p["cluster"] == 2 and p["tile_m"] == 256 and p["tile_n"] == (224 if mx else 256)
    if (variant & 0xFF) in (1, 2):
        assert p["stages"] >= 3


def test_quantize_validation():
    q = lambda **k: g.gemm_mxfp8_quantize(k.get("X", FAKE), k.get("rows", 4), k.get("K", 64),
                                          k.get("ldx", 64), k.get("Q", FAKE), k.get("ldq", 64),
                                          k.get("SF", FAKE), k.get("ldsf", 2), 0)
    assert q(rows=-1) == g.GEMM_ERR_INVALID_ARG
    assert q(K=-1) == g.GEMM_ERR_INVALID_ARG
    assert q(ldx=63) == g.GEMM_ERR_INVALID_ARG
    assert q(ldq=10) == g.GEMM_ERR_INVALID_ARG
    assert q(ldsf=1) == g.GEMM_ERR_INVALID_ARG
    assert q(X=NULL) == g.GEMM_ERR_INVALID_ARG
    assert q(rows=0) == g.GEMM_OK and q(K=0) == g.GEMM_OK


def test_streamk_validation_without_device():
    # a NULL workspace is refused before anything else
    assert g.gemm_bf16_streamk(2, FAKE, FAKE, FAKE, 4, 4, 16, 16, 16, 4, NULL, 1 << 20, 0) == \
        g.GEMM_ERR_INVALID_ARG
    assert g.gemm_mxfp8_streamk(1, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 4, 32, 32, 32, 16, 16, 4, NULL,
                                1 << 20, 0) == g.GEMM_ERR_INVALID_ARG
    # shapes are checked like the data-parallel entry points
    assert g.gemm_bf16_streamk(2, FAKE, FAKE, FAKE, -1, 4, 16, 16, 16, 4, FAKE, 1 << 20, 0) == \
        g.GEMM_ERR_INVALID_ARG
    assert g.gemm_bf16_streamk(0x40, FAKE, FAKE, FAKE, 4, 4, 16, 16, 16, 4, FAKE, 1 << 20, 0) == \
        g.GEMM_ERR_INVALID_ARG
    sched = g.gemm_last_schedule()
    assert set(sched) == {"clusters", "ctas_per_cluster", "dp_tiles", "sk_tiles", "sk_unit",
                          "half_tiles", "edge_last"}


def test_streamk_workspace_query_without_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert g.gemm_streamk_workspace_bytes(False, 2) == g.GEMM_ERR_UNSUPPORTED_DEVICE


def test_noalloc_variant_checked_before_device_setup():
    assert g.gemm_bf16_streamk_noalloc(3, FAKE, FAKE, FAKE, 4, 4, 16, 16, 16, 4, 0) == \
        g.GEMM_ERR_INVALID_ARG


def test_epilogue_struct_layout_matches_the_header(tmp_path):
    """The ctypes mirror of gemm_epilogue_t has the C compiler's layout."""
    import ctypes
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "gemm_gb300.h"\n'
        "int main(void) { printf(\"%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\\n\", sizeof(gemm_epilogue_t),"
        " offsetof(gemm_epilogue_t, alpha), offsetof(gemm_epilogue_t, beta),"
        " offsetof(gemm_epilogue_t, C), offsetof(gemm_epilogue_t, ldc),"
        " offsetof(gemm_epilogue_t, bias), offsetof(gemm_epilogue_t, bias_dtype),"
        " offsetof(gemm_epilogue_t, activation), offsetof(gemm_epilogue_t, out_dtype),"
        " offsetof(gemm_epilogue_t, reserved)); return 0; }\n")
    exe = tmp_path / "layout"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.run(["gcc", "-I", inc, "-o", str(exe), str(src)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    E = g.GemmEpilogue
    want = [ctypes.sizeof(E)] + [getattr(E, f).offset for f in
                                 ("alpha", "beta", "C", "ldc", "bias", "bias_dtype", "activation",
                                  "out_dtype", "reserved")]
    assert got == want


def test_fused_validation_without_device():
    e = g.GemmEpilogue()
    e.alpha = 1.0
    # the synchronous ladder kernels take no epilogue; checked before any device work
    assert g.gemm_bf16_fused(3, FAKE, FAKE, FAKE, 4, 4, 16, 16, 16, 4, e, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_bf16_fused(0x40, FAKE, FAKE, FAKE, 4, 4, 16, 16, 16, 4, e, 0) == \
        g.GEMM_ERR_INVALID_ARG
    assert g.gemm_bf16_fused(2, FAKE, FAKE, FAKE, -1, 4, 16, 16, 16, 4, e, 0) == \
        g.GEMM_ERR_INVALID_ARG
