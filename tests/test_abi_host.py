"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every entry point include/coda.h declares with the binding's
signature table, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "coda.h")


@pytest.fixture(scope="module")
def lib():
    from gemm_epilogue_transformer_gb300 import build_lib, _lib
    build_lib.build()
    return _lib.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(coda_\w+)\s*\(", src, flags=re.M)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("coda_gemm", "coda_gemm_res_rmsprep", "coda_rms_reduce", "coda_gemm_rowscale",
                     "coda_gemm_swiglu", "coda_gemm_rope", "coda_gemm_ce_lse", "coda_gemm_swiglu_bwd",
                     "coda_gemm_rope_bwd", "coda_gemm_ce_bwd", "coda_gemm_rowdot", "coda_gemm_rmsnorm_bwd",
                     "coda_unfused_add", "coda_unfused_rmsnorm"):
        assert required in names
    assert len(names) == len(set(names))


def test_checked_build_exports_the_same_symbols():
    """libcoda_checked.so (bounds-tested epilogues) is the same boundary."""
    from gemm_epilogue_transformer_gb300 import build_lib
    path = build_lib.build(checked=True)
    chk = ctypes.CDLL(path)
    for n in declared_functions():
        assert hasattr(chk, n), f"{n} not exported by the checked build"


def test_every_declared_symbol_is_exported_and_bound(lib):
    from gemm_epilogue_transformer_gb300 import _lib
    names = declared_functions()
    for n in names:
        assert hasattr(lib, n), f"{n} not exported by libcoda.so"
        assert n in _lib.SIGNATURES, f"{n} has no binding signature"
    assert set(_lib.SIGNATURES) == set(names)


def test_argument_count_matches_header():
    from gemm_epilogue_transformer_gb300 import _lib
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    for m in re.finditer(r"(coda_\w+)\s*\(([^)]*)\)\s*;", src):
        name, args = m.group(1), m.group(2).strip()
        n = 0 if args in ("", "void") else args.count(",") + 1
        assert len(_lib.SIGNATURES[name][1]) == n, name


def _p(v):
    return ctypes.c_void_p(v)


def test_host_validation_rejects_before_launch(lib):
    INVALID, UNSUPPORTED = -1, -2
    good = _p(0x10000)
    odd = _p(0x10008)
    # negative / inconsistent dimensions
    assert lib.coda_gemm(-1, 8, 8, good, 8, 0, good, 8, 0, good, 8, None) == INVALID
    assert lib.coda_gemm(8, 8, 8, good, 8, 2, good, 8, 0, good, 8, None) == INVALID
    assert b"transA" in lib.coda_last_error()
    # null and misaligned pointers
    assert lib.coda_gemm(8, 8, 8, None, 8, 0, good, 8, 0, good, 8, None) == INVALID
    assert lib.coda_gemm(8, 8, 8, odd, 8, 0, good, 8, 0, good, 8, None) == INVALID
    assert b"16-byte" in lib.coda_last_error()
    # leading dimensions
    assert lib.coda_gemm(8, 16, 8, good, 4, 0, good, 16, 0, good, 16, None) == INVALID
    assert lib.coda_gemm(8, 16, 8, good, 8, 0, good, 16, 0, good, 12, None) == INVALID
    # granularity
    assert lib.coda_gemm_rowscale(8, 12, 8, good, good, good, good, None) == UNSUPPORTED
    assert lib.coda_gemm_swiglu(8, 12, 8, good, good, good, None, None) == UNSUPPORTED
    assert lib.coda_gemm_rope(8, 256, 8, good, good, good, good, 16, 48, 128, good, None) == UNSUPPORTED
    assert lib.coda_gemm_rope(8, 256, 8, good, good, good, good, 16, 64, 96, good, None) == INVALID
    assert lib.coda_gemm_rope(8, 256, 8, good, good, good, good, 0, 64, 128, good, None) == INVALID
    assert lib.coda_rms_reduce(8, 0, 8, good, 1e-6, good, None) == INVALID
    assert lib.coda_rms_reduce(8, 2, 8, good, -1.0, good, None) == INVALID
    assert lib.coda_set_wait_timeout_ns(10) == INVALID
    # tile variants: 0 (automatic), 1 and 2 only; the setting is process-wide
    assert [lib.coda_set_cta_group(g) for g in (3, 4, 5, -1)] == [INVALID] * 4
    assert [lib.coda_set_cta_group(g) for g in (2, 1, 0)] == [0] * 3
    # stream-K tail: 0 (off), 1 (automatic) and 2 (wherever it applies) only
    assert [lib.coda_set_stream_k(m) for m in (3, -1)] == [INVALID] * 2
    assert [lib.coda_set_stream_k(m) for m in (0, 2, 1)] == [0] * 3
    assert lib.coda_unfused_rmsnorm_bwd(8, 65536, good, good, good, good, good, good, None) == UNSUPPORTED
    # empty problems are no-ops that never touch the device
    assert lib.coda_gemm(0, 8, 8, None, 8, 0, None, 8, 0, None, 8, None) == 0
    assert lib.coda_gemm_res_rmsprep(0, 8, 8, None, None, None, None, None, None, None, None) == 0
    assert lib.coda_gemm_ce_lse(0, 8, 8, None, None, None, None, None, None, None, None) == 0
    assert lib.coda_unfused_add(0, 8, None, None, None, None) == 0


def test_tile_counts(lib):
    assert [lib.coda_num_col_tiles(n) for n in (0, 1, 128, 129, 32768)] == [0, 1, 1, 2, 256]
    assert [lib.coda_num_row_tiles(m) for m in (0, 1, 32, 33, 8192)] == [0, 1, 1, 2, 256]


def test_no_device_is_reported_not_crashed(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    good = _p(0x10000)
    rc = lib.coda_gemm(128, 256, 64, good, 64, 0, good, 256, 0, good, 256, None)
    assert rc in (-2, -3)
    assert lib.coda_last_error()


def test_block_descriptor_layout_matches_c(tmp_path):
    """The ctypes mirror of coda_block_t has the C struct's size and field
    offsets (compiled with the host C compiler against include/coda.h)."""
    import shutil
    import subprocess
    from gemm_epilogue_transformer_gb300 import _lib
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    names = [f for f, _ in _lib.CodaBlock._fields_]
    src = tmp_path / "layout.c"
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"coda.h\"\nint main(void) {\n"
                   '  printf("%zu\\n", sizeof(coda_block_t));\n'
                   + "".join(f'  printf("%zu\\n", offsetof(coda_block_t, {n}));\n' for n in names) + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    assert got[0] == ctypes.sizeof(_lib.CodaBlock)
    assert got[1:] == [getattr(_lib.CodaBlock, n).offset for n in names]


def test_block_chain_host_validation(lib):
    INVALID, UNSUPPORTED = -1, -2
    good = _p(0x10000)
    assert lib.coda_block_fwd(None, None) == INVALID
    from gemm_epilogue_transformer_gb300 import _lib
    b = _lib.CodaBlock()
    b.M, b.d, b.F = 64, 100, 64
    b.workspace = 0x10000
    assert lib.coda_block_fwd(b, None) == UNSUPPORTED          # d not a multiple of 8
    b.d = 64
    b.workspace = 0x10010
    assert lib.coda_block_bwd(b, None) == INVALID              # workspace not 256-byte aligned
    # workspace size: partials (fused), plus the unfused intermediates
    M, d, F = 1000, 256, 384
    fused = lib.coda_block_workspace_bytes(M, d, F, 0)
    assert fused >= 4 * (M * 2 + M * 3 + 32 * d)
    assert lib.coda_block_workspace_bytes(M, d, F, 1) >= fused + 2 * M * (d + F + d)
    assert lib.coda_block_workspace_bytes(-1, d, F, 0) == 0
    # composed kernels: granularity and argument checks before any launch
    assert lib.coda_gemm_rowscale_rope(8, 256, 8, good, good, good, good, good, 16, 48, 128, good, None) == UNSUPPORTED
    assert lib.coda_gemm_rowscale_rope(8, 256, 8, good, good, None, good, good, 16, 64, 128, good, None) == INVALID
    assert lib.coda_gemm_rowscale_swiglu(8, 12, 8, good, good, good, good, None, None) == UNSUPPORTED
    assert lib.coda_gemm_swiglu_bwd_rowdot(8, 16, 8, good, good, good, None, good, good, None) == INVALID
    assert lib.coda_gemm_rmsnorm_bwd_res(8, 16, 8, good, good, good, good, good, good, None, good, good,
                                         None) == INVALID
    assert lib.coda_rope_bwd_rowdot(8, 96, good, good, good, good, good, 16, 12, 48, 32, good, good,
                                    None) == UNSUPPORTED
    assert lib.coda_rope_bwd_rowdot(8, 96, good, good, good, good, good, 16, 16, 40, 32, good, good,
                                    None) == INVALID
    assert lib.coda_rope_bwd_rowdot(8, 96, good, good, good, good, good, 16, 16, 48, 0, good, good, None) == INVALID


def test_block_fwd_noalloc_host_validation(lib):
    """The allocation-free forward refuses a null descriptor, negative sizes and
    partials past its static array before it looks up any device address."""
    INVALID, UNSUPPORTED = -1, -2
    from gemm_epilogue_transformer_gb300 import _lib
    assert lib.coda_block_fwd_noalloc(None, None) == INVALID
    b = _lib.CodaBlock()
    b.M, b.d, b.F = -1, 64, 64
    assert lib.coda_block_fwd_noalloc(b, None) == INVALID
    b.M, b.d, b.F = 16384 + 32, 8192, 8192  # 64 x 4 B per row: one row block past 4 MiB
    assert lib.coda_block_fwd_noalloc(b, None) == UNSUPPORTED
    assert b"static scratch" in lib.coda_last_error()
    b.M = 0
    assert lib.coda_block_fwd_noalloc(b, None) == 0  # nothing to do, nothing launched


def test_fp8_host_validation(lib):
    INVALID, UNSUPPORTED = -1, -2
    good = _p(0x10000)
    assert lib.coda_gemm_fp8(8, 16, 24, good, good, 1.0, good, None) == UNSUPPORTED      # K % 16
    assert lib.coda_gemm_fp8(8, 12, 32, good, good, 1.0, good, None) == UNSUPPORTED      # N % 8
    assert lib.coda_gemm_fp8(8, 16, 32, good, good, float("inf"), good, None) == INVALID
    assert lib.coda_gemm_fp8(8, 16, 32, _p(0x10008), good, 1.0, good, None) == INVALID  # misaligned A
    assert lib.coda_gemm_rope_fp8(8, 256, 32, good, good, 1.0, good, good, 16, 48, 128, good, None) == UNSUPPORTED
    assert lib.coda_gemm_swiglu_fp8(8, 12, 32, good, good, 1.0, good, None, None) == UNSUPPORTED
