"""The C-ABI library: it builds, loads, exports every declared entry point, and
its host-side checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from adapter_gemv_lora_gb300 import build, lora_delta
    build.build()
    return lora_delta.load_library()


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(lora_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 16
    for n in names:
        assert hasattr(lib, n), n
    # and nothing declared is missing from the binding
    from adapter_gemv_lora_gb300 import lora_delta
    for n in names:
        assert hasattr(lora_delta, n), n


def test_status_strings_and_counter(lib):
    from adapter_gemv_lora_gb300 import lora_delta as LD
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert LD.lora_status_string(code) != "unknown status"
    assert LD.lora_status_string(123) == "unknown status"
    assert LD.lora_launch_count() >= 0


def test_pool_bytes_shapes(lib):
    from adapter_gemv_lora_gb300 import lora_delta as LD
    b = LD.lora_pool_bytes(9, 16, 4096, [4096], 256)
    # factors: A + B^T + B, each 9 slots x 16 rows x 4096 bf16
    assert b >= 3 * 9 * 16 * 4096 * 2
    assert LD.lora_pool_bytes(9, 16, 4096, [4096, 1024, 1024], 17408) > b
    assert LD.lora_pool_bytes(1, 16, 4096, [4096], 1) == 0          # needs slot 0 + one adapter slot
    assert LD.lora_pool_bytes(9, 16, 4000, [4096], 1) == 0          # d_in not a multiple of 64
    assert LD.lora_pool_bytes(9, 16, 4096, [100], 1) == 0           # d_out not a multiple of 64
    assert LD.lora_pool_bytes(9, 129, 4096, [4096], 1) == 0         # rank above 128
    assert LD.lora_pool_bytes(9, 128, 4096, [64] * 4, 1) > 0        # 4 lanes x R16 128 = 512 TMEM columns
    assert LD.lora_pool_bytes(9, 16, 4096, [64] * 5, 1) == 0        # more than 4 lanes


def test_segments_bytes(lib):
    from adapter_gemv_lora_gb300 import lora_delta as LD
    assert LD.lora_segments_bytes(128, 16384, 65) > 16384 * 8
    assert LD.lora_segments_bytes(0, 16, 4) == 0
    assert LD.lora_segments_bytes(4, 16, 1) == 0
    assert LD.lora_segments_bytes(4, 16, 4097) == 0
    # the builder's per-sequence arrays move to the workspace (24 bytes a sequence) once they no
    # longer fit next to the per-slot counters in 227 KiB - 2 KiB of shared memory: no cap on max_seqs
    a, b = LD.lora_segments_bytes(7210, 16, 2048), LD.lora_segments_bytes(7211, 16, 2048)
    assert a > 0 and b >= a + 24 * 7211 - 256
    assert LD.lora_segments_bytes(20000, 16, 65) > LD.lora_segments_bytes(9523, 16, 65) + 24 * 20000 - 256
    assert LD.lora_segments_bytes(100000, 200000, 2048) > 0


def test_host_argument_errors_need_no_gpu(lib):
    from adapter_gemv_lora_gb300 import lora_delta as LD
    out = ctypes.c_void_p()
    # null memory / misaligned memory are refused before any CUDA call
    assert lib.lora_pool_create(ctypes.byref(out), None, 1 << 20, 4, 8, 256, 1,
                                (ctypes.c_int * 1)(256), 8, None) == LD.LORA_ERR_ARG
    assert lib.lora_pool_create(ctypes.byref(out), ctypes.c_void_p(0x1001), 1 << 20, 4, 8, 256, 1,
                                (ctypes.c_int * 1)(256), 8, None) == LD.LORA_ERR_ARG
    assert lib.lora_segments_create(ctypes.byref(out), None, 1 << 20, 4, 8, 4) == LD.LORA_ERR_ARG
    assert lib.lora_build_segments(None, None, None, 1, 1, None) == LD.LORA_ERR_ARG
    assert lib.lora_apply_shrink_expand(None, None, None, None, 256, 256, None) == LD.LORA_ERR_ARG
    assert lib.lora_pool_load(None, 1, 0, 8, 1.0, None, None, None) == LD.LORA_ERR_ARG
    with pytest.raises(LD.LoraError):
        LD.lora_pool_load(0, 1, 0, 8, 1.0, 0, 0)
