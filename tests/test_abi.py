"""The C ABI: the library builds for sm_103a, loads, exports every function that
include/tkg_gemm.h declares, and rejects bad arguments on the host before any
CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "tkg_gemm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tkg_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from dense_block_scaled_gb300 import build, tkg
    build.build()
    return tkg.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 10
    from dense_block_scaled_gb300 import tkg
    assert set(names) == set(tkg.EXPORTS)
    for name in names:
        assert hasattr(lib, name), name


def test_host_side_argument_checks(lib):
    from dense_block_scaled_gb300 import tkg
    # negative sizes are rejected before anything touches CUDA
    assert tkg.gemm_bf16_raw(-1, 8, 8, 16, 16, 16, 1.0, None) == tkg.ERR_INVALID_ARG
    assert tkg.gemm_mxfp8_raw(8, -8, 32, 16, 16, 16, 16, 16, 1.0, None) == tkg.ERR_INVALID_ARG
    assert tkg.gemm_nvfp4_raw(8, 8, -32, 16, 16, 16, 16, None, None, 16, 1.0, None) == tkg.ERR_INVALID_ARG
    # empty GEMMs are a no-op
    assert tkg.gemm_bf16_raw(0, 8, 8, None, None, None, 1.0, None) == tkg.OK
    assert tkg.gemm_nvfp4_raw(8, 0, 32, None, None, None, None, None, None, None, 1.0, None) == tkg.OK
    # misaligned output pitch / pointer
    assert tkg.gemm_bf16_raw(8, 12, 8, 16, 16, 16, 1.0, None) == tkg.ERR_ALIGNMENT
    assert tkg.gemm_bf16_raw(8, 8, 8, 16, 16, 24, 1.0, None) == tkg.ERR_ALIGNMENT
    assert tkg.gemm_bf16_raw(8, 8, 8, None, 16, 16, 1.0, None) == tkg.ERR_INVALID_ARG


def test_scale_bytes(lib):
    from dense_block_scaled_gb300 import tkg
    assert tkg.scale_bytes(1, 32, 32) == 128 * 4
    assert tkg.scale_bytes(128, 128, 32) == 128 * 4
    assert tkg.scale_bytes(129, 4000, 16) == 256 * 252
    assert tkg.scale_bytes(16384, 16384, 16) == 16384 * 1024
    assert tkg.scale_bytes(5, 64, 8) == 0


def test_options_roundtrip(lib):
    from dense_block_scaled_gb300 import tkg
    tkg.set_option(tkg.OPT_CTA_GROUP, 2)
    assert tkg.get_option(tkg.OPT_CTA_GROUP) == 2
    tkg.set_option(tkg.OPT_CTA_GROUP, 0)
    with pytest.raises(tkg.TkgError):
        tkg.set_option(tkg.OPT_CTA_GROUP, 3)
    # every option the header declares is settable; the next number is not
    for o in (tkg.OPT_CTA_GROUP, tkg.OPT_SINGLE_STAGE, tkg.OPT_TIMEOUT_MS, tkg.OPT_INJECT_STALL,
              tkg.OPT_MAX_CLUSTERS, tkg.OPT_ACC_STAGES, tkg.OPT_SCHEDULER, tkg.OPT_SPLIT_K,
              tkg.OPT_RASTER_GROUP, tkg.OPT_BF16_TILE_N, tkg.OPT_TAIL_SPLIT, tkg.OPT_EPILOGUE_STORE):
        tkg.set_option(o, 1)
        assert tkg.get_option(o) == 1
        tkg.set_option(o, 0)
    with pytest.raises(tkg.TkgError):
        tkg.set_option(tkg.OPT_EPILOGUE_STORE + 1, 0)
    assert lib.tkg_status_string(5) == b"device wait timed out"
    assert lib.tkg_status_string(6) == b"internal check failed"


def test_library_is_sm103a_only():
    # the build passes exactly one -gencode, for sm_103a
    from dense_block_scaled_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_grouped_host_checks():
    # argument checks that return before any device work
    import ctypes
    from dense_block_scaled_gb300 import tkg
    sizes = lambda *v: (ctypes.c_int * len(v))(*v)
    assert tkg.gemm_grouped_bf16_raw(0, sizes(1), 8, 8, None, None, None, 1.0, None) == tkg.ERR_INVALID_ARG
    assert tkg.gemm_grouped_bf16_raw(1, None, 8, 8, None, None, None, 1.0, None) == tkg.ERR_INVALID_ARG
    assert tkg.gemm_grouped_bf16_raw(2, sizes(3, -1), 8, 8, None, None, None, 1.0, None) == tkg.ERR_INVALID_ARG
    assert tkg.gemm_grouped_bf16_raw(129, sizes(*([1] * 129)), 8, 8, None, None, None, 1.0, None) == \
        tkg.ERR_UNSUPPORTED
    assert tkg.gemm_grouped_mxfp8_raw(2, sizes(0, 0), 8, 32, None, None, None, None, None, 1.0, None) == tkg.OK
    assert tkg.gemm_grouped_nvfp4_raw(1, sizes(4), 0, 32, None, None, None, None, None, None, None, 1.0,
                                      None) == tkg.OK


def test_grouped_scale_bytes():
    from dense_block_scaled_gb300 import tkg
    sizes = [0, 1, 128, 129]
    assert tkg.grouped_scale_bytes(sizes, 256, 16) == sum(tkg.scale_bytes(m, 256, 16) for m in sizes)
    assert tkg.grouped_scale_bytes([2, -1], 256, 16) == 0


def test_grouped_dev_host_checks():
    import ctypes
    from dense_block_scaled_gb300 import tkg
    lib = tkg.load()
    f = ctypes.c_float(1.0)
    fake = ctypes.c_void_p(4096)   # never dereferenced: these calls return before any device work
    assert lib.tkg_gemm_grouped_dev_bf16(0, fake, 8, 8, 8, None, None, None, f, None) == tkg.ERR_INVALID_ARG
    assert lib.tkg_gemm_grouped_dev_bf16(2, None, 8, 8, 8, None, None, None, f, None) == tkg.ERR_INVALID_ARG
    assert lib.tkg_gemm_grouped_dev_bf16(129, fake, 8, 8, 8, None, None, None, f, None) == tkg.ERR_UNSUPPORTED
    assert lib.tkg_gemm_grouped_dev_bf16(2, ctypes.c_void_p(4098), 8, 8, 8, None, None, None, f, None) == \
        tkg.ERR_ALIGNMENT
    assert lib.tkg_gemm_grouped_dev_bf16(2, fake, 0, 8, 8, None, None, None, f, None) == tkg.OK
    assert lib.tkg_gemm_grouped_dev_bf16(2, fake, 8, 8, 0, None, None, None, f, None) == tkg.ERR_UNSUPPORTED
    assert tkg.grouped_dev_scale_bytes(4, 1000, 256, 16) == \
        tkg.scale_bytes(1000, 256, 16) + 4 * tkg.scale_bytes(128, 256, 16)


def test_gemm_list_host_side_checks(lib):
    # every entry is checked before anything is launched; no CUDA call is made
    from dense_block_scaled_gb300 import tkg
    assert ctypes.sizeof(tkg.GemmDesc) == 80   # the C struct: 3 ints, 7 pointers, a float, padding
    ok = tkg.GemmDesc(64, 64, 64, 16, 16, 16, 16, None, None, 16, 1.0)
    assert tkg.gemm_list_raw("bf16", [], None) == tkg.ERR_INVALID_ARG
    assert tkg.gemm_list_raw("bf16", [ok] * (tkg.MAX_LIST + 1), None) == tkg.ERR_UNSUPPORTED
    bad_m = tkg.GemmDesc(-1, 64, 64, 16, 16, 16, 16, None, None, 16, 1.0)
    assert tkg.gemm_list_raw("bf16", [ok, bad_m], None) == tkg.ERR_INVALID_ARG
    bad_n = tkg.GemmDesc(64, 12, 64, 16, 16, 16, 16, None, None, 16, 1.0)
    assert tkg.gemm_list_raw("mxfp8", [ok, bad_n], None) == tkg.ERR_ALIGNMENT
    bad_k = tkg.GemmDesc(64, 64, 48, 16, 16, 16, 16, None, None, 16, 1.0)
    assert tkg.gemm_list_raw("nvfp4", [bad_k, ok], None) == tkg.ERR_ALIGNMENT
    no_scales = tkg.GemmDesc(64, 64, 64, 16, 16, None, 16, None, None, 16, 1.0)
    assert tkg.gemm_list_raw("mxfp8", [ok, no_scales], None) == tkg.ERR_INVALID_ARG
    bad_ta = tkg.GemmDesc(64, 64, 64, 16, 16, 16, 16, 18, None, 16, 1.0)
    assert tkg.gemm_list_raw("nvfp4", [ok, bad_ta], None) == tkg.ERR_ALIGNMENT
    # empty entries only: nothing to do
    empty = tkg.GemmDesc(0, 64, 64, None, None, None, None, None, None, None, 1.0)
    assert tkg.gemm_list_raw("bf16", [empty, empty], None) == tkg.OK


def test_strided_host_side_checks(lib):
    # pitches shorter than a row, or not a multiple of 16 bytes, are rejected before any CUDA call
    assert lib.tkg_gemm_bf16_strided(64, 64, 64, 16, 56, 16, 64, 16, 64, 1.0, None) == 1      # lda < k
    assert lib.tkg_gemm_bf16_strided(64, 64, 64, 16, 68, 16, 64, 16, 64, 1.0, None) == 2      # 136-byte pitch
    assert lib.tkg_gemm_bf16_strided(64, 64, 64, 16, 64, 16, 64, 16, 60, 1.0, None) == 1      # ldd < n
    assert lib.tkg_gemm_mxfp8_strided(64, 64, 64, 16, 72, 16, 64, 16, 16, 16, 64, 1.0, None) == 2   # 72 bytes
    assert lib.tkg_gemm_nvfp4_strided(64, 64, 64, 16, 16, 16, 32, 16, 16, None, None, 16, 64, 1.0, None) == 1  # < k/2
    assert lib.tkg_gemm_nvfp4_strided(64, 64, 64, 16, 40, 16, 32, 16, 16, None, None, 16, 64, 1.0, None) == 2
    assert lib.tkg_gemm_bf16_strided(0, 64, 64, None, 0, None, 0, None, 0, 1.0, None) == 0     # empty


def test_check_build_compiles_with_the_same_exports():
    # the check build (kernels verifying their invariants) builds and exports every declared symbol
    import ctypes
    from dense_block_scaled_gb300 import build
    path = build.build(check=True)
    assert path.endswith("libtkg_check.so")
    check = ctypes.CDLL(path)
    for name in _declared():
        assert hasattr(check, name), name


def test_no_multicast_tensor_loads_in_the_sources():
    # the kernels run as replicas on several GPUs (bench --gpus N): no TMA load
    # or copy may multicast tensor data across a cluster.  The multicast forms
    # that move no tensor data (the commit's barrier arrive, the cluster launch
    # control answer) are allowed.
    import re
    csrc = os.path.join(ROOT, "dense_block_scaled_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        text = open(os.path.join(csrc, name)).read()
        for line in text.splitlines():
            if "multicast" not in line or line.strip().startswith("//"):
                continue
            assert re.search(r"tcgen05\.commit|clusterlaunchcontrol\.try_cancel", line), (name, line.strip())
            assert "cp.async.bulk" not in line, (name, line.strip())
