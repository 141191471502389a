"""The C-ABI library builds for sm_103a, loads, exports every entry point the
header declares, and rejects invalid arguments on the host before touching
the GPU (no compute call runs here)."""
import ctypes
import os
import re

import pytest

from exact_io_aware_40_gb300 import build as fab

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    path = fab.build()
    from exact_io_aware_40_gb300 import fa
    return fa.load_library()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(fa_[a-z0-9_]+)\s*\(",
                                text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("fa_fwd", "fa_fwd_kvlen", "fa_bwd", "fa_bwd_prepare", "fa_bwd_dkdv",
              "fa_bwd_dq", "fa_bwd_workspace_bytes", "fa_check_error", "fa_status_string",
              "fa_selftest_stalled_wait", "fa_bwd_noalloc", "fa_fwd_masked", "fa_bwd_masked",
              "fa_fwd_dropout", "fa_bwd_dropout", "fa_fwd_fp8", "fa_fwd_fp8_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    from exact_io_aware_40_gb300 import fa
    assert fa.status_string(0) == "FA_OK"
    assert fa.status_string(4) == "FA_ERR_TIMEOUT"
    assert fa.status_string(99) == "FA_ERR_UNKNOWN"


def test_workspace_size(lib):
    from exact_io_aware_40_gb300 import fa
    B, H, N, d = 2, 3, 100, 64
    rows = B * H * N
    r256 = lambda x: (x + 255) // 256 * 256
    assert fa.fa_bwd_workspace_bytes(B, H, N, d) == r256(rows * 4)
    assert fa.fa_bwd_workspace_bytes(B, H, N, 96) == 0
    assert fa.fa_bwd_workspace_bytes(0, H, N, d) == 0


def test_invalid_arguments_are_rejected_on_the_host(lib):
    fake = ctypes.c_void_p(0x10000)        # 16-byte aligned, never dereferenced
    odd = ctypes.c_void_p(0x10008)         # 8-byte aligned only
    null = ctypes.c_void_p(0)
    f = ctypes.c_float
    # null pointer
    assert lib.fa_fwd(null, fake, fake, fake, fake, 1, 1, 128, 64, f(0.125), 0, null) == 1
    # unsupported head dim
    assert lib.fa_fwd(fake, fake, fake, fake, fake, 1, 1, 128, 96, f(0.125), 0, null) == 2
    # bad sizes and scale
    assert lib.fa_fwd(fake, fake, fake, fake, fake, 0, 1, 128, 64, f(0.125), 0, null) == 1
    assert lib.fa_fwd(fake, fake, fake, fake, fake, 1, 1, 0, 64, f(0.125), 0, null) == 1
    assert lib.fa_fwd(fake, fake, fake, fake, fake, 1, 1, 128, 64, f(float("nan")), 0, null) == 1
    assert lib.fa_fwd(fake, fake, fake, fake, fake, 1, 1, 128, 64, f(-1.0), 0, null) == 1
    # misaligned tensor
    assert lib.fa_fwd(odd, fake, fake, fake, fake, 1, 1, 128, 64, f(0.125), 0, null) == 1
    # backward: short workspace, null gradient
    args = [fake] * 9
    assert lib.fa_bwd(*args, 1, 1, 128, 64, f(0.125), 0, null, fake, 16, null) == 1
    args[6] = null
    assert lib.fa_bwd(*args, 1, 1, 128, 64, f(0.125), 0, null, fake, 1 << 20, null) == 1


def test_selftest_limit_is_validated_on_the_host(lib):
    null = ctypes.c_void_p(0)
    assert lib.fa_selftest_stalled_wait(0, null) == 1
    assert lib.fa_selftest_stalled_wait(20_000_000_000, null) == 1


def test_backward_stages_reject_invalid_arguments(lib):
    fake, null, f = ctypes.c_void_p(0x10000), ctypes.c_void_p(0), ctypes.c_float
    assert lib.fa_bwd_prepare(null, fake, 1, 1, 128, 64, fake, 1 << 20, null) == 1
    assert lib.fa_bwd_prepare(fake, fake, 1, 1, 128, 64, fake, 16, null) == 1
    assert lib.fa_bwd_prepare(fake, fake, 1, 1, 128, 96, fake, 1 << 20, null) == 2
    # workspace not 256-byte aligned
    assert lib.fa_bwd_dkdv(*([fake] * 7), 1, 1, 128, 64, f(0.1), 0, null, ctypes.c_void_p(0x10010),
                           1 << 20, null) == 1
    assert lib.fa_bwd_dq(*([fake] * 5), null, 1, 1, 128, 64, f(0.1), 0, null, fake, 1 << 20,
                         null) == 1
    # the no-allocation variant validates sizes before touching its scratch
    assert lib.fa_bwd_noalloc(*([fake] * 9), 1, 1, 128, 96, f(0.1), 0, null, null) == 2
    assert lib.fa_bwd_noalloc(*([fake] * 9), 0, 1, 128, 64, f(0.1), 0, null, null) == 1


def test_masked_entry_points_validate_the_mask_terms(lib):
    fake, null, f = ctypes.c_void_p(0x10000), ctypes.c_void_p(0), ctypes.c_float
    fwd = lambda d, window, bm: lib.fa_fwd_masked(*([fake] * 5), 1, 1, 256, d, f(0.1), 1, null,
                                                   window, bm, null)
    bwd = lambda d, window, bm: lib.fa_bwd_masked(*([fake] * 9), 1, 1, 256, d, f(0.1), 1, null,
                                                   window, bm, fake, 1 << 20, null)
    for call in (fwd, bwd):
        assert call(64, -2, null) == 1          # window below -1
        assert call(96, 8, null) == 2           # head dim
    # d = 256 takes the window and block-mask terms: these calls get past the
    # mask checks and stop at the short workspace
    for window, bm in ((8, null), (-1, fake)):
        assert lib.fa_bwd_masked(*([fake] * 9), 1, 1, 256, 256, f(0.1), 1, null, window, bm,
                                 fake, 16, null) == 1
    assert lib.fa_fwd_masked(null, *([fake] * 4), 1, 1, 256, 64, f(0.1), 1, null, 4, null,
                             null) == 1
    assert lib.fa_bwd_masked(*([fake] * 9), 1, 1, 256, 64, f(0.1), 1, null, 4, null, fake, 16,
                             null) == 1          # short workspace


def test_dropout_entry_points_validate_the_probability(lib):
    fake, null, f = ctypes.c_void_p(0x10000), ctypes.c_void_p(0), ctypes.c_float
    u64 = ctypes.c_uint64
    fwd = lambda d, p: lib.fa_fwd_dropout(*([fake] * 5), 1, 1, 256, d, f(0.1), 1, null, -1, null,
                                           f(p), u64(7), null)
    bwd = lambda d, p: lib.fa_bwd_dropout(*([fake] * 9), 1, 1, 256, d, f(0.1), 1, null, -1, null,
                                           f(p), u64(7), fake, 1 << 20, null)
    for call in (fwd, bwd):
        assert call(64, -0.1) == 1
        assert call(64, 1.0) == 1
        assert call(64, float("nan")) == 1
    # d = 256 takes dropout: the call gets past the probability check and stops
    # at the short workspace
    assert lib.fa_bwd_dropout(*([fake] * 9), 1, 1, 256, 256, f(0.1), 1, null, -1, null, f(0.1),
                              u64(7), fake, 16, null) == 1


def test_fp8_entry_point_validates_on_the_host(lib):
    from exact_io_aware_40_gb300 import fa
    fake, null, f = ctypes.c_void_p(0x10000), ctypes.c_void_p(0), ctypes.c_float
    assert fa.fa_fwd_fp8_workspace_bytes(1, 2, 100, 128) == (2 * 128 * 112 + 255) // 256 * 256
    assert fa.fa_fwd_fp8_workspace_bytes(1, 2, 100, 64) == 0
    call = lambda d, dq, ws_bytes: lib.fa_fwd_fp8(*([fake] * 5), 1, 2, 100, d, f(0.1), f(dq), f(1.0),
                                                  f(1.0), 1, null, fake, ws_bytes, null)
    assert call(64, 1.0, 1 << 20) == 2          # d must be 128
    assert call(128, 0.0, 1 << 20) == 1         # descale factor must be > 0
    assert call(128, float("inf"), 1 << 20) == 1
    assert call(128, 1.0, 64) == 1              # short workspace


def test_convenience_api_has_no_cpu_path():
    # CPU tensors are refused before any call: there is no host fallback.
    import torch
    from exact_io_aware_40_gb300 import fa
    q = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16)
    L = torch.zeros(1, 2, 128, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA"):
        fa.attention_fwd(q, q, q)
    with pytest.raises(ValueError, match="CUDA"):
        fa.attention_bwd(q, q, q, q, q, L)
    with pytest.raises(ValueError, match="one CUDA device"):
        fa._same_device(q, torch.zeros(1, device="meta"))


def _header_prototypes():
    """name -> (return type, [parameter types]) for every function in include/*.h."""
    protos = {}
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*((?:const\s+)?[A-Za-z_]\w*\s*\**)\s*(fa_\w+)\s*\(([^)]*)\)\s*;",
                             text, flags=re.M):
            params = [re.sub(r"\s*\b\w+$", "", p.strip()) for p in m.group(3).split(",")]
            protos[m.group(2)] = (m.group(1).strip(), [p for p in params if p])
    return protos


def _ctype(c):
    if "*" in c or c in ("fa_stream_t",):
        return ctypes.c_void_p
    return {"int": ctypes.c_int, "float": ctypes.c_float, "size_t": ctypes.c_size_t,
            "uint64_t": ctypes.c_uint64, "fa_status": ctypes.c_int}[c]


def test_binding_signatures_match_the_header(lib):
    # A parameter the binding declares with the wrong type or position would
    # hand the kernels a wrong pointer or size: every prototype is compared.
    protos = _header_prototypes()
    assert set(protos) == set(declared_functions())
    for name, (ret, params) in protos.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, name
        assert list(fn.argtypes) == [_ctype(p) for p in params], name
        want_ret = {"fa_status": ctypes.c_int, "size_t": ctypes.c_size_t,
                    "const char*": ctypes.c_char_p}[re.sub(r"\s+\*", "*", ret)]
        assert fn.restype == want_ret, name
