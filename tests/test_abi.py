"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before touching a GPU (CPU only)."""
import ctypes
import re

import pytest

import sink_sda_decode_gb300 as sda
from sink_sda_decode_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    from sink_sda_decode_gb300 import build
    build.build()
    return _lib.load()


def declared_functions():
    text = open(_lib.HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sda_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("sda_decode", "sda_decode_workspace_size", "sda_build_indices",
                     "sda_validate_indices", "sda_strerror"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in sda.h but not exported"


def test_binding_covers_every_declared_symbol():
    assert set(declared_functions()) <= set(_lib.SIGNATURES)


def test_strerror_and_version(lib):
    assert lib.sda_abi_version() == 1
    for code in range(5):
        assert lib.sda_strerror(code).decode().startswith("SDA")
    assert lib.sda_strerror(99)


def _decode(lib, N=2, H=16, D=512, total_pages=100, total_indices=10, ptr=1, ws_bytes=1 << 20):
    return lib.sda_decode(ptr, ptr, total_pages, ptr, total_indices, ptr, ptr, 0.1, N, H, D, ptr,
                          ptr, ws_bytes, None)


def test_decode_host_checks(lib):
    # pointers are fake (1): every case below must be rejected before any use
    assert _decode(lib, N=-1) == 1
    assert _decode(lib, total_pages=0) == 1
    assert _decode(lib, total_pages=1 << 31) == 1
    assert _decode(lib, total_indices=-1) == 1
    assert _decode(lib, H=16, D=100) == 2
    assert _decode(lib, H=0, D=512) == 2
    assert _decode(lib, H=300, D=512) == 2
    assert _decode(lib, N=0) == 0                      # empty batch: nothing to do
    assert lib.sda_decode(None, 16, 10, 16, 1, 16, 16, 1.0, 2, 16, 512, 16, 256, 1 << 20, None) == 1
    # misaligned q (not 16-byte aligned)
    assert lib.sda_decode(8, 16, 10, 16, 1, 16, 16, 1.0, 2, 16, 512, 16, 256, 1 << 20, None) == 1
    # misaligned workspace (not 256-byte aligned)
    assert lib.sda_decode(16, 16, 10, 16, 1, 16, 16, 1.0, 2, 16, 512, 16, 16, 1 << 20, None) == 4


def test_build_indices_host_checks(lib):
    args = dict(state_slot=16, swa_len=16, swa_head=16, comp_indptr=16, comp_block=16, comp_slot=16,
                comp_total=4, N=2, win=4, k_per_block=8, swa_pages=8, total_pages=100,
                kv_indices=16, capacity=100, kv_indptr=16, status=16)

    def call(**kw):
        a = dict(args, **kw)
        return lib.sda_build_indices(a["state_slot"], a["swa_len"], a["swa_head"], a["comp_indptr"],
                                     a["comp_block"], a["comp_slot"], a["comp_total"], a["N"],
                                     a["win"], a["k_per_block"], a["swa_pages"], a["total_pages"],
                                     a["kv_indices"], a["capacity"], a["kv_indptr"], a["status"],
                                     None)
    # the divide-by-zero-window failure: rejected on the host, never launched
    assert call(win=0) == 1
    assert call(win=-3) == 1
    assert call(k_per_block=0) == 1
    assert call(N=-1) == 1
    assert call(swa_pages=200) == 1                # swa region larger than the pool
    assert call(total_pages=1 << 31) == 1
    assert call(capacity=-1) == 1
    assert call(kv_indptr=None) == 1
    assert call(status=None) == 1
    assert call(comp_block=None) == 1


def test_validate_host_checks(lib):
    assert lib.sda_validate_indices(16, 4, 16, -1, 10, 16, None) == 1
    assert lib.sda_validate_indices(16, 4, 16, 2, 0, 16, None) == 1
    assert lib.sda_validate_indices(None, 4, 16, 2, 10, 16, None) == 1
    assert lib.sda_validate_indices(16, 4, 16, 2, 10, None, None) == 1


def test_workspace_size_args(lib):
    n = ctypes.c_size_t(0)
    assert lib.sda_decode_workspace_size(-1, 16, 512, 10, ctypes.byref(n)) == 1
    assert lib.sda_decode_workspace_size(2, 16, 512, 10, None) == 1


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        _lib.load()


def test_build_decode_host_extent_checks():
    """build_decode_host checks every host extent the kernels trust before it
    touches CUDA: a descriptor, comp_indptr, comp list or out of the wrong
    length raises ValueError (CPU tensors suffice: these checks come first)."""
    import torch
    N, H, D = 3, 16, 512
    q = torch.zeros(N, H, D, dtype=torch.bfloat16)
    i32 = lambda n: torch.zeros(n, dtype=torch.int32)  # noqa: E731
    good = dict(state_slot=i32(N), swa_len=i32(N), swa_head=i32(N), comp_indptr=i32(N + 1),
                comp_block=i32(5), comp_slot=i32(5))
    kw = dict(win=4, k_per_block=8, swa_pages=64)
    cases = [("state_slot", i32(N - 1)), ("swa_len", i32(N + 1)), ("swa_head", i32(0)),
             ("comp_indptr", i32(N)), ("comp_slot", i32(4))]
    for name, bad in cases:
        args = dict(good, **{name: bad})
        with pytest.raises(ValueError):
            sda.build_decode_host(q, None, None, 1.0, args["state_slot"], args["swa_len"],
                                  args["swa_head"], args["comp_indptr"], args["comp_block"],
                                  args["comp_slot"], **kw)
    with pytest.raises(ValueError):
        sda.build_decode_host(q, None, None, 1.0, *good.values(),
                              out=torch.zeros(N, H, D - 8, dtype=torch.bfloat16), **kw)
