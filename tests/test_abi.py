"""The C ABI without a GPU: the library builds and loads, exports every entry
point the header declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import re

import pytest

from block_fp8_expert_gb300 import build as B
from block_fp8_expert_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "moe_fp8.h")


@pytest.fixture(scope="module")
def L():
    B.build()
    return _lib.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert "moe_layer_forward" in names and len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(_lib.EXPORTED)


def test_version_and_status_strings(L):
    assert "sm_103a" in _lib.version()
    assert _lib.status_string(0) == "ok"
    assert _lib.status_string(3) == "workspace too small"
    assert _lib.status_string(99) == "unknown status"


def test_workspace_bytes_grows_with_tokens(L):
    a = _lib.workspace_bytes(_lib.dims(1, 2048, 768, 128, 8))
    b = _lib.workspace_bytes(_lib.dims(64, 2048, 768, 128, 8))
    c = _lib.workspace_bytes(_lib.dims(64, 2048, 512, 512, 10, 512))
    assert 0 < a < b and c > 0
    assert a % 256 == 0 and b % 256 == 0


def test_expert_regime_query(L, monkeypatch):
    """Host-only: the regime rule of moe_layer_forward and its override."""
    monkeypatch.delenv("MOE_FP8_EXPERT_PATH", raising=False)
    q = _lib.expert_uses_gemm
    assert q(_lib.dims(16, 2048, 768, 128, 8))          # 1 row per expert
    assert not q(_lib.dims(8, 2048, 768, 128, 8))       # 1/2 row per expert
    assert q(_lib.dims(4096, 2048, 768, 128, 8))
    assert q(_lib.dims(4096, 256, 128, 16, 2))          # H 256, I 128: smallest GEMM shapes
    assert not q(_lib.dims(4096, 2048 + 64, 768, 128, 8))  # H % 256 != 0
    assert not q(_lib.dims(100, 256, 128, 16, 2))       # small experts: 12.5 rows each
    assert q(_lib.dims(256, 256, 128, 16, 2))           # small experts: 32 rows each
    assert not q(_lib.dims(4096, 2048, 768 + 64, 128, 8))  # I % 128 != 0
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", "gemv")
    assert not q(_lib.dims(4096, 2048, 768, 128, 8))
    monkeypatch.setenv("MOE_FP8_EXPERT_PATH", "gemm")
    assert q(_lib.dims(1, 2048, 768, 128, 8))
    with pytest.raises(ValueError):
        q(_lib.dims(8, 100, 128, 16, 2))


@pytest.mark.parametrize("d,code", [
    ((8, 100, 128, 16, 2, 0), _lib.MOE_ERR_UNSUPPORTED),   # H not a multiple of 64
    ((8, 256, 96, 16, 2, 0), _lib.MOE_ERR_UNSUPPORTED),    # I not a multiple of 64
    ((8, 256, 128, 16, 17, 0), _lib.MOE_ERR_UNSUPPORTED),  # k > E
    ((8, 256, 128, 2000, 2, 0), _lib.MOE_ERR_UNSUPPORTED), # E > 1024
    ((8, 256, 128, 64, 33, 0), _lib.MOE_ERR_UNSUPPORTED),  # k > 32
    ((-1, 256, 128, 16, 2, 0), _lib.MOE_ERR_INVALID_ARG),  # T < 0
    ((8, 256, 128, 16, 2, 100), _lib.MOE_ERR_UNSUPPORTED), # I_shared
])
def test_bad_dims_rejected(L, d, code):
    with pytest.raises(_lib.MoeError) as ei:
        _lib.workspace_bytes(_lib.dims(*d))
    assert ei.value.status == code


def test_null_and_misaligned_pointers_rejected_before_cuda(L):
    d = _lib.dims(8, 256, 128, 16, 2)
    ws_n = _lib.workspace_bytes(d)
    st = L.moe_route(None, 0x1000, None, d, 0x2000, 0x3000, 0x4000, ws_n, None)
    assert st == _lib.MOE_ERR_INVALID_ARG
    assert b"x is NULL" in L.moe_last_error_message()
    st = L.moe_route(0x1008, 0x1000, None, d, 0x2000, 0x3000, 0x4000, ws_n, None)
    assert st == _lib.MOE_ERR_INVALID_ARG
    assert b"aligned" in L.moe_last_error_message()
    # workspace too small
    st = L.moe_permute(0x1000, d, 0x2000, 0x3000, 0x4000, 0x5000, ws_n - 1, None)
    assert st == _lib.MOE_ERR_WORKSPACE
    # shared expert given without I_shared
    f = _lib.ffn(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000)
    st = L.moe_layer_forward(0x1000, 0x1000, None, f, ctypes.byref(f), d, 0x1000, None, None,
                             0x1000, ws_n, None)
    assert st == _lib.MOE_ERR_INVALID_ARG
    # missing weights
    f0 = _lib.ffn(0x1000, None, 0x1000, 0x1000, 0x1000, 0x1000)
    st = L.moe_expert_ffn_fp8(0x1000, 0x1000, 0x1000, f0, d, 0x1000, 0x1000, ws_n, None)
    assert st == _lib.MOE_ERR_INVALID_ARG


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.lib()
