"""The C-ABI library builds, loads and exports every symbol include/moe.h
declares; host-side validation fails closed before any CUDA call (no GPU
needed: every case below returns before the library touches the device)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from moe_routed_expert_routing_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    from moe_routed_expert_routing_gb300 import binding
    return binding


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    syms = declared_symbols()
    for s in ("moe_dispatch", "moe_expert_compute", "moe_combine", "moe_forward", "moe_workspace_size"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(build_mod.lib_path())
    missing = [s for s in declared_symbols() if not hasattr(so, s)]
    assert not missing, missing
    assert set(declared_symbols()) == set(lib.EXPORTED_SYMBOLS)


def test_status_strings(lib):
    for s in range(7):
        assert lib.status_string(s).startswith("MOE_")
    # the code also covers a layout or form the shape cannot take, not only the device
    text = lib.status_string(5)
    assert "sm_103" in text and "layout" in text and "form" in text


def test_workspace_size_and_path(lib):
    P = lib.Problem.make
    for (T, E, k, H, I) in [(64, 8, 2, 256, 512), (1, 384, 6, 7168, 3072), (8192, 128, 8, 4096, 1536)]:
        p = P(T, E, k, H, I)
        n = lib.moe_workspace_size(p)
        cap = T * k
        assert n >= 2 * cap * (I + 2 * H) + 4 * cap
        assert n % 256 == 0
    assert lib.moe_resolve_path(P(1, 384, 6, 7168, 3072)) == (lib.MOE_PATH_SMALL_M, 16)
    assert lib.moe_resolve_path(P(8, 384, 6, 7168, 3072)) == (lib.MOE_PATH_SMALL_M, 16)
    assert lib.moe_resolve_path(P(128, 256, 8, 7168, 2048)) == (lib.MOE_PATH_SMALL_M, 32)
    assert lib.moe_resolve_path(P(2048, 384, 6, 7168, 3072)) == (lib.MOE_PATH_TILED_1CTA, 128)
    assert lib.moe_resolve_path(P(8192, 128, 8, 4096, 1536)) == (lib.MOE_PATH_TILED, 128)
    assert lib.moe_resolve_path(P(8192, 128, 8, 4096, 1536, path=lib.MOE_PATH_SMALL_M)) == (lib.MOE_PATH_SMALL_M, 64)
    assert lib.moe_resolve_path(P(1, 384, 6, 7168, 3072, path=lib.MOE_PATH_TILED)) == (lib.MOE_PATH_TILED, 128)
    assert lib.moe_resolve_path(P(64, 8, 2, 256, 512, path=lib.MOE_PATH_TILED_1CTA)) == (lib.MOE_PATH_TILED_1CTA, 128)


@pytest.mark.parametrize("bad,status", [
    (dict(T_max=0), 2), (dict(E=0), 2), (dict(E=1025), 2), (dict(k=0), 2), (dict(k=9, E=8), 2),
    (dict(H=300), 3), (dict(I=100), 3), (dict(capacity=5), 2), (dict(path=7), 2), (dict(path=-1), 2),
    (dict(weight_layout=3), 2), (dict(forward_form=3), 2), (dict(forward_form=-1), 2),
])
def test_problem_validation(lib, bad, status):
    args = dict(T_max=64, E=8, k=2, H=256, I=512, capacity=0, path=0, weight_layout=0)
    args.update(bad)
    p = lib.Problem.make(**args)
    with pytest.raises(lib.MoeError) as ei:
        lib.moe_workspace_size(p)
    assert ei.value.status == status


def test_entry_points_fail_closed_without_touching_the_device(lib):
    so = lib.load_library()
    p = lib.Problem.make(64, 8, 2, 256, 512)
    need = lib.moe_workspace_size(p)
    fake = 1 << 40  # never dereferenced: every call below fails validation first
    P = ctypes.byref(p)
    # NULL routing
    assert so.moe_dispatch(P, None, None, fake, fake, fake, None, None, fake, need, None) == 1
    # x without x_sorted
    assert so.moe_dispatch(P, fake, None, fake, fake, fake, fake, None, fake, need, None) == 1
    # misaligned workspace
    assert so.moe_dispatch(P, fake, None, fake, fake, fake, None, None, fake + 8, need, None) == 3
    # undersized workspace
    assert so.moe_dispatch(P, fake, None, fake, fake, fake, None, None, fake, need - 256, None) == 4
    assert so.moe_expert_compute(P, fake, fake, fake, fake, fake, fake, need - 1, None) == 4
    assert so.moe_expert_compute(P, fake + 2, fake, fake, fake, fake, fake, need, None) == 3
    assert so.moe_expert_compute(P, None, fake, fake, fake, fake, fake, need, None) == 1
    assert so.moe_combine(P, fake, None, fake, None, fake, None) == 1
    assert so.moe_combine(P, fake + 4, fake, fake, None, fake, None) == 3
    assert so.moe_forward(P, fake, fake, fake, None, fake, fake, fake, fake, fake, fake, need - 256, None) == 4
    assert so.moe_forward(P, fake, fake, None, None, fake, fake, fake, fake, fake, fake, need, None) == 1
    assert so.moe_forward(None, fake, fake, fake, None, fake, fake, fake, fake, fake, fake, need, None) == 1
    code = ctypes.c_int32(0)
    assert so.moe_last_device_error(None, None, ctypes.byref(code)) == 1
    assert so.moe_pack_weights(P, fake, fake, None, fake, None) == 1
    assert so.moe_pack_weights(P, fake, fake, fake + 8, fake, None) == 3


def test_weight_bytes_pure_host(lib):
    """Weight buffer sizes per layout, without a device: bf16 (row-major or
    packed) 2 bytes per element; MXFP8 1 byte per code plus 1 scale byte per 32."""
    p = lib.Problem.make(8, 384, 6, 7168, 3072)
    n13, n2 = 384 * 6144 * 7168, 384 * 7168 * 3072
    assert lib.moe_weight_bytes(p, lib.MOE_WEIGHTS_ROW_MAJOR) == (2 * n13, 2 * n2)
    assert lib.moe_weight_bytes(p, lib.MOE_WEIGHTS_PACKED) == (2 * n13, 2 * n2)
    assert lib.moe_weight_bytes(p, lib.MOE_WEIGHTS_MXFP8) == (n13 + n13 // 32, n2 + n2 // 32)
    with pytest.raises(lib.MoeError) as ei:
        lib.moe_weight_bytes(p, 7)
    assert ei.value.status == 2


class _DeviceStandIn:
    """Stands in for a CUDA tensor (device, dtype, element count) so that the
    binding's extent and dtype checks can be exercised without a GPU."""
    is_cuda = True

    def __init__(self, dtype, n):
        self.dtype, self._n = dtype, n

    def numel(self):
        return self._n


def test_binding_checks_fail_closed_before_the_library(lib, monkeypatch):
    import torch
    P = lib.Problem.make(16, 8, 2, 256, 128)
    # dtype and extent, per argument
    lib._need(_DeviceStandIn(torch.int32, 32), "topk_ids", torch.int32, 32)
    with pytest.raises(ValueError, match="int32"):
        lib._need(_DeviceStandIn(torch.int64, 32), "topk_ids", torch.int32, 32)
    with pytest.raises(ValueError, match="at least 32"):
        lib._need(_DeviceStandIn(torch.int32, 31), "topk_ids", torch.int32, 32)
    lib._need(1 << 40, "raw pointer", torch.int32, 32)          # a raw address is the caller's to vouch for
    with pytest.raises(ValueError, match="W13"):
        lib._need_weights(P, _DeviceStandIn(torch.bfloat16, 8 * 2 * 128 * 256 - 1),
                          _DeviceStandIn(torch.bfloat16, 8 * 256 * 128))
    Q = lib.Problem.make(16, 8, 2, 256, 128, weight_layout=lib.MOE_WEIGHTS_MXFP8)
    b13, b2 = lib.moe_weight_bytes(Q, lib.MOE_WEIGHTS_MXFP8)
    lib._need_weights(Q, _DeviceStandIn(torch.uint8, b13), _DeviceStandIn(torch.uint8, b2))
    with pytest.raises(ValueError, match="W2"):
        lib._need_weights(Q, _DeviceStandIn(torch.uint8, b13), _DeviceStandIn(torch.uint8, b2 - 1))

    # host tensors never reach the C entry points
    def no_library(*a, **k):
        raise AssertionError("the library was called")
    monkeypatch.setattr(lib, "load_library", no_library)
    x = torch.zeros((16, 256), dtype=torch.bfloat16)
    ids = torch.zeros((16, 2), dtype=torch.int32)
    w = torch.ones((16, 2), dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        lib.moe_forward(P, x, ids, w, 1 << 40, 1 << 40, 1 << 40, 1 << 40, 1 << 40, 1 << 40)
    with pytest.raises(ValueError, match="CUDA tensor"):
        lib.moe_combine(P, 1 << 40, 1 << 40, w, 1 << 40)


def test_missing_library_fails_loudly(lib, tmp_path, monkeypatch):
    """Without libmoe.so the binding raises; nothing falls back to a CPU path."""
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        lib.load_library(str(tmp_path / "libmoe.so"))
    monkeypatch.setattr(lib, "_lib", None)
    monkeypatch.setattr(lib, "lib_path", lambda: str(tmp_path / "absent" / "libmoe.so"))
    with pytest.raises(RuntimeError, match="not found"):
        lib.moe_workspace_size(lib.Problem.make(16, 8, 2, 256, 128))


def test_hidden_and_intermediate_multiples_of_64(lib):
    """H and I need only be multiples of 64 (FlashInfer moe_ep page, Shape
    Coverage & Guardrails: hidden and intermediate sizes that are multiples
    of 64, e.g. 2880); the PACKED and MXFP8 layouts, built of 128-row weight
    tiles, keep multiples of 128 and are refused otherwise, before any CUDA call."""
    P = lib.Problem.make
    for H, I in [(448, 192), (2880, 2880), (64, 64), (7168, 3072)]:
        assert lib.moe_workspace_size(P(64, 8, 2, H, I)) > 0
    for H, I in [(480, 192), (448, 160), (32, 64)]:
        with pytest.raises(lib.MoeError) as ei:
            lib.moe_workspace_size(P(64, 8, 2, H, I))
        assert ei.value.status == 3
    for layout in (lib.MOE_WEIGHTS_PACKED, lib.MOE_WEIGHTS_MXFP8):
        for H, I in [(448, 256), (512, 192)]:
            with pytest.raises(lib.MoeError) as ei:
                lib.moe_workspace_size(P(64, 8, 2, H, I, weight_layout=layout))
            assert ei.value.status == 3
        assert lib.moe_workspace_size(P(64, 8, 2, 512, 256, weight_layout=layout)) > 0
    so = lib.load_library()
    q = P(64, 8, 2, 448, 192)
    fake = 1 << 40   # never dereferenced: refused before the device is touched
    assert so.moe_pack_weights(ctypes.byref(q), fake, fake, fake, fake, None) == 3
    assert so.moe_quantize_weights(ctypes.byref(q), fake, fake, fake, fake, None) == 3
