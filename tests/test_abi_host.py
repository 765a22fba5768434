"""The C ABI on the host, without a GPU: the library builds and loads, exports
every entry point include/moe.h declares, sizes workspaces consistently, and
rejects bad arguments before touching the device."""
import ctypes
import functools
import os
import re

import pytest

from sparse_moe_ffn_gb300 import binding
from sparse_moe_ffn_gb300 import build as lib_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "moe.h")
OK, INVALID, SMALL, UNSUPPORTED = 0, 1, 2, 3
FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


@pytest.fixture(scope="module")
def L():
    lib_build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_are_exported(L):
    names = declared_functions()
    assert len(names) >= 12, names
    for name in names:
        assert hasattr(L, name), f"{name} declared in moe.h but not exported"


def test_status_strings(L):
    for code in range(7):
        assert L.moe_status_string(code)
    assert L.moe_status_string(99) == b"unknown status"


def test_layout_is_consistent(L):
    for args in [(64, 2048, 128, 768, 8, 0), (2048, 2048, 64, 768, 6, 2048), (16, 64, 6, 128, 2, 0)]:
        lay = binding.moe_forward_layout(*args)
        assert lay["total"] == binding.moe_forward_workspace_bytes(*args)
        offs = [v for k, v in lay.items() if k not in ("total", "capacity", "slots", "groups")]
        assert all(o % 256 == 0 for o in offs)
        N, H, E, I, k0, I_s = args
        # the shared expert adds ceil(I_s / I) slots per token and as many groups
        C = -(-I_s // I)
        assert lay["slots"] == k0 + C and lay["groups"] == E + C
        k, E = k0 + C, E + C
        cap = lay["capacity"]
        assert cap == L.moe_align_capacity(N, k, E, 128)
        assert lay["ypair"] >= lay["act"] + 4 * cap * I          # bf16 hi/lo or fp16 act
        assert lay["ypair_res"] >= lay["ypair"] + 2 * N * k * H  # pair rows: bf16 plane,
        assert lay["total"] >= lay["ypair_res"] + N * k * H      # then the int8 plane


def _fwd(L, N=64, H=2048, E=128, I=768, I_s=0, k=8, ws_bytes=None, shared=(None,) * 4,
         x=FAKE, ws=FAKE * 16, prepared=False):
    if ws_bytes is None:
        ws_bytes = L.moe_forward_workspace_bytes(N, H, E, I, k, I_s)
    fn = L.moe_forward_prepared if prepared else L.moe_forward
    return fn(x, FAKE, FAKE, FAKE, FAKE, *shared, N, H, E, I, I_s, k, 1, FAKE, ws, ws_bytes,
              None)


@pytest.mark.parametrize("prepared", [False, True])
def test_forward_argument_errors(L, prepared):
    fwd = functools.partial(_fwd, prepared=prepared)  # both entry points share every check
    assert fwd(L, k=0) == INVALID
    assert fwd(L, k=129) == INVALID
    assert fwd(L, H=2044) == INVALID
    assert fwd(L, I=770) == INVALID
    assert fwd(L, N=-1) == INVALID
    assert fwd(L, x=None) == INVALID
    assert fwd(L, x=FAKE + 2) == INVALID          # misaligned bf16 matrix
    assert fwd(L, ws=FAKE + 64) == INVALID        # workspace not 256-byte aligned
    assert fwd(L, E=300, k=8) == UNSUPPORTED
    assert fwd(L, shared=(FAKE, None, None, None), I_s=64) == INVALID
    assert fwd(L, shared=(FAKE,) * 4, I_s=60) == INVALID
    assert fwd(L, E=256, shared=(FAKE,) * 4, I_s=64) == UNSUPPORTED
    # the shared expert's chunks count as experts: 248 + ceil(72 / 8) > 256
    assert fwd(L, E=248, I=8, shared=(FAKE,) * 4, I_s=72) == UNSUPPORTED
    need = L.moe_forward_workspace_bytes(64, 2048, 128, 768, 8, 0)
    assert fwd(L, ws_bytes=need - 1) == SMALL
    assert b"needs" in L.moe_last_error()
    assert fwd(L, N=0) == OK                      # no-op, nothing launched
    assert fwd(L, N=1 << 27, k=8) == UNSUPPORTED  # N*k + E*128 beyond 2^30


def _fwd_host(L, N=64, H=2048, E=128, I=768, k=8, x_host=FAKE, out_host=FAKE, x_dev=FAKE,
              out_dev=FAKE, ws=FAKE * 16):
    ws_bytes = L.moe_forward_workspace_bytes(N, H, E, I, k, 0)
    return L.moe_forward_host(x_host, out_host, x_dev, out_dev, FAKE, FAKE, FAKE, FAKE,
                              None, None, None, None, N, H, E, I, 0, k, 1, ws, ws_bytes, None)


def test_forward_host_argument_errors(L):
    # every check runs before the input copy is enqueued
    assert _fwd_host(L, x_host=None) == INVALID
    assert _fwd_host(L, out_host=None) == INVALID
    assert _fwd_host(L, x_dev=FAKE + 2) == INVALID   # misaligned staging buffer
    assert _fwd_host(L, out_dev=None) == INVALID
    assert _fwd_host(L, k=0) == INVALID
    assert _fwd_host(L, N=0, x_host=None) == OK       # no-op, nothing enqueued


def _experts(L, R=64, H=2048, E=16, I=768, x=FAKE, ids=FAKE, y=FAKE, ws=FAKE * 16,
             ws_bytes=None, prepared=False):
    if ws_bytes is None:
        ws_bytes = L.moe_experts_workspace_bytes(R, H, E, I)
    fn = L.moe_experts_prepared if prepared else L.moe_experts
    return fn(x, ids, FAKE, R, H, E, I, FAKE, FAKE, FAKE, y, FAKE, ws, ws_bytes, None)


@pytest.mark.parametrize("prepared", [False, True])
def test_experts_and_combine_argument_errors(L, prepared):
    experts = functools.partial(_experts, prepared=prepared)

    # the expert-parallel receiving side: one routed row per (row, expert)
    # moe_forward's layout with one slot per row, without the pair-row planes
    # (the outputs go to the caller's y)
    assert L.moe_experts_workspace_bytes(64, 2048, 16, 768) == \
        binding.moe_forward_layout(64, 2048, 16, 768, 1, 0)["ypair"]
    assert experts(L, R=-1) == INVALID
    assert experts(L, H=2044) == INVALID
    assert experts(L, I=0) == INVALID
    assert experts(L, E=0) == UNSUPPORTED
    assert experts(L, ids=None) == INVALID
    assert experts(L, y=FAKE + 2) == INVALID
    assert experts(L, ws=FAKE + 64) == INVALID
    need = L.moe_experts_workspace_bytes(64, 2048, 16, 768)
    assert experts(L, ws_bytes=need - 1) == SMALL
    assert experts(L, R=0, x=None) == OK          # no-op, nothing launched
    P = FAKE
    assert L.moe_combine(P, P, None, None, 0, 16, 2048, 0, P, None) == INVALID
    assert L.moe_combine(P, P, None, None, 0, 16, 2044, 2, P, None) == INVALID
    assert L.moe_combine(None, P, None, None, 0, 16, 2048, 2, P, None) == INVALID
    assert L.moe_combine(P, None, None, None, 0, 16, 2048, 2, P, None) == INVALID
    assert L.moe_combine(P, P, P, None, 1, 16, 2048, 2, P, None) == INVALID   # one shared plane
    assert L.moe_combine(P, P, P + 2, P, 1, 16, 2048, 2, P, None) == INVALID  # misaligned
    assert L.moe_combine(P, P, P, P, 0, 16, 2048, 2, P, None) == INVALID      # no shared slots
    assert L.moe_combine(P, P, P, P, 257, 16, 2048, 2, P, None) == INVALID
    assert L.moe_combine(P, P, None, None, 0, 0, 2048, 2, None, None) == OK


def test_dense_mlp_argument_errors(L):
    P = FAKE
    need = L.moe_dense_mlp_workspace_bytes(300, 256, 192)
    for fn in (L.moe_dense_mlp, L.moe_dense_mlp_prepared):
        assert fn(P, P, P, P, 300, 250, 192, P, P * 16, need, None) == INVALID   # H % 8
        assert fn(P, P, P, None, 300, 256, 192, P, P * 16, need, None) == INVALID
        assert fn(P, P, P, P, 300, 256, 192, P, P * 16 + 64, need, None) == INVALID
        assert fn(P, P, P, P, 300, 256, 192, P, P * 16, need - 1, None) == SMALL
        assert fn(None, None, None, None, 0, 256, 192, None, None, 0, None) == OK


def test_convert_argument_errors(L):
    P = FAKE
    assert L.moe_convert_bf16_to_f16(P, P + 4096, -1, None, None) == INVALID
    assert L.moe_convert_bf16_to_f16(None, P, 8, None, None) == INVALID
    assert L.moe_convert_bf16_to_f16(P + 2, P + 4096, 8, None, None) == INVALID  # misaligned
    assert L.moe_convert_bf16_to_f16(P, P + 16, 64, None, None) == INVALID       # overlap
    assert L.moe_convert_bf16_to_f16(None, None, 0, None, None) == OK            # no-op


def test_route_and_align_argument_errors(L):
    P = FAKE
    assert L.moe_route(P, P, None, 16, 64, 6, 7, 1, P, P, None, None, None, 0, None) == INVALID
    assert L.moe_route(P, P, P, 16, 64, 6, 2, 1, P, P, None, None, None, 0, None) == INVALID
    assert L.moe_route(P, P, None, 16, 60, 6, 2, 1, P, P, None, None, None, 0, None) == INVALID
    assert L.moe_route(P, P, None, 16, 64, 6, 2, 1, P, P, None, None, P, 1, None) == SMALL
    assert L.moe_route(P, P, None, 0, 64, 6, 2, 1, P, P, None, None, None, 0, None) == OK
    need = L.moe_align_workspace_bytes(100, 2, 8, 16)
    assert L.moe_align(P, 100, 2, 8, 16, P, P, P, P, P, P, need - 1, None) == SMALL
    assert L.moe_align(P, 100, 2, 8, 0, P, P, P, P, P, P, need, None) == INVALID
    assert L.moe_align(P, 100, 2, 2000, 16, P, P, P, P, P, P, need, None) == UNSUPPORTED
    assert L.moe_align(None, 100, 2, 8, 16, P, P, P, P, P, P, need, None) == INVALID
    assert L.moe_align_capacity(3, 2, 5, 4) == 24  # round_up(6 + 5*3, 4)


def test_stage_events_argument_check(L):
    assert L.moe_set_stage_events(None, 0) == OK
    arr = (ctypes.c_void_p * 3)()
    assert L.moe_set_stage_events(arr, 3) == INVALID


def test_dispatch_and_indexed_combine_argument_errors(L):
    P = FAKE
    need = L.moe_ep_dispatch_workspace_bytes(64, 8, 2)
    assert need > 0 and L.moe_ep_dispatch_workspace_bytes(-1, 8, 2) == 0

    def disp(N=64, H=2048, k=8, E=128, world=2, x=P, ws=P * 16, ws_bytes=need):
        return L.moe_ep_dispatch(x, P, P, N, H, k, E, world, P, P, P, P, P, ws, ws_bytes, None)

    assert disp(world=0) == INVALID
    assert disp(H=2044) == INVALID
    assert disp(world=2000) == UNSUPPORTED
    assert disp(x=None) == INVALID
    assert disp(x=P + 2) == INVALID
    assert disp(ws=P * 16 + 64) == INVALID
    assert disp(ws_bytes=need - 1) == SMALL
    assert disp(N=0, x=None) == OK
    # indexed combine: row_index required, both shared planes or neither
    assert L.moe_combine_indexed(P, P, 10, None, None, None, 0, 4, 2048, 2, P, None) == INVALID
    assert L.moe_combine_indexed(P, P, 10, P, P, None, 1, 4, 2048, 2, P, None) == INVALID
    assert L.moe_combine_indexed(P, P, -1, P, None, None, 0, 4, 2048, 2, P, None) == INVALID
    assert L.moe_combine_indexed(P, P, 10, P, P, P, 0, 4, 2048, 2, P, None) == INVALID
    assert L.moe_combine_indexed(None, None, 0, None, None, None, 0, 0, 2048, 2, None,
                                 None) == OK


def _shared(L, N=64, H=2048, I=768, I_s=2048, x=FAKE, gamma=FAKE, y=FAKE, ws=FAKE * 16,
            ws_bytes=None, prepared=False):
    if ws_bytes is None:
        ws_bytes = L.moe_shared_expert_workspace_bytes(N, H, I, I_s)
    fn = L.moe_shared_expert_prepared if prepared else L.moe_shared_expert
    return fn(x, gamma, N, H, I, I_s, FAKE, FAKE, FAKE, y, FAKE, ws, ws_bytes, None)


@pytest.mark.parametrize("prepared", [False, True])
def test_shared_expert_argument_errors(L, prepared):
    shared = functools.partial(_shared, L, prepared=prepared)
    assert L.moe_shared_chunks(768, 2048) == 3
    assert L.moe_shared_chunks(768, 768) == 1
    assert L.moe_shared_chunks(64, 8) == 1
    # the layout of moe_forward with no routed experts and C chunk slots
    lay = binding.moe_forward_layout(64, 2048, 1, 768, 1, 2048)
    assert L.moe_shared_expert_workspace_bytes(64, 2048, 768, 2048) <= lay["total"]
    assert shared(N=-1) == INVALID
    assert shared(H=2044) == INVALID
    assert shared(I=0) == INVALID
    assert shared(I_s=60) == INVALID
    assert shared(I=8, I_s=8 * 257) == UNSUPPORTED   # 257 chunks
    assert shared(gamma=None) == INVALID
    assert shared(y=FAKE + 2) == INVALID
    assert shared(ws=FAKE + 64) == INVALID
    need = L.moe_shared_expert_workspace_bytes(64, 2048, 768, 2048)
    assert shared(ws_bytes=need - 1) == SMALL
    assert shared(N=0, x=None) == OK


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No CPU fallback: with the library absent, the binding raises instead
    of computing anything."""
    from sparse_moe_ffn_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB", str(tmp_path / "libsparse_moe_ffn.so"))
    with pytest.raises(RuntimeError, match="missing"):
        binding.lib()
    with pytest.raises(RuntimeError, match="missing"):
        binding.moe_shared_chunks(768, 2048)
