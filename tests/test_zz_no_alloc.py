"""moe_align_noalloc: the grouping step for callers that cannot allocate
device memory (code under CUDA-graph capture, plugin hosts that hand out only
I/O buffers, paths that must not take an allocator's locks).  Its scratch is
the library's static device array; its outputs must equal moe_align's,
which takes a caller-provided workspace.  This file is collected last so that
a run stopping at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from sparse_moe_ffn_gb300 import binding
from sparse_moe_ffn_gb300 import build as lib_build

MOE_OK, MOE_ERR_UNSUPPORTED, MOE_ERR_DEVICE_CHECK = 0, 3, 5


def _lib():
    lib_build.build()
    return binding.lib()


def test_rejects_sizes_beyond_the_static_scratch():
    L = _lib()
    p = ctypes.c_void_p(0x10000)
    # 2^22 tokens x 8 slots x 1024 experts needs far more than 1 MiB of scratch
    rc = L.moe_align_noalloc(p, 1 << 22, 8, 1024, 128, p, p, p, p, p, None, None)
    assert rc == MOE_ERR_UNSUPPORTED
    assert b"MOE_ALIGN_NOALLOC_SCRATCH_BYTES" in L.moe_last_error()


def _call_noalloc(L, ids, E, block_m):
    N, k = ids.shape
    cap = int(L.moe_align_capacity(N, k, E, block_m))
    out = {
        "sorted_pair": torch.full((cap,), -1, dtype=torch.int32, device="cuda"),
        "block_expert": torch.full((cap // block_m,), -1, dtype=torch.int32, device="cuda"),
        "counts": torch.empty(E, dtype=torch.int32, device="cuda"),
        "offsets": torch.empty(E + 1, dtype=torch.int32, device="cuda"),
        "num_padded": torch.empty(1, dtype=torch.int32, device="cuda"),
        "status": torch.full((1,), -7, dtype=torch.int32, device="cuda"),
    }
    ptr = {k_: ctypes.c_void_p(v.data_ptr()) for k_, v in out.items()}
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.moe_align_noalloc(ctypes.c_void_p(ids.data_ptr()), N, k, E, block_m,
                             ptr["sorted_pair"], ptr["block_expert"], ptr["counts"],
                             ptr["offsets"], ptr["num_padded"], ptr["status"], stream)
    assert rc == MOE_OK, L.moe_last_error()
    return out


@pytest.mark.gpu
def test_noalloc_matches_moe_align_on_two_calls_in_a_row():
    """Three-kernel grouping (more than 4096 pairs) and the single-CTA one
    (decode-sized: 64 tokens x 8 slots over 128 experts), each run twice in a
    row through the shared static scratch."""
    L = _lib()
    rng = np.random.default_rng(2024)
    for N, k, E, block_m in [(3000, 8, 128, 128), (700, 6, 64, 16), (3000, 8, 128, 128),
                             (64, 8, 128, 128), (64, 8, 128, 128)]:
        ids_np = rng.integers(0, E, size=(N, k)).astype(np.int32)
        ids_np[ids_np == 5] = 6  # one expert without pairs
        ids = torch.from_numpy(ids_np).cuda()
        got = _call_noalloc(L, ids, E, block_m)
        ref = binding.moe_align(ids, E, block_m)
        torch.cuda.synchronize()
        npad = int(ref["num_padded"].item())
        assert int(got["num_padded"].item()) == npad
        assert int(got["status"].item()) == 0
        for key in ("counts", "offsets"):
            assert torch.equal(got[key], ref[key]), key
        assert torch.equal(got["sorted_pair"][:npad], ref["sorted_pair"][:npad])
        assert torch.equal(got["block_expert"][:npad // block_m],
                           ref["block_expert"][:npad // block_m])


@pytest.mark.gpu
def test_noalloc_reports_bad_ids_and_zero_tokens():
    """An id outside [0, E) is skipped and reported through device_status,
    on both grouping paths; the next call (N = 0 included) reports 0 again."""
    L = _lib()
    for N, k, E in [(64, 8, 128), (1000, 8, 128)]:
        ids = torch.randint(0, E, (N, k), dtype=torch.int32).cuda()
        ids[3, 2] = E + 5
        got = _call_noalloc(L, ids, E, 128)
        torch.cuda.synchronize()
        assert int(got["status"].item()) == MOE_ERR_DEVICE_CHECK
        assert int(got["counts"].sum().item()) == N * k - 1
        ids[3, 2] = 0
        got = _call_noalloc(L, ids, E, 128)
        torch.cuda.synchronize()
        assert int(got["status"].item()) == 0
    empty = torch.empty((0, 8), dtype=torch.int32, device="cuda")
    got = _call_noalloc(L, empty, 128, 128)
    torch.cuda.synchronize()
    assert int(got["status"].item()) == 0  # written, not left at the -7 it held
