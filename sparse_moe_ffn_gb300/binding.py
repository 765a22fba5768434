"""ctypes binding of libsparse_moe_ffn.so, with the same entry-point names as
include/moe.h.  Argument marshalling only: torch tensors supply device
pointers and the current stream; every step of the layer runs in the
library's CUDA kernels.  There is no fallback: a missing library raises.

Down-projection weights may be the model's bf16 tensors or the fp16 copies
``prepare_weights`` makes once at load; the wrappers pick the library entry
point that takes that form (``moe_forward`` or ``moe_forward_prepared``, and
likewise for the host, experts and dense-MLP calls).
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB

MOE_OK = 0
MOE_BLOCK_M = 128
MOE_NUM_STAGES = 7
STAGE_NAMES = ("route", "align", "gather", "gate_up", "down", "shared", "combine")
SHARED_KEYS = ("shared_gate_proj", "shared_up_proj", "shared_down_proj", "shared_gate")


class MoEError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


class _Layout(ctypes.Structure):
    _fields_ = [(name, ctypes.c_size_t) for name in (
        "status", "topk_w", "topk_ids", "gamma", "counts", "offsets", "pad_offsets",
        "num_padded", "align_scratch", "sorted_pair", "block_expert", "ready", "x_sorted", "act",
        "ypair", "ypair_res", "total")] + [
        ("capacity", ctypes.c_int64), ("slots", ctypes.c_int), ("groups", ctypes.c_int)]


_lib = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB):
        raise RuntimeError(f"{LIB} is missing: build it first (python -m sparse_moe_ffn_gb300.build)")
    L = ctypes.CDLL(LIB)
    P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    sig = {
        "moe_status_string": ([i32], ctypes.c_char_p),
        "moe_last_error": ([], ctypes.c_char_p),
        "moe_route_workspace_bytes": ([], sz),
        "moe_route": ([P, P, P, i64, i32, i32, i32, i32, P, P, P, P, P, sz, P], i32),
        "moe_align_capacity": ([i64, i32, i32, i32], i64),
        "moe_align_workspace_bytes": ([i64, i32, i32, i32], sz),
        "moe_align": ([P, i64, i32, i32, i32, P, P, P, P, P, P, sz, P], i32),
        "moe_forward_workspace_bytes": ([i64, i32, i32, i32, i32, i32], sz),
        "moe_forward": ([P] * 9 + [i64, i32, i32, i32, i32, i32, i32, P, P, sz, P], i32),
        "moe_forward_prepared": ([P] * 9 + [i64, i32, i32, i32, i32, i32, i32, P, P, sz, P], i32),
        "moe_forward_host": ([P] * 12 + [i64, i32, i32, i32, i32, i32, i32, P, sz, P], i32),
        "moe_forward_host_prepared": ([P] * 12 + [i64, i32, i32, i32, i32, i32, i32, P, sz, P],
                                      i32),
        "moe_experts_workspace_bytes": ([i64, i32, i32, i32], sz),
        "moe_experts": ([P, P, P, i64, i32, i32, i32, P, P, P, P, P, P, sz, P], i32),
        "moe_experts_prepared": ([P, P, P, i64, i32, i32, i32, P, P, P, P, P, P, sz, P], i32),
        "moe_combine": ([P, P, P, P, i32, i64, i32, i32, P, P], i32),
        "moe_combine_indexed": ([P, P, i64, P, P, P, i32, i64, i32, i32, P, P], i32),
        "moe_shared_chunks": ([i32, i32], i32),
        "moe_shared_expert_workspace_bytes": ([i64, i32, i32, i32], sz),
        "moe_shared_expert": ([P, P, i64, i32, i32, i32, P, P, P, P, P, P, sz, P], i32),
        "moe_shared_expert_prepared": ([P, P, i64, i32, i32, i32, P, P, P, P, P, P, sz, P],
                                       i32),
        "moe_ep_dispatch_workspace_bytes": ([i64, i32, i32], sz),
        "moe_ep_dispatch": ([P, P, P, i64, i32, i32, i32, i32, P, P, P, P, P, P, sz, P], i32),
        "moe_convert_bf16_to_f16": ([P, P, i64, P, P], i32),
        "moe_forward_layout": ([i64, i32, i32, i32, i32, i32, ctypes.POINTER(_Layout)], i32),
        "moe_read_device_status": ([P, P], i32),
        "moe_kernel_launch_count": ([], ctypes.c_uint64),
        "moe_set_stage_events": ([P, i32], i32),
        "moe_selftest_wait_timeout": ([P, sz, ctypes.c_uint64, P], i32),
        "moe_align_noalloc": ([P, i64, i32, i32, i32, P, P, P, P, P, P, P], i32),
        "moe_dense_mlp_workspace_bytes": ([i64, i32, i32], sz),
        "moe_add_rmsnorm": ([P, P, P, i64, i32, ctypes.c_float, i32, P, P], i32),
        "moe_dense_mlp": ([P, P, P, P, i64, i32, i32, P, P, sz, P], i32),
        "moe_dense_mlp_prepared": ([P, P, P, P, i64, i32, i32, P, P, sz, P], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def _check(status: int, what: str) -> None:
    if status != MOE_OK:
        L = lib()
        detail = L.moe_last_error().decode()
        raise MoEError(status, f"{what}: {L.moe_status_string(status).decode()}"
                               + (f" -- {detail}" if detail else ""))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _bf16(t, name, shape=None):
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _f16(t, name, shape=None):
    if t.dtype != torch.float16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous fp16 CUDA tensor "
                         "(convert the bf16 weights once with prepare_weights)")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _down(t, name, shape=None) -> bool:
    """Checks a down-projection weight; True if it is the prepared fp16 copy."""
    if t.dtype == torch.float16:
        _f16(t, name, shape)
        return True
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bf16 (or its fp16 copy from prepare_weights)")
    _bf16(t, name, shape)
    return False


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def moe_kernel_launch_count() -> int:
    return int(lib().moe_kernel_launch_count())


def moe_route_raw(x, router, k: int, norm_topk_prob: bool, shared_gate=None,
                  want_bf16: bool = False):
    """Routing in the library's own types: (topk_w fp32 [N,k], topk_ids int32
    [N,k], gamma fp32 [N] or None, topk_w_bf16 or None)."""
    N, H = x.shape
    E = router.shape[0]
    _bf16(x, "x")
    _bf16(router, "router", (E, H))
    if shared_gate is not None:
        _bf16(shared_gate, "shared_gate", (1, H))
    dev = x.device
    w = torch.empty((N, k), dtype=torch.float32, device=dev)
    ids = torch.empty((N, k), dtype=torch.int32, device=dev)
    wb = torch.empty((N, k), dtype=torch.bfloat16, device=dev) if want_bf16 else None
    gamma = torch.empty(N, dtype=torch.float32, device=dev) if shared_gate is not None else None
    ws = torch.empty(lib().moe_route_workspace_bytes(), dtype=torch.uint8, device=dev)
    _check(lib().moe_route(_ptr(x), _ptr(router), _ptr(shared_gate), N, H, E, k,
                           int(bool(norm_topk_prob)), _ptr(w), _ptr(ids), _ptr(wb), _ptr(gamma),
                           _ptr(ws), ws.numel(), _stream()), "moe_route")
    return w, ids, gamma, wb


def moe_route(x, router, k: int, norm_topk_prob: bool = True):
    """The pages' route(): (weights in x.dtype, ids int64), each [N, k]."""
    _, ids, _, wb = moe_route_raw(x, router, k, norm_topk_prob, want_bf16=True)
    return wb, ids.long()


def moe_align(topk_ids, E: int, block_m: int = MOE_BLOCK_M):
    """Grouping of the pairs by expert; returns a dict of CUDA tensors."""
    if topk_ids.dtype != torch.int32 or not topk_ids.is_cuda or not topk_ids.is_contiguous():
        raise ValueError("topk_ids must be a contiguous int32 CUDA tensor")
    N, k = topk_ids.shape
    L = lib()
    cap = int(L.moe_align_capacity(N, k, E, block_m))
    dev = topk_ids.device
    sp = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
    be = torch.empty(max(cap // block_m, 1), dtype=torch.int32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    npad = torch.empty(1, dtype=torch.int32, device=dev)
    wsb = int(L.moe_align_workspace_bytes(N, k, E, block_m))
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    _check(L.moe_align(_ptr(topk_ids), N, k, E, block_m, _ptr(sp), _ptr(be), _ptr(counts),
                       _ptr(offsets), _ptr(npad), _ptr(ws), wsb, _stream()), "moe_align")
    return {"sorted_pair": sp, "block_expert": be, "counts": counts, "offsets": offsets,
            "num_padded": npad, "capacity": cap, "workspace": ws}


def moe_align_noalloc(topk_ids, E: int, block_m: int = MOE_BLOCK_M):
    """moe_align for callers that cannot allocate scratch (see moe.h): the
    library's static device array serves as the workspace.  Returns the same
    dict as moe_align, with "status" (int32 [1]) in place of "workspace"."""
    if topk_ids.dtype != torch.int32 or not topk_ids.is_cuda or not topk_ids.is_contiguous():
        raise ValueError("topk_ids must be a contiguous int32 CUDA tensor")
    N, k = topk_ids.shape
    L = lib()
    cap = int(L.moe_align_capacity(N, k, E, block_m))
    dev = topk_ids.device
    sp = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
    be = torch.empty(max(cap // block_m, 1), dtype=torch.int32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    npad = torch.empty(1, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    _check(L.moe_align_noalloc(_ptr(topk_ids), N, k, E, block_m, _ptr(sp), _ptr(be),
                               _ptr(counts), _ptr(offsets), _ptr(npad), _ptr(status), _stream()),
           "moe_align_noalloc")
    return {"sorted_pair": sp, "block_expert": be, "counts": counts, "offsets": offsets,
            "num_padded": npad, "capacity": cap, "status": status}


def moe_forward_layout(N, H, E, I, k, I_s=0) -> dict:
    lay = _Layout()
    _check(lib().moe_forward_layout(N, H, E, I, k, I_s, ctypes.byref(lay)), "moe_forward_layout")
    return {name: getattr(lay, name) for name, _ in _Layout._fields_}


def moe_forward_workspace_bytes(N, H, E, I, k, I_s=0) -> int:
    return int(lib().moe_forward_workspace_bytes(N, H, E, I, k, I_s))


def alloc_workspace(N, H, E, I, k, I_s=0, device="cuda"):
    """A workspace tensor for moe_forward (the caller owns it and may reuse it)."""
    return torch.empty(max(moe_forward_workspace_bytes(N, H, E, I, k, I_s), 256),
                       dtype=torch.uint8, device=device)


def moe_forward(x, router, w_gate, w_up, w_down, k: int, norm_topk_prob: bool = True,
                shared=None, out=None, workspace=None):
    """The whole layer.  ``shared`` is None or a dict with shared_gate_proj,
    shared_up_proj, shared_down_proj and shared_gate.  Every tensor is bf16,
    except that w_down and shared_down_proj may instead be the fp16 copies
    from ``prepare_weights`` (then moe_forward_prepared runs).  Returns out
    [N, H] bf16."""
    N, H = x.shape
    E, I, _ = w_gate.shape
    _bf16(x, "x")
    _bf16(router, "router", (E, H))
    _bf16(w_gate, "w_gate", (E, I, H))
    _bf16(w_up, "w_up", (E, I, H))
    prepared = _down(w_down, "w_down", (E, H, I))
    sp = [None] * 4
    I_s = 0
    if shared is not None:
        sp = [shared[n] for n in SHARED_KEYS]
        I_s = sp[0].shape[0]
        _bf16(sp[0], "shared_gate_proj", (I_s, H))
        _bf16(sp[1], "shared_up_proj", (I_s, H))
        if _down(sp[2], "shared_down_proj", (H, I_s)) != prepared:
            raise ValueError("w_down and shared_down_proj must both be bf16 or both fp16")
        _bf16(sp[3], "shared_gate", (1, H))
    if out is None:
        out = torch.empty((N, H), dtype=torch.bfloat16, device=x.device)
    _bf16(out, "out", (N, H))
    if workspace is None:
        workspace = alloc_workspace(N, H, E, I, k, I_s, x.device)
    fn = lib().moe_forward_prepared if prepared else lib().moe_forward
    _check(fn(_ptr(x), _ptr(router), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
              *[_ptr(t) for t in sp], N, H, E, I, I_s, k, int(bool(norm_topk_prob)), _ptr(out),
              _ptr(workspace), workspace.numel(), _stream()),
           "moe_forward_prepared" if prepared else "moe_forward")
    return out


def moe_add_rmsnorm(x, residual, weight, eps: float = 1e-6, gemma: bool = False, normed=None):
    """residual <- bf16(x + residual) in place; returns RMSNorm(residual) (bf16)."""
    N, H = x.shape
    _bf16(x, "x")
    _bf16(residual, "residual", (N, H))
    _bf16(weight, "weight", (H,))
    if normed is None:
        normed = torch.empty((N, H), dtype=torch.bfloat16, device=x.device)
    _bf16(normed, "normed", (N, H))
    _check(lib().moe_add_rmsnorm(_ptr(x), _ptr(residual), _ptr(weight), N, H, float(eps),
                                 int(bool(gemma)), _ptr(normed), _stream()), "moe_add_rmsnorm")
    return normed


def moe_dense_mlp(x, w_gate, w_up, w_down, out=None, workspace=None):
    """Dense SwiGLU MLP (silu(x Wg^T) * (x Wu^T)) Wd^T on the grouped GEMM
    kernels; w_down bf16 (moe_dense_mlp) or its fp16 copy (_prepared)."""
    N, H = x.shape
    I = w_gate.shape[0]
    _bf16(x, "x")
    _bf16(w_gate, "w_gate", (I, H))
    _bf16(w_up, "w_up", (I, H))
    prepared = _down(w_down, "w_down", (H, I))
    if out is None:
        out = torch.empty((N, H), dtype=torch.bfloat16, device=x.device)
    _bf16(out, "out", (N, H))
    L = lib()
    if workspace is None:
        workspace = torch.empty(max(int(L.moe_dense_mlp_workspace_bytes(N, H, I)), 256),
                                dtype=torch.uint8, device=x.device)
    fn = L.moe_dense_mlp_prepared if prepared else L.moe_dense_mlp
    _check(fn(_ptr(x), _ptr(w_gate), _ptr(w_up), _ptr(w_down), N, H, I, _ptr(out),
              _ptr(workspace), workspace.numel(), _stream()), "moe_dense_mlp")
    return out


def moe_experts(x_rows, ids, weights, w_gate, w_up, w_down, y=None, workspace=None):
    """Per-row expert outputs y[r] = weights[r] * Expert_{ids[r]}(x_rows[r]) as
    pair rows (``(hi bf16 [R, H], res int8 [R, H])``, the format moe.h
    describes): the receiving side of expert-parallel dispatch.  w_down bf16
    (moe_experts) or its fp16 copy (moe_experts_prepared).  Returns (y,
    workspace)."""
    R, H = x_rows.shape
    E, I, _ = w_gate.shape
    _bf16(x_rows, "x_rows")
    _bf16(w_gate, "w_gate", (E, I, H))
    _bf16(w_up, "w_up", (E, I, H))
    prepared = _down(w_down, "w_down", (E, H, I))
    if ids.dtype != torch.int32 or not ids.is_cuda or tuple(ids.shape) != (R,):
        raise ValueError("ids must be a CUDA int32 tensor of shape [R]")
    if weights.dtype != torch.float32 or not weights.is_cuda or tuple(weights.shape) != (R,):
        raise ValueError("weights must be a CUDA float32 tensor of shape [R]")
    ids, weights = ids.contiguous(), weights.contiguous()
    if y is None:
        y = alloc_pair_rows(R, H, x_rows.device)
    _check_pair_rows(y, R, H, "y")
    if workspace is None:
        workspace = torch.empty(max(lib().moe_experts_workspace_bytes(R, H, E, I), 256),
                                dtype=torch.uint8, device=x_rows.device)
    fn = lib().moe_experts_prepared if prepared else lib().moe_experts
    _check(fn(_ptr(x_rows), _ptr(ids), _ptr(weights), R, H, E, I, _ptr(w_gate), _ptr(w_up),
              _ptr(w_down), _ptr(y[0]), _ptr(y[1]), _ptr(workspace), workspace.numel(),
              _stream()), "moe_experts")
    return y, workspace


def alloc_pair_rows(R: int, H: int, device="cuda"):
    """Empty pair rows of [R, H] values: (hi bf16 [R, H], res int8 [R, H])."""
    return (torch.empty((R, H), dtype=torch.bfloat16, device=device),
            torch.empty((R, H), dtype=torch.int8, device=device))


def _check_pair_rows(y, R, H, name):
    hi, res = y
    if (hi.dtype != torch.bfloat16 or res.dtype != torch.int8 or tuple(hi.shape) != (R, H)
            or tuple(res.shape) != (R, H) or not hi.is_contiguous() or not res.is_contiguous()
            or not hi.is_cuda or not res.is_cuda):
        raise ValueError(f"{name} must be pair rows: (bf16 [{R}, {H}], int8 [{R}, {H}]) "
                         "contiguous CUDA tensors")


def _shared_rows(yshared, N, H):
    """(planes, S) of the shared expert's pair rows [N*S, H] (S rows per
    token, moe_shared_expert's output), or ((None, None), 0)."""
    if yshared is None:
        return (None, None), 0
    rows = yshared[0].shape[0]
    if N == 0 or rows % N or rows == 0:
        raise ValueError("yshared must hold S >= 1 rows per token ([N*S, H])")
    _check_pair_rows(yshared, rows, H, "yshared")
    return yshared, rows // N


def moe_combine(ypair, N: int, k: int, yshared=None, out=None):
    """out[n] = bf16(sum_j ypair[n*k + j] + sum_c yshared[n*S + c]) in fp32,
    slot order; ypair and yshared are pair rows (hi, res), yshared (optional)
    with S rows per token (moe_shared_expert's chunks)."""
    H = ypair[0].shape[1]
    _check_pair_rows(ypair, N * k, H, "ypair")
    sh, S = _shared_rows(yshared, N, H)
    if out is None:
        out = torch.empty((N, H), dtype=torch.bfloat16, device=ypair[0].device)
    _bf16(out, "out", (N, H))
    _check(lib().moe_combine(_ptr(ypair[0]), _ptr(ypair[1]), _ptr(sh[0]), _ptr(sh[1]), S, N, H,
                             k, _ptr(out), _stream()), "moe_combine")
    return out


def moe_combine_indexed(yrows, row_index, N: int, k: int, yshared=None, out=None):
    """moe_combine over pair rows in another order: pair p reads row
    row_index[p] of yrows (pair rows (hi, res), [R, H]); an index outside
    [0, R) contributes nothing."""
    R, H = yrows[0].shape
    _check_pair_rows(yrows, R, H, "yrows")
    if (row_index.dtype != torch.int32 or tuple(row_index.shape) != (N * k,) or
            not row_index.is_cuda or not row_index.is_contiguous()):
        raise ValueError("row_index must be a contiguous int32 CUDA tensor of shape [N*k]")
    sh, S = _shared_rows(yshared, N, H)
    if out is None:
        out = torch.empty((N, H), dtype=torch.bfloat16, device=row_index.device)
    _bf16(out, "out", (N, H))
    _check(lib().moe_combine_indexed(_ptr(yrows[0]), _ptr(yrows[1]), R, _ptr(row_index),
                                     _ptr(sh[0]), _ptr(sh[1]), S, N, H, k, _ptr(out),
                                     _stream()),
           "moe_combine_indexed")
    return out


def moe_shared_chunks(I: int, I_s: int) -> int:
    """C = ceil(I_s / I): the chunks (virtual experts) of the shared expert."""
    return int(lib().moe_shared_chunks(I, I_s))


def moe_shared_expert(x, gamma, I: int, shared_gate_proj, shared_up_proj, shared_down_proj,
                      y=None, workspace=None):
    """The gated shared expert on its own, as moe_forward computes it: pair
    rows [N*C, H], row n*C + c = gamma[n] * (chunk c of SharedMLP)(x[n]), C =
    ceil(I_s / I) with I the routed experts' intermediate size (moe.h).
    shared_down_proj bf16 or its fp16 copy.  Returns (y, workspace)."""
    N, H = x.shape
    I_s = shared_gate_proj.shape[0]
    _bf16(x, "x")
    _bf16(shared_gate_proj, "shared_gate_proj", (I_s, H))
    _bf16(shared_up_proj, "shared_up_proj", (I_s, H))
    prepared = _down(shared_down_proj, "shared_down_proj", (H, I_s))
    if gamma.dtype != torch.float32 or not gamma.is_cuda or tuple(gamma.shape) != (N,):
        raise ValueError("gamma must be a CUDA float32 tensor of shape [N]")
    gamma = gamma.contiguous()
    C = moe_shared_chunks(I, I_s)
    if y is None:
        y = alloc_pair_rows(N * C, H, x.device)
    _check_pair_rows(y, N * C, H, "y")
    if workspace is None:
        workspace = torch.empty(max(lib().moe_shared_expert_workspace_bytes(N, H, I, I_s), 256),
                                dtype=torch.uint8, device=x.device)
    fn = lib().moe_shared_expert_prepared if prepared else lib().moe_shared_expert
    _check(fn(_ptr(x), _ptr(gamma), N, H, I, I_s, _ptr(shared_gate_proj), _ptr(shared_up_proj),
              _ptr(shared_down_proj), _ptr(y[0]), _ptr(y[1]), _ptr(workspace), workspace.numel(),
              _stream()), "moe_shared_expert")
    return y, workspace


def moe_ep_dispatch(x, topk_ids, topk_w, E: int, world: int):
    """The sending side of expert-parallel dispatch on the device (moe.h):
    returns a dict with send_x [N*k, H] bf16, send_ids [N*k] int32 (local
    expert ids), send_w [N*k] fp32, send_counts [world] int32 (device),
    inv_order [N*k] int32 and the workspace (status word first)."""
    N, H = x.shape
    _bf16(x, "x")
    k = topk_ids.shape[1]
    if topk_ids.dtype != torch.int32 or tuple(topk_ids.shape) != (N, k) or not topk_ids.is_cuda:
        raise ValueError("topk_ids must be an int32 CUDA tensor of shape [N, k]")
    if topk_w.dtype != torch.float32 or tuple(topk_w.shape) != (N, k) or not topk_w.is_cuda:
        raise ValueError("topk_w must be a float32 CUDA tensor of shape [N, k]")
    topk_ids, topk_w = topk_ids.contiguous(), topk_w.contiguous()
    dev = x.device
    P = N * k
    r = {"send_x": torch.empty((P, H), dtype=torch.bfloat16, device=dev),
         "send_ids": torch.empty(P, dtype=torch.int32, device=dev),
         "send_w": torch.empty(P, dtype=torch.float32, device=dev),
         "send_counts": torch.zeros(world, dtype=torch.int32, device=dev),
         "inv_order": torch.empty(P, dtype=torch.int32, device=dev)}
    L = lib()
    wsb = int(L.moe_ep_dispatch_workspace_bytes(N, k, world))
    r["workspace"] = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    _check(L.moe_ep_dispatch(_ptr(x), _ptr(topk_ids), _ptr(topk_w), N, H, k, E, world,
                             _ptr(r["send_x"]), _ptr(r["send_ids"]), _ptr(r["send_w"]),
                             _ptr(r["send_counts"]), _ptr(r["inv_order"]), _ptr(r["workspace"]),
                             r["workspace"].numel(), _stream()), "moe_ep_dispatch")
    return r


def convert_bf16_to_f16(src, out=None, status=None):
    """fp16 copy of a bf16 CUDA tensor (round to nearest even; exact for
    |v| >= 2^-14).  ``status`` (int32 CUDA tensor, optional) receives
    MOE_ERR_DEVICE_CHECK when a value exceeds fp16's range or is NaN."""
    if src.dtype != torch.bfloat16 or not src.is_cuda or not src.is_contiguous():
        raise ValueError("src must be a contiguous bf16 CUDA tensor")
    if out is None:
        out = torch.empty(src.shape, dtype=torch.float16, device=src.device)
    _f16(out, "out", src.shape)
    _check(lib().moe_convert_bf16_to_f16(_ptr(src), _ptr(out), src.numel(), _ptr(status),
                                         _stream()), "moe_convert_bf16_to_f16")
    return out


DOWN_KEYS = ("w_down", "shared_down_proj")


def prepare_weights(weights: dict) -> dict:
    """The layer's weights in the form the *_prepared entry points take: the
    same dict with the down projections (w_down, shared_down_proj) converted
    to fp16 once; bf16 entries pass through.  Raises if a down weight is
    outside fp16's range."""
    out = dict(weights)
    dev = next(t.device for t in weights.values() if torch.is_tensor(t))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for name in DOWN_KEYS:
        if name in weights and weights[name].dtype == torch.bfloat16:
            out[name] = convert_bf16_to_f16(weights[name], status=status)
    code = int(status.item())
    if code != MOE_OK:
        raise MoEError(code, "prepare_weights: a down-projection weight exceeds fp16's range")
    return out


def moe_forward_from_host(x_host, out_host, x_dev, out_dev, weights: dict, k: int,
                          norm_topk_prob: bool, workspace):
    """End-to-end call with host buffers through moe_forward_host: x (pinned
    host) is copied to the device staging buffer x_dev, the layer runs, and
    the result is copied from out_dev back to pinned host memory, all on the
    current stream.  Weights stay resident on the device."""
    N, H = x_host.shape
    E, I, _ = weights["w_gate"].shape
    if x_host.is_cuda or out_host.is_cuda:
        raise ValueError("x_host and out_host must be host tensors")
    if x_host.dtype != torch.bfloat16 or out_host.dtype != torch.bfloat16:
        raise ValueError("x_host and out_host must be bf16")
    if not (x_host.is_contiguous() and out_host.is_contiguous()) or out_host.shape != (N, H):
        raise ValueError("x_host and out_host must be contiguous [N, H]")
    _bf16(x_dev, "x_dev", (N, H))
    _bf16(out_dev, "out_dev", (N, H))
    prepared = _down(weights["w_down"], "w_down", (E, H, I))
    shared = "shared_gate" in weights
    if shared and _down(weights["shared_down_proj"], "shared_down_proj") != prepared:
        raise ValueError("w_down and shared_down_proj must both be bf16 or both fp16")
    sp = [weights[n] if shared else None for n in SHARED_KEYS]
    I_s = weights["shared_gate_proj"].shape[0] if shared else 0
    fn = lib().moe_forward_host_prepared if prepared else lib().moe_forward_host
    _check(fn(x_host.data_ptr(), out_host.data_ptr(), _ptr(x_dev), _ptr(out_dev),
              _ptr(weights["router"]), _ptr(weights["w_gate"]), _ptr(weights["w_up"]),
              _ptr(weights["w_down"]), *[_ptr(t) for t in sp], N, H, E, I, I_s, k,
              int(bool(norm_topk_prob)), _ptr(workspace), workspace.numel(), _stream()),
           "moe_forward_host")
    return out_host


class ForwardGraph:
    """moe_forward captured once in a CUDA graph for a token bucket of
    `bucket` rows, then replayed: the serving decode loop's way of removing
    per-step launch cost.  A batch of n <= bucket tokens is copied into the
    first n rows of the static input (the rest zero); since every token's
    result is independent of the others, out[:n] equals an eager call on the
    n tokens bit for bit."""

    def __init__(self, weights: dict, k: int, norm_topk_prob: bool, bucket: int):
        dev = weights["router"].device
        H = weights["router"].shape[1]
        E, I, _ = weights["w_gate"].shape
        self.shared = ({n: weights[n] for n in SHARED_KEYS} if "shared_gate" in weights
                       else None)
        I_s = self.shared["shared_gate_proj"].shape[0] if self.shared else 0
        self.w, self.k, self.norm, self.bucket = weights, k, norm_topk_prob, bucket
        self.x = torch.zeros((bucket, H), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((bucket, H), dtype=torch.bfloat16, device=dev)
        self.ws = alloc_workspace(bucket, H, E, I, k, I_s, dev)
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for _ in range(2):
                self._call()
        torch.cuda.current_stream(dev).wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._call()

    def _call(self):
        w = self.w
        moe_forward(self.x, w["router"], w["w_gate"], w["w_up"], w["w_down"], self.k, self.norm,
                    self.shared, out=self.out, workspace=self.ws)

    def __call__(self, x):
        n = x.shape[0]
        if n > self.bucket:
            raise ValueError(f"{n} tokens exceed the graph's bucket of {self.bucket}")
        self.x[:n].copy_(x)
        if n < self.bucket:
            self.x[n:].zero_()
        self.graph.replay()
        return self.out[:n]


DECODE_BUCKETS = (1, 2, 4, 8, 16, 32, 64, 128)


class ForwardGraphSet:
    """The layer captured once per token bucket (1, 2, 4, ... 128 by default)
    and replayed for the smallest bucket that holds each step's batch: the
    decode loop of a serving engine, whose batch size changes from step to
    step, without per-step launch cost (the Nano-vLLM notes' model runner
    captures its decode step for a ladder of batch sizes the same way).

    Every bucket's graph reads the first b rows of one static input and
    writes the first b rows of one static output, and all of them use one
    workspace sized for the largest bucket: replays on one stream never
    overlap, and each graph carries its own workspace layout.  A batch of
    n tokens is copied into the input's first n rows (rows n..b-1 zeroed);
    since every token's result is independent of the others, the first n
    output rows equal an eager call on the n tokens bit for bit."""

    def __init__(self, weights: dict, k: int, norm_topk_prob: bool,
                 buckets=DECODE_BUCKETS):
        self.buckets = tuple(sorted(set(int(b) for b in buckets)))
        if not self.buckets or self.buckets[0] < 1:
            raise ValueError("buckets must be positive token counts")
        dev = weights["router"].device
        H = weights["router"].shape[1]
        E, I, _ = weights["w_gate"].shape
        self.shared = ({n: weights[n] for n in SHARED_KEYS} if "shared_gate" in weights
                       else None)
        I_s = self.shared["shared_gate_proj"].shape[0] if self.shared else 0
        self.w, self.k, self.norm = weights, k, norm_topk_prob
        top = self.buckets[-1]
        self.x = torch.zeros((top, H), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((top, H), dtype=torch.bfloat16, device=dev)
        self.ws = torch.empty(max(max(moe_forward_workspace_bytes(b, H, E, I, k, I_s)
                                      for b in self.buckets), 256),
                              dtype=torch.uint8, device=dev)
        self.graphs = {}
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for b in self.buckets:  # warm every shape once before capture
                self._call(b)
        torch.cuda.current_stream(dev).wait_stream(side)
        for b in self.buckets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._call(b)
            self.graphs[b] = g

    def _call(self, b):
        w = self.w
        moe_forward(self.x[:b], w["router"], w["w_gate"], w["w_up"], w["w_down"], self.k,
                    self.norm, self.shared, out=self.out[:b], workspace=self.ws)

    def bucket_of(self, n: int) -> int:
        for b in self.buckets:
            if b >= n:
                return b
        raise ValueError(f"{n} tokens exceed the largest bucket ({self.buckets[-1]})")

    def __call__(self, x):
        """out[:n] for this step's x [n, H] (a view of the static output,
        valid until the next call)."""
        n = x.shape[0]
        if n == 0:
            return self.out[:0]
        b = self.bucket_of(n)
        self.x[:n].copy_(x)
        if n < b:
            self.x[n:b].zero_()
        self.graphs[b].replay()
        return self.out[:n]

    def read_device_status(self) -> int:
        """Status word of the last replay (synchronises the stream)."""
        return moe_read_device_status(self.ws)


def decode_loop(graphs: ForwardGraphSet, steps):
    """Runs a multi-step decode: for each step's activations x_t [n_t, H]
    (n_t may change from step to step), the MoE layer by graph replay.
    Returns the per-step outputs (copies) and raises if a kernel recorded a
    device-side failure."""
    outs = [graphs(x).clone() for x in steps]
    status = graphs.read_device_status()
    if status != MOE_OK:
        raise MoEError(status, f"decode loop: {moe_status_string(status)}")
    return outs


def workspace_views(workspace, N, H, E, I, k, I_s=0) -> dict:
    """Typed views of moe_forward's intermediate buffers inside ``workspace``.

    With the shared expert every token has ``slots`` = k + C slots (the
    routed ones, then the shared expert's C chunks as virtual experts E + c)
    grouped over ``groups`` = E + C experts; topk_w / topk_ids / ypair hold
    all slots, ``routed_w`` / ``routed_ids`` only the first k."""
    lay = moe_forward_layout(N, H, E, I, k, I_s)
    cap = lay["capacity"]
    slots, groups = lay["slots"], lay["groups"]
    P = N * slots
    base = workspace

    def view(off, dtype, shape):
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return base[off:off + nbytes].view(dtype).view(shape)

    v = {
        "slots": slots,
        "groups": groups,
        "status": view(lay["status"], torch.int32, (1,)),
        "topk_w": view(lay["topk_w"], torch.float32, (N, slots)),
        "topk_ids": view(lay["topk_ids"], torch.int32, (N, slots)),
        "counts": view(lay["counts"], torch.int32, (groups,)),
        "offsets": view(lay["offsets"], torch.int32, (groups + 1,)),
        "pad_offsets": view(lay["pad_offsets"], torch.int32, (groups + 1,)),
        "num_padded": view(lay["num_padded"], torch.int32, (1,)),
        "sorted_pair": view(lay["sorted_pair"], torch.int32, (cap,)),
        "block_expert": view(lay["block_expert"], torch.int32, (cap // MOE_BLOCK_M,)),
        "x_sorted": view(lay["x_sorted"], torch.bfloat16, (cap, H)),
        # the activation: a bf16 hi/lo pair (bf16 down weights) or fp16
        # (prepared fp16 down weights), in the same bytes
        "act_hi": view(lay["act"], torch.bfloat16, (cap, I)),
        "act_lo": view(lay["act"] + 2 * cap * I, torch.bfloat16, (cap, I)),
        "act_f16": view(lay["act"], torch.float16, (cap, I)),
        # pair rows (hi, res) of w * Expert(x), one row per slot
        "ypair": (view(lay["ypair"], torch.bfloat16, (P, H)),
                  view(lay["ypair_res"], torch.int8, (P, H))),
    }
    v["routed_w"] = v["topk_w"][:, :k]
    v["routed_ids"] = v["topk_ids"][:, :k]
    if I_s:
        v["gamma"] = view(lay["gamma"], torch.float32, (N,))
    return v


def moe_selftest_wait_timeout(workspace, limit_ns: int) -> None:
    """Enqueue the device wait-timeout self-check (see moe.h)."""
    _check(lib().moe_selftest_wait_timeout(_ptr(workspace), workspace.numel(), int(limit_ns),
                                           _stream()), "moe_selftest_wait_timeout")


def moe_read_device_status(workspace) -> int:
    """Synchronise the current stream and return the workspace's status word."""
    return int(lib().moe_read_device_status(_ptr(workspace), _stream()))


def set_stage_events(events) -> None:
    """Record the given torch.cuda.Event objects (None entries skipped) around
    the stages of the next moe_forward calls on this thread (None to stop)."""
    L = lib()
    if events is None:
        _check(L.moe_set_stage_events(None, 0), "moe_set_stage_events")
        return
    if len(events) != MOE_NUM_STAGES + 1:
        raise ValueError(f"need {MOE_NUM_STAGES + 1} events")
    for e in events:
        if e is not None and not e.cuda_event:  # torch creates it on first record
            e.record()
    arr = (ctypes.c_void_p * len(events))(
        *[ctypes.c_void_p(e.cuda_event if e is not None else None) for e in events])
    _check(L.moe_set_stage_events(arr, len(events)), "moe_set_stage_events")
