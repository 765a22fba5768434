"""fp64 CPU oracle of the sparse MoE FFN layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never links, loads or
calls it, and it shares no code with that library: the C source
``moe_oracle.c`` widens raw bf16 bit patterns itself and computes every step
in fp64, following the M03 "Sparse MoE" drill (routing block, grouping
bookkeeping, shared expert) and the HF-style ``Qwen3MoeSparseMoeBlock`` of
the Nano-vLLM notes.

Inputs are numpy ``uint16`` arrays holding bf16 bit patterns (the exact values
the GPU receives).  ``bf16_bits`` converts a torch bf16 tensor to that form.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile an oracle C source into a shared library (gcc, portable C11)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-fPIC", "-shared", "-o", tmp, src,
               "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a, shape=None):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bf16 bit patterns, got {a.dtype}")
    if shape is not None and tuple(a.shape) != tuple(shape):
        raise ValueError(f"expected shape {shape}, got {a.shape}")
    return a


def bf16_bits(t) -> np.ndarray:
    """torch bf16 tensor (any device) -> numpy uint16 array of its bit patterns."""
    import torch
    if t.dtype != torch.bfloat16:
        raise TypeError(f"expected bfloat16, got {t.dtype}")
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def widen(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 (exact)."""
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def align_capacity(P: int, E: int, BM: int) -> int:
    """Largest padded length: round_up(P + E*(BM-1), BM)."""
    return -(-(P + E * (BM - 1)) // BM) * BM


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64, i32 = ctypes.c_int64, ctypes.c_int
        lib.oracle_route.argtypes = [P, P, i64, i32, i32, i32, i32, P, P, P, P]
        lib.oracle_route.restype = i32
        lib.oracle_align.argtypes = [P, i64, i32, i32, i32, P, P, P, P, i64, P, P]
        lib.oracle_align.restype = i32
        lib.oracle_moe_forward.argtypes = [P] * 9 + [i64, i32, i32, i32, i32, i32, i32,
                                                    P, i64, P, i32]
        lib.oracle_moe_forward.restype = i32
        lib.oracle_add_rmsnorm.argtypes = [P, P, P, i64, i32, ctypes.c_double, i32, P, P]
        lib.oracle_add_rmsnorm.restype = i32
        lib.oracle_hardware_threads.argtypes = []
        lib.oracle_hardware_threads.restype = i32
        self.lib = lib
        self.path = path

    def hardware_threads(self) -> int:
        return int(self.lib.oracle_hardware_threads())

    def route(self, x, router, k: int, norm: bool):
        """Routing of every token -> (logits [N,E], probs [N,E], w [N,k] f64, ids [N,k] i32)."""
        x = _u16(x)
        N, H = x.shape
        E = router.shape[0]
        router = _u16(router, (E, H))
        logits = np.zeros((N, E), np.float64)
        probs = np.zeros((N, E), np.float64)
        w = np.zeros((N, k), np.float64)
        ids = np.zeros((N, k), np.int32)
        rc = self.lib.oracle_route(_ptr(x), _ptr(router), N, H, E, k, int(bool(norm)),
                                   _ptr(logits), _ptr(probs), _ptr(w), _ptr(ids))
        if rc != 0:
            raise ValueError(f"oracle_route failed with code {rc}")
        return logits, probs, w, ids

    def align(self, ids, E: int, BM: int):
        """Grouping bookkeeping of the (token, slot) pairs -> dict of numpy arrays."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        N, k = ids.shape
        P = N * k
        cap = align_capacity(P, E, BM)
        counts = np.zeros(E, np.int32)
        offsets = np.zeros(E + 1, np.int32)
        order = np.zeros(max(P, 1), np.int32)
        sorted_pair = np.full(max(cap, 1), -1, np.int32)
        block_expert = np.full(max(cap // BM, 1), -1, np.int32)
        num_padded = np.zeros(1, np.int32)
        rc = self.lib.oracle_align(_ptr(ids), N, k, E, BM, _ptr(counts), _ptr(offsets),
                                   _ptr(order), _ptr(sorted_pair), cap, _ptr(block_expert),
                                   _ptr(num_padded))
        if rc != 0:
            raise ValueError(f"oracle_align failed with code {rc}")
        npad = int(num_padded[0])
        return {
            "counts": counts,
            "offsets": offsets,
            "order": order[:P],
            "sorted_pair": sorted_pair[:npad],
            "block_expert": block_expert[: npad // BM],
            "num_padded": npad,
            "flat_e": ids.reshape(-1).copy(),
            "flat_tok": np.repeat(np.arange(N, dtype=np.int64), k),
        }

    def add_rmsnorm(self, x, residual, weight, eps: float, gemma: bool = False):
        """(new residual as bf16 bits [N,H], normed [N,H] fp64)."""
        x = _u16(x)
        N, H = x.shape
        residual = _u16(residual, (N, H))
        weight = _u16(weight, (H,))
        res_out = np.zeros((N, H), np.uint16)
        normed = np.zeros((N, H), np.float64)
        rc = self.lib.oracle_add_rmsnorm(_ptr(x), _ptr(residual), _ptr(weight), N, H, float(eps),
                                         int(bool(gemma)), _ptr(res_out), _ptr(normed))
        if rc != 0:
            raise ValueError(f"oracle_add_rmsnorm failed with code {rc}")
        return res_out, normed

    def moe_forward(self, w: dict, k: int, norm: bool, rows=None, nthreads: int = 0):
        """out[r] = MoE(x[rows[r]]) in fp64.

        ``w`` holds uint16 bf16 bit arrays: x [N,H], router [E,H], w_gate/w_up
        [E,I,H], w_down [E,H,I] and optionally shared_gate_proj/shared_up_proj
        [I_s,H], shared_down_proj [H,I_s], shared_gate [1,H].  ``rows`` defaults
        to every token.  ``nthreads`` <= 0 uses every online core.
        """
        x = _u16(w["x"])
        N, H = x.shape
        router = _u16(w["router"])
        E = router.shape[0]
        wg = _u16(w["w_gate"])
        I = wg.shape[1]
        _u16(wg, (E, I, H))
        wu = _u16(w["w_up"], (E, I, H))
        wd = _u16(w["w_down"], (E, H, I))
        shared = [w.get(n) for n in SHARED_KEYS]
        I_s = 0
        if all(s is not None for s in shared):
            I_s = shared[0].shape[0]
            shared = [_u16(shared[0], (I_s, H)), _u16(shared[1], (I_s, H)),
                      _u16(shared[2], (H, I_s)), _u16(shared[3], (1, H))]
        elif any(s is not None for s in shared):
            raise ValueError("shared expert needs all four of gate_proj, up_proj, down_proj, gate")
        else:
            shared = [None] * 4
        if rows is None:
            rows = np.arange(N, dtype=np.int64)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.zeros((len(rows), H), np.float64)
        rc = self.lib.oracle_moe_forward(_ptr(x), _ptr(router), _ptr(wg), _ptr(wu), _ptr(wd),
                                         *[_ptr(s) for s in shared], N, H, E, I, I_s, int(k),
                                         int(bool(norm)), _ptr(rows), len(rows), _ptr(out),
                                         int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_moe_forward failed with code {rc}")
        return out


SHARED_KEYS = ("shared_gate_proj", "shared_up_proj", "shared_down_proj", "shared_gate")


def default() -> Oracle:
    """The oracle built from moe_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


_default = None


def hardware_threads() -> int:
    return default().hardware_threads()


def route(x, router, k: int, norm: bool):
    return default().route(x, router, k, norm)


def align(ids, E: int, BM: int):
    return default().align(ids, E, BM)


def moe_forward(w: dict, k: int, norm: bool, rows=None, nthreads: int = 0):
    return default().moe_forward(w, k, norm, rows, nthreads)


def add_rmsnorm(x, residual, weight, eps: float, gemma: bool = False):
    return default().add_rmsnorm(x, residual, weight, eps, gemma)
