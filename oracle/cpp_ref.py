"""Loader of the second CPU oracle, the plain C++ program in moe_oracle_ref.cpp
(test infrastructure only; the library's compute path never imports it).

build() compiles it with the host C++ compiler into liboracle_ref.so beside
the source; the functions below marshal numpy arrays to it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle_ref.cpp")
LIB = os.path.join(HERE, "liboracle_ref.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C++ oracle (g++, -O2, no machine-specific flags); returns the library path."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", SRC, "-o", LIB], check=True)
    return LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i = ctypes.c_int
        lib.oracle_ref_route.argtypes = [i, i, i, P, P, P]
        lib.oracle_ref_sort.argtypes = [i, i, i, P, P, P, P]
        lib.oracle_ref_forward.argtypes = [i, i, i, i, i] + [P] * 12 + [i]
        for f in (lib.oracle_ref_route, lib.oracle_ref_sort, lib.oracle_ref_forward):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def route(router_logits: np.ndarray, k: int):
    """(topk_ids int32 [T, k], topk_w fp64 [T, k])"""
    logits = np.ascontiguousarray(router_logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    if _load().oracle_ref_route(T, E, k, _p(logits), _p(ids), _p(w)) != 0:
        raise ValueError("oracle_ref_route rejected its arguments")
    return ids, w


def expert_sort(topk_ids: np.ndarray, E: int):
    """(expert_offsets int32 [E+1], sorted_slot int32 [S], slot_pos int32 [S])"""
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T, k = ids.shape
    off = np.empty(E + 1, dtype=np.int32)
    ss = np.empty(T * k, dtype=np.int32)
    sp = np.empty(T * k, dtype=np.int32)
    if _load().oracle_ref_sort(T, E, k, _p(ids), _p(off), _p(ss), _p(sp)) != 0:
        raise ValueError("oracle_ref_sort rejected its arguments")
    return off, ss, sp


def forward(x_bf16, router_logits, w13, w13_scale, w2, w2_scale, k: int, threads: int | None = None):
    """The whole layer; the same dict keys as oracle.forward (without slot_pos)."""
    x = np.ascontiguousarray(np.asarray(x_bf16).view(np.uint16))
    logits = np.ascontiguousarray(router_logits, dtype=np.float32)
    w13 = np.ascontiguousarray(w13, dtype=np.uint8)
    w13s = np.ascontiguousarray(w13_scale, dtype=np.uint8)
    w2 = np.ascontiguousarray(w2, dtype=np.uint8)
    w2s = np.ascontiguousarray(w2_scale, dtype=np.uint8)
    T, d = x.shape
    E = w13.shape[0]
    I = w13.shape[1] // 2
    S = T * k
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    off = np.empty(E + 1, dtype=np.int32)
    ss = np.empty(S, dtype=np.int32)
    h = np.empty((S, I), dtype=np.float64)
    out = np.empty((T, d), dtype=np.float64)
    nt = threads or os.cpu_count() or 1
    rc = _load().oracle_ref_forward(T, d, I, E, k, _p(x), _p(logits), _p(w13), _p(w13s), _p(w2), _p(w2s), _p(ids),
                                    _p(w), _p(off), _p(ss), _p(h), _p(out), int(nt))
    if rc != 0:
        raise ValueError("oracle_ref_forward rejected its arguments")
    return dict(topk_ids=ids, topk_w=w, expert_offsets=off, sorted_slot=ss, h=h, out=out)
