"""CPU oracle for MoE route-sort -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The product (the CUDA library and its binding) never touches it and
shares no code with it.

The arithmetic lives in ``moe_route_sort_oracle.c`` (plain single-threaded C, IEEE fp32,
libm ``expf``, built with ``-ffp-contract=off``); this module compiles it with gcc and
wraps its entry points for numpy arrays.  What each step computes, and the readings taken
where the source pages are silent, are stated in the C file's header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_route_sort_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmoe_route_sort_oracle.so")

FLAG_BAD_EXPERT_ID = 0x1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libmoe_route_sort_oracle.so`` (gcc, no fast-math)."""
    up_to_date = (
        os.path.exists(_LIB_PATH)
        and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    )
    if up_to_date and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = [
        "gcc", "-O2", "-std=c11", "-fPIC", "-shared",
        "-ffp-contract=off", "-fno-fast-math", "-fexcess-precision=standard",
        "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm",
    ]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32 = ctypes.c_int
        f32 = ctypes.c_float
        lib.oracle_bf16_to_float.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_float.restype = f32
        lib.oracle_sigmoid.argtypes = [f32]
        lib.oracle_sigmoid.restype = f32
        lib.oracle_bf16_to_float_n.argtypes = [P, ctypes.c_int64, P]
        lib.oracle_bf16_to_float_n.restype = None
        lib.oracle_sigmoid_n.argtypes = [P, ctypes.c_int64, P]
        lib.oracle_sigmoid_n.restype = None
        lib.oracle_scores_row.argtypes = [P, P, i32, P, P]
        lib.oracle_scores_row.restype = None
        lib.oracle_group_scores_row.argtypes = [P, i32, i32, P]
        lib.oracle_group_scores_row.restype = i32
        lib.oracle_kept_groups_row.argtypes = [P, i32, i32, P]
        lib.oracle_kept_groups_row.restype = i32
        lib.oracle_topk_row.argtypes = [P, i32, i32, P, i32, P]
        lib.oracle_topk_row.restype = i32
        lib.oracle_weights_row.argtypes = [P, P, i32, f32, P]
        lib.oracle_weights_row.restype = None
        lib.oracle_route.argtypes = [P, P, i32, i32, i32, i32, i32, f32, P, P]
        lib.oracle_route.restype = i32
        lib.oracle_route_softmax.argtypes = [P, i32, i32, i32, f32, P, P]
        lib.oracle_gate_logits.argtypes = [P, P, i32, i32, i32, P]
        lib.oracle_route_softmax.restype = i32
        lib.oracle_max_padded.argtypes = [i32, i32, i32, i32]
        lib.oracle_max_padded.restype = ctypes.c_int64
        lib.oracle_sort.argtypes = [P, P, i32, i32, i32, i32, P, P, P, P, P]
        lib.oracle_sort.restype = i32
        lib.oracle_margins.argtypes = [P, P, i32, i32, i32, i32, i32, P]
        lib.oracle_margins.restype = i32
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 logits must be passed as their uint16 bit patterns")
    return a


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


# ------------------------------------------------------------------ scalar steps
def bf16_to_float(bits: int) -> float:
    return float(_load().oracle_bf16_to_float(int(bits)))


def sigmoid(x: float) -> float:
    return float(_load().oracle_sigmoid(float(x)))


def bf16_to_float_array(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = _u16(bits).reshape(-1)
    out = np.empty(flat.shape[0], np.float32)
    lib.oracle_bf16_to_float_n(_ptr(flat), flat.shape[0], _ptr(out))
    return out.reshape(np.shape(bits))


def sigmoid_array(x: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = _f32(x).reshape(-1)
    out = np.empty(flat.shape[0], np.float32)
    lib.oracle_sigmoid_n(_ptr(flat), flat.shape[0], _ptr(out))
    return out.reshape(np.shape(x))


# --------------------------------------------------------------- per-row steps
def scores_row(logits_row: np.ndarray, bias: np.ndarray):
    """(s, key) of one token row."""
    lib = _load()
    row = _u16(logits_row).reshape(-1)
    b = _f32(bias)
    E = row.shape[0]
    s = np.empty(E, np.float32)
    key = np.empty(E, np.float32)
    lib.oracle_scores_row(_ptr(row), _ptr(b), E, _ptr(s), _ptr(key))
    return s, key


def group_scores_row(key: np.ndarray, n_group: int) -> np.ndarray:
    lib = _load()
    k = _f32(key)
    gs = np.empty(n_group, np.float32)
    _check(lib.oracle_group_scores_row(_ptr(k), k.shape[0], n_group, _ptr(gs)), "group_scores")
    return gs


def kept_groups_row(gs: np.ndarray, topk_group: int) -> np.ndarray:
    lib = _load()
    g = _f32(gs)
    kept = np.empty(g.shape[0], np.int32)
    _check(lib.oracle_kept_groups_row(_ptr(g), g.shape[0], topk_group, _ptr(kept)), "kept")
    return kept


def topk_row(key: np.ndarray, n_group: int, kept: np.ndarray, topk: int) -> np.ndarray:
    lib = _load()
    k = _f32(key)
    kf = _i32(kept)
    ids = np.empty(topk, np.int32)
    _check(lib.oracle_topk_row(_ptr(k), k.shape[0], n_group, _ptr(kf), topk, _ptr(ids)), "topk")
    return ids


def weights_row(s: np.ndarray, ids: np.ndarray, routed_scale: float) -> np.ndarray:
    lib = _load()
    sv = _f32(s)
    iv = _i32(ids)
    w = np.empty(iv.shape[0], np.float32)
    lib.oracle_weights_row(_ptr(sv), _ptr(iv), iv.shape[0], float(routed_scale), _ptr(w))
    return w


# ----------------------------------------------------------------- whole steps
def route(logits, bias, n_group, topk_group, topk, routed_scale):
    """topk_ids [T,K] int32, topk_weights [T,K] float32."""
    lib = _load()
    lg = _u16(logits)
    T, E = lg.shape
    b = _f32(bias)
    ids = np.empty((T, topk), np.int32)
    w = np.empty((T, topk), np.float32)
    _check(
        lib.oracle_route(_ptr(lg), _ptr(b), T, E, n_group, topk_group, topk,
                         float(routed_scale), _ptr(ids), _ptr(w)),
        "route",
    )
    return ids, w


def route_softmax(logits, topk, routed_scale):
    """Softmax variant (R9, no bias, no groups): topk_ids [T,K], topk_weights [T,K]."""
    lib = _load()
    lg = _u16(logits)
    T, E = lg.shape
    ids = np.empty((T, topk), np.int32)
    w = np.empty((T, topk), np.float32)
    _check(lib.oracle_route_softmax(_ptr(lg), T, E, topk, float(routed_scale), _ptr(ids),
                                    _ptr(w)), "route_softmax")
    return ids, w


def route_sort_softmax(logits, topk, routed_scale, block_m):
    ids, w = route_softmax(logits, topk, routed_scale)
    res = sort(ids, w, np.shape(logits)[1], block_m)
    res["topk_ids"] = ids
    res["topk_weights"] = w
    return res


def max_padded(T: int, E: int, topk: int, block_m: int) -> int:
    return int(_load().oracle_max_padded(T, E, topk, block_m))


class SortResult(dict):
    """sorted_token_ids / sorted_weights on [0, npp), expert_ids on [0, npp/B), npp, flags."""

    __getattr__ = dict.__getitem__


def sort(topk_ids, topk_weights, E: int, block_m: int) -> SortResult:
    lib = _load()
    ids = _i32(topk_ids)
    w = _f32(topk_weights)
    T, K = ids.shape
    P = max(max_padded(T, E, K, block_m), 1)
    sid = np.full(P, -1, np.int32)
    sw = np.zeros(P, np.float32)
    eid = np.full(max(P // block_m, 1), -1, np.int32)
    npp = np.zeros(1, np.int32)
    flags = np.zeros(1, np.int32)
    _check(
        lib.oracle_sort(_ptr(ids), _ptr(w), T, E, K, block_m, _ptr(sid), _ptr(sw), _ptr(eid),
                        _ptr(npp), _ptr(flags)),
        "sort",
    )
    n = int(npp[0])
    return SortResult(
        sorted_token_ids=sid[:n].copy(),
        sorted_weights=sw[:n].copy(),
        expert_ids=eid[: n // block_m].copy(),
        num_tokens_post_pad=n,
        flags=int(flags[0]),
    )


def route_sort(logits, bias, n_group, topk_group, topk, routed_scale, block_m):
    ids, w = route(logits, bias, n_group, topk_group, topk, routed_scale)
    E = np.shape(logits)[1]
    res = sort(ids, w, E, block_m)
    res["topk_ids"] = ids
    res["topk_weights"] = w
    return res


def gate_logits(hidden, w_gate) -> np.ndarray:
    """R14: bf16 logits [T,E] of bf16 hidden [T,H] and bf16 gate rows [E,H]: each the exact
    dot product rounded once to bf16 (nearest, ties to even)."""
    hs = _u16(hidden)
    ws = _u16(w_gate)
    T, H = hs.shape
    E, H2 = ws.shape
    if H != H2:
        raise ValueError("hidden and gate rows differ in length")
    out = np.empty((T, E), np.uint16)
    _check(_load().oracle_gate_logits(_ptr(hs), _ptr(ws), T, E, H, _ptr(out)), "gate_logits")
    return out


def gate_route_sort(hidden, w_gate, bias, n_group, topk_group, topk, routed_scale, block_m):
    """Gate projection (R14) then the whole path; the result also holds the logits."""
    logits = gate_logits(hidden, w_gate)
    res = route_sort(logits, bias, n_group, topk_group, topk, routed_scale, block_m)
    res["logits"] = logits
    return res


def margins(logits, bias, n_group, topk_group, topk) -> np.ndarray:
    """Per-token smallest selection gap (see the C header); used to redraw near-ties."""
    lib = _load()
    lg = _u16(logits)
    T, E = lg.shape
    b = _f32(bias)
    m = np.empty(T, np.float32)
    _check(lib.oracle_margins(_ptr(lg), _ptr(b), T, E, n_group, topk_group, topk, _ptr(m)),
           "margins")
    return m
