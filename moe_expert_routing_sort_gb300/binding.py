"""Thin Python binding of the route-sort C ABI (ctypes; argument marshalling only).

Each function has the name of its C entry point, takes torch CUDA tensors for the device
buffers, passes their data pointers and the current (or given) CUDA stream, and raises
``RouteSortError`` on a negative status.  Every step of the path runs in the library's
CUDA kernels; if the library has not been built this module raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

from ._build import LIB_PATH

DEVICE_BAD_EXPERT_ID = 0x1

_lock = threading.Lock()
_lib = None


class RouteSortError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what} failed with status {status}: {strerror(status)}")


def library_path() -> str:
    return LIB_PATH


def load() -> ctypes.CDLL:
    """Load ``libmoe_route_sort.so``; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')"
            )
        lib = ctypes.CDLL(LIB_PATH)
        P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.moe_sort_max_padded.argtypes = [I, I, I, I]
        lib.moe_sort_max_padded.restype = S
        lib.moe_sort_max_blocks.argtypes = [I, I, I, I]
        lib.moe_sort_max_blocks.restype = S
        lib.moe_route_sort_workspace_bytes.argtypes = [I, I, I, I]
        lib.moe_route_sort_workspace_bytes.restype = S
        lib.moe_route_sort_strerror.argtypes = [I]
        lib.moe_route_sort_map_host.argtypes = [P, ctypes.POINTER(ctypes.c_void_p)]
        lib.moe_route_sort_map_host.restype = I
        lib.moe_route_sort_strerror.restype = ctypes.c_char_p
        lib.moe_route_sort.argtypes = [P, P, I, I, I, I, I, F, I, P, P, P, P, P, P, P, S, P]
        lib.moe_route_sort.restype = I
        lib.moe_gate_route_sort.argtypes = [P, P, P, I, I, I, I, I, I, F, I, P, P, P, P, P, P,
                                            P, P, S, P]
        lib.moe_gate_route_sort.restype = I
        lib.moe_route_sort_softmax.argtypes = [P, I, I, I, F, I, P, P, P, P, P, P, P, S, P]
        lib.moe_route_sort_softmax.restype = I
        lib.moe_topk.argtypes = [P, P, I, I, I, I, I, F, P, P, P]
        lib.moe_topk.restype = I
        lib.moe_sort.argtypes = [P, P, I, I, I, I, P, P, P, P, P, S, P]
        lib.moe_sort_atomic.argtypes = [P, P, I, I, I, I, P, P, P, P, P, S, P]
        lib.moe_sort_atomic.restype = I
        lib.moe_sort.restype = I
        lib.moe_route_sort_noalloc.argtypes = [P, P, I, I, I, I, I, F, I, P, P, P, P, P, P, P]
        lib.moe_route_sort_noalloc.restype = I
        lib.moe_route_sort_from_host.argtypes = [P, P, P, I, I, I, I, I, F, I, P, P, P, P, P, P,
                                                 P, S, P, P, S, P]
        lib.moe_route_sort_from_host.restype = I
        lib.moe_route_sort_proxy_selftest.argtypes = [P, P]
        lib.moe_route_sort_proxy_selftest.restype = I
        lib.moe_route_sort_proxy_state.argtypes = [P, P]
        lib.moe_route_sort_proxy_state.restype = I
        lib.moe_route_sort_noalloc_status.argtypes = [P, P]
        lib.moe_route_sort_noalloc_status.restype = I
        lib.moe_route_sort_debug_set.argtypes = [I, ctypes.c_longlong]
        lib.moe_route_sort_debug_set.restype = I
        _lib = lib
        return lib


# ------------------------------------------------------------------ size queries
def moe_sort_max_padded(T: int, E: int, topk: int, block_m: int) -> int:
    return int(load().moe_sort_max_padded(T, E, topk, block_m))


def moe_sort_max_blocks(T: int, E: int, topk: int, block_m: int) -> int:
    return int(load().moe_sort_max_blocks(T, E, topk, block_m))


def moe_route_sort_workspace_bytes(T: int, E: int, topk: int, block_m: int) -> int:
    return int(load().moe_route_sort_workspace_bytes(T, E, topk, block_m))


def strerror(status: int) -> str:
    return load().moe_route_sort_strerror(int(status)).decode()


# ------------------------------------------------------------------ marshalling
def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _one_device(*tensors) -> torch.device:
    """The one CUDA device that every given tensor (None skipped) lives on.

    The library runs on the current device and reads every pointer from there, so a call whose
    buffers sit on different devices (or on the host) is refused here, before any launch."""
    devs = {t.device for t in tensors if t is not None}
    if len(devs) != 1:
        raise ValueError(f"all buffers must be on one device, got {sorted(map(str, devs))}")
    dev = devs.pop()
    if dev.type != "cuda":
        raise ValueError(f"buffers must be CUDA tensors, got {dev}")
    return dev


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RouteSortError(rc, what)


def _sort_sizes(T: int, E: int, topk: int, block_m: int):
    """Element counts the sort outputs need (sorted rows, block owners); 0 for a shape the
    library rejects anyway."""
    return moe_sort_max_padded(T, E, topk, block_m), moe_sort_max_blocks(T, E, topk, block_m)


def _need_room(T: int, topk: int, P: int, NB: int, **bufs) -> None:
    """Raise before any launch if an output is smaller than the shape needs (the kernels
    would write past it)."""
    want = {"topk_ids": T * topk, "topk_weights": T * topk, "sorted_token_ids": P,
            "sorted_weights": P, "expert_ids": NB, "num_tokens_post_pad": 1}
    for name, t in bufs.items():
        n = want[name] if T > 0 or name == "num_tokens_post_pad" else 0
        if n > 0 and t.numel() < n:
            raise ValueError(f"{name} holds {t.numel()} elements; this shape needs {n}")


# -------------------------------------------------------------------- operations
def moe_route_sort(logits, bias, n_group, topk_group, topk, routed_scale, block_m,
                   topk_ids, topk_weights, sorted_token_ids, sorted_weights, expert_ids,
                   num_tokens_post_pad, workspace, stream=None) -> None:
    """Whole path into caller-owned buffers (see include/moe_route_sort.h)."""
    T, E = logits.shape
    _need(logits, torch.bfloat16, "logits")
    _need(bias, torch.float32, "bias")
    for t, dt, n in [(topk_ids, torch.int32, "topk_ids"), (topk_weights, torch.float32,
                     "topk_weights"), (sorted_token_ids, torch.int32, "sorted_token_ids"),
                     (sorted_weights, torch.float32, "sorted_weights"),
                     (expert_ids, torch.int32, "expert_ids"),
                     (num_tokens_post_pad, torch.int32, "num_tokens_post_pad"),
                     (workspace, torch.uint8, "workspace")]:
        _need(t, dt, n)
    _need_room(T, topk, *_sort_sizes(T, E, topk, block_m), topk_ids=topk_ids,
               topk_weights=topk_weights, sorted_token_ids=sorted_token_ids,
               sorted_weights=sorted_weights, expert_ids=expert_ids,
               num_tokens_post_pad=num_tokens_post_pad)
    dev = _one_device(logits, bias, topk_ids, topk_weights, sorted_token_ids, sorted_weights,
                      expert_ids, num_tokens_post_pad, workspace)
    with torch.cuda.device(dev):
        rc = load().moe_route_sort(
            _ptr(logits), _ptr(bias), T, E, n_group, topk_group, topk, float(routed_scale),
            block_m, _ptr(topk_ids), _ptr(topk_weights), _ptr(sorted_token_ids),
            _ptr(sorted_weights), _ptr(expert_ids), _ptr(num_tokens_post_pad),
            _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check(rc, "moe_route_sort")


def moe_route_sort_softmax(logits, topk, routed_scale, block_m, topk_ids, topk_weights,
                           sorted_token_ids, sorted_weights, expert_ids, num_tokens_post_pad,
                           workspace, stream=None) -> None:
    """Whole path with softmax scoring (no bias, no groups) into caller-owned buffers."""
    T, E = logits.shape
    _need(logits, torch.bfloat16, "logits")
    for t, dt, n in [(topk_ids, torch.int32, "topk_ids"), (topk_weights, torch.float32,
                     "topk_weights"), (sorted_token_ids, torch.int32, "sorted_token_ids"),
                     (sorted_weights, torch.float32, "sorted_weights"),
                     (expert_ids, torch.int32, "expert_ids"),
                     (num_tokens_post_pad, torch.int32, "num_tokens_post_pad"),
                     (workspace, torch.uint8, "workspace")]:
        _need(t, dt, n)
    _need_room(T, topk, *_sort_sizes(T, E, topk, block_m), topk_ids=topk_ids,
               topk_weights=topk_weights, sorted_token_ids=sorted_token_ids,
               sorted_weights=sorted_weights, expert_ids=expert_ids,
               num_tokens_post_pad=num_tokens_post_pad)
    dev = _one_device(logits, topk_ids, topk_weights, sorted_token_ids, sorted_weights,
                      expert_ids, num_tokens_post_pad, workspace)
    with torch.cuda.device(dev):
        rc = load().moe_route_sort_softmax(
            _ptr(logits), T, E, topk, float(routed_scale), block_m, _ptr(topk_ids),
            _ptr(topk_weights), _ptr(sorted_token_ids), _ptr(sorted_weights),
            _ptr(expert_ids), _ptr(num_tokens_post_pad), _ptr(workspace), workspace.numel(),
            _stream_handle(stream))
    _check(rc, "moe_route_sort_softmax")


def route_sort_softmax(logits, topk, routed_scale, block_m,
                       out: Optional[RouteSortBuffers] = None, stream=None) -> RouteSortBuffers:
    """Allocate (unless ``out`` is given) and run moe_route_sort_softmax."""
    T, E = logits.shape
    if out is None:
        out = RouteSortBuffers.allocate(T, E, topk, block_m, device=logits.device)
    moe_route_sort_softmax(logits, topk, routed_scale, block_m, out.topk_ids, out.topk_weights,
                           out.sorted_token_ids, out.sorted_weights, out.expert_ids,
                           out.num_tokens_post_pad, out.workspace, stream=stream)
    return out


def moe_gate_route_sort(hidden, w_gate, bias, n_group, topk_group, topk, routed_scale,
                        block_m, logits, topk_ids, topk_weights, sorted_token_ids,
                        sorted_weights, expert_ids, num_tokens_post_pad, workspace,
                        stream=None) -> None:
    """Gate projection (hidden [T,H] x w_gate [E,H]) into ``logits`` [T,E], then the whole
    path, into caller-owned buffers (see include/moe_route_sort.h)."""
    T, H = hidden.shape
    E = w_gate.shape[0]
    _need(hidden, torch.bfloat16, "hidden")
    _need(w_gate, torch.bfloat16, "w_gate")
    _need(bias, torch.float32, "bias")
    _need(logits, torch.bfloat16, "logits")
    if tuple(w_gate.shape) != (E, H) or tuple(logits.shape) != (T, E):
        raise ValueError("w_gate must be [E, H] and logits [T, E] for hidden [T, H]")
    for t, dt, n in [(topk_ids, torch.int32, "topk_ids"), (topk_weights, torch.float32,
                     "topk_weights"), (sorted_token_ids, torch.int32, "sorted_token_ids"),
                     (sorted_weights, torch.float32, "sorted_weights"),
                     (expert_ids, torch.int32, "expert_ids"),
                     (num_tokens_post_pad, torch.int32, "num_tokens_post_pad"),
                     (workspace, torch.uint8, "workspace")]:
        _need(t, dt, n)
    _need_room(T, topk, *_sort_sizes(T, E, topk, block_m), topk_ids=topk_ids,
               topk_weights=topk_weights, sorted_token_ids=sorted_token_ids,
               sorted_weights=sorted_weights, expert_ids=expert_ids,
               num_tokens_post_pad=num_tokens_post_pad)
    dev = _one_device(hidden, w_gate, bias, logits, topk_ids, topk_weights, sorted_token_ids,
                      sorted_weights, expert_ids, num_tokens_post_pad, workspace)
    with torch.cuda.device(dev):
        rc = load().moe_gate_route_sort(
            _ptr(hidden), _ptr(w_gate), _ptr(bias), T, E, H, n_group, topk_group, topk,
            float(routed_scale), block_m, _ptr(logits), _ptr(topk_ids), _ptr(topk_weights),
            _ptr(sorted_token_ids), _ptr(sorted_weights), _ptr(expert_ids),
            _ptr(num_tokens_post_pad), _ptr(workspace), workspace.numel(),
            _stream_handle(stream))
    _check(rc, "moe_gate_route_sort")


def gate_route_sort(hidden, w_gate, bias, n_group, topk_group, topk, routed_scale, block_m,
                    out: Optional[RouteSortBuffers] = None, logits=None, stream=None):
    """Allocate (unless given) and run moe_gate_route_sort; returns (logits, buffers)."""
    T = hidden.shape[0]
    E = w_gate.shape[0]
    if out is None:
        out = RouteSortBuffers.allocate(T, E, topk, block_m, device=hidden.device)
    if logits is None:
        logits = torch.empty(T, E, dtype=torch.bfloat16, device=hidden.device)
    moe_gate_route_sort(hidden, w_gate, bias, n_group, topk_group, topk, routed_scale, block_m,
                        logits, out.topk_ids, out.topk_weights, out.sorted_token_ids,
                        out.sorted_weights, out.expert_ids, out.num_tokens_post_pad,
                        out.workspace, stream=stream)
    return logits, out


def moe_route_sort_noalloc(logits, bias, n_group, topk_group, topk, routed_scale, block_m,
                           topk_ids, topk_weights, sorted_token_ids, sorted_weights, expert_ids,
                           num_tokens_post_pad, stream=None) -> None:
    """moe_route_sort with the library's own static scratch (no workspace, no allocation).

    For callers that cannot provide or allocate scratch memory; see include/moe_route_sort.h.
    Calls that may overlap on the GPU share that scratch and must not be issued.
    """
    T, E = logits.shape
    _need(logits, torch.bfloat16, "logits")
    _need(bias, torch.float32, "bias")
    for t, dt, n in [(topk_ids, torch.int32, "topk_ids"), (topk_weights, torch.float32,
                     "topk_weights"), (sorted_token_ids, torch.int32, "sorted_token_ids"),
                     (sorted_weights, torch.float32, "sorted_weights"),
                     (expert_ids, torch.int32, "expert_ids"),
                     (num_tokens_post_pad, torch.int32, "num_tokens_post_pad")]:
        _need(t, dt, n)
    _need_room(T, topk, *_sort_sizes(T, E, topk, block_m), topk_ids=topk_ids,
               topk_weights=topk_weights, sorted_token_ids=sorted_token_ids,
               sorted_weights=sorted_weights, expert_ids=expert_ids,
               num_tokens_post_pad=num_tokens_post_pad)
    dev = _one_device(logits, bias, topk_ids, topk_weights, sorted_token_ids, sorted_weights,
                      expert_ids, num_tokens_post_pad)
    with torch.cuda.device(dev):
        rc = load().moe_route_sort_noalloc(
            _ptr(logits), _ptr(bias), T, E, n_group, topk_group, topk, float(routed_scale),
            block_m, _ptr(topk_ids), _ptr(topk_weights), _ptr(sorted_token_ids),
            _ptr(sorted_weights), _ptr(expert_ids), _ptr(num_tokens_post_pad),
            _stream_handle(stream))
    _check(rc, "moe_route_sort_noalloc")


def moe_route_sort_noalloc_status(dst, stream=None) -> None:
    """Copy the device status word of the last moe_route_sort_noalloc call on dst's device
    into dst[0] (an int32 CUDA tensor), enqueued on the stream."""
    _need(dst, torch.int32, "dst")
    dev = _one_device(dst)
    with torch.cuda.device(dev):
        rc = load().moe_route_sort_noalloc_status(_ptr(dst), _stream_handle(stream))
    _check(rc, "moe_route_sort_noalloc_status")


def moe_topk(logits, bias, n_group, topk_group, topk, routed_scale, topk_ids, topk_weights,
             stream=None) -> None:
    T, E = logits.shape
    _need(logits, torch.bfloat16, "logits")
    _need(bias, torch.float32, "bias")
    _need(topk_ids, torch.int32, "topk_ids")
    _need(topk_weights, torch.float32, "topk_weights")
    _need_room(T, topk, 0, 0, topk_ids=topk_ids, topk_weights=topk_weights)
    dev = _one_device(logits, bias, topk_ids, topk_weights)
    with torch.cuda.device(dev):
        rc = load().moe_topk(_ptr(logits), _ptr(bias), T, E, n_group, topk_group, topk,
                             float(routed_scale), _ptr(topk_ids), _ptr(topk_weights),
                             _stream_handle(stream))
    _check(rc, "moe_topk")


def moe_sort(topk_ids, topk_weights, E, block_m, sorted_token_ids, sorted_weights, expert_ids,
             num_tokens_post_pad, workspace, stream=None, atomic=False) -> None:
    """Sort step only.  ``atomic=True`` calls moe_sort_atomic (order inside each expert's
    segment unspecified; see include/moe_route_sort.h)."""
    T, K = topk_ids.shape
    _need(topk_ids, torch.int32, "topk_ids")
    _need(topk_weights, torch.float32, "topk_weights")
    _need(sorted_token_ids, torch.int32, "sorted_token_ids")
    _need(sorted_weights, torch.float32, "sorted_weights")
    _need(expert_ids, torch.int32, "expert_ids")
    _need(num_tokens_post_pad, torch.int32, "num_tokens_post_pad")
    _need(workspace, torch.uint8, "workspace")
    if topk_weights.numel() < T * K:
        raise ValueError("topk_weights must hold T * topk weights")
    _need_room(T, K, *_sort_sizes(T, E, K, block_m), sorted_token_ids=sorted_token_ids,
               sorted_weights=sorted_weights, expert_ids=expert_ids,
               num_tokens_post_pad=num_tokens_post_pad)
    fn = load().moe_sort_atomic if atomic else load().moe_sort
    dev = _one_device(topk_ids, topk_weights, sorted_token_ids, sorted_weights, expert_ids,
                      num_tokens_post_pad, workspace)
    with torch.cuda.device(dev):
        rc = fn(_ptr(topk_ids), _ptr(topk_weights), T, E, K, block_m, _ptr(sorted_token_ids),
                _ptr(sorted_weights), _ptr(expert_ids), _ptr(num_tokens_post_pad),
                _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check(rc, "moe_sort_atomic" if atomic else "moe_sort")


def moe_route_sort_proxy_selftest(out2, stream=None) -> None:
    """Largest |cheap sigmoid - exact sigmoid| over all bf16 inputs -> out2[0]; bound -> out2[1]."""
    _need(out2, torch.float32, "out2")
    if out2.numel() < 2:
        raise ValueError("out2 needs 2 floats")
    with torch.cuda.device(_one_device(out2)):
        rc = load().moe_route_sort_proxy_selftest(_ptr(out2), _stream_handle(stream))
    _check(rc, "moe_route_sort_proxy_selftest")


def moe_route_sort_proxy_state(dst, stream=None) -> None:
    """The library's record of its proxy-bound check on dst's device into dst[0] (int32):
    0 not checked yet, 1 bound holds (pruning), 2 bound failed (exact keys everywhere)."""
    _need(dst, torch.int32, "dst")
    with torch.cuda.device(_one_device(dst)):
        rc = load().moe_route_sort_proxy_state(_ptr(dst), _stream_handle(stream))
    _check(rc, "moe_route_sort_proxy_state")


DEBUG_WAIT_LIMIT_NS = 1
DEBUG_FORCE_PROXY_FAIL = 2
DEBUG_CLUSTER_TOKENS = 3
DEBUG_GRID_TOKENS = 4
DEBUG_WARP_GRID_TOKENS = 5


def moe_route_sort_debug_set(knob: int, value: int) -> None:
    """Test hook of the library (see include/moe_route_sort.h): process-wide."""
    _check(load().moe_route_sort_debug_set(int(knob), int(value)), "moe_route_sort_debug_set")


# ---------------------------------------------------------- convenience buffers
@dataclass
class RouteSortBuffers:
    """Caller-owned output buffers plus workspace for one (T, E, topk, block_m) shape.

    ``allocate`` places the six outputs in one contiguous device block (``outputs``, bytes),
    so a caller can bring every result to the host with a single copy."""

    topk_ids: torch.Tensor
    topk_weights: torch.Tensor
    sorted_token_ids: torch.Tensor
    sorted_weights: torch.Tensor
    expert_ids: torch.Tensor
    num_tokens_post_pad: torch.Tensor
    workspace: torch.Tensor
    outputs: Optional[torch.Tensor] = None
    host_alias: Optional[int] = None  # device address of `outputs` when it is pinned host memory
    shape: Optional[tuple] = None  # (T, E, topk, block_m) the buffers were allocated for

    @classmethod
    def allocate(cls, T, E, topk, block_m, device="cuda") -> "RouteSortBuffers":
        P = max(moe_sort_max_padded(T, E, topk, block_m), 1)
        NB = max(moe_sort_max_blocks(T, E, topk, block_m), 1)
        ws = moe_route_sort_workspace_bytes(T, E, topk, block_m)
        if ws == 0:
            raise ValueError("invalid shape for route-sort buffers")
        parts = [("topk_ids", torch.int32, (T, topk)), ("topk_weights", torch.float32, (T, topk)),
                 ("sorted_token_ids", torch.int32, (P,)), ("sorted_weights", torch.float32, (P,)),
                 ("expert_ids", torch.int32, (NB,)), ("num_tokens_post_pad", torch.int32, (1,))]
        offs, total = [], 0
        for _, _, shape in parts:
            n = 4
            for d in shape:
                n *= d
            offs.append((total, n))
            total += (n + 15) // 16 * 16
        block = torch.empty(max(total, 16), dtype=torch.uint8, device=device)
        views = {name: block[o:o + n].view(dt).view(shape)
                 for (name, dt, shape), (o, n) in zip(parts, offs)}
        return cls(workspace=torch.empty(ws, dtype=torch.uint8, device=device), outputs=block,
                   shape=(T, E, topk, block_m), **views)

    @classmethod
    def allocate_pinned(cls, T, E, topk, block_m) -> "RouteSortBuffers":
        """Like ``allocate``, but the outputs block is pinned host memory mapped into the
        device's address space (zero-copy): the kernels write the results straight to the host.
        The workspace stays in device memory."""
        dev = cls.allocate(T, E, topk, block_m, device="cuda")
        block = torch.empty(dev.outputs.numel(), dtype=torch.uint8, pin_memory=True)
        base = dev.outputs.data_ptr()
        views = {}
        for name in ("topk_ids", "topk_weights", "sorted_token_ids", "sorted_weights",
                     "expert_ids", "num_tokens_post_pad"):
            t = getattr(dev, name)
            o = t.data_ptr() - base
            views[name] = block[o:o + t.numel() * 4].view(t.dtype).view(t.shape)
        return cls(workspace=dev.workspace, outputs=block, host_alias=map_host(block),
                   shape=dev.shape, **views)

    def addr(self, t: torch.Tensor) -> int:
        """Device address of one of the output views."""
        if self.host_alias is None:
            return t.data_ptr()
        return self.host_alias + (t.data_ptr() - self.outputs.data_ptr())

    def status_word(self) -> int:
        """Device status bits of the last completed call (synchronises the device)."""
        return int(self.workspace[:4].view(torch.int32).item())


def route_sort_from_host(logits_host, logits_dev, bias, n_group, topk_group, topk,
                         routed_scale, block_m, out: RouteSortBuffers, result_host,
                         stream=None) -> RouteSortBuffers:
    """moe_route_sort_from_host: copy the host logits in, run, copy every output back.

    ``logits_host`` is a pinned CPU bf16 tensor [T, E]; ``logits_dev`` a device tensor of the
    same shape that receives it; ``out`` buffers from ``RouteSortBuffers.allocate``, whose
    ``outputs`` block is copied into ``result_host`` (pinned CPU uint8, same size).  All of
    it is enqueued on the stream; the host copy is valid once the stream reaches its end."""
    T, E = logits_host.shape
    if logits_host.is_cuda or logits_host.dtype != torch.bfloat16:
        raise ValueError("logits_host must be a CPU bf16 tensor")
    if not logits_host.is_contiguous() or tuple(logits_dev.shape) != (T, E):
        raise ValueError("logits_host must be contiguous and match logits_dev")
    _need(logits_dev, torch.bfloat16, "logits_dev")
    _need(bias, torch.float32, "bias")
    if out.outputs is None or result_host.is_cuda or result_host.numel() != out.outputs.numel():
        raise ValueError("out must come from RouteSortBuffers.allocate; result_host must be a "
                         "CPU tensor of out.outputs' size")
    dev = _one_device(logits_dev, bias, out.outputs, out.workspace)
    with torch.cuda.device(dev):
        rc = load().moe_route_sort_from_host(
            logits_host.data_ptr(), logits_dev.data_ptr(), bias.data_ptr(), T, E, n_group,
            topk_group, topk, float(routed_scale), block_m, out.topk_ids.data_ptr(),
            out.topk_weights.data_ptr(), out.sorted_token_ids.data_ptr(),
            out.sorted_weights.data_ptr(), out.expert_ids.data_ptr(),
            out.num_tokens_post_pad.data_ptr(), out.workspace.data_ptr(),
            out.workspace.numel(), out.outputs.data_ptr(), result_host.data_ptr(),
            out.outputs.numel(), _stream_handle(stream))
    _check(rc, "moe_route_sort_from_host")
    return out


def map_host(t: torch.Tensor) -> int:
    """Device address of a pinned CPU tensor's memory (moe_route_sort_map_host)."""
    if t.is_cuda or not t.is_pinned():
        raise ValueError("map_host needs a pinned CPU tensor")
    d = ctypes.c_void_p()
    _check(load().moe_route_sort_map_host(t.data_ptr(), ctypes.byref(d)), "moe_route_sort_map_host")
    return int(d.value)


def route_sort_mapped(logits_addr: int, T: int, E: int, bias, n_group, topk_group, topk,
                      routed_scale, block_m, out: RouteSortBuffers, stream=None):
    """moe_route_sort with the logits at device address ``logits_addr`` (for example the
    ``map_host`` address of pinned host logits) and the outputs of ``out`` (device buffers, or
    pinned host buffers from ``RouteSortBuffers.allocate_pinned``): zero-copy when host."""
    _need(bias, torch.float32, "bias")
    _need_room(T, topk, *_sort_sizes(T, E, topk, block_m), topk_ids=out.topk_ids,
               topk_weights=out.topk_weights, sorted_token_ids=out.sorted_token_ids,
               sorted_weights=out.sorted_weights, expert_ids=out.expert_ids,
               num_tokens_post_pad=out.num_tokens_post_pad)
    dev = _one_device(bias, out.workspace)
    with torch.cuda.device(dev):
        rc = load().moe_route_sort(
            logits_addr, bias.data_ptr(), T, E, n_group, topk_group, topk,
            float(routed_scale), block_m, out.addr(out.topk_ids), out.addr(out.topk_weights),
            out.addr(out.sorted_token_ids), out.addr(out.sorted_weights),
            out.addr(out.expert_ids), out.addr(out.num_tokens_post_pad),
            out.workspace.data_ptr(), out.workspace.numel(), _stream_handle(stream))
    _check(rc, "moe_route_sort")
    return out


def route_sort(logits, bias, n_group, topk_group, topk, routed_scale, block_m,
               out: Optional[RouteSortBuffers] = None, stream=None) -> RouteSortBuffers:
    """Allocate (unless ``out`` is given) and run moe_route_sort; returns the buffers."""
    T, E = logits.shape
    if out is None:
        out = RouteSortBuffers.allocate(T, E, topk, block_m, device=logits.device)
    if out.outputs is None or out.shape != (T, E, topk, block_m) or out.host_alias is not None:
        moe_route_sort(logits, bias, n_group, topk_group, topk, routed_scale, block_m,
                       out.topk_ids, out.topk_weights, out.sorted_token_ids, out.sorted_weights,
                       out.expert_ids, out.num_tokens_post_pad, out.workspace, stream=stream)
        return out
    # buffers from allocate() have the right types and layout: check the inputs only
    _need(logits, torch.bfloat16, "logits")
    _need(bias, torch.float32, "bias")
    dev = _one_device(logits, bias, out.outputs, out.workspace)
    with torch.cuda.device(dev):
        rc = load().moe_route_sort(
            logits.data_ptr(), bias.data_ptr(), T, E, n_group, topk_group, topk,
            float(routed_scale), block_m, out.topk_ids.data_ptr(), out.topk_weights.data_ptr(),
            out.sorted_token_ids.data_ptr(), out.sorted_weights.data_ptr(),
            out.expert_ids.data_ptr(), out.num_tokens_post_pad.data_ptr(),
            out.workspace.data_ptr(), out.workspace.numel(), _stream_handle(stream))
    _check(rc, "moe_route_sort")
    return out
