"""The C-ABI library on the host: it loads, exports every declared symbol, answers size
queries, and rejects bad arguments before touching any device (no GPU needed)."""
import ctypes
import glob
import os
import re

import pytest
import torch

import moe_expert_routing_sort_gb300 as mrs
from moe_expert_routing_sort_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return mrs.load()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(moe_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"moe_route_sort", "moe_topk", "moe_sort"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_size_queries():
    assert mrs.moe_sort_max_padded(1, 896, 16, 32) == 16 + 16 * 31
    assert mrs.moe_sort_max_padded(16384, 4096, 8, 128) == 131072 + 4096 * 127
    assert mrs.moe_sort_max_blocks(1, 896, 16, 32) == (16 + 16 * 31) // 32
    assert mrs.moe_sort_max_padded(0, 64, 6, 16) == 0
    assert mrs.moe_sort_max_padded(4, 64, 6, 3) == 0  # block_m not a power of two
    for E in range(1, 4097, 37):
        assert mrs.moe_route_sort_workspace_bytes(512, E, 8, 64) >= 4 * E
    assert mrs.moe_route_sort_workspace_bytes(1, 0, 1, 1) == 0
    assert mrs.moe_route_sort_workspace_bytes(1, 4097, 1, 1) == 0
    assert mrs.moe_route_sort_workspace_bytes(16384, 4096, 8, 128) % 16 == 0


def test_strerror_covers_codes():
    for code in range(-16, 1):
        assert mrs.strerror(code) != "unknown status"
    assert mrs.strerror(-99) == "unknown status"


# Host-side validation runs before any CUDA call, so fake device addresses are safe here:
# every call below must be rejected without dereferencing anything.
BASE = 0x7F0000000000


def _route_sort(lib, T=4, E=64, G=8, Kg=4, K=6, R=2.5, B=16, logits=BASE, bias=BASE + 0x10000,
                ids=BASE + 0x20000, w=BASE + 0x30000, sid=BASE + 0x40000, sw=BASE + 0x80000,
                eid=BASE + 0xC0000, npp=BASE + 0xD0000, ws=BASE + 0x100000, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = mrs.moe_route_sort_workspace_bytes(max(T, 0), E, K, B) if E > 0 else 1 << 20
    return lib.moe_route_sort(logits, bias, T, E, G, Kg, K, R, B, ids, w, sid, sw, eid, npp, ws,
                              ws_bytes, None)


def test_route_sort_rejects_bad_shapes(lib):
    assert _route_sort(lib, E=0) == -2
    assert _route_sort(lib, E=4097) == -2
    assert _route_sort(lib, G=7) == -3  # 64 % 7 != 0
    assert _route_sort(lib, E=128, G=128, Kg=4, K=4) == -3  # more than 64 groups
    assert _route_sort(lib, Kg=9) == -3
    assert _route_sort(lib, Kg=0) == -3
    assert _route_sort(lib, K=0) == -4
    assert _route_sort(lib, K=33, E=256, G=1, Kg=1) == -4
    assert _route_sort(lib, K=33) == -4  # more than Kg * g = 32
    assert _route_sort(lib, B=3) == -5
    assert _route_sort(lib, B=2048) == -5
    assert _route_sort(lib, T=-1) == -6
    assert _route_sort(lib, T=(1 << 31) // 6 + 1) == -7
    assert _route_sort(lib, R=float("nan")) == -11
    assert _route_sort(lib, R=float("inf")) == -11


def test_route_sort_rejects_bad_buffers(lib):
    assert _route_sort(lib, logits=0) == -1
    assert _route_sort(lib, sid=0) == -1
    assert _route_sort(lib, ws=0) == -10
    assert _route_sort(lib, ws_bytes=16) == -10
    assert _route_sort(lib, logits=BASE + 8) == -8  # logits need 16-byte alignment
    assert _route_sort(lib, ids=BASE + 0x20002) == -8
    assert _route_sort(lib, ws=BASE + 0x100004) == -8
    assert _route_sort(lib, sw=BASE + 0x40000) == -9  # sorted weights over sorted ids
    assert _route_sort(lib, ids=BASE + 0x10) == -9  # topk ids over the logits
    assert _route_sort(lib, npp=BASE + 0x100010) == -9  # npp inside the workspace
    assert _route_sort(lib, eid=BASE + 0x10000) == -9  # expert ids over the bias


def test_moe_sort_and_topk_validate(lib):
    P = mrs.moe_sort_max_padded(4, 64, 6, 16)
    ws = mrs.moe_route_sort_workspace_bytes(4, 64, 6, 16)
    args = [BASE, BASE + 0x1000, 4, 64, 6, 16, BASE + 0x2000, BASE + 0x2000 + 4 * P,
            BASE + 0x8000, BASE + 0x9000, BASE + 0x10000, ws, None]
    bad = list(args)
    bad[5] = 12
    assert lib.moe_sort(*bad) == -5
    bad = list(args)
    bad[7] = BASE + 0x2000  # sorted weights over sorted ids
    assert lib.moe_sort(*bad) == -9
    bad = list(args)
    bad[11] = 8
    assert lib.moe_sort(*bad) == -10
    assert lib.moe_topk(BASE, BASE + 0x1000, 4, 64, 8, 4, 33, 1.0, BASE + 0x2000,
                        BASE + 0x3000, None) == -4
    assert lib.moe_topk(BASE + 2, BASE + 0x1000, 4, 64, 8, 4, 6, 1.0, BASE + 0x2000,
                        BASE + 0x3000, None) == -8
    # T == 0 needs no buffers for moe_topk and launches nothing
    assert lib.moe_topk(0, 0, 0, 64, 8, 4, 6, 1.0, 0, 0, None) == 0


def _from_host(lib, logits_host=BASE + 0x200000, logits_dev=BASE, result_dev=BASE + 0x300000,
               result_host=BASE + 0x400000, result_bytes=64):
    ws_bytes = mrs.moe_route_sort_workspace_bytes(4, 64, 6, 16)
    return lib.moe_route_sort_from_host(
        logits_host, logits_dev, BASE + 0x10000, 4, 64, 8, 4, 6, 2.5, 16, BASE + 0x20000,
        BASE + 0x30000, BASE + 0x40000, BASE + 0x80000, BASE + 0xC0000, BASE + 0xD0000,
        BASE + 0x100000, ws_bytes, result_dev, result_host, result_bytes, None)


def test_from_host_rejects_missing_copy_pointers(lib):
    # checked before anything is enqueued: no pointer is dereferenced
    assert _from_host(lib, logits_host=None) == -1
    assert _from_host(lib, logits_dev=None) == -1
    assert _from_host(lib, result_dev=None) == -1
    assert _from_host(lib, result_host=None) == -1


def _from_host_full(lib, B=16, ws=BASE + 0x100000, ws_bytes=None, logits_dev=BASE,
                    ids=BASE + 0x20000):
    if ws_bytes is None:
        ws_bytes = mrs.moe_route_sort_workspace_bytes(4, 64, 6, 16)
    return lib.moe_route_sort_from_host(
        BASE + 0x200000, logits_dev, BASE + 0x10000, 4, 64, 8, 4, 6, 2.5, B, ids,
        BASE + 0x30000, BASE + 0x40000, BASE + 0x80000, BASE + 0xC0000, BASE + 0xD0000, ws,
        ws_bytes, BASE + 0x300000, BASE + 0x400000, 64, None)


def test_from_host_checks_everything_before_the_copy(lib):
    # Every check of moe_route_sort runs before the host-to-device copy is enqueued.  With fake
    # addresses (and no GPU here) an enqueued copy would fail with the launch status -12, so
    # each specific status below also shows that nothing was enqueued first.
    assert _from_host_full(lib, B=12) == -5                       # bad block_m
    assert _from_host_full(lib, ws_bytes=16) == -10               # short workspace
    assert _from_host_full(lib, ws=0) == -10                      # no workspace
    assert _from_host_full(lib, logits_dev=BASE + 8) == -8        # misaligned device logits
    assert _from_host_full(lib, logits_dev=BASE + 0x100000) == -9  # device logits over workspace
    assert _from_host_full(lib, logits_dev=BASE + 0x40000) == -9   # over sorted_token_ids
    assert _from_host_full(lib, ids=BASE + 0x10) == -9             # topk ids over device logits


def test_noalloc_checks_shapes_first(lib):
    # a shape the library rejects gets its own status, before the scratch size check and the
    # device address lookup (which would give -12 here, with no GPU)
    args = [BASE, BASE + 0x100000, 600000, 4096, 16, 4, 8, 1.0, 128, BASE + 0x200000,
            BASE + 0x300000, BASE + 0x400000, BASE + 0x500000, BASE + 0x600000,
            BASE + 0x700000, None]
    for i, v, code in [(8, 3, -5), (3, 0, -2), (3, 4097, -2), (4, 7, -3), (6, 0, -4),
                       (2, -1, -6), (7, float("nan"), -11)]:
        bad = list(args)
        bad[i] = v
        assert lib.moe_route_sort_noalloc(*bad) == code, (i, v, code)
    assert lib.moe_route_sort_noalloc(*args) == -13  # valid shape, too large for the scratch


def test_state_accessors_validate(lib):
    assert lib.moe_route_sort_noalloc_status(None, None) == -1
    assert lib.moe_route_sort_noalloc_status(BASE + 2, None) == -8
    assert lib.moe_route_sort_proxy_state(None, None) == -1
    assert lib.moe_route_sort_proxy_state(BASE + 1, None) == -8


def test_debug_knobs(lib):
    assert lib.moe_route_sort_debug_set(99, 0) == -16
    assert lib.moe_route_sort_debug_set(0, 0) == -16
    assert lib.moe_route_sort_debug_set(1, 0) == 0   # wait limit 0 ...
    assert lib.moe_route_sort_debug_set(1, -1) == 0  # ... and back to the default
    assert lib.moe_route_sort_debug_set(2, 1) == 0   # forced proxy failure ...
    assert lib.moe_route_sort_debug_set(2, 0) == 0   # ... and back to the real check
    assert lib.moe_route_sort_debug_set(3, 0) == 0   # cluster path off ...
    assert lib.moe_route_sort_debug_set(3, -1) == 0  # ... and back to the default
    assert lib.moe_route_sort_debug_set(4, 0) == 0   # per-token grid path off ...
    assert lib.moe_route_sort_debug_set(4, -1) == 0  # ... and back to the default
    assert lib.moe_route_sort_debug_set(5, 1 << 30) == 0  # warp-per-token grid path off ...
    assert lib.moe_route_sort_debug_set(5, -1) == 0       # ... and back to the default


def test_binding_refuses_buffers_on_different_devices():
    # the library runs on one device and reads every pointer there: the binding refuses a mix
    from moe_expert_routing_sort_gb300 import binding
    with pytest.raises(ValueError, match="one device"):
        binding._one_device(torch.empty(1), torch.empty(1, device="meta"))
    with pytest.raises(ValueError, match="CUDA"):
        binding._one_device(torch.empty(1), None, torch.empty(2))


def _softmax(lib, T=4, E=64, K=6, R=1.0, B=16, logits=BASE, ids=BASE + 0x20000,
             ws=BASE + 0x100000, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = mrs.moe_route_sort_workspace_bytes(max(T, 0), E, K, B) if E > 0 else 1 << 20
    return lib.moe_route_sort_softmax(logits, T, E, K, R, B, ids, BASE + 0x30000,
                                      BASE + 0x40000, BASE + 0x80000, BASE + 0xC0000,
                                      BASE + 0xD0000, ws, ws_bytes, None)


def test_softmax_variant_validates(lib):
    # no groups: K is bounded by E itself (and by 32)
    assert _softmax(lib, E=0) == -2
    assert _softmax(lib, E=5, K=6) == -4
    assert _softmax(lib, E=256, K=33) == -4
    assert _softmax(lib, K=0) == -4
    assert _softmax(lib, B=24) == -5
    assert _softmax(lib, T=-3) == -6
    assert _softmax(lib, R=float("nan")) == -11
    assert _softmax(lib, logits=0) == -1
    assert _softmax(lib, logits=BASE + 4) == -8
    assert _softmax(lib, ws_bytes=16) == -10
    assert _softmax(lib, ids=BASE + 0x30000) == -9  # topk ids over topk weights


def _gate(lib, T=2, E=64, H=256, hidden=BASE + 0x200000, w_gate=BASE + 0x210000,
          logits=BASE + 0x300000, ids=BASE + 0x20000, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = mrs.moe_route_sort_workspace_bytes(max(T, 0), E, 6, 16)
    return lib.moe_gate_route_sort(hidden, w_gate, BASE + 0x10000, T, E, H, 8, 4, 6, 2.5, 16,
                                   logits, ids, BASE + 0x30000, BASE + 0x40000, BASE + 0x80000,
                                   BASE + 0xC0000, BASE + 0xD0000, BASE + 0x100000, ws_bytes,
                                   None)


def test_gate_variant_validates(lib):
    assert _gate(lib, T=9) == -6       # at most 8 tokens
    assert _gate(lib, H=7) == -14
    assert _gate(lib, H=0) == -14
    assert _gate(lib, H=8200) == -14
    assert _gate(lib, hidden=0) == -1
    assert _gate(lib, logits=0) == -1
    assert _gate(lib, w_gate=BASE + 0x210008) == -8
    assert _gate(lib, logits=BASE + 0x300002) == -8
    assert _gate(lib, hidden=BASE + 0x300000) == -9  # hidden over the logits output
    assert _gate(lib, w_gate=BASE + 0x100000) == -9  # gate rows over the workspace
    assert _gate(lib, ids=BASE + 0x300010) == -9     # topk ids over the logits
    assert _gate(lib, logits=BASE + 0x10000) == -9   # the gate's logits over the bias
    assert _gate(lib, ws_bytes=16) == -10


def test_map_host_rejects_null(lib):
    d = ctypes.c_void_p()
    assert lib.moe_route_sort_map_host(None, ctypes.byref(d)) == -1
    assert lib.moe_route_sort_map_host(BASE, None) == -1


def test_moe_sort_atomic_validates(lib):
    # same contract as moe_sort: checked before the memset or any launch
    P = mrs.moe_sort_max_padded(4, 64, 6, 16)
    ws = mrs.moe_route_sort_workspace_bytes(4, 64, 6, 16)
    args = [BASE, BASE + 0x1000, 4, 64, 6, 16, BASE + 0x2000, BASE + 0x2000 + 4 * P,
            BASE + 0x8000, BASE + 0x9000, BASE + 0x10000, ws, None]
    for i, v, code in [(5, 12, -5), (3, 0, -2), (4, 33, -4), (2, -1, -6),
                       (7, BASE + 0x2000, -9), (11, 8, -10), (10, 0, -10), (0, 0, -1),
                       (6, BASE + 0x2002, -8)]:
        bad = list(args)
        bad[i] = v
        assert lib.moe_sort_atomic(*bad) == code, (i, v, code)


def test_binding_rejects_undersized_outputs(lib):
    # the Python binding checks buffer sizes against the shape before calling the library
    from moe_expert_routing_sort_gb300 import binding
    T, E, K, B = 5, 64, 6, 16
    P, NB = binding._sort_sizes(T, E, K, B)
    assert (P, NB) == (mrs.moe_sort_max_padded(T, E, K, B), mrs.moe_sort_max_blocks(T, E, K, B))
    ok = dict(topk_ids=torch.empty(T * K), topk_weights=torch.empty(T * K),
              sorted_token_ids=torch.empty(P), sorted_weights=torch.empty(P),
              expert_ids=torch.empty(NB), num_tokens_post_pad=torch.empty(1))
    binding._need_room(T, K, P, NB, **ok)
    for name in ok:
        bad = dict(ok)
        bad[name] = torch.empty(max(ok[name].numel() - 1, 0))
        with pytest.raises(ValueError, match=name):
            binding._need_room(T, K, P, NB, **bad)
    binding._need_room(0, K, 0, 0, topk_ids=torch.empty(0), num_tokens_post_pad=torch.empty(1))
    b = mrs.RouteSortBuffers.allocate(T, E, K, B, device="cpu")
    assert b.shape == (T, E, K, B)
    binding._need_room(T, K, P, NB, topk_ids=b.topk_ids, topk_weights=b.topk_weights,
                       sorted_token_ids=b.sorted_token_ids, sorted_weights=b.sorted_weights,
                       expert_ids=b.expert_ids, num_tokens_post_pad=b.num_tokens_post_pad)


def test_header_is_plain_c(tmp_path):
    # the C ABI header compiles as C99 (no C++ or torch types leak into the signatures)
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    cuda_inc = "/usr/local/cuda/include"
    if gcc is None or not os.path.isdir(cuda_inc):
        pytest.skip("gcc or the CUDA headers are not available")
    src = tmp_path / "use.c"
    src.write_text('#include "moe_route_sort.h"\nint main(void) { return MOE_RS_OK; }\n')
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
