"""Host-side checks of the C ABI (no GPU): the library loads, exports every
function include/kda.h declares, and rejects bad arguments before launching
anything.  Fake, never-dereferenced pointer values are used: validation must
return before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def L():
    from kda_linear_attention_gb300 import build
    build.build()
    import kda_linear_attention_gb300 as kda
    return kda.lib()


def _declared_functions():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(HEADER_DIR, fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        for m in re.finditer(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\(", src):
            name = m.group(1)
            if name.startswith("kda_"):
                names.add(name)
    return names


def test_exports_every_declared_symbol(L):
    names = _declared_functions()
    assert {"kda_prefill_chunked", "kda_decode_step", "kda_version",
            "kda_status_string"} <= names
    for n in names:
        assert hasattr(L, n), "libkda_gb300.so does not export %s" % n


def test_version_and_status_strings(L):
    assert L.kda_version() >= 100
    for s in range(0, 9):
        assert len(L.kda_status_string(s)) > 0
        assert L.kda_status_string(s) != b"unknown status"
    assert L.kda_status_string(12345) == b"unknown status"


GOOD = ctypes.c_void_p(0x10000)   # aligned, never dereferenced


def _prefill(L, **kw):
    a = dict(q=GOOD, k=GOOD, v=GOOD, g=GOOD, beta=GOOD, S0=None, o=GOOD, S_out=GOOD, cu=GOOD,
             N=1, T=64, H=2, dk=128, dv=128, chunk=64, dtype=0, stream=None)
    a.update(kw)
    return L.kda_prefill_chunked(a["q"], a["k"], a["v"], a["g"], a["beta"], a["S0"], a["o"],
                                 a["S_out"], a["cu"], a["N"], a["T"], a["H"], a["dk"], a["dv"],
                                 a["chunk"], a["dtype"], a["stream"])


def _decode(L, **kw):
    a = dict(q=GOOD, k=GOOD, v=GOOD, g=GOOD, beta=GOOD, S=GOOD, o=GOOD, B=4, H=2, dk=128, dv=128,
             dtype=0, stream=None)
    a.update(kw)
    return L.kda_decode_step(a["q"], a["k"], a["v"], a["g"], a["beta"], a["S"], a["o"], a["B"],
                             a["H"], a["dk"], a["dv"], a["dtype"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=7), 5),
    (dict(dk=64), 2), (dict(dv=256), 2), (dict(N=0), 2), (dict(H=0), 2), (dict(T=-1), 2),
    (dict(T=1 << 31), 2),
    (dict(chunk=48), 3), (dict(chunk=128), 3), (dict(chunk=0), 3),
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(g=None), 1),
    (dict(beta=None), 1), (dict(o=None), 1), (dict(S_out=None), 1), (dict(cu=None), 1),
    (dict(q=ctypes.c_void_p(0x10004)), 4), (dict(S0=ctypes.c_void_p(0x10008)), 4),
    (dict(cu=ctypes.c_void_p(0x10002)), 4), (dict(o=ctypes.c_void_p(0x1000c)), 4),
])
def test_prefill_rejects_bad_arguments(L, kw, status):
    assert _prefill(L, **kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=-1), 5), (dict(dk=127), 2), (dict(H=0), 2), (dict(B=-3), 2),
    (dict(q=None), 1), (dict(S=None), 1), (dict(o=None), 1), (dict(beta=None), 1),
    (dict(S=ctypes.c_void_p(0x10004)), 4), (dict(v=ctypes.c_void_p(0x10001)), 4),
])
def test_decode_rejects_bad_arguments(L, kw, status):
    assert _decode(L, **kw) == status


@pytest.mark.parametrize("fn", ["kda_prefill_chunked_noalloc", "kda_prefill_chunked_events"])
@pytest.mark.parametrize("kw,status", [
    (dict(dk=64), 2), (dict(N=0), 2), (dict(q=None), 1), (dict(S_out=None), 1),
    (dict(q=ctypes.c_void_p(0x10004)), 4),
])
def test_prefill_variants_reject_bad_arguments(L, fn, kw, status):
    a = dict(q=GOOD, k=GOOD, v=GOOD, g=GOOD, beta=GOOD, S0=None, o=GOOD, S_out=GOOD, cu=GOOD,
             N=1, T=64, H=2, dk=128, dv=128, chunk=64, dtype=0, stream=None)
    a.update(kw)
    args = [a["q"], a["k"], a["v"], a["g"], a["beta"], a["S0"], a["o"], a["S_out"], a["cu"],
            a["N"], a["T"], a["H"], a["dk"], a["dv"], a["chunk"], a["dtype"], a["stream"]]
    if fn == "kda_prefill_chunked_events":
        evs = (ctypes.c_void_p * 4)(GOOD, GOOD, GOOD, GOOD)
        args.append(ctypes.cast(evs, ctypes.POINTER(ctypes.c_void_p)))
    assert getattr(L, fn)(*args) == status


def _prefill_ws(L, ws=GOOD, ws_bytes=None, **kw):
    a = dict(q=GOOD, k=GOOD, v=GOOD, g=GOOD, beta=GOOD, S0=None, o=GOOD, S_out=GOOD, cu=GOOD,
             N=1, T=64, H=2, dk=128, dv=128, chunk=64, dtype=0, stream=None)
    a.update(kw)
    if ws_bytes is None:
        ws_bytes = L.kda_prefill_workspace_bytes(a["N"], a["T"], a["H"], a["dk"], a["dv"],
                                                 a["chunk"], a["dtype"])
    return L.kda_prefill_chunked_ws(a["q"], a["k"], a["v"], a["g"], a["beta"], a["S0"], a["o"],
                                    a["S_out"], a["cu"], a["N"], a["T"], a["H"], a["dk"], a["dv"],
                                    a["chunk"], a["dtype"], ws, ctypes.c_size_t(ws_bytes),
                                    a["stream"])


def test_prefill_workspace_bytes(L):
    """The caller-owned workspace of the tensor-core path: the chunk offsets
    and a job counter (4 (N + 2) bytes) and the chunk table (8 bytes per
    chunk), each rounded up to 1 KB, then one 60,416-byte record per (chunk,
    head), with one spare chunk per sequence for a partial tail; no workspace
    for the CUDA-core path or for invalid sizes."""
    for N, T, H in [(1, 64, 2), (1, 4096, 96), (3, 130, 5), (300, 4096, 4), (255, 4096, 2)]:
        chunks = -(-T // 64) + N
        want = 1024 * (-(-4 * (N + 2) // 1024)) + 1024 * (-(-8 * chunks // 1024)) + chunks * H * 60416
        assert L.kda_prefill_workspace_bytes(N, T, H, 128, 128, 64, 0) == want
    assert L.kda_prefill_workspace_bytes(1, 64, 2, 128, 128, 64, 1) == 0    # fp32 inputs
    assert L.kda_prefill_workspace_bytes(1, 64, 2, 128, 128, 32, 0) == 0    # chunk 32
    assert L.kda_prefill_workspace_bytes(1, 0, 2, 128, 128, 64, 0) == 0     # no tokens
    assert L.kda_prefill_workspace_bytes(0, 64, 2, 128, 128, 64, 0) == 0    # no sequences
    assert L.kda_prefill_workspace_bytes(1, 64, 2, 64, 128, 64, 0) == 0     # unsupported dk


@pytest.mark.parametrize("kw,status", [
    (dict(dk=64), 2), (dict(N=0), 2), (dict(chunk=48), 3), (dict(dtype=7), 5),
    (dict(q=None), 1), (dict(S_out=None), 1), (dict(q=ctypes.c_void_p(0x10004)), 4),
    (dict(ws=None), 6),                                  # the tensor-core path needs one
    (dict(ws_bytes=1024), 6),                            # too small
    (dict(ws=ctypes.c_void_p(0x10010)), 4),              # not 256-byte aligned
])
def test_prefill_ws_rejects_bad_arguments(L, kw, status):
    assert _prefill_ws(L, **kw) == status


def test_prefill_events_needs_events_and_the_tensor_core_path(L):
    def call(evs, dtype=0, chunk=64):
        return L.kda_prefill_chunked_events(GOOD, GOOD, GOOD, GOOD, GOOD, None, GOOD, GOOD, GOOD,
                                            1, 64, 2, 128, 128, chunk, dtype, None, evs)
    assert call(None) == 1
    four = (ctypes.c_void_p * 4)(GOOD, GOOD, None, GOOD)
    assert call(ctypes.cast(four, ctypes.POINTER(ctypes.c_void_p))) == 1
    four = (ctypes.c_void_p * 4)(GOOD, GOOD, GOOD, GOOD)
    ptr = ctypes.cast(four, ctypes.POINTER(ctypes.c_void_p))
    assert call(ptr, dtype=1) == 3 and call(ptr, chunk=32) == 3


def test_decode_batch_zero_is_noop(L):
    # B = 0 returns before touching any pointer or the GPU
    assert _decode(L, B=0, q=None, S=None) == 0


def test_binding_fails_loudly_without_cuda_tensors():
    torch = pytest.importorskip("torch")
    import kda_linear_attention_gb300 as kda
    x = torch.zeros(4, 2, 128)
    with pytest.raises(ValueError):
        kda.decode_step(x, x, x, x, torch.zeros(4, 2), torch.zeros(4, 2, 128, 128))


def _prologue(L, **kw):
    a = dict(xq=GOOD, xk=GOOD, xv=GOOD, w=GOOD, cin=None, cout=GOOD, q=GOOD, k=GOOD, v=GOOD,
             cu=GOOD, N=1, T=64, H=2, d=128, qs=0.088, eps=1e-6, stream=None)
    a.update(kw)
    return L.kda_conv_prologue(a["xq"], a["xk"], a["xv"], a["w"], a["cin"], a["cout"], a["q"],
                               a["k"], a["v"], a["cu"], a["N"], a["T"], a["H"], a["d"], a["qs"],
                               a["eps"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(d=64), 2), (dict(N=0), 2), (dict(H=0), 2), (dict(T=-1), 2),
    (dict(eps=-1.0), 8), (dict(eps=float("nan")), 8), (dict(qs=float("inf")), 8),
    (dict(qs=float("nan")), 8), (dict(cin=GOOD, cout=GOOD), 8),
    (dict(xq=None), 1), (dict(w=None), 1), (dict(v=None), 1), (dict(cu=None), 1),
    (dict(xk=ctypes.c_void_p(0x10004)), 4), (dict(cout=ctypes.c_void_p(0x10002)), 4),
])
def test_prologue_rejects_bad_arguments(L, kw, status):
    assert _prologue(L, **kw) == status


def test_prologue_without_tokens_or_windows_is_noop(L):
    assert _prologue(L, T=0, cout=None, xq=None, q=None) == 0


def _gated(L, **kw):
    a = dict(q=GOOD, k=GOOD, v=GOOD, g=GOOD, beta=GOOD, S0=None, gate=GOOD, w=GOOD, eps=1e-6,
             out=GOOD, S_out=GOOD, cu=GOOD, N=1, T=64, H=2, dk=128, dv=128, chunk=64, dtype=0,
             stream=None)
    a.update(kw)
    return L.kda_prefill_chunked_gated(a["q"], a["k"], a["v"], a["g"], a["beta"], a["S0"],
                                       a["gate"], a["w"], a["eps"], a["out"], a["S_out"], a["cu"],
                                       a["N"], a["T"], a["H"], a["dk"], a["dv"], a["chunk"],
                                       a["dtype"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=3), 5), (dict(dk=64), 2), (dict(N=0), 2), (dict(chunk=8), 3),
    (dict(eps=-0.5), 8), (dict(gate=None), 1), (dict(w=None), 1), (dict(out=None), 1),
    (dict(S_out=None), 1), (dict(gate=ctypes.c_void_p(0x10006)), 4),
    (dict(w=ctypes.c_void_p(0x10004)), 4),
])
def test_gated_prefill_rejects_bad_arguments(L, kw, status):
    assert _gated(L, **kw) == status


def _layer_step(L, **kw):
    a = dict(xq=GOOD, xk=GOOD, xv=GOOD, w=GOOD, cp=GOOD, g=GOOD, beta=GOOD, gate=GOOD, nw=GOOD,
             S=GOOD, sdt=1, idx=None, P=4, out=GOOD, B=4, H=2, dk=128, dv=128, qs=0.088,
             l2=1e-6, ne=1e-6, stream=None)
    a.update(kw)
    return L.kda_decode_layer_step(a["xq"], a["xk"], a["xv"], a["w"], a["cp"], a["g"], a["beta"],
                                   a["gate"], a["nw"], a["S"], a["sdt"], a["idx"], a["P"],
                                   a["out"], a["B"], a["H"], a["dk"], a["dv"], a["qs"], a["l2"],
                                   a["ne"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(sdt=2), 5), (dict(dk=64), 2), (dict(H=0), 2), (dict(B=-1), 2), (dict(P=3), 2),
    (dict(l2=-1.0), 8), (dict(ne=float("nan")), 8), (dict(qs=float("-inf")), 8),
    (dict(cp=None), 1), (dict(gate=None), 1), (dict(nw=None), 1), (dict(S=None), 1),
    (dict(out=None), 1), (dict(cp=ctypes.c_void_p(0x10008)), 4),
    (dict(idx=ctypes.c_void_p(0x10004)), 4),
])
def test_decode_layer_rejects_bad_arguments(L, kw, status):
    assert _layer_step(L, **kw) == status


def test_decode_layer_with_slots_allows_small_pool_and_empty_batch(L):
    assert _layer_step(L, B=0, xq=None, S=None) == 0


def _layer_prefill(L, **kw):
    a = dict(xq=GOOD, xk=GOOD, xv=GOOD, w=GOOD, cin=None, cout=GOOD, g=GOOD, beta=GOOD, S0=None,
             gate=GOOD, nw=GOOD, qs=0.088, l2=1e-6, ne=1e-6, out=GOOD, S_out=GOOD, cu=GOOD, N=1,
             T=64, H=2, dk=128, dv=128, stream=None)
    a.update(kw)
    return L.kda_layer_prefill(a["xq"], a["xk"], a["xv"], a["w"], a["cin"], a["cout"], a["g"],
                               a["beta"], a["S0"], a["gate"], a["nw"], a["qs"], a["l2"], a["ne"],
                               a["out"], a["S_out"], a["cu"], a["N"], a["T"], a["H"], a["dk"],
                               a["dv"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(dk=64), 2), (dict(dv=256), 2), (dict(N=0), 2), (dict(H=0), 2), (dict(T=-1), 2),
    (dict(T=1 << 31), 2), (dict(l2=-1.0), 8), (dict(ne=float("nan")), 8),
    (dict(qs=float("inf")), 8), (dict(cin=GOOD, cout=GOOD), 8),
    (dict(xq=None), 1), (dict(w=None), 1), (dict(g=None), 1), (dict(gate=None), 1),
    (dict(nw=None), 1), (dict(out=None), 1), (dict(S_out=None), 1), (dict(cu=None), 1),
    (dict(xv=ctypes.c_void_p(0x10004)), 4), (dict(S0=ctypes.c_void_p(0x10008)), 4),
    (dict(cout=ctypes.c_void_p(0x10002)), 4),
])
def test_layer_prefill_rejects_bad_arguments(L, kw, status):
    assert _layer_prefill(L, **kw) == status
