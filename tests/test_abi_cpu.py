"""The C-ABI library on a machine without a GPU: it loads, exports every
symbol the header declares, and rejects bad arguments on the host before
touching the device."""
import ctypes
import os
import re

import pytest

from mixture_experts_atomic_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


def _lib():
    try:
        return B.lib()
    except RuntimeError as e:  # not built yet in this checkout
        import __graft_entry__
        __graft_entry__.build()
        return B.lib()


def _declared_functions():
    names = []
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            txt = open(os.path.join(HEADER_DIR, fn)).read()
            names += re.findall(r"MOEBLAZE_API\s+[\w\s\*]+?\b(moeblaze_\w+)\s*\(", txt)
    return names


def test_library_exports_every_declared_symbol():
    lib = _lib()
    declared = _declared_functions()
    assert len(declared) >= 13
    for n in declared:
        assert hasattr(lib, n), n
    assert sorted(declared) == sorted(B.EXPORTS)
    assert lib.moeblaze_version() == 10000


def test_status_strings():
    _lib()
    for st in range(7):
        assert B.status_string(st)
    assert "workspace" in B.status_string(B.ERR_WORKSPACE)


FAKE = ctypes.c_void_p(0x100000)      # aligned, never dereferenced: validation fails first
MISALIGNED = ctypes.c_void_p(0x100004)


def _disp():
    return B.Dispatch(0x100000, 0x100000, 0x100000, 0x100000, 0x100000)


def test_sizes_and_shape_validation():
    _lib()
    s = B.make_shape(512, 64, 128, 8, 2, B.F32, "swiglu")
    assert B.moeblaze_dispatch_meta_bytes(s) > 0
    rows = (1024 + 8 * 255 + 255) // 256 * 256   # L*K plus 255 padding rows per expert
    assert B.moeblaze_saved_bytes(s) == 2 * rows * 128 * 4
    bad = [
        B.make_shape(512, 64, 128, 2, 3, B.F32, "swiglu"),        # K > E
        B.make_shape(-1, 64, 128, 8, 2, B.F32, "swiglu"),         # L < 0
        B.make_shape(512, 64, 128, 8, 2, 7, "swiglu"),            # dtype
        B.make_shape(512, 64, 128, 8, 2, B.F32, 9),               # act
    ]
    for sh in bad:
        assert B.moeblaze_saved_bytes(sh) == 0
        st = B.moeblaze_dispatch_build(sh, FAKE, _disp(), FAKE, 1 << 30, 0, None)
        assert st == B.ERR_INVALID_ARG
    unsup = [
        B.make_shape(512, 96, 128, 8, 2, B.BF16, "swiglu"),       # bf16 needs d % 128 == 0
        B.make_shape(512, 128, 200, 8, 2, B.BF16, "silu"),        # and h % 128 == 0
        B.make_shape(512, 128, 128, 600, 2, B.BF16, "swiglu"),    # E > 512
        B.make_shape(512, 128, 128, 16, 9, B.BF16, "swiglu"),     # K > 8
        B.make_shape(1 << 30, 128, 128, 16, 4, B.BF16, "swiglu"), # L*K >= 2^31
    ]
    for sh in unsup:
        st = B.moeblaze_forward(sh, FAKE, FAKE, _disp(), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None)
        assert st == B.ERR_UNSUPPORTED


def test_pointer_and_workspace_validation():
    _lib()
    s = B.make_shape(4096, 128, 256, 8, 2, B.BF16, "swiglu")
    need = B.moeblaze_dispatch_workspace_bytes(s)
    assert B.moeblaze_dispatch_build(s, None, _disp(), FAKE, need, 0, None) == B.ERR_INVALID_ARG
    assert B.moeblaze_dispatch_build(s, MISALIGNED, _disp(), FAKE, need, 0, None) == B.ERR_INVALID_ARG
    assert B.moeblaze_dispatch_build(s, FAKE, _disp(), FAKE, need - 1, 0, None) == B.ERR_WORKSPACE
    d = _disp()
    d.meta = None
    assert B.moeblaze_dispatch_build(s, FAKE, d, FAKE, need, 0, None) == B.ERR_INVALID_ARG
    fw = B.moeblaze_forward_workspace_bytes(s)
    # missing W2 for SwiGLU
    assert B.moeblaze_forward(s, FAKE, FAKE, _disp(), FAKE, None, FAKE, FAKE, FAKE, FAKE, fw, None) == B.ERR_INVALID_ARG
    assert B.moeblaze_forward(s, FAKE, FAKE, _disp(), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, fw - 1, None) == B.ERR_WORKSPACE
    bw = B.moeblaze_backward_workspace_bytes(s)
    assert B.moeblaze_backward(s, FAKE, FAKE, FAKE, _disp(), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None,
                               FAKE, bw, None) == B.ERR_INVALID_ARG
    assert B.moeblaze_backward(s, FAKE, FAKE, FAKE, _disp(), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                               FAKE, bw - 1, None) == B.ERR_WORKSPACE
    # a misaligned dgates pointer is rejected
    assert B.moeblaze_backward(s, FAKE, FAKE, FAKE, _disp(), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                               MISALIGNED, FAKE, bw, None) == B.ERR_INVALID_ARG
    # SiLU takes no W2 / dW2
    s2 = B.make_shape(4096, 128, 256, 8, 2, B.BF16, "silu")
    assert B.moeblaze_saved_bytes(s2) * 2 == B.moeblaze_saved_bytes(s)
    # identity needs no weights and no scratch
    s3 = B.make_shape(4096, 128, 0, 8, 2, B.BF16, "identity")
    assert B.moeblaze_saved_bytes(s3) == 0 and B.moeblaze_forward_workspace_bytes(s3) == 0


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        B.lib()


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "mixture_experts_atomic_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in txt and "from oracle" not in txt, fn


def test_router_validation_codes():
    _lib()
    ok = B.make_shape(4096, 1024, 0, 8, 2, B.BF16, "silu")
    ws = B.moeblaze_router_backward_workspace_bytes(ok)
    assert ws > 0
    # more than 256 experts, d not a multiple of 64: unsupported
    for bad in (B.make_shape(4096, 1024, 0, 300, 2, B.BF16, "silu"), B.make_shape(4096, 96, 0, 8, 2, B.BF16, "silu")):
        assert B.moeblaze_router_forward(bad, FAKE, FAKE, None, FAKE, FAKE, None) == B.ERR_UNSUPPORTED
        assert B.moeblaze_router_backward_workspace_bytes(bad) == 0
    # K > E, missing Wr, misaligned x, missing outputs: invalid
    assert B.moeblaze_router_forward(B.make_shape(16, 64, 0, 2, 3, B.F32, "silu"), FAKE, FAKE, None, FAKE, FAKE,
                                     None) == B.ERR_INVALID_ARG
    assert B.moeblaze_router_forward(ok, FAKE, None, None, FAKE, FAKE, None) == B.ERR_INVALID_ARG
    assert B.moeblaze_router_forward(ok, MISALIGNED, FAKE, None, FAKE, FAKE, None) == B.ERR_INVALID_ARG
    assert B.moeblaze_router_forward(ok, FAKE, FAKE, None, None, FAKE, None) == B.ERR_INVALID_ARG
    assert B.moeblaze_router_backward(ok, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE, ws, None) \
        == B.ERR_INVALID_ARG
    assert B.moeblaze_router_backward(ok, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, ws - 1, None) \
        == B.ERR_WORKSPACE


def test_dispatch_meta_check_compares_the_recorded_shape():
    """The comparison the forward/backward kernels make on the device header
    (words 3, 4, 5 = the L, E, K the build recorded), run on a host copy."""
    import struct
    _lib()
    s = B.make_shape(70000, 128, 128, 64, 6, B.BF16, "swiglu")

    def hdr(L, E, K):
        return ctypes.create_string_buffer(struct.pack("<8i", 0, 5, 640, L, E, K, 0, 0), 32)

    assert B.moeblaze_dispatch_meta_check(s, hdr(70000, 64, 6)) == B.OK
    for L, E, K in [(69999, 64, 6), (70000, 63, 6), (70000, 64, 5), (0, 0, 0)]:
        assert B.moeblaze_dispatch_meta_check(s, hdr(L, E, K)) == B.ERR_INVALID_ARG, (L, E, K)
    # a build for no tokens records only L = 0 and serves any L = 0 call
    s0 = B.make_shape(0, 128, 128, 64, 6, B.BF16, "swiglu")
    assert B.moeblaze_dispatch_meta_check(s0, hdr(0, 0, 0)) == B.OK
    assert B.moeblaze_dispatch_meta_check(s0, hdr(1, 64, 6)) == B.ERR_INVALID_ARG
    assert B.moeblaze_dispatch_meta_check(s, None) == B.ERR_INVALID_ARG


def test_recompute_flag_sizes_and_validation():
    """MOEBLAZE_RECOMPUTE_H drops H (padded_rows x h) from the forward
    scratch and Hg from the backward scratch of the bf16 expert layers, and
    keeps one fp32 gate per padded row in the saved buffer instead; fp32 and
    identity layers ignore it; unknown flag bits are refused."""
    _lib()
    for act in ("swiglu", "silu"):
        a = B.make_shape(70000, 256, 384, 16, 2, B.BF16, act)
        r = B.make_shape(70000, 256, 384, 16, 2, B.BF16, act, B.RECOMPUTE_H)
        rows = -(-(70000 * 2 + 255 * 16) // 256) * 256
        assert rows == B.padded_rows(a)
        h_bytes = -(-(rows * 384 * 2) // 256) * 256
        assert B.moeblaze_forward_workspace_bytes(a) - B.moeblaze_forward_workspace_bytes(r) == h_bytes
        assert B.moeblaze_backward_workspace_bytes(a) - B.moeblaze_backward_workspace_bytes(r) == h_bytes
        assert B.moeblaze_saved_bytes(r) - B.moeblaze_saved_bytes(a) == rows * 4
    for dt, act in ((B.F32, "swiglu"), (B.BF16, "identity")):
        a = B.make_shape(700, 64, 128, 8, 2, dt, act)
        r = B.make_shape(700, 64, 128, 8, 2, dt, act, B.RECOMPUTE_H)
        assert B.moeblaze_forward_workspace_bytes(a) == B.moeblaze_forward_workspace_bytes(r)
        assert B.moeblaze_backward_workspace_bytes(a) == B.moeblaze_backward_workspace_bytes(r)
    bad = B.make_shape(700, 128, 128, 8, 2, B.BF16, "swiglu", 2)
    assert B.moeblaze_saved_bytes(bad) == 0
    assert B.moeblaze_dispatch_build(bad, FAKE, _disp(), FAKE, 1 << 30, 0, None) == B.ERR_INVALID_ARG


def test_bf16_backward_scratch_has_no_gradient_buffer():
    """The bf16 backward writes dA and dB over the saved A and B: its scratch
    is Hg (rows x h) and the fp32 dX accumulator (L x d) plus 256 bytes of
    tile counters; the fp32 layer keeps its own dA|dB buffer."""
    _lib()
    L, d, h, E, K = 5000, 256, 384, 8, 2
    s = B.make_shape(L, d, h, E, K, B.BF16, "swiglu")
    rows = B.padded_rows(s)
    up = lambda n: -(-n // 256) * 256
    assert B.moeblaze_backward_workspace_bytes(s) == up(rows * h * 2) + up(L * d * 4) + 256
    f = B.make_shape(L, d, h, E, K, B.F32, "swiglu")
    assert B.moeblaze_backward_workspace_bytes(f) == up(rows * 2 * h * 4) + up(rows * h * 4)


def test_router_dispatch_validation_codes():
    """moeblaze_router_dispatch_build: both the dispatch's and the router's
    shape rules apply, and its scratch holds the dispatch's plus, on the
    fused path (bf16 x, <= 64 experts, >= 128 tokens), the split router
    weights (3 x 8 rows of d bf16, rounded up to 16 rows, for <= 8 experts)."""
    _lib()
    ok = B.make_shape(4096, 1024, 1024, 8, 2, B.BF16, "silu")
    n = B.moeblaze_router_dispatch_workspace_bytes(ok)
    split = 32 * 1024 * 2
    assert n == B.moeblaze_dispatch_workspace_bytes(ok) + split
    # the unfused shapes need only the dispatch's scratch
    for sh in (B.make_shape(4096, 1024, 1024, 8, 2, B.F32, "silu"),      # fp32 x
               B.make_shape(4096, 1024, 1024, 100, 2, B.BF16, "silu"),   # more than 64 experts
               B.make_shape(100, 1024, 1024, 8, 2, B.BF16, "silu")):     # fewer than 128 tokens
        assert B.moeblaze_router_dispatch_workspace_bytes(sh) == B.moeblaze_dispatch_workspace_bytes(sh)
    # router limits (E > 256) and dispatch limits (bf16 d % 128) both refuse
    assert B.moeblaze_router_dispatch_workspace_bytes(B.make_shape(4096, 1024, 1024, 300, 2, B.BF16, "silu")) == 0
    assert B.moeblaze_router_dispatch_workspace_bytes(B.make_shape(4096, 192, 1024, 8, 2, B.BF16, "silu")) == 0
    call = lambda sh, x=FAKE, Wr=FAKE, ids=FAKE, g=FAKE, d=None, ws=FAKE, nb=n: B.moeblaze_router_dispatch_build(
        sh, x, Wr, None, ids, g, _disp() if d is None else d, ws, nb, None)
    assert call(ok, nb=n - 1) == B.ERR_WORKSPACE
    assert call(ok, Wr=None) == B.ERR_INVALID_ARG
    assert call(ok, x=MISALIGNED) == B.ERR_INVALID_ARG
    assert call(ok, ids=None) == B.ERR_INVALID_ARG
    assert call(ok, ws=None) == B.ERR_INVALID_ARG
    d = _disp()
    d.meta = None
    assert call(ok, d=d) == B.ERR_INVALID_ARG
    assert call(B.make_shape(16, 128, 128, 2, 3, B.BF16, "silu")) == B.ERR_INVALID_ARG  # K > E
