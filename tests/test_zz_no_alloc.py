"""moeblaze_dispatch_build_static: the dispatch build for callers that cannot
allocate device memory (for example a runtime that only hands over input and
output buffers from a fixed, fully claimed pool).  It keeps its scratch in a
fixed array inside the library instead of a caller-provided workspace.

These checks call it through the C ABI and compare its outputs with those of
moeblaze_dispatch_build (caller scratch) on two calls in a row, so the second
call runs on scratch that still holds the first call's contents.  Index
structures are integers: the comparison is bit-exact.  This file is
collected last so that a run stopping at the first failure has already run
every other test."""
import ctypes

import pytest
import torch

from mixture_experts_atomic_gb300 import binding as B
from mixture_experts_atomic_gb300 import inputs as I


def test_static_scratch_limit_is_checked_on_the_host():
    B.lib()
    # the 2M-token, 256-expert dispatch needs ~36 MB of scratch: over the limit
    big = B.make_shape(2097152, 128, 0, 256, 4, B.BF16, "identity")
    assert B.moeblaze_dispatch_workspace_bytes(big) > B.STATIC_SCRATCH_BYTES
    fake = 0x100000
    d = B.Dispatch(fake, fake, fake, fake, fake)
    st = B.moeblaze_dispatch_build_static(big, ctypes.c_void_p(fake), d, 0, None)
    assert st == B.ERR_WORKSPACE


def _compare(shape, ids_dev, validate):
    ref = B.alloc_dispatch(shape, "cuda")
    B.dispatch_build(shape, ids_dev, ref)               # caller-provided scratch
    out = B.alloc_dispatch(shape, "cuda")
    st = B.moeblaze_dispatch_build_static(shape, ctypes.c_void_p(ids_dev.data_ptr()), out.struct(), validate,
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == B.OK, B.status_string(st)
    torch.cuda.synchronize()
    for a, b in zip(B.index_views(shape, ref), B.index_views(shape, out)):
        assert torch.equal(a, b)
    ra, rb = B.meta_arrays(shape, ref), B.meta_arrays(shape, out)
    assert ra[0] == rb[0]
    for a, b in zip(ra[1:], rb[1:]):
        assert torch.equal(a, b)
    mt = B.meta_arrays(shape, out)[0]
    E = shape.E
    tiles_ref = ref.meta.view(torch.int32)[8 + 3 * E + 1:8 + 3 * E + 1 + mt]
    tiles_out = out.meta.view(torch.int32)[8 + 3 * E + 1:8 + 3 * E + 1 + mt]
    assert torch.equal(tiles_ref, tiles_out)
    assert B.device_error(shape, out) == 0


@pytest.mark.gpu
def test_static_scratch_dispatch_matches_caller_scratch_twice():
    try:
        B.lib()
    except RuntimeError:
        import __graft_entry__
        __graft_entry__.build()
    assert torch.cuda.is_available()
    # first call: a skewed 6-of-64 routing; second call: a different shape and
    # contents on the same (now dirty) scratch, with validation on
    ids1, _ = I.random_routing(70000, 64, 6, 21, one_expert=5)
    s1 = B.make_shape(70000, 128, 128, 64, 6, B.BF16, "swiglu")
    _compare(s1, ids1.cuda(), validate=0)
    ids2, _ = I.random_routing(16384, 8, 2, 22)
    s2 = B.make_shape(16384, 1024, 4096, 8, 2, B.BF16, "silu")
    _compare(s2, ids2.cuda(), validate=1)
    # third call: larger than the first, so it reads scratch words neither
    # earlier call wrote; L is not a multiple of the 1024-token chunk, so its
    # last chunk is partial
    ids3, _ = I.random_routing(200001, 64, 6, 23, one_expert=63)
    s3 = B.make_shape(200001, 128, 128, 64, 6, B.BF16, "swiglu")
    assert B.moeblaze_dispatch_workspace_bytes(s3) > B.moeblaze_dispatch_workspace_bytes(s1)
    assert B.moeblaze_dispatch_workspace_bytes(s3) <= B.STATIC_SCRATCH_BYTES
    _compare(s3, ids3.cuda(), validate=1)
    # and a small ragged case after it: 1537 tokens, 3 experts, K = 3
    ids4, _ = I.random_routing(1537, 3, 3, 24)
    _compare(B.make_shape(1537, 128, 128, 3, 3, B.BF16, "silu"), ids4.cuda(), validate=0)
