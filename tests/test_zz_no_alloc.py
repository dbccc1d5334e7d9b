"""The allocation-free top-t select against the regular one.

Callers that cannot allocate device memory or hand the library a workspace
(for example code under a memory planner that forbids allocation on the
serving path) use lc_select_topt_noalloc, whose scratch is a fixed array
compiled into the library.  Its results must equal lc_select_topt's, call
after call.  This file is collected last, so a failure here leaves every
other test already run."""
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def _ptr(x):
    return ctypes.c_void_p(x.data_ptr())


def test_noalloc_select_equals_workspace_select():
    import torch
    from kv_cache_compaction_gb300 import build
    build.build()
    import kv_cache_compaction_gb300 as lc

    torch.cuda.set_device(0)
    lib = lc.load_library()
    comp = lc.Compactor(0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [
        (8, 8192, 256, synth.continuous_scores(8, 8192, 71)),
        (3, 1000, 333, synth.tie_heavy_scores(3, 1000, 72)),
    ]
    for H, T, t, u in cases:  # two calls in a row through the shared array
        ud = torch.from_numpy(np.ascontiguousarray(u, dtype=np.float32)).cuda()
        ref = comp.select_topt(ud, t)
        out = torch.full((H, t), -1, dtype=torch.int32, device="cuda")
        assert lib.lc_select_topt_noalloc(H, T, t, _ptr(ud), _ptr(out), stream) == 0
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    # beyond the fixed array: rejected before anything is enqueued
    small = torch.zeros((1, 8), dtype=torch.float32, device="cuda")
    idx = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    too_many = lc.load_library()
    assert too_many.lc_select_topt_noalloc(2, 1 << 20, 4, _ptr(small), _ptr(idx), stream) == 2
