"""The C ABI without a GPU: the library builds and loads, exports every symbol
include/lc.h declares, and rejects bad shapes on the host."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from kv_cache_compaction_gb300 import build as b
    b.build()
    import kv_cache_compaction_gb300 as lc
    return lc.load_library()


def declared_symbols():
    with open(os.path.join(ROOT, "include", "lc.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:lc_status|const char\*)\s+(lc_\w+)\(", text, re.M)))


def test_header_declares_the_entry_points():
    syms = declared_symbols()
    for name in ("lc_compact_layer", "lc_full_attn_stats", "lc_fit_only", "lc_key_scores",
                 "lc_select_topt", "lc_workspace_bytes", "lc_get_report"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    import kv_cache_compaction_gb300 as lc
    syms = declared_symbols()
    missing = [s for s in syms if not hasattr(lib, s)]
    assert not missing, missing
    assert sorted(lc.EXPORTS) == syms


def _shape(**kw):
    import kv_cache_compaction_gb300 as lc
    base = dict(n_kv_heads=8, n_q=32768, T=8192, d=128, t=256, in_dtype=0, scale=0.0,
                nnls_max_iter=0)
    base.update(kw)
    return lc.Shape(**base)


@pytest.mark.parametrize("kw,code", [
    ({}, 0),
    ({"d": 96}, 2),
    ({"t": 8193}, 1),
    ({"t": 2048, "T": 4096}, 2),
    ({"t": 0}, 1),
    ({"T": 0}, 1),
    ({"n_q": 0}, 1),
    ({"in_dtype": 1}, 2),          # fp32 needs d = 64
    ({"in_dtype": 1, "d": 64}, 0),
    ({"in_dtype": 7}, 1),
    ({"scale": -1.0}, 1),
    ({"scale": float("nan")}, 1),
    ({"n_kv_heads": 0}, 1),
    ({"n_kv_heads": 5000}, 1),
])
def test_workspace_query_validates_shape(lib, kw, code):
    n = ctypes.c_size_t(0)
    s = _shape(**kw)
    assert lib.lc_workspace_bytes(ctypes.byref(s), ctypes.byref(n)) == code
    if code == 0:
        assert n.value > 0


def test_workspace_grows_with_the_problem(lib):
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    s1, s2 = _shape(), _shape(T=16384, n_q=65536)
    lib.lc_workspace_bytes(ctypes.byref(s1), ctypes.byref(a))
    lib.lc_workspace_bytes(ctypes.byref(s2), ctypes.byref(b))
    assert b.value > a.value
    h = ctypes.c_size_t()
    lib.lc_host_workspace_bytes(ctypes.byref(s1), ctypes.byref(h))
    assert h.value > a.value


def test_null_handle_and_status_strings(lib):
    s = _shape()
    assert lib.lc_compact_layer(None, ctypes.byref(s), None, None, None, None, None, None, None,
                                None, 0, None) != 0
    assert lib.lc_status_string(0) == b"ok"
    for code in range(8):
        assert lib.lc_status_string(code)
    assert lib.lc_destroy(None) == 1


@pytest.mark.parametrize("kw,n_sub,k,code", [
    ({}, 256, 4, 0),
    ({}, 32768, 1, 0),
    ({}, 0, 4, 1),                 # empty query subset
    ({}, 32769, 4, 1),             # more subset rows than queries
    ({}, 256, 0, 1),
    ({"in_dtype": 1, "d": 64}, 256, 4, 2),   # fp32 inputs: bf16 only
    ({"d": 96}, 256, 4, 2),
    ({"t": 0}, 256, 4, 1),
])
def test_fast_workspace_query_validates(lib, kw, n_sub, k, code):
    n = ctypes.c_size_t(0)
    s = _shape(**kw)
    assert lib.lc_fast_workspace_bytes(ctypes.byref(s), n_sub, k, ctypes.byref(n)) == code
    if code == 0:
        assert n.value > 0


def test_fast_workspace_grows_with_the_shortlist(lib):
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    s = _shape()
    lib.lc_fast_workspace_bytes(ctypes.byref(s), 256, 1, ctypes.byref(a))
    lib.lc_fast_workspace_bytes(ctypes.byref(s), 256, 8, ctypes.byref(b))
    assert b.value > a.value
    # k t beyond T caps the shortlist at T
    c8, c64 = ctypes.c_size_t(), ctypes.c_size_t()
    lib.lc_fast_workspace_bytes(ctypes.byref(s), 256, 32, ctypes.byref(c8))
    lib.lc_fast_workspace_bytes(ctypes.byref(s), 256, 64, ctypes.byref(c64))
    assert c8.value == c64.value


def test_compact_attention_validates_before_any_device_work(lib):
    vp = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    args = dict(n_heads=2, n=4, t=3, n_new=0, d=128)

    def call(**kw):
        a = dict(args, **kw)
        return lib.lc_compact_attention(None, a["n_heads"], a["n"], a["t"], a["n_new"], a["d"],
                                        ctypes.c_float(kw.get("scale", 0.0)), vp, vp, vp, vp,
                                        None, None, None, vp, None, None)
    assert call(n=0) == 1
    assert call(n_heads=0) == 1
    assert call(t=-1) == 1
    assert call(n_new=2) == 1          # appended tokens without Knew / Vnew
    assert call(d=96) == 2
    assert call(scale=float("nan")) == 1
    assert call() == 1                 # valid arguments, null handle


def test_heldout_workspace_query(lib):
    n = ctypes.c_size_t(0)
    s = _shape(n_q=4096)
    assert lib.lc_heldout_workspace_bytes(ctypes.byref(s), ctypes.byref(n)) == 0
    base = ctypes.c_size_t(0)
    lib.lc_workspace_bytes(ctypes.byref(s), ctypes.byref(base))
    assert n.value > base.value
    s = _shape(in_dtype=1, d=64)
    assert lib.lc_heldout_workspace_bytes(ctypes.byref(s), ctypes.byref(n)) == 2


def test_farthest_first_validates(lib):
    vp = ctypes.c_void_p(16)  # never dereferenced: validation fails first

    def call(H=2, T=100, d=128, n_seed=2, M=10, out=vp):
        return lib.lc_farthest_first(None, H, T, d, vp, vp, n_seed, M, out, None)
    assert call(n_seed=0) == 1
    assert call(M=1) == 1          # fewer keys in all than seeds
    assert call(M=101) == 1        # more than T
    assert call(d=96) == 2
    assert call(out=None) == 1
    assert call(M=2, out=None) == 0  # nothing to add: no device work at all
    assert call() == 1               # valid arguments, null handle


def test_baseline_workspace_query(lib):
    n, base = ctypes.c_size_t(0), ctypes.c_size_t(0)
    s = _shape()
    assert lib.lc_baseline_workspace_bytes(ctypes.byref(s), ctypes.byref(n)) == 0
    lib.lc_workspace_bytes(ctypes.byref(s), ctypes.byref(base))
    assert n.value > base.value
    s = _shape(in_dtype=1, d=64)
    assert lib.lc_baseline_workspace_bytes(ctypes.byref(s), ctypes.byref(n)) == 2


def test_layers_workspace_query(lib):
    one, two = ctypes.c_size_t(0), ctypes.c_size_t(0)
    s = _shape()
    assert lib.lc_layers_workspace_bytes(ctypes.byref(s), 1, ctypes.byref(one)) == 0
    assert lib.lc_layers_workspace_bytes(ctypes.byref(s), 36, ctypes.byref(two)) == 0
    assert two.value == 2 * one.value
    assert lib.lc_layers_workspace_bytes(ctypes.byref(s), 0, ctypes.byref(one)) == 1
