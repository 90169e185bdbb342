"""The C-ABI library on a machine without a GPU: it loads, exports every
entry point include/mac.h declares, and its host-only logic (sizes,
configuration checks, argument checks) behaves.  No call here reaches CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def native():
    from kv_cache_computation_gb300 import build
    build.build()
    from kv_cache_computation_gb300 import _native
    return _native


def _declared():
    src = open(os.path.join(ROOT, "include", "mac.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mac_[a-z_]+)\s*\(", src)))


def test_every_declared_entry_point_is_exported(native):
    names = _declared()
    assert len(names) >= 19
    L = native.lib()
    for n in names:
        assert hasattr(L, n), f"{n} declared in mac.h but not exported"
    assert set(names) == set(native.SIGNATURES), "binding signatures out of step with mac.h"


def _cfg(native, **kw):
    from kv_cache_computation_gb300 import make_config
    base = dict(heads=32, kv_heads=8, head_dim=128, ring_len=16, band_r=64, tau=0.3, max_batch=1,
                max_ctx=131072, page_size=16)
    base.update(kw)
    return make_config(**base)


def _sizes(native, cfg):
    kv, ring, scr = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    st = native.lib().mac_query_sizes(ctypes.byref(cfg), ctypes.byref(kv), ctypes.byref(ring), ctypes.byref(scr))
    return st, kv.value, ring.value, scr.value


def test_kv_bytes_are_exact(native):
    st, kv, ring, scr = _sizes(native, _cfg(native))
    assert st == 0
    assert kv == 131072 * 8 * 128 * 2 * 2
    st, kv_c, _, _ = _sizes(native, _cfg(native, page_size=0, max_ctx=4097, max_batch=2))
    assert st == 0 and kv_c == 2 * 2 * 8 * 4112 * 128 * 2     # contiguous: rounded up to whole pages


def test_ring_layout_reproduces_table7():
    """Ring slot = bf16 q~ + fp32 o + fp32 lse per query head (772 B at d=128)
    plus an int32 position per request; at 128K context (8 KV heads) this is
    the auxiliary HBM overhead the paper's Table 7 reports."""
    from kv_cache_computation_gb300 import _native as native
    native_lib = native
    rows = [tuple(map(float, ln.split())) for ln in open(os.path.join(ROOT, "tests", "golden", "table7_aux_hbm.txt"))
            if ln.strip() and not ln.startswith("#")]
    st, kv, r32, _ = _sizes(native_lib, _cfg(native_lib, ring_len=32))
    st2, _, r64, _ = _sizes(native_lib, _cfg(native_lib, ring_len=64))
    assert st == 0 and st2 == 0
    per_slot = (r64 - r32) / 32
    # 772 B per query head; the per-request int32 position may vanish in the 256-B alignment
    assert 32 * 772 <= per_slot <= 32 * 772 + 4
    for K, pct in rows:
        got = 100.0 * K * per_slot / kv
        assert abs(got - pct) <= 0.1, (K, got, pct)


@pytest.mark.parametrize("bad", [dict(head_dim=64), dict(heads=24, kv_heads=8), dict(heads=30, kv_heads=8),
                                 dict(ring_len=0), dict(ring_len=4097), dict(band_r=0), dict(tau=-0.1),
                                 dict(tau=float("inf")), dict(max_batch=0), dict(max_ctx=0),
                                 dict(max_ctx=(1 << 30) + 1), dict(page_size=8), dict(plan_mode=2),
                                 dict(heads=64, kv_heads=1), dict(sm_scale=-1.0),
                                 dict(amend_band=2), dict(max_batch=129, kv_heads=8)])
def test_invalid_configs_are_rejected(native, bad):
    st, *_ = _sizes(native, _cfg(native, **bad))
    assert st == -1


def test_create_checks_buffers_before_touching_the_gpu(native):
    cfg = _cfg(native, max_ctx=1024)
    st, kv, ring, scr = _sizes(native, cfg)
    L = native.lib()
    h = ctypes.c_void_p()
    assert L.mac_create(ctypes.byref(cfg), None, kv, None, ring, None, scr, ctypes.byref(h)) == -1
    # misaligned and too-small buffers (never dereferenced)
    assert L.mac_create(ctypes.byref(cfg), ctypes.c_void_p(0x1000 + 8), kv, ctypes.c_void_p(0x2000), ring,
                        ctypes.c_void_p(0x3000), scr, ctypes.byref(h)) == -2
    assert L.mac_create(ctypes.byref(cfg), ctypes.c_void_p(0x1000), kv - 1, ctypes.c_void_p(0x2000), ring,
                        ctypes.c_void_p(0x3000), scr, ctypes.byref(h)) == -2
    assert L.mac_create(ctypes.byref(cfg), ctypes.c_void_p(0x1000), kv, ctypes.c_void_p(0x2000), ring,
                        ctypes.c_void_p(0x3000), scr, None) == -1


def test_null_handle_calls_fail_cleanly(native):
    L = native.lib()
    assert L.mac_decode_step(None, 1, None, None, None, None, None, None, None) == -1
    assert L.mac_decode_step_host(None, 1, None, None, None, None, None, None, None) == -1
    assert L.mac_sync(None, 0) == -1
    assert L.mac_destroy(None) == -1
    assert L.mac_last_error(None) == b""


def test_status_strings(native):
    L = native.lib()
    for code in range(0, -7, -1):
        s = L.mac_status_string(code)
        assert s and s != b"unknown status"
    assert L.mac_status_string(5) == b"unknown status"


def test_host_binding_refuses_what_the_kernels_cannot_address():
    """The host-buffer binding takes pinned CPU tensors only: pageable memory,
    a wrong dtype or shape is refused before anything reaches the library."""
    import torch
    from kv_cache_computation_gb300.attention import _host
    t = torch.zeros((2, 4, 128), dtype=torch.bfloat16)   # pageable
    with pytest.raises(TypeError, match="pinned"):
        _host(t, "q_pre", torch.bfloat16, (2, 4, 128))
    if torch.cuda.is_available():
        p = t.pin_memory()
        assert _host(p, "q_pre", torch.bfloat16, (2, 4, 128)).value == p.data_ptr()
        with pytest.raises(TypeError):
            _host(p, "q_pre", torch.float32)
        with pytest.raises(ValueError):
            _host(p, "q_pre", torch.bfloat16, (2, 4, 64))


def _struct_fields(name):
    """(type, field) pairs of the typedef struct `name` in include/mac.h."""
    src = open(os.path.join(ROOT, "include", "mac.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    body = re.search(r"typedef struct\s*\{([^}]*)\}\s*" + name + r"\s*;", src).group(1)
    return re.findall(r"\b(u?int\d+_t|int|float|double)\s+(\w+)\s*;", body)


@pytest.mark.parametrize("cname,pyname", [("mac_config", "MacConfig"), ("mac_stats", "MacStats"),
                                          ("mac_profile", "MacProfile")])
def test_binding_structs_match_the_header(native, cname, pyname):
    """The ctypes structures the binding passes to the library declare the
    header's fields in the header's order with the header's widths."""
    width = {"int": 4, "float": 4, "double": 8, "int32_t": 4, "uint32_t": 4, "int64_t": 8, "uint64_t": 8}
    hdr = _struct_fields(cname)
    py = getattr(native, pyname)._fields_
    assert [f for _, f in hdr] == [f for f, _ in py]
    assert [width[t] for t, _ in hdr] == [ctypes.sizeof(t) for _, t in py]
