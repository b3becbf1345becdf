"""The C ABI library builds, loads without a GPU, exports every declared
symbol, and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_softmax_gb300 as sv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specv.h")
FAKE = ctypes.c_void_p(0x10000)     # never dereferenced: every case fails host validation


@pytest.fixture(scope="module")
def L():
    sv.build()
    return sv.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(spec_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_exported_calls():
    assert sorted(sv.EXPORTED) == declared_functions()


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_workspace_sizes(L):
    assert L.spec_verify_workspace_bytes(64, 16, 131072, sv.BF16) > 0
    assert L.spec_verify_workspace_bytes(0, 16, 131072, sv.BF16) > 0
    assert L.spec_verify_workspace_bytes(4097, 16, 1024, sv.BF16) == 0
    assert L.spec_verify_workspace_bytes(4, 33, 1024, sv.BF16) == 0
    assert L.spec_verify_workspace_bytes(4, 4, 0, sv.F32) == 0
    assert L.spec_verify_workspace_bytes(4, 4, 10, 7) == 0
    assert L.spec_schedule_workspace_bytes(64, 16) >= 4


def _verify(L, B=4, gamma=4, V=1024, dt=sv.F32, target=FAKE, draft=FAKE, tokens=FAKE, vl=None,
            T=1.0, uniforms=FAKE, out_t=FAKE, out_n=FAKE, ws=FAKE, ws_bytes=1 << 40):
    return L.spec_verify(target, draft, dt, B, gamma, V, tokens, vl, ctypes.c_float(T), uniforms,
                         out_t, out_n, ws, ws_bytes, None)


def test_host_errors(L):
    assert _verify(L, B=-1) == sv.ERR_SHAPE
    assert _verify(L, B=4097) == sv.ERR_SHAPE
    assert _verify(L, gamma=33) == sv.ERR_SHAPE
    assert _verify(L, V=0) == sv.ERR_SHAPE
    assert _verify(L, dt=3) == sv.ERR_SHAPE
    assert _verify(L, T=-1.0) == sv.ERR_TEMPERATURE
    assert _verify(L, T=float("nan")) == sv.ERR_TEMPERATURE
    assert _verify(L, T=1e-5) == sv.ERR_TEMPERATURE
    assert _verify(L, T=2e4) == sv.ERR_TEMPERATURE
    assert _verify(L, target=None) == sv.ERR_NULL
    assert _verify(L, draft=None) == sv.ERR_NULL
    assert _verify(L, uniforms=None) == sv.ERR_NULL
    assert _verify(L, tokens=None) == sv.ERR_NULL
    assert _verify(L, ws=None) == sv.ERR_NULL
    assert _verify(L, target=ctypes.c_void_p(0x10001)) == sv.ERR_ALIGN
    assert _verify(L, dt=sv.BF16, target=ctypes.c_void_p(0x10001)) == sv.ERR_ALIGN
    assert _verify(L, dt=sv.BF16, target=ctypes.c_void_p(0x10002), ws_bytes=16) == sv.ERR_WORKSPACE
    assert _verify(L, ws=ctypes.c_void_p(0x10008)) == sv.ERR_ALIGN
    assert _verify(L, out_n=ctypes.c_void_p(0x10002)) == sv.ERR_ALIGN
    assert _verify(L, ws_bytes=16) == sv.ERR_WORKSPACE


def test_empty_batch_is_a_no_op(L):
    assert _verify(L, B=0, target=None, draft=None, tokens=None, uniforms=None, out_t=None, out_n=None,
                   ws=None) == sv.OK


def test_greedy_needs_no_draft_or_uniforms(L):
    # T == 0 with NULL draft / uniforms passes host validation up to the workspace check
    assert _verify(L, T=0.0, draft=None, uniforms=None, ws_bytes=16) == sv.ERR_WORKSPACE


def test_schedule_host_errors(L):
    table = sv.CostTable.from_knots([0.0, 512.0, 513.0], [8.0, 18.24, 20.0])

    def sched(B=4, gamma=4, cost=table, min_len=0, mode=0, conf=FAKE, out=FAKE, ws=FAKE, ws_bytes=256):
        return L.spec_schedule(conf, B, gamma, ctypes.byref(cost) if cost is not None else None,
                               min_len, mode, None, out, ws, ws_bytes, None)

    assert sched(B=-1) == sv.ERR_SHAPE
    assert sched(min_len=5) == sv.ERR_SHAPE
    assert sched(B=4096, gamma=32) == sv.ERR_SHAPE         # more than 16384 candidates
    assert sched(mode=3) == sv.ERR_SHAPE
    assert sched(mode=2) == sv.ERR_COST_TABLE                # knots 512 and 513 are not ratios in (0, 1]
    assert sched(cost=None) == sv.ERR_NULL
    assert sched(cost=sv.CostTable.from_knots([1.0, 1.0], [1.0, 2.0])) == sv.ERR_COST_TABLE
    assert sched(cost=sv.CostTable.from_knots([0.0, 1.0], [1.0, 0.0])) == sv.ERR_COST_TABLE
    assert sched(cost=sv.CostTable.from_knots([], [])) == sv.ERR_COST_TABLE
    assert sched(ws_bytes=8) == sv.ERR_WORKSPACE
    assert sched(ws=ctypes.c_void_p(0x10004)) == sv.ERR_ALIGN
    assert sched(B=0, conf=None, out=None, ws=None) == sv.OK


def test_schedule_static_host_errors(L):
    T = (ctypes.c_float * 4)(1.0, 0.5, 2.0, 1.0)
    Tbad = (ctypes.c_float * 4)(1.0, 0.0, 2.0, 1.0)

    def st(B=4, gamma=4, th=0.5, max_len=4, min_len=0, sts=None, conf=FAKE, out=FAKE, ws=FAKE, ws_bytes=256):
        return L.spec_schedule_static(conf, B, gamma, ctypes.c_float(th), max_len, min_len, sts, out, ws,
                                      ws_bytes, None)

    assert st(B=-1) == sv.ERR_SHAPE
    assert st(max_len=5) == sv.ERR_SHAPE
    assert st(min_len=3, max_len=2) == sv.ERR_SHAPE
    assert st(th=float("nan")) == sv.ERR_SHAPE
    assert st(sts=Tbad) == sv.ERR_SHAPE
    assert st(conf=None) == sv.ERR_NULL
    assert st(ws=ctypes.c_void_p(0x10004)) == sv.ERR_ALIGN
    assert st(sts=T, ws_bytes=8) == sv.ERR_WORKSPACE
    assert st(B=0, conf=None, out=None, ws=None) == sv.OK


def test_schedule_rejects_bad_temperatures(L):
    table = sv.CostTable.from_knots([0.0, 512.0], [8.0, 18.24])
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        T = (ctypes.c_float * 4)(1.0, 1.0, bad, 1.0)
        assert L.spec_schedule(FAKE, 4, 4, ctypes.byref(table), 0, 0, T, FAKE, FAKE, 256, None) == sv.ERR_SHAPE


def test_verify_packed_host_errors(L):
    def vp(B=4, gamma=4, V=1024, Kt=20, Kd=16, trow=FAKE, drow=FAKE, T=1.0, ws_bytes=1 << 40, **kw):
        return L.spec_verify_packed(kw.get("target", FAKE), Kt, kw.get("draft", FAKE), Kd, trow, drow, sv.F32, B,
                                    gamma, V, FAKE, None, ctypes.c_float(T), FAKE, FAKE, FAKE, FAKE, ws_bytes, None)

    assert vp(Kt=-1) == sv.ERR_SHAPE
    assert vp(trow=None) == sv.ERR_NULL
    assert vp(drow=None) == sv.ERR_NULL
    assert vp(drow=None, T=0.0, ws_bytes=16) == sv.ERR_WORKSPACE     # greedy reads no draft rows
    assert vp(trow=ctypes.c_void_p(0x10002)) == sv.ERR_ALIGN
    assert vp(B=4097) == sv.ERR_SHAPE
    assert vp(ws_bytes=16) == sv.ERR_WORKSPACE
    assert vp(B=0, trow=None, drow=None, target=None, draft=None) == sv.OK


def test_pack_rows_host_errors(L):
    assert L.spec_pack_rows(FAKE, 4097, 4, FAKE, FAKE, FAKE, None) == sv.ERR_SHAPE
    assert L.spec_pack_rows(FAKE, 4, 33, FAKE, FAKE, FAKE, None) == sv.ERR_SHAPE
    assert L.spec_pack_rows(None, 4, 4, FAKE, FAKE, FAKE, None) == sv.ERR_NULL
    assert L.spec_pack_rows(FAKE, 4, 4, FAKE, FAKE, None, None) == sv.ERR_NULL
    assert L.spec_pack_rows(FAKE, 4, 4, ctypes.c_void_p(0x10001), FAKE, FAKE, None) == sv.ERR_ALIGN


def test_selftest_wait_host_errors(L):
    assert L.spec_selftest_wait(10, FAKE, FAKE, None) == sv.ERR_SHAPE
    assert L.spec_selftest_wait(10 ** 10, FAKE, FAKE, None) == sv.ERR_SHAPE
    assert L.spec_selftest_wait(10 ** 6, None, FAKE, None) == sv.ERR_NULL
    assert L.spec_selftest_wait(10 ** 6, FAKE, ctypes.c_void_p(0x10004), None) == sv.ERR_ALIGN


def test_status_strings(L):
    for code in range(-14, 1):
        assert sv.status_string(code) and "unknown" not in sv.status_string(code)
    assert "unknown" in sv.status_string(-99)


def test_kernel_count(L):
    assert sv.kernel_count(0, 1.0) == 0
    assert sv.kernel_count(4, 0.0) == 2
    assert sv.kernel_count(4, 1.0) == 2
