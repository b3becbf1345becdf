"""Oracle: the plain fp64 CPU definition of speculative verification and of the
verify-length scheduler (``oracle.c``), with a ctypes wrapper.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code with
the CUDA library and the CUDA library never calls it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

# Per-request status values (the library's error-code numbers).
OK, ERR_SHAPE, ERR_TEMPERATURE, ERR_VERIFY_LEN, ERR_TOKEN = 0, -2, -4, -5, -6
ERR_COST_TABLE, ERR_NONFINITE, ERR_UNIFORM, ERR_CONFIDENCE = -8, -9, -12, -13
EV_RESIDUAL_EMPTY, EV_NO_BIN = 1, 2


def build(force: bool = False) -> str:
    """Compile oracle.c (gcc -O2, no FP contraction, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c99", "-ffp-contract=off",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _L():
    global _lib
    if _lib is not None:
        return _lib
    with _lock:  # the test helpers call the oracle from several host threads
        return _load()


def _load():
    global _lib
    if _lib is None:
        # A mutated copy of the oracle may be substituted (the pin-sensitivity
        # test plants mistakes in oracle.c and expects the pins to fail).
        alt = os.environ.get("SPECV_ORACLE_LIB")
        if alt:
            lib = ctypes.CDLL(alt)
        else:
            build()
            lib = ctypes.CDLL(_LIB)
        vp, i32, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.oracle_verify.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, dbl, vp, vp, vp,
                                      vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.oracle_verify_probs.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp, vp]
        lib.oracle_draw_cdf.argtypes = [vp, vp, i32, i32, i32, i32, vp, dbl, i32, i32, vp, i32, vp, vp]
        lib.oracle_cost_at.argtypes = [dbl, vp, vp, i32, vp]
        lib.oracle_sched_exact.argtypes = [vp, i32, i32, vp, vp, i32, i32, vp, vp, vp]
        lib.oracle_sched_alg1.argtypes = [vp, i32, i32, vp, vp, i32, i32, vp]
        lib.oracle_sched_brute.argtypes = [vp, i32, i32, vp, vp, i32, i32, vp, vp, vp]
        lib.oracle_set_sts.argtypes = [vp]
        lib.oracle_sched_dcut.argtypes = [vp, i32, i32, vp, vp, i32, i32, vp, vp, vp]
        lib.oracle_sched_threshold.argtypes = [vp, i32, i32, dbl, i32, i32, vp]
        lib.oracle_sts_ece.argtypes = [vp, vp, i32, i32, vp]
        lib.oracle_sts_fit.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp]
        for f in ("oracle_verify", "oracle_verify_probs", "oracle_draw_cdf", "oracle_cost_at", "oracle_sched_exact",
                  "oracle_sched_alg1", "oracle_sched_brute", "oracle_set_sts", "oracle_sched_dcut",
                  "oracle_sched_threshold", "oracle_sts_ece", "oracle_sts_fit"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def verify(target, draft, dtype: str, tokens, verify_len, T: float, uniforms, *,
           b0: int = 0, b1: int | None = None) -> dict:
    """Run the oracle on requests [b0, b1) of a batch.

    ``target``/``draft`` are the stored logits ([B, gamma+1, V] / [B, gamma, V];
    uint16 bf16 bits or float32).  ``T`` is the fp32 temperature widened to fp64.
    Returns the outputs and diagnostics as numpy arrays.
    """
    B_all, G1, V = target.shape
    gamma = G1 - 1
    b1 = B_all if b1 is None else b1
    B = b1 - b0
    dt = 1 if dtype == "bf16" else 0
    t = np.ascontiguousarray(target[b0:b1])
    d = np.ascontiguousarray(draft[b0:b1]) if draft is not None and gamma > 0 else None
    x = np.ascontiguousarray(tokens[b0:b1], np.int32)
    vl = None if verify_len is None else np.ascontiguousarray(verify_len[b0:b1], np.int32)
    u = None if uniforms is None else np.ascontiguousarray(uniforms[b0:b1], np.float32)
    out = dict(tokens=np.empty((B, G1), np.int32), accept_len=np.empty(B, np.int32),
               px=np.empty((B, gamma)), qx=np.empty((B, gamma)), margin=np.empty((B, gamma)),
               resid_mass=np.empty(B), cdf_lo=np.empty(B), cdf_hi=np.empty(B),
               u_draw=np.empty(B), status=np.empty(B, np.int32), events=np.empty(B, np.int32))
    rc = _L().oracle_verify(_p(t), _p(d), dt, B, gamma, V, _p(x), _p(vl),
                            float(np.float32(T)), _p(u), _p(out["tokens"]), _p(out["accept_len"]),
                            _p(out["px"]), _p(out["qx"]), _p(out["margin"]), _p(out["resid_mass"]),
                            _p(out["cdf_lo"]), _p(out["cdf_hi"]), _p(out["u_draw"]),
                            _p(out["status"]), _p(out["events"]))
    out["rc"] = rc
    return out


def draw_cdf(target, draft, dtype: str, verify_len, T: float, b: int, n: int, query) -> tuple:
    """Normalised CDF edges (lo, hi) of the tokens in ``query`` in the oracle's
    own draw for request ``b`` after ``n`` accepted drafts (the residual
    max(p - q, 0) of row n after a rejection, else p of row verify_len[b]).
    T > 0; arrays laid out as for :func:`verify`."""
    B_all, G1, V = target.shape
    gamma = G1 - 1
    dt = 1 if dtype == "bf16" else 0
    t = np.ascontiguousarray(target[b:b + 1])
    d = np.ascontiguousarray(draft[b:b + 1]) if draft is not None and gamma > 0 else None
    vl = None if verify_len is None else np.ascontiguousarray(verify_len[b:b + 1], np.int32)
    q = np.ascontiguousarray(np.atleast_1d(query), np.int32)
    lo = np.empty(len(q))
    hi = np.empty(len(q))
    rc = _L().oracle_draw_cdf(_p(t), _p(d), dt, 1, gamma, V, _p(vl), float(np.float32(T)), 0, int(n),
                              _p(q), len(q), _p(lo), _p(hi))
    if rc != OK:
        raise ValueError(f"oracle_draw_cdf rejected request {b}, n={n}: {rc}")
    return lo, hi


def verify_probs(P, Q, tokens, uniforms) -> dict:
    """Verification on probability vectors given directly (fp64)."""
    P = np.ascontiguousarray(P, np.float64)
    Q = np.ascontiguousarray(Q, np.float64)
    B, G1, V = P.shape
    gamma = G1 - 1
    x = np.ascontiguousarray(tokens, np.int32)
    u = np.ascontiguousarray(uniforms, np.float64)
    out = dict(tokens=np.empty((B, G1), np.int32), accept_len=np.empty(B, np.int32),
               resid_mass=np.empty(B))
    rc = _L().oracle_verify_probs(_p(P), _p(Q), B, gamma, V, _p(x), _p(u), _p(out["tokens"]),
                                  _p(out["accept_len"]), _p(out["resid_mass"]))
    out["rc"] = rc
    return out


def pack_rows(verify_len, gamma: int) -> dict:
    """Dense request-major row index of ragged prefixes."""
    vl = np.ascontiguousarray(verify_len, np.int32)
    B = vl.shape[0]
    tr = np.empty(B, np.int32)
    dr = np.empty(B, np.int32)
    tot = np.empty(2, np.int32)
    rc = _L().oracle_pack_rows(_p(vl), B, gamma, _p(tr), _p(dr), _p(tot))
    return dict(rc=rc, target_row=tr, draft_row=dr, K_target=int(tot[0]), K_draft=int(tot[1]))


def _knots(cost):
    kt = np.ascontiguousarray(cost[0], np.float64)
    kc = np.ascontiguousarray(cost[1], np.float64)
    return kt, kc


def cost_at(N: float, cost) -> float:
    kt, kc = _knots(cost)
    r = ctypes.c_double()
    _L().oracle_cost_at(float(N), _p(kt), _p(kc), len(kt), ctypes.byref(r))
    return r.value


_sts_keep = None


def _set_sts(sts_T):
    """Calibration temperatures for the next scheduler call (None: none)."""
    global _sts_keep
    _sts_keep = None if sts_T is None else np.ascontiguousarray(sts_T, np.float64)
    _L().oracle_set_sts(_p(_sts_keep))


def _sched(fn, conf, cost, min_len, with_obj=True, sts_T=None):
    _set_sts(sts_T)
    conf = np.ascontiguousarray(conf, np.float32)
    B, gamma = conf.shape
    kt, kc = _knots(cost)
    out = np.full(B, -1, np.int32)
    if with_obj:
        obj, gap = ctypes.c_double(np.nan), ctypes.c_double(np.nan)
        rc = fn(_p(conf), B, gamma, _p(kt), _p(kc), len(kt), min_len, _p(out),
                ctypes.byref(obj), ctypes.byref(gap))
        return dict(rc=rc, verify_len=out, obj=obj.value, gap=gap.value)
    rc = fn(_p(conf), B, gamma, _p(kt), _p(kc), len(kt), min_len, _p(out))
    return dict(rc=rc, verify_len=out)


def sched_exact(conf, cost, min_len: int = 0, sts_T=None) -> dict:
    return _sched(_L().oracle_sched_exact, conf, cost, min_len, sts_T=sts_T)


def sched_alg1(conf, cost, min_len: int = 0, sts_T=None) -> dict:
    return _sched(_L().oracle_sched_alg1, conf, cost, min_len, with_obj=False, sts_T=sts_T)


def sched_brute(conf, cost, min_len: int = 0, sts_T=None) -> dict:
    return _sched(_L().oracle_sched_brute, conf, cost, min_len, sts_T=sts_T)


def sched_dcut(conf, ratios, costs, min_len: int = 0, sts_T=None) -> dict:
    """D-cut: the best of the budgets ceil(rho * B(gamma+1)) by progress / cost."""
    _set_sts(sts_T)
    conf = np.ascontiguousarray(conf, np.float32)
    B, gamma = conf.shape
    r = np.ascontiguousarray(ratios, np.float64)
    c = np.ascontiguousarray(costs, np.float64)
    out = np.full(B, -1, np.int32)
    choice = ctypes.c_int(-1)
    obj = np.full(len(r), np.nan)
    rc = _L().oracle_sched_dcut(_p(conf), B, gamma, _p(r), _p(c), len(r), min_len, _p(out), ctypes.byref(choice),
                                _p(obj))
    return dict(rc=rc, verify_len=out, choice=choice.value, obj=obj)


def sched_threshold(conf, threshold: float, min_len: int = 0, sts_T=None, max_len: int | None = None) -> dict:
    _set_sts(sts_T)
    conf = np.ascontiguousarray(conf, np.float32)
    B, gamma = conf.shape
    out = np.full(B, -1, np.int32)
    ml = gamma if max_len is None else max_len
    rc = _L().oracle_sched_threshold(_p(conf), B, gamma, float(threshold), ml, min_len, _p(out))
    return dict(rc=rc, verify_len=out)


def sts_ece(a, y, bins: int = 15) -> float:
    a = np.ascontiguousarray(a, np.float64)
    y = np.ascontiguousarray(y, np.int32)
    out = ctypes.c_double()
    _L().oracle_sts_ece(_p(a), _p(y), len(a), bins, ctypes.byref(out))
    return out.value


def sts_fit(conf, accept_len, grid: int = 100, bins: int = 15) -> dict:
    """STS temperatures (one per position) from confidences [n, gamma] and the
    accept lengths observed when verifying all gamma positions."""
    conf = np.ascontiguousarray(conf, np.float32)
    n, gamma = conf.shape
    al = np.ascontiguousarray(accept_len, np.int32)
    T = np.empty(gamma)
    e = np.empty(gamma)
    rc = _L().oracle_sts_fit(_p(conf), _p(al), n, gamma, grid, bins, _p(T), _p(e))
    return dict(rc=rc, T=T, ece=e)
