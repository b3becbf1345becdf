"""GB300-native speculative-decoding verification.

Thin ctypes binding over ``libspecv.so`` (C ABI declared in ``include/specv.h``).
Every step of verification and scheduling runs in the library's CUDA kernels;
this module only checks tensor properties, allocates outputs/workspaces with
PyTorch and passes pointers and the current CUDA stream.  There is no CPU
fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_CSRC = os.path.join(_HERE, "csrc")
LIB_PATH = os.path.join(_HERE, "libspecv.so")
SOURCES = ["specv_verify.cu", "specv_sched.cu", "specv_api.cu", "specv_static.cu"]
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3", "-std=c++17",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-O2"]

# status codes (include/specv.h)
OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_TEMPERATURE = 0, -1, -2, -3, -4
ERR_VERIFY_LEN, ERR_TOKEN, ERR_WORKSPACE, ERR_COST_TABLE = -5, -6, -7, -8
ERR_NONFINITE, ERR_TIMEOUT, ERR_CUDA, ERR_UNIFORM, ERR_CONFIDENCE = -9, -10, -11, -12, -13
ERR_ROW_INDEX = -14
F32, BF16 = 0, 1
SCHED_EXACT, SCHED_ALGORITHM1, SCHED_DCUT = 0, 1, 2
MAX_BATCH, MAX_GAMMA, MAX_SCHED_CANDIDATES = 4096, 32, 16384

EXPORTED = ["spec_verify_workspace_bytes", "spec_verify", "spec_verify_stats",
            "spec_schedule_workspace_bytes", "spec_schedule", "spec_read_status",
            "spec_status_string", "spec_profile_events", "spec_verify_kernel_count",
            "spec_verify_static", "spec_schedule_static", "spec_sts_fit", "spec_verify_packed",
            "spec_pack_rows", "spec_selftest_wait", "spec_selftest_expire_first_wait"]
STATIC_WORKSPACE_BYTES = 8 << 20


class SpecError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (code {code})" if where else status_string(code))


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/*.cu for sm_103a into libspecv.so (in-tree, parallel TUs)."""
    srcs = [os.path.join(_CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(_CSRC, "specv_common.cuh"), os.path.join(_CSRC, "specv_rowstats.cuh"),
                   os.path.join(_CSRC, "specv_trace.h"), os.path.join(_ROOT, "include", "specv.h")]
    if (not force and os.path.exists(LIB_PATH)
            and all(os.path.getmtime(LIB_PATH) >= os.path.getmtime(d) for d in deps)):
        return LIB_PATH
    bdir = os.path.join(_HERE, "_build")
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src).replace(".cu", ".o"))
        cmd = [nvcc, *NVCC_FLAGS, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(len(srcs)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp, *objs],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded libspecv.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build() "
                                       "(or speculative_decoding_verification_softmax_gb300.build())")
                L = ctypes.CDLL(LIB_PATH)
                vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
                L.spec_verify_workspace_bytes.argtypes = [i32, i32, i32, i32]
                L.spec_verify_workspace_bytes.restype = sz
                L.spec_verify.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, f32, vp, vp, vp, vp, sz, vp]
                L.spec_verify.restype = i32
                L.spec_verify_stats.argtypes = [vp, sz, i32, i32, i32, i32, vp, vp, vp, vp, vp]
                L.spec_verify_stats.restype = i32
                L.spec_schedule_workspace_bytes.argtypes = [i32, i32]
                L.spec_schedule_workspace_bytes.restype = sz
                L.spec_schedule.argtypes = [vp, i32, i32, vp, i32, i32, vp, vp, vp, sz, vp]
                L.spec_schedule_static.argtypes = [vp, i32, i32, f32, i32, i32, vp, vp, vp, sz, vp]
                L.spec_schedule_static.restype = i32
                L.spec_sts_fit.argtypes = [vp, vp, i32, i32, vp, vp]
                L.spec_sts_fit.restype = i32
                L.spec_schedule.restype = i32
                L.spec_read_status.argtypes = [vp, vp, ctypes.POINTER(i32)]
                L.spec_read_status.restype = i32
                L.spec_status_string.argtypes = [i32]
                L.spec_status_string.restype = ctypes.c_char_p
                L.spec_profile_events.argtypes = [vp, vp]
                L.spec_profile_events.restype = i32
                L.spec_verify_kernel_count.argtypes = [i32, f32]
                L.spec_verify_kernel_count.restype = i32
                L.spec_verify_static.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, f32, vp, vp, vp, vp]
                L.spec_verify_static.restype = i32
                L.spec_verify_packed.argtypes = [vp, i32, vp, i32, vp, vp, i32, i32, i32, i32, vp, vp, f32, vp,
                                                 vp, vp, vp, sz, vp]
                L.spec_verify_packed.restype = i32
                L.spec_pack_rows.argtypes = [vp, i32, i32, vp, vp, vp, vp]
                L.spec_pack_rows.restype = i32
                L.spec_selftest_wait.argtypes = [ctypes.c_longlong, vp, vp, vp]
                L.spec_selftest_wait.restype = i32
                L.spec_selftest_expire_first_wait.argtypes = [i32]
                L.spec_selftest_expire_first_wait.restype = i32
                _lib = L
    return _lib


class CostTable(ctypes.Structure):
    """spec_cost_table: piecewise-linear round cost, knots (tokens[i], cost_ms[i])."""
    _fields_ = [("n", ctypes.c_int), ("tokens", ctypes.c_double * 32), ("cost_ms", ctypes.c_double * 32)]

    @classmethod
    def from_knots(cls, tokens, cost_ms) -> "CostTable":
        t = cls()
        t.n = len(tokens)
        if len(cost_ms) != t.n or not 1 <= t.n <= 32:
            t.n = 0 if t.n == 0 else 33  # rejected by the library
            return t
        for i, (a, b) in enumerate(zip(tokens, cost_ms)):
            t.tokens[i] = float(a)
            t.cost_ms[i] = float(b)
        return t


def status_string(code: int) -> str:
    try:
        return lib().spec_status_string(int(code)).decode()
    except RuntimeError:
        return f"status {code}"


def _check(rc: int, where: str):
    if rc != OK:
        raise SpecError(rc, where)


# ------------------------------------------------------------ torch helpers
def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _check_tensor(name, t, dtype, shape, required=True):
    """A contiguous tensor of `dtype` and `shape` on the current CUDA device
    (the device whose current stream the call uses), or None if allowed."""
    torch = _torch()
    if t is None:
        if required:
            raise ValueError(f"{name} is required")
        return
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, but the current device is cuda:{torch.cuda.current_device()}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _check_verify_inputs(B, gamma, V, ldtype, draft_logits, draft_shape, draft_tokens, verify_len, temperature,
                         uniforms, out_tokens, out_accept_len):
    """Shapes, dtypes and devices of every tensor a verify call reads or writes
    (the library reads them with the sizes it is given, so a mismatch here
    would be an out-of-bounds access on the device)."""
    torch = _torch()
    greedy = float(temperature) == 0.0
    _check_tensor("draft_logits", draft_logits, ldtype, draft_shape, required=not greedy and gamma > 0)
    _check_tensor("draft_tokens", draft_tokens, torch.int32, (B, gamma), required=gamma > 0)
    _check_tensor("verify_len", verify_len, torch.int32, (B,), required=False)
    _check_tensor("uniforms", uniforms, torch.float32, (B, gamma + 2), required=not greedy)
    _check_tensor("out_tokens", out_tokens, torch.int32, (B, gamma + 1), required=False)
    _check_tensor("out_accept_len", out_accept_len, torch.int32, (B,), required=False)


def verify_workspace_bytes(B: int, gamma: int, V: int, dtype_code: int) -> int:
    return int(lib().spec_verify_workspace_bytes(B, gamma, V, dtype_code))


def alloc_verify_workspace(B: int, gamma: int, V: int, dtype_code: int, device=None):
    """A verification workspace (its contents need no initialisation)."""
    torch = _torch()
    n = verify_workspace_bytes(B, gamma, V, dtype_code)
    if n == 0:
        raise SpecError(ERR_SHAPE, "spec_verify_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def verify(target_logits, draft_logits, draft_tokens, verify_len, temperature: float, uniforms,
           *, out_tokens=None, out_accept_len=None, workspace=None, stream=None):
    """Run spec_verify on device tensors (see include/specv.h).

    target_logits [B, gamma+1, V] and draft_logits [B, gamma, V] (bf16 or fp32,
    contiguous), draft_tokens [B, gamma] int32, verify_len [B] int32 or None,
    uniforms [B, gamma+2] fp32 (None at temperature 0).  Returns
    (out_tokens [B, gamma+1] int32, out_accept_len [B] int32, workspace).
    """
    torch = _torch()
    B, G1, V = target_logits.shape
    gamma = G1 - 1
    dt = _dtype_code(target_logits)
    dev = target_logits.device
    _check_tensor("target_logits", target_logits, target_logits.dtype, (B, G1, V))
    _check_verify_inputs(B, gamma, V, target_logits.dtype, draft_logits, (B, gamma, V), draft_tokens, verify_len,
                         temperature, uniforms, out_tokens, out_accept_len)
    if workspace is not None:
        _check_tensor("workspace", workspace, torch.uint8, (workspace.numel(),))
    if out_tokens is None:
        out_tokens = torch.empty((B, G1), dtype=torch.int32, device=dev)
    if out_accept_len is None:
        out_accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = alloc_verify_workspace(B, gamma, V, dt, dev)
    rc = lib().spec_verify(_ptr(target_logits), _ptr(draft_logits), dt, B, gamma, V, _ptr(draft_tokens),
                           _ptr(verify_len), ctypes.c_float(temperature), _ptr(uniforms), _ptr(out_tokens),
                           _ptr(out_accept_len), _ptr(workspace), workspace.numel(),
                           _stream_handle(stream))
    _check(rc, "spec_verify")
    return out_tokens, out_accept_len, workspace


def verify_static(target_logits, draft_logits, draft_tokens, verify_len, temperature: float, uniforms,
                  *, out_tokens=None, out_accept_len=None, stream=None):
    """spec_verify_static: verification without a workspace, for callers that
    cannot allocate device memory where they verify.  The scratch is a fixed
    8 MiB array on the device (shared by all calls; order overlapping calls on
    one stream).  Only the outputs, if not given, are allocated here.
    Returns (out_tokens, out_accept_len)."""
    torch = _torch()
    B, G1, V = target_logits.shape
    gamma = G1 - 1
    dt = _dtype_code(target_logits)
    dev = target_logits.device
    _check_tensor("target_logits", target_logits, target_logits.dtype, (B, G1, V))
    _check_verify_inputs(B, gamma, V, target_logits.dtype, draft_logits, (B, gamma, V), draft_tokens, verify_len,
                         temperature, uniforms, out_tokens, out_accept_len)
    if out_tokens is None:
        out_tokens = torch.empty((B, G1), dtype=torch.int32, device=dev)
    if out_accept_len is None:
        out_accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    rc = lib().spec_verify_static(_ptr(target_logits), _ptr(draft_logits), dt, B, gamma, V, _ptr(draft_tokens),
                                  _ptr(verify_len), ctypes.c_float(temperature), _ptr(uniforms),
                                  _ptr(out_tokens), _ptr(out_accept_len), _stream_handle(stream))
    _check(rc, "spec_verify_static")
    return out_tokens, out_accept_len


def verify_packed(target_logits, draft_logits, target_row, draft_row, draft_tokens, verify_len,
                  temperature: float, uniforms, *, out_tokens=None, out_accept_len=None, workspace=None,
                  stream=None):
    """Run spec_verify_packed: target_logits [K_target, V] and draft_logits
    [K_draft, V] (bf16 or fp32, contiguous; draft may be None at temperature 0),
    the row index target_row / draft_row [B] int32, draft_tokens [B, gamma]
    int32, verify_len [B] int32 or None, uniforms [B, gamma+2] fp32.
    Returns (out_tokens [B, gamma+1], out_accept_len [B], workspace)."""
    torch = _torch()
    Kt, V = target_logits.shape
    B, gamma = draft_tokens.shape
    Kd = draft_logits.shape[0] if draft_logits is not None else 0
    dt = _dtype_code(target_logits)
    dev = target_logits.device
    _check_tensor("target_logits", target_logits, target_logits.dtype, (Kt, V))
    _check_verify_inputs(B, gamma, V, target_logits.dtype, draft_logits, (Kd, V), draft_tokens, verify_len,
                         temperature, uniforms, out_tokens, out_accept_len)
    _check_tensor("target_row", target_row, torch.int32, (B,))
    _check_tensor("draft_row", draft_row, torch.int32, (B,), required=float(temperature) != 0.0 and gamma > 0)
    if workspace is not None:
        _check_tensor("workspace", workspace, torch.uint8, (workspace.numel(),))
    if out_tokens is None:
        out_tokens = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    if out_accept_len is None:
        out_accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = alloc_verify_workspace(B, gamma, V, dt, dev)
    rc = lib().spec_verify_packed(_ptr(target_logits), Kt, _ptr(draft_logits), Kd, _ptr(target_row),
                                  _ptr(draft_row), dt, B, gamma, V, _ptr(draft_tokens), _ptr(verify_len),
                                  ctypes.c_float(temperature), _ptr(uniforms), _ptr(out_tokens),
                                  _ptr(out_accept_len), _ptr(workspace), workspace.numel(),
                                  _stream_handle(stream))
    _check(rc, "spec_verify_packed")
    return out_tokens, out_accept_len, workspace


def pack_rows(verify_len, gamma: int, *, target_row=None, draft_row=None, totals=None, stream=None):
    """Run spec_pack_rows on verify_len [B] int32 (CUDA): the dense request-major
    row index.  Returns (target_row [B], draft_row [B], totals [2] = (K_target,
    K_draft)), all int32 on the device."""
    torch = _torch()
    B = verify_len.shape[0]
    dev = verify_len.device
    _check_tensor("verify_len", verify_len, torch.int32, (B,))
    for name, t, shp in (("target_row", target_row, (B,)), ("draft_row", draft_row, (B,)), ("totals", totals, (2,))):
        _check_tensor(name, t, torch.int32, shp, required=False)
    if target_row is None:
        target_row = torch.empty((B,), dtype=torch.int32, device=dev)
    if draft_row is None:
        draft_row = torch.empty((B,), dtype=torch.int32, device=dev)
    if totals is None:
        totals = torch.empty((2,), dtype=torch.int32, device=dev)
    rc = lib().spec_pack_rows(_ptr(verify_len), B, gamma, _ptr(target_row), _ptr(draft_row), _ptr(totals),
                              _stream_handle(stream))
    _check(rc, "spec_pack_rows")
    return target_row, draft_row, totals


def verify_stats(workspace, B: int, gamma: int, V: int, dtype_code: int, stream=None):
    """Diagnostics of the last verify on `workspace`: (px, qx, resid_mass, status)."""
    torch = _torch()
    dev = workspace.device
    px = torch.empty((B, gamma), dtype=torch.float64, device=dev)
    qx = torch.empty((B, gamma), dtype=torch.float64, device=dev)
    mass = torch.empty((B,), dtype=torch.float64, device=dev)
    st = torch.empty((B,), dtype=torch.int32, device=dev)
    rc = lib().spec_verify_stats(_ptr(workspace), workspace.numel(), B, gamma, V, dtype_code, _ptr(px),
                                 _ptr(qx), _ptr(mass), _ptr(st), _stream_handle(stream))
    _check(rc, "spec_verify_stats")
    return px, qx, mass, st


def _sts_arg(sts, gamma):
    if sts is None:
        return None, None
    import numpy as np
    arr = np.ascontiguousarray(np.asarray(sts, dtype=np.float32).reshape(-1))
    if arr.size != gamma:
        raise ValueError("sts temperatures need one value per draft position")
    return arr, arr.ctypes.data_as(ctypes.c_void_p)


def schedule(confidence, cost, min_len: int = 0, mode: int = SCHED_EXACT, *, sts=None, out_verify_len=None,
             workspace=None, stream=None):
    """Run spec_schedule: confidence [B, gamma] fp32 CUDA tensor, cost = (tokens, cost_ms)
    knots or a CostTable (for SCHED_DCUT: (ratios, costs)); sts = per-position STS
    temperatures or None.  Returns (out_verify_len [B] int32, workspace)."""
    torch = _torch()
    B, gamma = confidence.shape
    _check_tensor("confidence", confidence, torch.float32, (B, gamma))
    _check_tensor("out_verify_len", out_verify_len, torch.int32, (B,), required=False)
    table = cost if isinstance(cost, CostTable) else CostTable.from_knots(*cost)
    if out_verify_len is None:
        out_verify_len = torch.empty((B,), dtype=torch.int32, device=confidence.device)
    if workspace is None:
        workspace = torch.zeros(max(256, int(lib().spec_schedule_workspace_bytes(B, gamma))),
                                dtype=torch.uint8, device=confidence.device)
    keep, sts_p = _sts_arg(sts, gamma)
    rc = lib().spec_schedule(_ptr(confidence), B, gamma, ctypes.byref(table), min_len, mode, sts_p,
                             _ptr(out_verify_len), _ptr(workspace), workspace.numel(),
                             _stream_handle(stream))
    _check(rc, "spec_schedule")
    return out_verify_len, workspace


def schedule_static(confidence, threshold: float, max_len: int, min_len: int = 0, *, sts=None,
                    out_verify_len=None, workspace=None, stream=None):
    """Run spec_schedule_static: leading positions with confidence >= threshold,
    clamped to [min_len, max_len] (threshold <= 0: fixed length max_len)."""
    torch = _torch()
    B, gamma = confidence.shape
    _check_tensor("confidence", confidence, torch.float32, (B, gamma), required=threshold > 0)
    _check_tensor("out_verify_len", out_verify_len, torch.int32, (B,), required=False)
    if out_verify_len is None:
        out_verify_len = torch.empty((B,), dtype=torch.int32, device=confidence.device)
    if workspace is None:
        workspace = torch.zeros(256, dtype=torch.uint8, device=confidence.device)
    keep, sts_p = _sts_arg(sts, gamma)
    rc = lib().spec_schedule_static(_ptr(confidence), B, gamma, ctypes.c_float(threshold), max_len, min_len, sts_p,
                                    _ptr(out_verify_len), _ptr(workspace), workspace.numel(),
                                    _stream_handle(stream))
    _check(rc, "spec_schedule_static")
    return out_verify_len, workspace


def sts_fit(confidence, accept_len):
    """spec_sts_fit on host arrays: confidences [n, gamma] and the accept lengths
    observed at verify_len = gamma.  Returns (temperatures [gamma] fp32, ece [gamma])."""
    import numpy as np
    c = np.ascontiguousarray(confidence, np.float32)
    al = np.ascontiguousarray(accept_len, np.int32)
    n, gamma = c.shape
    T = np.empty(gamma, np.float32)
    e = np.empty(gamma, np.float64)
    rc = lib().spec_sts_fit(c.ctypes.data_as(ctypes.c_void_p), al.ctypes.data_as(ctypes.c_void_p), n, gamma,
                            T.ctypes.data_as(ctypes.c_void_p), e.ctypes.data_as(ctypes.c_void_p))
    _check(rc, "spec_sts_fit")
    return T, e


def selftest_wait(limit_ns: int = 1_000_000, stream=None):
    """Run spec_selftest_wait: returns ((status_blocked, status_completed),
    (elapsed_ns_blocked, elapsed_ns_completed)) after synchronising."""
    torch = _torch()
    st = torch.full((2,), 99, dtype=torch.int32, device="cuda")
    el = torch.zeros((2,), dtype=torch.int64, device="cuda")
    _check(lib().spec_selftest_wait(int(limit_ns), _ptr(st), _ptr(el), _stream_handle(stream)), "spec_selftest_wait")
    torch.cuda.synchronize()
    return tuple(int(v) for v in st.cpu()), tuple(int(v) for v in el.cpu())


def selftest_expire_first_wait(on: bool) -> None:
    """Test hook: while on, the first copy wait of every streaming warp in later
    verify calls counts as expired (the timeout path; see include/specv.h)."""
    _check(lib().spec_selftest_expire_first_wait(1 if on else 0), "spec_selftest_expire_first_wait")


def read_status(workspace, stream=None) -> int:
    """Synchronise the stream, read and clear the workspace's device status word."""
    v = ctypes.c_int(0)
    _check(lib().spec_read_status(_ptr(workspace), _stream_handle(stream), ctypes.byref(v)),
           "spec_read_status")
    return v.value


def profile_events(before=None, after=None):
    """Register torch.cuda.Event pair recorded around the row-statistics kernel."""
    b = ctypes.c_void_p(before.cuda_event) if before is not None else None
    a = ctypes.c_void_p(after.cuda_event) if after is not None else None
    _check(lib().spec_profile_events(b, a), "spec_profile_events")


def kernel_count(B: int, temperature: float) -> int:
    return int(lib().spec_verify_kernel_count(B, ctypes.c_float(temperature)))
