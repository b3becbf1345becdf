"""Seeded synthetic inputs for verification and scheduling.

This module is shared by the tests, the benchmark and ``__graft_entry__``.  It
holds no step of the verification or scheduling arithmetic: it only draws
random numbers (SplitMix64 counter streams, Box-Muller normals, Gumbel-max
draft sampling) and encodes logits as bf16 / fp32.  Both the CUDA path and the
oracle receive the arrays it produces.

Workload recipes stand in for the served benchmarks the pages measure on
(chat, code and maths traffic at concurrency 4-64, draft blocks of 3-16 tokens,
vocabularies of 32k-152k); no benchmark item is used.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so next to it (plain gcc, no SIMD flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        u64, i32, dbl, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.synth_raw64.argtypes = [u64, u64, u64, vp]
        lib.synth_uniform_f64.argtypes = [u64, u64, u64, vp]
        lib.synth_uniform_f32.argtypes = [u64, u64, u64, vp]
        lib.synth_normal_f64.argtypes = [u64, u64, u64, dbl, dbl, i32, vp]
        lib.synth_to_bf16.argtypes = [vp, u64, vp]
        lib.synth_bf16_to_f32.argtypes = [vp, u64, vp]
        lib.synth_to_f32.argtypes = [vp, u64, vp]
        lib.synth_gumbel_argmax.argtypes = [vp, u64, u64, dbl, u64, u64, vp]
        lib.synth_row_argmax.argtypes = [vp, u64, u64, vp]
        for f in ("synth_raw64", "synth_uniform_f64", "synth_uniform_f32", "synth_normal_f64",
                  "synth_to_bf16", "synth_bf16_to_f32", "synth_to_f32", "synth_gumbel_argmax",
                  "synth_row_argmax"):
            getattr(lib, f).restype = None
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- primitives
def raw64(seed: int, n: int, start: int = 0) -> np.ndarray:
    out = np.empty(n, np.uint64)
    _L().synth_raw64(seed, start, n, _p(out))
    return out


def uniform_f64(seed: int, n: int, start: int = 0) -> np.ndarray:
    out = np.empty(n, np.float64)
    _L().synth_uniform_f64(seed, start, n, _p(out))
    return out


def uniform_f32(seed: int, n: int, start: int = 0) -> np.ndarray:
    """24-bit uniforms in [0, 1), exact in fp32."""
    out = np.empty(n, np.float32)
    _L().synth_uniform_f32(seed, start, n, _p(out))
    return out


def normal_f64(seed: int, n: int, mean: float = 0.0, std: float = 1.0, start: int = 0,
               out: np.ndarray | None = None) -> np.ndarray:
    """mean + std * N(0,1); with ``out`` given, the draw is added to it."""
    acc = 1 if out is not None else 0
    if out is None:
        out = np.empty(n, np.float64)
    _L().synth_normal_f64(seed, start, n, float(mean), float(std), acc, _p(out))
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    _L().synth_to_bf16(_p(x), x.size, _p(out))
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, np.uint16)
    out = np.empty(b.shape, np.float32)
    _L().synth_bf16_to_f32(_p(b), b.size, _p(out))
    return out


def gumbel_argmax(logits_f32: np.ndarray, inv_t: float, seed: int, start_row: int = 0) -> np.ndarray:
    """Draw one index per row from softmax(logits * inv_t) by the Gumbel-max trick."""
    x = np.ascontiguousarray(logits_f32, np.float32)
    R, V = x.reshape(-1, x.shape[-1]).shape
    out = np.empty(R, np.int32)
    _L().synth_gumbel_argmax(_p(x), R, V, float(inv_t), seed, start_row, _p(out))
    return out


def row_argmax(logits_f32: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(logits_f32, np.float32)
    R, V = x.reshape(-1, x.shape[-1]).shape
    out = np.empty(R, np.int32)
    _L().synth_row_argmax(_p(x), R, V, _p(out))
    return out


def distinct_ids(seed: int, row: int, k: int, V: int) -> np.ndarray:
    """k distinct ids uniform in [0, V): sequential draws, duplicates skipped."""
    ids: list[int] = []
    pos = row * 4096
    while len(ids) < min(k, V):
        u = uniform_f64(seed, 64, start=pos)
        pos += 64
        for x in (u * V).astype(np.int64):
            if x not in ids:
                ids.append(int(x))
                if len(ids) == min(k, V):
                    break
    return np.array(ids, np.int64)


# ------------------------------------------------------------------ recipes
@dataclass
class VerifySpec:
    """Shape and value recipe of one synthetic verification batch."""
    name: str
    B: int
    gamma: int
    V: int
    dtype: str              # "f32" or "bf16"
    T: float
    target_std: float
    draft_noise_std: float
    boost: float = 0.0      # added to `boost_count` distinct ids of every target row
    boost_count: int = 0
    greedy_draft_p: float | None = None   # T == 0 recipe: draft = argmax w.p. p else uniform id
    seed_logits: int = 0
    seed_noise: int = 0
    seed_tokens: int = 0
    seed_uniforms: int = 0
    seed_boost: int = 0
    verify_len: int | None = None          # None -> gamma for every request


CONFIGS: dict[str, VerifySpec] = {
    # B=4, gamma=4, V=1024, fp32, T=1: z_t ~ N(0, 2^2), z_d = z_t + N(0, 0.7^2)
    "tiny": VerifySpec("tiny", 4, 4, 1024, "f32", 1.0, 2.0, 0.7,
                       seed_logits=100, seed_noise=101, seed_tokens=0, seed_uniforms=1),
    # B=16, gamma=4, V=32000, bf16, T=0.8: N(0, 3^2) with +6 on 32 ids, noise N(0, 1.5^2)
    "mtp_chat": VerifySpec("mtp_chat", 16, 4, 32000, "bf16", 0.8, 3.0, 1.5, boost=6.0, boost_count=32,
                           seed_logits=200, seed_noise=201, seed_tokens=202, seed_uniforms=203,
                           seed_boost=204),
    # B=64, gamma=16, V=131072, bf16, T=1: N(0, 2^2) with +10 on one id, noise N(0, 0.3^2)
    "block_diffusion": VerifySpec("block_diffusion", 64, 16, 131072, "bf16", 1.0, 2.0, 0.3,
                                  boost=10.0, boost_count=1, seed_logits=300, seed_noise=301,
                                  seed_tokens=302, seed_uniforms=303, seed_boost=304),
    # B=32, gamma=8, V=151936, bf16, T=0: N(0, 2^2); draft = argmax w.p. 0.7 else uniform id
    "greedy": VerifySpec("greedy", 32, 8, 151936, "bf16", 0.0, 2.0, 1.0, greedy_draft_p=0.7,
                         seed_logits=400, seed_noise=401, seed_tokens=402, seed_uniforms=403),
}

# Scheduled ragged workload: confidences sigmoid(N(1.5, 1)) [64, 16], then the
# block-diffusion logits verified at the scheduled lengths.
SCHED_SEED = 500
SCHED_B, SCHED_GAMMA, SCHED_MIN_LEN = 64, 16, 1


@dataclass
class VerifyCase:
    spec: VerifySpec
    target: np.ndarray        # [B, gamma+1, V] uint16 (bf16 bits) or float32
    draft: np.ndarray         # [B, gamma, V]
    draft_tokens: np.ndarray  # [B, gamma] int32
    verify_len: np.ndarray    # [B] int32
    uniforms: np.ndarray      # [B, gamma+2] float32
    extra: dict = field(default_factory=dict)

    @property
    def B(self): return self.spec.B

    @property
    def gamma(self): return self.spec.gamma

    @property
    def V(self): return self.spec.V

    @property
    def T(self): return self.spec.T

    @property
    def dtype(self): return self.spec.dtype


def _encode(x64: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return to_bf16_bits(x64)
    out = np.empty(x64.shape, np.float32)
    _L().synth_to_f32(_p(np.ascontiguousarray(x64)), x64.size, _p(out))
    return out


def as_f32(enc: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_f32(enc) if dtype == "bf16" else np.ascontiguousarray(enc, np.float32)


def make_verify_case(spec: VerifySpec | str, **overrides) -> VerifyCase:
    """Generate one batch: target/draft logits, draft tokens, uniforms, lengths."""
    if isinstance(spec, str):
        spec = CONFIGS[spec]
    if overrides:
        spec = VerifySpec(**{**spec.__dict__, **overrides})
    B, g, V = spec.B, spec.gamma, spec.V
    edt = np.uint16 if spec.dtype == "bf16" else np.float32
    target = np.empty((B, g + 1, V), edt)
    draft = np.empty((B, g, V), edt)
    tokens = np.empty((B, g), np.int32)
    for b in range(B):
        rows_t = normal_f64(spec.seed_logits, (g + 1) * V, 0.0, spec.target_std, start=b * (g + 1) * V)
        rows_t = rows_t.reshape(g + 1, V)
        if spec.boost_count:
            for j in range(g + 1):
                ids = distinct_ids(spec.seed_boost, b * (g + 1) + j, spec.boost_count, V)
                rows_t[j, ids] += spec.boost
        target[b] = _encode(rows_t, spec.dtype)
        if g:
            rows_d = np.ascontiguousarray(rows_t[:g]).reshape(-1)
            normal_f64(spec.seed_noise, g * V, 0.0, spec.draft_noise_std, start=b * g * V, out=rows_d)
            draft[b] = _encode(rows_d.reshape(g, V), spec.dtype)
            if spec.greedy_draft_p is not None:
                am = row_argmax(as_f32(target[b, :g], spec.dtype))
                u = uniform_f64(spec.seed_tokens, 2 * g, start=2 * b * g).reshape(g, 2)
                rnd = np.minimum((u[:, 1] * V).astype(np.int64), V - 1).astype(np.int32)
                tokens[b] = np.where(u[:, 0] < spec.greedy_draft_p, am, rnd)
            else:
                tokens[b] = gumbel_argmax(as_f32(draft[b], spec.dtype), 1.0 / spec.T,
                                          spec.seed_tokens, start_row=b * g)
    uniforms = uniform_f32(spec.seed_uniforms, B * (g + 2)).reshape(B, g + 2)
    vl = np.full(B, g if spec.verify_len is None else spec.verify_len, np.int32)
    return VerifyCase(spec, target, draft, tokens, vl, uniforms)


def make_confidences(B: int = SCHED_B, gamma: int = SCHED_GAMMA, seed: int = SCHED_SEED,
                     mean: float = 1.5, std: float = 1.0) -> np.ndarray:
    """Per-position confidences sigmoid(N(mean, std^2)) as fp32 [B, gamma]."""
    z = normal_f64(seed, B * gamma, mean, std)
    return (1.0 / (1.0 + np.exp(-z))).astype(np.float32).reshape(B, gamma)


# Round-cost tables for the scheduled workload: "8 ms + 0.02 ms per verified
# token, saturating at +12 ms above 512 tokens".  The three numbers do not agree
# (0.02 * 512 = 10.24), so three readings are kept:
#   B' (default): knots (0, 8), (512, 18.24), (513, 20), flat after.
#   A:            8 + min(0.02 N, 12)      -> knots (0, 8), (600, 20)
#   C:            8 + 0.02 min(N, 512)     -> knots (0, 8), (512, 18.24)
COST_TABLES = {
    "Bprime": ([0.0, 512.0, 513.0], [8.0, 18.24, 20.0]),
    "A": ([0.0, 600.0], [8.0, 20.0]),
    "C": ([0.0, 512.0], [8.0, 18.24]),
    "affine": ([0.0, 100000.0], [8.0, 8.0 + 0.02 * 100000.0]),
}


def make_replicated_case(P: np.ndarray, Q: np.ndarray, B: int, seed_tokens: int,
                         seed_uniforms: int, T: float = 1.0, dtype: str = "f32",
                         verify_len: int | None = None) -> VerifyCase:
    """B requests sharing the same rows: target logits T*log(P) ([gamma+1, V]) and
    draft logits T*log(Q) ([gamma, V]); draft tokens drawn from softmax(draft / T)
    by Gumbel-max, so x_j ~ Q_j; fresh uniforms per request.  Zero probabilities
    become -inf logits (masked vocabulary entries)."""
    P = np.asarray(P, np.float64)
    Q = np.asarray(Q, np.float64)
    gamma, V = Q.shape
    with np.errstate(divide="ignore"):
        lt = T * np.log(P)
        ld = T * np.log(Q)
    enc_t, enc_d = _encode(lt, dtype), _encode(ld, dtype)
    target = np.ascontiguousarray(np.broadcast_to(enc_t, (B, gamma + 1, V)))
    draft = np.ascontiguousarray(np.broadcast_to(enc_d, (B, gamma, V)))
    rows = np.ascontiguousarray(np.broadcast_to(as_f32(enc_d, dtype), (B, gamma, V)))
    tokens = gumbel_argmax(rows.reshape(B * gamma, V), 1.0 / T, seed_tokens).reshape(B, gamma)
    uniforms = uniform_f32(seed_uniforms, B * (gamma + 2)).reshape(B, gamma + 2)
    vl = np.full(B, gamma if verify_len is None else verify_len, np.int32)
    spec = VerifySpec("replicated", B, gamma, V, dtype, T, 0.0, 0.0)
    return VerifyCase(spec, target, draft, tokens, vl, uniforms)


def to_device(case: VerifyCase, device="cuda"):
    """The case's arrays as torch tensors on ``device`` (bf16 bits reinterpreted
    as torch.bfloat16): target, draft, draft tokens, verify lengths, uniforms.
    Marshalling only; torch is imported here so that the generators above work
    without it."""
    import torch
    if case.dtype == "bf16":
        t = torch.from_numpy(case.target.view(np.int16)).to(device).view(torch.bfloat16)
        d = torch.from_numpy(case.draft.view(np.int16)).to(device).view(torch.bfloat16)
    else:
        t = torch.from_numpy(case.target).to(device)
        d = torch.from_numpy(case.draft).to(device)
    x = torch.from_numpy(case.draft_tokens).to(device)
    vl = torch.from_numpy(case.verify_len).to(device)
    u = torch.from_numpy(case.uniforms).to(device)
    return t, d, x, vl, u
