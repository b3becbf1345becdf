"""Shared test helpers: run the oracle in request slices on host threads, move
synthetic cases to the GPU, and compare GPU results with the oracle under the
flagging rules for near-ties."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

import oracle
import specsynth

# Tolerances (the flag rules are explained in the design notes):
#   accept decisions may differ only where |u - p(x)/q(x)| < ACCEPT_FLAG;
#   a drawn token t' may differ from the oracle's t only where u lies within
#   DRAW_FLAG of the oracle's own CDF bin of t' (normalised CDF units), i.e.
#   u is that close to the boundary between the two tokens and the mass the
#   oracle puts strictly between them is below DRAW_FLAG;
#   such excused positions stay below FLAG_FRACTION of all positions;
#   p(x), q(x) and the draw's total weight agree within PROB_TOL absolute.
ACCEPT_FLAG = 1e-5
DRAW_FLAG = 1e-5
FLAG_FRACTION = 1e-4
PROB_TOL = 1e-5


def oracle_verify(case: specsynth.VerifyCase, T: float | None = None, verify_len=None,
                  threads: int | None = None) -> dict:
    """Oracle over all requests, split into request slices across host threads
    (ctypes releases the GIL; each slice runs the unchanged oracle)."""
    T = case.T if T is None else T
    vl = case.verify_len if verify_len is None else verify_len
    B = case.B
    threads = threads or min(B, os.cpu_count() or 1, 32)
    bounds = np.linspace(0, B, threads + 1).astype(int)
    uni = None if T == 0 else case.uniforms

    def run(i):
        return oracle.verify(case.target, case.draft, case.dtype, case.draft_tokens, vl, T, uni,
                             b0=int(bounds[i]), b1=int(bounds[i + 1]))

    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(run, range(threads)))
    out = {}
    for k in parts[0]:
        if k == "rc":
            out[k] = max(abs(p[k]) for p in parts) * (-1 if any(p[k] for p in parts) else 1)
        else:
            out[k] = np.concatenate([p[k] for p in parts])
    # request ids (kept through sub-selections) and the oracle's CDF lookup
    out["req"] = np.arange(B)
    if T != 0:
        out["_draw_cdf"] = lambda b, n, toks: oracle.draw_cdf(case.target, case.draft, case.dtype, vl, T,
                                                              b, n, toks)
    return out


to_device = specsynth.to_device


@dataclass
class Parity:
    requests: int = 0
    positions: int = 0
    accept_flagged: int = 0
    draw_flagged: int = 0
    mismatches: list = field(default_factory=list)
    max_p_err: float = 0.0
    max_mass_err: float = 0.0

    @property
    def flagged(self):
        return self.accept_flagged + self.draw_flagged


def draw_distance(o: dict, b: int, n: int, tok: int, draw_cdf=None) -> float:
    """Distance, in the oracle's normalised CDF units, from the draw's uniform
    of request b (row b of ``o``) to the oracle's own bin of token ``tok``:
    how far u would have to move for ``tok`` to be the correct draw.  inf when
    the oracle's CDF is not available or the token is out of range."""
    draw_cdf = draw_cdf or o.get("_draw_cdf")
    if draw_cdf is None:
        return float("inf")
    lo, hi = draw_cdf(int(o["req"][b]), int(n), [int(tok)])
    lo, hi, u = float(lo[0]), float(hi[0]), float(o["u_draw"][b])
    if not (lo == lo and hi == hi):
        return float("inf")
    return max(lo - u, u - hi, 0.0)


def compare(o: dict, g_tokens, g_len, g_px=None, g_qx=None, g_mass=None, g_status=None,
            greedy=False, draw_flag=DRAW_FLAG, accept_flag=ACCEPT_FLAG, draw_cdf=None) -> Parity:
    """Compare GPU outputs with the oracle request by request."""
    P = Parity()
    B, G1 = o["tokens"].shape
    gamma = G1 - 1
    for b in range(B):
        P.requests += 1
        if g_status is not None:
            assert g_status[b] == o["status"][b], (b, g_status[b], o["status"][b])
        no, ng = int(o["accept_len"][b]), int(g_len[b])
        if no < 0 or ng < 0:
            if no != ng or (g_tokens[b] != o["tokens"][b]).any():
                P.mismatches.append((b, "invalid", no, ng))
            continue
        P.positions += max(no, 0) + 1
        flagged = False
        if no != ng:
            k = min(no, ng)
            if not greedy and o["margin"][b, k] < accept_flag:
                P.accept_flagged += 1
                flagged = True
            else:
                P.mismatches.append((b, "accept_len", no, ng))
                continue
        if not flagged:
            if (g_tokens[b, :no] != o["tokens"][b, :no]).any():
                P.mismatches.append((b, "prefix"))
                continue
            if (g_tokens[b, no + 1:] != -1).any():
                P.mismatches.append((b, "tail"))
                continue
            if g_tokens[b, no] != o["tokens"][b, no]:
                dist = float("inf") if greedy else draw_distance(o, b, no, g_tokens[b, no], draw_cdf)
                if dist < draw_flag:
                    P.draw_flagged += 1
                else:
                    P.mismatches.append((b, "draw", int(o["tokens"][b, no]), int(g_tokens[b, no]),
                                         float(o["u_draw"][b]), dist))
                    continue
        if not greedy and g_px is not None:
            ell = int((~np.isnan(o["px"][b])).sum())
            if ell:
                P.max_p_err = max(P.max_p_err, float(np.max(np.abs(g_px[b, :ell] - o["px"][b, :ell]))),
                                  float(np.max(np.abs(g_qx[b, :ell] - o["qx"][b, :ell]))))
            if g_mass is not None and not flagged:
                P.max_mass_err = max(P.max_mass_err, abs(float(g_mass[b]) - float(o["resid_mass"][b])))
    return P


def assert_parity(P: Parity, prob: bool = True) -> None:
    """The parity bar: no unexcused disagreement, excused (flagged) positions
    below FLAG_FRACTION of all positions, and (prob) p(x), q(x) and the draw's
    total weight within PROB_TOL."""
    assert not P.mismatches, P.mismatches[:5]
    assert P.flagged <= FLAG_FRACTION * P.positions, (P.accept_flagged, P.draw_flagged, P.positions)
    if prob:
        assert P.max_p_err <= PROB_TOL, P.max_p_err
        assert P.max_mass_err <= PROB_TOL, P.max_mass_err


def gpu_verify(case: specsynth.VerifyCase, T: float | None = None, verify_len_dev=None, with_stats=True):
    """Run the CUDA path on a case; returns numpy outputs (and stats)."""
    import torch
    import speculative_decoding_verification_softmax_gb300 as sv
    T = case.T if T is None else T
    t, d, x, vl, u = to_device(case)
    if verify_len_dev is not None:
        vl = verify_len_dev
    tok, n, ws = sv.verify(t, d, x, vl, T, u if T != 0 else None)
    res = dict(tokens=tok.cpu().numpy(), accept_len=n.cpu().numpy())
    if with_stats:
        dt = sv.BF16 if case.dtype == "bf16" else sv.F32
        px, qx, mass, st = sv.verify_stats(ws, case.B, case.gamma, case.V, dt)
        res.update(px=px.cpu().numpy(), qx=qx.cpu().numpy(), mass=mass.cpu().numpy(),
                   status=st.cpu().numpy())
    res["device_status"] = sv.read_status(ws)
    torch.cuda.synchronize()
    return res
