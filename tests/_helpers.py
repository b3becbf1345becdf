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
#   a drawn token may differ only where u lies within DRAW_FLAG of an edge of
#   the oracle's chosen bin (normalised CDF units);
#   p(x), q(x) and the draw's total weight agree within PROB_TOL absolute.
ACCEPT_FLAG = 1e-5
DRAW_FLAG = 1e-5
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
    return out


def to_device(case: specsynth.VerifyCase, device="cuda"):
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


def compare(o: dict, g_tokens, g_len, g_px=None, g_qx=None, g_mass=None, g_status=None,
            greedy=False, draw_flag=DRAW_FLAG, accept_flag=ACCEPT_FLAG) -> Parity:
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
                u, lo, hi = o["u_draw"][b], o["cdf_lo"][b], o["cdf_hi"][b]
                if not greedy and min(u - lo, hi - u) < draw_flag:
                    P.draw_flagged += 1
                else:
                    P.mismatches.append((b, "draw", int(o["tokens"][b, no]), int(g_tokens[b, no]),
                                         float(u), float(lo), float(hi)))
                    continue
        if not greedy and g_px is not None:
            ell = int((~np.isnan(o["px"][b])).sum())
            if ell:
                P.max_p_err = max(P.max_p_err, float(np.max(np.abs(g_px[b, :ell] - o["px"][b, :ell]))),
                                  float(np.max(np.abs(g_qx[b, :ell] - o["qx"][b, :ell]))))
            if g_mass is not None and not flagged:
                P.max_mass_err = max(P.max_mass_err, abs(float(g_mass[b]) - float(o["resid_mass"][b])))
    return P


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
