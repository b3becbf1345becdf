"""Out-of-bounds writes: every output and workspace buffer handed to the library
is a view into a larger buffer whose guard bands before and after are filled
with a canary pattern; after each call the bands must be untouched.  Covers
the padded and packed verification (T > 0 and greedy, ragged and invalid
requests, unaligned vocabularies), the diagnostics copy, the packing and every
scheduler mode."""
import numpy as np
import pytest

import specsynth
from tests import _helpers as H

pytestmark = pytest.mark.gpu

GUARD = 4096            # bytes on each side
CANARY = 0x5A


def _guarded(torch, nbytes, dev):
    """A uint8 buffer with guard bands; returns (whole, inner view)."""
    whole = torch.full((nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device=dev)
    return whole, whole[GUARD:GUARD + nbytes]


def _typed(torch, shape, dtype, dev, bufs):
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    whole, inner = _guarded(torch, n, dev)
    bufs.append(whole)
    return inner.view(dtype).view(*shape)


def _check(torch, bufs):
    torch.cuda.synchronize()
    for w in bufs:
        h = w.cpu().numpy()
        assert (h[:GUARD] == CANARY).all(), "write before the buffer"
        assert (h[-GUARD:] == CANARY).all(), "write after the buffer"


def _case(name, **kw):
    case = specsynth.make_verify_case(name, **kw)
    rng = np.random.default_rng(7)
    vl = rng.integers(0, case.gamma + 1, case.B).astype(np.int32)
    vl[0] = case.gamma + 3      # invalid length
    vl[1] = 0
    case.verify_len[:] = vl
    return case


@pytest.mark.parametrize("name,kw", [("mtp_chat", dict(B=12, V=3001)), ("greedy", dict(B=9, V=2049)),
                                     ("tiny", dict(B=6, V=1001))])
def test_verify_writes_stay_in_bounds(name, kw):
    import torch
    import speculative_decoding_verification_softmax_gb300 as sv
    case = _case(name, **kw)
    dev = torch.device("cuda", 0)
    t, d, x, vl, u = H.to_device(case, dev)
    B, g, V = case.B, case.gamma, case.V
    dt = sv.BF16 if case.dtype == "bf16" else sv.F32
    bufs = []
    ot = _typed(torch, (B, g + 1), torch.int32, dev, bufs)
    on = _typed(torch, (B,), torch.int32, dev, bufs)
    ws = _typed(torch, (sv.verify_workspace_bytes(B, g, V, dt),), torch.uint8, dev, bufs)
    sv.verify(t, d, x, vl, case.T, u if case.T != 0 else None, out_tokens=ot, out_accept_len=on, workspace=ws)
    _check(torch, bufs)
    assert on.cpu().numpy()[0] == -1
    # the diagnostics copy into guarded outputs
    px = _typed(torch, (B, g), torch.float64, dev, bufs)
    qx = _typed(torch, (B, g), torch.float64, dev, bufs)
    mass = _typed(torch, (B,), torch.float64, dev, bufs)
    st = _typed(torch, (B,), torch.int32, dev, bufs)
    L = sv.lib()
    rc = L.spec_verify_stats(sv._ptr(ws), ws.numel(), B, g, V, dt, sv._ptr(px), sv._ptr(qx), sv._ptr(mass),
                             sv._ptr(st), sv._stream_handle(None))
    assert rc == 0
    _check(torch, bufs)


def test_packed_verify_and_packing_stay_in_bounds():
    import torch
    import speculative_decoding_verification_softmax_gb300 as sv
    case = _case("mtp_chat", B=10, V=3001)
    dev = torch.device("cuda", 0)
    t, d, x, vl, u = H.to_device(case, dev)
    B, g, V = case.B, case.gamma, case.V
    bufs = []
    tr = _typed(torch, (B,), torch.int32, dev, bufs)
    dr = _typed(torch, (B,), torch.int32, dev, bufs)
    tot = _typed(torch, (2,), torch.int32, dev, bufs)
    sv.pack_rows(vl, g, target_row=tr, draft_row=dr, totals=tot)
    _check(torch, bufs)
    vl_h = case.verify_len
    ok = (vl_h >= 0) & (vl_h <= g)
    ti = np.concatenate([b * (g + 1) + np.arange(vl_h[b] + 1) for b in range(B) if ok[b]])
    di = np.concatenate([b * g + np.arange(vl_h[b]) for b in range(B) if ok[b]])
    tp = t.view(B * (g + 1), V)[torch.from_numpy(ti).to(dev)].contiguous()
    dp = d.view(B * g, V)[torch.from_numpy(di).to(dev)].contiguous()
    ot = _typed(torch, (B, g + 1), torch.int32, dev, bufs)
    on = _typed(torch, (B,), torch.int32, dev, bufs)
    ws = _typed(torch, (sv.verify_workspace_bytes(B, g, V, sv.BF16),), torch.uint8, dev, bufs)
    sv.verify_packed(tp, dp, tr, dr, x, vl, case.T, u, out_tokens=ot, out_accept_len=on, workspace=ws)
    _check(torch, bufs)
    ref_t, ref_n, _ = sv.verify(t, d, x, vl, case.T, u)
    assert (ref_t.cpu().numpy() == ot.cpu().numpy()).all()
    assert (ref_n.cpu().numpy() == on.cpu().numpy()).all()


@pytest.mark.parametrize("B,gamma", [(5, 3), (64, 16), (200, 32)])
def test_schedulers_stay_in_bounds(B, gamma):
    import torch
    import speculative_decoding_verification_softmax_gb300 as sv
    dev = torch.device("cuda", 0)
    conf = torch.from_numpy(specsynth.make_confidences(B, gamma, seed=900 + B)).to(dev)
    cost = specsynth.COST_TABLES["Bprime"]
    sts = np.linspace(0.8, 1.6, gamma).astype(np.float32)
    bufs = []
    runs = [
        lambda out, ws: sv.schedule(conf, cost, 1, sv.SCHED_EXACT, out_verify_len=out, workspace=ws),
        lambda out, ws: sv.schedule(conf, cost, 0, sv.SCHED_ALGORITHM1, out_verify_len=out, workspace=ws),
        lambda out, ws: sv.schedule(conf, ([0.25, 0.5, 1.0], [10.0, 13.0, 19.0]), 1, sv.SCHED_DCUT,
                                    out_verify_len=out, workspace=ws),
        lambda out, ws: sv.schedule(conf, cost, 1, sv.SCHED_EXACT, sts=sts, out_verify_len=out, workspace=ws),
        lambda out, ws: sv.schedule_static(conf, 0.6, gamma, 1, out_verify_len=out, workspace=ws),
        lambda out, ws: sv.schedule_static(conf, 0.6, gamma, 0, sts=sts, out_verify_len=out, workspace=ws),
    ]
    for run in runs:
        out = _typed(torch, (B,), torch.int32, dev, bufs)
        ws = _typed(torch, (sv.lib().spec_schedule_workspace_bytes(B, gamma),), torch.uint8, dev, bufs)
        run(out, ws)
        _check(torch, bufs)
        v = out.cpu().numpy()
        assert ((v >= 0) & (v <= gamma)).all()
