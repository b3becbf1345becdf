"""Calls on different CUDA streams, each with its own workspace, are
independent: interleaved launches give exactly the results of the same calls
run one at a time."""
import numpy as np
import pytest

import specsynth
from tests import _helpers as H

pytestmark = pytest.mark.gpu


def test_interleaved_streams_match_sequential():
    import torch
    import speculative_decoding_verification_softmax_gb300 as sv
    sv.build()
    cases = [specsynth.make_verify_case("tiny", B=16, V=20000),
             specsynth.make_verify_case("mtp_chat", B=16, V=32000),
             specsynth.make_verify_case("greedy", B=8, V=30011)]
    dev = [H.to_device(c) for c in cases]
    conf = torch.from_numpy(specsynth.make_confidences(64, 16, seed=31)).cuda()
    cost = specsynth.COST_TABLES["Bprime"]

    def run(i, stream=None):
        c = cases[i]
        t, d, x, vl, u = dev[i]
        tok, n, ws = sv.verify(t, d, x, vl, c.T, u if c.T != 0 else None, stream=stream)
        return tok, n, ws

    seq = []
    for i in range(len(cases)):
        tok, n, ws = run(i)
        torch.cuda.synchronize()
        seq.append((tok.cpu().numpy(), n.cpu().numpy()))
    vseq, _ = sv.schedule(conf, cost, 1)
    vseq = vseq.cpu().numpy()

    streams = [torch.cuda.Stream() for _ in range(4)]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    outs = []
    for rep in range(5):
        for i, s in enumerate(streams[:3]):
            with torch.cuda.stream(s):
                outs.append((i, run(i, s)))
        with torch.cuda.stream(streams[3]):
            outs.append((-1, sv.schedule(conf, cost, 1, stream=streams[3])))
    torch.cuda.synchronize()
    for i, res in outs:
        if i < 0:
            assert np.array_equal(res[0].cpu().numpy(), vseq)
            assert sv.read_status(res[1]) == 0
        else:
            tok, n, ws = res
            assert np.array_equal(tok.cpu().numpy(), seq[i][0]) and np.array_equal(n.cpu().numpy(), seq[i][1])
            assert sv.read_status(ws) == 0


def test_inputs_written_just_before_the_call_are_seen():
    """Stream order with the programmatic dependent launches: kernels that
    rewrite the inputs (verify lengths, uniforms, logits) right before each
    call on the same stream, with no host synchronisation, are seen by that
    call; each call matches the same call run alone."""
    import torch
    import speculative_decoding_verification_softmax_gb300 as sv
    sv.build()
    case = specsynth.make_verify_case("mtp_chat", B=16, V=32000)
    t, d, x, vl, u = H.to_device(case)
    rng = np.random.default_rng(11)
    vls = [torch.from_numpy(rng.integers(0, case.gamma + 1, case.B).astype(np.int32)).cuda() for _ in range(6)]
    us = [torch.from_numpy(rng.uniform(0, 1, u.shape).astype(np.float32)).cuda() for _ in range(6)]
    scales = [1.0, 0.5, 2.0, 1.0, 0.25, 1.5]
    t0, d0 = t.clone(), d.clone()
    ws = sv.alloc_verify_workspace(case.B, case.gamma, case.V, sv.BF16)

    # back to back: the inputs are rewritten in place by torch kernels before each call
    outs = []
    for k in range(6):
        vl.copy_(vls[k])
        u.copy_(us[k])
        torch.mul(t0, scales[k], out=t)
        torch.mul(d0, scales[k], out=d)
        tok, n, _ = sv.verify(t, d, x, vl, case.T, u, workspace=ws)
        outs.append((tok.clone(), n.clone()))
    torch.cuda.synchronize()

    for k in range(6):
        tk, dk = (t0 * scales[k]).contiguous(), (d0 * scales[k]).contiguous()
        torch.cuda.synchronize()
        tok, n, _ = sv.verify(tk, dk, x, vls[k].clone(), case.T, us[k].clone())
        torch.cuda.synchronize()
        assert (tok.cpu().numpy() == outs[k][0].cpu().numpy()).all(), k
        assert (n.cpu().numpy() == outs[k][1].cpu().numpy()).all(), k
    assert sv.read_status(ws) == 0
