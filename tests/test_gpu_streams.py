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
