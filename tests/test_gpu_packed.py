"""Verification on the packed logit layout ("AngelSpec" §4.2, "Packing and
correctness": the kept prefixes form one dense verification batch).

The packed call must give the oracle's results (the oracle reads the same
logical rows from the padded layout) and exactly the padded call's results:
only the addresses of the rows differ, not the arithmetic."""
import numpy as np
import pytest

import oracle
import specsynth
from tests import _helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_softmax_gb300 as m
    m.build()
    return m


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _logits_dev(arr, dtype):
    import torch
    if dtype == "bf16":
        return _dev(arr.view(np.int16)).view(torch.bfloat16)
    return _dev(arr)


def _pack(case, vl, trow, drow, Kt, Kd, fill):
    """Host gather of the kept rows of a padded case into [Kt, V] / [Kd, V]
    arrays at the given row index; rows not written hold `fill`."""
    V = case.V
    tp = np.full((Kt, V), fill, case.target.dtype)
    dp = np.full((max(Kd, 1), V), fill, case.draft.dtype)
    for b in range(case.B):
        ell = int(vl[b])
        if 0 <= ell <= case.gamma:
            tp[trow[b]:trow[b] + ell + 1] = case.target[b, :ell + 1]
            if ell:
                dp[drow[b]:drow[b] + ell] = case.draft[b, :ell]
    return tp, dp


def _nan_fill(dtype):
    return specsynth.to_bf16_bits(np.array([np.nan]))[0] if dtype == "bf16" else np.float32(np.nan)


def _ragged(case, seed, lo=0):
    rng = np.random.default_rng(seed)
    return rng.integers(lo, case.gamma + 1, case.B).astype(np.int32)


def _run_packed(sv, case, vl, tp, dp, trow, drow):
    T = case.T
    tok, n, ws = sv.verify_packed(_logits_dev(tp, case.dtype), _logits_dev(dp, case.dtype) if T != 0 else None,
                                  _dev(trow.astype(np.int32)), _dev(drow.astype(np.int32)) if T != 0 else None,
                                  _dev(case.draft_tokens), _dev(vl), T, _dev(case.uniforms) if T != 0 else None)
    dt = sv.BF16 if case.dtype == "bf16" else sv.F32
    px, qx, mass, st = sv.verify_stats(ws, case.B, case.gamma, case.V, dt)
    return dict(tokens=tok.cpu().numpy(), accept_len=n.cpu().numpy(), px=px.cpu().numpy(), qx=qx.cpu().numpy(),
                mass=mass.cpu().numpy(), status=st.cpu().numpy(), device_status=sv.read_status(ws))


def test_pack_rows_matches_oracle(sv):
    rng = np.random.default_rng(8)
    for trial in range(40):
        B, gamma = int(rng.integers(1, 4097)), int(rng.integers(0, 33))
        vl = rng.integers(-2, gamma + 3, B).astype(np.int32)   # some out of range
        tr, dr, tot = sv.pack_rows(_dev(vl), gamma)
        r = oracle.pack_rows(vl, gamma)
        assert (tr.cpu().numpy() == r["target_row"]).all()
        assert (dr.cpu().numpy() == r["draft_row"]).all()
        assert list(tot.cpu().numpy()) == [r["K_target"], r["K_draft"]]


@pytest.mark.parametrize("name", ["tiny", "mtp_chat", "block_diffusion", "greedy"])
def test_dense_packed_equals_padded_and_oracle(sv, name):
    case = specsynth.make_verify_case(name)
    vl = _ragged(case, 40 + len(name))
    case.verify_len[:] = vl
    r = oracle.pack_rows(vl, case.gamma)
    tp, dp = _pack(case, vl, r["target_row"], r["draft_row"], r["K_target"], r["K_draft"], 0)
    g = _run_packed(sv, case, vl, tp, dp, r["target_row"], r["draft_row"])
    pad = H.gpu_verify(case)
    for k in ("tokens", "accept_len", "status"):
        assert (g[k] == pad[k]).all(), k
    if case.T != 0:
        for k in ("px", "qx", "mass"):
            np.testing.assert_array_equal(g[k], pad[k])
    o = H.oracle_verify(case)
    P = H.compare(o, g["tokens"], g["accept_len"], g["px"], g["qx"], g["mass"], g["status"], greedy=case.T == 0)
    assert g["device_status"] == 0
    H.assert_parity(P)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_shuffled_placement_with_gap_rows(sv, dtype):
    """Requests placed in a random order with unused rows between them; the
    unused rows hold NaN, so reading one would mark its request invalid."""
    case = specsynth.make_verify_case("mtp_chat", B=12, V=4096, dtype=dtype)
    vl = _ragged(case, 5)
    case.verify_len[:] = vl
    rng = np.random.default_rng(6)
    order = rng.permutation(case.B)
    trow, drow = np.zeros(case.B, np.int64), np.zeros(case.B, np.int64)
    t = d = 0
    for b in order:
        t += int(rng.integers(0, 3))
        d += int(rng.integers(0, 3))
        trow[b], drow[b] = t, d
        t += vl[b] + 1
        d += vl[b]
    tp, dp = _pack(case, vl, trow, drow, t + 2, d + 2, _nan_fill(dtype))
    g = _run_packed(sv, case, vl, tp, dp, trow, drow)
    pad = H.gpu_verify(case)
    assert g["device_status"] == 0
    for k in ("tokens", "accept_len", "px", "qx", "mass"):
        np.testing.assert_array_equal(g[k], pad[k])


def test_unaligned_packed_base(sv):
    """Packed arrays that start off a 16-byte boundary take the general
    (head/tail) streaming variant and give the same results."""
    import torch
    case = specsynth.make_verify_case("tiny", B=6, V=3001, dtype="bf16")
    vl = _ragged(case, 9)
    case.verify_len[:] = vl
    r = oracle.pack_rows(vl, case.gamma)
    tp, dp = _pack(case, vl, r["target_row"], r["draft_row"], r["K_target"], r["K_draft"], 0)
    t = _logits_dev(tp, "bf16")
    d = _logits_dev(dp, "bf16")
    tb = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
    t2 = tb[1:].view(t.shape)
    t2.copy_(t)
    assert t2.data_ptr() % 16 != 0
    tok, n, ws = sv.verify_packed(t2, d, _dev(r["target_row"]), _dev(r["draft_row"]), _dev(case.draft_tokens),
                                  _dev(vl), case.T, _dev(case.uniforms))
    pad = H.gpu_verify(case)
    assert (tok.cpu().numpy() == pad["tokens"]).all() and (n.cpu().numpy() == pad["accept_len"]).all()


def test_row_index_out_of_range_marks_the_request(sv):
    case = specsynth.make_verify_case("tiny", B=6)
    vl = np.array([4, 2, 3, 0, 1, 4], np.int32)
    case.verify_len[:] = vl
    r = oracle.pack_rows(vl, case.gamma)
    trow, drow = r["target_row"].copy(), r["draft_row"].copy()
    tp, dp = _pack(case, vl, trow, drow, r["K_target"], r["K_draft"], 0)
    trow[1] = r["K_target"] - 2      # 3 rows from K-2: one past the end
    drow[4] = -1
    trow[5] = -7
    g = _run_packed(sv, case, vl, tp, dp, trow, drow)
    pad = H.gpu_verify(case)
    bad = [1, 4, 5]
    assert list(g["status"][bad]) == [sv.ERR_ROW_INDEX] * 3
    assert (g["accept_len"][bad] == -1).all() and (g["tokens"][bad] == -1).all()
    good = [0, 2, 3]
    assert (g["tokens"][good] == pad["tokens"][good]).all()
    assert g["device_status"] == sv.ERR_ROW_INDEX


def test_schedule_pack_verify_in_one_graph(sv):
    """D-cut schedule, dense packing and packed verification: three calls, no
    host synchronisation, captured in one CUDA graph and replayed."""
    import torch
    case = specsynth.make_verify_case("mtp_chat", B=16, V=8192)
    conf = _dev(specsynth.make_confidences(16, case.gamma, seed=21))
    ratios, costs = [0.25, 0.5, 0.75, 1.0], [6.0, 7.0, 8.5, 10.0]
    vl, sws = sv.schedule(conf, (ratios, costs), 0, sv.SCHED_DCUT)
    tr, dr, tot = sv.pack_rows(vl, case.gamma)
    torch.cuda.synchronize()
    vl_h, tr_h, dr_h = vl.cpu().numpy(), tr.cpu().numpy(), dr.cpu().numpy()
    Kt, Kd = [int(v) for v in tot.cpu().numpy()]
    case.verify_len[:] = vl_h
    tp, dp = _pack(case, vl_h, tr_h, dr_h, Kt, Kd, 0)
    t, d = _logits_dev(tp, case.dtype), _logits_dev(dp, case.dtype)
    x, u = _dev(case.draft_tokens), _dev(case.uniforms)
    out_t = torch.empty((case.B, case.gamma + 1), dtype=torch.int32, device="cuda")
    out_n = torch.empty((case.B,), dtype=torch.int32, device="cuda")
    ws = sv.alloc_verify_workspace(case.B, case.gamma, case.V, sv.BF16)

    def step():
        sv.schedule(conf, (ratios, costs), 0, sv.SCHED_DCUT, out_verify_len=vl, workspace=sws)
        sv.pack_rows(vl, case.gamma, target_row=tr, draft_row=dr, totals=tot)
        sv.verify_packed(t, d, tr, dr, x, vl, case.T, u, out_tokens=out_t, out_accept_len=out_n, workspace=ws)

    step()
    torch.cuda.synchronize()
    ref_t, ref_n = out_t.cpu().numpy().copy(), out_n.cpu().numpy().copy()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            step()
    torch.cuda.current_stream().wait_stream(side)
    out_t.fill_(-7)
    out_n.fill_(-7)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert (out_t.cpu().numpy() == ref_t).all() and (out_n.cpu().numpy() == ref_n).all()
    assert sv.read_status(ws) == 0 and sv.read_status(sws) == 0
    pad = H.gpu_verify(case)
    assert (ref_t == pad["tokens"]).all() and (ref_n == pad["accept_len"]).all()


@pytest.mark.parametrize("name", ["tiny", "greedy"])
def test_packed_no_drafts(sv, name):
    """gamma = 0: one target row per request, a pure draw from p (or its argmax)."""
    case = specsynth.make_verify_case(name, B=5, gamma=0, V=3000)
    vl = np.zeros(case.B, np.int32)
    r = oracle.pack_rows(vl, 0)
    assert (r["K_target"], r["K_draft"]) == (case.B, 0)
    tp, dp = _pack(case, vl, r["target_row"], r["draft_row"], r["K_target"], r["K_draft"], 0)
    g = _run_packed(sv, case, vl, tp, dp, r["target_row"], r["draft_row"])
    pad = H.gpu_verify(case)
    assert g["device_status"] == 0
    assert (g["tokens"] == pad["tokens"]).all() and (g["accept_len"] == 0).all()


@pytest.mark.parametrize("name", ["mtp_chat", "greedy"])
def test_packed_beyond_the_row_table(sv, name):
    """More compact rows than the streaming kernel's shared-memory row table
    holds (4096): the rows and their packed positions then come from the
    request prefix and the row index in global memory.  512 requests with
    ragged lengths, small vocabulary; identical to the padded call and at
    parity with the oracle."""
    case = specsynth.make_verify_case(name, B=512, gamma=16, V=520, seed_logits=910, seed_noise=911,
                                      seed_tokens=912, seed_uniforms=913)
    vl = _ragged(case, 77, lo=8)
    case.verify_len[:] = vl
    rows = int(((vl + 1) if case.T == 0 else (2 * vl + 1)).sum())
    assert rows > 4096
    r = oracle.pack_rows(vl, case.gamma)
    tp, dp = _pack(case, vl, r["target_row"], r["draft_row"], r["K_target"], r["K_draft"], 0)
    g = _run_packed(sv, case, vl, tp, dp, r["target_row"], r["draft_row"])
    pad = H.gpu_verify(case)
    for k in ("tokens", "accept_len", "status"):
        assert (g[k] == pad[k]).all(), k
    o = H.oracle_verify(case)
    P = H.compare(o, g["tokens"], g["accept_len"], g["px"], g["qx"], g["mass"], g["status"], greedy=case.T == 0)
    assert g["device_status"] == 0
    H.assert_parity(P)


@pytest.mark.parametrize("name,gamma", [("mtp_chat", 2), ("greedy", 1)])
def test_packed_row_map_read_from_global_memory(sv, name, gamma):
    """1400 requests with ragged lengths on packed logits, with the row table
    (T = 0: at most 2800 rows) and without it (T > 0: more than 4096 rows).
    Identical to the padded call and at parity with the oracle; then one
    request's target row moved past the end of the packed array is marked
    and the others are unchanged."""
    case = specsynth.make_verify_case(name, B=1400, gamma=gamma, V=520, seed_logits=920, seed_noise=921,
                                      seed_tokens=922, seed_uniforms=923)
    vl = _ragged(case, 78)
    case.verify_len[:] = vl
    r = oracle.pack_rows(vl, case.gamma)
    tp, dp = _pack(case, vl, r["target_row"], r["draft_row"], r["K_target"], r["K_draft"], 0)
    g = _run_packed(sv, case, vl, tp, dp, r["target_row"], r["draft_row"])
    pad = H.gpu_verify(case)
    for k in ("tokens", "accept_len", "status"):
        assert (g[k] == pad[k]).all(), k
    o = H.oracle_verify(case)
    P = H.compare(o, g["tokens"], g["accept_len"], g["px"], g["qx"], g["mass"], g["status"], greedy=case.T == 0)
    assert g["device_status"] == 0
    H.assert_parity(P)

    bad = int(np.flatnonzero(vl > 0)[-1])
    trow = r["target_row"].copy()
    trow[bad] = r["K_target"] - int(vl[bad])  # its last row one past the end
    g2 = _run_packed(sv, case, vl, tp, dp, trow, r["draft_row"])
    assert g2["status"][bad] == sv.ERR_ROW_INDEX and g2["accept_len"][bad] == -1
    keep = np.arange(case.B) != bad
    assert (g2["tokens"][keep] == pad["tokens"][keep]).all() and (g2["accept_len"][keep] == pad["accept_len"][keep]).all()
    assert g2["device_status"] == sv.ERR_ROW_INDEX
