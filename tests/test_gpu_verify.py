"""Parity of the CUDA verification path with the oracle on the GPU.

Every case runs the C ABI through the Python binding on seeded synthetic
inputs and compares request by request with the fp64 oracle: accept lengths
and tokens bit-exact except at flagged near-ties, p(x), q(x) and the draw's
total weight within 1e-5 absolute.
"""
import numpy as np
import pytest

import oracle
import specsynth
from tests import _helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import speculative_decoding_verification_softmax_gb300 as sv
    sv.build()


def _run(case, T=None, vl_dev=None, o=None, **kw):
    T = case.T if T is None else T
    g = H.gpu_verify(case, T=T, verify_len_dev=vl_dev)
    if o is None:
        o = H.oracle_verify(case, T=T)
    P = H.compare(o, g["tokens"], g["accept_len"], g["px"], g["qx"], g["mass"], g["status"],
                  greedy=(T == 0), **kw)
    return g, o, P


def _report(name, P):
    print(f"\n[{name}] requests={P.requests} positions={P.positions} accept_flagged={P.accept_flagged} "
          f"draw_flagged={P.draw_flagged} max|dp|={P.max_p_err:.2e} max|dmass|={P.max_mass_err:.2e} "
          f"mismatches={P.mismatches[:5]}")


# ------------------------------------------------------------ the workloads
@pytest.mark.parametrize("name", ["tiny", "mtp_chat", "block_diffusion", "greedy"])
def test_parity_configs(name):
    case = specsynth.make_verify_case(name)
    g, o, P = _run(case)
    _report(name, P)
    assert g["device_status"] == 0
    H.assert_parity(P)


@pytest.mark.parametrize("offset", [1000, 2000])
@pytest.mark.parametrize("name", ["mtp_chat", "block_diffusion", "greedy"])
def test_parity_configs_other_seeds(name, offset):
    """The same workloads at full size on two more seed sets (every seed of
    the recipe moved by the offset): other logits, drafts and uniforms, so
    other rejection positions and draws."""
    spec = specsynth.CONFIGS[name]
    case = specsynth.make_verify_case(name, seed_logits=spec.seed_logits + offset, seed_noise=spec.seed_noise + offset,
                                      seed_tokens=spec.seed_tokens + offset,
                                      seed_uniforms=spec.seed_uniforms + offset, seed_boost=spec.seed_boost + offset)
    g, o, P = _run(case)
    _report(f"{name}+{offset}", P)
    assert g["device_status"] == 0
    H.assert_parity(P)


def test_parity_scheduled_ragged():
    """Schedule on the GPU (lengths stay on the device), then verify the
    block-diffusion logits at those ragged lengths."""
    import torch
    import speculative_decoding_verification_softmax_gb300 as sv
    conf = specsynth.make_confidences()
    cost = specsynth.COST_TABLES["Bprime"]
    vl_dev, ws = sv.schedule(torch.from_numpy(conf).cuda(), cost, specsynth.SCHED_MIN_LEN)
    assert sv.read_status(ws) == 0
    ref = oracle.sched_exact(conf, cost, specsynth.SCHED_MIN_LEN)
    vl = vl_dev.cpu().numpy()
    assert (vl == ref["verify_len"]).all()
    case = specsynth.make_verify_case("block_diffusion")
    o = H.oracle_verify(case, verify_len=vl)
    g, o, P = _run(case, vl_dev=vl_dev, o=o)
    _report("scheduled_ragged", P)
    H.assert_parity(P)


# -------------------------------------------------------------- edge cases
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [1, 2, 5, 7, 8, 9, 1001, 2047, 2048, 2049, 4097, 65537])
def test_ragged_vocabularies(dtype, V):
    case = specsynth.make_verify_case("tiny", B=6, gamma=3, V=V, dtype=dtype, seed_logits=700 + V)
    g, o, P = _run(case)
    H.assert_parity(P)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_unaligned_row_starts(dtype):
    """Rows whose byte offsets are not 16-byte aligned (V * size % 16 != 0) and a
    base pointer off a 16-byte boundary exercise the scalar head/tail paths."""
    import torch
    import speculative_decoding_verification_softmax_gb300 as sv
    case = specsynth.make_verify_case("tiny", B=5, gamma=4, V=3001, dtype=dtype)
    o = H.oracle_verify(case)
    t, d, x, vl, u = H.to_device(case)
    tb = torch.empty(t.numel() + 3, dtype=t.dtype, device="cuda")
    db = torch.empty(d.numel() + 1, dtype=d.dtype, device="cuda")
    t2 = tb[3:].view(t.shape)
    d2 = db[1:].view(d.shape)
    t2.copy_(t)
    d2.copy_(d)
    assert t2.data_ptr() % 16 != 0
    tok, n, ws = sv.verify(t2, d2, x, vl, case.T, u)
    P = H.compare(o, tok.cpu().numpy(), n.cpu().numpy())
    H.assert_parity(P, prob=False)


@pytest.mark.parametrize("gamma", [0, 1, 32])
def test_draft_depths(gamma):
    case = specsynth.make_verify_case("mtp_chat", B=8, gamma=gamma, V=4000)
    g, o, P = _run(case)
    H.assert_parity(P)
    if gamma == 0:
        assert (g["accept_len"] == 0).all()


def test_ragged_verify_lengths_including_zero():
    case = specsynth.make_verify_case("mtp_chat", B=33, gamma=8, V=5000)
    case.verify_len[:] = np.arange(33) % 9
    g, o, P = _run(case)
    H.assert_parity(P)
    assert (g["accept_len"] <= case.verify_len).all()


@pytest.mark.parametrize("dtype,V", [("bf16", 2_500_001), ("bf16", 4_300_003), ("f32", 1_500_001),
                                     ("f32", 2_200_001)])
def test_very_large_vocabularies(dtype, V):
    """More than 1024 chunks per row (round sums of the draw leave shared
    memory) and more than 2048 (chunk totals go to the workspace)."""
    case = specsynth.make_verify_case("tiny", B=4, gamma=2, V=V, dtype=dtype, seed_logits=800 + V % 97,
                                      seed_noise=801, seed_tokens=802, seed_uniforms=803)
    g, o, P = _run(case)
    _report(f"V={V} {dtype}", P)
    assert g["device_status"] == 0
    H.assert_parity(P)
    assert (o["accept_len"] < case.gamma).any()      # at least one residual draw


def test_large_batch_small_vocab():
    case = specsynth.make_verify_case("tiny", B=4096, gamma=4, V=64)
    g, o, P = _run(case)
    H.assert_parity(P)


def test_equal_rows_accept_everything():
    case = specsynth.make_verify_case("mtp_chat", B=8, V=3000)
    case.draft[:] = case.target[:, :-1]
    case.draft_tokens[:] = specsynth.gumbel_argmax(specsynth.as_f32(case.draft, case.dtype).reshape(-1, case.V),
                                                   1.0 / case.T, 5).reshape(case.B, case.gamma)
    g, o, P = _run(case)
    assert (g["accept_len"] == case.gamma).all()
    H.assert_parity(P)


def test_small_temperature_equals_greedy():
    case = specsynth.make_verify_case("tiny", B=16, V=300, dtype="bf16")
    tf = specsynth.as_f32(case.target, "bf16")
    am = tf.argmax(-1)
    srt = np.sort(tf, -1)
    ok = (srt[..., -1] - srt[..., -2]) >= 0.1
    case.draft[:] = case.target[:, :-1]
    case.draft_tokens[:] = am[:, :-1]
    case.uniforms[:] = np.minimum(case.uniforms, np.float32(1 - 1e-6))
    gs = H.gpu_verify(case, T=1e-3)
    gg = H.gpu_verify(case, T=0.0)
    keep = ok.all(axis=1)
    assert keep.sum() >= 4
    assert (gs["accept_len"][keep] == gg["accept_len"][keep]).all()
    assert (gs["tokens"][keep] == gg["tokens"][keep]).all()


def test_invalid_inputs_marked_per_request():
    import speculative_decoding_verification_softmax_gb300 as sv
    case = specsynth.make_verify_case("tiny", B=7)
    case.verify_len[1] = case.gamma + 1
    case.draft_tokens[2, 1] = -3
    case.uniforms[3, case.gamma + 1] = 1.0
    case.target[4, 2, 17] = np.nan
    case.draft[5, 0, :] = -np.inf
    case.target[6, 0, 3] = np.inf
    g, o, P = _run(case)
    H.assert_parity(P)
    assert list(g["status"]) == list(o["status"])
    assert list(o["status"]) == [0, sv.ERR_VERIFY_LEN, sv.ERR_TOKEN, sv.ERR_UNIFORM, sv.ERR_NONFINITE,
                                 sv.ERR_NONFINITE, sv.ERR_NONFINITE]
    assert (g["accept_len"][1:] == -1).all() and (g["tokens"][1:] == -1).all()
    assert g["device_status"] in (sv.ERR_VERIFY_LEN, sv.ERR_TOKEN, sv.ERR_UNIFORM, sv.ERR_NONFINITE)


@pytest.mark.parametrize("name", ["tiny", "mtp_chat"])
def test_logit_scale_beyond_fp32_is_reported(name):
    """At T > 0 the streaming pass keeps each chunk's scale max|z| * log2(e) / T
    as an fp32 integer; a row where that leaves the fp32 range (here |z| = 3e38
    at T = 1) is reported as SPEC_ERR_NONFINITE (the fp64 oracle still computes
    it), and the other requests are unaffected."""
    import speculative_decoding_verification_softmax_gb300 as sv
    case = specsynth.make_verify_case(name, B=6, V=1000)
    big = np.array([3e38, -3e38], np.float32)
    if case.dtype == "bf16":
        big = specsynth.to_bf16_bits(big)
    case.target[1, 0, 5] = big[0]      # 3e38 * log2(e) / T overflows fp32 for T <= 1
    case.draft[2, 1, :] = big[1]       # a row whose max is -3e38
    g = H.gpu_verify(case)
    o = H.oracle_verify(case)
    assert g["status"][1] == sv.ERR_NONFINITE and g["status"][2] == sv.ERR_NONFINITE
    assert g["accept_len"][1] == -1 and g["accept_len"][2] == -1
    assert g["device_status"] == sv.ERR_NONFINITE
    others = np.array([0, 3, 4, 5])
    assert (g["status"][others] == 0).all() and (o["status"][others] == 0).all()
    # the other requests against the oracle (near-ties excused as everywhere)
    sub = {k: v[others] for k, v in o.items() if isinstance(v, np.ndarray) and v.shape[:1] == (case.B,)}
    P = H.compare(sub, g["tokens"][others], g["accept_len"][others], g["px"][others], g["qx"][others],
                  g["mass"][others], g["status"][others], draw_cdf=o["_draw_cdf"])
    H.assert_parity(P)


@pytest.mark.parametrize("T", [1e-4, 1e-2, 5e-2, 5.0, 100.0, 1e4])
def test_temperature_extremes(T):
    """Parity at the ends of the temperature range, with the draft tokens drawn
    from q at that temperature (as a drafter sampling at T would).  At small T
    most probabilities underflow fp32 (about 1e-38 of the row's largest); the
    tested ones do not, because the drafted tokens are likely under q and the
    residual of a rejection sits on the target's likely tokens."""
    case = specsynth.make_verify_case("mtp_chat", B=64, V=32000, T=T)
    g, o, P = _run(case)
    _report(f"T={T:g}", P)
    assert g["device_status"] == 0
    H.assert_parity(P)


def test_masked_vocabulary_entries():
    """-inf logits (masked tokens) carry zero probability and are never drawn."""
    case = specsynth.make_verify_case("mtp_chat", B=8, V=2000)
    case.target[:, :, 1000:] = specsynth.to_bf16_bits(np.array([-np.inf]))[0]
    case.draft[:, :, 1500:] = specsynth.to_bf16_bits(np.array([-np.inf]))[0]
    case.draft_tokens[:] = np.minimum(case.draft_tokens, 1499)
    g, o, P = _run(case)
    H.assert_parity(P)
    valid = g["accept_len"] >= 0
    drawn = g["tokens"][valid, :][np.arange(valid.sum()), g["accept_len"][valid]]
    assert (drawn < 1000).all()


def test_repeated_calls_are_deterministic():
    case = specsynth.make_verify_case("mtp_chat", B=16, V=32000)
    a = H.gpu_verify(case)
    b = H.gpu_verify(case)
    assert (a["tokens"] == b["tokens"]).all() and (a["accept_len"] == b["accept_len"]).all()
    assert np.array_equal(a["px"], b["px"], equal_nan=True)


def test_wrappers_reject_mismatched_inputs():
    """The binding checks dtype, shape and device of every tensor against
    (B, gamma, V) before calling the library, for spec_verify and
    spec_verify_static alike: a draft in another dtype or a short token,
    length or uniform array would otherwise be read out of bounds."""
    import torch
    import speculative_decoding_verification_softmax_gb300 as sv
    case = specsynth.make_verify_case("mtp_chat", B=4, V=1000)
    t, d, x, vl, u = H.to_device(case)
    bad = {
        "draft dtype": dict(d=d.float()),
        "draft shape": dict(d=d[:, :-1].contiguous()),
        "tokens dtype": dict(x=x.long()),
        "tokens shape": dict(x=x[:-1].contiguous()),
        "verify_len shape": dict(vl=vl[:-1].contiguous()),
        "uniforms shape": dict(u=u[:, :-1].contiguous()),
        "uniforms missing": dict(u=None),
        "tokens on the host": dict(x=x.cpu()),
        "draft not contiguous": dict(d=d.transpose(0, 1).contiguous().transpose(0, 1)),
    }
    for fn in (lambda a: sv.verify(a["t"], a["d"], a["x"], a["vl"], case.T, a["u"]),
               lambda a: sv.verify_static(a["t"], a["d"], a["x"], a["vl"], case.T, a["u"])):
        for what, over in bad.items():
            args = {**dict(t=t, d=d, x=x, vl=vl, u=u), **over}
            with pytest.raises((TypeError, ValueError)):
                fn(args)
        fn(dict(t=t, d=d, x=x, vl=vl, u=u))   # the well-formed call still runs
    torch.cuda.synchronize()



@pytest.mark.parametrize("u_draw", [0.0, float(np.nextafter(np.float32(1.0), np.float32(0.0)))])
@pytest.mark.parametrize("name", ["mtp_chat", "block_diffusion"])
def test_draws_at_the_ends_of_the_cdf(name, u_draw):
    """Residual and bonus draws with u = 0 (the first bin with positive
    weight: the CDF test is strict) and u = 1 - 2^-24 (the last bins, where
    rounding of the prefix sums may leave no bin above u * W and the draw
    takes the last bin with positive weight): parity with the oracle."""
    kw = dict(B=16) if name == "block_diffusion" else {}
    case = specsynth.make_verify_case(name, **kw)
    case.uniforms[:, case.gamma:] = np.float32(u_draw)
    g, o, P = _run(case)
    _report(f"{name} u={u_draw:.8f}", P)
    assert g["device_status"] == 0
    H.assert_parity(P)
