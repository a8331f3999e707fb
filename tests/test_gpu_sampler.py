"""Device sampler against the oracle: the hand-derived inverse-CDF fixture, greedy
ties, and thousands of draws over the 129280-token vocabulary with the same
uniform on both sides (xorshift64*)."""
import os

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden")


def undecidable(info, token: int) -> bool:
    """Draws whose token the device may legitimately choose differently.

    The device computes each p in f32 (z = l / T, exp(z - max z)): a relative error
    of at most ~2e-6 per token, independent across tokens, so a cumulative sum
    moves by about 2e-6 * sqrt(sum p^2) (taken x4).  Sums themselves are exact on
    the device.  If the top-p cut lies within that noise, or the crossing token's p
    is within 4e-6 of a different p, the kept set may differ by the crossing token
    or the one after it (in top-p order).  That changes the kept total (moving the
    target u * total by up to u times that token's probability) and moves the CDF
    boundaries of tokens after it in vocabulary order by its probability.
    """
    noise = 8e-6 * info.p_rms
    band = noise
    if info.cut_index >= 0 and (info.cut_sum_margin < noise or info.cut_gap_margin < 4e-6):
        band += info.cut_p
        first = min(i for i in (info.cut_index, info.cut_next_index) if i >= 0)
        if token >= first:
            band += info.cut_p
    return info.cdf_margin < band


def undecidable_min_p(info, token: int) -> bool:
    """As undecidable(), and a token of the top-p set whose p lies within f32 noise
    (4e-6 relative) of the min-p bound may be kept on one side and not the other:
    that moves the kept total by up to that token's p (at most min_p * max p)."""
    if info.minp_margin < 4e-6:
        return True
    return undecidable(info, token)


def workspace(n):
    import torch
    import prefill_decode_layer_gb300 as pdl
    return torch.empty(pdl.sample_workspace_bytes(n), dtype=torch.uint8, device="cuda")


def test_hand_derived_fixture_on_device():
    import torch
    import prefill_decode_layer_gb300 as pdl
    from test_oracle_pins import load_sampler_fixture
    logits, cases = load_sampler_fixture()
    lg = torch.from_numpy(logits).cuda()
    ws = workspace(len(logits))
    for T, tp, u, expect in cases:
        u24 = int(round(u * (1 << 24)))
        assert pdl.sample_u(lg, T, tp, min(u24, (1 << 24) - 1), ws) == expect, (T, tp, u)


def test_greedy_matches_argmax_and_ties_go_low():
    import torch
    import prefill_decode_layer_gb300 as pdl
    V = 129280
    ws = workspace(V)
    lg = synth.host_logits(V, 2.0, stream=3)
    lg[[777, 100000]] = lg.max() + 1.0          # exact tie at the top
    t = torch.from_numpy(lg).cuda()
    tok, st = pdl.sample(t, 0.0, 0.9, 12345, ws)
    assert tok == 777 == oracle.argmax(lg) and st == 12345
    lg2 = synth.host_logits(V, 1.0, stream=4)
    assert pdl.sample(torch.from_numpy(lg2).cuda(), -1.0, 1.0, 1, ws)[0] == int(np.argmax(lg2))


# stream 9 at (2.0, 0.7, 0.95) puts the top-p target within f32 noise of a cut boundary
# (an undecidable kept set); the other instances have clear cuts.
@pytest.mark.parametrize("sigma,T,top_p,stream", [(2.0, 0.7, 0.95, 10), (2.0, 0.7, 0.95, 9),
                                                  (1.0, 1.0, 1.0, 10), (3.0, 0.5, 0.5, 10),
                                                  (0.3, 1.3, 0.9, 10)])
def test_draws_match_oracle(sigma, T, top_p, stream):
    import torch
    import prefill_decode_layer_gb300 as pdl
    from synth import torch_weights as tw
    V = 129280
    ws = workspace(V)
    dev = tw.dev_logits(V, sigma, stream_id=stream)
    host = synth.host_logits(V, sigma, stream=stream)
    assert np.array_equal(dev.cpu().numpy(), host)
    state = 0x9E3779B97F4A7C15
    n, ambiguous = 300, 0
    for i in range(n):
        tok, new_state = pdl.sample(dev, T, top_p, state, ws)
        u, ostate = oracle.uniform(state)
        assert new_state == ostate
        otok, info = oracle.sample(host, T, top_p, u)
        if undecidable(info, otok):
            ambiguous += 1
        else:
            assert tok == otok, f"draw {i}: {tok} vs {otok} (u={u})"
        state = new_state
    assert ambiguous <= (3 * n) // 10, ambiguous   # the rest (>= 70%) matched exactly


def test_min_p_hand_derived_cases_on_device():
    """The hand-derived min-p cases of the oracle pins, on the device."""
    import torch
    import prefill_decode_layer_gb300 as pdl
    lg = np.array([np.log(8.0), np.log(4.0), np.log(2.0), 0.0, -5.0], dtype=np.float32)
    t = torch.from_numpy(lg).cuda()
    ws = workspace(len(lg))
    for mp, tp, u, expect in [(0.3, 1.0, 0.5, 0), (0.3, 1.0, 0.9, 1), (0.2, 1.0, 0.95, 2),
                              (0.1, 0.6, 0.9, 1), (0.1, 1.0, 0.99, 3), (1.0, 1.0, 0.999, 0),
                              (0.0005, 1.0, 0.9999, 4), (0.001, 1.0, 0.9999, 3)]:
        u24 = int(round(u * (1 << 24)))
        assert pdl.sample_u(t, 1.0, tp, u24, ws, min_p=mp) == expect, (mp, tp, u)
    assert pdl.sample_u(t, 1.0, 1.0, 5, ws, min_p=1.5) == pdl.ds4g.EINVAL


@pytest.mark.parametrize("sigma,T,top_p,min_p", [(2.0, 0.7, 0.95, 0.05), (1.0, 1.0, 1.0, 0.2),
                                                 (3.0, 0.5, 0.9, 0.01), (0.3, 1.3, 1.0, 0.9)])
def test_min_p_draws_match_oracle(sigma, T, top_p, min_p):
    import torch
    import prefill_decode_layer_gb300 as pdl
    from synth import torch_weights as tw
    V = 129280
    ws = workspace(V)
    dev = tw.dev_logits(V, sigma, stream_id=12)
    host = synth.host_logits(V, sigma, stream=12)
    state = 0x9E3779B97F4A7C15
    n, ambiguous = 200, 0
    for i in range(n):
        tok, new_state = pdl.sample(dev, T, top_p, state, ws, min_p=min_p)
        u, ostate = oracle.uniform(state)
        assert new_state == ostate
        otok, info = oracle.sample(host, T, top_p, u, min_p=min_p)
        if undecidable_min_p(info, otok):
            ambiguous += 1
        else:
            assert tok == otok, f"draw {i}: {tok} vs {otok} (u={u})"
        state = new_state
    assert ambiguous <= (3 * n) // 10, ambiguous
