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


def undecided_band(info, token: int) -> float:
    """Width (in units of the kept total) of the band around u * total in which the
    device may legitimately choose a different token; 0 when the draw is decided.

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
    return band if info.cdf_margin < band else 0.0


def undecided_band_min_p(info, token: int, min_p: float) -> float:
    """As undecided_band(); besides, a token of the top-p set whose p lies within f32
    noise (4e-6 relative) of the min-p bound may be kept on one side and not the
    other, which moves the kept total and the CDF by up to that token's p (at most
    min_p times the largest p, so at most min_p of the kept total)."""
    if info.minp_margin < 4e-6:
        return 8e-6 * info.p_rms + 2.0 * min_p
    return undecided_band(info, token)


def within_band(host, T, top_p, u, band, tok, info, min_p=0.0) -> bool:
    """The device's token of an undecided draw lies among the tokens the oracle
    draws for uniforms in [u - band, u + band] (the walk is monotone in u for a
    fixed kept set), or is the crossing token or the one after it in top-p order."""
    if tok in (info.cut_index, info.cut_next_index):
        return True
    lo = oracle.sample(host, T, top_p, max(0.0, u - band), min_p=min_p)[0]
    hi = oracle.sample(host, T, top_p, min(1.0 - 2.0 ** -53, u + band), min_p=min_p)[0]
    return lo <= tok <= hi


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
# (an undecidable kept set): 66 of its 300 draws are undecided.  The other instances
# have clear cuts; their undecided draws are those whose u * total falls within the
# f32 noise of a CDF boundary: 0 of 300, except 5 of 300 for top-p = 1 over the flat
# sigma = 1 logits (129280 tokens of p ~ 8e-6 each, so the boundaries are dense).
# The limits are those counts plus one or two draws.
@pytest.mark.parametrize("sigma,T,top_p,stream,max_undecided",
                         [(2.0, 0.7, 0.95, 10, 2), (2.0, 0.7, 0.95, 9, 90),
                          (1.0, 1.0, 1.0, 10, 7), (3.0, 0.5, 0.5, 10, 2),
                          (0.3, 1.3, 0.9, 10, 2)])
def test_draws_match_oracle(sigma, T, top_p, stream, max_undecided):
    import torch
    import prefill_decode_layer_gb300 as pdl
    from synth import torch_weights as tw
    V = 129280
    ws = workspace(V)
    dev = tw.dev_logits(V, sigma, stream_id=stream)
    host = synth.host_logits(V, sigma, stream=stream)
    assert np.array_equal(dev.cpu().numpy(), host)
    state = 0x9E3779B97F4A7C15
    n, undecided, differ = 300, 0, 0
    for i in range(n):
        tok, new_state = pdl.sample(dev, T, top_p, state, ws)
        u, ostate = oracle.uniform(state)
        assert new_state == ostate
        otok, info = oracle.sample(host, T, top_p, u)
        band = undecided_band(info, otok)
        if band > 0.0:
            undecided += 1
            differ += tok != otok
            assert within_band(host, T, top_p, u, band, tok, info), f"draw {i}: {tok} vs {otok}"
        else:
            assert tok == otok, f"draw {i}: {tok} vs {otok} (u={u})"
        state = new_state
    print(f"sigma={sigma} T={T} top_p={top_p} stream={stream}: {undecided} of {n} draws "
          f"undecided, {differ} of them differ")
    assert undecided <= max_undecided, undecided


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


# Undecided counts of these instances (oracle only): 9 of 200 for the first (tokens
# of the top-p set within f32 noise of the min-p bound), 0 for the others.
@pytest.mark.parametrize("sigma,T,top_p,min_p,max_undecided",
                         [(2.0, 0.7, 0.95, 0.05, 10), (1.0, 1.0, 1.0, 0.2, 2),
                          (3.0, 0.5, 0.9, 0.01, 2), (0.3, 1.3, 1.0, 0.9, 2)])
def test_min_p_draws_match_oracle(sigma, T, top_p, min_p, max_undecided):
    import torch
    import prefill_decode_layer_gb300 as pdl
    from synth import torch_weights as tw
    V = 129280
    ws = workspace(V)
    dev = tw.dev_logits(V, sigma, stream_id=12)
    host = synth.host_logits(V, sigma, stream=12)
    state = 0x9E3779B97F4A7C15
    n, undecided, differ = 200, 0, 0
    for i in range(n):
        tok, new_state = pdl.sample(dev, T, top_p, state, ws, min_p=min_p)
        u, ostate = oracle.uniform(state)
        assert new_state == ostate
        otok, info = oracle.sample(host, T, top_p, u, min_p=min_p)
        band = undecided_band_min_p(info, otok, min_p)
        if band > 0.0:
            undecided += 1
            differ += tok != otok
            assert within_band(host, T, top_p, u, band, tok, info, min_p), \
                f"draw {i}: {tok} vs {otok}"
        else:
            assert tok == otok, f"draw {i}: {tok} vs {otok} (u={u})"
        state = new_state
    print(f"sigma={sigma} T={T} top_p={top_p} min_p={min_p}: {undecided} of {n} draws "
          f"undecided, {differ} of them differ")
    assert undecided <= max_undecided, undecided


# Vocabularies above 256 chunks of 1024 tokens (the one-launch form reads one chunk
# sum per thread in its draw) take the per-pass kernels instead; 700000 tokens
# exercise them.  Undecided draws (oracle only): 2 and 7 of 100; the flat sigma = 1
# logits over 700000 tokens have dense CDF boundaries.
@pytest.mark.parametrize("sigma,T,top_p,max_undecided", [(2.0, 0.7, 0.95, 4), (1.0, 1.0, 1.0, 9)])
def test_large_vocabulary_draws_match_oracle(sigma, T, top_p, max_undecided):
    import torch
    import prefill_decode_layer_gb300 as pdl
    from synth import torch_weights as tw
    V = 700000
    ws = workspace(V)
    dev = tw.dev_logits(V, sigma, stream_id=13)
    host = synth.host_logits(V, sigma, stream=13)
    state = 0x9E3779B97F4A7C15
    undecided = 0
    for i in range(100):
        tok, new_state = pdl.sample(dev, T, top_p, state, ws)
        u, _ = oracle.uniform(state)
        otok, info = oracle.sample(host, T, top_p, u)
        band = undecided_band(info, otok)
        if band > 0.0:
            undecided += 1
            assert within_band(host, T, top_p, u, band, tok, info), f"draw {i}"
        else:
            assert tok == otok, f"draw {i}: {tok} vs {otok}"
        state = new_state
    print(f"V={V} sigma={sigma} T={T} top_p={top_p}: {undecided} of 100 draws undecided")
    assert undecided <= max_undecided, undecided
    assert pdl.sample(dev, 0.0, 1.0, None, ws)[0] == oracle.argmax(host)
