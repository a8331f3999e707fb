"""Router top-k on exact ties, checked against the kernels' own scores.

Router rows are duplicated (and negated) so that the selected set always holds
experts with bit-identical scores.  The selection must then equal a stable sort of
the scores the kernel computed (larger score first, equal scores to the lower
expert id), and the gate weights the softmax over the selected scores.  No
tolerance is involved in the ids, so the check is exact at any size."""
import numpy as np
import pytest

import synth
from helpers import DECODE_KERNELS, to_np

pytestmark = pytest.mark.gpu

# (shape, groups of rows made identical: each group copies a source row scaled by a
# power of two; a negated copy of every group puts one of the two near the top)
CASES = {
    "layer": (synth.LAYER, [(11, 64.0, [3, 40]), (150, 32.0, [12, 150, 151])]),
    "tiny": (synth.TINY, [(7, 64.0, [3, 9])]),
}


def stable_topk(scores, k):
    s = np.where(np.isnan(scores), -np.inf, scores.astype(np.float64))
    order = sorted(range(len(s)), key=lambda e: (-s[e], e))
    return order[:k]


@pytest.mark.parametrize("kernel", DECODE_KERNELS, ids=["persistent", "staged"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_router_ties_go_to_lower_id(case, kernel):
    import torch
    import prefill_decode_layer_gb300 as pdl
    from synth import torch_weights as tw
    shape, groups = CASES[case]
    E, K = shape.n_experts, shape.top_k
    emb, lm, layers = tw.dev_model(shape, 0)
    r = layers[0]["w_router"]
    used = set()
    neg_base = E - 1
    for src, scale, rows in groups:
        v = (r[src].float() * scale).to(r.dtype)
        for row in rows:
            r[row] = v
            used.add(row)
        for j in range(len(rows)):   # the negated group, on rows from the top down
            while neg_base in used:
                neg_base -= 1
            r[neg_base] = -v
            used.add(neg_base)
    torch.cuda.synchronize()
    gm = pdl.Model(shape, emb, lm, layers, decode_kernel=kernel)
    sess = pdl.Session(gm, 64)
    toks = synth.host_tokens(6, shape.vocab, stream=21)
    tied_steps = 0
    for t in toks:
        assert sess.decode_layers(int(t)) == 0
        torch.cuda.synchronize()
        sc = to_np(sess.debug("scores", E)).astype(np.float32)
        ids, w = sess.router(0)
        want = stable_topk(sc, K)
        assert list(ids) == want, f"{list(ids)} vs {want} (scores {sc[want]})"
        sel = sc[want].astype(np.float64)
        ew = np.exp(sel - sel[0])
        ew /= ew.sum()
        assert np.max(np.abs(np.asarray(w, dtype=np.float64) - ew)) <= 1e-6
        tied_steps += any(sc[want[i]] == sc[want[i + 1]] for i in range(K - 1))
    # a scaled group outranks the unscaled rows unless its source score is near zero
    assert tied_steps >= len(toks) // 2
    assert sess.status() == 0
