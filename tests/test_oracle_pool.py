"""The multi-process oracle driver used by the full-size GPU parity tests
(host logic only, no GPU): the spawn pool returns, per head and tensor, the
same errors as a direct oracle call, and the summary combines them into
whole-tensor and worst-head ratios."""

import numpy as np

from oracle import attention_backward
from oracle_pool import TENSORS, run_heads, summarize


def _tasks(perturb):
    rng = np.random.default_rng(5)
    tasks, refs = [], []
    for h in range(3):
        q, k, v, g = (rng.standard_normal((70, 16)).astype(np.float32) for _ in range(4))
        ref = attention_backward(*(x.astype(np.float64) for x in (q, k, v, g)), 0.25, h % 2 == 1)
        outs = {n: getattr(ref, n)[0, 0].copy() for n in TENSORS}
        outs["dK"][3, 5] += perturb * (h + 1)  # a known error in one element per head
        tasks.append((q, k, v, g, 0.25, h % 2 == 1, outs))
        refs.append(ref)
    return tasks, refs


def test_pool_matches_direct_oracle():
    tasks, refs = _tasks(1e-3)
    per_head = run_heads(tasks, workers=2)
    assert len(per_head) == 3
    for h, e in enumerate(per_head):
        for n in TENSORS:
            diff, ref_max, finite = e[n]
            assert finite
            assert ref_max == float(np.abs(getattr(refs[h], n)).max())
            expect = 1e-3 * (h + 1) if n == "dK" else 0.0
            assert abs(diff - expect) <= 1e-12
    whole, worst = summarize(per_head)
    dk_max = max(float(np.abs(r.dK).max()) for r in refs)
    assert abs(whole["dK"] - 3e-3 / dk_max) <= 1e-12
    assert abs(worst["dK"] - max(1e-3 * (h + 1) / float(np.abs(refs[h].dK).max()) for h in range(3))) <= 1e-12
    assert whole["dQ"] == 0.0 and worst["O"] == 0.0


def test_pool_flags_non_finite_outputs():
    tasks, _ = _tasks(0.0)
    tasks[1][6]["dV"][0, 0] = np.nan
    per_head = run_heads(tasks, workers=2)
    assert not per_head[1]["dV"][2] and per_head[1]["dV"][0] == float("inf")
    assert per_head[0]["dV"][2] and per_head[2]["dV"][2]
