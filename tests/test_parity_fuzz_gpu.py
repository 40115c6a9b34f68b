"""Seeded random configurations of the verify step on the GPU against the float64 oracle.

The hand-written parity cases follow the workloads and the edge cases one can name; this file
draws 128 configurations from a fixed seed over the whole space the C ABI accepts, so that the
combinations nobody wrote down also meet the oracle: greedy or stochastic mode, fp32 or bf16
rows, K in 1..8, vocabularies from 7 ids to 152064 (so rows of one and of many ring chunks per
CTA), ragged or full lengths, a bias set and top-F ids, cluster sizes 0 (the library's choice,
which may take the small-batch routes) to 8, the diagnostics entry point, and a few planted
invalid sequences (length out of range, an id outside the vocabulary, a uniform of 1, a NaN in a
row). The bar is the same as everywhere: bit-exact outcomes, decisions closer than 1e-6 to their
threshold flagged.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from speculative_decoding_verification_33_gb300 import api  # noqa: E402
from speculative_decoding_verification_33_gb300 import workloads as W  # noqa: E402
from tests.test_parity_gpu import check, run_gpu  # noqa: E402

VOCABS = (7, 100, 3001, 9000, 20000, 40000, 65537, 152064)


def draw_case(i: int):
    rng = np.random.default_rng([2026, i])
    greedy = rng.random() < 0.25
    K = int(rng.integers(1, 9))
    V = int(VOCABS[rng.integers(len(VOCABS))])
    B = int(rng.integers(1, 13))
    dtype = "bf16" if rng.random() < 0.6 else "f32"
    bias_k, beta, fanout = 0, 1.0, None
    if not greedy and rng.random() < 0.3:
        bias_k, beta = int(min(V, rng.integers(1, 9))), 0.5
    if not greedy and rng.random() < 0.3:
        fanout = tuple(int(f) for f in rng.integers(1, 9, size=K))
    w = W.Workload(100 + i, f"fuzz{i}", B=B, K=K, V=V, dtype=dtype,
                   mode="greedy" if greedy else "stochastic",
                   temperature=0.0 if greedy else float(rng.choice([0.6, 1.0, 1.5])),
                   sigma_t=float(rng.choice([1.0, 2.0])), sigma_d=float(rng.choice([0.3, 1.0])),
                   zipf=bool(rng.random() < 0.5), ragged=bool(rng.random() < 0.5), beta=beta,
                   bias_k=bias_k, fanout=fanout)
    min_c = (V + 65535) // 65536  # a CTA's slice holds at most 65536 ids
    cluster = int(rng.choice([c for c in (0, 1, 2, 4, 8) if c == 0 or c >= min_c]))
    debug = bool(rng.random() < 0.25)
    n_plant = int(rng.integers(0, 3)) if B >= 3 else 0  # keep valid sequences in every batch
    plant = [int(x) for x in rng.integers(0, 5, size=n_plant)]
    return w, cluster, debug, plant


CASES = [draw_case(i) for i in range(128)]


def plant_invalid(d, w, kinds, rng):
    """0: length out of range, 1: id outside the vocabulary, 2: final uniform of 1, 3: NaN in the
    first target row, 4: NaN in a row the outcome never reads (harmless)."""
    nan = W.BF16_NAN if w.dtype == "bf16" else np.float32(np.nan)
    for kind in kinds:
        b = int(rng.integers(w.B))
        if kind == 0:
            d["draft_lens"][b] = w.K + 1 if rng.random() < 0.5 else 0
        elif kind == 1:
            d["draft_tokens"][b, int(rng.integers(w.K))] = w.V
        elif kind == 2:
            d["uniforms"][b, w.K] = 1.0
        elif kind == 3:
            d["target"][b, 0, int(rng.integers(w.V))] = nan
        elif kind == 4 and d["draft_lens"][b] < w.K:
            d["target"][b, w.K, int(rng.integers(w.V))] = nan


@pytest.mark.parametrize("case", range(len(CASES)))
def test_fuzz(case):
    w, cluster, debug, plant = CASES[case]
    d = W.make_inputs(w)
    plant_invalid(d, w, plant, np.random.default_rng([7, case]))
    g = run_gpu(d, w, cluster_hint=cluster, debug=debug)
    assert api.device_error() == 0, (w, cluster, debug, plant)
    rep = check(d, w, g)
    print(w.name, w.mode, w.dtype, f"B={w.B} K={w.K} V={w.V}", f"C={cluster}",
          "debug" if debug else "", f"bias={w.bias_k}", f"F={w.fanout}", plant, rep.summary())
