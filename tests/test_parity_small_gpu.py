"""GPU parity of stochastic verification for small batches (every row a sequence has read at
once: row statistics, the draw's slice masses, one pick per sequence), against the float64
oracle. The library takes that route for a stochastic batch whose padded rows fit in 256 MiB,
when the caller leaves the cluster size to it (cluster_hint 0) and asks for no diagnostics; with
a bias set or top-F ids the statistics launch also keeps each draft row slice's 8 largest
logits. Each case here also runs the chained cluster walk (cluster_hint 4) on the same inputs,
so both routes face the same bar."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from speculative_decoding_verification_33_gb300 import _lib  # noqa: E402
from speculative_decoding_verification_33_gb300 import workloads as W  # noqa: E402
from tests.test_parity_gpu import check, oracle, run_gpu  # noqa: E402


def both_paths(d, w, **kw):
    reps = []
    for hint in (0, 4):
        g = run_gpu(d, w, cluster_hint=hint, debug=False, **kw)
        reps.append((check(d, w, g), g))
    return reps


def route_of(w, hint=0):
    prob, _keep = _lib.make_problem(w.B, w.K, w.V, _lib.SV_DTYPE_BF16 if w.dtype == "bf16"
                                    else _lib.SV_DTYPE_F32, w.V, w.V, w.bias_k, w.fanout,
                                    cluster_hint=hint)
    return _lib.route(prob, _lib.SV_MODE_GREEDY if w.mode == "greedy"
                      else _lib.SV_MODE_STOCHASTIC)


def test_routes_of_the_workloads():
    R = _lib
    assert route_of(W.WORKLOADS[1]) == (R.SV_ROUTE_SMALL, 3)
    assert route_of(W.WORKLOADS[2]) == (R.SV_ROUTE_GREEDY_ROWS, 2)
    assert route_of(W.WORKLOADS[3]) == (R.SV_ROUTE_SMALL, 3)            # 181 MB of rows
    # the stochastic walk defers its draws to two launches after it
    assert route_of(W.small_variant(W.WORKLOADS[3], B=96)) == (R.SV_ROUTE_WALK, 3)  # 271 MB
    assert route_of(W.WORKLOADS[4]) == (R.SV_ROUTE_SMALL, 3)            # top 8 kept per slice
    assert route_of(W.WORKLOADS[4], hint=4) == (R.SV_ROUTE_WALK, 2)
    assert route_of(W.WORKLOADS[5]) == (R.SV_ROUTE_WALK, 3)
    assert route_of(W.WORKLOADS[1], hint=4) == (R.SV_ROUTE_WALK, 3)


@pytest.mark.parametrize("w", [W.WORKLOADS[1], W.WORKLOADS[3],
                               W.small_variant(W.WORKLOADS[5], B=24)],
                         ids=["B1_K4_V32000_f32", "B64_K5_V128256_bf16", "B24_K8_V152064_ragged"])
def test_small_path_workloads(w):
    assert route_of(w)[0] == _lib.SV_ROUTE_SMALL
    d = W.make_inputs(w)
    (rep, g), (_, g4) = both_paths(d, w)
    print(w.name, rep.summary())
    assert (g["accept_len"] >= 0).all()


@pytest.mark.parametrize("fanout,beta,bias_k", [
    ((8, 4, 2, 1, 1), 0.5, 8),     # workload 4: bias set and top-F ids
    (None, 0.5, 8),                # bias set only
    ((3, 3, 3, 3, 3), 1.0, 0),     # top-F ids only
    (None, 0.25, 1),               # a bias set of one id
])
def test_small_path_bias_and_topf(fanout, beta, bias_k):
    """The draft rows' top 8 (merged from the slices' lists) drive the bias set (q' = q
    reweighted by beta on the bias_k most likely draft ids, renormalised) in the accept tests and
    the residual draw, and give the top-F ids of rows below L (-1 elsewhere and for invalid
    sequences)."""
    w = W.WORKLOADS[4].replace(fanout=fanout, beta=beta, bias_k=bias_k, ragged=True)
    assert route_of(w)[0] == _lib.SV_ROUTE_SMALL
    d = W.make_inputs(w)
    d["draft_tokens"][3, 1] = w.V                # an invalid sequence
    for rep, g in both_paths(d, w):
        assert g["accept_len"][3] == -1
        if fanout is not None:
            assert (g["topf"][3] == -1).all()


@pytest.mark.parametrize("V", [1, 3, 7, 9, 1000, 70001])
def test_small_path_top8_vocabularies(V):
    """Vocabularies below 8 ids (the missing keys read as no id), one partial vector, and
    several slices per row."""
    w = W.small_variant(W.WORKLOADS[4], B=5, V=V).replace(ragged=True)
    w = w.replace(bias_k=min(w.bias_k, V))
    assert route_of(w)[0] == _lib.SV_ROUTE_SMALL
    d = W.make_inputs(w)
    both_paths(d, w)


def test_small_path_top8_ties_zeros_and_sparse_rows():
    """Draft rows that stress the per-slice top 8: every logit equal (ties go to the lower id),
    -0 and +0 as the largest value (one value), -inf but for 5 ids (fewer finite ids than the
    list holds), logits that grow along the row (every later element enters), and a row whose 8
    largest sit in its last 8 ids (a whole vector and the 3-id tail that the bulk copies leave
    to plain loads: row stride V + 5)."""
    w = W.small_variant(W.WORKLOADS[4], B=6, V=20011).replace(ragged=False)
    assert route_of(w)[0] == _lib.SV_ROUTE_SMALL
    d = W.make_inputs(w)
    V, K = w.V, w.K
    dr = d["draft"]
    rng = np.random.default_rng(7)
    dr[0] = 0x3F80                                                   # all 1.0
    dr[1] = rng.choice(np.array([0x8000, 0x0000, 0xBF80], np.uint16), size=dr[1].shape)
    dr[2] = 0xFF80                                                   # -inf ...
    for i in range(K):
        dr[2, i, rng.choice(V, 5, replace=False)] = rng.integers(0x3F00, 0x4000, 5)
    dr[3] = (0x3F80 + np.arange(V) // 4).astype(np.uint16)         # nondecreasing
    dr[4, :, V - 8:] = 0x4100                                        # 8.0 in the last 8 ids
    for b in range(5):                       # drafts the rows can have drawn (q(x) > 0)
        for i in range(K):
            d["draft_tokens"][b, i] = int(np.argmax(W.bf16_bits_to_f32(dr[b, i])))
    for fanout, beta, bias_k in (((8, 4, 2, 1, 1), 0.5, 8), ((8, 8, 8, 8, 8), 1.0, 0)):
        w2 = w.replace(fanout=fanout, beta=beta, bias_k=bias_k)
        for rep, g in both_paths(d, w2, stride_pad=5):
            assert (g["accept_len"] >= 0).all()


@pytest.mark.parametrize("fanout", [(8, 4, 2, 1, 1), None])
def test_small_path_bad_draft_row_below_L(fanout):
    """With top-F ids every draft row below L is needed, so a NaN in the last draft row makes
    the sequence invalid even when the decision stops before it; with a bias set alone it
    matters only where the decision reads the row."""
    w = W.small_variant(W.WORKLOADS[4], B=8, V=3000).replace(ragged=False, fanout=fanout)
    d = W.make_inputs(w)
    d["draft"][:, w.K - 1, 11] = W.BF16_NAN
    for rep, g in both_paths(d, w):
        if fanout is not None:
            assert (g["accept_len"] == -1).all()
            assert (g["topf"] == -1).all()


def test_small_path_top8_unaligned_and_f32():
    """Top 8 kept by the element-by-element path (bf16 rows of stride V + 1, fp32 rows of odd
    stride) and by the bulk copies of fp32 rows with a 3-id tail (stride V + 1 = 5004)."""
    w = W.small_variant(W.WORKLOADS[4], B=5, V=3001).replace(ragged=True)
    both_paths(W.make_inputs(w), w, stride_pad=1)
    w = w.replace(dtype="f32", V=5003)
    d = W.make_inputs(w)
    both_paths(d, w)
    both_paths(d, w, stride_pad=1)


@pytest.mark.parametrize("B,K,V,dtype", [
    (1, 1, 7, "f32"),          # one partial vector per row
    (3, 8, 50001, "bf16"),     # K at its maximum, a ragged last vector
    (17, 3, 4099, "f32"),
    (2, 5, 200000, "bf16"),    # 32 draw slices
    (40, 6, 10000, "bf16"),
])
def test_small_path_shapes(B, K, V, dtype):
    base = W.WORKLOADS[3] if dtype == "bf16" else W.WORKLOADS[1]
    w = W.small_variant(base, B=B, V=V).replace(K=K, ragged=True)
    d = W.make_inputs(w)
    both_paths(d, w)


def test_small_path_unaligned_rows():
    """Row stride V + 1: no 16-byte vectors, every element loaded on its own."""
    w = W.small_variant(W.WORKLOADS[3], B=5, V=3001)
    d = W.make_inputs(w)
    both_paths(d, w, stride_pad=1)


def test_small_path_bonus_draws():
    """u = 0 accepts every draft with p(x) > 0: the draw is from p_L."""
    w = W.small_variant(W.WORKLOADS[3], B=9, V=6000).replace(ragged=True)
    d = W.make_inputs(w)
    d["uniforms"][:, : w.K] = 0.0
    for rep, g in both_paths(d, w):
        assert (g["accept_len"] == d["draft_lens"]).all()


def test_small_path_invalid_sequences():
    w = W.small_variant(W.WORKLOADS[3], B=8, V=600)
    d = W.make_inputs(w)
    d["draft_lens"][0] = 0                    # length out of range
    d["draft_lens"][7] = w.K + 1
    d["draft_tokens"][1, 2] = w.V             # draft id out of range
    d["uniforms"][2, w.K] = 1.0               # final uniform out of range
    d["target"][3, 0, 17] = W.BF16_NAN        # NaN in a needed row
    d["draft"][4, 0, :] = 0xFF80              # draft row of -inf only
    d["target"][5, 0, 5] = 0x7F80             # +inf
    d["target"][6, 0, 3] = 0xFF80             # a single -inf is legal
    for rep, g in both_paths(d, w):
        assert (g["accept_len"][[0, 1, 2, 3, 4, 5, 7]] == -1).all()
        assert (g["tokens"][[0, 1, 2, 3, 4, 5, 7]] == -1).all()
        assert g["accept_len"][6] >= 0


def test_small_path_nan_after_the_stop():
    """Rows after the decided position hold NaN: the statistics read them, the decision must
    not."""
    w = W.small_variant(W.WORKLOADS[3], B=6, V=700)
    d = W.make_inputs(w)
    res = oracle(d, w, all_rows=False)
    for b, r in enumerate(res):
        a = r.accept_len
        if a < w.K:
            d["target"][b, a + 1:] = W.BF16_NAN
            d["draft"][b, a + 1:] = W.BF16_NAN
    for rep, g in both_paths(d, w):
        assert (g["accept_len"] >= 0).all()


def test_small_path_zero_draft_probability_and_ties():
    V, K, B = 64, 3, 4
    w = W.Workload(0, "crafted", B=B, K=K, V=V, dtype="f32", mode="stochastic",
                   temperature=1.0, sigma_t=1, sigma_d=1, zipf=False)
    rng = np.random.default_rng(0)
    tgt = rng.integers(-2, 2, (B, K + 1, V)).astype(np.float32)   # many ties
    dft = rng.integers(-2, 2, (B, K, V)).astype(np.float32)
    dft[0, 0, 5] = -np.inf                                          # q(x) = 0 < p(x)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    tok[0, 0] = 5
    d = {"target": tgt, "draft": dft, "draft_tokens": tok,
         "draft_lens": np.full(B, K, np.int32),
         "uniforms": rng.random((B, K + 1), dtype=np.float32)}
    both_paths(d, w)


def test_small_path_repeated_calls_agree():
    """The workspace's partials, decisions and masses are rewritten each call: repeated calls
    (and a call of another shape in between) give the same outcome."""
    w = W.small_variant(W.WORKLOADS[3], B=12, V=9000).replace(ragged=True)
    d = W.make_inputs(w)
    g1 = run_gpu(d, w, debug=False)
    w2 = W.small_variant(W.WORKLOADS[1], B=3, V=1000)
    run_gpu(W.make_inputs(w2), w2, debug=False)
    g2 = run_gpu(d, w, debug=False)
    assert (g1["accept_len"] == g2["accept_len"]).all()
    assert (g1["tokens"] == g2["tokens"]).all()
