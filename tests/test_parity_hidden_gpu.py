"""GPU parity of the verify step taken from hidden states (``spec_verify_hidden``), called
through the C ABI, against the float64 oracle (``oracle.lmhead.verify_hidden_batch``).

Two kinds of input:
* exact: hidden states and head on dyadic grids (``workloads.hidden_inputs(exact=True)``), so
  every logit is exact in float32 whatever the order of the tensor cores' sums. The GPU then
  sees the oracle's logits, and the outcome must match with the verify step's own bar: decisions
  closer than 1e-6 to their threshold are flagged, everything else equal.
* continuous: bf16 values of a normal distribution. A logit then carries float32 rounding; for a
  sum of d exact products it behaves like a random walk of about sqrt(d) * 2^-24 * |z|, so 10
  standard deviations on both logits of the ratio and both normalisers stay below 1e-3
  relative for d <= 4096 and |z| <= 40: decisions closer than 1e-3 are flagged. With V in the
  thousands a draw's relative CDF gap is about 1/V, so most draws are flagged there and these
  tests mostly check the accept decisions, lengths and accepted ids; the exact inputs check the
  draws.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from oracle import lmhead as HO  # noqa: E402
from speculative_decoding_verification_33_gb300 import api  # noqa: E402
from speculative_decoding_verification_33_gb300 import workloads as W  # noqa: E402
from tests import parity  # noqa: E402

CONTINUOUS_MARGIN = 1e-3


def bf16(bits: np.ndarray) -> "torch.Tensor":
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def run_gpu(x, w, beta=1.0, bias_k=0, fanout=None):
    greedy = w.mode == "greedy"
    out = api.verify_hidden(bf16(x["hidden_target"]),
                            None if greedy else bf16(x["hidden_draft"]), bf16(x["weight"]),
                            torch.from_numpy(x["draft_tokens"]).cuda(),
                            torch.from_numpy(x["draft_lens"]).cuda(),
                            None if greedy else torch.from_numpy(x["uniforms"]).cuda(),
                            temperature=w.temperature, beta=beta, bias_k=bias_k, fanout=fanout,
                            mode=w.mode)
    torch.cuda.synchronize()
    return (out["accept_len"].cpu().numpy(), out["tokens"].cpu().numpy(),
            out["topf"].cpu().numpy() if fanout is not None else None)


def check(x, w, margin, seqs=None, weight64=None, beta=1.0, bias_k=0, fanout=None,
          topf_exact=True):
    greedy = w.mode == "greedy"
    acc, tok, topf = run_gpu(x, w, beta, bias_k, fanout)
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    res = HO.verify_hidden_batch(x["hidden_target"], None if greedy else x["hidden_draft"],
                                 x["weight"] if weight64 is None else weight64,
                                 x["draft_tokens"], x["draft_lens"], x["uniforms"],
                                 temperature=w.temperature, mode=w.mode, beta=beta,
                                 bias_k=bias_k, fanout=fanout, seqs=seqs)
    rep = parity.compare(res, seqs, acc, tok, topf if topf_exact else None, margin=margin)
    assert rep.ok(), (rep.summary(), rep.mismatches[:4])
    return rep, res, topf


@pytest.mark.parametrize("B,K,V,d,T,mode", [
    (40, 4, 3000, 256, 0.8, "stochastic"),    # one tile of pairs, ragged column tile
    (130, 3, 5000, 128, 1.0, "stochastic"),   # three tiles of pairs, partly empty
    (24, 5, 2048, 192, 1.0, "greedy"),
    (7, 8, 777, 64, 1.3, "stochastic"),       # smallest d, K at its maximum
])
def test_hidden_exact(B, K, V, d, T, mode):
    w = W.HiddenWorkload(f"exact_{B}_{K}_{V}_{d}", B=B, K=K, V=V, d=d, mode=mode, temperature=T,
                         exact=True)
    x = W.hidden_inputs(w)
    rep, res, _ = check(x, w, margin=1e-6)
    assert sum(r.accept_len for r in res if r.valid) > 0  # accept and reject paths both ran
    assert rep.flagged <= max(1, B // 20)


@pytest.mark.parametrize("mode,B", [("stochastic", 64), ("greedy", 32)])
def test_hidden_exact_full_vocabulary(mode, B):
    """Exact-grid inputs at the bench's vocabulary (V = 152064: the whole split of the vocabulary
    over column tiles, with its ragged last tile) and the deepest K loop the exact grid allows
    (d = 1024), ragged K = 8: every draw is compared at the 1e-6 margin, so a wrong token at full
    size shows here."""
    w = W.HiddenWorkload(f"exact_full_{mode}", B=B, K=8, V=152064, d=1024, mode=mode,
                         exact=True, drafter="prior")
    x = W.hidden_inputs(w)
    weight64 = HO.bf16_to_f64(x["weight"])  # converted once for the oracle's B head products
    rep, res, _ = check(x, w, margin=1e-6, weight64=weight64)
    print(w.name, rep.summary())
    assert sum(r.accept_len for r in res if r.valid) > 0
    assert rep.flagged <= max(1, B // 20)


@pytest.mark.parametrize("fanout,beta,bias_k", [
    ((8, 4, 2, 1, 1), 0.5, 8),     # the Saguaro workload's options
    (None, 0.3, 3),                # bias set only
    ((3, 3, 3, 3, 3), 1.0, 0),     # top-F ids only
])
def test_hidden_exact_bias_set_and_top_f(fanout, beta, bias_k):
    """The bias set (the bias_k largest draft logits, merged from the head GEMM's vocabulary
    ranges) in the accept tests and the residual draw, and the top-F draft ids, on exact-grid
    inputs: ids, lengths and tokens equal the oracle's."""
    w = W.HiddenWorkload("exact_bias", B=40, K=5, V=3000, d=256, exact=True)
    x = W.hidden_inputs(w)
    x["draft_tokens"][3, 1] = w.V  # an invalid sequence: -1 everywhere, top-F ids included
    rep, res, topf = check(x, w, margin=1e-6, beta=beta, bias_k=bias_k, fanout=fanout)
    assert sum(r.accept_len for r in res if r.valid) > 0
    assert rep.flagged <= max(1, w.B // 20)
    if fanout is not None:
        assert (topf[3] == -1).all()
        assert (topf >= 0).sum() > 0


def test_hidden_exact_bias_set_full_vocabulary():
    """The bias set and top-F ids at the bench's vocabulary (V = 152064 over many ranges of the
    head GEMM, K = 8 ragged): the merge over ranges must find each draft row's 8 largest."""
    w = W.HiddenWorkload("exact_full_bias", B=48, K=8, V=152064, d=1024, exact=True,
                         drafter="prior")
    x = W.hidden_inputs(w)
    weight64 = HO.bf16_to_f64(x["weight"])
    rep, res, topf = check(x, w, margin=1e-6, weight64=weight64, beta=0.5, bias_k=8,
                           fanout=(8, 4, 2, 1, 1, 1, 1, 1))
    print(w.name, rep.summary())
    assert sum(r.accept_len for r in res if r.valid) > 0
    assert rep.flagged <= max(1, w.B // 20)


def test_hidden_continuous_bias_set_and_top_f():
    """Continuous inputs: the accept decisions at the float32 margin, and every top-F id within
    the logits' rounding of the oracle's id at that rank (near ties may swap)."""
    w = W.HiddenWorkload("cont_bias", B=32, K=5, V=4000, d=512, temperature=0.9)
    x = W.hidden_inputs(w)
    fan = (6, 3, 2, 1, 1)
    rep, res, topf = check(x, w, margin=CONTINUOUS_MARGIN, beta=0.5, bias_k=8, fanout=fan,
                           topf_exact=False)
    assert sum(r.accept_len for r in res) > 0
    swaps = 0
    for b, r in enumerate(res):
        if not r.valid:
            assert (topf[b] == -1).all()
            continue
        L = int(x["draft_lens"][b])
        z = HO.head_logits(x["hidden_draft"][b, :L], x["weight"])
        err = HO.logit_error_bound(x["hidden_draft"][b, :L], x["weight"])
        for i in range(L):
            for f in range(fan[i]):
                g, o = int(topf[b, i, f]), int(r.topf[i, f])
                if g != o:
                    swaps += 1
                    assert abs(z[i, g] - z[i, o]) <= 2 * (err[i, g] + err[i, o])
    assert swaps <= 2


def test_hidden_every_draft_accepted_and_invalid_rows():
    """Bonus draws (all drafts accepted: the draft row of the pair is zeros, the draw is from p),
    and invalid sequences (length 0 or > K, an id outside the vocabulary, a uniform of 1)."""
    w = W.HiddenWorkload("exact_bonus", B=12, K=3, V=1500, d=128, exact=True, ragged=False,
                         sigma_d=0.0)
    x = W.hidden_inputs(w)
    x["uniforms"][:6, :3] = 0.0          # u = 0 accepts every draft with p(x) > 0
    x["draft_lens"][7] = 0
    x["draft_lens"][8] = 4
    x["draft_tokens"][9, 1] = 1500
    x["uniforms"][10, 3] = 1.0
    rep, res, _ = check(x, w, margin=1e-6)
    assert all(res[b].accept_len == 3 for b in range(6))
    assert rep.invalid == 4


def test_hidden_continuous():
    w = W.HiddenWorkload("cont", B=48, K=5, V=4000, d=512, temperature=0.9)
    x = W.hidden_inputs(w)
    rep, res, _ = check(x, w, margin=CONTINUOUS_MARGIN)
    assert rep.flagged < rep.sequences
    assert sum(r.accept_len for r in res) > 0


def test_hidden_full_size_sampled():
    """The bench's batch (B=256, K=8, V=152064, d=3584), oracle on sampled sequences."""
    w = W.HIDDEN_WORKLOADS["hv_B256_K8_V152064_d3584"]
    x = W.hidden_inputs(w)
    seqs = list(range(0, w.B, 16)) + [w.B - 1]
    rep, res, _ = check(x, w, margin=CONTINUOUS_MARGIN, seqs=seqs)
    # At this margin a draw's relative CDF gap (about 1 / V) is almost always below it, so the
    # draws here are flagged and only the accept decisions, lengths and accepted ids are compared;
    # test_hidden_exact_full_vocabulary compares the draws at this vocabulary.
    print(w.name, rep.summary())
    assert sum(r.accept_len for r in res) > 0
    assert rep.flagged <= len(seqs)


def test_hidden_rejects_bad_arguments():
    h = torch.zeros(2, 3, 96, dtype=torch.bfloat16, device="cuda")  # d not a multiple of 64
    wt = torch.zeros(10, 96, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(2, 2, dtype=torch.int32, device="cuda")
    with pytest.raises(RuntimeError):
        api.verify_hidden(h, None, wt, x, torch.ones(2, dtype=torch.int32, device="cuda"),
                          mode="greedy")
    h = torch.zeros(2, 3, 64, dtype=torch.bfloat16, device="cuda")
    wt = torch.zeros(10, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError):  # stochastic mode needs the draft rows and uniforms
        api.verify_hidden(h, None, wt, x, torch.ones(2, dtype=torch.int32, device="cuda"))
