"""GPU parity: the CUDA verify path, called through the C ABI, against the float64 oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from oracle import verify as O  # noqa: E402
from speculative_decoding_verification_33_gb300 import api  # noqa: E402
from speculative_decoding_verification_33_gb300 import workloads as W  # noqa: E402
from tests.parity import compare  # noqa: E402


def run_gpu(d, w, cluster_hint=0, debug=True, lens=True, stride_pad=0, entry="spec_verify"):
    tgt, dft = d["target"], d["draft"]
    if stride_pad:
        tgt = np.pad(tgt, ((0, 0), (0, 0), (0, stride_pad)))
        dft = np.pad(dft, ((0, 0), (0, 0), (0, stride_pad)))
    T = api.to_device_logits(tgt)
    D = api.to_device_logits(dft) if w.mode == "stochastic" else None
    if stride_pad:
        T = T[:, :, : w.V]
        D = D[:, :, : w.V] if D is not None else None
    tok = torch.from_numpy(d["draft_tokens"]).cuda()
    ln = torch.from_numpy(d["draft_lens"]).cuda() if lens else None
    uni = torch.from_numpy(d["uniforms"]).cuda()
    out = api.verify(T, D, tok, ln, uni, temperature=w.temperature, beta=w.beta, mode=w.mode,
                     bias_k=w.bias_k, fanout=w.fanout, debug=debug and w.mode == "stochastic",
                     cluster_hint=cluster_hint)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def oracle(d, w, all_rows=True, seqs=None):
    return O.verify_batch(d["target"], d["draft"] if w.mode == "stochastic" else None,
                          d["draft_tokens"], d["draft_lens"], d["uniforms"],
                          temperature=w.temperature, mode=w.mode, beta=w.beta,
                          bias_k=w.bias_k, fanout=w.fanout, all_rows=all_rows, seqs=seqs)


def check(d, w, g, seqs=None):
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    res = oracle(d, w, seqs=seqs)
    dbg = {k: g[k] for k in ("lse_t", "lse_d", "p_x", "q_x")} if "lse_t" in g else None
    rep = compare(res, seqs, g["accept_len"], g["tokens"], g.get("topf"), dbg)
    assert rep.ok(), (rep.summary(), rep.mismatches[:5], rep.diag_bad[:5])
    return rep


# ---------------------------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_workload_full(cfg):
    w = W.WORKLOADS[cfg]
    d = W.make_inputs(w)
    rep = check(d, w, run_gpu(d, w))
    print(w.name, rep.summary())


def test_workload5_full_size():
    w = W.WORKLOADS[5]
    d = W.make_inputs(w)
    rep = check(d, w, run_gpu(d, w, debug=False))
    print(w.name, rep.summary())
    assert rep.flagged < 0.35 * w.B


def test_workload5_diagnostics_sample():
    w = W.WORKLOADS[5].replace(B=24)
    d = W.make_inputs(w)
    check(d, w, run_gpu(d, w, debug=True))


@pytest.mark.parametrize("cfg", [1, 3, 4])
@pytest.mark.parametrize("cluster", [1, 2, 4, 8, 16])
def test_cluster_sizes(cfg, cluster):
    w = W.small_variant(W.WORKLOADS[cfg], B=6, V=3001)
    d = W.make_inputs(w)
    check(d, w, run_gpu(d, w, cluster_hint=cluster))


# ---------------------------------------------------------------------------------------------
# shapes and layouts
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("V", [1, 2, 3, 7, 8, 9, 31, 257, 1000])
@pytest.mark.parametrize("cfg", [2, 4])
def test_tiny_vocab(V, cfg):
    w = W.small_variant(W.WORKLOADS[cfg], B=5, V=V)
    w = w.replace(bias_k=min(w.bias_k, V))
    d = W.make_inputs(w)
    for cl in (1, 4, 16):
        check(d, w, run_gpu(d, w, cluster_hint=cl))


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_unaligned_row_stride(cfg):
    """Row strides that are not a multiple of 16 bytes take the plain-load staging path."""
    w = W.small_variant(W.WORKLOADS[cfg], B=4, V=1003)
    d = W.make_inputs(w)
    check(d, w, run_gpu(d, w, stride_pad=3))


def test_many_sequences_dynamic_queue():
    w = W.small_variant(W.WORKLOADS[5], B=700, V=512)
    d = W.make_inputs(w)
    g1 = run_gpu(d, w, cluster_hint=2, debug=False)
    check(d, w, g1)
    g2 = run_gpu(d, w, cluster_hint=2, debug=False)  # the queue resets between launches
    assert np.array_equal(g1["accept_len"], g2["accept_len"])
    assert np.array_equal(g1["tokens"], g2["tokens"])


def test_batch_above_ordering_threshold():
    """Batches above 4096 sequences keep the natural order (no longest-first permutation)."""
    w = W.small_variant(W.WORKLOADS[5], B=4200, V=64).replace(K=3)
    d = W.make_inputs(w)
    check(d, w, run_gpu(d, w, debug=False), seqs=range(0, 4200, 7))


def test_greedy_without_draft_logits_and_lens():
    w = W.small_variant(W.WORKLOADS[2], B=9)
    d = W.make_inputs(w)
    check(d, w, run_gpu(d, w, lens=False))


def test_empty_batch():
    t = torch.zeros(0, 3, 16, dtype=torch.bfloat16, device="cuda")
    out = api.verify(t, None, torch.zeros(0, 2, dtype=torch.int32, device="cuda"), mode="greedy")
    assert out["accept_len"].numel() == 0


# ---------------------------------------------------------------------------------------------
# invalid and degenerate sequences
# ---------------------------------------------------------------------------------------------
def test_invalid_sequences():
    w = W.small_variant(W.WORKLOADS[4], B=8, V=600)
    d = W.make_inputs(w)
    d["draft_lens"][0] = 0                    # length out of range
    d["draft_tokens"][1, 2] = w.V             # draft id out of range
    d["uniforms"][2, w.K] = 1.0               # final uniform out of range
    d["target"][3, 0, 17] = W.BF16_NAN        # NaN in a needed row
    d["draft"][4, 0, :] = 0xFF80              # draft row of -inf only
    d["target"][5, 0, 5] = 0x7F80             # +inf
    d["target"][6, 0, 3] = 0xFF80             # a single -inf is legal
    check(d, w, run_gpu(d, w))
    g = run_gpu(d, w, debug=False)
    assert (g["accept_len"][[0, 1, 2, 3, 4, 5]] == -1).all()
    assert g["accept_len"][6] >= 0


@pytest.mark.parametrize("cluster", [4, 8])
def test_greedy_walk_long_rows(cluster):
    """Greedy rows of 152064 ids take several ring chunks per CTA, and with 8 sequences no
    cluster has a second one: a stop that lands while the next position streams must still end
    the sequence (the producer marks the stage after a stop) instead of leaving the consumers
    waiting for chunks that will not come."""
    w = W.small_variant(W.WORKLOADS[5], B=8).replace(mode="greedy", temperature=0.0)
    d = W.make_inputs(w)
    g = run_gpu(d, w, cluster_hint=cluster, debug=False)
    assert api.device_error() == 0
    check(d, w, g)
    assert (g["accept_len"] >= 0).all()


def test_invalid_row_mid_walk_long_rows():
    """A NaN in the second position's target row, read after the first draft is accepted, makes
    the sequence invalid while the third position streams; with one sequence per cluster and
    rows of several chunks the walk must end it without waiting out its bounded waits."""
    w = W.small_variant(W.WORKLOADS[5], B=6).replace(ragged=False)
    d = W.make_inputs(w)
    d["uniforms"][:, 0] = 0.0                  # u = 0 accepts the first draft when p(x) > 0
    d["target"][:, 1, 17] = W.BF16_NAN
    for cluster in (4, 8):
        g = run_gpu(d, w, cluster_hint=cluster, debug=False)
        assert api.device_error() == 0
        check(d, w, g)
        assert (g["accept_len"] == -1).all()


def test_greedy_walk_many_short_sequences():
    """Many greedy sequences of one chunk per position on the walk: a stop's marker stage
    that the consumers no longer wait for is dropped when they move to the next sequence."""
    w = W.small_variant(W.WORKLOADS[2], B=256)
    d = W.make_inputs(w)
    g = run_gpu(d, w, cluster_hint=4, debug=False)
    assert api.device_error() == 0
    check(d, w, g)


def test_nan_after_rejection_is_not_read():
    w = W.small_variant(W.WORKLOADS[3], B=6, V=700)
    d = W.make_inputs(w)
    res = oracle(d, w, all_rows=False)
    for b, r in enumerate(res):
        a = r.accept_len
        if a < w.K:
            d["target"][b, a + 1:] = W.BF16_NAN
            d["draft"][b, a + 1:] = W.BF16_NAN
    g = run_gpu(d, w, debug=False)
    check(d, w, g)
    assert (g["accept_len"] >= 0).all()


def test_zero_draft_probability_and_ties():
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
    check(d, w, run_gpu(d, w))
    wg = w.replace(mode="greedy", temperature=0.0)
    check(d, wg, run_gpu(d, wg))


def test_beta_bias_without_topf():
    w = W.small_variant(W.WORKLOADS[4], B=10, V=5000).replace(fanout=None)
    d = W.make_inputs(w)
    check(d, w, run_gpu(d, w))


@pytest.mark.parametrize("hint", [0, 4])
def test_fanout_with_zero_widths(hint):
    """Fan-out widths of 0 leave a position's top-F ids at -1 and the others take the first F_i
    of the draft row's order: on the small route (no hint at this size) and on the cluster walk
    with the top-8 prepass (hint 4)."""
    w = W.small_variant(W.WORKLOADS[4], B=12, V=20000).replace(fanout=(3, 0, 5, 0, 1))
    d = W.make_inputs(w)
    g = run_gpu(d, w, cluster_hint=hint)
    check(d, w, g)
    assert (g["topf"][:, 1] == -1).all() and (g["topf"][:, 3] == -1).all()


# ---------------------------------------------------------------------------------------------
# other entry points give the same answer
# ---------------------------------------------------------------------------------------------
def test_workspace_and_host_entry_points():
    w = W.small_variant(W.WORKLOADS[4], B=12, V=4099)
    d = W.make_inputs(w)
    ref = run_gpu(d, w, debug=False)
    T = api.to_device_logits(d["target"])
    D = api.to_device_logits(d["draft"])
    tok = torch.from_numpy(d["draft_tokens"]).cuda()
    ln = torch.from_numpy(d["draft_lens"]).cuda()
    uni = torch.from_numpy(d["uniforms"]).cuda()
    acc = torch.empty(w.B, dtype=torch.int32, device="cuda")
    toks = torch.empty(w.B, w.K + 1, dtype=torch.int32, device="cuda")
    topf = torch.empty(w.B, w.K, 8, dtype=torch.int32, device="cuda")
    ws = torch.zeros(api.workspace_bytes(w.B) // 4, dtype=torch.int32, device="cuda")
    for _ in range(2):
        api.spec_verify(T, D, tok, ln, uni, w.temperature, w.beta, w.mode, acc, toks, topf,
                        bias_k=w.bias_k, fanout=w.fanout, workspace=ws)
        torch.cuda.synchronize()
        assert np.array_equal(acc.cpu().numpy(), ref["accept_len"])
        assert np.array_equal(toks.cpu().numpy(), ref["tokens"])
    h_acc = np.empty(w.B, np.int32)
    h_tok = np.empty((w.B, w.K + 1), np.int32)
    h_topf = np.empty((w.B, w.K, 8), np.int32)
    api.verify_host(d["target"], d["draft"], d["draft_tokens"], d["draft_lens"], d["uniforms"],
                    h_acc, h_tok, h_topf, dtype=w.dtype, temperature=w.temperature, beta=w.beta,
                    mode=w.mode, bias_k=w.bias_k, fanout=w.fanout)
    assert np.array_equal(h_acc, ref["accept_len"])
    assert np.array_equal(h_tok, ref["tokens"])
    assert np.array_equal(h_topf, ref["topf"])
    assert api.device_error() == 0


@pytest.mark.parametrize("cfg", [5, 2, 1])
def test_host_rows_read_in_place(cfg):
    """Rows in pinned host memory are read in place by the kernel (no staging copy); the outcome
    equals the device-buffer call and the oracle's."""
    w = W.WORKLOADS[cfg] if cfg != 5 else W.small_variant(W.WORKLOADS[5], B=48)
    d = W.make_inputs(w)
    greedy = w.mode == "greedy"

    def pinned(a):
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).pin_memory()
    hT = pinned(d["target"])
    hD = None if greedy else pinned(d["draft"])
    h_acc = torch.empty(w.B, dtype=torch.int32).pin_memory()
    h_tok = torch.empty(w.B, w.K + 1, dtype=torch.int32).pin_memory()
    api.verify_host(hT, hD, torch.from_numpy(d["draft_tokens"]).pin_memory(),
                    torch.from_numpy(d["draft_lens"]).pin_memory(),
                    torch.from_numpy(d["uniforms"]).pin_memory(), h_acc, h_tok,
                    dtype=w.dtype, temperature=w.temperature, mode=w.mode)
    T = api.to_device_logits(d["target"])
    D = None if greedy else api.to_device_logits(d["draft"])
    out = api.verify(T, D, torch.from_numpy(d["draft_tokens"]).cuda(),
                     torch.from_numpy(d["draft_lens"]).cuda(),
                     torch.from_numpy(d["uniforms"]).cuda(), temperature=w.temperature,
                     mode=w.mode)
    torch.cuda.synchronize()
    res = O.verify_batch(d["target"], None if greedy else d["draft"], d["draft_tokens"],
                         d["draft_lens"], d["uniforms"], temperature=w.temperature, mode=w.mode)
    rep = compare(res, range(w.B), h_acc.numpy(), h_tok.numpy())
    assert rep.ok(), (rep.summary(), rep.mismatches[:3])
    # the device call may take another route than the in-place host rows (the walk):
    # both calls equal the oracle, and each other wherever no decision is flagged
    d_acc, d_tok = out["accept_len"].cpu().numpy(), out["tokens"].cpu().numpy()
    rep_d = compare(res, range(w.B), d_acc, d_tok)
    assert rep_d.ok(), (rep_d.summary(), rep_d.mismatches[:3])
    for b, r in enumerate(res):
        if r.first_flag(O.MARGIN) is None:
            assert h_acc.numpy()[b] == d_acc[b] and np.array_equal(h_tok.numpy()[b], d_tok[b])
    assert api.device_error() == 0
