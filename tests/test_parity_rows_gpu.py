"""GPU parity of the row kernels (draft draw with exit confidence, exact-residual top-F and the
cache-hit flag), called through the C ABI, against the float64 oracle."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from oracle import rows as RO  # noqa: E402
from oracle import verify as O  # noqa: E402
from speculative_decoding_verification_33_gb300 import api  # noqa: E402
from speculative_decoding_verification_33_gb300 import workloads as W  # noqa: E402

REL_TOL = 1e-5
MARGIN = 1e-6


# ---------------------------------------------------------------------------------------------
# draft draw
# ---------------------------------------------------------------------------------------------
def draft_rows(w, R, offset=0):
    """[R, V] draft rows and [R] uniforms from the workload's generator (rows past a sequence's
    draft length are NaN, so some rows are bad on purpose)."""
    d = W.make_inputs(w, offset=offset)
    rows = d["draft"].reshape(-1, w.V)[:R]
    uni = d["uniforms"].reshape(-1)[:R].copy()
    return rows, uni


def check_draws(rows, uni, *, T, beta, bias_k, tau, pad=0, seqs=None):
    host = np.pad(rows, ((0, 0), (0, pad))) if pad else rows
    D = api.to_device_logits(host)
    if pad:
        D = D[:, : rows.shape[1]]
    out = api.draft_sample(D, torch.from_numpy(uni).cuda(), temperature=T, beta=beta,
                           bias_k=bias_k, tau=tau)
    torch.cuda.synchronize()
    tok, conf, ex = (out[k].cpu().numpy() for k in ("tokens", "conf", "exit"))
    seqs = range(rows.shape[0]) if seqs is None else seqs
    flagged = checked = 0
    for r in seqs:
        o = RO.draft_sample(rows[r], float(uni[r]), temperature=T, beta=beta, bias_k=bias_k,
                            tau=tau)
        checked += 1
        if math.isnan(o.conf):
            assert tok[r] == -1 and ex[r] == -1 and math.isnan(conf[r]), r
            continue
        assert abs(float(conf[r]) - o.conf) <= REL_TOL * o.conf, (r, conf[r], o.conf)
        if abs(o.conf - tau) > REL_TOL * o.conf:
            assert ex[r] == o.exit, (r, ex[r], o.exit)
        if o.margin < MARGIN:
            flagged += 1
            assert tok[r] >= 0
            continue
        assert tok[r] == o.token, (r, tok[r], o.token, o.margin)
    return checked, flagged


@pytest.mark.parametrize("cfg", [1, 3, 4, 5])
def test_draft_draw_workload_rows(cfg):
    w = W.small_variant(W.WORKLOADS[cfg], B=8)
    rows, uni = draft_rows(w, 8 * w.K)
    T = w.temperature if w.mode == "stochastic" else 1.0
    checked, flagged = check_draws(rows, uni, T=T, beta=w.beta, bias_k=w.bias_k, tau=0.05)
    assert flagged <= checked // 10


@pytest.mark.parametrize("V", [1, 2, 7, 8, 9, 1000, 12289, 40000, 98305, 262144])
def test_draft_draw_vocab_sizes(V):
    """Cluster sizes 1 to 16 and ragged slice tails."""
    w = W.small_variant(W.WORKLOADS[4], B=3, V=V).replace(bias_k=min(8, V))
    rows, uni = draft_rows(w, 3 * w.K)
    check_draws(rows, uni, T=1.0, beta=0.5, bias_k=w.bias_k, tau=0.2)
    check_draws(rows, uni, T=0.7, beta=1.0, bias_k=0, tau=0.2)


def test_draft_draw_unaligned_stride_and_f32():
    w = W.small_variant(W.WORKLOADS[1], B=4, V=5003)
    rows, uni = draft_rows(w, 4 * w.K)
    check_draws(rows, uni, T=1.3, beta=0.3, bias_k=4, tau=0.01, pad=3)


def test_draft_draw_bad_uniforms_and_rows():
    w = W.small_variant(W.WORKLOADS[3], B=2, V=3000)
    rows, uni = draft_rows(w, 2 * w.K)
    rows = rows.copy()
    uni[0], uni[1], uni[2] = 1.0, -0.5, np.nan
    rows[3, 11] = W.BF16_NAN
    rows[4, :] = 0xFF80  # all -inf
    check_draws(rows, uni, T=0.8, beta=1.0, bias_k=0, tau=0.5)


def _planted_rows(V, dtype):
    """Draft rows whose bias set decides the draws (bf16 bit patterns or float32): (a) 12 large,
    close logits over N(0, 1) noise (most of the mass, the 8th and 9th close); (b) groups of 4
    ever larger logits planted in chunks 2, 5, 8, ... of the stream, so the kept candidate groups
    fill up and are compacted; (c) a decreasing row (the first chunk holds the 8 largest); (d) an
    increasing row (every later group reaches the kept bound: the store runs over and the groups
    are read again); (e) a row of equal values."""
    rng = np.random.default_rng(21)
    base = rng.standard_normal((5, V)).astype(np.float32)
    ids = rng.choice(V, 12, replace=False)
    base[0, ids] = 14.0 + 0.05 * np.arange(12)
    chunk = 8192 if dtype == "bf16" else 4096
    for j, ch in enumerate(range(2, (V + chunk - 1) // chunk, 3)):
        lo = ch * chunk
        at = lo + rng.choice(min(chunk, V - lo), 4, replace=False)
        base[1, at] = 12.0 + j + 0.1 * np.arange(4)
    base[2] = np.linspace(8.0, -8.0, V)
    base[3] = np.linspace(-8.0, 8.0, V)
    base[4] = 1.0
    return W.f32_to_bf16_bits(base) if dtype == "bf16" else base


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_draft_draw_bias_set_decides_the_draws(dtype):
    """Each planted row drawn at 96 evenly spaced uniforms: the tokens sweep the inverse CDF of
    q' = q reweighted by beta on the 8 largest logits, so a wrong bias set (kept groups missing
    one of the 8, a compaction that drops one, a fallback that does not read the groups again)
    moves tokens across the CDF."""
    V = 152064 if dtype == "bf16" else 70001
    base = _planted_rows(V, dtype)
    n = 96
    rows = np.repeat(base, n, axis=0)
    uni = np.tile((np.arange(n, dtype=np.float64) + 0.5) / n, base.shape[0]).astype(np.float32)
    checked, flagged = check_draws(rows, uni, T=1.0, beta=0.3, bias_k=8, tau=0.1,
                                   seqs=range(2 * n))  # the planted rows, where the set decides
    assert flagged <= checked // 20
    check_draws(rows, uni, T=1.0, beta=0.3, bias_k=8, tau=0.1, seqs=range(2 * n, rows.shape[0]))


def test_draft_draw_frequencies_follow_biased_draft():
    """Many draws of one row: token frequencies match q' (chi-square style bound)."""
    V, n = 64, 1 << 16
    rng = np.random.default_rng(9)
    z = (rng.standard_normal(V) * 1.5).astype(np.float32)
    D = torch.from_numpy(np.tile(z, (n, 1))).cuda()
    uni = torch.from_numpy(rng.random(n, dtype=np.float32)).cuda()
    out = api.draft_sample(D, uni, temperature=0.9, beta=0.4, bias_k=3)
    tok = out["tokens"].cpu().numpy()
    q, _ = O.softmax(z.astype(np.float64), 0.9)
    qb, _ = O.biased_draft(q, z.astype(np.float64), 0.4, 3)
    freq = np.bincount(tok, minlength=V) / n
    assert np.all(np.abs(freq - qb) <= 5 * np.sqrt(qb * (1 - qb) / n) + 1e-9)


def test_draft_draw_empty_and_full_size_sample():
    e = api.draft_sample(torch.zeros(0, 16, dtype=torch.bfloat16, device="cuda"),
                         torch.zeros(0, dtype=torch.float32, device="cuda"))
    assert e["tokens"].numel() == 0
    w = W.WORKLOADS[5]
    rows, uni = draft_rows(w, w.B * w.K)
    check_draws(rows, uni, T=1.0, beta=0.5, bias_k=8, tau=0.1, seqs=range(0, w.B * w.K, 37))


# ---------------------------------------------------------------------------------------------
# exact-residual top-F and cache hits
# ---------------------------------------------------------------------------------------------
def residual_gpu(d, w, verify_out=None, pad=0):
    tgt, dft = d["target"], d["draft"]
    if pad:
        tgt = np.pad(tgt, ((0, 0), (0, 0), (0, pad)))
        dft = np.pad(dft, ((0, 0), (0, 0), (0, pad)))
    T = api.to_device_logits(tgt)
    D = api.to_device_logits(dft)
    if pad:
        T, D = T[:, :, : w.V], D[:, :, : w.V]
    ln = torch.from_numpy(d["draft_lens"]).cuda()
    out = api.residual_topf(T, D, ln, w.fanout, temperature=w.temperature, beta=w.beta,
                            bias_k=w.bias_k, verify_out=verify_out)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def compare_residual(d, w, r2, seqs):
    """Exact ids where the oracle's residual values are separated; at a near tie (within the
    float32 error of p and q') any id of equal residual is accepted."""
    near = 0
    fmax = r2.shape[2]
    for b in seqs:
        L = int(d["draft_lens"][b])
        for i in range(w.K):
            got = r2[b, i].tolist()
            if i >= L:
                assert got == [-1] * fmax, (b, i, got)
                continue
            zt, zd = O.row_to_f64(d["target"][b, i]), O.row_to_f64(d["draft"][b, i])
            if O.row_is_bad(zt) or O.row_is_bad(zd):
                assert got == [-1] * fmax, (b, i, got)
                continue
            p, _ = O.softmax(zt, w.temperature)
            q, _ = O.softmax(zd, w.temperature)
            qb, _ = O.biased_draft(q, zd, w.beta, w.bias_k)
            r, ids = RO.residual_order(d["target"][b, i], d["draft"][b, i],
                                       temperature=w.temperature, beta=w.beta, bias_k=w.bias_k)
            tol = 4e-6 * (p + qb) + 1e-12
            F = min(w.fanout[i], 8)
            assert got[F:] == [-1] * (fmax - F), (b, i, got)
            real = [g for g in got[:F] if g >= 0]
            assert len(set(real)) == len(real), (b, i, got)
            for f in range(F):
                o = int(ids[f]) if f < len(ids) else -1
                g = got[f]
                if g == o:
                    continue
                near += 1
                ro = r[o] if o >= 0 else 0.0
                to = tol[o] if o >= 0 else 0.0
                rg = (p[g] - qb[g]) if g >= 0 else 0.0
                tg = tol[g] if g >= 0 else 0.0
                assert abs(rg - ro) <= tg + to, (b, i, f, g, o, rg, ro)
    return near


@pytest.mark.parametrize("cfg", [4, 3, 5])
def test_residual_topf_and_hits(cfg):
    w = W.WORKLOADS[cfg]
    if w.fanout is None:
        w = w.replace(fanout=(8, 4, 2, 1, 1, 1, 1, 1)[: w.K])
    if cfg == 5:
        w = w.replace(B=24)
    d = W.make_inputs(w)
    Tt = api.to_device_logits(d["target"])
    Dd = api.to_device_logits(d["draft"])
    vo = api.verify(Tt, Dd, torch.from_numpy(d["draft_tokens"]).cuda(),
                    torch.from_numpy(d["draft_lens"]).cuda(),
                    torch.from_numpy(d["uniforms"]).cuda(), temperature=w.temperature,
                    beta=w.beta, mode="stochastic", bias_k=w.bias_k, fanout=w.fanout)
    g = residual_gpu(d, w, verify_out=vo)
    near = compare_residual(d, w, g["r2"], range(w.B))
    assert near <= w.B * w.K // 20
    # hit flags: the oracle's own verify outcome against its own top-F keys
    res = O.verify_batch(d["target"], d["draft"], d["draft_tokens"], d["draft_lens"],
                         d["uniforms"], temperature=w.temperature, mode="stochastic",
                         beta=w.beta, bias_k=w.bias_k, fanout=w.fanout)
    hits = 0
    for b, r in enumerate(res):
        if r.first_flag() is not None:
            continue
        ref = RO.cache_hit(r.accept_len, r.tokens, r.topf, int(d["draft_lens"][b]), w.fanout)
        assert g["hit"][b] == ref, (b, g["hit"][b], ref)
        hits += ref == 1
    print(w.name, "near ties", near, "hits", hits)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_residual_topf_planted_bias_sets(dtype):
    """Draft rows whose bias sets take every path of the kernel's selection of the draft's 8
    largest: one per group (random rows), several in one group (8 groups holding two planted
    logits each; a decreasing row), more tied candidates than the kernel lists (a row of equal
    values); ever larger logits planted across the stream. The target rows are the draft plus
    noise, so beta on the set's ids moves the residual order there."""
    V = 152064 if dtype == "bf16" else 70001
    base = _planted_rows(V, dtype)
    zd = W.bf16_bits_to_f32(base) if dtype == "bf16" else base.copy()
    rng = np.random.default_rng(33)
    pair = rng.standard_normal(V).astype(np.float32)
    groups = rng.choice(V // 64, 8, replace=False)
    for j, g in enumerate(groups):
        pair[64 * g + 5] = 11.0 + 0.25 * j
        pair[64 * g + 40] = 11.1 + 0.25 * j
    noise = rng.standard_normal((2, V)).astype(np.float32)
    zd = np.concatenate([zd, pair[None], noise[:1]], axis=0)
    B = zd.shape[0]
    zt = zd + 0.7 * rng.standard_normal(zd.shape).astype(np.float32)
    tgt = np.stack([zt, zt[::-1]], axis=1)  # position 1: the bonus row, not read here
    if dtype == "bf16":
        tgt, dft = W.f32_to_bf16_bits(tgt), W.f32_to_bf16_bits(zd[:, None])
    else:
        dft = zd[:, None].copy()
    w = W.small_variant(W.WORKLOADS[4], B=B, V=V).replace(
        K=1, fanout=(8,), beta=0.3, bias_k=8, temperature=1.0, dtype=dtype)
    d = {"target": tgt, "draft": dft, "draft_lens": np.ones(B, np.int32)}
    compare_residual(d, w, residual_gpu(d, w)["r2"], range(B))
    w3 = w.replace(fanout=(3,))
    compare_residual(d, w3, residual_gpu(d, w3)["r2"], range(B))


def test_residual_topf_zero_widths():
    """Positions whose fan-out width is 0 get no residual ids (all -1); the others their first
    F_i."""
    w = W.small_variant(W.WORKLOADS[4], B=6, V=20000).replace(fanout=(3, 0, 5, 0, 1))
    d = W.make_inputs(w)
    r2 = residual_gpu(d, w)["r2"]
    compare_residual(d, w, r2, range(w.B))
    assert (r2[:, 1] == -1).all() and (r2[:, 3] == -1).all()


def test_residual_topf_fewer_positive_than_wanted():
    """Draft rows equal to the target rows: with beta = 1 every residual is zero (all ids -1);
    with beta = 0.5 on 3 ids exactly those 3 are positive (p - beta q / N > 0 there, p - q / N < 0
    elsewhere), fewer than the 8 or 2 ids asked for, so the search must end on having no positive
    bound left rather than on an F-th best residual."""
    rng = np.random.default_rng(34)
    V, B, K = 50000, 4, 2
    zt = rng.standard_normal((B, K + 1, V)).astype(np.float32) * 2.0
    tgt = W.f32_to_bf16_bits(zt)
    dft = tgt[:, :K].copy()
    d = {"target": tgt, "draft": dft, "draft_lens": np.full(B, K, np.int32)}
    base = W.small_variant(W.WORKLOADS[4], B=B, V=V).replace(K=K, fanout=(8, 2),
                                                             temperature=1.0)
    for beta, bias_k in ((1.0, 0), (0.5, 3)):
        w = base.replace(beta=beta, bias_k=bias_k)
        r2 = residual_gpu(d, w)["r2"]
        compare_residual(d, w, r2, range(B))
        want = 0 if bias_k == 0 else bias_k
        for b in range(B):
            for i in range(K):
                got = [g for g in r2[b, i].tolist() if g >= 0]
                assert len(got) == min(want, w.fanout[i]), (beta, b, i, got)


@pytest.mark.parametrize("V", [1, 9, 3001, 50000])
def test_residual_topf_vocab_sizes_and_stride(V):
    w = W.small_variant(W.WORKLOADS[4], B=4, V=V).replace(bias_k=min(8, V))
    d = W.make_inputs(w)
    d["draft_lens"][1] = 0  # invalid length: every position -1
    compare_residual(d, w, residual_gpu(d, w)["r2"], range(w.B))
    compare_residual(d, w, residual_gpu(d, w, pad=5)["r2"], range(w.B))
    w1 = w.replace(beta=1.0, bias_k=0)
    compare_residual(d, w1, residual_gpu(d, w1)["r2"], range(w.B))
