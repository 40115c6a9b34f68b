"""Seeded synthetic inputs for the batched speculative-sampling verify step.

This module only *makes inputs*. It holds none of the verify step's own arithmetic (no softmax,
no acceptance ratio, no residual, no inverse CDF). Both the CUDA path and the float64 oracle are
fed from here, and neither of them imports the other.

The five workloads mirror the Llama/Qwen-class shapes the pages talk about (Llama-3, the
Llama-2-7B LayerSkip checkpoint and Qwen-3 are named on the SSD and LayerSkip pages); the vocab
sizes 32000 / 128256 / 152064 are those of the Llama-2, Llama-3 and Qwen families. No dataset is
read: every logit is drawn from a seeded generator.

Generation recipe (per workload ``c`` and sequence ``b``):

* Target logits ``z_t``: i.i.d. normal (workloads 1, 2) or a Zipf(1.1)-shaped log-prior
  ``l(v) = -1.1 * ln(1 + pi(v))`` plus N(0, 1) noise (workloads 3-5), where ``pi`` is a seeded
  permutation of the vocabulary shared by all rows, so frequent ids are spread over the row.
* Draft logits ``z_d = z_t + N(0, sigma_d^2)``, computed in float32 and then rounded to the
  storage type (bf16 with round-to-nearest-even, or kept as float32).
* Draft tokens: the drafter samples from its own distribution at temperature ``T`` with the
  Gumbel-max rule ``x = argmax_v(z_d[v]/T + ln f(v) + G_v)``, ``G_v ~ Gumbel(0, 1)`` in float64.
  ``f(v) = beta`` for the ``bias_k`` ids with the largest draft logit (ties to the lower id) and
  1 elsewhere; this is the Saguaro-style down-weighting of the most likely draft tokens (SSD page,
  "Method"), applied before drafting. Greedy drafters take ``argmax_v z_d[v]`` (first occurrence).
* Draft lengths: all ``K``, or uniform on ``1..K`` for the ragged workload (the dynamic
  draft length of Kangaroo's confidence exit, Kangaroo page, "Double Early Exiting").
* Uniforms: ``numpy.random.default_rng(0).random((B, K+1), float32)``; ``u[b, i]`` drives accept
  test ``i`` and ``u[b, K]`` the final sample.
* Rows that the verify step never reads (target rows ``i > L_b``, draft rows ``i >= L_b``) are
  filled with NaN so that any stray read shows up as an invalid sequence.

Seeds are ``numpy.random.default_rng([tag, c, b, offset])`` with tags 100 (target), 200 (draft
noise), 300 (drafting), 400 (Zipf permutation, per workload) and 500 (lengths); ``offset``
separates replicas (e.g. ranks of a multi-GPU weak-scaling run).
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Tuple

import numpy as np

BF16_NAN = np.uint16(0x7FC0)
F32_NAN = np.float32(np.nan)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic verify workload (shapes, dtype, mode and generation parameters)."""

    cfg_id: int
    name: str
    B: int
    K: int
    V: int
    dtype: str  # "f32" or "bf16"
    mode: str  # "stochastic" or "greedy"
    temperature: float
    sigma_t: float  # std of the target noise
    sigma_d: float  # std of the draft-vs-target noise
    zipf: bool
    ragged: bool = False
    beta: float = 1.0
    bias_k: int = 0
    fanout: Optional[Tuple[int, ...]] = None

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    1: Workload(1, "B1_K4_V32000_f32_stochastic", B=1, K=4, V=32000, dtype="f32",
                mode="stochastic", temperature=1.0, sigma_t=2.0, sigma_d=0.5, zipf=False),
    2: Workload(2, "B8_K5_V32000_bf16_greedy", B=8, K=5, V=32000, dtype="bf16",
                mode="greedy", temperature=0.0, sigma_t=3.0, sigma_d=1.0, zipf=False),
    3: Workload(3, "B64_K5_V128256_bf16_T0.8", B=64, K=5, V=128256, dtype="bf16",
                mode="stochastic", temperature=0.8, sigma_t=1.0, sigma_d=0.7, zipf=True),
    4: Workload(4, "B32_K5_V128256_bf16_saguaro_beta0.5_F84211", B=32, K=5, V=128256,
                dtype="bf16", mode="stochastic", temperature=1.0, sigma_t=1.0, sigma_d=0.7,
                zipf=True, beta=0.5, bias_k=8, fanout=(8, 4, 2, 1, 1)),
    5: Workload(5, "B256_K8_V152064_bf16_ragged", B=256, K=8, V=152064, dtype="bf16",
                mode="stochastic", temperature=1.0, sigma_t=1.0, sigma_d=0.5, zipf=True,
                ragged=True),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest, ties to even) and return the 16-bit patterns."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = bits + np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))
    out = (rounded >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = BF16_NAN
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def zipf_log_prior(w: Workload, offset: int = 0) -> np.ndarray:
    """l(v) = -1.1 ln(1 + pi(v)) with a seeded permutation pi, float32 [V]."""
    perm = np.random.default_rng([400, w.cfg_id, offset]).permutation(w.V)
    return (-1.1 * np.log1p(perm.astype(np.float64))).astype(np.float32)


def draft_lengths(w: Workload, offset: int = 0) -> np.ndarray:
    if not w.ragged:
        return np.full(w.B, w.K, dtype=np.int32)
    return np.random.default_rng([500, w.cfg_id, offset]).integers(
        1, w.K + 1, size=w.B).astype(np.int32)


def uniforms(w: Workload, offset: int = 0) -> np.ndarray:
    seed = 0 if offset == 0 else [0, offset]
    return np.random.default_rng(seed).random((w.B, w.K + 1), dtype=np.float32)


def _top_set(zd: np.ndarray, k: int) -> np.ndarray:
    """Ids of the k largest entries (ties to the lower id) -- the drafter's down-weighted set."""
    k = min(k, zd.shape[0])
    if k <= 0:
        return np.zeros(0, dtype=np.int64)
    order = np.lexsort((np.arange(zd.shape[0]), -zd.astype(np.float64)))
    return order[:k]


def _draw_draft(zd_row: np.ndarray, w: Workload, rng: np.random.Generator) -> int:
    z = zd_row.astype(np.float64)
    if w.mode == "greedy":
        return int(np.argmax(z))
    score = z / w.temperature
    if w.beta < 1.0 and w.bias_k > 0:
        score[_top_set(z, w.bias_k)] += np.log(w.beta)
    return int(np.argmax(score + rng.gumbel(size=z.shape[0])))


def _make_sequence(w: Workload, b: int, L: int, prior, offset: int, tgt_out, dft_out, tok_out):
    rng_t = np.random.default_rng([100, w.cfg_id, b, offset])
    rng_d = np.random.default_rng([200, w.cfg_id, b, offset])
    rng_x = np.random.default_rng([300, w.cfg_id, b, offset])
    V, K = w.V, w.K
    rows_t = L + 1
    zt = rng_t.standard_normal((rows_t, V), dtype=np.float32)
    zt *= np.float32(w.sigma_t)
    if prior is not None:
        zt += prior
    zd = zt[:L] + np.float32(w.sigma_d) * rng_d.standard_normal((L, V), dtype=np.float32)
    if w.dtype == "bf16":
        tgt_out[b, :rows_t] = f32_to_bf16_bits(zt)
        tgt_out[b, rows_t:] = BF16_NAN
        zd_store = f32_to_bf16_bits(zd)
        dft_out[b, :L] = zd_store
        dft_out[b, L:] = BF16_NAN
        zd_seen = bf16_bits_to_f32(zd_store)
    else:
        tgt_out[b, :rows_t] = zt
        tgt_out[b, rows_t:] = F32_NAN
        dft_out[b, :L] = zd
        dft_out[b, L:] = F32_NAN
        zd_seen = zd
    tok_out[b, :] = 0
    for i in range(L):
        tok_out[b, i] = _draw_draft(zd_seen[i], w, rng_x)


def make_inputs(w: Workload, offset: int = 0, threads: Optional[int] = None) -> dict:
    """Generate one batch for workload ``w``.

    Returns a dict of numpy arrays: ``target`` [B, K+1, V] and ``draft`` [B, K, V] (uint16 bf16
    bit patterns or float32), ``draft_tokens`` [B, K] int32, ``draft_lens`` [B] int32 and
    ``uniforms`` [B, K+1] float32, plus the workload itself under ``workload``.
    """
    B, K, V = w.B, w.K, w.V
    store = np.uint16 if w.dtype == "bf16" else np.float32
    tgt = np.empty((B, K + 1, V), dtype=store)
    dft = np.empty((B, K, V), dtype=store)
    tok = np.zeros((B, K), dtype=np.int32)
    lens = draft_lengths(w, offset)
    prior = zipf_log_prior(w, offset) if w.zipf else None
    if threads is None:
        threads = min(16, len(os.sched_getaffinity(0)))
    if B:
        with ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
            list(ex.map(lambda b: _make_sequence(w, b, int(lens[b]), prior, offset,
                                                 tgt, dft, tok), range(B)))
    return {"workload": w, "target": tgt, "draft": dft, "draft_tokens": tok,
            "draft_lens": lens, "uniforms": uniforms(w, offset)}


def small_variant(w: Workload, B: int, V: Optional[int] = None) -> Workload:
    """Same generation recipe at a smaller batch (and optionally vocabulary)."""
    return w.replace(B=B, V=V if V is not None else w.V)


# ---------------------------------------------------------------------------------------------
# LM-head inputs: hidden states and a head matrix whose product gives logits of the shape above
# ---------------------------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class HeadWorkload:
    """Hidden states [R, d] and an LM head [V, d] (bf16) for the fused head statistics.

    ``R`` counts the rows one verify step scores: ``B * (K + 1)`` target rows plus ``B * K``
    draft rows of the matching verify workload (the early-exit draft of LayerSkip and Kangaroo
    shares the full model's head, so both go through the same matrix). ``d`` is the hidden size
    of the model family the vocabulary belongs to (4096 for Llama-2/3 8B-class models, 3584 for
    the Qwen model with 152064 ids)."""

    name: str
    R: int
    d: int
    V: int
    temperature: float
    sigma: float = 2.0  # standard deviation of the logits' noise part
    zipf: bool = True


HEAD_WORKLOADS = {
    "head_B64_K5_V128256_d4096": HeadWorkload("head_B64_K5_V128256_d4096", R=64 * 6 + 64 * 5,
                                              d=4096, V=128256, temperature=0.8),
    "head_B256_K8_V152064_d3584": HeadWorkload("head_B256_K8_V152064_d3584",
                                               R=256 * 9 + 256 * 8, d=3584, V=152064,
                                               temperature=1.0),
}


def head_inputs(w: HeadWorkload, offset: int = 0) -> dict:
    """Seeded hidden states, head and ids for ``w``.

    Recipe: hidden ``h[r, j] ~ N(0, 1)`` for ``j < d - 1`` and ``h[r, d-1] = 1``; head
    ``W[v, j] ~ N(0, sigma^2 / (d - 1))`` for ``j < d - 1`` and ``W[v, d-1]`` = the Zipf(1.1)
    log-prior of the verify workloads (0 when ``zipf`` is off). The logits ``h W^T`` are then
    about prior + N(0, sigma^2) per row, the shape of the verify workloads' target rows. Both
    are rounded to bf16 (round to nearest even). ``ids[r]`` is a uniform id in ``[0, V)``.
    Seeds: ``default_rng([600 | 800 | 400, R, d, V, offset])`` (hidden, ids, prior) and
    ``default_rng([700, R, d, V, offset, v0])`` for the head's rows ``v0 .. v0 + 4095``.
    Returns ``hidden`` [R, d] and ``weight`` [V, d] as uint16 bit patterns and ``ids`` [R]
    int32."""
    R, d, V = w.R, w.d, w.V
    rng_h = np.random.default_rng([600, R, d, V, offset])
    rng_i = np.random.default_rng([800, R, d, V, offset])
    h = rng_h.standard_normal((R, d), dtype=np.float32)
    h[:, d - 1] = 1.0
    hidden = f32_to_bf16_bits(h)
    del h
    weight = np.empty((V, d), dtype=np.uint16)
    scale = np.float32(w.sigma / np.sqrt(max(1, d - 1)))
    if w.zipf:
        perm = np.random.default_rng([400, R, d, V, offset]).permutation(V)
        prior = (-1.1 * np.log1p(perm.astype(np.float64))).astype(np.float32)
    else:
        prior = np.zeros(V, dtype=np.float32)
    step = 4096

    def fill(v0: int) -> None:
        rng_w = np.random.default_rng([700, R, d, V, offset, v0])
        blk = rng_w.standard_normal((min(step, V - v0), d), dtype=np.float32)
        blk *= scale
        blk[:, d - 1] = prior[v0:v0 + blk.shape[0]]
        weight[v0:v0 + blk.shape[0]] = f32_to_bf16_bits(blk)

    threads = min(16, len(os.sched_getaffinity(0)))
    with ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
        list(ex.map(fill, range(0, V, step)))
    ids = rng_i.integers(0, V, size=R).astype(np.int32)
    return {"workload": w, "hidden": hidden, "weight": weight, "ids": ids}


def small_head(R: int, d: int, V: int, temperature: float = 1.0, zipf: bool = True,
               sigma: float = 2.0) -> HeadWorkload:
    """A head workload of the same recipe at other sizes (tests)."""
    return HeadWorkload(f"head_R{R}_d{d}_V{V}", R=R, d=d, V=V, temperature=temperature,
                        sigma=sigma, zipf=zipf)


# ---------------------------------------------------------------------------------------------
# verify-from-hidden-states inputs
# ---------------------------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class HiddenWorkload:
    """Hidden states of the target and early-exit draft rows of B sequences and an LM head."""

    name: str
    B: int
    K: int
    V: int
    d: int
    mode: str = "stochastic"
    temperature: float = 1.0
    ragged: bool = True
    sigma: float = 2.0        # standard deviation of a logit's noise part
    sigma_d: float = 0.25     # draft hidden state = target's + N(0, sigma_d^2) per unit
    exact: bool = False       # values on dyadic grids: every logit is exact in float32
    drafter: str = "head"     # "head": x ~ the draft head's softmax; "prior": x ~ softmax(prior/T)


HIDDEN_WORKLOADS = {
    "hv_B256_K8_V152064_d3584": HiddenWorkload("hv_B256_K8_V152064_d3584", B=256, K=8,
                                               V=152064, d=3584, drafter="prior"),
}


def _grid(x: np.ndarray, step: float, lim: int) -> np.ndarray:
    """x rounded to a multiple of `step` with at most `lim` steps either way."""
    return (np.clip(np.rint(x / step), -lim, lim) * step).astype(np.float32)


def hidden_inputs(w: HiddenWorkload, offset: int = 0) -> dict:
    """Seeded hidden states, head, draft ids, lengths and uniforms for ``w``.

    Recipe: head rows ``W[v, j] ~ N(0, sigma^2 / (d - 1))`` for ``j < d - 1`` and ``W[v, d-1]`` the
    Zipf(1.1) log-prior; target hidden states ``h ~ N(0, 1)`` with ``h[d-1] = 1``; draft hidden
    states ``h + N(0, sigma_d^2)`` (last unit 1), so the draft logits are the target's plus noise.
    With ``exact`` every value sits on a dyadic grid (h on 1/8 within +-31/8, W on 1/256 within
    +-127/256, the prior on 1/16) so that any float32 sum of d <= 1024 products is exact. All are
    rounded to bf16. Rows past a sequence's draft length are NaN (never to be read). Draft ids:
    with ``drafter="head"`` the drafter scores its rows with the head in float32 and samples by
    the Gumbel-max rule at temperature T (greedy: argmax); with ``"prior"`` it samples from
    softmax(prior / T) alone (cheap at full size). Lengths: all K, or uniform on 1..K when
    ragged; uniforms as ``uniforms``. Seeds: ``default_rng([tag, B, K, V, d, offset])`` with tags
    900 (head), 901 (hidden), 902 (draft noise), 903 (drafting), 904 (prior), 905 (lengths).
    """
    B, K, V, d = w.B, w.K, w.V, w.d
    key = [B, K, V, d, offset]
    perm = np.random.default_rng([904] + key).permutation(V)
    prior = (-1.1 * np.log1p(perm.astype(np.float64))).astype(np.float32)
    if w.exact:
        prior = _grid(prior, 1.0 / 16, 255)
    weight = np.empty((V, d), dtype=np.uint16)
    scale = np.float32(w.sigma / np.sqrt(max(1, d - 1)))
    step = 4096

    def fill(v0: int) -> None:
        rng = np.random.default_rng([900] + key + [v0])
        blk = rng.standard_normal((min(step, V - v0), d), dtype=np.float32) * scale
        if w.exact:
            blk = _grid(blk, 1.0 / 256, 127)
        blk[:, d - 1] = prior[v0:v0 + blk.shape[0]]
        weight[v0:v0 + blk.shape[0]] = f32_to_bf16_bits(blk)

    threads = min(16, len(os.sched_getaffinity(0)))
    with ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
        list(ex.map(fill, range(0, V, step)))
    if w.ragged:
        lens = np.random.default_rng([905] + key).integers(1, K + 1, size=B).astype(np.int32)
    else:
        lens = np.full(B, K, dtype=np.int32)
    h = np.random.default_rng([901] + key).standard_normal((B, K + 1, d), dtype=np.float32)
    hd = h[:, :K] + np.float32(w.sigma_d) * np.random.default_rng([902] + key).standard_normal(
        (B, K, d), dtype=np.float32)
    if w.exact:
        h, hd = _grid(h, 1.0 / 8, 31), _grid(hd, 1.0 / 8, 31)
    h[..., d - 1] = 1.0
    hd[..., d - 1] = 1.0
    ht_bits, hd_bits = f32_to_bf16_bits(h), f32_to_bf16_bits(hd)
    del h
    rng_x = np.random.default_rng([903] + key)
    tok = np.zeros((B, K), dtype=np.int32)
    Wf = bf16_bits_to_f32(weight) if w.drafter == "head" else None
    T = w.temperature if w.mode == "stochastic" else 1.0
    for b in range(B):
        L = int(lens[b])
        if w.drafter == "head":
            zd = bf16_bits_to_f32(hd_bits[b, :L]) @ Wf.T
        else:
            zd = np.broadcast_to(prior, (L, V))
        for i in range(L):
            z = zd[i].astype(np.float64)
            if w.mode == "greedy":
                tok[b, i] = int(np.argmax(z))
            else:
                tok[b, i] = int(np.argmax(z / T + rng_x.gumbel(size=V)))
        ht_bits[b, L + 1:] = BF16_NAN
        hd_bits[b, L:] = BF16_NAN
    uni = np.random.default_rng(0 if offset == 0 else [0, offset]).random((B, K + 1),
                                                                           dtype=np.float32)
    return {"workload": w, "hidden_target": ht_bits, "hidden_draft": hd_bits, "weight": weight,
            "draft_tokens": tok, "draft_lens": lens, "uniforms": uni}
