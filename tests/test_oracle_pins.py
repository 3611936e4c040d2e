"""Pins for the fp64 oracle, checked against things other than the oracle itself.

The attention page (oxicuda-dnn 0.1.8 hopper.rs) prints no attention values,
so every pin here is fixed by mathematics: a hand-derived worked example,
brute force on tiny inputs by independent pure-Python loops, closed forms,
invariants, and a library special case.  ``test_pins_catch_planted_mistakes``
plants plausible mistakes in the oracle (on the CPU) and checks that at least
one pin fails for each.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import oracle.attention as oa

RNG = np.random.default_rng(12345)


def _fwd(q, k, v, causal, scale, row_block=512):
    return oracle.attention_forward(q, k, v, causal=causal, scale=scale, row_block=row_block)


def _loops(q, k, v, causal, scale, offset=0):
    """Attention by explicit Python loops over one head: q [S_q][d] lists."""
    S_q, S_k, d = len(q), len(k), len(q[0])
    o, lse = [], []
    for i in range(S_q):
        logits = []
        for j in range(S_k):
            if causal and j > i + offset:
                continue
            dot = 0.0
            for c in range(d):
                dot += q[i][c] * k[j][c]
            logits.append((j, scale * dot))
        mx = max(t for _, t in logits)
        w = [(j, math.exp(t - mx)) for j, t in logits]
        tot = sum(x for _, x in w)
        o.append([sum(x * v[j][c] for j, x in w) / tot for c in range(len(v[0]))])
        lse.append(mx + math.log(tot))
    return o, lse


# --------------------------------------------------------------------------- pins
def pin_worked_example():
    """A 2×2, d=2 example derived by hand (asymmetric, so transposes show)."""
    q = np.array([[[[1.0, 0.0], [0.0, 2.0]]]])
    k = np.array([[[[1.0, 1.0], [0.0, -1.0]]]])
    v = np.array([[[[3.0, 0.0], [0.0, 5.0]]]])
    e = math.e
    # non-causal: row 0 logits (0.5, 0); row 1 logits (1, -1)
    o, lse = _fwd(q, k, v, False, 0.5)
    r0 = np.array([3 * math.exp(0.5), 5.0]) / (math.exp(0.5) + 1)
    r1 = np.array([3 * e, 5 / e]) / (e + 1 / e)
    np.testing.assert_allclose(o[0, 0, 0], r0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(o[0, 0, 1], r1, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], [math.log(math.exp(0.5) + 1), math.log(e + 1 / e)],
                               rtol=0, atol=1e-14)
    # causal: row 0 sees key 0 only
    o, lse = _fwd(q, k, v, True, 0.5)
    np.testing.assert_allclose(o[0, 0, 0], [3.0, 0.0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0, 0], 0.5, rtol=0, atol=1e-14)
    np.testing.assert_allclose(o[0, 0, 1], r1, rtol=0, atol=1e-14)


def pin_brute_force():
    """Tiny random cases against independent pure-Python loops."""
    for (S_q, S_k, d, dv) in [(2, 2, 1, 1), (4, 4, 2, 2), (3, 5, 2, 3), (5, 3, 3, 2)]:
        for causal in (False, True):
            q = RNG.standard_normal((1, 2, S_q, d))
            k = RNG.standard_normal((1, 2, S_k, d))
            v = RNG.standard_normal((1, 2, S_k, dv))
            scale = 0.7
            o, lse = _fwd(q, k, v, causal, scale)
            for h in range(2):
                ro, rl = _loops(q[0, h].tolist(), k[0, h].tolist(), v[0, h].tolist(), causal, scale)
                np.testing.assert_allclose(o[0, h], np.array(ro), rtol=0, atol=1e-13)
                np.testing.assert_allclose(lse[0, h], np.array(rl), rtol=0, atol=1e-13)


def pin_constant_v():
    """V = c in every row gives O = c for every query (softmax rows sum to 1)."""
    q = RNG.standard_normal((2, 3, 37, 8))
    k = RNG.standard_normal((2, 3, 41, 8))
    c = RNG.standard_normal(8)
    v = np.broadcast_to(c, (2, 3, 41, 8)).copy()
    for causal in (False, True):
        o, _ = _fwd(q, k, v, causal, 0.9)
        np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-13)


def pin_scale_zero():
    """scale = 0: O is the mean of the visible V rows, LSE = ln(#visible)."""
    q = RNG.standard_normal((1, 2, 19, 4))
    k = RNG.standard_normal((1, 2, 19, 4))
    v = RNG.standard_normal((1, 2, 19, 4))
    o, lse = _fwd(q, k, v, False, 0.0)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape),
                               rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, math.log(19), rtol=0, atol=1e-13)
    o, lse = _fwd(q, k, v, True, 0.0)
    n = np.arange(1, 20)
    np.testing.assert_allclose(o, np.cumsum(v, axis=2) / n[None, None, :, None], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(n), lse.shape), rtol=0, atol=1e-13)


def pin_causal_first_row():
    """Causal row 0 attends to key 0 alone: O_0 = V_0 and LSE_0 = scale·q_0·k_0."""
    q = RNG.standard_normal((2, 2, 9, 16))
    k = RNG.standard_normal((2, 2, 9, 16))
    v = RNG.standard_normal((2, 2, 9, 16))
    o, lse = _fwd(q, k, v, True, 0.3)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[:, :, 0], 0.3 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]),
                               rtol=0, atol=1e-13)


def pin_one_hot_selection():
    """One-hot keys and a large scale select the V row of the matching key."""
    S, d = 6, 8
    k = np.eye(d)[:S][None, None]
    target = np.array([3, 0, 5, 1, 4, 2])
    q = np.eye(d)[target][None, None]
    v = RNG.standard_normal((1, 1, S, d))
    o, lse = _fwd(q, k, v, False, 200.0)
    np.testing.assert_allclose(o[0, 0], v[0, 0, target], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], 200.0, rtol=0, atol=1e-12)


def pin_key_permutation():
    """Non-causal attention is invariant under a joint permutation of K and V rows."""
    q = RNG.standard_normal((1, 2, 13, 8))
    k = RNG.standard_normal((1, 2, 21, 8))
    v = RNG.standard_normal((1, 2, 21, 5))
    perm = RNG.permutation(21)
    o1, l1 = _fwd(q, k, v, False, 0.4)
    o2, l2 = _fwd(q, k[:, :, perm], v[:, :, perm], False, 0.4)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def pin_key_shift():
    """K + u in every row: O unchanged, LSE_i shifted by scale·q_i·u."""
    q = RNG.standard_normal((1, 2, 11, 8))
    k = RNG.standard_normal((1, 2, 11, 8))
    v = RNG.standard_normal((1, 2, 11, 8))
    u = RNG.standard_normal(8)
    for causal in (False, True):
        o1, l1 = _fwd(q, k, v, causal, 0.6)
        o2, l2 = _fwd(q, k + u, v, causal, 0.6)
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l2 - l1, 0.6 * (q @ u), rtol=0, atol=1e-12)


def pin_log_domain_form():
    """O_i = Σ_j exp(scale·q_i·k_j − LSE_i)·v_j over the visible keys."""
    q = RNG.standard_normal((1, 1, 10, 4))
    k = RNG.standard_normal((1, 1, 10, 4))
    v = RNG.standard_normal((1, 1, 10, 3))
    for causal in (False, True):
        o, lse = _fwd(q, k, v, causal, 1.3)
        for i in range(10):
            vis = range(i + 1) if causal else range(10)
            acc = np.zeros(3)
            for j in vis:
                acc += math.exp(1.3 * float(q[0, 0, i] @ k[0, 0, j]) - lse[0, 0, i]) * v[0, 0, j]
            np.testing.assert_allclose(o[0, 0, i], acc, rtol=0, atol=1e-12)


def pin_library_sdpa():
    """PyTorch's fp64 CPU scaled_dot_product_attention and logsumexp agree."""
    g = torch.Generator().manual_seed(7)
    for (S_q, S_k, causal) in [(33, 33, False), (33, 33, True), (17, 40, False), (40, 17, True)]:
        q = torch.randn(2, 3, S_q, 16, generator=g, dtype=torch.float64)
        k = torch.randn(2, 3, S_k, 16, generator=g, dtype=torch.float64)
        v = torch.randn(2, 3, S_k, 16, generator=g, dtype=torch.float64)
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=0.25)
        s = 0.25 * q @ k.transpose(-1, -2)
        if causal:
            s = s.masked_fill(torch.ones(S_q, S_k, dtype=torch.bool).triu(1), float("-inf"))
        ref_lse = torch.logsumexp(s, dim=-1)
        o, lse = _fwd(q.numpy(), k.numpy(), v.numpy(), causal, 0.25)
        np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=0, atol=1e-12)


def pin_rows_and_blocks_agree():
    """Sampled-row evaluation and any row blocking give the same rows."""
    q = RNG.standard_normal((1, 2, 70, 8))
    k = RNG.standard_normal((1, 2, 70, 8))
    v = RNG.standard_normal((1, 2, 70, 8))
    for causal in (False, True):
        o, lse = _fwd(q, k, v, causal, 0.5)
        o7, lse7 = _fwd(q, k, v, causal, 0.5, row_block=7)
        np.testing.assert_array_equal(o, o7)
        np.testing.assert_array_equal(lse, lse7)
        rows = [0, 5, 31, 69]
        ro, rl = oracle.attention_rows(q[0, 1], k[0, 1], v[0, 1], rows, causal, 0.5)
        np.testing.assert_allclose(ro, o[0, 1, rows], rtol=0, atol=1e-14)
        np.testing.assert_allclose(rl, lse[0, 1, rows], rtol=0, atol=1e-14)


def pin_bottom_right_square_is_top_left():
    """With S_q = S_k the two causal alignments coincide."""
    q, k, v = RNG.standard_normal((3, 1, 2, 23, 8))
    a = _fwd(q, k, v, True, 0.3)
    b = oracle.attention_forward(q, k, v, causal=True, scale=0.3, bottom_right=True)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def pin_bottom_right_is_tail_of_square():
    """S_q < S_k, bottom-right: the last S_q rows of a top-left causal S_k × S_k problem."""
    S_q, S_k, d = 9, 30, 8
    k, v = RNG.standard_normal((2, 1, 1, S_k, d))
    q_tail = RNG.standard_normal((1, 1, S_q, d))
    q_full = np.concatenate([RNG.standard_normal((1, 1, S_k - S_q, d)), q_tail], axis=2)
    full_o, full_l = _fwd(q_full, k, v, True, 0.4)
    o, l = oracle.attention_forward(q_tail, k, v, causal=True, scale=0.4, bottom_right=True)
    np.testing.assert_allclose(o, full_o[:, :, S_k - S_q:], rtol=0, atol=1e-13)
    np.testing.assert_allclose(l, full_l[:, :, S_k - S_q:], rtol=0, atol=1e-13)


def pin_bottom_right_loops():
    """Brute force with the shifted mask, S_q = 5 against S_k = 8."""
    q, k, v = RNG.standard_normal((5, 3)), RNG.standard_normal((8, 3)), RNG.standard_normal((8, 2))
    lo, ll = _loops(q.tolist(), k.tolist(), v.tolist(), True, 0.8, offset=3)
    o, l = oracle.attention_forward(q[None, None], k[None, None], v[None, None], causal=True,
                                    scale=0.8, bottom_right=True)
    np.testing.assert_allclose(o[0, 0], np.array(lo), rtol=0, atol=1e-13)
    np.testing.assert_allclose(l[0, 0], np.array(ll), rtol=0, atol=1e-13)


def pin_negative_scale():
    """Any finite scale: a negative one against PyTorch's fp64 SDPA and a closed form.

    With one-hot keys, q_i = e_t and scale −200, key t gets logit −200 and every
    other key 0, so O_i is the mean of the other V rows and LSE_i = ln(S − 1 + e^−200).
    """
    g = torch.Generator().manual_seed(9)
    for causal in (False, True):
        q, k, v = (torch.randn(1, 2, 21, 8, generator=g, dtype=torch.float64) for _ in range(3))
        if causal:
            # (PyTorch's math SDPA returns NaN for a negative scale under is_causal, so the
            # masked case goes through torch.softmax directly.)
            s = (-0.4 * q @ k.transpose(-1, -2)).masked_fill(
                torch.ones(21, 21, dtype=torch.bool).triu(1), float("-inf"))
            ref = torch.softmax(s, dim=-1) @ v
        else:
            ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=-0.4)
        o, _ = _fwd(q.numpy(), k.numpy(), v.numpy(), causal, -0.4)
        np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
    S, d = 6, 8
    k = np.eye(d)[:S][None, None]
    target = np.array([3, 0, 5, 1, 4, 2])
    q = np.eye(d)[target][None, None]
    v = RNG.standard_normal((1, 1, S, d))
    o, lse = _fwd(q, k, v, False, -200.0)
    for i, t in enumerate(target):
        others = [j for j in range(S) if j != t]
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, others].mean(axis=0), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], math.log(S - 1 + math.exp(-200.0)), rtol=0, atol=1e-13)


PINS = [pin_worked_example, pin_brute_force, pin_constant_v, pin_scale_zero,
        pin_causal_first_row, pin_one_hot_selection, pin_key_permutation, pin_key_shift,
        pin_log_domain_form, pin_library_sdpa, pin_rows_and_blocks_agree,
        pin_bottom_right_square_is_top_left, pin_bottom_right_is_tail_of_square,
        pin_bottom_right_loops, pin_negative_scale]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin()


def pin_probs_worked_example(probs):
    """attention_probs on a 2×2 case derived by hand: with q = k = I and scale = ln 3 the
    logits are [[ln 3, 0], [0, ln 3]], so the rows are [3/4, 1/4] and [1/4, 3/4]; scale −ln 3
    swaps them; causal row 0 is [1, 0] and row 1 stays [1/4, 3/4]."""
    eye = np.eye(2)
    ln3 = math.log(3.0)
    np.testing.assert_allclose(probs(eye, eye, causal=False, scale=ln3),
                               [[0.75, 0.25], [0.25, 0.75]], rtol=0, atol=1e-15)
    np.testing.assert_allclose(probs(eye, eye, causal=False, scale=-ln3),
                               [[0.25, 0.75], [0.75, 0.25]], rtol=0, atol=1e-15)
    np.testing.assert_allclose(probs(eye, eye, causal=True, scale=ln3),
                               [[1.0, 0.0], [0.25, 0.75]], rtol=0, atol=1e-15)
    # an asymmetric case, so a transposed product shows: logits [[ln 3, 0], [2 ln 3, 0]]
    q = np.array([[1.0, 0.0], [2.0, 0.0]])
    k = np.array([[1.0, 0.0], [0.0, 1.0]])
    np.testing.assert_allclose(probs(q, k, causal=False, scale=ln3),
                               [[0.75, 0.25], [0.9, 0.1]], rtol=0, atol=1e-15)


def test_probs_worked_example():
    pin_probs_worked_example(oracle.attention_probs)


@pytest.mark.parametrize("kind", ["no_scale", "inverse_scale", "transposed", "mask_flipped"])
def test_probs_pin_catches_planted_mistakes(kind):
    def probs(q, k, causal=False, scale=None):
        s = scale * (q @ k.T)
        if kind == "no_scale":
            s = q @ k.T
        elif kind == "inverse_scale":
            s = (q @ k.T) / scale
        elif kind == "transposed":
            s = scale * (k @ q.T)
        if causal:
            i = np.arange(q.shape[0])[:, None]
            j = np.arange(k.shape[0])[None, :]
            s = np.where((j < i) if kind == "mask_flipped" else (j > i), -np.inf, s)
        e = np.exp(s - s.max(axis=1, keepdims=True))
        return e / e.sum(axis=1, keepdims=True)
    with pytest.raises(AssertionError):
        pin_probs_worked_example(probs)


def test_probs_rows_sum_to_one_and_mask():
    q = RNG.standard_normal((23, 8))
    k = RNG.standard_normal((23, 8))
    for causal in (False, True):
        p = oracle.attention_probs(q, k, causal=causal, scale=0.8)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        assert (p >= 0).all()
        if causal:
            assert (np.triu(p, 1) == 0).all()
            assert (np.diag(p) > 0).all()


def test_default_scale_is_inverse_sqrt_d():
    q = RNG.standard_normal((1, 1, 5, 16))
    k = RNG.standard_normal((1, 1, 5, 16))
    v = RNG.standard_normal((1, 1, 5, 16))
    o1, l1 = oracle.attention_forward(q, k, v)
    o2, l2 = oracle.attention_forward(q, k, v, scale=0.25)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_half_inputs_are_widened_exactly():
    t = torch.randn(1, 1, 4, 8).to(torch.bfloat16)
    assert oa._as_f64(t).dtype == np.float64
    np.testing.assert_array_equal(oa._as_f64(t), t.float().numpy().astype(np.float64))


# ------------------------------------------------------- planted mistakes
def _mutant(kind):
    def head(q, k, v, rows, causal, scale, offset=0):
        if kind == "offset_ignored":
            offset = 0
        if kind == "offset_sign":
            offset = -offset
        s = scale * (q[rows] @ k.T)
        if kind == "no_scale":
            s = q[rows] @ k.T
        if kind == "inverse_scale":
            s = (q[rows] @ k.T) / scale if scale else s
        if kind == "transposed":
            s = scale * (k @ q.T)[: len(rows)][:, : k.shape[0]] if k.shape[0] == q.shape[0] else s.T
        if causal:
            keys = np.arange(k.shape[0])
            r = rows[:, None] + offset
            if kind == "mask_off_by_one":
                s = np.where(keys[None, :] >= r, -np.inf, s)
            elif kind == "mask_flipped":
                s = np.where(keys[None, :] < r, -np.inf, s)
            elif kind == "mask_zero_score":
                s = np.where(keys[None, :] > r, 0.0, s)
            else:
                s = np.where(keys[None, :] > r, -np.inf, s)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=1, keepdims=True)
        o = (p @ v) / l
        if kind == "no_normalise":
            o = p @ v
        lse = m[:, 0] + np.log(l[:, 0])
        if kind == "lse_log2":
            lse = m[:, 0] + np.log2(l[:, 0])
        if kind == "lse_no_max":
            lse = np.log(l[:, 0])
        if kind == "lse_unscaled":
            lse = (m[:, 0] + np.log(l[:, 0])) / scale if scale else lse
        return o, lse
    return head


MUTANTS = ["no_scale", "inverse_scale", "transposed", "mask_off_by_one", "mask_flipped",
           "mask_zero_score", "no_normalise", "lse_log2", "lse_no_max", "lse_unscaled",
           "offset_ignored", "offset_sign"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_catch_planted_mistakes(kind, monkeypatch):
    monkeypatch.setattr(oa, "_head", _mutant(kind))
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {kind!r}"


def test_unmutated_head_passes_all_pins(monkeypatch):
    """The mutant harness with no mistake planted passes, so failures above are the plants'."""
    monkeypatch.setattr(oa, "_head", _mutant("none"))
    for pin in PINS:
        pin()
