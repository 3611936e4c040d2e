"""Pins for the fp64 backward oracle, fixed by things other than the oracle itself.

* central finite differences of the forward oracle (a separate code path:
  it never forms a gradient) on tiny inputs, every element of Q, K and V;
* torch autograd in fp64 through an independently written attention;
* invariants of softmax attention: key gradients sum to zero (a softmax row
  does not change when a constant is added to its logits), Σ_j dV_j = Σ_i dO_i,
  identical keys give dQ = 0, under causal masking query 0 sees one key so
  dQ_0 = 0, scale 0 gives dQ = dK = 0 and uniform weights in dV;
* the page's two forms of D agree: rowsum(dP ∘ P) = rowsum(dO ∘ O).

``test_bwd_pins_catch_planted_mistakes`` plants plausible mistakes in the
oracle (on the CPU) and checks that some pin fails for each.
"""

import numpy as np
import pytest
import torch

import oracle
import oracle.attention_bwd as oab

RNG = np.random.default_rng(2024)


def _rand(*shape):
    return RNG.standard_normal(shape)


def _loss(q, k, v, do, causal, scale, bottom_right=False):
    o, _ = oracle.attention_forward(q, k, v, causal=causal, scale=scale, bottom_right=bottom_right)
    return float((o * do).sum())


# --------------------------------------------------------------------------- pins
def pin_finite_differences():
    h = 1e-6
    for causal in (False, True):
        q, k, v = _rand(1, 1, 3, 3), _rand(1, 1, 4, 3), _rand(1, 1, 4, 2)
        do = _rand(1, 1, 3, 2)
        scale = 0.7
        dq, dk, dv = oab.attention_backward(q, k, v, do, causal=causal, scale=scale)
        for x, g in ((q, dq), (k, dk), (v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                x0 = x[idx]
                x[idx] = x0 + h
                lp = _loss(q, k, v, do, causal, scale)
                x[idx] = x0 - h
                lm = _loss(q, k, v, do, causal, scale)
                x[idx] = x0
                num[idx] = (lp - lm) / (2 * h)
            np.testing.assert_allclose(g, num, rtol=0, atol=2e-7)


def pin_finite_differences_bottom_right():
    """The shifted mask (S_q = 3 against S_k = 5) against differences of the forward oracle."""
    h = 1e-6
    q, k, v, do = _rand(1, 1, 3, 3), _rand(1, 1, 5, 3), _rand(1, 1, 5, 2), _rand(1, 1, 3, 2)
    dq, dk, dv = oab.attention_backward(q, k, v, do, causal=True, scale=0.6, bottom_right=True)
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            x0 = x[idx]
            x[idx] = x0 + h
            lp = _loss(q, k, v, do, True, 0.6, True)
            x[idx] = x0 - h
            lm = _loss(q, k, v, do, True, 0.6, True)
            x[idx] = x0
            num[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=0, atol=2e-7)


def pin_torch_autograd():
    for causal in (False, True):
        S_q, S_k, d = 37, 53, 16
        q, k, v, do = _rand(1, 2, S_q, d), _rand(1, 2, S_k, d), _rand(1, 2, S_k, d), _rand(1, 2, S_q, d)
        scale = 0.3
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        logits = scale * tq @ tk.transpose(-1, -2)
        if causal:
            keep = torch.ones(S_q, S_k, dtype=torch.bool).tril()
            logits = logits.masked_fill(~keep, float("-inf"))
        out = torch.softmax(logits, dim=-1) @ tv
        (out * torch.tensor(do)).sum().backward()
        dq, dk, dv = oab.attention_backward(q, k, v, do, causal=causal, scale=scale)
        np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-11)
        np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-11)
        np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-11)


def pin_invariants():
    for causal in (False, True):
        q, k, v, do = _rand(1, 1, 20, 8), _rand(1, 1, 20, 8), _rand(1, 1, 20, 8), _rand(1, 1, 20, 8)
        dq, dk, dv = oab.attention_backward(q, k, v, do, causal=causal, scale=0.4)
        np.testing.assert_allclose(dk[0, 0].sum(axis=0), 0.0, atol=1e-12)
        np.testing.assert_allclose(dv[0, 0].sum(axis=0), do[0, 0].sum(axis=0), atol=1e-12)
        if causal:
            np.testing.assert_allclose(dq[0, 0, 0], 0.0, atol=1e-14)
    # identical keys: every softmax row is uniform whatever Q is
    q, v, do = _rand(1, 1, 6, 4), _rand(1, 1, 9, 4), _rand(1, 1, 6, 4)
    k = np.repeat(_rand(1, 1, 1, 4), 9, axis=2)
    dq, _, _ = oab.attention_backward(q, k, v, do, causal=False, scale=0.9)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)
    # scale 0: uniform weights, no logit gradients
    q, k, v, do = _rand(1, 1, 5, 4), _rand(1, 1, 7, 4), _rand(1, 1, 7, 4), _rand(1, 1, 5, 4)
    dq, dk, dv = oab.attention_backward(q, k, v, do, causal=False, scale=0.0)
    np.testing.assert_allclose(dq, 0.0, atol=0)
    np.testing.assert_allclose(dk, 0.0, atol=0)
    np.testing.assert_allclose(dv[0, 0], np.tile(do[0, 0].sum(axis=0) / 7, (7, 1)), atol=1e-14)


def pin_two_forms_of_d():
    for causal in (False, True):
        q, k, v, do = _rand(30, 8), _rand(41, 8), _rand(41, 8), _rand(30, 8)
        t = oab.backward_terms(q, k, v, do, causal=causal, scale=0.5)
        np.testing.assert_allclose((t["dP"] * t["P"]).sum(axis=1), t["D"], atol=1e-12)
        o, _ = oracle.attention_rows(q, k, v, np.arange(30), causal=causal, scale=0.5)
        np.testing.assert_allclose(t["O"], o, atol=1e-13)


PINS = [pin_finite_differences, pin_finite_differences_bottom_right, pin_torch_autograd,
        pin_invariants, pin_two_forms_of_d]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_bwd_oracle_pin(pin):
    pin()


def test_default_scale_is_inverse_sqrt_d():
    q, k, v, do = _rand(1, 1, 5, 16), _rand(1, 1, 6, 16), _rand(1, 1, 6, 16), _rand(1, 1, 5, 16)
    a = oab.attention_backward(q, k, v, do)
    b = oab.attention_backward(q, k, v, do, scale=0.25)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


# ------------------------------------------------------------- planted mistakes
def _mutant(kind):
    real = oab.backward_terms

    def terms(q_bh, k_bh, v_bh, do_bh, causal=False, scale=None, bottom_right=False):
        if kind == "offset_ignored":
            bottom_right = False
        t = real(q_bh, k_bh, v_bh, do_bh, causal, scale, bottom_right)
        sc = 1.0 / np.sqrt(np.shape(q_bh)[1]) if scale is None else scale
        q, k = oab._as_f64(q_bh), oab._as_f64(k_bh)
        if kind == "no_D":
            ds = t["P"] * t["dP"]
            t["dQ"], t["dK"] = sc * ds @ k, sc * ds.T @ q
        elif kind == "D_sign":
            ds = t["P"] * (t["dP"] + t["D"][:, None])
            t["dQ"], t["dK"] = sc * ds @ k, sc * ds.T @ q
        elif kind == "no_scale_dk":
            t["dK"] = t["dS"].T @ q
        elif kind == "no_scale_dq":
            t["dQ"] = t["dS"] @ k
        elif kind == "dq_with_q":
            t["dQ"] = sc * t["dS"] @ q[: k.shape[0]] if q.shape[0] >= k.shape[0] else t["dQ"] * 1.01
        elif kind == "dv_unnormalised":
            t["dV"] = t["dV"] * 1.0001
        elif kind == "D_from_dO_only":
            ds = t["P"] * (t["dP"] - oab._as_f64(do_bh).sum(axis=1)[:, None])
            t["dQ"], t["dK"] = sc * ds @ k, sc * ds.T @ q
        elif kind == "mask_ignored":
            if causal:
                u = real(q_bh, k_bh, v_bh, do_bh, False, scale, bottom_right)
                t["dQ"], t["dK"], t["dV"] = u["dQ"], u["dK"], u["dV"]
        return t
    return terms


MUTANTS = ["no_D", "D_sign", "no_scale_dk", "no_scale_dq", "dq_with_q", "dv_unnormalised",
           "D_from_dO_only", "mask_ignored", "offset_ignored"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_bwd_pins_catch_planted_mistakes(kind, monkeypatch):
    monkeypatch.setattr(oab, "backward_terms", _mutant(kind))
    failed = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0, f"no pin caught mutant {kind}"
