"""Pins for the attention oracle, against facts other than the oracle itself.

The oracle follows "TileLang で GPU カーネル設計を解説" §6 (FlashAttention):
O[b, i, h] = sum_j softmax_j(q_i . k_j / sqrt(dim)) v_j over all keys, or over
j <= i when causal, tensors [batch, seq, heads, dim].  The page checks its
kernel against torch's scaled_dot_product_attention; here that library routine
(in float64, on the CPU) is one pin, and the others are closed forms and
invariants:

  * torch float64 SDPA on random shapes (several batch, seq, heads, dim,
    causal and not, both 16-bit formats);
  * zero queries: uniform weights, so each output row is the mean of the
    value rows it may attend (prefix means when causal);
  * one key: the output is that key's value row;
  * permuting keys and values together (not causal) changes nothing;
  * adding one vector to every key shifts all of a query's scores equally,
    which changes nothing (exact small-integer keys);
  * the |V| magnitude equals the output on |V|, and row subsets equal rows of
    the full result.

Every pin takes the attention function as an argument, so the mutation tests
at the bottom can show that a planted mistake (no 1/sqrt(dim) scale, the
causal mask off by one, softmax over queries instead of keys, the weights not
normalised, heads mixed up) fails at least one pin.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

DTS = {oracle.F16: torch.float16, oracle.BF16: torch.bfloat16}


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def rand_qkv(B, S, H, D, dt, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return [(torch.randn(B, S, H, D, generator=g) * scale).to(DTS[dt]) for _ in range(3)]


def sdpa64(q, k, v, causal):
    t = lambda x: x.double().transpose(1, 2)
    o = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=causal)
    return o.transpose(1, 2).contiguous().numpy()


def run(fn, q, k, v, causal, dt, **kw):
    B, S, H, D = q.shape
    return fn(bits(q), bits(k), bits(v), B, S, H, D, causal, dt, **kw).reshape(B, S, H, D)


def pin_library_sdpa(fn):
    for dt in (oracle.F16, oracle.BF16):
        for (B, S, H, D, seed) in [(1, 1, 1, 8, 1), (2, 7, 3, 16, 2), (1, 33, 2, 64, 3), (2, 130, 1, 64, 4)]:
            q, k, v = rand_qkv(B, S, H, D, dt, seed, scale=1.5)
            for causal in (False, True):
                got = run(fn, q, k, v, causal, dt)
                ref = sdpa64(q, k, v, causal)
                assert np.allclose(got, ref, rtol=1e-12, atol=1e-13), (dt, B, S, H, D, causal)


def pin_zero_queries(fn):
    dt = oracle.F16
    B, S, H, D = 2, 9, 3, 16
    _, k, v = rand_qkv(B, S, H, D, dt, 5)
    q = torch.zeros(B, S, H, D, dtype=torch.float16)
    vv = v.double().numpy()
    full = run(fn, q, k, v, False, dt)
    assert np.allclose(full, np.broadcast_to(vv.mean(axis=1, keepdims=True), vv.shape), rtol=1e-13, atol=1e-14)
    causal = run(fn, q, k, v, True, dt)
    prefix = np.cumsum(vv, axis=1) / np.arange(1, S + 1)[None, :, None, None]
    assert np.allclose(causal, prefix, rtol=1e-13, atol=1e-14)


def pin_single_key(fn):
    for dt in (oracle.F16, oracle.BF16):
        q, k, v = rand_qkv(3, 1, 2, 32, dt, 6, scale=4.0)
        for causal in (False, True):
            assert np.array_equal(run(fn, q, k, v, causal, dt), v.double().numpy())


def pin_key_permutation(fn):
    dt = oracle.F16
    B, S, H, D = 1, 17, 2, 32
    q, k, v = rand_qkv(B, S, H, D, dt, 7)
    perm = torch.randperm(S, generator=torch.Generator().manual_seed(8))
    a = run(fn, q, k, v, False, dt)
    b = run(fn, q, k[:, perm], v[:, perm], False, dt)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-13)


def pin_score_shift(fn):
    # Small-integer keys and shift: K + c is exact in fp16, and every score of
    # query i moves by the same amount q_i . c / sqrt(D).
    dt = oracle.F16
    B, S, H, D = 1, 11, 2, 16
    g = torch.Generator().manual_seed(9)
    q = (torch.randint(-2, 3, (B, S, H, D), generator=g).float() / 4).half()
    k = torch.randint(-3, 4, (B, S, H, D), generator=g).half()
    v = torch.randn(B, S, H, D, generator=g).half()
    c = torch.randint(-5, 6, (D,), generator=g).half()
    for causal in (False, True):
        a = run(fn, q, k, v, causal, dt)
        b = run(fn, q, k + c, v, causal, dt)
        assert np.allclose(a, b, rtol=1e-12, atol=1e-13)


def pin_magnitude_and_rows(fn):
    dt = oracle.BF16
    B, S, H, D = 2, 13, 3, 16
    q, k, v = rand_qkv(B, S, H, D, dt, 10)
    for causal in (False, True):
        mag = run(fn, q, k, v, causal, dt, abs_v=True)
        on_abs = run(fn, q, k, v.abs(), causal, dt)
        assert np.array_equal(mag, on_abs)
        full = run(fn, q, k, v, causal, dt).reshape(-1, D)
        rows = [0, 5, 17, B * S * H - 1]
        sub = fn(bits(q), bits(k), bits(v), B, S, H, D, causal, dt, rows=rows)
        assert np.array_equal(sub, full[rows])


ALL_PINS = [pin_library_sdpa, pin_zero_queries, pin_single_key, pin_key_permutation, pin_score_shift,
            pin_magnitude_and_rows]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_attention_oracle_pin(pin):
    pin(oracle.attention_f64)


def test_workload_shape_runs():
    # The page's workload size (B, S, H, D) = (4, 1024, 8, 64), on sampled rows.
    B, S, H, D = 4, 1024, 8, 64
    q, k, v = rand_qkv(B, S, H, D, oracle.F16, 11)
    rows = [0, 1023 * H + 7, (3 * S + 511) * H + 2]
    for causal in (False, True):
        got = oracle.attention_f64(bits(q), bits(k), bits(v), B, S, H, D, causal, oracle.F16, rows=rows)
        ref = sdpa64(q, k, v, causal).reshape(-1, D)[rows]
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------- mutation tests
# Plain numpy restatements with one planted mistake each (test-only).
def _decode(b, dt):
    return oracle.decode(b, dt)


def _mutant(mistake):
    def fn(Q, K, V, B, S, H, D, causal, dt, rows=None, abs_v=False):
        q = _decode(Q, dt).reshape(B, S, H, D)
        k = _decode(K, dt).reshape(B, S, H, D)
        v = np.abs(_decode(V, dt)).reshape(B, S, H, D) if abs_v else _decode(V, dt).reshape(B, S, H, D)
        scale = 1.0 if mistake == "no_scale" else 1.0 / np.sqrt(D)
        out = np.zeros((B, S, H, D))
        for b in range(B):
            for h in range(H):
                qh, kh = q[b, :, h], k[b, :, h]
                if mistake == "heads_mixed":
                    kh = k[b, :, (h + 1) % H]
                s = scale * qh @ kh.T
                if causal:
                    off = -1 if mistake == "causal_off_by_one" else 0
                    mask = np.tril(np.ones((S, S), dtype=bool), k=off)
                    s = np.where(mask, s, -np.inf)
                axis = 0 if mistake == "softmax_over_queries" else 1
                with np.errstate(invalid="ignore", divide="ignore"):
                    w = np.exp(s - np.max(s, axis=axis, keepdims=True))
                    if mistake != "not_normalised":
                        w = w / np.sum(w, axis=axis, keepdims=True)
                w = np.nan_to_num(w)
                out[b, :, h] = w @ v[b, :, h]
        out = out.reshape(-1, D)
        return out[np.asarray(rows)] if rows is not None else out
    fn.__name__ = "_mut_" + mistake
    return fn


MUTANTS = [_mutant(m) for m in ("no_scale", "causal_off_by_one", "softmax_over_queries", "not_normalised",
                                "heads_mixed")]


def test_unmutated_restatement_passes():
    # The test-only restatement itself (no mistake) passes the pins that a
    # correct attention must pass, so a failing mutant fails for its mistake.
    fn = _mutant("none")
    for pin in (pin_library_sdpa, pin_zero_queries, pin_single_key, pin_key_permutation, pin_score_shift):
        pin(fn)


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m.__name__)
def test_pins_catch_planted_mistake(mutant):
    failed = 0
    for pin in ALL_PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed += 1
    assert failed > 0, f"no pin caught {mutant.__name__}"
