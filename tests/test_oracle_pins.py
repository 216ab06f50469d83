"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test states an expected value that comes from mathematics or from what the
pages fix, never from re-running the oracle's own formula:
  * brute force at 50 significant digits on tiny inputs (materialised masked
    score matrix, softmax without max subtraction);
  * closed forms: one visible key, constant V, q = 0, a dominant key, the
    two-key logistic weight, identity-V probabilities;
  * the pages' invariants: folded == full-KV for any page size and page
    permutation (CFR-Atlas README, "Core contract"); suffix rows == decode at the
    shorter context (CPUAttn README, "Parallel example" / "Operator model");
    GQA == MHA with duplicated K/V heads; split + structured merge == unsplit
    (CPUAttn README, "Operator model");
  * a library routine on tiny shapes: torch's fp64 scaled_dot_product_attention
    with an explicit causal-offset mask;
  * a hand-worked example stored under tests/golden/;
  * for the score/mask variants (window, softcap, sinks): the same brute force
    with the variant applied, their limits (a window covering every key, a huge
    cap, a sink at -1e4), closed forms (window 1; one key with a sink; q = 0 with
    a sink), the sink as one more merge state, and torch SDPA with a band mask.
"""
import json
import math
import os

import mpmath
import numpy as np
import pytest
import torch

import oracle
from tests.paging import page_kv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_problem(seed, B, Hq, Hkv, D, lens, q_len, P, scale=None, spread=1.0):
    rng = np.random.default_rng(seed)
    Lmax = max(lens)
    q = (rng.standard_normal((B, Hq, q_len, D)) * spread).astype(np.float32)
    k = (rng.standard_normal((B, Hkv, Lmax, D)) * spread).astype(np.float32)
    v = rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float32)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    return q, k, v, scale


def run_oracle(fn, q, k, v, lens, P, Hq, Hkv, scale, seed=3, **kw):
    kp, vp, table = page_kv(k, v, lens, P, seed=seed)
    return fn(q, kp, vp, table, np.asarray(lens, np.int32), Hq, Hkv, scale, **kw)


def brute_force(q, k, v, lens, Hq, Hkv, scale, digits=50, window=0, softcap=0.0, sinks=None):
    """Materialise s = scale * q k^T with the causal-suffix (and window) mask, apply the
    softcap, softmax without shift with exp(sink) in the denominator."""
    mpmath.mp.dps = digits
    B, _, q_len, D = q.shape
    G = Hq // Hkv
    out = np.zeros(q.shape, dtype=np.float64)
    for b in range(B):
        L = lens[b]
        for h in range(Hq):
            g = h // G
            for i in range(q_len):
                pos = L - q_len + i
                w = {}
                for t in range(L):
                    if t > pos or (window and pos - t >= window):
                        continue
                    s = mpmath.mpf(0)
                    for d in range(D):
                        s += mpmath.mpf(float(q[b, h, i, d])) * mpmath.mpf(float(k[b, g, t, d]))
                    s = mpmath.mpf(scale) * s
                    if softcap:
                        s = mpmath.mpf(softcap) * mpmath.tanh(s / mpmath.mpf(softcap))
                    w[t] = mpmath.exp(s)
                z = mpmath.fsum(w.values())
                if sinks is not None:
                    z += mpmath.exp(mpmath.mpf(float(sinks[h])))
                for d in range(D):
                    num = mpmath.fsum(wt * mpmath.mpf(float(v[b, g, t, d])) for t, wt in w.items())
                    out[b, h, i, d] = float(num / z)
    return out


@pytest.mark.parametrize("case", [
    dict(B=1, Hq=2, Hkv=1, D=4, lens=[7], q_len=1, P=2),
    dict(B=2, Hq=4, Hkv=2, D=3, lens=[9, 5], q_len=3, P=4),
    dict(B=1, Hq=3, Hkv=3, D=5, lens=[6], q_len=6, P=1),
    dict(B=2, Hq=2, Hkv=1, D=2, lens=[11, 4], q_len=4, P=3),
])
def test_brute_force_50_digits(case):
    q, k, v, scale = rand_problem(11, case["B"], case["Hq"], case["Hkv"], case["D"],
                                  case["lens"], case["q_len"], case["P"])
    ref = brute_force(q, k, v, case["lens"], case["Hq"], case["Hkv"], scale)
    for fn in (oracle.attn, oracle.folded):
        got = run_oracle(fn, q, k, v, case["lens"], case["P"], case["Hq"], case["Hkv"], scale)
        np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)


def test_single_visible_key_returns_its_value_row():
    # Decode at context 1 and prefill row 0 both see exactly one key.
    q, k, v, scale = rand_problem(5, 2, 4, 2, 16, [1, 1], 1, 16)
    out = run_oracle(oracle.attn, q, k, v, [1, 1], 16, 4, 2, scale)
    for b in range(2):
        for h in range(4):
            assert np.array_equal(out[b, h, 0], v[b, h // 2, 0].astype(np.float64))
    q, k, v, scale = rand_problem(6, 1, 2, 1, 8, [33], 33, 8)
    out = run_oracle(oracle.attn, q, k, v, [33], 8, 2, 1, scale)
    assert np.array_equal(out[0, 1, 0], v[0, 0, 0].astype(np.float64))


def test_constant_values_return_the_constant():
    q, k, _, scale = rand_problem(7, 2, 4, 2, 8, [40, 17], 5, 16, spread=2.0)
    const = np.float32([0.5, -1.25, 3.0, 0.0, 7.5, -2.0, 1e-3, 4.0])
    v = np.broadcast_to(const, k.shape).copy()
    for fn in (oracle.attn, oracle.folded):
        out = run_oracle(fn, q, k, v, [40, 17], 16, 4, 2, scale)
        ref = np.broadcast_to(const.astype(np.float64), out.shape)
        np.testing.assert_allclose(out, ref, rtol=4 * np.finfo(np.float64).eps, atol=1e-18)


def test_zero_query_returns_mean_of_visible_values():
    B, Hq, Hkv, D, lens, q_len = 2, 2, 1, 6, [12, 9], 3
    _, k, v, scale = rand_problem(8, B, Hq, Hkv, D, lens, q_len, 4)
    q = np.zeros((B, Hq, q_len, D), np.float32)
    out = run_oracle(oracle.attn, q, k, v, lens, 4, Hq, Hkv, scale)
    for b in range(B):
        for i in range(q_len):
            n = lens[b] - q_len + i + 1
            mean = v[b, 0, :n].astype(np.float64).mean(axis=0)
            for h in range(Hq):
                np.testing.assert_allclose(out[b, h, i], mean, rtol=1e-14, atol=1e-15)


def test_dominant_key_returns_its_value_row():
    # One key aligned with q at a score ~1000 above the others: every other
    # weight is exp(-1000) == 0 in fp64, so the output is that key's V row.
    B, Hq, Hkv, D, L = 1, 1, 1, 4, 20
    q = np.zeros((B, Hq, 1, D), np.float32)
    q[0, 0, 0, 0] = 1.0
    rng = np.random.default_rng(9)
    k = rng.standard_normal((B, Hkv, L, D)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, L, D)).astype(np.float32)
    k[0, 0, 13, 0] = 1000.0
    out = run_oracle(oracle.attn, q, k, v, [L], 4, 1, 1, 1.0)
    assert np.array_equal(out[0, 0, 0], v[0, 0, 13].astype(np.float64))


def test_identity_values_expose_probabilities():
    # With V rows e_t the output is the probability row: non-negative, sums to 1,
    # and for two keys equals the logistic function of the score difference.
    L = 6
    rng = np.random.default_rng(10)
    q = rng.standard_normal((1, 1, L, L)).astype(np.float32)
    k = rng.standard_normal((1, 1, L, L)).astype(np.float32)
    v = np.eye(L, dtype=np.float32)[None, None]
    scale = 0.7
    out = run_oracle(oracle.attn, q, k, v, [L], 2, 1, 1, scale)
    probs = out[0, 0]
    assert (probs >= 0).all()
    np.testing.assert_allclose(probs.sum(axis=1), 1.0, rtol=0, atol=2e-15)
    assert np.all(probs[np.triu_indices(L, 1)] == 0.0)  # causal: row i ignores keys > i
    s0 = scale * float(np.dot(q[0, 0, 1].astype(np.float64), k[0, 0, 0].astype(np.float64)))
    s1 = scale * float(np.dot(q[0, 0, 1].astype(np.float64), k[0, 0, 1].astype(np.float64)))
    np.testing.assert_allclose(probs[1, 0], 1.0 / (1.0 + math.exp(s1 - s0)), rtol=1e-14)


@pytest.mark.parametrize("P", [1, 2, 16, 64, 77])
def test_fold_equals_full_for_any_page_size_and_permutation(P):
    lens = [77, 40, 1]
    q, k, v, scale = rand_problem(12, 3, 4, 2, 16, lens, 1, P, spread=1.5)
    full = run_oracle(oracle.attn, q, k, v, lens, P, 4, 2, scale, seed=100)
    for perm_seed in (1, 2, 3):
        for fn in (oracle.attn, oracle.folded):
            got = run_oracle(fn, q, k, v, lens, P, 4, 2, scale, seed=perm_seed)
            np.testing.assert_allclose(got, full, rtol=1e-13, atol=1e-14)


def test_gqa_equals_mha_with_duplicated_heads():
    B, Hq, Hkv, D, lens, q_len = 2, 8, 2, 8, [30, 21], 4
    q, k, v, scale = rand_problem(13, B, Hq, Hkv, D, lens, q_len, 8)
    gqa = run_oracle(oracle.attn, q, k, v, lens, 8, Hq, Hkv, scale)
    k_mha = np.repeat(k, Hq // Hkv, axis=1)
    v_mha = np.repeat(v, Hq // Hkv, axis=1)
    mha = run_oracle(oracle.attn, q, k_mha, v_mha, lens, 8, Hq, Hq, scale)
    np.testing.assert_allclose(gqa, mha, rtol=0, atol=0)


def test_suffix_rows_equal_decode_at_shorter_context():
    B, Hq, Hkv, D, lens, SQ = 2, 4, 2, 8, [25, 16], 16
    q, k, v, scale = rand_problem(14, B, Hq, Hkv, D, lens, SQ, 4)
    suffix = run_oracle(oracle.attn, q, k, v, lens, 4, Hq, Hkv, scale)
    for b in range(B):
        for i in range(SQ):
            n = lens[b] - SQ + i + 1
            dec = run_oracle(oracle.attn, q[b:b + 1, :, i:i + 1], k[b:b + 1, :, :n],
                             v[b:b + 1, :, :n], [n], 4, Hq, Hkv, scale)
            np.testing.assert_allclose(suffix[b, :, i], dec[0, :, 0], rtol=1e-14, atol=1e-15)


def test_prefill_equals_suffix_with_full_query_length():
    L = 19
    q, k, v, scale = rand_problem(15, 1, 2, 1, 8, [L], L, 4)
    pre = run_oracle(oracle.attn, q, k, v, [L], 4, 2, 1, scale)
    for i in (0, 5, L - 1):
        dec = run_oracle(oracle.attn, q[:, :, i:i + 1], k[:, :, :i + 1], v[:, :, :i + 1],
                         [i + 1], 4, 2, 1, scale)
        np.testing.assert_allclose(pre[0, :, i], dec[0, :, 0], rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("cuts", [[0, 300], [0, 1, 300], [0, 64, 128, 200, 300],
                                  [0, 0, 150, 150, 300], [0, 299, 300]])
def test_split_and_merge_equals_unsplit(cuts):
    L = 300
    q, k, v, scale = rand_problem(16, 1, 2, 1, 16, [L], 1, 16, spread=1.7)
    kp, vp, table = page_kv(k, v, [L], 16, seed=4)
    lens = np.asarray([L], np.int32)
    full, full_lse = oracle.attn(q, kp, vp, table, lens, 2, 1, scale, want_lse=True)
    for row in range(2):
        parts = [oracle.state(q, kp, vp, table, lens, 2, 1, scale, row, a, b)
                 for a, b in zip(cuts[:-1], cuts[1:])]
        o, lse = oracle.merge([p[0] for p in parts], [p[1] for p in parts],
                              np.stack([p[2] for p in parts]))
        np.testing.assert_allclose(o, full.reshape(2, -1)[row], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse, full_lse.reshape(-1)[row], rtol=1e-14)


def test_lse_matches_brute_force_log_partition():
    mpmath.mp.dps = 50
    q, k, v, scale = rand_problem(17, 1, 1, 1, 4, [9], 1, 2)
    _, lse = run_oracle(oracle.attn, q, k, v, [9], 2, 1, 1, scale, want_lse=True)
    z = mpmath.fsum(mpmath.exp(mpmath.mpf(scale) * mpmath.fsum(
        mpmath.mpf(float(q[0, 0, 0, d])) * mpmath.mpf(float(k[0, 0, t, d])) for d in range(4)))
        for t in range(9))
    np.testing.assert_allclose(lse.reshape(-1)[0], float(mpmath.log(z)), rtol=1e-14)


@pytest.mark.parametrize("case", [
    # the CPUAttn README "Parallel example" shape: q (1,8,16,64), k/v (1,2,256,64),
    # scale 0.125, causal, kv_cache=True (queries are the suffix of K/V)
    dict(B=1, Hq=8, Hkv=2, D=64, lens=[256], q_len=16, P=32, scale=0.125),
    dict(B=3, Hq=6, Hkv=3, D=32, lens=[50, 9, 33], q_len=9, P=8, scale=None),
])
def test_library_pin_torch_sdpa_fp64(case):
    B, Hq, Hkv, D, lens, q_len = (case[x] for x in ("B", "Hq", "Hkv", "D", "lens", "q_len"))
    q, k, v, scale = rand_problem(18, B, Hq, Hkv, D, lens, q_len, case["P"], scale=case["scale"])
    got = run_oracle(oracle.attn, q, k, v, lens, case["P"], Hq, Hkv, scale)
    G = Hq // Hkv
    for b in range(B):
        L = lens[b]
        qt = torch.from_numpy(q[b:b + 1]).double()
        kt = torch.from_numpy(k[b:b + 1, :, :L]).double().repeat_interleave(G, dim=1)
        vt = torch.from_numpy(v[b:b + 1, :, :L]).double().repeat_interleave(G, dim=1)
        pos = torch.arange(q_len)[:, None] + (L - q_len)
        mask = torch.arange(L)[None, :] <= pos
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                               scale=scale)
        np.testing.assert_allclose(got[b], ref[0].numpy(), rtol=1e-12, atol=1e-13)


def test_golden_hand_worked_example():
    with open(os.path.join(GOLDEN, "hand_worked_decode.json")) as f:
        case = json.load(f)
    q = np.asarray(case["q"], np.float32)[None, None, None]
    k = np.asarray(case["k"], np.float32)[None, None]
    v = np.asarray(case["v"], np.float32)[None, None]
    L = k.shape[2]
    for P in (1, 2, 3):
        out = run_oracle(oracle.attn, q, k, v, [L], P, 1, 1, case["scale"])
        np.testing.assert_allclose(out[0, 0, 0], case["expected"], rtol=case["rtol"])


def test_invalid_inputs_are_rejected():
    q, k, v, scale = rand_problem(19, 1, 3, 2, 4, [8], 1, 4)
    kp, vp, table = page_kv(k, v, [8], 4)
    with pytest.raises(oracle.OracleError):  # Hq not a multiple of Hkv
        oracle.attn(q, kp, vp, table, np.asarray([8], np.int32), 3, 2, scale)
    q, k, v, scale = rand_problem(19, 1, 2, 1, 4, [8], 2, 4)
    kp, vp, table = page_kv(k, v, [8], 4)
    bad = table.copy()
    bad[0, 1] = kp.shape[0] + 5
    with pytest.raises(oracle.OracleError):  # page id out of range
        oracle.attn(q, kp, vp, bad, np.asarray([8], np.int32), 2, 1, scale)
    with pytest.raises(oracle.OracleError):  # context beyond the page table
        oracle.attn(q, kp, vp, table, np.asarray([9], np.int32), 2, 1, scale)
    with pytest.raises(oracle.OracleError):  # fewer keys than query rows
        oracle.attn(q, kp, vp, table, np.asarray([1], np.int32), 2, 1, scale)


# ---------------------------------------------------------------- score / mask variants
# (ferrox-core crate index: causal_gqa_attention_windowed, _softcap, _sinks)

@pytest.mark.parametrize("variant", [
    dict(window=3), dict(softcap=2.5), dict(sinks=[0.7, -1.2, 3.0, 0.0]),
    dict(window=5, softcap=1.5, sinks=[-0.3, 2.0, 0.1, -4.0]),
])
def test_variants_brute_force_50_digits(variant):
    B, Hq, Hkv, D, lens, q_len, P = 2, 4, 2, 3, [9, 6], 3, 2
    q, k, v, scale = rand_problem(21, B, Hq, Hkv, D, lens, q_len, P, spread=1.8)
    kw = dict(variant)
    if "sinks" in kw:
        kw["sinks"] = np.asarray(kw["sinks"], np.float32)
    ref = brute_force(q, k, v, lens, Hq, Hkv, scale, **kw)
    for fn in (oracle.attn, oracle.folded):
        got = run_oracle(fn, q, k, v, lens, P, Hq, Hkv, scale, **kw)
        np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)


def test_window_limits():
    lens, q_len = [23, 11], 5
    q, k, v, scale = rand_problem(22, 2, 2, 1, 8, lens, q_len, 4)
    plain = run_oracle(oracle.attn, q, k, v, lens, 4, 2, 1, scale)
    wide = run_oracle(oracle.attn, q, k, v, lens, 4, 2, 1, scale, window=23)
    np.testing.assert_array_equal(plain, wide)  # a window covering every key changes nothing
    one = run_oracle(oracle.attn, q, k, v, lens, 4, 2, 1, scale, window=1)
    for b, L in enumerate(lens):           # window 1: only the row's own position
        for i in range(q_len):
            pos = L - q_len + i
            for h in range(2):
                assert np.array_equal(one[b, h, i], v[b, 0, pos].astype(np.float64))


def test_softcap_limit_and_sink_limits():
    lens = [30]
    q, k, v, scale = rand_problem(23, 1, 2, 1, 8, lens, 4, 8, spread=2.0)
    plain = run_oracle(oracle.attn, q, k, v, lens, 8, 2, 1, scale)
    huge_cap = run_oracle(oracle.attn, q, k, v, lens, 8, 2, 1, scale, softcap=1e7)
    np.testing.assert_allclose(huge_cap, plain, rtol=1e-9, atol=1e-12)
    dead_sink = run_oracle(oracle.attn, q, k, v, lens, 8, 2, 1, scale,
                           sinks=np.float32([-1e4, -1e4]))
    np.testing.assert_array_equal(dead_sink, plain)  # exp(-1e4) is 0 in fp64


def test_sink_closed_forms():
    # one visible key with score s and a sink sigma: o = v / (1 + exp(sigma - s))
    q = np.float32([[[[1.0, 0.0]]]])
    k = np.float32([[[[0.75, 3.0]]]])
    v = np.float32([[[[2.0, -6.0]]]])
    out = run_oracle(oracle.attn, q, k, v, [1], 1, 1, 1, 1.0, sinks=np.float32([1.25]))
    np.testing.assert_allclose(out[0, 0, 0],
                               v[0, 0, 0].astype(np.float64) / (1.0 + math.exp(1.25 - 0.75)),
                               rtol=1e-15)
    # q = 0: n equal weights and the sink: o = mean(v) * n / (n + exp(sigma))
    L = 7
    _, k, v, scale = rand_problem(24, 1, 1, 1, 5, [L], 1, 4)
    q = np.zeros((1, 1, 1, 5), np.float32)
    out = run_oracle(oracle.attn, q, k, v, [L], 4, 1, 1, scale, sinks=np.float32([0.5]))
    expect = v[0, 0, :L].astype(np.float64).mean(0) * L / (L + math.exp(0.5))
    np.testing.assert_allclose(out[0, 0, 0], expect, rtol=1e-14)


def test_sink_is_one_more_merge_state_and_window_splits():
    L, W = 60, 37
    q, k, v, scale = rand_problem(25, 1, 2, 1, 16, [L], 1, 8, spread=1.3)
    kp, vp, table = page_kv(k, v, [L], 8, seed=5)
    lens = np.asarray([L], np.int32)
    sinks = np.float32([0.9, -0.4])
    full, full_lse = oracle.attn(q, kp, vp, table, lens, 2, 1, scale, want_lse=True,
                                 window=W, softcap=3.0, sinks=sinks)
    for row in range(2):
        parts = [oracle.state(q, kp, vp, table, lens, 2, 1, scale, row, a, b_,
                              window=W, softcap=3.0)
                 for a, b_ in ((0, 20), (20, 41), (41, 60))]
        ms = [p_[0] for p_ in parts] + [float(sinks[row])]
        ls = [p_[1] for p_ in parts] + [1.0]
        accs = np.stack([p_[2] for p_ in parts] + [np.zeros(16)])
        o, lse = oracle.merge(ms, ls, accs)
        np.testing.assert_allclose(o, full.reshape(2, -1)[row], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse, full_lse.reshape(-1)[row], rtol=1e-14)


def test_window_library_pin_torch_sdpa():
    B, Hq, Hkv, D, lens, q_len, W = 2, 4, 2, 16, [40, 25], 6, 9
    q, k, v, scale = rand_problem(26, B, Hq, Hkv, D, lens, q_len, 8)
    got = run_oracle(oracle.attn, q, k, v, lens, 8, Hq, Hkv, scale, window=W)
    for b in range(B):
        L = lens[b]
        qt = torch.from_numpy(q[b:b + 1]).double()
        kt = torch.from_numpy(k[b:b + 1, :, :L]).double().repeat_interleave(2, dim=1)
        vt = torch.from_numpy(v[b:b + 1, :, :L]).double().repeat_interleave(2, dim=1)
        pos = torch.arange(q_len)[:, None] + (L - q_len)
        t = torch.arange(L)[None, :]
        mask = (t <= pos) & (pos - t < W)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                               scale=scale)
        np.testing.assert_allclose(got[b], ref[0].numpy(), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- ragged queries, append

def test_ragged_rows_equal_each_sequence_alone_and_brute_force():
    B, Hq, Hkv, D, q_len = 3, 4, 2, 6, 7
    lens, q_lens = [20, 9, 7], [7, 3, 1]
    q, k, v, scale = rand_problem(27, B, Hq, Hkv, D, lens, q_len, 4, spread=1.4)
    got = run_oracle(oracle.attn, q, k, v, lens, 4, Hq, Hkv, scale, q_lens=q_lens)
    for b in range(B):
        qn = q_lens[b]
        alone = run_oracle(oracle.attn, q[b:b + 1, :, :qn], k[b:b + 1], v[b:b + 1], [lens[b]],
                           4, Hq, Hkv, scale)
        np.testing.assert_allclose(got[b, :, :qn], alone[0], rtol=1e-14, atol=1e-15)
        ref = brute_force(q[b:b + 1, :, :qn], k[b:b + 1], v[b:b + 1], [lens[b]], Hq, Hkv, scale)
        np.testing.assert_allclose(got[b, :, :qn], ref[0], rtol=1e-13, atol=1e-14)
        assert np.all(got[b, :, qn:] == 0.0)  # padding rows are not queries


def test_append_then_gather_is_concatenation():
    from tests.paging import gather_kv
    rng = np.random.default_rng(28)
    B, Hkv, D, P = 3, 2, 8, 4
    old, new = [5, 8, 0], [3, 1, 6]
    max_new = max(new)
    total = [o + n for o, n in zip(old, new)]
    k_log = rng.standard_normal((B, Hkv, max(total), D)).astype(np.float32)
    v_log = rng.standard_normal((B, Hkv, max(total), D)).astype(np.float32)
    # pages sized for the final lengths, filled with the old tokens only
    kp, vp, table = page_kv(k_log, v_log, total, P, seed=6)
    for b in range(B):
        for t in range(old[b], total[b]):
            phys = table[b, t // P]
            kp[phys, :, t % P] = np.nan
            vp[phys, :, t % P] = np.nan
    k_new = np.zeros((B, Hkv, max_new, D), np.float32)
    v_new = np.zeros((B, Hkv, max_new, D), np.float32)
    for b in range(B):
        k_new[b, :, :new[b]] = k_log[b, :, old[b]:total[b]]
        v_new[b, :, :new[b]] = v_log[b, :, old[b]:total[b]]
    kp2, vp2 = oracle.kv_append(k_new, v_new, kp, vp, table, np.int32(old), np.int32(new))
    kg, vg = gather_kv(kp2, vp2, table, total)
    for b in range(B):
        np.testing.assert_array_equal(kg[b, :, :total[b]], k_log[b, :, :total[b]])
        np.testing.assert_array_equal(vg[b, :, :total[b]], v_log[b, :, :total[b]])
    bad = table.copy()
    bad[0, 1] = kp.shape[0]
    with pytest.raises(oracle.OracleError):
        oracle.kv_append(k_new, v_new, kp, vp, bad, np.int32(old), np.int32(new))
