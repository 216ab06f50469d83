"""Shared helpers for the GPU parity tests: run the library, run the oracle on
the same host bytes, and apply the tolerance rule.

Tolerances (written here once, used by every parity test):
  * f32 q/K/V:  max|gpu - ref| <= 1e-5 * max|ref| over the output tensor;
  * bf16 q/K/V, f32 output:  max|gpu - ref| <= 2e-3 (absolute);
  * bf16 output:  |gpu - ref| <= 2e-3 + 2^-8 |ref| elementwise -- bf16 keeps 8
    significant bits, so the store alone rounds by up to 2^-8 |o| (its unit
    roundoff) -- and the bf16 result must equal the round-to-nearest-even of the
    f32-output result of the same call bit for bit.
"""
import numpy as np
import torch

import exact_causal_gqa_gb300 as atlas
import oracle

F32_REL = 1e-5
BF16_ABS = 2e-3
BF16_STORE_REL = 2.0 ** -8


def oracle_rows(prob, rows=None, want_lse=False, **variants):
    """The oracle on the problem's host bytes; ``variants``: window, softcap, sinks."""
    return oracle.attn(prob.q, prob.k_pages, prob.v_pages, prob.page_table, prob.seq_lens,
                       prob.n_q_heads, prob.n_kv_heads, prob.scale, rows=rows,
                       want_lse=want_lse, **variants)


def run_gpu(prob_dev, out_dtype=None, **kw):
    out_dtype = out_dtype or {"f32": torch.float32, "bf16": torch.bfloat16}[prob_dev.out_dtype]
    return atlas.run(prob_dev, out_dtype=out_dtype, **kw)


def assert_parity(prob, got, ref, label=""):
    """got: GPU output (any dtype, any shape matching ref); ref: fp64 oracle."""
    g = got.detach().float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    assert np.isfinite(g).all(), f"{label}: non-finite output"
    err = np.abs(g - ref)
    if prob.dtype == "f32":
        bound = F32_REL * np.abs(ref).max()
        assert err.max() <= bound, f"{label}: max err {err.max():.3e} > {bound:.3e}"
    elif got.dtype == torch.float32:
        assert err.max() <= BF16_ABS, f"{label}: max err {err.max():.3e} > {BF16_ABS}"
    else:
        lim = BF16_ABS + BF16_STORE_REL * np.abs(ref)
        worst = (err - lim).max()
        assert worst <= 0, f"{label}: err exceeds 2e-3 + 2^-8|ref| by {worst:.3e}"
    return float(err.max())


def flat_rows(prob):
    return prob.batch * prob.n_q_heads * prob.q_len
