"""GQA against MHA with duplicated K/V heads on the GPU, and non-finite inputs.

- GQA mapping (kv head = h / G): the same attention with every kv head repeated G
  times (Hkv = Hq) matches it on every kernel path; the two runs take different
  kernels or tilings, so they agree within the tolerance, each with the oracle.
- Non-finite K/V are not scanned (a second read of the cache would cost as much as
  the attention); they propagate: a NaN in a visible key makes the rows that see it
  NaN and leaves every other row as it was.
"""
import numpy as np
import pytest
import torch

from exact_causal_gqa_gb300 import inputs
from tests.gpu_helpers import assert_parity, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu


def to_dev(host):
    return inputs.Problem(**{k: (v.to("cuda") if torch.is_tensor(v) else v)
                             for k, v in vars(host).items()})


def as_mha(host):
    """The same problem with each kv head repeated G times (Hkv = Hq)."""
    G = host.n_q_heads // host.n_kv_heads
    mha = inputs.Problem(**vars(host))
    mha.k_pages = host.k_pages.repeat_interleave(G, dim=1).contiguous()
    mha.v_pages = host.v_pages.repeat_interleave(G, dim=1).contiguous()
    mha.n_kv_heads = host.n_q_heads
    return mha


@pytest.mark.parametrize("kind,dtype,Hq,Hkv,D,P,q_len,lens", [
    ("decode", "bf16", 16, 4, 128, 16, 1, (900, 2500)),      # split kernel; MHA: G = 1
    ("suffix", "bf16", 32, 4, 128, 32, 16, (1200, 3000)),    # tensor cores vs split kernel
    ("prefill", "bf16", 8, 2, 128, 64, 384, (384, 384)),     # tensor cores both, G 4 vs 1
    ("decode", "f32", 8, 2, 64, 16, 1, (700, 1800)),         # fp32 ring kernel
])
def test_gqa_equals_mha_with_duplicated_heads(kind, dtype, Hq, Hkv, D, P, q_len, lens):
    host = inputs.make(kind, len(lens), Hq, Hkv, D, P, list(lens), q_len=q_len, dtype=dtype,
                       out_dtype=dtype, seed=Hq + q_len, device="cpu")
    mha = as_mha(host)
    ref = oracle_rows(host)
    np.testing.assert_array_equal(ref, oracle_rows(mha))  # the oracle: identical
    out_gqa = run_gpu(to_dev(host), out_dtype=torch.float32)
    out_mha = run_gpu(to_dev(mha), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_parity(host, out_gqa, ref, "GQA")
    assert_parity(host, out_mha, ref, "MHA with duplicated heads")


@pytest.mark.parametrize("kind,dtype,Hq,Hkv,D,P,q_len", [
    ("suffix", "bf16", 32, 4, 128, 32, 16),   # tensor cores (G * q_len = 128)
    ("suffix", "bf16", 8, 4, 128, 16, 4),     # split kernel (G * q_len = 8)
    ("suffix", "f32", 16, 2, 128, 16, 16),    # fp32 tensor-core kernel (3 x tf32)
    ("suffix", "f32", 4, 2, 64, 16, 2),       # fp32 ring kernel
])
def test_nan_key_reaches_exactly_the_rows_that_see_it(kind, dtype, Hq, Hkv, D, P, q_len):
    L = 1000
    host = inputs.make(kind, 1, Hq, Hkv, D, P, [L], q_len=q_len, dtype=dtype, out_dtype=dtype,
                       seed=3, device="cpu")
    t = L - q_len + q_len // 2          # rows i >= q_len // 2 see key t (row i sees <= L-q_len+i)
    phys = int(host.page_table[0, t // P])
    host.k_pages[phys, 0, t % P, 5] = float("nan")   # kv head 0: q heads 0 .. G-1
    out = run_gpu(to_dev(host), out_dtype=torch.float32).cpu().numpy()[0]
    torch.cuda.synchronize()
    G = Hq // Hkv
    sees = np.zeros((Hq, q_len), dtype=bool)
    sees[:G, q_len // 2:] = True
    rows_nan = np.isnan(out).any(-1)
    np.testing.assert_array_equal(rows_nan, sees)
    # every other row is the oracle's (the oracle rows are computed on the same bytes)
    ref = oracle_rows(host)[0]
    ok = ~sees
    err = np.abs(out[ok] - ref[ok]).max()
    assert err <= (1e-5 * np.abs(ref[ok]).max() if dtype == "f32" else 2e-3)
