"""Seeded random shapes on every entry point against the fp64 oracle: kind, dtype,
head_dim, page size, group size, batch, context lengths, query rows, split size and
the score variants are drawn per case, so that the plan's choices (direct output,
cluster merge, split + merge, tensor-core tiles, balanced splits) meet shapes no
hand-written case picked.  Sizes stay where the oracle takes well under a second.
Needs a GB300."""
import random

import numpy as np
import pytest
import torch

from exact_causal_gqa_gb300 import inputs
from tests.gpu_helpers import assert_parity, flat_rows, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"
N_CASES = 96


def draw(i):
    r = random.Random(1000 + i)
    kind = r.choice(["decode", "decode", "suffix", "suffix", "prefill"])
    dtype = r.choice(["bf16", "bf16", "f32"])
    D = r.choice([64, 128])
    P = r.choice([8, 16, 32, 64, 128])
    Hkv = r.choice([1, 2, 4, 8])
    G = r.choice([1, 2, 3, 4, 8])
    B = r.randint(1, 4)
    if kind == "prefill":
        L = r.randint(1, 700)
        lens, q_len = [L] * B, L
    else:
        lens = [r.randint(1, 3000) for _ in range(B)]
        q_len = 1 if kind == "decode" else r.randint(1, min(40, min(lens)))
    kw = {}
    if r.random() < 0.3:
        kw["split_tokens"] = 64 * r.randint(1, 12)
    var = {}
    if r.random() < 0.25:
        var["window"] = r.randint(1, 800)
    if r.random() < 0.2:
        var["softcap"] = r.choice([2.0, 10.0, 30.0])
    sinks = r.random() < 0.2
    return dict(kind=kind, dtype=dtype, D=D, P=P, Hkv=Hkv, G=G, B=B, lens=lens, q_len=q_len,
                kw=kw, var=var, sinks=sinks, seed=2000 + i)


CASES = [draw(i) for i in range(N_CASES)]


def label(c):
    return (f"{c['kind']}-{c['dtype']}-D{c['D']}-P{c['P']}-G{c['G']}x{c['Hkv']}-B{c['B']}"
            f"-q{c['q_len']}-L{max(c['lens'])}")


@pytest.mark.parametrize("c", CASES, ids=[label(c) for c in CASES])
def test_random_shape(c):
    Hq = c["G"] * c["Hkv"]
    prob = inputs.make(c["kind"], c["B"], Hq, c["Hkv"], c["D"], c["P"], c["lens"],
                       q_len=c["q_len"], dtype=c["dtype"], seed=c["seed"])
    var = dict(c["var"])
    call = dict(var)
    if c["sinks"]:
        g = torch.Generator().manual_seed(c["seed"])
        s = (torch.randn(Hq, generator=g) * 2.0).float()
        var["sinks"] = s
        call["sinks"] = s.to(DEV)
    ref, ref_lse = oracle_rows(prob, want_lse=True, **var)
    dev = prob.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    lse = torch.empty(flat_rows(prob), dtype=torch.float32, device=DEV)
    out = run_gpu(dev, out_dtype=torch.float32, lse=lse, status=status, **c["kw"], **call)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_parity(prob, out, ref, label(c))
    tol = 1e-4 if c["dtype"] == "bf16" else 2e-5
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.reshape(-1), rtol=0, atol=tol)
