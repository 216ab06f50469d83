"""Direct prefill with more tile pairs than SMs runs persistent CTAs: each walks
several (sequence, kv head, prompt-row) items in a snake order, with every barrier
phase running on across items.  A small ``sm_count`` forces that on small shapes;
the outputs must equal, bit for bit, the one-item-per-CTA grid of the same plan, and
match the fp64 oracle.  Needs a GB300."""
import numpy as np
import pytest
import torch

import exact_causal_gqa_gb300 as atlas
from exact_causal_gqa_gb300 import inputs
from tests.gpu_helpers import assert_parity, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"
DIRECT = atlas.DEBUG_TC_DIRECT

CASES = [
    dict(B=2, Hq=8, Hkv=2, D=128, P=64, S=512, sms=4),
    dict(B=1, Hq=8, Hkv=2, D=64, P=16, S=768, sms=3),
    dict(B=3, Hq=4, Hkv=1, D=128, P=32, S=384, sms=5),
    dict(B=1, Hq=16, Hkv=2, D=128, P=128, S=640, sms=7),
    dict(B=2, Hq=4, Hkv=2, D=128, P=8, S=256, sms=2),
]


def label(c):
    return f"B{c['B']}-H{c['Hq']}x{c['Hkv']}-D{c['D']}-P{c['P']}-S{c['S']}-sms{c['sms']}"


@pytest.mark.parametrize("c", CASES, ids=[label(c) for c in CASES])
def test_persistent_prefill_equals_the_grid_and_the_oracle(c):
    prob = inputs.make("prefill", c["B"], c["Hq"], c["Hkv"], c["D"], c["P"], [c["S"]] * c["B"],
                       seed=40 + c["S"])
    dev = prob.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    grid = run_gpu(dev, out_dtype=torch.float32, debug_flags=DIRECT)
    pers = run_gpu(dev, out_dtype=torch.float32, debug_flags=DIRECT, sm_count=c["sms"],
                   status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(grid, pers)
    assert_parity(prob, pers, oracle_rows(prob), label(c))


@pytest.mark.parametrize("var", [dict(window=200), dict(softcap=10.0), dict(sinks=True)],
                         ids=["window", "softcap", "sinks"])
def test_persistent_prefill_variants(var):
    prob = inputs.make("prefill", 2, 8, 2, 128, 64, [512, 512], seed=51)
    dev = prob.to(DEV)
    var = dict(var)
    ref_kw = dict(var)
    if var.get("sinks"):
        s = (torch.randn(8, generator=torch.Generator().manual_seed(5)) * 2.0).float()
        var["sinks"] = s.to(DEV)
        ref_kw["sinks"] = s
    grid = run_gpu(dev, out_dtype=torch.float32, debug_flags=DIRECT, **var)
    pers = run_gpu(dev, out_dtype=torch.float32, debug_flags=DIRECT, sm_count=3, **var)
    torch.cuda.synchronize()
    assert torch.equal(grid, pers)
    assert_parity(prob, pers, oracle_rows(prob, **ref_kw), str(var))


def test_persistent_prefill_bf16_output_and_lse():
    prob = inputs.make("prefill", 2, 8, 2, 128, 64, [384, 384], seed=52)
    dev = prob.to(DEV)
    rows = 2 * 8 * 384
    la = torch.empty(rows, dtype=torch.float32, device=DEV)
    lb = torch.empty(rows, dtype=torch.float32, device=DEV)
    a = run_gpu(dev, out_dtype=torch.bfloat16, debug_flags=DIRECT, lse=la)
    b = run_gpu(dev, out_dtype=torch.bfloat16, debug_flags=DIRECT, lse=lb, sm_count=2)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(la, lb)
    ref, ref_lse = oracle_rows(prob, want_lse=True)
    assert_parity(prob, b, ref, "bf16 out")
    np.testing.assert_allclose(lb.cpu().numpy(), ref_lse.reshape(-1), rtol=0, atol=1e-4)


def test_persistent_prefill_bad_page_and_seq_len():
    # sequence 0: page 5 (keys 320..383) outside the pool, read by the tiles from row
    # 256 on; sequence 2: seq_len differs from q_len; sequence 1 is unaffected
    prob = inputs.make("prefill", 3, 8, 2, 128, 64, [512] * 3, seed=53)
    clean = run_gpu(prob.to(DEV), out_dtype=torch.float32, debug_flags=DIRECT)
    prob.page_table[0, 5] = -1
    prob.seq_lens[2] = 511
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_gpu(prob.to(DEV), out_dtype=torch.float32, debug_flags=DIRECT, sm_count=4,
                  status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == atlas.DEV_BAD_PAGE | atlas.DEV_BAD_SEQLEN
    assert torch.isnan(out[0, :, 256:]).all() and torch.isnan(out[2]).all()
    assert torch.equal(out[0, :, :256], clean[0, :, :256])
    assert torch.equal(out[1], clean[1])


def draw(i):
    import random
    r = random.Random(7000 + i)
    Hkv = r.choice([1, 2, 4])
    G = r.choice([2, 4, 6, 8])
    return dict(B=r.randint(1, 3), Hq=G * Hkv, Hkv=Hkv, D=r.choice([64, 128]),
                P=r.choice([8, 16, 32, 64, 128]), S=128 * r.randint(1, 6),
                sms=r.randint(1, 6), seed=8000 + i,
                var=r.choice([{}, {}, {"window": r.randint(1, 500)}, {"softcap": 20.0}]))


RANDOM = [draw(i) for i in range(16)]


@pytest.mark.parametrize("c", RANDOM, ids=[label(c) for c in RANDOM])
def test_persistent_prefill_random_shapes(c):
    prob = inputs.make("prefill", c["B"], c["Hq"], c["Hkv"], c["D"], c["P"], [c["S"]] * c["B"],
                       seed=c["seed"])
    dev = prob.to(DEV)
    grid = run_gpu(dev, out_dtype=torch.float32, debug_flags=DIRECT, **c["var"])
    pers = run_gpu(dev, out_dtype=torch.float32, debug_flags=DIRECT, sm_count=c["sms"],
                   **c["var"])
    torch.cuda.synchronize()
    assert torch.equal(grid, pers)
    assert_parity(prob, pers, oracle_rows(prob, **c["var"]), label(c))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_persistent_prefill_output_only_16_byte_aligned(dtype):
    # the epilogue writes 32-byte pieces when the output allows; an output that is
    # only 16-byte aligned takes 16-byte stores with the same values
    prob = inputs.make("prefill", 2, 8, 2, 128, 64, [384, 384], seed=54)
    dev = prob.to(DEV)
    n = prob.q.numel()
    shift = 16 // torch.tensor([], dtype=dtype).element_size()
    buf = torch.empty(n + shift, dtype=dtype, device=DEV)
    out = buf[shift:].view(prob.q.shape)
    assert out.data_ptr() % 32 == 16
    aligned = run_gpu(dev, out_dtype=dtype, debug_flags=DIRECT, sm_count=3)
    run_gpu(dev, out_dtype=dtype, debug_flags=DIRECT, sm_count=3, out=out)
    torch.cuda.synchronize()
    assert torch.equal(aligned, out)


@pytest.mark.parametrize("S", [4096, 4224])
def test_persistent_prefill_full_item_lists(S):
    # 128 tile pairs with one SM allowed: two CTAs of exactly 64 items each (the
    # per-CTA limit, every bit of the item mask in use); 132 pairs: three CTAs
    prob = inputs.make("prefill", 1, 8, 2, 128, 64, [S], seed=55)
    dev = prob.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    grid = run_gpu(dev, out_dtype=torch.float32, debug_flags=DIRECT)
    pers = run_gpu(dev, out_dtype=torch.float32, debug_flags=DIRECT, sm_count=1, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(grid, pers)
    assert_parity(prob, pers, oracle_rows(prob), f"S{S}")


def test_persistent_prefill_every_item_skipped():
    # a bad seq_len makes all 64 items of both CTAs skip: the rows are NaN, the
    # status says why, and the CTAs leave before their setup
    prob = inputs.make("prefill", 1, 8, 2, 128, 64, [4096], seed=56)
    prob.seq_lens[0] = 4095
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_gpu(prob.to(DEV), out_dtype=torch.float32, debug_flags=DIRECT, sm_count=1,
                  status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == atlas.DEV_BAD_SEQLEN
    assert torch.isnan(out).all()
