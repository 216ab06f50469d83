"""Parity of the split-KV decode path (and its LSE merge) with the fp64 oracle,
through the C ABI, on the same seeded host bytes.  Needs a GB300."""
import numpy as np
import pytest
import torch

import exact_causal_gqa_gb300 as atlas
from exact_causal_gqa_gb300 import inputs
from tests.gpu_helpers import assert_parity, flat_rows, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu

DEV = "cuda"


def small(kind="decode", B=3, Hq=8, Hkv=2, D=128, P=16, lens=(100, 257, 16), q_len=None,
          dtype="bf16", seed=0, **kw):
    return inputs.make(kind, B, Hq, Hkv, D, P, list(lens), q_len=q_len, dtype=dtype, seed=seed,
                       **kw)


CASES = [
    # (D, P, Hq, Hkv, lens) -- page boundaries and +-1, several splits and tails
    (128, 16, 8, 2, (1, 15, 16, 17, 64, 65, 1000)),
    (128, 8, 4, 4, (7, 8, 9, 300)),
    (128, 32, 32, 4, (31, 32, 33, 511)),
    (128, 64, 16, 2, (63, 64, 65, 4097)),
    (128, 128, 8, 8, (127, 128, 129, 2000)),
    (64, 16, 4, 1, (5, 16, 700)),
    (64, 64, 16, 1, (64, 65, 1234)),
    (128, 16, 16, 1, (333, 48)),          # G = 16: two column tiles of 8 in one CTA
]


@pytest.mark.parametrize("D,P,Hq,Hkv,lens", CASES)
@pytest.mark.parametrize("split", [0, 64, 192])
def test_decode_bf16_parity(D, P, Hq, Hkv, lens, split):
    prob = small(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, P=P, lens=lens, seed=D + P + Hq)
    ref, ref_lse = oracle_rows(prob, want_lse=True)
    dev = prob.to(DEV)
    lse = torch.empty(flat_rows(prob), dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out32 = run_gpu(dev, out_dtype=torch.float32, lse=lse, status=status, split_tokens=split)
    out16 = run_gpu(dev, out_dtype=torch.bfloat16, split_tokens=split)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_parity(prob, out32, ref, "f32 out")
    assert_parity(prob, out16, ref, "bf16 out")
    # the bf16 store is the RNE of the f32 result of the same split plan
    assert torch.equal(out16, out32.to(torch.bfloat16))
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.reshape(-1), rtol=0, atol=1e-4)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("split", [0, 64])
@pytest.mark.parametrize("lens", [(1, 17, 512, 777), (1, 17, 300, 512)])
def test_decode_f32_parity(D, split, lens):
    # contexts up to 512 keys with the automatic plan: at most 8 splits, merged inside
    # a thread-block cluster; longer ones, or split 64, go through the merge kernel
    prob = small(B=4, Hq=8, Hkv=4, D=D, P=16, lens=lens, dtype="f32", seed=D)
    ref, ref_lse = oracle_rows(prob, want_lse=True)
    lse = torch.empty(flat_rows(prob), dtype=torch.float32, device=DEV)
    out = run_gpu(prob.to(DEV), lse=lse, split_tokens=split)
    assert_parity(prob, out, ref, "f32")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.reshape(-1), rtol=0, atol=1e-5)


def test_config1_full_parity():
    prob = inputs.make_config(1)
    ref = oracle_rows(prob)
    out = run_gpu(prob.to(DEV))
    assert_parity(prob, out, ref, "config 1")


@pytest.mark.parametrize("index", [2, 3])
def test_full_size_decode_every_row(index):
    """The GQA decode (256 (sequence, kv head) groups) and the long-context decode
    (4 x 131072 keys, 1 % outlier K rows) at full size, in the launch configuration
    bench.py times: every output row against the oracle, bf16 and f32 outputs."""
    prob = inputs.make_config(index)
    dev = prob.to(DEV)
    out = run_gpu(dev)
    out32 = run_gpu(dev, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = oracle_rows(prob)
    assert_parity(prob, out, ref, "bf16 out")
    assert_parity(prob, out32, ref, "f32 out")
    assert torch.equal(out, out32.to(torch.bfloat16))


def outlier_dominated_rows(prob, min_weight=0.5):
    """Rows of a decode problem whose largest softmax weight belongs to an outlier K
    row (scaled x8 by the input recipe; its norm is ~8x the others'), with that weight
    above min_weight.  Scores come from the host bytes in numpy (selection only; the
    expected outputs are the oracle's)."""
    q = prob.q.float().numpy()
    k = prob.k_pages.float().numpy()
    table = prob.page_table.numpy()
    lens = prob.seq_lens.numpy()
    G = prob.n_q_heads // prob.n_kv_heads
    P, D = prob.page_tokens, prob.head_dim
    picked, weights = [], []
    for b in range(prob.batch):
        L = int(lens[b])
        pages = table[b, :(L + P - 1) // P]
        for g in range(prob.n_kv_heads):
            keys = k[pages, g].reshape(-1, D)[:L]
            norms = np.linalg.norm(keys, axis=1)
            outlier = norms > 4.0 * np.median(norms)
            qg = q[b, g * G:(g + 1) * G, 0, :]
            s = (qg @ keys.T).astype(np.float64) * prob.scale
            top = s.argmax(axis=1)
            w = 1.0 / np.exp(s - s.max(axis=1, keepdims=True)).sum(axis=1)
            for j in range(G):
                weights.append(w[j])
                if outlier[top[j]] and w[j] > min_weight:
                    picked.append((b * prob.n_q_heads + g * G + j))
    return np.asarray(picked, dtype=np.int64), np.asarray(weights)


def test_config3_outlier_dominated_rows():
    """Long-context decode with 1 % of K rows scaled x8: the rows whose softmax is
    dominated by one outlier key (the softmax-max stress of that workload) match the
    oracle at the bf16 bound, with nothing non-finite anywhere."""
    prob = inputs.make_config(3)
    rows, weights = outlier_dominated_rows(prob)
    # the recipe makes most rows outlier-dominated; the check below needs many
    assert rows.size >= 0.5 * flat_rows(prob), (rows.size, flat_rows(prob))
    dev = prob.to(DEV)
    out32 = run_gpu(dev, out_dtype=torch.float32)
    out16 = run_gpu(dev)
    torch.cuda.synchronize()
    assert torch.isfinite(out32).all() and torch.isfinite(out16.float()).all()
    ref = oracle_rows(prob, rows=rows)
    idx = torch.from_numpy(rows).to(DEV)
    D = prob.head_dim
    assert_parity(prob, out32.reshape(-1, D)[idx], ref, "f32 out, outlier rows")
    assert_parity(prob, out16.reshape(-1, D)[idx], ref, "bf16 out, outlier rows")


def test_page_permutation_is_bitwise_invariant():
    prob = small(lens=(300, 45, 129), P=16, extra_pages=5)
    dev = prob.to(DEV)
    base = run_gpu(dev, out_dtype=torch.float32)
    # move every page to a new slot and rewrite the table accordingly
    perm = torch.randperm(prob.num_pages, generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(prob.num_pages)
    k2 = torch.empty_like(prob.k_pages)
    v2 = torch.empty_like(prob.v_pages)
    k2[inv] = prob.k_pages
    v2[inv] = prob.v_pages
    table2 = inv[prob.page_table.long()].to(torch.int32)
    prob2 = inputs.Problem(**{**prob.__dict__, "k_pages": k2, "v_pages": v2,
                              "page_table": table2})
    again = run_gpu(prob2.to(DEV), out_dtype=torch.float32)
    assert torch.equal(base, again)


def test_deterministic_and_padding_never_read():
    prob = small(lens=(1000, 3, 640), pad_page=10 ** 6)  # padding ids are out of range
    dev = prob.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    a = run_gpu(dev, status=status)
    b = run_gpu(dev, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(a, b)


# split 0: short contexts, one split writing the output directly (bf16) or splits
# merged inside a thread-block cluster (f32); 64: split + merge kernel
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("split", [0, 64])
def test_bad_page_id_flags_status_and_poisons_only_that_sequence(split, dtype):
    prob = small(lens=(100, 200, 50), dtype=dtype)
    prob.page_table[1, 3] = prob.num_pages + 7
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_gpu(prob.to(DEV), out_dtype=torch.float32, status=status, split_tokens=split)
    torch.cuda.synchronize()
    assert int(status.item()) & atlas.DEV_BAD_PAGE
    assert torch.isnan(out[1]).all()
    assert torch.isfinite(out[0]).all() and torch.isfinite(out[2]).all()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("split", [0, 64])
def test_bad_seq_len_flags_status_and_poisons_rows(split, dtype):
    prob = small(lens=(100, 200, 50), dtype=dtype)
    prob.seq_lens[2] = prob.max_pages * prob.page_tokens + 1
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_gpu(prob.to(DEV), out_dtype=torch.float32, status=status, split_tokens=split)
    torch.cuda.synchronize()
    assert int(status.item()) & atlas.DEV_BAD_SEQLEN
    assert torch.isnan(out[2]).all()
    assert torch.isfinite(out[:2]).all()


def test_small_workspace_is_rejected():
    prob = small(lens=(2000, 300, 16)).to(DEV)  # long enough to be split
    with pytest.raises(atlas.AtlasError) as e:
        run_gpu(prob, workspace=torch.empty(16, dtype=torch.uint8, device=DEV))
    assert e.value.status == 3


@pytest.mark.parametrize("split", [0, 64])
def test_bounded_wait_reports_timeout_and_context_survives(split):
    # The producer withholds its first stage: the consumers' bounded wait runs
    # out (about 2 s), the kernel records ATLAS_DEV_TIMEOUT and returns.
    prob = small(B=1, lens=(300,))
    dev = prob.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_gpu(dev, out_dtype=torch.float32, status=status, split_tokens=split,
                  debug_flags=atlas.DEBUG_WITHHOLD_STAGE)
    torch.cuda.synchronize()
    assert int(status.item()) & atlas.DEV_TIMEOUT
    assert torch.isnan(out).all()
    ref = oracle_rows(prob)
    good = run_gpu(dev, out_dtype=torch.float32)
    assert_parity(prob, good, ref, "after timeout")
