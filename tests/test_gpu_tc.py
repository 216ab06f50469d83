"""Parity of the tensor-core (tcgen05 / TMEM) suffix and prefill path with the
fp64 oracle, through the C ABI, on the same seeded host bytes.  Needs a GB300."""
import numpy as np
import pytest
import torch

import exact_causal_gqa_gb300 as atlas
from exact_causal_gqa_gb300 import inputs
from tests.gpu_helpers import assert_parity, flat_rows, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def check(prob, split=0, flags=0):
    ref, ref_lse = oracle_rows(prob, want_lse=True)
    dev = prob.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    lse = torch.empty(flat_rows(prob), dtype=torch.float32, device=DEV)
    out32 = run_gpu(dev, out_dtype=torch.float32, lse=lse, status=status, split_tokens=split,
                    debug_flags=flags)
    out16 = run_gpu(dev, out_dtype=torch.bfloat16, split_tokens=split, debug_flags=flags)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_parity(prob, out32, ref, "f32 out")
    assert_parity(prob, out16, ref, "bf16 out")
    assert torch.equal(out16, out32.to(torch.bfloat16))
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.reshape(-1), rtol=0, atol=2e-4)
    return out32


SUFFIX = [
    # (B, Hq, Hkv, P, SQ, lens)
    (3, 32, 4, 32, 16, (16, 300, 1000)),       # G*SQ = 128: one tile per (seq, kv head)
    (2, 8, 1, 16, 16, (129, 4097)),            # one tile, P = 16
    (2, 16, 2, 64, 4, (64, 777)),              # G*SQ = 32: a partial tile
    (1, 16, 1, 128, 32, (1024,)),              # G*SQ = 512: four tiles, P = 128
    (2, 12, 4, 8, 8, (33, 2000)),              # G = 3, G*SQ = 24, P = 8
]


@pytest.mark.parametrize("B,Hq,Hkv,P,SQ,lens", SUFFIX)
@pytest.mark.parametrize("split", [0, 128, 384])
def test_suffix_parity(B, Hq, Hkv, P, SQ, lens, split):
    prob = inputs.make("suffix", B, Hq, Hkv, 128, P, list(lens), q_len=SQ, seed=B + Hq + P + SQ)
    check(prob, split=split)


D64 = [
    # (kind, B, Hq, Hkv, P, q_len, lens)
    ("suffix", 1, 8, 2, 16, 16, (256,)),        # the CPUAttn example: q (1,8,16,64), k/v (1,2,256,64)
    ("suffix", 3, 32, 4, 32, 16, (16, 300, 1000)),
    ("suffix", 2, 12, 4, 8, 8, (33, 2000)),
    ("prefill", 1, 4, 1, 64, 128, None),
    ("prefill", 2, 8, 2, 16, 300, None),
    ("prefill", 1, 32, 8, 64, 200, None),
]


@pytest.mark.parametrize("kind,B,Hq,Hkv,P,q_len,lens", D64)
@pytest.mark.parametrize("mode", ["auto", "split256", "direct"])
def test_head_dim_64_parity(kind, B, Hq, Hkv, P, q_len, lens, mode):
    """bf16 head_dim 64 with many query rows per kv head (suffix and prefill)."""
    lens = list(lens) if lens else [q_len] * B
    prob = inputs.make(kind, B, Hq, Hkv, 64, P, lens, q_len=q_len, seed=64 + B + Hq + P)
    split = 256 if mode == "split256" else 0
    flags = atlas.DEBUG_TC_DIRECT if mode == "direct" else 0
    check(prob, split=split, flags=flags)


PREFILL = [
    # (B, Hq, Hkv, P, S)
    (1, 4, 1, 64, 128),
    (2, 4, 2, 64, 129),
    (1, 8, 2, 16, 300),
    (1, 2, 2, 128, 1000),
    (2, 8, 8, 32, 640),
    (1, 32, 8, 64, 100),
]


@pytest.mark.parametrize("B,Hq,Hkv,P,S", PREFILL)
@pytest.mark.parametrize("mode", ["direct", "split256", "auto"])
def test_prefill_parity(B, Hq, Hkv, P, S, mode):
    prob = inputs.make("prefill", B, Hq, Hkv, 128, P, [S] * B, seed=S + Hq + P)
    split = 256 if mode == "split256" else 0
    flags = atlas.DEBUG_TC_DIRECT if mode == "direct" else 0
    check(prob, split=split, flags=flags)


def test_prefill_direct_is_deterministic_and_page_order_invariant():
    prob = inputs.make("prefill", 2, 8, 2, 128, 32, [700, 700], seed=9, extra_pages=3)
    dev = prob.to(DEV)
    a = run_gpu(dev, out_dtype=torch.float32, debug_flags=atlas.DEBUG_TC_DIRECT)
    b = run_gpu(dev, out_dtype=torch.float32, debug_flags=atlas.DEBUG_TC_DIRECT)
    assert torch.equal(a, b)
    perm = torch.randperm(prob.num_pages, generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(prob.num_pages)
    k2 = torch.empty_like(prob.k_pages)
    v2 = torch.empty_like(prob.v_pages)
    k2[inv] = prob.k_pages
    v2[inv] = prob.v_pages
    prob2 = inputs.Problem(**{**prob.__dict__, "k_pages": k2, "v_pages": v2,
                              "page_table": inv[prob.page_table.long()].to(torch.int32)})
    c = run_gpu(prob2.to(DEV), out_dtype=torch.float32, debug_flags=atlas.DEBUG_TC_DIRECT)
    assert torch.equal(a, c)


@pytest.mark.parametrize("flags,split", [(atlas.DEBUG_TC_DIRECT, 0), (0, 256)])
def test_tc_bad_page_and_seq_len(flags, split):
    prob = inputs.make("suffix", 3, 32, 4, 128, 32, [300, 400, 500], q_len=16, seed=4)
    prob.page_table[1, 2] = -3
    prob.seq_lens[2] = 7  # fewer keys than query rows
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_gpu(prob.to(DEV), out_dtype=torch.float32, status=status, split_tokens=split,
                  debug_flags=flags)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st & atlas.DEV_BAD_PAGE and st & atlas.DEV_BAD_SEQLEN
    assert torch.isnan(out[1]).all() and torch.isnan(out[2]).all()
    assert torch.isfinite(out[0]).all()


@pytest.mark.parametrize("flags", [atlas.DEBUG_TC_DIRECT, 0])
@pytest.mark.parametrize("bad", ["negative", "num_pages", "huge"])
def test_prefill_bad_page_id_poisons_the_rows_that_read_it(bad, flags):
    # page 3 of sequence 0 holds keys 192..255: rows from 192 on read it, rows below
    # 128 sit in tiles whose key range ends before it
    prob = inputs.make("prefill", 2, 8, 2, 128, 64, [384, 384], seed=6)
    prob.page_table[0, 3] = {"negative": -1, "num_pages": prob.num_pages, "huge": 1 << 30}[bad]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_gpu(prob.to(DEV), out_dtype=torch.float32, status=status, debug_flags=flags)
    torch.cuda.synchronize()
    assert int(status.item()) == atlas.DEV_BAD_PAGE
    assert torch.isnan(out[0, :, 192:]).all()
    assert torch.isfinite(out[0, :, :128]).all() and torch.isfinite(out[1]).all()


def test_prefill_rejects_seq_len_different_from_q_len():
    prob = inputs.make("prefill", 2, 8, 2, 128, 64, [256, 256], seed=5)
    prob.seq_lens[1] = 255
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_gpu(prob.to(DEV), out_dtype=torch.float32, status=status,
                  debug_flags=atlas.DEBUG_TC_DIRECT)
    torch.cuda.synchronize()
    assert int(status.item()) & atlas.DEV_BAD_SEQLEN
    assert torch.isnan(out[1]).all() and torch.isfinite(out[0]).all()


def sampled(prob, rows, out32, out16):
    ref = oracle_rows(prob, rows=rows)
    D = prob.head_dim
    idx = torch.from_numpy(rows).to(DEV)
    assert_parity(prob, out32.reshape(-1, D)[idx], ref, "f32 out")
    assert_parity(prob, out16.reshape(-1, D)[idx], ref, "bf16 out")
    assert torch.equal(out16, out32.to(torch.bfloat16))
    assert torch.isfinite(out32).all()


def test_config4_suffix_full_size_every_row():
    """Suffix queries at full size (16 sequences x 32 heads x 16 rows, contexts up to
    64K keys), in bench.py's launch configuration: every output row."""
    prob = inputs.make_config(4)
    dev = prob.to(DEV)
    out16 = run_gpu(dev)
    out32 = run_gpu(dev, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = oracle_rows(prob)
    assert_parity(prob, out32, ref, "f32 out")
    assert_parity(prob, out16, ref, "bf16 out")
    assert torch.equal(out16, out32.to(torch.bfloat16))


def test_config5_prefill_full_size_whole_group_and_samples():
    """Causal prefill at full size (2 x 8192 rows, 32 / 8 heads): every row of one
    whole (sequence, kv head) group -- all its G q heads, all 8192 positions -- plus a
    spread of rows over the other groups, including the first rows of tiles."""
    prob = inputs.make_config(5)
    dev = prob.to(DEV)
    out16 = run_gpu(dev)
    out32 = run_gpu(dev, out_dtype=torch.float32)
    torch.cuda.synchronize()
    S, H = prob.q_len, prob.n_q_heads
    G = H // prob.n_kv_heads
    b, g = 1, 5
    group = [(b * H + h) * S + i for h in range(g * G, (g + 1) * G) for i in range(S)]
    rng = np.random.default_rng(5)
    early = [(bb * H + h) * S + i for bb in range(2) for h in (0, 13, 31)
             for i in (0, 1, 2, 63, 127, 128, 511, 512, 4095, S - 1)]
    rows = np.unique(np.concatenate([group, early,
                                     rng.choice(flat_rows(prob), 256, replace=False)]))
    sampled(prob, rows, out32, out16)


@pytest.mark.parametrize("scale", [-0.07, 0.0, 0.31])
def test_tc_any_finite_scale(scale):
    # S = -Q K^T with |scale| for negative scales; scale 0 gives uniform weights.
    prob = inputs.make("suffix", 2, 32, 4, 128, 32, [200, 1000], q_len=16, seed=7, scale=scale)
    check(prob)
    prob = inputs.make("prefill", 1, 8, 2, 128, 64, [384], seed=8, scale=scale)
    check(prob, flags=atlas.DEBUG_TC_DIRECT)


def test_decode_any_finite_scale():
    prob = inputs.make("decode", 3, 16, 4, 128, 16, [5, 300, 2000], seed=9, scale=-0.2)
    check(prob)


@pytest.mark.parametrize("kind,q_len,lens", [("prefill", 2048, [2048]), ("suffix", 64, [3000, 5000])])
def test_late_score_jumps(kind, q_len, lens):
    # K rows scaled x16 (about 0.2 % of keys) give later blocks scores far above the
    # running max: the plain-path blocks after the first must rescale the P they
    # already wrote with the old reference.
    prob = inputs.make(kind, len(lens), 8, 2, 128, 64, lens, q_len=q_len, seed=21,
                       k_outlier_prob=0.002, k_outlier_scale=16.0)
    check(prob)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_suffix_batch_past_the_longest_first_order(dtype):
    """More sequences than the kernels order longest-first (kTcOrderMaxSeqs = 128): the
    automatic plan falls back to fixed chunks in grid order, with split + merge."""
    B = 131
    g = np.random.default_rng(5)
    lens = [int(x) for x in g.integers(20, 2500, size=B)]
    prob = inputs.make("suffix", B, 8, 1, 64, 32, lens, q_len=4, dtype=dtype, seed=41)
    ref, ref_lse = oracle_rows(prob, want_lse=True)
    dev = prob.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    lse = torch.empty(flat_rows(prob), dtype=torch.float32, device=DEV)
    out = run_gpu(dev, out_dtype=torch.float32, lse=lse, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_parity(prob, out, ref, f"B{B} {dtype}")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.reshape(-1), rtol=0,
                               atol=2e-4 if dtype == "bf16" else 2e-5)


@pytest.mark.parametrize("kind,lens,q_len,outlier,scale", [
    ("prefill", [2048], 2048, (0.02, 3.0), None),
    ("prefill", [2048], 2048, (0.002, 4.0), None),
    ("prefill", [2048], 2048, (0.0, 1.0), 1.15),
    ("prefill", [2048], 2048, (0.0, 1.0), 1.24),
    ("suffix", [3000, 5000], 64, (0.002, 4.0), None),
    ("suffix", [3000, 5000], 64, (0.02, 3.0), None),
])
def test_hilo_threshold_margin(kind, lens, q_len, outlier, scale):
    # The inputs that came closest to the bound when the per-block hi + lo threshold was
    # chosen (outlier K rows, scores as sharp as the limit above which every block takes
    # hi + lo): the largest error must keep a margin of 2 to 2e-3.
    prob = inputs.make(kind, len(lens), 8, 2, 128, 64, lens, q_len=q_len, seed=102,
                       k_outlier_prob=outlier[0], k_outlier_scale=outlier[1],
                       scale=None if scale is None else scale / np.sqrt(128))
    out = run_gpu(prob.to(DEV), out_dtype=torch.float32,
                  debug_flags=atlas.DEBUG_TC_DIRECT if kind == "prefill" else 0)
    torch.cuda.synchronize()
    err = assert_parity(prob, out, oracle_rows(prob), kind)
    assert err <= 1e-3, f"{kind}: max err {err:.3e} leaves less than a 2x margin"
