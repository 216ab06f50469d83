"""The allocation-free decode entry point (atlas_attn_decode_static_scratch).

It serves callers that cannot allocate device memory on the decode path, so it
keeps the split-KV scratch in a library-owned device array.  This test calls it
through the C ABI twice in a row, on different problems, and checks each result
against the ordinary atlas_attn_decode (which is itself checked against the
fp64 oracle elsewhere) within the parity tolerance: the second call must not
be affected by what the first left in the shared array.  It also checks that a
call needing more scratch than the array holds is refused.

Collected last on purpose (file name), and self-contained: it builds and loads
the library itself, so it passes alone in a fresh process as well.
"""
import ctypes

import numpy as np
import pytest
import torch

import exact_causal_gqa_gb300 as atlas
from exact_causal_gqa_gb300 import inputs

pytestmark = pytest.mark.gpu

STATIC_BYTES = 16 << 20
BF16_ABS = 2e-3
BF16_STORE_REL = 2.0 ** -8


def static_fn():
    lib = atlas.load_library(build_if_missing=True)
    fn = lib.atlas_attn_decode_static_scratch
    fn.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int32] * 4 + [ctypes.c_float,
                                                                  ctypes.POINTER(atlas._Launch)]
    fn.restype = ctypes.c_int
    return fn


def call_static(prob, out, phase=atlas.PHASE_ALL):
    stream = torch.cuda.current_stream().cuda_stream
    L = atlas._launch(prob.q, prob.k_pages, prob.page_table, out.dtype, out=out, stream=stream,
                      phase=phase)
    return static_fn()(prob.q.data_ptr(), prob.k_pages.data_ptr(), prob.v_pages.data_ptr(),
                       prob.page_table.data_ptr(), prob.seq_lens.data_ptr(), prob.n_q_heads,
                       prob.n_kv_heads, prob.head_dim, prob.page_tokens, prob.scale,
                       ctypes.byref(L))


def assert_close(got, ref):
    g = got.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all()
    if got.dtype == torch.float32:
        assert np.abs(g - r).max() <= BF16_ABS
    else:
        assert (np.abs(g - r) <= BF16_ABS + BF16_STORE_REL * np.abs(r)).all()


def test_static_scratch_decode_matches_decode_on_two_calls_in_a_row():
    probs = [
        inputs.make("decode", 4, 32, 8, 128, 16, [5000, 17, 1024, 3333], seed=21).to("cuda"),
        inputs.make("decode", 3, 16, 2, 64, 64, [64, 9000, 130], seed=22).to("cuda"),
    ]
    for prob, dtype in zip(probs, (torch.bfloat16, torch.float32)):
        need = atlas.workspace_size("decode", prob.q.shape, prob.n_q_heads, prob.n_kv_heads,
                                    prob.head_dim, prob.page_tokens, prob.max_pages,
                                    prob.num_pages, dtype=prob.q.dtype, out_dtype=dtype)
        assert 0 < need <= STATIC_BYTES
        out = torch.full(prob.q.shape, float("nan"), dtype=dtype, device="cuda")
        assert call_static(prob, out) == 0
        ref = atlas.run(prob, out_dtype=dtype)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        assert_close(out, ref)


def test_static_scratch_refuses_calls_beyond_its_size():
    # 64 sequences x 64 q heads with a 2^20-token page table: the automatic split
    # plan needs far more than 16 MiB of partials.
    q = torch.zeros((64, 64, 1, 128), dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros((1, 8, 128, 128), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((64, 8192), dtype=torch.int32, device="cuda")
    lens = torch.ones(64, dtype=torch.int32, device="cuda")
    prob = inputs.Problem("decode", q, pool, pool, table, lens, 64, 8, 128, 128, 0.1, 1,
                          "bf16", "bf16")
    need = atlas.workspace_size("decode", q.shape, 64, 8, 128, 128, 8192, 1)
    assert need > STATIC_BYTES
    out = torch.empty_like(q)
    assert call_static(prob, out) == 3  # ATLAS_ERR_WORKSPACE, nothing launched


def test_static_scratch_refuses_calls_spread_over_launches():
    # The partials of a chunked call would sit in the shared array between its
    # launches, where another call could overwrite them: only whole calls run here.
    prob = inputs.make("decode", 2, 8, 2, 128, 16, [300, 41], seed=23).to("cuda")
    out = torch.empty(prob.q.shape, dtype=torch.bfloat16, device="cuda")
    assert call_static(prob, out, phase=atlas.PHASE_CHUNKS) == 2  # ATLAS_ERR_UNSUPPORTED
    assert call_static(prob, out, phase=atlas.PHASE_MERGE) == 2
