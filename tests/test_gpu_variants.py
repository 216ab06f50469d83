"""Score / mask variants (sliding window, logit softcap, attention sinks) on every
kernel path, against the fp64 oracle with the same variant.  Needs a GB300."""
import numpy as np
import pytest
import torch

import exact_causal_gqa_gb300 as atlas
from exact_causal_gqa_gb300 import inputs
from tests.gpu_helpers import assert_parity, flat_rows, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"

# (label, problem factory, extra call kwargs): one per kernel path
PATHS = [
    ("decode bf16 split", lambda: inputs.make("decode", 3, 16, 4, 128, 16, [700, 45, 2100], seed=31), {}),
    ("decode bf16 split 64", lambda: inputs.make("decode", 2, 8, 2, 128, 32, [1000, 333], seed=32),
     dict(split_tokens=64)),
    # short contexts: bf16 one split writing the output directly, f32 splits merged
    # inside a thread-block cluster; then the same f32 call split + merged
    ("decode bf16 direct", lambda: inputs.make("decode", 3, 16, 4, 128, 16, [200, 45, 400],
                                               seed=30), {}),
    ("decode f32 cluster", lambda: inputs.make("decode", 2, 8, 4, 64, 16, [300, 77], dtype="f32",
                                               seed=33), {}),
    ("decode f32 split 64", lambda: inputs.make("decode", 2, 8, 4, 64, 16, [300, 77], dtype="f32",
                                                seed=33), dict(split_tokens=64)),
    ("suffix f32 cluster", lambda: inputs.make("suffix", 2, 8, 2, 128, 16, [400, 90], q_len=3,
                                               dtype="f32", seed=29), {}),
    ("suffix split kernel", lambda: inputs.make("suffix", 2, 8, 4, 128, 16, [500, 90], q_len=4,
                                                seed=34), {}),
    ("suffix tensor core", lambda: inputs.make("suffix", 2, 32, 4, 128, 32, [900, 300], q_len=16,
                                               seed=35), dict(split_tokens=256)),
    # automatic splits: each sequence cut into equal splits, longest first
    ("suffix tensor core balanced", lambda: inputs.make("suffix", 3, 32, 4, 128, 32,
                                                        [3000, 300, 1500], q_len=16, seed=27), {}),
    ("suffix f32 tensor core balanced", lambda: inputs.make("suffix", 3, 16, 2, 64, 32,
                                                            [3000, 300, 1500], q_len=16,
                                                            dtype="f32", seed=26), {}),
    ("prefill direct pair", lambda: inputs.make("prefill", 1, 8, 2, 128, 64, [640], seed=36),
     dict(debug_flags=atlas.DEBUG_TC_DIRECT)),
    ("prefill direct single", lambda: inputs.make("prefill", 1, 6, 2, 128, 16, [384], seed=37),
     dict(debug_flags=atlas.DEBUG_TC_DIRECT)),
    ("prefill split", lambda: inputs.make("prefill", 2, 8, 2, 128, 32, [300, 300], seed=38),
     dict(split_tokens=128)),
]

VARIANTS = [
    dict(window=1),
    dict(window=17),
    dict(window=300, softcap=3.0),
    dict(softcap=1.5),
    dict(sinks=True),
    dict(window=64, softcap=5.0, sinks=True),
]


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: "-".join(f"{k}{v[k]}" for k in v))
@pytest.mark.parametrize("label,make,kw", PATHS, ids=[p[0] for p in PATHS])
def test_variant_parity(label, make, kw, variant):
    prob = make()
    variant = dict(variant)
    sinks_host = None
    if variant.pop("sinks", False):
        g = torch.Generator().manual_seed(prob.n_q_heads)
        sinks_host = (torch.randn(prob.n_q_heads, generator=g) * 2.0).float()
        variant["sinks"] = sinks_host
    ref, ref_lse = oracle_rows(prob, want_lse=True, **variant)
    call = dict(variant)
    if sinks_host is not None:
        call["sinks"] = sinks_host.to(DEV)
    dev = prob.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    lse = torch.empty(flat_rows(prob), dtype=torch.float32, device=DEV)
    out32 = run_gpu(dev, out_dtype=torch.float32, lse=lse, status=status, **kw, **call)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_parity(prob, out32, ref, f"{label} {variant}")
    tol = 1e-4 if prob.dtype == "bf16" else 2e-5
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.reshape(-1), rtol=0, atol=tol)
    if prob.dtype == "bf16":
        out16 = run_gpu(dev, out_dtype=torch.bfloat16, **kw, **call)
        assert torch.equal(out16, out32.to(torch.bfloat16))


def test_variant_arguments_are_checked():
    prob = inputs.make("decode", 1, 4, 1, 128, 16, [40], seed=39).to(DEV)
    with pytest.raises(atlas.AtlasError):
        run_gpu(prob, window=-1)
    with pytest.raises(atlas.AtlasError):
        run_gpu(prob, softcap=float("nan"))
    with pytest.raises(ValueError):
        run_gpu(prob, sinks=torch.zeros(3, device=DEV))
