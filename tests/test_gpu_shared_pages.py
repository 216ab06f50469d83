"""Shared prefix pages (ferrox-core paged KV sharing; CFR-Atlas pages named by identity,
not by owner): several sequences' page tables point at the same physical pages.  Every
kernel path must read them like any other page: parity with the oracle, and a sequence
that is an exact copy of another (same q, same pages, same length) gives the same bits."""
import pytest
import torch

from exact_causal_gqa_gb300 import inputs
from tests.gpu_helpers import assert_parity, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind,dtype,Hq,Hkv,D,P,q_len,lens,shared", [
    ("decode", "bf16", 32, 8, 128, 16, 1, (2000, 1500, 2000), 40),    # mma.sync split kernel
    ("suffix", "bf16", 32, 4, 128, 32, 16, (3000, 2600, 3000), 50),   # tcgen05, split + merge
    ("prefill", "bf16", 8, 2, 128, 64, 300, (300, 300, 300), 3),       # tcgen05, direct
    ("decode", "f32", 8, 4, 64, 16, 1, (900, 700, 900), 20),           # fp32 ring kernel
    ("suffix", "f32", 16, 2, 128, 16, 16, (1200, 1000, 1200), 30),     # fp32 tensor-core kernel (3 x tf32)
])
def test_shared_prefix_pages(kind, dtype, Hq, Hkv, D, P, q_len, lens, shared):
    host = inputs.make(kind, 3, Hq, Hkv, D, P, list(lens), q_len=q_len, dtype=dtype,
                       out_dtype=dtype, seed=len(lens) + shared, device="cpu")
    # sequence 1 reads sequence 0's first `shared` pages; sequence 2 is sequence 0 again
    host.page_table[1, :shared] = host.page_table[0, :shared]
    host.page_table[2] = host.page_table[0]
    host.q[2] = host.q[0]
    dev = inputs.Problem(**{k: (v.to("cuda") if torch.is_tensor(v) else v)
                            for k, v in vars(host).items()})
    out = run_gpu(dev, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_parity(host, out, oracle_rows(host), f"{kind} {dtype} shared pages")
    assert torch.equal(out[2], out[0])
