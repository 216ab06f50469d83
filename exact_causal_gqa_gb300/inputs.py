"""Seeded synthetic inputs for paged causal GQA attention.

This module only draws and lays out data: it holds none of the attention
arithmetic, so both the CUDA path's tests and the CPU oracle can consume the
same host bytes.  Shapes follow the five workloads the library is measured on
(decode, GQA decode, long-context decode, suffix queries, causal prefill).

Recipe (all draws from ``torch.Generator`` seeded per problem):
  * per-sequence context lengths: integers uniform on [lo, hi], both ends inclusive;
  * pool pages: exactly sum_b ceil(L_b / P) pages (plus ``extra_pages`` unused
    ones), logical page p of sequence b stored at a slot chosen by one seeded
    random permutation of the pool;
  * q, K, V values: N(0, 1) drawn in fp32, optionally K rows scaled by
    ``k_outlier_scale`` with probability ``k_outlier_prob`` per (sequence,
    kv head, token), then rounded once to the storage dtype (RNE);
  * slots past a sequence's length in its last page, and unused pages, are
    filled with NaN unless ``poison=False``: no correct kernel ever reads them;
  * page-table entries past a sequence's last page hold ``pad_page`` (0 by
    default; tests pass an out-of-range id to show they are never read).

Layouts: q / out [B][Hq][q_len][D]; k_pages / v_pages [num_pages][Hkv][P][D];
page_table [B][max_pages] int32; seq_lens [B] int32.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

# The five workloads.  kind: decode (q_len 1), suffix (q_len SQ), prefill (q_len = L).
CONFIGS = {
    1: dict(name="decode_mha_f32_b1_h4_d64_ctx512_p16", kind="decode", B=1, Hq=4, Hkv=4,
            D=64, P=16, ctx=(512, 512), q_len=1, dtype="f32", out_dtype="f32",
            scale=1.0 / 8.0),
    2: dict(name="gqa_decode_bf16_b32_h32x8_d128_ctx1k-32k_p16", kind="decode", B=32, Hq=32,
            Hkv=8, D=128, P=16, ctx=(1024, 32768), q_len=1, dtype="bf16",
            out_dtype="bf16", scale=1.0 / math.sqrt(128)),
    3: dict(name="long_decode_bf16_b4_h64x8_d128_ctx128k_p64_outliers", kind="decode", B=4,
            Hq=64, Hkv=8, D=128, P=64, ctx=(131072, 131072), q_len=1, dtype="bf16",
            out_dtype="bf16", scale=1.0 / math.sqrt(128), k_outlier_prob=0.01,
            k_outlier_scale=8.0),
    4: dict(name="suffix_bf16_b16_sq16_h32x4_d128_ctx4k-64k_p32", kind="suffix", B=16, Hq=32,
            Hkv=4, D=128, P=32, ctx=(4096, 65536), q_len=16, dtype="bf16",
            out_dtype="bf16", scale=1.0 / math.sqrt(128)),
    5: dict(name="prefill_bf16_b2_s8192_h32x8_d128_p64", kind="prefill", B=2, Hq=32, Hkv=8,
            D=128, P=64, ctx=(8192, 8192), q_len=8192, dtype="bf16", out_dtype="bf16",
            scale=1.0 / math.sqrt(128)),
}

_TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclasses.dataclass
class Problem:
    """One attention call's inputs (all tensors on ``device``)."""
    kind: str
    q: torch.Tensor
    k_pages: torch.Tensor
    v_pages: torch.Tensor
    page_table: torch.Tensor
    seq_lens: torch.Tensor
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    page_tokens: int
    scale: float
    q_len: int
    dtype: str
    out_dtype: str
    name: str = ""

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def num_pages(self) -> int:
        return self.k_pages.shape[0]

    @property
    def max_pages(self) -> int:
        return self.page_table.shape[1]

    def to(self, device) -> "Problem":
        moved = {f.name: getattr(self, f.name) for f in dataclasses.fields(self)}
        for key in ("q", "k_pages", "v_pages", "page_table", "seq_lens"):
            moved[key] = moved[key].to(device)
        return Problem(**moved)

    def kv_bytes(self) -> int:
        """K and V bytes a decode/suffix call must read: every visible key once."""
        elem = self.k_pages.element_size()
        return 2 * int(self.seq_lens.to(torch.int64).sum()) * self.n_kv_heads * self.head_dim * elem


def _normal(shape, gen, device, dtype, scale_rows=None):
    """N(0,1) in fp32 rounded once to ``dtype``; drawn in slabs to bound memory."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(shape[0], -1)
    step = max(1, (1 << 26) // max(1, flat.shape[1]))
    for s in range(0, shape[0], step):
        e = min(shape[0], s + step)
        x = torch.randn((e - s,) + tuple(shape[1:]), generator=gen, device=device,
                        dtype=torch.float32)
        if scale_rows is not None:
            x.mul_(scale_rows[s:e].unsqueeze(-1))
        out[s:e].copy_(x)  # RNE for bf16
    return out


def make(kind: str, B: int, Hq: int, Hkv: int, D: int, P: int,
         seq_lens: Sequence[int], q_len: Optional[int] = None, dtype: str = "bf16",
         out_dtype: Optional[str] = None, scale: Optional[float] = None,
         seed: int = 0, device="cpu", max_pages: Optional[int] = None,
         extra_pages: int = 0, poison: bool = True, pad_page: int = 0,
         k_outlier_prob: float = 0.0, k_outlier_scale: float = 1.0,
         name: str = "") -> Problem:
    """Build a problem with explicit per-sequence context lengths."""
    lens = [int(x) for x in seq_lens]
    assert len(lens) == B
    if kind == "decode":
        q_len = 1 if q_len is None else q_len
    elif kind == "prefill":
        q_len = lens[0] if q_len is None else q_len
    assert q_len is not None and q_len >= 1
    tdt = _TORCH_DTYPES[dtype]
    out_dtype = out_dtype or dtype
    scale = 1.0 / math.sqrt(D) if scale is None else scale

    host = torch.Generator(device="cpu").manual_seed(seed)
    gen = torch.Generator(device=device).manual_seed(seed + 7919)

    pages_per_seq = [(n + P - 1) // P for n in lens]
    used = sum(pages_per_seq)
    num_pages = max(1, used + extra_pages)
    if max_pages is None:
        max_pages = max(1, max(pages_per_seq))
    assert max_pages >= max(pages_per_seq)

    perm = torch.randperm(num_pages, generator=host)
    table = torch.full((B, max_pages), pad_page, dtype=torch.int32)
    cursor = 0
    for b, n in enumerate(pages_per_seq):
        table[b, :n] = perm[cursor:cursor + n].to(torch.int32)
        cursor += n

    q = _normal((B, Hq, q_len, D), gen, device, tdt)
    scale_rows = None
    if k_outlier_prob > 0.0:
        hit = torch.rand((num_pages, Hkv, P), generator=gen, device=device) < k_outlier_prob
        scale_rows = torch.where(hit, torch.tensor(k_outlier_scale, device=device),
                                 torch.tensor(1.0, device=device))
    k_pages = _normal((num_pages, Hkv, P, D), gen, device, tdt, scale_rows)
    v_pages = _normal((num_pages, Hkv, P, D), gen, device, tdt)

    if poison:
        nan = float("nan")
        for b, n in enumerate(lens):
            tail = n % P
            if tail:
                last = int(table[b, pages_per_seq[b] - 1])
                k_pages[last, :, tail:, :] = nan
                v_pages[last, :, tail:, :] = nan
        if extra_pages:
            unused = perm[used:].to(device)
            k_pages[unused] = nan
            v_pages[unused] = nan

    return Problem(kind=kind, q=q, k_pages=k_pages, v_pages=v_pages,
                   page_table=table.to(device),
                   seq_lens=torch.tensor(lens, dtype=torch.int32, device=device),
                   n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, page_tokens=P, scale=scale,
                   q_len=q_len, dtype=dtype, out_dtype=out_dtype, name=name)


def make_config(index: int, seed: Optional[int] = None, device="cpu", **overrides) -> Problem:
    """One of the five workloads, seeded by its index unless ``seed`` is given."""
    cfg = dict(CONFIGS[index])
    cfg.update(overrides)
    seed = index if seed is None else seed
    host = torch.Generator(device="cpu").manual_seed(seed * 1000003 + 17)
    lo, hi = cfg["ctx"]
    lens = torch.randint(lo, hi + 1, (cfg["B"],), generator=host).tolist()
    q_len = cfg["q_len"]
    max_pages = (hi + cfg["P"] - 1) // cfg["P"]
    return make(cfg["kind"], cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["P"], lens,
                q_len=q_len, dtype=cfg["dtype"], out_dtype=cfg["out_dtype"],
                scale=cfg["scale"], seed=seed, device=device, max_pages=max_pages,
                k_outlier_prob=cfg.get("k_outlier_prob", 0.0),
                k_outlier_scale=cfg.get("k_outlier_scale", 1.0),
                poison=cfg.get("poison", True), name=cfg["name"])
