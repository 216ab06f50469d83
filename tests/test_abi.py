"""CPU-side checks of the C ABI: the library builds and loads, exports every
function include/*.h declares, and its host-only logic (argument
checks, workspace sizing, status strings) behaves as documented.  No kernel is
launched: every call here returns before any CUDA work."""
import ctypes
import os
import re
import subprocess

import pytest

import exact_causal_gqa_gb300 as atlas
from exact_causal_gqa_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return atlas.load_library()


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            text = open(os.path.join(inc, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(atlas_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("atlas_attn_decode", "atlas_attn_suffix", "atlas_attn_prefill",
              "atlas_attn_workspace_size", "atlas_attn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(\w+)$", out, flags=re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"not exported: {missing}"
    for n in declared_functions():
        assert hasattr(lib, n)


def test_status_strings(lib):
    for code in range(6):
        assert atlas.status_string(code)
    assert atlas.status_string(99) == "unknown status"


def launch(**kw):
    L = atlas._Launch()
    L.batch, L.max_pages_per_seq, L.num_pages, L.q_len = 2, 8, 16, 1
    L.q_dtype = L.kv_dtype = L.out_dtype = 1
    for k, v in kw.items():
        setattr(L, k, v)
    return L


def ws(lib, kind=0, Hq=8, Hkv=2, D=128, P=16, **kw):
    L = launch(**kw)
    return lib.atlas_attn_workspace_size(kind, Hq, Hkv, D, P, ctypes.byref(L))


SIZE_MAX = ctypes.c_size_t(-1).value


def test_workspace_size_matches_the_split_layout(lib):
    # 2 sequences x 8 q heads x 1 row, context <= 128 keys, 64-key splits -> 2 splits
    n = ws(lib, split_tokens=64)
    rows, splits, D = 2 * 8, 2, 128
    acc = rows * splits * D * 4
    assert n == (acc + 255) // 256 * 256 + rows * splits * 2 * 4
    # fp32 K/V: the same layout
    assert ws(lib, split_tokens=64, q_dtype=0, kv_dtype=0, out_dtype=0) == n


@pytest.mark.parametrize("kw,expect", [
    (dict(Hq=6, Hkv=4), SIZE_MAX),          # Hq not a multiple of Hkv
    (dict(D=96), SIZE_MAX),                 # unsupported head_dim
    (dict(P=12), SIZE_MAX),                 # page_tokens not a power of two
    (dict(P=256), SIZE_MAX),                # page_tokens above 128
    (dict(q_len=2), SIZE_MAX),              # decode takes one query row
    (dict(split_tokens=100), SIZE_MAX),     # splits must be multiples of 64
    (dict(out_dtype=0, q_dtype=0, kv_dtype=1), SIZE_MAX),  # q and K/V dtypes differ
    (dict(kv_dtype=0, q_dtype=0, out_dtype=1), SIZE_MAX),  # f32 K/V only gives f32 out
    (dict(batch=1 << 23, Hq=256), SIZE_MAX),  # batch * n_q_heads * q_len >= 2^31 - 1
])
def test_invalid_plans_are_rejected(lib, kw, expect):
    assert ws(lib, **kw) == expect


def test_entry_points_check_arguments_before_any_launch(lib):
    L = launch()
    args = [None] * 5 + [8, 2, 128, 16, ctypes.c_float(0.1), ctypes.byref(L)]
    for name in ("atlas_attn_decode", "atlas_attn_suffix", "atlas_attn_prefill"):
        assert getattr(lib, name)(*args) == 1  # null pointers -> ATLAS_ERR_INVALID_ARG
    # misaligned pointers are rejected too
    fake = 0x1000
    L.out = fake + 8
    args = [fake, fake, fake, fake, fake, 8, 2, 128, 16, ctypes.c_float(0.1), ctypes.byref(L)]
    assert lib.atlas_attn_decode(*args) == 1
    # unsupported head_dim
    L.out = fake
    args = [fake, fake, fake, fake, fake, 8, 2, 80, 16, ctypes.c_float(0.1), ctypes.byref(L)]
    assert lib.atlas_attn_decode(*args) == 2
    # missing workspace (a context long enough to be split: 16K keys per sequence)
    L.max_pages_per_seq = 1024
    args = [fake, fake, fake, fake, fake, 8, 2, 128, 16, ctypes.c_float(0.1), ctypes.byref(L)]
    assert lib.atlas_attn_decode(*args) == 3
    # non-finite scale
    args = [fake, fake, fake, fake, fake, 8, 2, 128, 16, ctypes.c_float(float("nan")),
            ctypes.byref(L)]
    assert lib.atlas_attn_decode(*args) == 1


def split_tokens(lib, kind=0, Hq=8, Hkv=2, D=128, P=16, **kw):
    L = launch(**kw)
    return lib.atlas_attn_split_tokens(kind, Hq, Hkv, D, P, ctypes.byref(L))


def test_split_tokens_and_phases(lib):
    # the chunk size the pool's planner needs: the same as the plan's
    assert split_tokens(lib, split_tokens=64) == 64
    assert split_tokens(lib, split_tokens=64, phase=1) == 64
    # invalid phase, invalid sizes
    assert split_tokens(lib, phase=3) == -1
    assert split_tokens(lib, Hq=7) == -1
    assert lib.atlas_attn_workspace_size(0, 8, 2, 128, 16, ctypes.byref(launch(phase=7))) == SIZE_MAX
    # a tensor-core call that would write its output directly has no chunks with
    # phase ALL under the debug flag, and refuses the chunked phases then
    tc = dict(q_len=64, batch=1, max_pages_per_seq=64, num_pages=64)
    assert split_tokens(lib, kind=1, Hq=32, Hkv=4, debug_flags=atlas.DEBUG_TC_DIRECT, **tc) == 0
    assert split_tokens(lib, kind=1, Hq=32, Hkv=4, debug_flags=atlas.DEBUG_TC_DIRECT, phase=1,
                        **tc) == -1
    # without the flag a chunked phase always gets chunks (multiples of 128 there)
    n = split_tokens(lib, kind=1, Hq=32, Hkv=4, phase=1, **tc)
    assert n > 0 and n % 128 == 0


def test_split_plan_sizes(lib):
    """The automatic split sizes are a pure function of the call's sizes: bf16 decode
    aims for 152 x 2 x 2 CTAs, the fp32 ring kernel with 4 or 8 columns (4-warp CTAs,
    three per SM) for 152 x 3 x 4, both capped at 2560 keys and rounded to 64."""
    f32 = dict(q_dtype=0, kv_dtype=0, out_dtype=0)

    def plan(batch, Hq, Hkv, ctx, P=16, **kw):
        pages = ctx // P
        return split_tokens(lib, Hq=Hq, Hkv=Hkv, P=P, batch=batch, max_pages_per_seq=pages,
                            num_pages=batch * pages, **kw)

    def expect(units, ctx, target):
        chunk = -(-(-(-ctx * units // target)) // 64) * 64
        return min(max(chunk, 64), 2560)

    # bf16 GQA decode, 32 x 8 (sequence, kv head) units at 32K keys: the cap
    assert plan(32, 32, 8, 32768) == 2560
    assert plan(4, 32, 8, 32768) == max(512, expect(32, 32768, 608))
    # fp32, 4 columns (G = 4): 1824-CTA target
    assert plan(4, 32, 8, 32768, **f32) == expect(32, 32768, 1824) == 576
    assert plan(1, 32, 8, 32768, **f32) == expect(8, 32768, 1824) == 192
    assert plan(32, 32, 8, 32768, **f32) == 2560
    # fp32, 8 columns (G = 8), long context
    assert plan(4, 64, 8, 131072, P=64, **f32) == expect(32, 131072, 1824) == 2304
    # fp32, 16 columns (G = 16): 8-warp CTAs, the 608-CTA target
    assert plan(2, 32, 2, 16384, **f32) == expect(4, 16384, 608) == 128


def test_tensor_core_plan_sizes(lib):
    """Tensor-core calls (bf16, G * q_len > 16): splits of 1024-8192 keys in multiples of
    128, aiming for 152 x 3 CTAs; prefill with at least 304 query tiles writes the output
    directly (no chunks)."""
    def plan(kind, batch, Hq, Hkv, q_len, ctx, P):
        pages = ctx // P
        return split_tokens(lib, kind=kind, Hq=Hq, Hkv=Hkv, P=P, batch=batch, q_len=q_len,
                            max_pages_per_seq=pages, num_pages=batch * pages)

    # suffix of 16 rows, G = 8, contexts up to 64K keys: 64 tiles -> the 8192-key cap
    assert plan(1, 16, 32, 4, 16, 65536, 32) == 8192
    # one short suffix: the 1024-key floor
    assert plan(1, 1, 32, 4, 16, 4096, 32) == 1024
    # causal prefill of 2 x 8192 rows, 32 / 8 heads: 4096 tiles, direct
    assert plan(2, 2, 32, 8, 8192, 8192, 64) == 0
    # a small prefill (64 tiles) is split, capped at its own length
    assert plan(2, 1, 8, 2, 1024, 1024, 64) == 1024


def test_split_plan_follows_the_sm_count(lib):
    """The automatic plan fills the SMs it is given (atlas_launch.sm_count): the split
    targets scale with the count, and a count of 0 means the device's own (152, one
    GB300, on a host without a GPU)."""
    def plan(sms, batch=4, Hq=32, Hkv=8, ctx=32768, P=16, kind=0, q_len=1, **kw):
        pages = ctx // P
        return split_tokens(lib, kind=kind, Hq=Hq, Hkv=Hkv, P=P, batch=batch, q_len=q_len,
                            max_pages_per_seq=pages, num_pages=batch * pages, sm_count=sms,
                            **kw)

    def expect(units, ctx, target, lo, hi):
        chunk = -(-(-(-ctx * units // target)) // 64) * 64
        return min(max(chunk, lo), hi)

    # bf16 decode: SMs x 2 x 2 CTAs, 512..2560 keys
    for sms in (152, 148, 132, 76, 20):
        assert plan(sms) == expect(32, 32768, sms * 4, 512, 2560), sms
    assert plan(0) == plan(152)
    # fp32 ring (G = 4): SMs x 3 x 4 CTAs
    f32 = dict(q_dtype=0, kv_dtype=0, out_dtype=0)
    for sms in (152, 76):
        assert plan(sms, batch=1, **f32) == expect(8, 32768, sms * 12, 64, 2560)
    # tensor-core suffix: SMs x 3 CTAs, 1024..8192 keys in multiples of 128
    for sms in (152, 40):
        n = plan(sms, batch=1, Hq=32, Hkv=4, ctx=65536, P=32, kind=1, q_len=16)
        tiles = 4
        want = -(-(65536 * tiles) // (sms * 3))
        want = min(max(-(-want // 128) * 128, 1024), 8192)
        assert n == want, sms
    # prefill writes its output directly at >= SMs x 2 query tiles (4096 here), so a
    # part with 4096 / 2 + 1 SMs would split it
    assert plan(152, batch=2, Hq=32, Hkv=8, ctx=8192, P=64, kind=2, q_len=8192) == 0
    assert plan(2049, batch=2, Hq=32, Hkv=8, ctx=8192, P=64, kind=2, q_len=8192) > 0
    # a negative count is an invalid argument
    assert plan(-1) == -1


def test_short_decode_contexts_write_their_output_directly(lib):
    """A decode-like call whose context per (sequence, kv head) holds at most 256 KB of
    K/V runs one split per unit that writes the output itself: no chunks, no
    workspace.  Longer contexts, a fixed split size or a chunked phase keep the split
    form."""
    def both(P=16, pages=8, D=128, **kw):
        return (ws(lib, D=D, P=P, max_pages_per_seq=pages, **kw),
                split_tokens(lib, D=D, P=P, max_pages_per_seq=pages, **kw))

    f32 = dict(q_dtype=0, kv_dtype=0, out_dtype=0)
    # 512 keys x 2 x 64 x 4 B = 256 KB (fp32, head_dim 64, as the single-sequence decode)
    assert both(pages=32, D=64, Hq=4, Hkv=4, **f32) == (0, 0)
    assert both(pages=33, D=64, Hq=4, Hkv=4, **f32)[0] > 0
    # bf16, head_dim 128: 512 keys = 256 KB
    assert both(pages=32) == (0, 0)
    assert both(pages=33)[0] > 0
    # a fixed split size or a chunked phase keeps the split form
    assert both(pages=8, split_tokens=64)[0] > 0
    assert both(pages=8, phase=1)[1] > 0
