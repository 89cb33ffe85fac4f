"""Sizes past the 32-bit element range and long contexts: every row offset, tensor-map row
coordinate and key count must be carried in 64 bits (or stay below 2^31 by construction).
Checked on sampled rows against the oracle, one query token at a time (token t is query 0 of a
one-token prefill at position t, which sees the same keys), so the host never holds the whole
query tensor.

Caches and key tables past 2^31 elements: the used pages (or listed rows) of a small seeded case
sit at the top of a cache of more than 3.73M rows (row x 576 past 2^31), everything below them
NaN, so an offset that wrapped or a row read from the wrong place shows in the output.  The
oracle runs on the small case itself; only the placement differs."""
import numpy as np
import pytest
import torch

import oracle.mla_oracle as mo
from mla_attention_gb300 import inputs as gen
from mla_attention_gb300 import (check_device_status, mla_decode, mla_decode_fp8, mla_prefill, mla_rope_append,
                                 mla_sparse, set_tile_keys)
from tests.helpers import assert_lse_close, assert_out_close, dev, to_np

pytestmark = [pytest.mark.gpu, pytest.mark.full]


def test_prefill_past_2_31_query_elements():
    """32768 tokens x 128 heads, causal over 32768 keys: q holds 2.4e9 elements and out 2^31."""
    T, H = 32768, 128
    d = dev()
    q = gen.randn_bf16_device((T, H, 576), 301, d)
    kv = gen.randn_bf16_device((T, 576), 302, d)
    assert q.numel() > 2 ** 31
    out, lse = mla_prefill(q, kv, gen.SCALE_192, causal=True)
    torch.cuda.synchronize()
    check_device_status()
    assert out.numel() >= 2 ** 31
    kv_h = kv.cpu()
    for t in gen.sample_rows(T, 6, seed=303, must=[0, 1, 16383, 32767]):
        ro, rl = mo.mla_prefill(q[t:t + 1].cpu(), kv_h, gen.SCALE_192, causal=True, q_pos0=t, kv_pos0=0)
        assert_out_close(out[t:t + 1], ro, what=f"out[token {t}]")
        assert_lse_close(lse[:, t:t + 1], rl, what=f"lse[token {t}]")
    del q, kv, out, lse
    torch.cuda.empty_cache()


def test_decode_128k_context():
    """One request of 131072 keys beside a short one, 64-token pages, H=128, default split."""
    D = gen.decode_inputs([131072, 300], H=128, seed=304, page_size=64)
    d = dev()
    out, lse = mla_decode(D.q.to(d), D.cache.to(d), D.block_table.to(d), D.lens.to(d), D.scale)
    torch.cuda.synchronize()
    check_device_status()
    ro, rl = mo.mla_decode(D.q, D.cache, D.block_table, D.lens, D.scale)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


BIG_PAGES = 60000          # 64-token pages: 3.84M rows, row x 576 past 2^31 (4.4 GB as bf16)
BF16_NAN_BITS = 0x7FC0     # torch's bf16 NaN
E4M3_NAN_BITS = 0x7F


def _lift_pages(D, big_pages, fill_bits, dtype, cache=None):
    """The small case's pages placed at the top of a NaN-filled cache of big_pages pages, and its
    block table moved with them."""
    d = dev()
    n = D.cache.shape[0]
    off = big_pages - n
    itype = torch.int16 if dtype == torch.bfloat16 else torch.uint8
    big = torch.full((big_pages, D.page_size, 576), fill_bits, dtype=itype, device=d).view(dtype)
    big[off:] = (D.cache if cache is None else cache).to(d)
    bt = torch.where(D.block_table >= 0, D.block_table + off, D.block_table)
    return big, bt, off


def _still_nan(big, off, fill_bits):
    """Every page below the lifted ones still holds the fill (nothing was written there)."""
    itype = torch.int16 if big.element_size() == 2 else torch.uint8
    raw = big.view(itype)
    for p0 in range(0, off, 8192):
        assert bool((raw[p0:min(off, p0 + 8192)] == fill_bits).all()), f"pages {p0}.. changed"


@pytest.fixture(params=[128, 64], ids=["decode128", "decode64"])
def decode_engine(request):
    set_tile_keys(decode_keys=request.param)
    yield request.param
    set_tile_keys(0, 0)


def test_decode_cache_past_2_31_elements(decode_engine):
    D = gen.decode_inputs([300, 4097, 65, 1000], H=128, seed=306, page_size=64)
    big, bt, off = _lift_pages(D, BIG_PAGES, BF16_NAN_BITS, torch.bfloat16)
    assert big.numel() > 2 ** 31 and off * 64 * 576 > 2 ** 31
    d = dev()
    out, lse = mla_decode(D.q.to(d), big, bt.to(d), D.lens.to(d), D.scale)
    torch.cuda.synchronize()
    check_device_status()
    ro, rl = mo.mla_decode(D.q, D.cache, D.block_table, D.lens, D.scale)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)
    del big, out, lse
    torch.cuda.empty_cache()


def test_fp8_decode_cache_past_2_31_bytes():
    """The e4m3 cache's byte offsets pass 2^31 (the producers' own loads where a half spans pages,
    16-token pages here, and the L2 prefetch)."""
    big_pages = 4 * BIG_PAGES
    D = gen.decode_inputs([300, 4097, 65, 1000], H=128, seed=307, page_size=16)
    kv_scale = 0.37
    c8 = (D.cache.float() / kv_scale).to(torch.float8_e4m3fn)
    big, bt, off = _lift_pages(D, big_pages, E4M3_NAN_BITS, torch.float8_e4m3fn, cache=c8)
    assert off * 16 * 576 > 2 ** 31
    d = dev()
    q = D.q.unsqueeze(1)  # [B, 1, H, 576]
    out, lse = mla_decode_fp8(q.to(d), big, kv_scale, bt.to(d), D.lens.to(d), D.scale)
    torch.cuda.synchronize()
    check_device_status()
    ro, rl = mo.mla_decode_fp8(q, c8, kv_scale, D.block_table, D.lens, D.scale)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)
    del big, out, lse
    torch.cuda.empty_cache()


def test_rope_append_cache_past_2_31_elements():
    """The appended rows land past element 2^31 of the cache; the cache below stays as it was."""
    lens = [0, 63, 130, 1000]
    D = gen.decode_inputs([n + 1 for n in lens], H=128, seed=308, page_size=64)
    g = torch.Generator().manual_seed(309)
    B = len(lens)
    q_pe = gen.randn_bf16((B, 128, 64), g)
    c_kv = gen.randn_bf16((B, 512), g)
    k_pe = gen.randn_bf16((B, 64), g)
    pos = torch.tensor(lens, dtype=torch.int32)
    cs = gen.rope_cos_sin(2048)
    big, bt, off = _lift_pages(D, BIG_PAGES, BF16_NAN_BITS, torch.bfloat16)
    d = dev()
    q_out = D.q.to(d).clone()
    mla_rope_append(q_pe.to(d), c_kv.to(d), k_pe.to(d), pos.to(d), cs.to(d), big, bt.to(d), q_out)
    torch.cuda.synchronize()
    check_device_status()
    q_rope, new_cache = mo.mla_rope_append(q_pe, c_kv, k_pe, pos, cs, False, D.cache, D.block_table, 64)
    got = to_np(big[off:])
    changed = np.any(new_cache != to_np(D.cache), axis=-1)
    assert int(changed.sum()) == B
    np.testing.assert_array_equal(got[~changed], to_np(D.cache)[~changed])
    np.testing.assert_array_equal(got[changed][:, :512], new_cache[changed][:, :512])
    err = np.abs(got[changed][:, 512:] - new_cache[changed][:, 512:])
    assert (err <= np.abs(new_cache[changed][:, 512:]) * 2.0 ** -8 + 1e-6).all(), "rotated k_pe"
    err = np.abs(to_np(q_out[:, :, 512:]) - q_rope)
    assert (err <= np.abs(q_rope) * 2.0 ** -8 + 1e-6).all(), "rotated q_pe"
    _still_nan(big, off, BF16_NAN_BITS)
    del big, q_out
    torch.cuda.empty_cache()


@pytest.fixture(params=[128, 64], ids=["sparse128", "sparse64"])
def sparse_engine(request):
    set_tile_keys(prefill_keys=request.param)
    yield request.param
    set_tile_keys(0, 0)


def test_sparse_rows_past_2_31_elements(sparse_engine):
    """Listed rows past element 2^31 of c_kv (row x 512) and of the 16-byte gathers' addresses."""
    S_small, S_big = 3000, 4400000
    SI = gen.sparse_inputs(40, S_small, 128, 700, 2500, seed=310)
    d = dev()
    off = S_big - S_small
    c_kv = torch.full((1, S_big, 512), BF16_NAN_BITS, dtype=torch.int16, device=d).view(torch.bfloat16)
    k_pe = torch.full((1, S_big, 64), BF16_NAN_BITS, dtype=torch.int16, device=d).view(torch.bfloat16)
    c_kv[:, off:] = SI.c_kv.to(d)
    k_pe[:, off:] = SI.k_pe.to(d)
    topk = torch.where(SI.topk >= 0, SI.topk + off, SI.topk)
    assert off * 512 > 2 ** 31
    out, lse = mla_sparse(SI.q_lift.to(d), SI.q_pe.to(d), c_kv, k_pe, topk.to(d), SI.scale)
    torch.cuda.synchronize()
    check_device_status()
    ro, rl = mo.mla_sparse(SI.q_lift, SI.q_pe, SI.c_kv, SI.k_pe, SI.topk, SI.scale)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)
    del c_kv, k_pe, out, lse
    torch.cuda.empty_cache()
