"""Parity of mla_decode (paged, split-K + reduction) and mla_sparse (top-k gather) with the oracle,
plus bit-exact checks of the gathered row sets."""
import math

import numpy as np
import pytest
import torch

import oracle.mla_oracle as mo
from mla_attention_gb300 import inputs as gen
from mla_attention_gb300 import MLAError, check_device_status, mla_decode, mla_sparse, set_tile_keys
from tests.helpers import assert_lse_close, assert_out_close, dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[128, 64], ids=["tile128", "tile64"])
def tile_keys(request):
    """Both decode engines: 64-key score tiles (the default) and 128-key tiles."""
    set_tile_keys(decode_keys=request.param)
    yield request.param
    set_tile_keys(0, 0)


def _decode(D, num_splits=0):
    out, lse = mla_decode(D.q.to(dev()), D.cache.to(dev()), D.block_table.to(dev()), D.lens.to(dev()), D.scale,
                          num_splits=num_splits)
    torch.cuda.synchronize()
    check_device_status()
    return out, lse


@pytest.mark.parametrize("lens,H,page,splits", [
    ([1, 63, 64, 65, 200], 128, 64, 0),
    ([1, 63, 64, 65, 200], 128, 64, 1),
    ([300, 17, 0, 129], 16, 16, 3),        # a request with no key, 16-token pages
    ([513, 96, 33], 64, 32, 7),
    ([4096, 100, 1000], 128, 128, 0),       # 128-token pages
])
def test_decode_parity(lens, H, page, splits, tile_keys):
    D = gen.decode_inputs(lens, H=H, seed=sum(lens) + H, page_size=page, extra_pages=2)
    out, lse = _decode(D, splits)
    ro, rl = mo.mla_decode(D.q, D.cache, D.block_table, D.lens, D.scale)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_decode_row_set_is_exact(tile_keys):
    """q = 0 makes every score equal; one-hot V rows encode each cache row's id, so
    out * len must be the exact histogram of the rows the page table selects."""
    lens = [64, 128, 7, 256]
    D = gen.decode_inputs(lens, H=8, seed=5, page_size=16)
    D.q.zero_()
    rows = D.cache.shape[0] * D.cache.shape[1]
    assert rows <= 512
    flat = torch.zeros((rows, 576), dtype=torch.bfloat16)
    flat[torch.arange(rows), torch.arange(rows)] = 1.0
    D.cache = flat.view(D.cache.shape)
    out, lse = _decode(D, 2)
    o = to_np(out)
    for b, n in enumerate(lens):
        want = np.zeros(512)
        for j in range(n):
            want[int(D.block_table[b, j // 16]) * 16 + j % 16] += 1
        got = np.rint(o[b, 0] * n)
        assert (got == want).all(), f"request {b}: gathered row set differs"
        assert abs(float(lse[b, 0]) - math.log(n)) < 5e-3


@pytest.mark.parametrize("lens,bad", [([100, 50], (0, 1)),     # in a partial tile
                                      ([300, 50], (0, 2)),     # in a whole tile, mid-request
                                      ([64, 250], (1, 0))])    # first tile of a request
def test_decode_bad_page_reported(lens, bad, tile_keys):
    D = gen.decode_inputs(lens, H=16, seed=9, page_size=64)
    D.block_table[bad] = 1 << 20           # out of range
    out, lse = mla_decode(D.q.to(dev()), D.cache.to(dev()), D.block_table.to(dev()), D.lens.to(dev()), D.scale)
    torch.cuda.synchronize()
    with pytest.raises(MLAError) as e:
        check_device_status()
    assert e.value.status == 5
    check_device_status()                  # cleared after reading


@pytest.mark.full
def test_decode_full_size_all_rows():
    lens = gen.decode_lens(64, 4096, 32768, seed=4)
    D = gen.decode_inputs(lens, H=128, seed=4, page_size=64)
    out, lse = _decode(D)
    ro, rl = mo.mla_decode(D.q, D.cache, D.block_table, D.lens, D.scale)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


# ---------------------------------------------------------------------------
@pytest.fixture(params=[128, 64], ids=["sparse128", "sparse64"])
def sparse_engine(request):
    """Both tile engines for mla_sparse (it follows the prefill setting): 128-key tiles (the
    default) and 64-key tiles."""
    set_tile_keys(prefill_keys=request.param)
    yield request.param
    set_tile_keys(0, 0)


def _sparse(SI, lse=None):
    out, lse = mla_sparse(SI.q_lift.to(dev()), SI.q_pe.to(dev()), SI.c_kv.to(dev()), SI.k_pe.to(dev()),
                          SI.topk.to(dev()), SI.scale, lse=lse)
    torch.cuda.synchronize()
    check_device_status()
    return out, lse


@pytest.mark.parametrize("S,S_kv,H,K,pos0", [
    (64, 300, 16, 128, 200),
    (40, 2048, 128, 256, 1900),
    (33, 100, 128, 130, 0),        # a second tile with two listed keys
    (9, 5000, 128, 512, 4990),     # H = 128: rows staged and stored by TMA
    (21, 3000, 64, 384, 2900),     # H = 64: rows stored by the row threads
    (1, 700, 100, 200, 650),       # one token, H not a multiple of 32
    (300, 4000, 128, 256, 3900),   # several items per CTA pair (Q handed from item to item)
    (200, 1000, 16, 384, 900),
])
def test_sparse_parity(S, S_kv, H, K, pos0, sparse_engine):
    SI = gen.sparse_inputs(S, S_kv, H, K, pos0, seed=S + K)
    # plant padding and a duplicate
    SI.topk[0, 0, 5] = -1
    if S > 1:
        SI.topk[0, 1, 7] = S_kv + 5
        SI.topk[0, 2, 9] = SI.topk[0, 2, 8]
    if K >= 192 and S > 3:
        SI.topk[0, 3, 64:128] = -1         # a whole 64-key tile of padding mid-list
    if K >= 384 and S > 4:
        SI.topk[0, 4, 128:256] = -1        # a whole 128-key tile of padding mid-list
    out, lse = _sparse(SI)
    ro, rl = mo.mla_sparse(SI.q_lift, SI.q_pe, SI.c_kv, SI.k_pe, SI.topk, SI.scale)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


@pytest.mark.parametrize("H", [128, 48])
def test_sparse_without_lse(H, sparse_engine):
    """lse is optional: the output is the same without it."""
    SI = gen.sparse_inputs(12, 800, H, 256, 700, seed=77)
    out, none = _sparse(SI, lse=False)
    assert none is None
    ro, _ = mo.mla_sparse(SI.q_lift, SI.q_pe, SI.c_kv, SI.k_pe, SI.topk, SI.scale)
    assert_out_close(out, ro)


def test_sparse_row_set_is_exact(sparse_engine):
    S, S_kv, H, K = 16, 512, 4, 128
    SI = gen.sparse_inputs(S, S_kv, H, K, pos0=S_kv - S, seed=11)
    SI.topk[0, 3, 10:20] = -1
    SI.topk[0, 4, 0] = SI.topk[0, 4, 1]
    SI.q_lift.zero_()
    SI.q_pe.zero_()
    c = torch.zeros((1, S_kv, 512), dtype=torch.bfloat16)
    c[0, torch.arange(S_kv), torch.arange(S_kv)] = 1.0
    SI.c_kv = c
    out, lse = _sparse(SI)
    o = to_np(out).reshape(S, H, 512)
    for s in range(S):
        idx = SI.topk[0, s]
        idx = idx[(idx >= 0) & (idx < S_kv)]
        want = np.bincount(idx.numpy(), minlength=512).astype(float)
        n = len(idx)
        got = np.rint(o[s, 1] * n)
        assert (got == want).all(), f"token {s}: gathered row multiset differs"
        assert abs(float(lse[0, s, 1]) - math.log(n)) < 5e-3


def test_sparse_all_padding_row(sparse_engine):
    SI = gen.sparse_inputs(4, 64, 16, 64, pos0=60, seed=12)
    SI.topk[0, 2, :] = -1
    out, lse = _sparse(SI)
    assert torch.all(out[0, 2] == 0)
    assert torch.all(torch.isneginf(lse[0, 2]))


@pytest.mark.full
def test_sparse_full_size_sampled():
    SI = gen.sparse_inputs(4096, 32768, 128, 2048, pos0=28672, seed=5)
    out, lse = _sparse(SI)
    toks = gen.sample_rows(4096, 256, seed=5, must=[0, 4095])
    ro, rl = mo.mla_sparse(SI.q_lift, SI.q_pe, SI.c_kv, SI.k_pe, SI.topk, SI.scale, tokens=toks)
    assert_out_close(out[0, toks], ro[0])
    assert_lse_close(lse[0, toks], rl[0])
