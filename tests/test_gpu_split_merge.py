"""Parity of mla_prefill_split (Ascend split layout) and mla_merge_lse with the oracle."""
import numpy as np
import pytest
import torch

import oracle.mla_oracle as mo
from mla_attention_gb300 import inputs as gen
from mla_attention_gb300 import check_device_status, mla_merge_lse, mla_prefill_split
from tests.helpers import assert_lse_close, assert_out_close, dev

pytestmark = pytest.mark.gpu


def _split(si, mask_type, with_prev=False, seq_len=None):
    d = dev()
    kw = {}
    if with_prev:
        kw = dict(prev_out=si.prev_out.to(d), prev_lse=si.prev_lse.to(d))
    out, lse = mla_prefill_split(si.q_nope.to(d), si.q_pe.to(d), si.k_nope.to(d), si.k_pe.to(d), si.v.to(d),
                                 si.seq_len if seq_len is None else seq_len, si.head_num, si.kv_head_num, si.scale,
                                 mask_type, **kw)
    torch.cuda.synchronize()
    check_device_status()
    return out, lse


@pytest.mark.parametrize("qlens,kvlens,H,Hkv,mt,prev", [
    ([5, 130, 257], [5, 130, 257], 4, 2, 1, False),
    ([5, 130, 257], [5, 130, 257], 4, 4, 1, True),
    ([64, 100], [300, 100], 8, 1, 1, True),     # q shorter than kv: bottom-right causal
    ([77, 1], [77, 129], 2, 2, 0, False),       # NO_MASK
    ([128, 256], [128, 256], 128, 128, 1, True),
])
def test_split_parity(qlens, kvlens, H, Hkv, mt, prev):
    si = gen.split_inputs(qlens, kvlens, H, Hkv, seed=sum(qlens) + H, with_prev=prev, prev_lse_range=(2.0, 5.0))
    out, lse = _split(si, mt, with_prev=prev)
    kw = dict(prev_out=si.prev_out, prev_lse=si.prev_lse) if prev else {}
    ro, rl = mo.mla_prefill_split(si.q_nope, si.q_pe, si.k_nope, si.k_pe, si.v, si.seq_len, H, Hkv, si.scale, mt,
                                  **kw)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


@pytest.mark.parametrize("scale", [-0.09, 0.0, -0.0])
def test_split_negative_and_zero_scale(scale):
    """A negative scale runs the instantiation whose row extreme is the minimum of the raw scores;
    a zero scale (either sign) gives every visible key the same weight."""
    si = gen.split_inputs([70, 200], [70, 260], 4, 2, seed=17, scale=scale, with_prev=True, prev_lse_range=(2.0, 5.0))
    out, lse = _split(si, 1, with_prev=True)
    ro, rl = mo.mla_prefill_split(si.q_nope, si.q_pe, si.k_nope, si.k_pe, si.v, si.seq_len, 4, 2, scale, 1,
                                  prev_out=si.prev_out, prev_lse=si.prev_lse)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_split_query_tiles_without_keys():
    """KV shorter than the queries under TRIU (bottom-right): the first query tiles see no key and
    keep the previous output; a sequence with no key at all keeps it entirely."""
    si = gen.split_inputs([300, 5, 130], [50, 0, 200], 4, 4, seed=23, with_prev=True, prev_lse_range=(2.0, 5.0))
    out, lse = _split(si, 1, with_prev=True)
    ro, rl = mo.mla_prefill_split(si.q_nope, si.q_pe, si.k_nope, si.k_pe, si.v, si.seq_len, 4, 4, si.scale, 1,
                                  prev_out=si.prev_out, prev_lse=si.prev_lse)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_split_many_sequences():
    """40 sequences of mixed lengths, some empty: every work item is claimed once and finds its
    sequence (the per-CTA item claiming and the sequence search over the tile offsets)."""
    g = np.random.default_rng(29)
    qlens = [int(x) for x in g.integers(0, 200, size=40)]
    qlens[3] = qlens[17] = 0
    kvlens = [q + int(x) for q, x in zip(qlens, g.integers(0, 60, size=40))]
    si = gen.split_inputs(qlens, kvlens, 2, 1, seed=31)
    out, lse = _split(si, 1)
    ro, rl = mo.mla_prefill_split(si.q_nope, si.q_pe, si.k_nope, si.k_pe, si.v, si.seq_len, 2, 1, si.scale, 1)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_split_seq_len_one_row_and_kv_head_zero():
    si = gen.split_inputs([40, 90], [40, 90], 4, 4, seed=3)
    out1, lse1 = _split(si, 1)
    si.kv_head_num = 0
    out2, lse2 = _split(si, 1, seq_len=si.seq_len[0])
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


@pytest.mark.full
def test_split_full_size_sampled():
    lens = gen.split_lens(4, 1024, 8192, seed=3)
    si = gen.split_inputs(lens, lens, 128, 128, seed=3, with_prev=True)
    out, lse = _split(si, 1, with_prev=True)
    toks = []
    off = 0
    for i, L in enumerate(lens):
        toks += [off + t for t in gen.sample_rows(L, 256, seed=30 + i, must=[0, L - 1])]
        off += L
    ro, rl = mo.mla_prefill_split(si.q_nope, si.q_pe, si.k_nope, si.k_pe, si.v, si.seq_len, 128, 128, si.scale, 1,
                                  prev_out=si.prev_out, prev_lse=si.prev_lse, tokens=toks)
    assert_out_close(out[toks], ro)
    assert_lse_close(lse[:, toks], rl)


@pytest.mark.parametrize("dv,alias", [(512, "a"), (128, "a"), (128, "b"), (8, "none")])
def test_merge_parity_and_in_place(dv, alias):
    """dv = 512 (the absorbed path), 128 (the split layout's width), 8 (the smallest allowed);
    the result written over side a, over side b, or to fresh buffers."""
    g = torch.Generator().manual_seed(8 + dv)
    rows, H = 300, 16
    oa = gen.randn_bf16((rows, H, dv), g)
    ob = gen.randn_bf16((rows, H, dv), g)
    la = torch.randn((H, rows), generator=g) * 3
    lb = torch.randn((H, rows), generator=g) * 3
    la[0, :10] = -float("inf")
    lb[0, 5:15] = -float("inf")          # rows 5..9: both sides empty
    ro, rl = mo.merge(oa.double().numpy().transpose(1, 0, 2), la.double().numpy(),
                      ob.double().numpy().transpose(1, 0, 2), lb.double().numpy())
    d = dev()
    a_o, a_l, b_o, b_l = oa.to(d), la.to(d), ob.to(d), lb.to(d)
    dst = {"a": (a_o, a_l), "b": (b_o, b_l), "none": (None, None)}[alias]
    out, lse = mla_merge_lse(a_o, a_l, b_o, b_l, out=dst[0], lse=dst[1])
    torch.cuda.synchronize()
    if alias != "none":
        assert out.data_ptr() == dst[0].data_ptr() and lse.data_ptr() == dst[1].data_ptr()
    assert_out_close(out, ro.transpose(1, 0, 2))
    assert_lse_close(lse, rl)
    assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    assert (out[5:10, 0] == 0).all() and torch.isneginf(lse[0, 5:10]).all()  # both sides empty
