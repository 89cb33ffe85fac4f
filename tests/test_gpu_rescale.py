"""Scores that climb along the keys by far more than the lazy-rescale threshold (2^8 in exp2
units) per key tile, so a row's running offset moves on every tile: the kernels' rescale of O
(and the 128-key engine's second pass over a tile) run on every tile instead of almost never, as
with N(0, 1) inputs.  Both signs of the scale (the extreme of the raw scores is their maximum or
their minimum).  The ramp sits in a RoPE column, outside V, so the outputs stay O(1)."""
import pytest
import torch

import oracle.mla_oracle as mo
from mla_attention_gb300 import inputs as gen
from mla_attention_gb300 import (check_device_status, mla_decode, mla_decode_ex, mla_prefill, mla_prefill_split,
                                 mla_sparse, set_tile_keys)
from tests.helpers import assert_lse_close, assert_out_close, dev

pytestmark = pytest.mark.gpu

LOG2E = 1.4426950408889634
CLIMB_PER_128_KEYS = 24.0  # exp2 units the scaled scores climb over 128 keys


def ramp(n, scale):
    """Per-key values whose scaled scores climb CLIMB_PER_128_KEYS exp2 units per 128 keys when the
    query holds +-1 in the same column (bf16, so large values come out as a staircase)."""
    slope = CLIMB_PER_128_KEYS / (128 * abs(scale) * LOG2E)
    return (torch.arange(n, dtype=torch.float64) * slope).to(torch.bfloat16)


@pytest.fixture(params=[128, 64], ids=["tile128", "tile64"])
def tile_keys(request):
    set_tile_keys(request.param, request.param)
    yield request.param
    set_tile_keys(0, 0)


@pytest.mark.parametrize("sign", [1.0, -1.0], ids=["scale+", "scale-"])
def test_prefill_climbing_scores(tile_keys, sign):
    P = gen.prefill_inputs(T=150, H=16, Tkv=900, seed=71, scale=sign * gen.SCALE_192)
    P.kv[:, 512] = ramp(900, P.scale)
    P.q[:, :, 512] = sign
    kw = dict(causal=True, q_pos0=740, kv_pos0=0)
    out, lse = mla_prefill(P.q.to(dev()), P.kv.to(dev()), P.scale, **kw)
    torch.cuda.synchronize()
    check_device_status()
    ro, rl = mo.mla_prefill(P.q, P.kv, P.scale, **kw)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_prefill_climbing_scores_with_prev(tile_keys):
    """The same climb merged with a previous result whose LSEs are of the same size, so both sides
    of the merge carry weight."""
    P = gen.prefill_inputs(T=150, H=16, Tkv=900, seed=75)
    P.kv[:, 512] = ramp(900, P.scale)
    P.q[:, :, 512] = 1.0
    po, pl = gen.prev_inputs(150, 16, 512, seed=76, lse_lo=95.0, lse_hi=125.0)
    kw = dict(causal=True, q_pos0=740, kv_pos0=0)
    out, lse = mla_prefill(P.q.to(dev()), P.kv.to(dev()), P.scale, prev_out=po.to(dev()), prev_lse=pl.to(dev()), **kw)
    torch.cuda.synchronize()
    check_device_status()
    ro, rl = mo.mla_prefill(P.q, P.kv, P.scale, prev_out=po, prev_lse=pl, **kw)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_multi_token_decode_climbing_scores_with_sinks(tile_keys):
    """Two query tokens per request (causal between them) and per-head sinks of the same size as
    the climbing scores' LSEs."""
    D = gen.decode_inputs([700, 1300, 260], H=16, seed=77, page_size=16)
    bt = D.block_table.numpy()
    for b, n in enumerate(D.lens.tolist()):
        r = ramp(n, D.scale)
        for j in range(n):
            D.cache[int(bt[b, j // D.page_size]), j % D.page_size, 512] = r[j]
    g = torch.Generator().manual_seed(78)
    q2 = gen.randn_bf16((3, 2, 16, 576), g)
    q2[..., 512] = 1.0
    sinks = (90.0 + 40.0 * torch.rand((16,), generator=g)).float()
    out, lse = mla_decode_ex(q2.to(dev()), D.cache.to(dev()), D.block_table.to(dev()), D.lens.to(dev()), D.scale,
                             sinks=sinks.to(dev()), num_splits=4)
    torch.cuda.synchronize()
    check_device_status()
    ro, rl = mo.mla_decode_ex(q2, D.cache, D.block_table, D.lens, D.scale, sinks=sinks)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


@pytest.mark.parametrize("sign", [1.0, -1.0], ids=["scale+", "scale-"])
def test_decode_climbing_scores(tile_keys, sign):
    D = gen.decode_inputs([700, 1300, 5, 260], H=16, seed=72, page_size=16, scale=sign * gen.SCALE_192)
    bt = D.block_table.numpy()
    for b, n in enumerate(D.lens.tolist()):
        r = ramp(n, D.scale)
        for j in range(n):  # logical key j of request b, wherever its page sits
            D.cache[int(bt[b, j // D.page_size]), j % D.page_size, 512] = r[j]
    D.q[:, :, 512] = sign
    out, lse = mla_decode(D.q.to(dev()), D.cache.to(dev()), D.block_table.to(dev()), D.lens.to(dev()), D.scale,
                          num_splits=5)
    torch.cuda.synchronize()
    check_device_status()
    ro, rl = mo.mla_decode(D.q, D.cache, D.block_table, D.lens, D.scale)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_sparse_climbing_scores(tile_keys):
    """mla_sparse takes a positive softmax scale only."""
    sign = 1.0
    SI = gen.sparse_inputs(60, 2000, 16, 600, 1500, seed=73, scale=gen.SCALE_192)
    SI.k_pe[0, :, 0] = ramp(2000, SI.scale)
    SI.q_pe[..., 0] = sign
    SI.topk = torch.sort(SI.topk, dim=-1).values  # listed rows in ascending order: scores climb along the list
    out, lse = mla_sparse(SI.q_lift.to(dev()), SI.q_pe.to(dev()), SI.c_kv.to(dev()), SI.k_pe.to(dev()),
                          SI.topk.to(dev()), SI.scale)
    torch.cuda.synchronize()
    check_device_status()
    ro, rl = mo.mla_sparse(SI.q_lift, SI.q_pe, SI.c_kv, SI.k_pe, SI.topk, SI.scale)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


@pytest.mark.parametrize("sign", [1.0, -1.0], ids=["scale+", "scale-"])
def test_split_climbing_scores(sign):
    lens = [700, 300]
    si = gen.split_inputs(lens, lens, 4, 2, seed=74, scale=sign * gen.SCALE_192, with_prev=True,
                          prev_lse_range=(2.0, 5.0))
    off = 0
    for n in lens:
        si.k_pe[off:off + n, :, 0] = ramp(n, si.scale)[:, None]
        off += n
    si.q_pe[:, :, 0] = sign
    out, lse = mla_prefill_split(si.q_nope.to(dev()), si.q_pe.to(dev()), si.k_nope.to(dev()), si.k_pe.to(dev()),
                                 si.v.to(dev()), si.seq_len, 4, 2, si.scale, 1, prev_out=si.prev_out.to(dev()),
                                 prev_lse=si.prev_lse.to(dev()))
    torch.cuda.synchronize()
    check_device_status()
    ro, rl = mo.mla_prefill_split(si.q_nope, si.q_pe, si.k_nope, si.k_pe, si.v, si.seq_len, 4, 2, si.scale, 1,
                                  prev_out=si.prev_out, prev_lse=si.prev_lse)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)
