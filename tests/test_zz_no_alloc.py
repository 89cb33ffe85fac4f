"""mla_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (plug-ins handed only their input and output buffers by a
framework that owns every device allocation, processes that forbid device
allocation after start-up) cannot pass mla_decode a workspace.  The no-alloc
entry point keeps the split-K scratch in a fixed device array of the library
instead.  These tests call it through the C ABI and check, on two calls in a
row with different request mixes (so stale scratch from the first call would
show), that it matches mla_decode with a workspace within the parity
tolerance, and the oracle; on both tile engines and several split counts; that
an out-of-range page id reads as a zero row, as in mla_decode; and that sizes
beyond the array are refused.  This file is collected last so that a run
stopping at its first failure has run every other test already; it also passes
alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle.mla_oracle as mo
from mla_attention_gb300 import inputs as gen
from mla_attention_gb300 import MLAError, check_device_status, mla_decode, mla_decode_noalloc, set_tile_keys
from tests.helpers import TOL_LSE, TOL_O, assert_lse_close, assert_out_close, dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[128, 64], ids=["keys128", "keys64"])
def engine(request):
    set_tile_keys(decode_keys=request.param)
    yield request.param
    set_tile_keys(0, 0)


def _args(D):
    return (D.q.to(dev()), D.cache.to(dev()), D.block_table.to(dev()), D.lens.to(dev()), D.scale)


@pytest.mark.parametrize("splits", [0, 3, 17])
def test_no_alloc_matches_workspace_decode_on_two_calls(engine, splits):
    first = gen.decode_inputs([1, 63, 64, 65, 200, 4100], H=128, seed=91, page_size=64)
    second = gen.decode_inputs([3000, 17, 0, 129, 64], H=128, seed=92, page_size=64, extra_pages=3)
    for D in (first, second):
        a = _args(D)
        ref_out, ref_lse = mla_decode(*a, num_splits=splits)
        out, lse = mla_decode_noalloc(*a, num_splits=splits)
        torch.cuda.synchronize()
        assert_out_close(out, to_np(ref_out), tol=TOL_O)
        assert_lse_close(lse, to_np(ref_lse), tol=TOL_LSE)
        ro, rl = mo.mla_decode(D.q, D.cache, D.block_table, D.lens, D.scale)
        assert_out_close(out, ro)
        assert_lse_close(lse, rl)
    check_device_status()


def test_no_alloc_bad_page_reads_as_zero_rows(engine):
    """A page id outside the cache is read as zero rows (score 0, value 0), as mla_decode does; the
    no-alloc call has no workspace to report it through, and the other requests are untouched."""
    D = gen.decode_inputs([300, 200, 130], H=128, seed=94, page_size=64)
    bt = D.block_table.clone()
    num_pages = D.cache.shape[0]
    bt[1, 2] = num_pages + 5                    # keys 128..191 of request 1
    out, lse = mla_decode_noalloc(D.q.to(dev()), D.cache.to(dev()), bt.to(dev()), D.lens.to(dev()), D.scale)
    torch.cuda.synchronize()
    # expected: the same page id pointing at an all-zero page
    cache0 = torch.cat([D.cache, torch.zeros((1,) + tuple(D.cache.shape[1:]), dtype=D.cache.dtype)])
    bt0 = D.block_table.clone()
    bt0[1, 2] = num_pages
    ro, rl = mo.mla_decode(D.q, cache0, bt0, D.lens, D.scale)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)
    ref_out, ref_lse = mla_decode(*_args(D))
    torch.cuda.synchronize()
    for b in (0, 2):
        np.testing.assert_array_equal(to_np(out[b]), to_np(ref_out[b]))


def test_no_alloc_refuses_sizes_beyond_its_array():
    D = gen.decode_inputs([64, 64], H=128, seed=93, page_size=64)
    q, cache, bt, lens, scale = _args(D)
    with pytest.raises(MLAError) as e:
        mla_decode_noalloc(q, cache, bt, lens, scale, num_splits=200)   # (2 + 200) * 128 > 24576
    assert e.value.status == 1
