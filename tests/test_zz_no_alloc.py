"""mla_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (plug-ins handed only their input and output buffers by a
framework that owns every device allocation, processes that forbid device
allocation after start-up) cannot pass mla_decode a workspace.  The no-alloc
entry point keeps the split-K scratch in a fixed device array of the library
instead.  These tests call it through the C ABI and check, on two calls in a
row with different request mixes (so stale scratch from the first call would
show), that it matches mla_decode with a workspace within the parity
tolerance, and that sizes beyond the array are refused.  This file is
collected last so that a run stopping at its first failure has run every
other test already; it also passes alone in a fresh process.
"""
import pytest
import torch

from mla_attention_gb300 import inputs as gen
from mla_attention_gb300 import MLAError, mla_decode, mla_decode_noalloc
from tests.helpers import TOL_LSE, TOL_O, assert_lse_close, assert_out_close, dev, to_np

pytestmark = pytest.mark.gpu


def _args(D):
    return (D.q.to(dev()), D.cache.to(dev()), D.block_table.to(dev()), D.lens.to(dev()), D.scale)


def test_no_alloc_matches_workspace_decode_on_two_calls():
    first = gen.decode_inputs([1, 63, 64, 65, 200, 4100], H=128, seed=91, page_size=64)
    second = gen.decode_inputs([3000, 17, 0, 129, 64], H=128, seed=92, page_size=64, extra_pages=3)
    for D in (first, second):
        a = _args(D)
        ref_out, ref_lse = mla_decode(*a)
        out, lse = mla_decode_noalloc(*a)
        torch.cuda.synchronize()
        assert_out_close(out, to_np(ref_out), tol=TOL_O)
        assert_lse_close(lse, to_np(ref_lse), tol=TOL_LSE)


def test_no_alloc_refuses_sizes_beyond_its_array():
    D = gen.decode_inputs([64, 64], H=128, seed=93, page_size=64)
    q, cache, bt, lens, scale = _args(D)
    with pytest.raises(MLAError) as e:
        mla_decode_noalloc(q, cache, bt, lens, scale, num_splits=200)   # (2 + 200) * 128 > 24576
    assert e.value.status == 1
