"""Failure detection without a GPU fault.  A wait that cannot finish (a barrier that
nothing arrives on, switched on from the host) runs out of its bound; the kernel
records MLA_ERR_TIMEOUT, drains and exits; the context stays usable afterwards."""
import pytest
import torch

from mla_attention_gb300 import inputs as gen
from mla_attention_gb300 import (MLAError, check_device_status, inject_stall, mla_decode, mla_prefill,
                                 mla_prefill_split, mla_sparse, set_spin_limit, set_tile_keys)
from tests.helpers import dev

pytestmark = pytest.mark.gpu


def _expect_timeout(run):
    check_device_status()
    set_spin_limit(4096)
    inject_stall(True)
    try:
        run()
        torch.cuda.synchronize()
    finally:
        inject_stall(False)
        set_spin_limit(0)
    with pytest.raises(MLAError) as e:
        check_device_status()
    assert e.value.status == 4
    check_device_status()   # the word was cleared


@pytest.fixture(params=[128, 64], ids=["keys128", "keys64"])
def engine(request):
    """Both tile engines (prefill, decode and sparse): the abort path of each instantiation is driven."""
    set_tile_keys(request.param, request.param)
    yield request.param
    set_tile_keys(0, 0)


def test_prefill_timeout_and_context_survives(engine):
    P = gen.prefill_inputs(T=64, H=128, Tkv=256, seed=1)
    q, kv = P.q.to(dev()), P.kv.to(dev())
    _expect_timeout(lambda: mla_prefill(q, kv, P.scale, q_pos0=192))
    out, lse = mla_prefill(q, kv, P.scale, q_pos0=192)
    torch.cuda.synchronize()
    check_device_status()
    assert torch.isfinite(out.float()).all()


def test_split_kernel_timeout():
    si = gen.split_inputs([300], [300], 2, 2, seed=2)
    d = dev()
    args = [si.q_nope.to(d), si.q_pe.to(d), si.k_nope.to(d), si.k_pe.to(d), si.v.to(d), si.seq_len, 2, 2, si.scale, 1]
    _expect_timeout(lambda: mla_prefill_split(*args))
    mla_prefill_split(*args)
    torch.cuda.synchronize()
    check_device_status()


def test_decode_timeout(engine):
    D = gen.decode_inputs([200, 70], H=16, seed=3)
    a = [D.q.to(dev()), D.cache.to(dev()), D.block_table.to(dev()), D.lens.to(dev()), D.scale]
    _expect_timeout(lambda: mla_decode(*a))
    out, lse = mla_decode(*a)
    torch.cuda.synchronize()
    check_device_status()
    assert torch.isfinite(out.float()).all()


def test_sparse_timeout(engine):
    S = gen.sparse_inputs(S=8, S_kv=300, H=16, K=128, pos0=200, seed=4)
    d = dev()
    a = [S.q_lift.to(d), S.q_pe.to(d), S.c_kv.to(d), S.k_pe.to(d), S.topk.to(d), S.scale]
    _expect_timeout(lambda: mla_sparse(*a))
    out, lse = mla_sparse(*a)
    torch.cuda.synchronize()
    check_device_status()
    assert torch.isfinite(out.float()).all()
