"""Failure detection without a GPU fault: a bound on every device wait turns a wait that
cannot finish into MLA_ERR_TIMEOUT, and the context stays usable afterwards."""
import pytest
import torch

from mla_attention_gb300 import inputs as gen
from mla_attention_gb300 import MLAError, check_device_status, mla_prefill, mla_prefill_split, set_spin_limit
from tests.helpers import dev

pytestmark = pytest.mark.gpu


def test_wait_bound_reports_timeout_and_context_survives():
    P = gen.prefill_inputs(T=64, H=128, Tkv=256, seed=1)
    q, kv = P.q.to(dev()), P.kv.to(dev())
    check_device_status()
    set_spin_limit(1)
    try:
        mla_prefill(q, kv, P.scale, q_pos0=192)
        torch.cuda.synchronize()
    finally:
        set_spin_limit(0)
    with pytest.raises(MLAError) as e:
        check_device_status()
    assert e.value.status == 4
    # the same call with the default bound succeeds on the same context
    out, lse = mla_prefill(q, kv, P.scale, q_pos0=192)
    torch.cuda.synchronize()
    check_device_status()
    assert torch.isfinite(out.float()).all()


def test_split_wait_bound_reports_timeout():
    si = gen.split_inputs([300], [300], 2, 2, seed=2)
    d = dev()
    set_spin_limit(1)
    try:
        mla_prefill_split(si.q_nope.to(d), si.q_pe.to(d), si.k_nope.to(d), si.k_pe.to(d), si.v.to(d), si.seq_len,
                          2, 2, si.scale, 1)
        torch.cuda.synchronize()
    finally:
        set_spin_limit(0)
    with pytest.raises(MLAError) as e:
        check_device_status()
    assert e.value.status == 4
