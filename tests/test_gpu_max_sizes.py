"""Sizes past the 32-bit element range and long contexts: every row offset, tensor-map row
coordinate and key count must be carried in 64 bits (or stay below 2^31 by construction).
Checked on sampled rows against the oracle, one query token at a time (token t is query 0 of a
one-token prefill at position t, which sees the same keys), so the host never holds the whole
query tensor."""
import pytest
import torch

import oracle.mla_oracle as mo
from mla_attention_gb300 import inputs as gen
from mla_attention_gb300 import check_device_status, mla_decode, mla_prefill
from tests.helpers import assert_lse_close, assert_out_close, dev

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
