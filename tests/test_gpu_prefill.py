"""Parity of mla_prefill (absorbed causal MLA, CUDA path through the C ABI) with the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle.mla_oracle as mo
from mla_attention_gb300 import inputs as gen
from mla_attention_gb300 import check_device_status, mla_prefill, set_tile_keys
from tests.helpers import assert_lse_close, assert_out_close, dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[128, 64], ids=["tile128", "tile64"])
def tile_keys(request):
    """Both prefill kernels: 128-key score tiles (the default) and 64-key tiles."""
    set_tile_keys(prefill_keys=request.param)
    yield request.param
    set_tile_keys(0, 0)


def _run(P, **kw):
    q = P.q.to(dev())
    kv = P.kv.to(dev())
    out, lse = mla_prefill(q, kv, P.scale, **kw)
    torch.cuda.synchronize()
    check_device_status()
    return out, lse


def test_tiny_config_full_parity(tile_keys):
    """B=1, H=16, T=Tkv=256 causal, every row (rows pack 8 tokens x 16 heads per tile)."""
    P = gen.prefill_inputs(T=256, H=16, Tkv=256, seed=1)
    out, lse = _run(P)
    ro, rl = mo.mla_prefill(P.q, P.kv, P.scale, causal=True)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


@pytest.mark.parametrize("T,H,Tkv,q_pos0,kv_pos0,kv_valid,causal", [
    (100, 7, 77, 50, 20, 70, True),       # ragged rows/tiles, padded chunk, offsets
    (37, 128, 200, 0, 10, 200, True),     # tokens 0..9 see no key: O = 0, lse = -inf
    (64, 3, 130, 0, 0, 130, False),       # FULL mask (a cached chunk)
    (5, 128, 1, 0, 0, 1, True),           # a single key
    (130, 128, 64, 1000, 0, 64, True),    # every token sees the whole chunk
])
def test_ragged_and_edge_cases(T, H, Tkv, q_pos0, kv_pos0, kv_valid, causal, tile_keys):
    P = gen.prefill_inputs(T=T, H=H, Tkv=Tkv, seed=T + H)
    out, lse = _run(P, causal=causal, q_pos0=q_pos0, kv_pos0=kv_pos0, kv_valid=kv_valid)
    ro, rl = mo.mla_prefill(P.q, P.kv, P.scale, causal=causal, q_pos0=q_pos0, kv_pos0=kv_pos0, kv_valid=kv_valid)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_empty_rows_are_zero_and_neg_inf(tile_keys):
    P = gen.prefill_inputs(T=20, H=16, Tkv=64, seed=3)
    out, lse = _run(P, q_pos0=0, kv_pos0=100)   # no token reaches the chunk
    assert torch.all(out == 0)
    assert torch.all(torch.isneginf(lse))


def test_prev_merge_and_in_place(tile_keys):
    T, H = 96, 128
    P = gen.prefill_inputs(T=T, H=H, Tkv=96, seed=4)
    prev_out, prev_lse = gen.prev_inputs(T, H, 512, seed=44, lse_lo=1.0, lse_hi=6.0)
    prev_lse[:, :5] = -float("inf")           # rows with an empty previous part
    ro, rl = mo.mla_prefill(P.q, P.kv, P.scale, causal=True, q_pos0=40, kv_pos0=0, prev_out=prev_out,
                            prev_lse=prev_lse)
    po = prev_out.to(dev())
    pl = prev_lse.to(dev())
    out, lse = _run(P, q_pos0=40, kv_pos0=0, prev_out=po, prev_lse=pl, out=po, lse=pl)   # in place
    assert out.data_ptr() == po.data_ptr()
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_chunked_ring_equals_one_pass(tile_keys):
    """4 KV chunks in sequence, each merged in place into (out, lse), equal one causal pass."""
    T, H, C = 512, 128, 128
    P = gen.prefill_inputs(T=T, H=H, Tkv=T, seed=2)
    q = P.q.to(dev())
    kv = P.kv.to(dev())
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev())
    lse = torch.empty((H, T), dtype=torch.float32, device=dev())
    for j in range(T // C):
        prev = (out, lse) if j > 0 else (None, None)
        mla_prefill(q, kv[j * C:(j + 1) * C], P.scale, causal=True, q_pos0=0, kv_pos0=j * C,
                    prev_out=prev[0], prev_lse=prev[1], out=out, lse=lse)
    torch.cuda.synchronize()
    check_device_status()
    toks = gen.sample_rows(T, 96, seed=7, must=[0, 127, 128, 255, 256, 383, 384, 511])
    ro, rl = mo.mla_prefill(P.q, P.kv, P.scale, causal=True, tokens=toks)
    assert_out_close(out[toks], ro)
    assert_lse_close(lse[:, toks], rl)


def test_strided_q(tile_keys):
    T, H = 40, 16
    P = gen.prefill_inputs(T=T, H=H, Tkv=50, seed=6)
    big = torch.zeros((T, H, 640), dtype=torch.bfloat16)
    big[:, :, :576] = P.q
    qv = big.to(dev())[:, :, :576]
    out, lse = mla_prefill(qv, P.kv.to(dev()), P.scale, causal=True, q_pos0=10)
    torch.cuda.synchronize()
    ro, rl = mo.mla_prefill(P.q, P.kv, P.scale, causal=True, q_pos0=10)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


@pytest.mark.full
def test_full_size_chunked_config_sampled():
    """H=128, 8192 tokens, 4 chunks of 2048 keys in sequence with prev merge in place;
    256 sampled tokens x all heads (every chunk boundary included) against the oracle."""
    T, H, C = 8192, 128, 2048
    P = gen.prefill_inputs(T=T, H=H, Tkv=T, seed=2)
    q = P.q.to(dev())
    kv = P.kv.to(dev())
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev())
    lse = torch.empty((H, T), dtype=torch.float32, device=dev())
    for j in range(4):
        prev = (out, lse) if j > 0 else (None, None)
        mla_prefill(q, kv[j * C:(j + 1) * C], P.scale, causal=True, q_pos0=0, kv_pos0=j * C,
                    prev_out=prev[0], prev_lse=prev[1], out=out, lse=lse)
    torch.cuda.synchronize()
    check_device_status()
    toks = gen.sample_rows(T, 256, seed=2, must=[0, 2047, 2048, 4095, 4096, 6143, 6144, 8191])
    ro, rl = mo.mla_prefill(P.q, P.kv, P.scale, causal=True, tokens=toks)
    assert_out_close(out[toks], ro)
    assert_lse_close(lse[:, toks], rl)


@pytest.mark.parametrize("scale_mul", [-1.0, 0.0])
def test_negative_and_zero_scale(scale_mul, tile_keys):
    """A negative scale makes the row extreme the smallest raw score; a zero scale gives
    every visible key the same weight (the mean of V)."""
    P = gen.prefill_inputs(T=100, H=16, Tkv=150, seed=9)
    scale = P.scale * scale_mul
    out, lse = mla_prefill(P.q.to(dev()), P.kv.to(dev()), scale, causal=True, q_pos0=40)
    torch.cuda.synchronize()
    check_device_status()
    ro, rl = mo.mla_prefill(P.q, P.kv, scale, causal=True, q_pos0=40)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


@pytest.mark.parametrize("H", [128, 16])
def test_varlen_batch_with_prev_and_empty_sequences(tile_keys, H):
    """Four packed sequences of unequal lengths (one with no query, one with a cached prefix longer
    than its queries, one with no key), causal, merged in place with a previous pair; each
    sequence against the oracle's single-sequence prefill with its bottom-right alignment."""
    from mla_attention_gb300 import mla_prefill_varlen
    q_lens = [70, 0, 33, 200, 5]
    kv_lens = [70, 10, 150, 200, 0]
    g = torch.Generator().manual_seed(90 + H)
    Tq, Tk = sum(q_lens), sum(kv_lens)
    q = gen.randn_bf16((Tq, H, 576), g)
    kv = gen.randn_bf16((Tk, 576), g)
    prev_out, prev_lse = gen.prev_inputs(Tq, H, 512, seed=91, lse_lo=1.0, lse_hi=6.0)
    prev_lse[:, :3] = -float("inf")
    cq = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(kv_lens)]).astype(np.int32)
    d = dev()
    po, pl = prev_out.to(d), prev_lse.to(d)
    out, lse = mla_prefill_varlen(q.to(d), kv.to(d), cq, ck, gen.SCALE_192, causal=True, prev_out=po, prev_lse=pl,
                                  out=po, lse=pl)
    torch.cuda.synchronize()
    check_device_status()
    for b in range(len(q_lens)):
        if q_lens[b] == 0:
            continue
        qs, ks = slice(cq[b], cq[b + 1]), slice(ck[b], ck[b + 1])
        ro, rl = mo.mla_prefill(q[qs], kv[ks], gen.SCALE_192, causal=True, q_pos0=kv_lens[b] - q_lens[b], kv_pos0=0,
                                prev_out=prev_out[qs], prev_lse=prev_lse[:, qs])
        assert_out_close(out[qs], ro, what=f"out of sequence {b}")
        assert_lse_close(lse[:, qs], rl, what=f"lse of sequence {b}")
