"""The decode step around the latent attention: RoPE and the paged latent-cache append
(mla_rope_append), against the oracle, alone and followed by mla_decode."""
import numpy as np
import pytest
import torch

import oracle.mla_oracle as mo
from mla_attention_gb300 import inputs as gen
from mla_attention_gb300 import MLAError, check_device_status, mla_decode, mla_rope_append
from tests.helpers import assert_lse_close, assert_out_close, dev, to_np

pytestmark = pytest.mark.gpu


def _bf16_close(gpu, ref, what):
    """Rotations are computed in fp32 and stored as bf16: within half a bf16 step of the exact value."""
    g = to_np(gpu)
    r = np.asarray(ref)
    err = np.abs(g - r)
    bound = np.abs(r) * 2.0 ** -8 + 1e-6
    assert (err <= bound).all(), f"{what}: worst excess {float((err - bound).max()):.3e}"


def _step_inputs(lens, H, seed, page_size=64):
    """A cache with room for one more row per request; the new token goes to row lens[b]."""
    D = gen.decode_inputs([n + 1 for n in lens], H=H, seed=seed, page_size=page_size)
    g = torch.Generator().manual_seed(seed + 1000)
    B = len(lens)
    q_pe = gen.randn_bf16((B, H, 64), g)
    c_kv = gen.randn_bf16((B, 512), g)
    k_pe = gen.randn_bf16((B, 64), g)
    pos = torch.tensor(lens, dtype=torch.int32)
    return D, q_pe, c_kv, k_pe, pos


@pytest.mark.parametrize("neox", [False, True], ids=["interleaved", "halves"])
@pytest.mark.parametrize("page_size", [64, 16])
def test_rope_append_parity(neox, page_size):
    lens = [0, 10, 63, 64, 130, 301]
    D, q_pe, c_kv, k_pe, pos = _step_inputs(lens, H=128, seed=31, page_size=page_size)
    cs = gen.rope_cos_sin(512)
    d = dev()
    cache = D.cache.to(d)
    q_out = D.q.to(d).clone()
    mla_rope_append(q_pe.to(d), c_kv.to(d), k_pe.to(d), pos.to(d), cs.to(d), cache, D.block_table.to(d), q_out,
                    is_neox=neox)
    torch.cuda.synchronize()
    check_device_status()
    q_rope, new_cache = mo.mla_rope_append(q_pe, c_kv, k_pe, pos, cs, neox, D.cache, D.block_table, page_size)
    _bf16_close(q_out[:, :, 512:], q_rope, "rotated q_pe")
    np.testing.assert_array_equal(to_np(q_out[:, :, :512]), to_np(D.q[:, :, :512]))   # latent part untouched
    got = to_np(cache)
    changed = np.any(new_cache != to_np(D.cache), axis=-1)
    np.testing.assert_array_equal(got[~changed], to_np(D.cache)[~changed])           # every other row untouched
    np.testing.assert_array_equal(got[changed][:, :512], new_cache[changed][:, :512])  # c_kv copied exactly
    _bf16_close(cache.view(-1, 576)[torch.from_numpy(changed.reshape(-1)).to(d)][:, 512:],
                new_cache[changed][:, 512:], "rotated k_pe")


def test_decode_step_rope_append_then_attention():
    """One full decode step: the latent query part (given), RoPE + append, then attention over
    len + 1 keys; the oracle runs the same two steps."""
    lens = [5, 200, 64, 1000]
    D, q_pe, c_kv, k_pe, pos = _step_inputs(lens, H=128, seed=32)
    cs = gen.rope_cos_sin(2048, base=50000.0)
    d = dev()
    cache = D.cache.to(d)
    q = D.q.to(d).clone()
    bt = D.block_table.to(d)
    mla_rope_append(q_pe.to(d), c_kv.to(d), k_pe.to(d), pos.to(d), cs.to(d), cache, bt, q)
    out, lse = mla_decode(q, cache, bt, (pos + 1).to(d), D.scale)
    torch.cuda.synchronize()
    check_device_status()
    q_rope, new_cache = mo.mla_rope_append(q_pe, c_kv, k_pe, pos, cs, False, D.cache, D.block_table, 64)
    # the attention reads the query the GPU formed (bf16 rotated q_pe); the oracle forms the same
    q_ref = to_np(q)
    ro, rl = mo.mla_decode(q_ref, to_np(cache), D.block_table, pos + 1, D.scale)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)
    _bf16_close(q[:, :, 512:], q_rope, "rotated q_pe")
    ro2, rl2 = mo.mla_decode(np.concatenate([to_np(D.q[:, :, :512]), q_rope], -1), new_cache, D.block_table,
                             pos + 1, D.scale)
    assert_out_close(out, ro2)
    assert_lse_close(lse, rl2)


def test_rope_append_out_of_range_position_is_reported_and_skipped():
    lens = [10, 20]
    D, q_pe, c_kv, k_pe, pos = _step_inputs(lens, H=16, seed=33)
    pos[1] = 5000                                   # past this request's pages
    d = dev()
    cache = D.cache.to(d)
    q_out = D.q.to(d).clone()
    mla_rope_append(q_pe.to(d), c_kv.to(d), k_pe.to(d), pos.to(d), gen.rope_cos_sin(8192).to(d), cache,
                    D.block_table.to(d), q_out)
    with pytest.raises(MLAError) as e:
        check_device_status()
    assert e.value.status == 5
    np.testing.assert_array_equal(to_np(q_out[1]), to_np(D.q[1]))    # request 1 untouched
    assert not torch.equal(q_out[0].cpu(), D.q[0])                   # request 0 done


# ---------------------------------------------------------------------------
# the absorption BMMs
# ---------------------------------------------------------------------------
def _gemm_close(gpu, ref, what, k):
    """bf16 result of a K-term fp32 dot product: half a bf16 step of the value plus the fp32
    accumulation error, bounded by k * 2^-22 times the magnitude of the terms (taken as 4)."""
    g = to_np(gpu)
    r = np.asarray(ref)
    err = np.abs(g - r)
    bound = np.abs(r) * 2.0 ** -8 + k * 2.0 ** -22 * 4 + 1e-6
    assert (err <= bound).all(), f"{what}: worst excess {float((err - bound).max()):.3e}"


@pytest.mark.parametrize("T,H", [(300, 16), (128, 128), (1, 3), (2048, 32)])   # the last: several items per CTA
def test_absorb_q_parity_strided_input(T, H):
    from mla_attention_gb300 import mla_absorb_q
    g = torch.Generator().manual_seed(40 + T)
    q = gen.randn_bf16((T, H, 192), g)             # projection output: 128 nope + 64 rope per head
    wk, _ = gen.absorb_weights(H, seed=41)
    d = dev()
    qd = q.to(d)
    fused = torch.full((T, H, 576), 7.0, dtype=torch.bfloat16, device=d)
    mla_absorb_q(qd[:, :, :128], wk.to(d), q_out=fused)
    torch.cuda.synchronize()
    check_device_status()
    _gemm_close(fused[:, :, :512], mo.absorb_q(q[:, :, :128], wk), "q_lift", 128)
    assert (fused[:, :, 512:] == 7.0).all()       # the RoPE columns are not written


@pytest.mark.parametrize("T,H", [(300, 16), (129, 128), (1500, 64)])
def test_project_out_parity(T, H):
    from mla_attention_gb300 import mla_project_out
    g = torch.Generator().manual_seed(50 + T)
    o = gen.randn_bf16((T, H, 512), g)
    _, wv = gen.absorb_weights(H, seed=51)
    d = dev()
    out = mla_project_out(o.to(d), wv.to(d))
    torch.cuda.synchronize()
    check_device_status()
    _gemm_close(out, mo.project_out(o, wv), "projected out", 512)


@pytest.mark.full
def test_absorption_bmms_full_size_sampled_tokens():
    """Both BMMs at the measured size (T = 8192 tokens, H = 128): every token is its own
    per-head product, so sampled tokens against the oracle check the whole launch's indexing
    (the q side reads a strided [T, H, 128] view of a [T, H, 192] projection)."""
    from mla_attention_gb300 import mla_absorb_q, mla_project_out
    T, H = 8192, 128
    d = dev()
    q = gen.randn_bf16_device((T, H, 192), 311, d)
    o = gen.randn_bf16_device((T, H, 512), 312, d)
    wk, wv = gen.absorb_weights(H, seed=313)
    fused = torch.full((T, H, 576), 7.0, dtype=torch.bfloat16, device=d)
    mla_absorb_q(q[:, :, :128], wk.to(d), q_out=fused)
    out = mla_project_out(o, wv.to(d))
    torch.cuda.synchronize()
    check_device_status()
    for t in gen.sample_rows(T, 8, seed=314, must=[0, 127, 128, T - 1]):
        _gemm_close(fused[t:t + 1, :, :512], mo.absorb_q(q[t:t + 1, :, :128].cpu(), wk), f"q_lift[{t}]", 128)
        _gemm_close(out[t:t + 1], mo.project_out(o[t:t + 1].cpu(), wv), f"projected out[{t}]", 512)
    assert bool((fused[:, :, 512:] == 7.0).all())
    del q, o, fused, out
    torch.cuda.empty_cache()


def test_absorbed_chain_equals_non_absorbed_attention():
    """q_nope -> q_lift (tensor cores) -> latent causal attention over [c_kv | k_pe] -> O x v_b_proj^T
    equals, within the parity tolerance, per-head attention over the explicitly up-projected
    k_nope = c W_k[h] and v = c W_v[h]^T (the oracle's non-absorbed form)."""
    from mla_attention_gb300 import mla_absorb_q, mla_prefill, mla_project_out
    T, H = 256, 16
    g = torch.Generator().manual_seed(60)
    q_nope = gen.randn_bf16((T, H, 128), g)
    q_pe = gen.randn_bf16((T, H, 64), g)
    c = gen.randn_bf16((T, 512), g)
    k_pe = gen.randn_bf16((T, 64), g)
    wk, wv = gen.absorb_weights(H, seed=61)
    scale = gen.SCALE_192
    d = dev()
    q = torch.empty((T, H, 576), dtype=torch.bfloat16, device=d)
    q[:, :, 512:] = q_pe.to(d)
    mla_absorb_q(q_nope.to(d), wk.to(d), q_out=q)
    kv = torch.cat([c, k_pe], 1).to(d)
    o_lat, lse = mla_prefill(q, kv, scale, causal=True)
    out = mla_project_out(o_lat, wv.to(d))
    torch.cuda.synchronize()
    check_device_status()
    # (1) the chain with the method's bf16 storage points: the fused query and the latent output are
    #     bf16 tensors (TensorRT-LLM allocates fused_q with q's dtype), so the oracle rounds there too
    bf = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()  # noqa: E731
    q_ref = np.concatenate([bf(mo.absorb_q(q_nope, wk)), q_pe.double().numpy()], -1)
    kv_ref = np.concatenate([c.double().numpy(), k_pe.double().numpy()], 1)
    o_ref, l_ref = mo.mla_prefill(q_ref, kv_ref, scale, causal=True)
    assert_out_close(o_lat, o_ref)
    assert_lse_close(lse, l_ref)
    assert_out_close(out, mo.project_out(bf(o_ref), wv))
    # (2) absorbed = non-absorbed: per-head attention over k_nope = c W_k[h], v = c W_v[h]^T.  The
    #     bf16 fused query moves each score by about scale * 2^-9 * sqrt(512) ~ 3e-3, so the LSE
    #     bound here is 1e-2; the output bound is the usual one.
    W_k = wk.double().numpy()
    W_v = wv.double().numpy()
    cd = c.double().numpy()
    k_nope = np.stack([cd @ W_k[h] for h in range(H)], 1)           # [T, H, 128]
    v = np.stack([cd @ W_v[h].T for h in range(H)], 1)              # [T, H, 128]
    k_pe_h = np.repeat(k_pe.double().numpy()[:, None, :], H, 1)
    ro, rl = mo.mla_prefill_split(q_nope, q_pe, k_nope, k_pe_h, v, [T], H, H, scale, 1)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl, tol=1e-2)


# ---------------------------------------------------------------------------
# several query tokens per request, attention sinks
# ---------------------------------------------------------------------------
@pytest.fixture(params=[128, 64], ids=["keys128", "keys64"])
def decode_engine(request):
    from mla_attention_gb300 import set_tile_keys
    set_tile_keys(decode_keys=request.param)
    yield request.param
    set_tile_keys(0, 0)


@pytest.mark.parametrize("S,H,sinks,splits", [(2, 128, False, 0), (4, 16, True, 0), (3, 128, True, 7),
                                              (1, 64, True, 0)])
def test_multi_token_decode_with_sinks(decode_engine, S, H, sinks, splits):
    from mla_attention_gb300 import mla_decode_ex
    lens = [1, 3, 64, 129, 700, 2]                     # tokens of the short requests see few or no keys
    D = gen.decode_inputs(lens, H=H, seed=70 + S, page_size=64)
    g = torch.Generator().manual_seed(71 + S)
    q = gen.randn_bf16((len(lens), S, H, 576), g)
    sk = (torch.randn((H,), generator=g) * 2.0).float() if sinks else None
    d = dev()
    out, lse = mla_decode_ex(q.to(d), D.cache.to(d), D.block_table.to(d), D.lens.to(d), D.scale,
                             sinks=None if sk is None else sk.to(d), num_splits=splits)
    torch.cuda.synchronize()
    check_device_status()
    ro, rl = mo.mla_decode_ex(q, D.cache, D.block_table, D.lens, D.scale, sinks=sk)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


# ---------------------------------------------------------------------------
# FP8 (e4m3) latent cache
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("lens,S,H,page_size,splits,sinks", [
    ([1, 63, 64, 65, 200, 4100], 1, 128, 64, 0, False),
    ([3000, 17, 0, 129, 64], 2, 16, 64, 7, True),
    ([70, 5, 130, 300], 1, 128, 16, 0, False),
    ([300, 129, 1000, 64], 1, 128, 128, 0, False),   # 128-token pages: halves at offsets 0 and 64 of a page
])
def test_fp8_cache_decode(lens, S, H, page_size, splits, sinks):
    from mla_attention_gb300 import mla_decode_fp8
    D = gen.decode_inputs(lens, H=H, seed=80 + S, page_size=page_size)
    kv_scale = 0.37
    c8 = (D.cache.float() / kv_scale).to(torch.float8_e4m3fn)      # the caller's quantised cache
    g = torch.Generator().manual_seed(81)
    q = gen.randn_bf16((len(lens), S, H, 576), g)
    sk = (torch.randn((H,), generator=g) * 2.0).float() if sinks else None
    d = dev()
    out, lse = mla_decode_fp8(q.to(d), c8.to(d), kv_scale, D.block_table.to(d), D.lens.to(d), D.scale,
                              sinks=None if sk is None else sk.to(d), num_splits=splits)
    torch.cuda.synchronize()
    check_device_status()
    ro, rl = mo.mla_decode_fp8(q, c8, kv_scale, D.block_table, D.lens, D.scale, sinks=sk)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_fp8_cache_row_set_is_exact():
    """q = 0 makes every score equal; one-hot e4m3 value rows then give out = (keys' one-hots) / n,
    so a wrong or missed row shows up exactly."""
    from mla_attention_gb300 import mla_decode_fp8
    lens = [5, 64, 129, 300]
    D = gen.decode_inputs(lens, H=16, seed=85, page_size=64)
    pages = D.cache.shape[0]
    cache = torch.zeros((pages, 64, 576))
    ids = torch.arange(pages * 64)
    cache.view(-1, 576)[ids, ids % 512] = 1.0                      # row i holds a one at column i % 512
    c8 = cache.to(torch.float8_e4m3fn)
    q = torch.zeros((len(lens), 16, 576), dtype=torch.bfloat16)
    d = dev()
    out, _ = mla_decode_fp8(q.to(d), c8.to(d), 1.0, D.block_table.to(d), D.lens.to(d), D.scale)
    torch.cuda.synchronize()
    check_device_status()
    for b, n in enumerate(lens):
        want = torch.zeros(512, dtype=torch.float64)
        for j in range(n):
            row = int(D.block_table[b, j // 64]) * 64 + j % 64
            want[row % 512] += 1.0 / n
        np.testing.assert_allclose(to_np(out[b, 0]), want.numpy(), atol=2.0 ** -8)


@pytest.mark.full
@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "e4m3"])
def test_decode_step_variants_full_size_sampled_requests(fp8):
    """The measured decode-step variants at full size (B = 64, H = 128, lens U[4096, 32768],
    64-token pages): bf16 with two query tokens per request and per-head sinks, and the e4m3
    cache with one.  The GPU runs every request; the oracle checks 12 sampled ones (each
    request's rows depend only on its own keys)."""
    from mla_attention_gb300 import mla_decode_ex, mla_decode_fp8
    lens = gen.decode_lens(64, 4096, 32768, seed=4)
    D = gen.decode_inputs(lens, H=128, seed=315, page_size=64)
    g = torch.Generator().manual_seed(316)
    S = 1 if fp8 else 2
    q = gen.randn_bf16((64, S, 128, 576), g)
    d = dev()
    if fp8:
        kv_scale = 0.05
        c8 = (D.cache.float() / kv_scale).to(torch.float8_e4m3fn)
        out, lse = mla_decode_fp8(q.to(d), c8.to(d), kv_scale, D.block_table.to(d), D.lens.to(d), D.scale)
    else:
        sinks = (torch.randn((128,), generator=g) * 2.0).float()
        out, lse = mla_decode_ex(q.to(d), D.cache.to(d), D.block_table.to(d), D.lens.to(d), D.scale,
                                 sinks=sinks.to(d))
    torch.cuda.synchronize()
    check_device_status()
    reqs = gen.sample_rows(64, 12, seed=317, must=[0, 63, int(np.argmax(lens)), int(np.argmin(lens))])
    bt, ln = D.block_table[reqs], D.lens[reqs]
    if fp8:
        ro, rl = mo.mla_decode_fp8(q[reqs], c8, kv_scale, bt, ln, D.scale)
    else:
        ro, rl = mo.mla_decode_ex(q[reqs], D.cache, bt, ln, D.scale, sinks=sinks)
    assert_out_close(out[reqs], ro)
    assert_lse_close(lse[reqs], rl)
