"""Pins of the fp64 oracle to things other than itself (CPU only).

Each check ties an oracle function to something it does not compute itself:
hand-derived closed forms (tests/golden/closed_form_cases.json), a
pure-Python scalar brute force written independently here, a library routine
(torch scaled_dot_product_attention in fp64), and identities of the
mathematics that the pages state (chunked prefill merged by LSE equals one
pass; sparse attention over the full causal prefix equals dense causal
attention; decode equals the last row of causal prefill; absorbed equals
non-absorbed attention).  test_oracle_mutations.py plants mistakes in the
oracle and checks that these pins catch each one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.mla_oracle as mo
from mla_attention_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")


def _num(x):
    return -math.inf if x == "-inf" else x


# ---------------------------------------------------------------------------
# independent scalar brute force (pure Python loops; no numpy arithmetic)
# ---------------------------------------------------------------------------
def brute_attend(q, keys, vals, scale):
    """One query row against a list of keys, in plain Python floats."""
    if len(keys) == 0:
        return [0.0] * (len(vals[0]) if vals else 0), -math.inf
    scores = []
    for k in keys:
        acc = 0.0
        for a, b in zip(q, k):
            acc += a * b
        scores.append(scale * acc)
    top = max(scores)
    ws = [math.exp(s - top) for s in scores]
    tot = sum(ws)
    dv = len(vals[0])
    out = [sum(ws[j] * vals[j][c] for j in range(len(keys))) / tot for c in range(dv)]
    return out, top + math.log(tot)


def tolist(a):
    return np.asarray(a, dtype=np.float64).tolist()


# ---------------------------------------------------------------------------
# the checks (plain functions so that the mutation tests can rerun them)
# ---------------------------------------------------------------------------
def check_golden_attend():
    cases = json.load(open(GOLDEN))["attend"]
    for c in cases:
        o, l_ = mo.attend(np.array(c["q"], float), np.array(c["k"], float), np.array(c["v"], float), c["scale"])
        np.testing.assert_allclose(o, np.array(c["out"]), rtol=0, atol=1e-12, err_msg=c["name"])
        np.testing.assert_allclose(l_, np.array(c["lse"]), rtol=0, atol=1e-12, err_msg=c["name"])


def check_golden_merge():
    cases = json.load(open(GOLDEN))["merge"]
    for c in cases:
        o, l_ = mo.merge(np.array(c["out_a"]), np.array(_num(c["lse_a"])),
                         np.array(c["out_b"]), np.array(_num(c["lse_b"])))
        assert not np.isnan(o).any() and not np.isnan(l_).any(), c["name"]
        np.testing.assert_allclose(o, np.array(c["out"]), rtol=0, atol=1e-12, err_msg=c["name"])
        exp_l = _num(c["lse"])
        if exp_l == -math.inf:
            assert np.isneginf(l_), c["name"]
        else:
            assert abs(float(l_) - exp_l) < 1e-12, c["name"]
        # the merge is symmetric in its two sides
        o2, l2 = mo.merge(np.array(c["out_b"]), np.array(_num(c["lse_b"])),
                          np.array(c["out_a"]), np.array(_num(c["lse_a"])))
        np.testing.assert_allclose(o2, o, atol=1e-12)


def check_prefill_brute(seed=11):
    rng = np.random.default_rng(seed)
    T, H, dk, dv, Tkv = 5, 3, 10, 6, 7
    q = rng.standard_normal((T, H, dk))
    kv = rng.standard_normal((Tkv, dk))
    scale = 0.37
    for (causal, q_pos0, kv_pos0, kv_valid) in [(True, 0, 0, 7), (True, 4, 1, 7), (False, 0, 0, 5),
                                                 (True, 2, 3, 6), (True, 0, 3, 7)]:
        out, lse = mo.mla_prefill(q, kv, scale, dv=dv, causal=causal, q_pos0=q_pos0,
                                  kv_pos0=kv_pos0, kv_valid=kv_valid)
        for t in range(T):
            keys = [tolist(kv[j]) for j in range(Tkv)
                    if j < kv_valid and (not causal or kv_pos0 + j <= q_pos0 + t)]
            vals = [k[:dv] for k in keys]
            for h in range(H):
                bo, bl = brute_attend(tolist(q[t, h]), keys, vals, scale)
                if not keys:
                    assert np.isneginf(lse[h, t]) and np.all(out[t, h] == 0)
                    continue
                np.testing.assert_allclose(out[t, h], bo, rtol=1e-12, atol=1e-12)
                assert abs(lse[h, t] - bl) < 1e-12


def check_prefill_prev_brute(seed=12):
    """The prev merge, computed by hand from the brute force of the two key sets."""
    rng = np.random.default_rng(seed)
    T, H, dk, dv = 4, 2, 8, 5
    q = rng.standard_normal((T, H, dk))
    kv_a = rng.standard_normal((6, dk))
    kv_b = rng.standard_normal((6, dk))
    scale = 0.5
    # ring step: chunk a holds keys 0..5, chunk b keys 6..11; queries at 6..9
    out_a, lse_a = mo.mla_prefill(q, kv_a, scale, dv=dv, causal=True, q_pos0=6, kv_pos0=0)
    out, lse = mo.mla_prefill(q, kv_b, scale, dv=dv, causal=True, q_pos0=6, kv_pos0=6,
                              prev_out=out_a, prev_lse=lse_a)
    kv_all = np.concatenate([kv_a, kv_b])
    for t in range(T):
        keys = [tolist(kv_all[j]) for j in range(6 + t + 1)]
        vals = [k[:dv] for k in keys]
        for h in range(H):
            bo, bl = brute_attend(tolist(q[t, h]), keys, vals, scale)
            np.testing.assert_allclose(out[t, h], bo, rtol=1e-11, atol=1e-12)
            assert abs(lse[h, t] - bl) < 1e-11


def check_closed_forms_prefill():
    """Single key, equal scores and causal row 0 on the MLA geometry."""
    P = gen.prefill_inputs(T=4, H=3, Tkv=4, seed=5, scale=gen.SCALE_192)
    q = P.q.double().numpy()
    kv = P.kv.double().numpy()
    out, lse = mo.mla_prefill(q, kv, P.scale, dv=512, causal=True)
    # causal row 0 sees only key 0: O = kv[0][:512], lse = scale * q0.k0
    for h in range(3):
        np.testing.assert_allclose(out[0, h], kv[0, :512], rtol=0, atol=1e-12)
        s0 = P.scale * sum(float(a) * float(b) for a, b in zip(q[0, h], kv[0]))
        assert abs(lse[h, 0] - s0) < 1e-9
    # q = 0: all scores equal, O = mean of V rows, lse = ln(#keys)
    out0, lse0 = mo.mla_prefill(np.zeros_like(q), kv, P.scale, dv=512, causal=True)
    for t in range(4):
        np.testing.assert_allclose(out0[t, 0], kv[: t + 1, :512].mean(axis=0), atol=1e-12)
        assert abs(lse0[0, t] - math.log(t + 1)) < 1e-12
    # all keys identical: O = that value row for every query, lse = s + ln n
    kv_same = np.repeat(kv[1:2], 4, axis=0)
    o3, l3 = mo.mla_prefill(q, kv_same, P.scale, dv=512, causal=True)
    for t in range(4):
        np.testing.assert_allclose(o3[t, 2], kv[1, :512], atol=1e-12)
        s = P.scale * float(q[t, 2] @ kv[1])
        assert abs(l3[2, t] - (s + math.log(t + 1))) < 1e-9


def check_rope_columns_count():
    """QK^T spans all 576 columns: scores change when only the RoPE part changes."""
    P = gen.prefill_inputs(T=1, H=1, Tkv=2, seed=21)
    q = P.q.double().numpy()
    kv = P.kv.double().numpy()
    kv2 = kv.copy()
    kv2[1, 512:] += 1.0     # only RoPE columns of key 1 change
    _, l1 = mo.mla_prefill(q, kv, 1.0, dv=512, causal=False)
    _, l2 = mo.mla_prefill(q, kv2, 1.0, dv=512, causal=False)
    assert abs(l1[0, 0] - l2[0, 0]) > 1e-6
    # and V is the latent prefix: changing RoPE columns never enters O directly
    q0 = np.zeros_like(q)
    o1, _ = mo.mla_prefill(q0, kv, 1.0, dv=512, causal=False)
    o2, _ = mo.mla_prefill(q0, kv2, 1.0, dv=512, causal=False)
    np.testing.assert_allclose(o1, o2, atol=0)


def check_chunk_merge_equals_one_pass():
    """Cached chunks (FULL mask) + current chunk (CAUSAL) merged by LSE equals one causal pass."""
    T, H, Tkv = 24, 2, 24
    P = gen.prefill_inputs(T=T, H=H, Tkv=Tkv, seed=2)
    q = P.q.double().numpy()
    kv = P.kv.double().numpy()
    ref_o, ref_l = mo.mla_prefill(q, kv, P.scale, causal=True)
    run_o = run_l = None
    for c0 in range(0, Tkv, 8):          # ring order 0, 1, 2
        o, l_ = mo.mla_prefill(q, kv[c0:c0 + 8], P.scale, causal=True, q_pos0=0, kv_pos0=c0,
                               prev_out=run_o, prev_lse=run_l)
        run_o, run_l = o, l_
    np.testing.assert_allclose(run_o, ref_o, atol=1e-12)
    np.testing.assert_allclose(run_l, ref_l, atol=1e-12)
    # the merge is order independent: process the chunks backwards
    run_o = run_l = None
    for c0 in reversed(range(0, Tkv, 8)):
        o, l_ = mo.mla_prefill(q, kv[c0:c0 + 8], P.scale, causal=True, q_pos0=0, kv_pos0=c0,
                               prev_out=run_o, prev_lse=run_l)
        run_o, run_l = o, l_
    np.testing.assert_allclose(run_o, ref_o, atol=1e-12)
    np.testing.assert_allclose(run_l, ref_l, atol=1e-12)


def check_invariances():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((4, 9))
    k = rng.standard_normal((7, 9))
    v = rng.standard_normal((7, 5))
    o, l_ = mo.attend(q, k, v, 0.3)
    perm = rng.permutation(7)
    o2, l2 = mo.attend(q, k[perm], v[perm], 0.3)
    np.testing.assert_allclose(o2, o, atol=1e-13)
    np.testing.assert_allclose(l2, l_, atol=1e-13)
    # adding the same constant c to every score: append a column q=c/scale, k=1
    c = 2.5
    q3 = np.concatenate([q, np.full((4, 1), c / 0.3)], axis=1)
    k3 = np.concatenate([k, np.ones((7, 1))], axis=1)
    o3, l3 = mo.attend(q3, k3, v, 0.3)
    np.testing.assert_allclose(o3, o, atol=1e-12)
    np.testing.assert_allclose(l3, l_ + c, atol=1e-12)


def check_sparse_full_prefix_equals_dense():
    S, S_kv, H, pos0 = 6, 10, 3, 4
    K = 16                               # padded with -1 beyond the prefix
    g = torch.Generator().manual_seed(7)
    topk = torch.full((S, K), -1, dtype=torch.int32)
    for s in range(S):
        n = pos0 + s + 1
        topk[s, :n] = torch.randperm(n, generator=g).to(torch.int32)
    SI = gen.sparse_inputs(S, S_kv, H, K, pos0, seed=9, topk=topk)
    out, lse = mo.mla_sparse(SI.q_lift, SI.q_pe, SI.c_kv, SI.k_pe, SI.topk, SI.scale)
    q = torch.cat([SI.q_lift[0], SI.q_pe[0]], dim=-1)            # [S,H,576]
    kv = torch.cat([SI.c_kv[0], SI.k_pe[0]], dim=-1)             # [S_kv,576]
    d_out, d_lse = mo.mla_prefill(q, kv, SI.scale, causal=True, q_pos0=pos0, kv_pos0=0)
    np.testing.assert_allclose(out[0].reshape(S, H, 512), d_out, atol=1e-12)
    np.testing.assert_allclose(lse[0], d_lse.T, atol=1e-12)
    # brute force on one query and head, with padding and a duplicate index
    idx = [3, -1, 0, 3, 40]
    tk = torch.tensor([[idx]], dtype=torch.int32)
    SJ = gen.sparse_inputs(1, 5, 1, len(idx), 0, seed=13, topk=tk)
    o, l_ = mo.mla_sparse(SJ.q_lift, SJ.q_pe, SJ.c_kv, SJ.k_pe, SJ.topk, SJ.scale)
    ck = SJ.c_kv[0].double().numpy()
    kp = SJ.k_pe[0].double().numpy()
    keys = [tolist(np.concatenate([ck[j], kp[j]])) for j in [3, 0, 3]]
    vals = [tolist(ck[j]) for j in [3, 0, 3]]
    qrow = tolist(np.concatenate([SJ.q_lift[0, 0, 0].double().numpy(), SJ.q_pe[0, 0, 0].double().numpy()]))
    bo, bl = brute_attend(qrow, keys, vals, SJ.scale)
    np.testing.assert_allclose(o[0, 0], bo, atol=1e-12)
    assert abs(l_[0, 0, 0] - bl) < 1e-12


def check_decode_equals_prefill_last_row():
    lens = [1, 5, 64, 130, 77]
    D = gen.decode_inputs(lens, H=3, seed=4, page_size=16, extra_pages=3)
    out, lse = mo.mla_decode(D.q, D.cache, D.block_table, D.lens, D.scale)
    cache = D.cache.double().numpy()
    for b, n in enumerate(lens):
        rows = np.stack([cache[int(D.block_table[b, j // 16]), j % 16] for j in range(n)])
        qb = np.zeros((n, 3, 576))
        qb[n - 1] = D.q[b].double().numpy()
        po, pl = mo.mla_prefill(qb, rows, D.scale, causal=True, tokens=[n - 1])
        np.testing.assert_allclose(out[b], po[0], atol=1e-12)
        np.testing.assert_allclose(lse[b], pl[:, 0], atol=1e-12)
    # brute force for one (request, head)
    b, h = 1, 2
    rows = [tolist(cache[int(D.block_table[b, j // 16]), j % 16]) for j in range(lens[b])]
    bo, bl = brute_attend(tolist(D.q[b, h].double().numpy()), rows, [r[:512] for r in rows], D.scale)
    np.testing.assert_allclose(out[b, h], bo, atol=1e-12)
    assert abs(lse[b, h] - bl) < 1e-12


def _sdpa_split(si, mask_type):
    """torch SDPA (fp64, CPU) per sequence with an explicit bottom-right causal mask."""
    ql = si.seq_len[0].tolist()
    kl = si.seq_len[1].tolist()
    H, Hkv = si.head_num, si.kv_head_num or si.head_num
    outs = []
    qo = ko = 0
    for b in range(len(ql)):
        q = torch.cat([si.q_nope[qo:qo + ql[b]], si.q_pe[qo:qo + ql[b]]], -1).double().transpose(0, 1)
        k = torch.cat([si.k_nope[ko:ko + kl[b]], si.k_pe[ko:ko + kl[b]]], -1).double().transpose(0, 1)
        v = si.v[ko:ko + kl[b]].double().transpose(0, 1)
        k = k.repeat_interleave(H // Hkv, dim=0)
        v = v.repeat_interleave(H // Hkv, dim=0)
        mask = None
        if mask_type == 1:
            i = torch.arange(ql[b])[:, None]
            j = torch.arange(kl[b])[None, :]
            mask = j <= (kl[b] - ql[b] + i)
        o = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None], attn_mask=mask,
                                                             scale=si.scale)[0]
        outs.append(o.transpose(0, 1))
        qo += ql[b]
        ko += kl[b]
    return torch.cat(outs).numpy()


def check_split_equals_library_sdpa():
    for (qlens, kvlens, H, Hkv, mt) in [([5, 9, 1], [5, 9, 1], 4, 4, 1), ([3, 4], [7, 4], 4, 2, 1),
                                          ([6, 2], [6, 5], 4, 1, 0)]:
        si = gen.split_inputs(qlens, kvlens, H, Hkv, seed=31)
        out, lse = mo.mla_prefill_split(si.q_nope, si.q_pe, si.k_nope, si.k_pe, si.v, si.seq_len,
                                        H, Hkv, si.scale, mt)
        ref = _sdpa_split(si, mt)
        np.testing.assert_allclose(out, ref, atol=1e-12)
    # kvHeadNum = 0 means kvHeadNum = headNum; a [batch] seqLen means q = kv lengths
    si = gen.split_inputs([4, 3], [4, 3], 2, 2, seed=32)
    o1, l1 = mo.mla_prefill_split(si.q_nope, si.q_pe, si.k_nope, si.k_pe, si.v, si.seq_len, 2, 0, si.scale, 1)
    o2, l2 = mo.mla_prefill_split(si.q_nope, si.q_pe, si.k_nope, si.k_pe, si.v, si.seq_len[0], 2, 2, si.scale, 1)
    np.testing.assert_allclose(o1, o2, atol=0)
    np.testing.assert_allclose(l1, l2, atol=0)


def check_split_lse_brute():
    si = gen.split_inputs([3, 2], [4, 2], 2, 1, seed=33)
    out, lse = mo.mla_prefill_split(si.q_nope, si.q_pe, si.k_nope, si.k_pe, si.v, si.seq_len, 2, 1, si.scale, 1)
    # token 1 = sequence 0, query 1, position 4 - 3 + 1 = 2 -> keys 0..2 of KV head 0
    qrow = tolist(torch.cat([si.q_nope[1, 1], si.q_pe[1, 1]]).double())
    keys = [tolist(torch.cat([si.k_nope[j, 0], si.k_pe[j, 0]]).double()) for j in range(3)]
    vals = [tolist(si.v[j, 0].double()) for j in range(3)]
    bo, bl = brute_attend(qrow, keys, vals, si.scale)
    np.testing.assert_allclose(out[1, 1], bo, atol=1e-12)
    assert abs(lse[1, 1] - bl) < 1e-12


def check_absorbed_equals_non_absorbed():
    """absorb_q (q_nope times k_b_proj_trans^T) and project_out (O times v_b_proj^T) around the
    latent attention reproduce MHA over the explicitly up-projected keys and values."""
    rng = np.random.default_rng(8)
    T, H, L, R, dn, dvh = 5, 2, 16, 4, 6, 5
    c = rng.standard_normal((T, L))           # latent cache rows
    k_pe = rng.standard_normal((T, R))
    q_nope = rng.standard_normal((T, H, dn))
    q_pe = rng.standard_normal((T, H, R))
    W_k = rng.standard_normal((H, L, dn)) / 4    # k_b_proj_trans: k_nope[h] = c @ W_k[h]
    W_v = rng.standard_normal((H, dvh, L)) / 4   # v_b_proj: v[h] = c @ W_v[h].T
    scale = 0.3
    q_lift = mo.absorb_q(q_nope, W_k)
    q_abs = np.concatenate([q_lift, q_pe], -1)
    kv = np.concatenate([c, k_pe], -1)
    o_lat, lse_a = mo.mla_prefill(q_abs, kv, scale, dv=L, causal=True)
    o_abs = mo.project_out(o_lat, W_v)
    for h in range(H):
        k_nope = c @ W_k[h]
        v = c @ W_v[h].T
        q = np.concatenate([q_nope[:, h], q_pe[:, h]], -1)
        k = np.concatenate([k_nope, k_pe], -1)
        qs = torch.from_numpy(q)[None, None]
        ks = torch.from_numpy(k)[None, None]
        vs = torch.from_numpy(v)[None, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, is_causal=True, scale=scale)[0, 0]
        np.testing.assert_allclose(o_abs[:, h], ref.numpy(), atol=1e-12)
    # one entry by hand: q_lift[t, h, l] = sum_d q_nope[t, h, d] W_k[h, l, d]
    assert abs(q_lift[3, 1, 7] - sum(q_nope[3, 1, d] * W_k[1, 7, d] for d in range(dn))) < 1e-12
    assert abs(o_abs[2, 0, 4] - sum(o_lat[2, 0, l] * W_v[0, 4, l] for l in range(L))) < 1e-12


def check_rope_golden():
    """Hand-rotated pairs.  x = (1, 2, 3, 4): pair 0 turns by 90 degrees (cos 0, sin 1), pair 1 by 0.
    Interleaved pairs (1, 2), (3, 4): (1, 2) -> (1*0 - 2*1, 1*1 + 2*0) = (-2, 1); (3, 4) stays.
    Halves pairs (1, 3), (2, 4): (1, 3) -> (-3, 1) at positions 0 and 2; (2, 4) stays."""
    x = np.array([1.0, 2.0, 3.0, 4.0])
    c, s = np.array([0.0, 1.0]), np.array([1.0, 0.0])
    np.testing.assert_array_equal(mo.rope(x, c, s, False), [-2.0, 1.0, 3.0, 4.0])
    np.testing.assert_array_equal(mo.rope(x, c, s, True), [-3.0, 2.0, 1.0, 4.0])
    # the identity angle leaves any vector unchanged
    y = np.random.default_rng(3).standard_normal(64)
    np.testing.assert_array_equal(mo.rope(y, np.ones(32), np.zeros(32), False), y)


def _rope_table(max_pos, R=64, base=10000.0):
    inv = base ** (-np.arange(0, R, 2) / R)          # R/2 frequencies
    ang = np.arange(max_pos)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], 1)


def check_rope_properties():
    """Rotation keeps each pair's length; scores depend on the position difference only; the halves
    layout is the interleaved one under the pair permutation."""
    rng = np.random.default_rng(12)
    cs = _rope_table(64)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    for neox in (False, True):
        for m in (0, 5, 40):
            r = mo.rope(q, cs[m, :32], cs[m, 32:], neox)
            pairs = (lambda v: np.stack([v[:32], v[32:]])) if neox else (lambda v: np.stack([v[0::2], v[1::2]]))
            np.testing.assert_allclose(np.linalg.norm(pairs(r), axis=0), np.linalg.norm(pairs(q), axis=0), atol=1e-12)
        for m, n in ((7, 3), (50, 50), (63, 0)):
            lhs = mo.rope(q, cs[m, :32], cs[m, 32:], neox) @ mo.rope(k, cs[n, :32], cs[n, 32:], neox)
            rhs = mo.rope(q, cs[m - n, :32], cs[m - n, 32:], neox) @ k
            assert abs(lhs - rhs) < 1e-10
    perm = np.empty(64, dtype=int)          # interleaved index 2i <- halves i, 2i+1 <- halves i + 32
    perm[0::2], perm[1::2] = np.arange(32), np.arange(32) + 32
    x = rng.standard_normal(64)
    inter = mo.rope(x[perm], cs[9, :32], cs[9, 32:], False)
    back = np.empty(64)
    back[perm] = inter
    np.testing.assert_allclose(mo.rope(x, cs[9, :32], cs[9, 32:], True), back, atol=1e-12)


def check_rope_append():
    """The appended row lands at (block_table[b][pos // P], pos % P) and nowhere else, holds
    [c_kv | rotated k_pe], and a decode over pos + 1 keys then attends to it like any other key."""
    rng = np.random.default_rng(21)
    B, H, P, L, R = 2, 3, 4, 8, 4
    pages = 5
    cache = rng.standard_normal((pages, P, L + R))
    bt = np.array([[3, 0, -1], [1, 4, 2]])
    pos = np.array([5, 9])
    q_pe, c_kv, k_pe = rng.standard_normal((B, H, R)), rng.standard_normal((B, L)), rng.standard_normal((B, R))
    cs = _rope_table(16, R)
    q_rope, new = mo.mla_rope_append(q_pe, c_kv, k_pe, pos, cs, False, cache, bt, P)
    changed = np.argwhere(np.any(new != cache, axis=-1))
    assert sorted(map(tuple, changed)) == [(0, 1), (2, 1)]        # (page 0, slot 1) and (page 2, slot 1)
    np.testing.assert_array_equal(new[0, 1, :L], c_kv[0])
    np.testing.assert_allclose(new[2, 1, L:], mo.rope(k_pe[1], cs[9, :2], cs[9, 2:], False), atol=1e-15)
    np.testing.assert_allclose(q_rope[1, 2], mo.rope(q_pe[1, 2], cs[9, :2], cs[9, 2:], False), atol=1e-15)
    q_lat = rng.standard_normal((B, H, L))
    q = np.concatenate([q_lat, q_rope], -1)
    out, lse = mo.mla_decode(q, new, bt, pos + 1, 0.5, dv=L)
    keys = np.stack([new[bt[1, j // P], j % P] for j in range(10)])
    o_ref, l_ref = mo.attend(q[1], keys, keys[:, :L], 0.5)
    np.testing.assert_allclose(out[1], o_ref, atol=1e-12)
    np.testing.assert_allclose(lse[1], l_ref, atol=1e-12)


def _small_decode():
    D = gen.decode_inputs([5, 64, 130, 2], H=3, seed=6, page_size=16, extra_pages=2)
    return {"q": D.q.double().numpy(), "cache": D.cache.double().numpy(), "bt": D.block_table.numpy(),
            "lens": D.lens.numpy(), "dv": 512}


def check_decode_ex():
    """Several query tokens per request: token i equals the causal prefill row at position
    len - s + i over the request's gathered rows; one token and no sinks is mla_decode; a sink
    adds e^{sink} to the denominator (closed form with one key) and -inf sinks change nothing."""
    D = _small_decode()
    rng = np.random.default_rng(30)
    B, H = D["q"].shape[0], D["q"].shape[1]
    S = 3
    q = rng.standard_normal((B, S, H, D["q"].shape[2]))
    out, lse = mo.mla_decode_ex(q, D["cache"], D["bt"], D["lens"], 0.4, dv=D["dv"])
    for b in range(B):
        n = int(D["lens"][b])
        rows = mo.gather_pages(D["cache"], D["bt"][b], n, D["cache"].shape[1])
        for i in range(S):
            po, pl = mo.mla_prefill(q[b, i][None], rows, 0.4, dv=D["dv"], causal=True, q_pos0=n - S + i)
            np.testing.assert_allclose(out[b, i], po[0], atol=1e-12)
            np.testing.assert_allclose(lse[b, i], pl[:, 0], atol=1e-12)
    o1, l1 = mo.mla_decode_ex(D["q"][:, None], D["cache"], D["bt"], D["lens"], 0.4, dv=D["dv"])
    o0, l0 = mo.mla_decode(D["q"], D["cache"], D["bt"], D["lens"], 0.4, dv=D["dv"])
    np.testing.assert_allclose(o1[:, 0], o0, atol=1e-12)
    np.testing.assert_allclose(l1[:, 0], l0, atol=1e-12)
    on, ln_ = mo.mla_decode_ex(q, D["cache"], D["bt"], D["lens"], 0.4, sinks=np.full(H, -np.inf), dv=D["dv"])
    np.testing.assert_allclose(on, out, atol=1e-12)
    # one key of score s and value v with a sink z: out = v e^s / (e^s + e^z), lse = ln(e^s + e^z)
    cache = np.zeros((1, 4, 3))
    cache[0, 0] = [2.0, 1.5, -1.0]                     # key (dk = 3), value = first 2 columns
    qq = np.array([[[[0.5, 1.0, 2.0]]]])               # s = 0.5 * (1 + 1.5 - 2) = 0.25
    o, l_ = mo.mla_decode_ex(qq, cache, np.array([[0]]), np.array([1]), 0.5, sinks=np.array([1.0]), dv=2)
    w = np.exp(0.25) / (np.exp(0.25) + np.exp(1.0))
    np.testing.assert_allclose(o[0, 0, 0], w * np.array([2.0, 1.5]), atol=1e-15)
    assert abs(l_[0, 0, 0] - np.log(np.exp(0.25) + np.exp(1.0))) < 1e-14
    # a token that sees no key: out = 0, lse = the sink (or -inf without one)
    o, l_ = mo.mla_decode_ex(np.zeros((1, 2, 1, 3)), cache, np.array([[0]]), np.array([1]), 0.5,
                             sinks=np.array([0.7]), dv=2)
    assert (o[0, 0] == 0).all() and l_[0, 0, 0] == 0.7


def check_decode_fp8():
    """An e4m3 cache stands for its values times kv_scale: the same keys/values given in fp64 (scaled)
    give the same result; doubling kv_scale doubles every score and every output value."""
    D = _small_decode()
    rng = np.random.default_rng(33)
    c8 = torch.from_numpy(D["cache"] / 3.0).to(torch.float8_e4m3fn)
    vals = c8.double().numpy()
    q = rng.standard_normal((D["q"].shape[0], 2, D["q"].shape[1], D["q"].shape[2]))
    out, lse = mo.mla_decode_fp8(q, c8, 3.0, D["bt"], D["lens"], 0.2)
    ro, rl = mo.mla_decode_ex(q, vals * 3.0, D["bt"], D["lens"], 0.2)
    np.testing.assert_allclose(out, ro, atol=1e-12)
    np.testing.assert_allclose(lse, rl, atol=1e-12)
    o2, l2 = mo.mla_decode_fp8(q, c8, 6.0, D["bt"], D["lens"], 0.1)   # scores unchanged, values doubled
    np.testing.assert_allclose(o2, 2.0 * out, atol=1e-12)
    np.testing.assert_allclose(l2, lse, atol=1e-12)


def check_flop_count():
    # causal T = Tkv = n: n(n+1)/2 pairs
    assert mo.causal_pairs(256, 256, 0, 0) == 256 * 257 // 2
    # chunk j of the 4 x 2048 ring over 8192 queries
    per = [mo.causal_pairs(8192, 2048, 0, 2048 * j) for j in range(4)]
    assert sum(per) == 8192 * 8193 // 2
    assert mo.attention_flops(1, 128, 576, 512) == 2 * 128 * 1088


ALL_CHECKS = [
    check_golden_attend, check_golden_merge, check_prefill_brute, check_prefill_prev_brute,
    check_closed_forms_prefill, check_rope_columns_count, check_chunk_merge_equals_one_pass,
    check_invariances, check_sparse_full_prefix_equals_dense, check_decode_equals_prefill_last_row,
    check_split_equals_library_sdpa, check_split_lse_brute, check_absorbed_equals_non_absorbed,
    check_flop_count, check_rope_golden, check_rope_properties, check_rope_append, check_decode_ex, check_decode_fp8,
]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check()


def test_every_exported_function_is_reached_by_a_pin():
    """Each function the oracle exports runs inside at least one pin (directly or through a
    caller), so none of them can drift unchecked."""
    import sys
    called = set()
    src = mo.__file__

    def tracer(frame, event, arg):
        if event == "call" and frame.f_code.co_filename == src:
            called.add(frame.f_code.co_name)

    sys.setprofile(tracer)
    try:
        for check in ALL_CHECKS:
            check()
    finally:
        sys.setprofile(None)
    exported = {n for n in mo.__all__ if callable(getattr(mo, n))}
    assert exported - called == set(), f"oracle functions no pin reaches: {sorted(exported - called)}"
