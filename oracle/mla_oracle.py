"""fp64 CPU oracle for the Multi-head Latent Attention (MLA) forward.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run this module.  The product
path (the CUDA library and its Python binding) never calls it; it shares no
code, table or helper with that path.

What it computes is the plain definition, written out step by step, in fp64
(numpy), on the bf16 values the caller holds (inputs are decoded exactly):

  for each query row r and its key set J(r):
      s_j   = scale * <q_r, k_j>                      (all dk columns)
      m     = max_j s_j ;  l = sum_j exp(s_j - m)
      O_r   = sum_j exp(s_j - m) * v_j / l            (v_j = value row of key j)
      lse_r = m + ln l                                (natural log)
  an empty J(r) gives O_r = 0 and lse_r = -inf.
  With a previous pair (O_p, lse_p):
      m' = max(lse_p, lse_r); m' = -inf -> (0, -inf)
      O  = (e^(lse_p-m') O_p + e^(lse_r-m') O_r) / (e^(lse_p-m') + e^(lse_r-m'))
      lse = m' + ln(e^(lse_p-m') + e^(lse_r-m'))

Passages followed (pages by title, with their sections):
  * Tenstorrent "ttnn.transformer.ring_mla": one shared KV head; QK^T over the
    full KV width; the first head_dim_v columns of KV are V; causal; outputs
    the attention output and streaming statistics.
  * Huawei Ascend "RingMLAOperation", parameter table: split q/k (128 no-PE +
    64 RoPE), value 128, seqLen [batch] or [2, batch], kvHeadNum (0 = headNum),
    qkScale, maskType NO_MASK/TRIU, prevOut/prevLse in, softmaxLse [headNum,
    qNTokens] float out, calcType (first ring step passes no prev).
  * NVIDIA TensorRT-LLM "mla.py": forward_context_with_chunked_prefill (cached
    chunks with a FULL mask, current chunk CAUSAL, each partial merged into the
    running output and softmax statistics by merge_attention_for_mla);
    _attn_forward_gen (a fully masked row must not poison a combine with NaN).
  * Modular Mojo "mha_single_batch_pipelined": token generation, seqlen = 1,
    split-K over keys needs a separate reduction.
  * AWS NKI "MLA Sparse Attention CTE Kernel API Reference": per query,
    absorbed latent + RoPE attention over the top-k selected cache rows.

Readings where the pages are silent:
  * lse is the natural log of sum exp(scale * q.k) (Ascend: "exp, sum, and log
    ... in sequence"); prev_lse is fp32 (the page's "float16" for prevLse
    contradicts its float softmaxLse output).
  * Split layout causal alignment is bottom-right: query i of a sequence with
    q_len queries and kv_len keys sits at position kv_len - q_len + i.
  * Sparse: indices outside [0, S_kv) are padding and skipped; a repeated
    index counts once per occurrence; no causal mask beyond the list itself.
  * Decode: the single query sees all len keys of its request.

Pins: every function here is checked in tests/test_oracle_pins.py against
closed forms, a pure-Python brute force, library routines and identities of
the mathematics (see that file).  No function is "parity unpinned".
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

NEG_INF = -np.inf


def _f64(x) -> np.ndarray:
    """Decode a tensor/array (bf16, fp32, ...) exactly into float64."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def _i64(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu").to(torch.int64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.int64)


# ---------------------------------------------------------------------------
# the core definition
# ---------------------------------------------------------------------------
def attend(q_rows: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float):
    """Softmax attention of R query rows over one key set J.

    q_rows [R, dk], keys [|J|, dk], values [|J|, dv] (fp64).
    Returns (O [R, dv], lse [R]).  |J| = 0 gives O = 0, lse = -inf.
    """
    R = q_rows.shape[0]
    dv = values.shape[1]
    if keys.shape[0] == 0:
        return np.zeros((R, dv)), np.full((R,), NEG_INF)
    s = scale * (q_rows @ keys.T)                  # [R, |J|]
    m = s.max(axis=1, keepdims=True)               # row max
    p = np.exp(s - m)                              # unnormalised weights
    l = p.sum(axis=1, keepdims=True)               # row sum
    out = (p @ values) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse


def merge(out_a: np.ndarray, lse_a: np.ndarray, out_b: np.ndarray, lse_b: np.ndarray):
    """Merge two partial results of the same rows by their log-sum-exp.

    out_* [..., dv], lse_* [...] (matching leading shape).  A side with
    lse = -inf contributes nothing; both -inf gives (0, -inf), never NaN.
    This is the combine of merge_attention_for_mla / Ascend prevOut+prevLse.
    """
    out_a = np.asarray(out_a, dtype=np.float64)
    out_b = np.asarray(out_b, dtype=np.float64)
    lse_a = np.asarray(lse_a, dtype=np.float64)
    lse_b = np.asarray(lse_b, dtype=np.float64)
    m = np.maximum(lse_a, lse_b)
    empty = np.isneginf(m)
    m_safe = np.where(empty, 0.0, m)
    w_a = np.where(np.isneginf(lse_a), 0.0, np.exp(lse_a - m_safe))
    w_b = np.where(np.isneginf(lse_b), 0.0, np.exp(lse_b - m_safe))
    w = w_a + w_b
    w_div = np.where(empty, 1.0, w)
    out = (w_a[..., None] * out_a + w_b[..., None] * out_b) / w_div[..., None]
    out = np.where(empty[..., None], 0.0, out)
    lse = np.where(empty, NEG_INF, m_safe + np.log(np.where(empty, 1.0, w)))
    return out, lse


# ---------------------------------------------------------------------------
# absorbed dense prefill: many heads over one shared KV head
# ---------------------------------------------------------------------------
def prefill_key_set(t: int, Tkv: int, causal: bool, q_pos0: int, kv_pos0: int, kv_valid: int) -> np.ndarray:
    """Keys visible to query token t: j < kv_valid and (causal: kv_pos0 + j <= q_pos0 + t)."""
    n = min(Tkv, kv_valid)
    if causal:
        n = min(n, q_pos0 + t - kv_pos0 + 1)
    return np.arange(max(0, n))


def mla_prefill(q, kv, scale: float, dv: int = 512, causal: bool = True,
                q_pos0: int = 0, kv_pos0: int = 0, kv_valid: Optional[int] = None,
                prev_out=None, prev_lse=None, tokens: Optional[Sequence[int]] = None):
    """Absorbed causal MLA prefill over one shared KV head (ring_mla semantics).

    q [T, H, dk], kv [Tkv, dk]; V = kv[:, :dv].  Query token t sits at global
    position q_pos0 + t, key j at kv_pos0 + j; only keys j < kv_valid exist.
    Returns out [n, H, dv] and lse [H, n] for the requested tokens (all by
    default).  With prev_out [T, H, dv] / prev_lse [H, T] the result is merged
    with the previous pair (ring step / chunked prefill).
    """
    q = _f64(q)
    kv = _f64(kv)
    T, H, dk = q.shape
    Tkv = kv.shape[0]
    if kv_valid is None:
        kv_valid = Tkv
    toks = list(range(T)) if tokens is None else [int(t) for t in tokens]
    out = np.zeros((len(toks), H, dv))
    lse = np.full((H, len(toks)), NEG_INF)
    for i, t in enumerate(toks):
        J = prefill_key_set(t, Tkv, causal, q_pos0, kv_pos0, kv_valid)
        o, l_ = attend(q[t], kv[J], kv[J, :dv], scale)
        out[i], lse[:, i] = o, l_
    if prev_out is not None:
        po = _f64(prev_out)[toks]
        pl = _f64(prev_lse)[:, toks]
        mo, ml = merge(po, pl.T, out, lse.T)
        out, lse = mo, ml.T
    return out, lse


# ---------------------------------------------------------------------------
# Ascend split layout (non-absorbed), varlen, GQA, NO_MASK / TRIU
# ---------------------------------------------------------------------------
def attend_masked(q_rows: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float, visible: np.ndarray):
    """attend() where row r sees only the keys with visible[r, j] true (a row may see none)."""
    R, dv = q_rows.shape[0], values.shape[1]
    out = np.zeros((R, dv))
    lse = np.full((R,), NEG_INF)
    if keys.shape[0] == 0:
        return out, lse
    s = scale * (q_rows @ keys.T)
    s = np.where(visible, s, NEG_INF)
    has = visible.any(axis=1)
    m = np.where(has, s.max(axis=1), 0.0)[:, None]
    p = np.where(visible, np.exp(s - m), 0.0)
    l = p.sum(axis=1, keepdims=True)
    l_safe = np.where(l > 0, l, 1.0)
    out = np.where(has[:, None], (p @ values) / l_safe, 0.0)
    lse = np.where(has, (m + np.log(l_safe))[:, 0], NEG_INF)
    return out, lse


def mla_prefill_split(q_nope, q_pe, k_nope, k_pe, v, seq_len, head_num: int, kv_head_num: int,
                      scale: float, mask_type: int, prev_out=None, prev_lse=None,
                      tokens: Optional[Sequence[int]] = None):
    """Ascend RingMLAOperation forward on the BSND split layout.

    q_nope [Nq,H,128], q_pe [Nq,H,64], k_nope/k_pe/v [Nkv,Hkv,*]; seq_len
    [batch] (q = kv lengths) or [2, batch].  Head h reads KV head
    h // (H / Hkv); kv_head_num 0 means head_num.  mask_type 0 = NO_MASK,
    1 = TRIU (query i of a sequence sees keys j <= kv_len - q_len + i).
    Returns out [n, H, 128], lse [H, n] for the requested global query tokens.
    """
    qn, qp = _f64(q_nope), _f64(q_pe)
    kn, kp, vv = _f64(k_nope), _f64(k_pe), _f64(v)
    sl = _i64(seq_len)
    if sl.ndim == 1:
        q_lens, kv_lens = sl, sl
    else:
        q_lens, kv_lens = sl[0], sl[1]
    H = int(head_num)
    Hkv = int(kv_head_num) if kv_head_num else H
    group = H // Hkv
    Nq = qn.shape[0]
    dv = vv.shape[2]
    q_off = np.concatenate([[0], np.cumsum(q_lens)])
    kv_off = np.concatenate([[0], np.cumsum(kv_lens)])
    toks = np.arange(Nq) if tokens is None else np.asarray([int(t) for t in tokens], dtype=np.int64)
    out = np.zeros((len(toks), H, dv))
    lse = np.full((H, len(toks)), NEG_INF)
    seq_of = np.searchsorted(q_off, toks, side="right") - 1
    for b in range(len(q_lens)):
        sel = np.nonzero(seq_of == b)[0]               # positions in `toks` of this sequence
        if len(sel) == 0:
            continue
        ql, kl = int(q_lens[b]), int(kv_lens[b])
        qi = toks[sel] - q_off[b]                       # query index inside the sequence
        j = np.arange(kl)
        if mask_type == 0:
            visible = np.ones((len(sel), kl), dtype=bool)
        else:
            visible = j[None, :] <= (kl - ql + qi)[:, None]
        ks = slice(kv_off[b], kv_off[b] + kl)
        for h in range(H):
            g = h // group
            qrows = np.concatenate([qn[toks[sel], h], qp[toks[sel], h]], axis=1)
            keys = np.concatenate([kn[ks, g], kp[ks, g]], axis=1)
            o, l_ = attend_masked(qrows, keys, vv[ks, g], scale, visible)
            out[sel, h] = o
            lse[h, sel] = l_
    if prev_out is not None:
        po = _f64(prev_out)[toks]
        pl = _f64(prev_lse)[:, toks]
        mo, ml = merge(po, pl.T, out, lse.T)
        out, lse = mo, ml.T
    return out, lse


# ---------------------------------------------------------------------------
# decode: one query token per request over a paged latent cache
# ---------------------------------------------------------------------------
def gather_pages(cache, block_table_row, n: int, page_size: int) -> np.ndarray:
    """Rows 0..n-1 of one request: row j lives at cache[block_table[j // P], j % P]."""
    cache = _f64(cache) if not isinstance(cache, np.ndarray) else cache
    bt = _i64(block_table_row)
    j = np.arange(n)
    return cache[bt[j // page_size], j % page_size]


def mla_decode(q, cache, block_table, lens, scale: float, dv: int = 512,
               requests: Optional[Sequence[int]] = None):
    """Absorbed MLA decode (seqlen = 1): each request's query sees all its len keys.

    q [B, H, dk], cache [pages, page_size, dk], block_table [B, max_pages],
    lens [B].  Returns out [n, H, dv] and lse [n, H].
    """
    qq = _f64(q)
    cc = _f64(cache)
    bt = _i64(block_table)
    ln = _i64(lens)
    B, H, dk = qq.shape
    P = cc.shape[1]
    reqs = list(range(B)) if requests is None else [int(b) for b in requests]
    out = np.zeros((len(reqs), H, dv))
    lse = np.full((len(reqs), H), NEG_INF)
    for i, b in enumerate(reqs):
        rows = gather_pages(cc, bt[b], int(ln[b]), P)
        o, l_ = attend(qq[b], rows, rows[:, :dv], scale)
        out[i], lse[i] = o, l_
    return out, lse


def mla_decode_ex(q, cache, block_table, lens, scale: float, sinks=None, dv: int = 512):
    """Decode with q_per_req query tokens per request and optional attention sinks.

    q [B, s, H, dk].  Token i of request b sits at position lens[b] - s + i and sees keys
    0 .. lens[b] - s + i (TensorRT-LLM "mla.py", predicted_tokens_per_seq: several generated
    tokens per request in one step, causal among them).  With sinks [H], head h's sink logit
    joins the softmax denominator as one more term with no value (Modular Mojo
    "mha_single_batch_pipelined", sink_weights): the result is the attention output merged by
    LSE with an empty-valued partial (O = 0, lse = sinks[h]).
    Returns out [B, s, H, dv], lse [B, s, H].
    """
    qq = _f64(q)
    cc = _f64(cache)
    bt = _i64(block_table)
    ln = _i64(lens)
    B, S, H, dk = qq.shape
    P = cc.shape[1]
    out = np.zeros((B, S, H, dv))
    lse = np.full((B, S, H), NEG_INF)
    for b in range(B):
        for i in range(S):
            n = max(0, int(ln[b]) - S + 1 + i)
            rows = gather_pages(cc, bt[b], n, P)
            out[b, i], lse[b, i] = attend(qq[b, i], rows, rows[:, :dv], scale)
    if sinks is not None:
        sk = _f64(sinks)
        out, lse = merge(out, lse, np.zeros_like(out), np.broadcast_to(sk, lse.shape))
    return out, lse


def mla_decode_fp8(q, cache_e4m3, kv_scale: float, block_table, lens, scale: float, sinks=None, dv: int = 512):
    """Decode over an FP8 (e4m3) latent cache with one per-tensor scale (TensorRT-LLM "mla.py":
    FP8 KV cache, use_fp8_mla, with the cache's scale applied to both BMMs, mla_bmm1_scale and
    mla_bmm2_scale): every cache value stands for e4m3_value * kv_scale.  cache_e4m3 holds the
    e4m3 values (decoded exactly); q as in mla_decode_ex ([B, s, H, dk])."""
    return mla_decode_ex(q, _f64(cache_e4m3) * float(kv_scale), block_table, lens, scale, sinks=sinks, dv=dv)


# ---------------------------------------------------------------------------
# top-k sparse latent + RoPE attention
# ---------------------------------------------------------------------------
def mla_sparse(q_lift, q_pe, c_kv, k_pe, topk, scale: float,
               tokens: Optional[Sequence[int]] = None):
    """NKI sparse MLA: query (b, s) attends the cache rows listed in topk[b, s].

    q_lift [B,S,H,L], q_pe [B,S,H,R], c_kv [B,S_kv,L], k_pe [B,S_kv,R],
    topk [B,S,K] int.  Indices outside [0, S_kv) are skipped; each listed
    occurrence counts.  Output in natural order: out [B, n, H*L], lse [B, n, H].
    """
    ql, qp = _f64(q_lift), _f64(q_pe)
    ck, kp = _f64(c_kv), _f64(k_pe)
    tk = _i64(topk)
    B, S, H, L = ql.shape
    S_kv = ck.shape[1]
    toks = list(range(S)) if tokens is None else [int(t) for t in tokens]
    out = np.zeros((B, len(toks), H * L))
    lse = np.full((B, len(toks), H), NEG_INF)
    for b in range(B):
        for i, s in enumerate(toks):
            idx = tk[b, s]
            idx = idx[(idx >= 0) & (idx < S_kv)]
            keys = np.concatenate([ck[b, idx], kp[b, idx]], axis=1)
            qrows = np.concatenate([ql[b, s], qp[b, s]], axis=1)     # [H, L+R]
            o, l_ = attend(qrows, keys, ck[b, idx], scale)
            out[b, i] = o.reshape(-1)
            lse[b, i] = l_
    return out, lse


# ---------------------------------------------------------------------------
# decode step before attention: RoPE and the paged latent-cache append
# ---------------------------------------------------------------------------
def rope(x, cos, sin, is_neox: bool) -> np.ndarray:
    """Rotary position embedding of the last axis (2n values = n rotation pairs).

    Pair i is rotated by the angle whose cosine and sine are cos[..., i], sin[..., i]:
    (a, b) -> (a cos - b sin, a sin + b cos).  The pairs are (x[2i], x[2i+1]) (interleaved)
    or, with is_neox, (x[i], x[i+n]) (halves) -- the two layouts TensorRT-LLM "mla.py"
    selects with RotaryEmbedding(..., is_neox=...) for the qk_rope_head_dim part.
    """
    x = _f64(x)
    c = _f64(cos)
    s = _f64(sin)
    n = x.shape[-1] // 2
    out = np.empty_like(x)
    if is_neox:
        a, b = x[..., :n], x[..., n:]
        out[..., :n] = a * c - b * s
        out[..., n:] = a * s + b * c
    else:
        a, b = x[..., 0::2], x[..., 1::2]
        out[..., 0::2] = a * c - b * s
        out[..., 1::2] = a * s + b * c
    return out


def mla_rope_append(q_pe, c_kv, k_pe, positions, cos_sin, is_neox: bool, cache, block_table, page_size: int):
    """One decode step's RoPE and latent-cache append (TensorRT-LLM "mla.py",
    forward_absorption_generation: q_pe and k_pe rotated at the new token's position
    (apply_rope), the rotated q_pe forms the RoPE part of the fused query, and the latent
    cache row of the new token receives [compressed_kv | rotated k_pe]
    (mla_rope_generation / mla_rope_append_paged_kv_assign_q append it to the paged cache)).

    q_pe [B, H, R], c_kv [B, L], k_pe [B, R], positions [B] (the token's index in its
    request's cache), cos_sin [max_pos, R] (cos of the R/2 angles, then their sin),
    cache [pages, page_size, L + R], block_table [B, max_pages].
    Returns (q_rope [B, H, R], cache after the append (a new array)).
    """
    qp, ck, kp = _f64(q_pe), _f64(c_kv), _f64(k_pe)
    cs = _f64(cos_sin)
    pos = _i64(positions)
    bt = _i64(block_table)
    new_cache = _f64(cache).copy()
    R = qp.shape[-1]
    n = R // 2
    q_rope = np.empty_like(qp)
    for b in range(qp.shape[0]):
        c, s = cs[pos[b], :n], cs[pos[b], n:]
        q_rope[b] = rope(qp[b], c[None, :], s[None, :], is_neox)
        page = bt[b, pos[b] // page_size]
        new_cache[page, pos[b] % page_size] = np.concatenate([ck[b], rope(kp[b], c, s, is_neox)])
    return q_rope, new_cache


# ---------------------------------------------------------------------------
# the absorption BMMs around the latent attention
# ---------------------------------------------------------------------------
def absorb_q(q_nope, k_b_proj_trans) -> np.ndarray:
    """q_lift[t, h, l] = sum_d q_nope[t, h, d] W[h, l, d] with W = k_b_proj_trans [H, L, D_nope]
    (TensorRT-LLM "mla.py", forward_absorption_generation: q_nope (per head) times
    k_b_proj_trans transposed, written into the latent part of the fused query)."""
    return np.einsum("thd,hld->thl", _f64(q_nope), _f64(k_b_proj_trans))


def project_out(o_latent, v_b_proj) -> np.ndarray:
    """out[t, h, v] = sum_l O[t, h, l] W[h, v, l] with W = v_b_proj [H, D_v, L] (TensorRT-LLM
    "mla.py": the latent attention output times v_b_proj transposed, per head)."""
    return np.einsum("thl,hvl->thv", _f64(o_latent), _f64(v_b_proj))


def attention_flops(pairs: int, H: int, dk: int, dv: int) -> float:
    """Algorithmic FLOPs of attention over `pairs` unmasked (query token, key) pairs."""
    return 2.0 * float(pairs) * H * (dk + dv)


def causal_pairs(T: int, Tkv: int, q_pos0: int, kv_pos0: int, kv_valid: Optional[int] = None) -> int:
    """Number of unmasked (token, key) pairs of a causal dense prefill call."""
    if kv_valid is None:
        kv_valid = Tkv
    tot = 0
    n_cap = min(Tkv, kv_valid)
    for t in range(T):
        tot += max(0, min(n_cap, q_pos0 + t - kv_pos0 + 1))
    return tot


__all__ = [
    "attend", "attend_masked", "merge", "prefill_key_set", "mla_prefill", "mla_prefill_split",
    "gather_pages", "mla_decode", "mla_decode_ex", "mla_decode_fp8", "mla_sparse", "rope", "mla_rope_append", "absorb_q", "project_out",
    "attention_flops", "causal_pairs", "NEG_INF",
]
