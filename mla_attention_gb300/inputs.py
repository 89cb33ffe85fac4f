"""Seeded synthetic inputs for the MLA attention forward.

This module only draws numbers: it holds none of the attention arithmetic.
Both the CPU oracle (through the tests) and the CUDA path consume what it
makes, so the two sides always see bit-identical inputs.

Every tensor is drawn on the CPU from ``torch.Generator('cpu')`` as fp32
N(0, 1) and rounded (round-to-nearest-even) to bf16, which makes the values
identical on x86 and Arm hosts.  Integer metadata (lengths, page tables, top-k
lists) come from the same generator.

Shapes follow the workloads of the pages:
  * DeepSeek latent geometry: one shared KV head, rows of 512 latent + 64 RoPE
    columns, V = the first 512 columns (Tenstorrent ``ring_mla``, "Causal Ring
    MLA attention over a single KV tensor"; AWS NKI MLA sparse attention CTE
    kernel, "Dimensions").
  * Ascend ``RingMLAOperation`` split layout: q/k = 128 no-PE + 64 RoPE columns,
    v = 128 columns, ``seqLen`` [2, batch].
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

LATENT = 512          # kv_lora_rank
ROPE = 64             # qk_rope_head_dim
DK = LATENT + ROPE    # 576: width of the shared KV row and of absorbed q
DV = LATENT           # V is the latent prefix of the KV row
SPLIT_NOPE = 128      # Ascend split layout: q/k no-PE width
SPLIT_PE = 64         # Ascend split layout: q/k RoPE width
SPLIT_V = 128         # Ascend split layout: v width
SCALE_192 = 192.0 ** -0.5


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, g: torch.Generator, chunk_elems: int = 1 << 26) -> torch.Tensor:
    """fp32 N(0,1) rounded to bf16, drawn in chunks to bound host memory."""
    out = torch.empty(shape, dtype=torch.bfloat16)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        flat[s:e] = torch.randn(e - s, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return out


# ---------------------------------------------------------------------------
# absorbed dense prefill (one shared KV head)
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class PrefillInputs:
    q: torch.Tensor            # [T, H, 576] bf16
    kv: torch.Tensor           # [Tkv, 576] bf16
    scale: float


def prefill_inputs(T: int, H: int, Tkv: int, seed: int, scale: float = SCALE_192) -> PrefillInputs:
    g = _gen(seed)
    q = randn_bf16((T, H, DK), g)
    kv = randn_bf16((Tkv, DK), g)
    return PrefillInputs(q=q, kv=kv, scale=scale)


def prev_inputs(T: int, H: int, dv: int, seed: int, lse_lo: float, lse_hi: float):
    """A caller-held previous (out, lse) pair: out bf16 N(0,1) [T,H,dv], lse fp32 U[lo,hi] [H,T]."""
    g = _gen(seed)
    prev_out = randn_bf16((T, H, dv), g)
    prev_lse = lse_lo + (lse_hi - lse_lo) * torch.rand((H, T), generator=g, dtype=torch.float32)
    return prev_out, prev_lse


# ---------------------------------------------------------------------------
# Ascend-style split layout, varlen
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class SplitInputs:
    q_nope: torch.Tensor       # [Nq, H, 128]
    q_pe: torch.Tensor         # [Nq, H, 64]
    k_nope: torch.Tensor       # [Nkv, Hkv, 128]
    k_pe: torch.Tensor         # [Nkv, Hkv, 64]
    v: torch.Tensor            # [Nkv, Hkv, 128]
    seq_len: torch.Tensor      # int32 [2, batch] (row 0: q lens, row 1: kv lens)
    head_num: int
    kv_head_num: int
    scale: float
    prev_out: Optional[torch.Tensor] = None   # [Nq, H, 128] bf16
    prev_lse: Optional[torch.Tensor] = None   # [H, Nq] fp32


def split_inputs(q_lens, kv_lens, H: int, Hkv: int, seed: int, scale: float = SCALE_192,
                 with_prev: bool = False, prev_lse_range=(7.4, 9.5)) -> SplitInputs:
    g = _gen(seed)
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    Nq, Nkv = sum(q_lens), sum(kv_lens)
    q_nope = randn_bf16((Nq, H, SPLIT_NOPE), g)
    q_pe = randn_bf16((Nq, H, SPLIT_PE), g)
    k_nope = randn_bf16((Nkv, Hkv, SPLIT_NOPE), g)
    k_pe = randn_bf16((Nkv, Hkv, SPLIT_PE), g)
    v = randn_bf16((Nkv, Hkv, SPLIT_V), g)
    seq_len = torch.tensor([q_lens, kv_lens], dtype=torch.int32)
    si = SplitInputs(q_nope, q_pe, k_nope, k_pe, v, seq_len, H, Hkv, scale)
    if with_prev:
        si.prev_out = randn_bf16((Nq, H, SPLIT_V), g)
        lo, hi = prev_lse_range
        si.prev_lse = lo + (hi - lo) * torch.rand((H, Nq), generator=g, dtype=torch.float32)
    return si


def split_lens(batch: int, lo: int, hi: int, seed: int):
    """Sequence lengths drawn uniformly from [lo, hi] (inclusive)."""
    g = _gen(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (batch,), generator=g)]


# ---------------------------------------------------------------------------
# paged decode
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class DecodeInputs:
    q: torch.Tensor            # [B, H, 576]
    cache: torch.Tensor        # [num_pages, page_size, 576]
    block_table: torch.Tensor  # int32 [B, max_pages]; unused slots hold -1
    lens: torch.Tensor         # int32 [B]
    page_size: int
    scale: float


def decode_inputs(lens, H: int, seed: int, page_size: int = 64, scale: float = SCALE_192,
                  extra_pages: int = 0) -> DecodeInputs:
    """A paged latent cache whose pages are handed out in a random permutation."""
    g = _gen(seed)
    lens = [int(x) for x in lens]
    B = len(lens)
    pages_per = [(n + page_size - 1) // page_size for n in lens]
    num_pages = sum(pages_per) + int(extra_pages)
    max_pages = max(1, max(pages_per) if pages_per else 1)
    perm = torch.randperm(num_pages, generator=g).to(torch.int32)
    block_table = torch.full((B, max_pages), -1, dtype=torch.int32)
    o = 0
    for b, n in enumerate(pages_per):
        block_table[b, :n] = perm[o:o + n]
        o += n
    q = randn_bf16((B, H, DK), g)
    cache = randn_bf16((num_pages, page_size, DK), g)
    return DecodeInputs(q, cache, block_table, torch.tensor(lens, dtype=torch.int32), page_size, scale)


def decode_lens(batch: int, lo: int, hi: int, seed: int):
    g = _gen(seed * 7919 + 1)
    return [int(x) for x in torch.randint(lo, hi + 1, (batch,), generator=g)]


# ---------------------------------------------------------------------------
# top-k sparse
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class SparseInputs:
    q_lift: torch.Tensor       # [B, S, H, 512]
    q_pe: torch.Tensor         # [B, S, H, 64]
    c_kv: torch.Tensor         # [B, S_kv, 512]
    k_pe: torch.Tensor         # [B, S_kv, 64]
    topk: torch.Tensor         # int32 [B, S, K]
    pos: torch.Tensor          # int64 [S]: global position of each query (for the recipe only)
    scale: float


def sparse_topk(S: int, S_kv: int, K: int, pos0: int, g: torch.Generator, pad_to: Optional[int] = None):
    """K distinct indices per query drawn uniformly from its causal prefix [0, pos].

    Queries whose prefix holds fewer than K rows list the whole prefix and pad
    the rest with -1.
    """
    rows = []
    for s in range(S):
        pos = pos0 + s
        n = min(pos + 1, S_kv)
        if n >= K:
            # uniform K-subset of [0, n): the K smallest of n uniform keys
            keys = torch.rand(n, generator=g)
            idx = torch.topk(keys, K, largest=False).indices.to(torch.int32)
        else:
            idx = torch.cat([torch.randperm(n, generator=g).to(torch.int32),
                             torch.full((K - n,), -1, dtype=torch.int32)])
        rows.append(idx)
    return torch.stack(rows, 0)


def sparse_inputs(S: int, S_kv: int, H: int, K: int, pos0: int, seed: int,
                  scale: float = SCALE_192, topk: Optional[torch.Tensor] = None) -> SparseInputs:
    g = _gen(seed)
    q_lift = randn_bf16((1, S, H, LATENT), g)
    q_pe = randn_bf16((1, S, H, ROPE), g)
    c_kv = randn_bf16((1, S_kv, LATENT), g)
    k_pe = randn_bf16((1, S_kv, ROPE), g)
    if topk is None:
        topk = sparse_topk(S, S_kv, K, pos0, g)
    topk = topk.reshape(1, S, -1).to(torch.int32)
    pos = torch.arange(pos0, pos0 + S, dtype=torch.int64)
    return SparseInputs(q_lift, q_pe, c_kv, k_pe, topk, pos, scale)


def sample_rows(n: int, count: int, seed: int, must=()) -> list:
    """A seeded sorted subset of range(n) of about ``count`` rows that always includes ``must``."""
    g = _gen(seed + 1000003)
    base = set(int(x) for x in must if 0 <= int(x) < n)
    if count >= n:
        return list(range(n))
    extra = torch.randperm(n, generator=g)[: max(0, count - len(base))].tolist()
    return sorted(base.union(int(x) for x in extra))


def randn_bf16_device(shape, seed: int, device) -> torch.Tensor:
    """fp32 N(0,1) rounded to bf16, drawn on the device by a seeded CUDA generator.

    Same distribution as randn_bf16, used for full-size timing inputs that the
    CPU generator would take tens of seconds to draw.
    """
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


# ---------------------------------------------------------------------------
# decode step inputs: RoPE angle table and the absorption weights
# ---------------------------------------------------------------------------
def rope_cos_sin(max_pos: int, base: float = 10000.0, rope: int = ROPE) -> torch.Tensor:
    """fp32 [max_pos, rope]: for position p the rope/2 cosines, then the sines, of the angles
    p * base^(-2i / rope) (the usual geometric frequency ladder; any table is valid input)."""
    inv = base ** (-torch.arange(0, rope, 2, dtype=torch.float64) / rope)
    ang = torch.arange(max_pos, dtype=torch.float64)[:, None] * inv[None, :]
    return torch.cat([torch.cos(ang), torch.sin(ang)], 1).to(torch.float32)


def absorb_weights(H: int, seed: int, nope: int = 128, v_head: int = 128):
    """Synthetic k_b_proj_trans [H, 512, nope] and v_b_proj [H, v_head, 512] (bf16), scaled so the
    lifted query and the projected output stay of order one for N(0,1) activations."""
    g = _gen(seed)
    wk = (torch.randn((H, LATENT, nope), generator=g) / nope ** 0.5).to(torch.bfloat16)
    wv = (torch.randn((H, v_head, LATENT), generator=g) / LATENT ** 0.5).to(torch.bfloat16)
    return wk, wv
