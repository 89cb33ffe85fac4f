"""Plant plausible mistakes in the oracle (on the CPU) and check the pins catch each.

Each mutant is the oracle's own source with one textual change (a dropped
term, a wrong sign, index or base, a transposed operand), loaded as a fresh
module; the pins of test_oracle_pins.py run against it and at least one of
them must fail.  The real oracle is never modified.
"""
import inspect
import types

import numpy as np
import pytest

import oracle.mla_oracle as mo
import tests.test_oracle_pins as pins

MUTANTS = {
    "scores drop the last column": ("s = scale * (q_rows @ keys.T)                  # [R, |J|]",
                                    "s = scale * (q_rows[:, :-1] @ keys[:, :-1].T)"),
    "scale applied twice": ("s = scale * (q_rows @ keys.T)                  # [R, |J|]",
                            "s = scale * scale * (q_rows @ keys.T)"),
    "masked scores drop the RoPE part": ("    s = scale * (q_rows @ keys.T)\n    s = np.where(visible, s, NEG_INF)",
                                         "    s = scale * (q_rows[:, :128] @ keys[:, :128].T)\n"
                                         "    s = np.where(visible, s, NEG_INF)"),
    "masked lse in base 2": ("lse = np.where(has, (m + np.log(l_safe))[:, 0], NEG_INF)",
                             "lse = np.where(has, (m + np.log2(l_safe))[:, 0], NEG_INF)"),
    "lse in base 2": ("lse = (m + np.log(l))[:, 0]", "lse = (m + np.log2(l))[:, 0]"),
    "lse without the max": ("lse = (m + np.log(l))[:, 0]", "lse = (np.log(l))[:, 0]"),
    "softmax not normalised": ("out = (p @ values) / l", "out = (p @ values)"),
    "causal off by one": ("n = min(n, q_pos0 + t - kv_pos0 + 1)", "n = min(n, q_pos0 + t - kv_pos0)"),
    "kv offset sign": ("n = min(n, q_pos0 + t - kv_pos0 + 1)", "n = min(n, q_pos0 + t + kv_pos0 + 1)"),
    "V taken from the RoPE end": ("o, l_ = attend(q[t], kv[J], kv[J, :dv], scale)",
                                  "o, l_ = attend(q[t], kv[J], kv[J, -dv:], scale)"),
    "merge weights swapped": ("out = (w_a[..., None] * out_a + w_b[..., None] * out_b)",
                              "out = (w_b[..., None] * out_a + w_a[..., None] * out_b)"),
    "merge lse missing log": ("lse = np.where(empty, NEG_INF, m_safe + np.log(np.where(empty, 1.0, w)))",
                              "lse = np.where(empty, NEG_INF, m_safe + np.where(empty, 1.0, w))"),
    "merge without the empty-row guard": [
        ("w_a = np.where(np.isneginf(lse_a), 0.0, np.exp(lse_a - m_safe))", "w_a = np.exp(lse_a - m)"),
        ("w_b = np.where(np.isneginf(lse_b), 0.0, np.exp(lse_b - m_safe))", "w_b = np.exp(lse_b - m)"),
        ("out = np.where(empty[..., None], 0.0, out)", "pass"),
    ],
    "sparse keeps padding": ("idx = idx[(idx >= 0) & (idx < S_kv)]", "idx = idx[idx < S_kv]"),
    "sparse drops duplicates": ("idx = idx[(idx >= 0) & (idx < S_kv)]",
                                "idx = np.unique(idx[(idx >= 0) & (idx < S_kv)])"),
    "decode page index transposed": ("return cache[bt[j // page_size], j % page_size]",
                                     "return cache[bt[j % page_size], j // page_size]"),
    "split GQA head map": ("g = h // group", "g = h % Hkv"),
    "split causal top-left": ("visible = j[None, :] <= (kl - ql + qi)[:, None]",
                              "visible = j[None, :] <= qi[:, None]"),
    "split rope/nope swapped in q": ("qrows = np.concatenate([qn[toks[sel], h], qp[toks[sel], h]], axis=1)",
                                     "qrows = np.concatenate([qp[toks[sel], h], qn[toks[sel], h]], axis=1)"),
    "masked softmax keeps hidden keys": [("s = np.where(visible, s, NEG_INF)", "pass"),
                                         ("p = np.where(visible, np.exp(s - m), 0.0)", "p = np.exp(s - m)")],
    "rope sine sign (interleaved)": ("out[..., 0::2] = a * c - b * s", "out[..., 0::2] = a * c + b * s"),
    "rope halves paired as neighbours": ("a, b = x[..., :n], x[..., n:]", "a, b = x[..., 0::2], x[..., 1::2]"),
    "rope second output uses cos twice": ("out[..., n:] = a * s + b * c", "out[..., n:] = a * c + b * c"),
    "appended row in the next slot": ("new_cache[page, pos[b] % page_size] =",
                                      "new_cache[page, (pos[b] + 1) % page_size] ="),
    "appended row keeps k_pe unrotated": ("np.concatenate([ck[b], rope(kp[b], c, s, is_neox)])",
                                          "np.concatenate([ck[b], kp[b]])"),
    "absorb sums over the latent axis": ('return np.einsum("thd,hld->thl", _f64(q_nope), _f64(k_b_proj_trans))',
                                         'return np.einsum("thd,hld->thl", _f64(q_nope), '
                                         '_f64(k_b_proj_trans)[:, ::-1, :])'),
    "multi-token decode: every token sees all keys": ("n = max(0, int(ln[b]) - S + 1 + i)", "n = int(ln[b])"),
    "multi-token decode: token order reversed": ("n = max(0, int(ln[b]) - S + 1 + i)",
                                                  "n = max(0, int(ln[b]) - i)"),
    "fp8 cache scale dropped": ("return mla_decode_ex(q, _f64(cache_e4m3) * float(kv_scale), block_table,",
                                "return mla_decode_ex(q, _f64(cache_e4m3), block_table,"),
    "sink weight ignored": ("out, lse = merge(out, lse, np.zeros_like(out), np.broadcast_to(sk, lse.shape))",
                            "pass"),
    "project_out with the head's weight of the next head": (
        'return np.einsum("thl,hvl->thv", _f64(o_latent), _f64(v_b_proj))',
        'return np.einsum("thl,hvl->thv", _f64(o_latent), np.roll(_f64(v_b_proj), 1, axis=0))'),
}


def _mutant_module(subs) -> types.ModuleType:
    src = inspect.getsource(mo)
    if isinstance(subs, tuple):
        subs = [subs]
    for old, new in subs:
        assert src.count(old) == 1, f"mutation anchor not unique/found: {old!r}"
        src = src.replace(old, new)
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src, "<oracle_mutant>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    mut = _mutant_module(MUTANTS[name])
    monkeypatch.setattr(pins, "mo", mut)
    caught = []
    for check in pins.ALL_CHECKS:
        try:
            with np.errstate(all="ignore"):
                check()
        except Exception:  # any failure (assertion, NaN, index error) counts as caught
            caught.append(check.__name__)
    assert caught, f"no pin caught the planted mistake: {name}"


def test_real_oracle_passes_all_pins():
    for check in pins.ALL_CHECKS:
        check()
